"""GPU parity of svp_dvl_allocate_pack against the allocator / packer reference
(oracle/dvl.py): integer outputs bit-exact ("DScale", SIII-C, Algorithm 1, Fig. 6)."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_packed_gb300 as svp
from oracle import dvl

pytestmark = pytest.mark.gpu

FIG6_GROW = [[1, 1, 1, 1, 0.6], [1] * 9 + [0.55], [1] * 6 + [0.52], [1] * 8 + [0.51]]


def _scores(rows, w=16):
    s = np.zeros((len(rows), w - 1), dtype=np.float32)
    for i, r in enumerate(rows):
        s[i, :len(r)] = r
    return s


def _run(s, n_live, per, m_cap, fields=True, seed=0, fills=(0, 0, -1), reference=True):
    n_bs, wm1 = s.shape
    w = wm1 + 1
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, 250000, (n_bs, w)).astype(np.int32)
    pos = rng.integers(0, 1 << 20, (n_bs, w)).astype(np.int32)
    ref = rng.integers(0, 1 << 30, (n_bs, w)).astype(np.int32)
    t = lambda a: torch.from_numpy(a).cuda()
    nl = torch.tensor([n_live], dtype=torch.int32, device="cuda")
    ws = svp.Workspace(256)
    g = svp.dvl_allocate_pack(t(s), n_live=nl, budget_per_req=per, m_cap=m_cap,
                              tokens=t(tok) if fields else None, positions=t(pos) if fields else None,
                              kv_refs=t(ref) if fields else None, fill_token=fills[0], fill_pos=fills[1],
                              fill_ref=fills[2], ws=ws)
    torch.cuda.synchronize()
    if not reference:
        return g, None, ws
    o = dvl.dvl_allocate_pack(s, n_live, per, m_cap, tok if fields else None, pos if fields else None,
                              ref if fields else None, *fills)
    return g, o, ws


def _assert_same(g, o, fields=True):
    assert g["k_init"].cpu().tolist() == o["k0"].tolist()
    assert g["k"].cpu().tolist() == o["k"].tolist()
    assert g["cu_slots"].cpu().tolist() == o["cu"].tolist()
    assert int(g["n_adjust"].item()) == o["adjustments"]
    if fields:
        for name in ("tokens", "positions", "kv_refs"):
            assert g[name].cpu().tolist() == o[name].tolist(), name


def test_fig6_on_gpu():
    g, o, ws = _run(_scores(FIG6_GROW), 4, 8, 64)
    _assert_same(g, o)
    assert g["k"].cpu().tolist() == [6, 10, 7, 9]
    assert g["cu_slots"].cpu().tolist() == [0, 6, 16, 23, 32]
    assert ws.read_status() == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_batches_match_reference(seed):
    rng = np.random.default_rng(1000 + seed)
    n_bs = int(rng.choice([1, 3, 8, 64, 257, 1024, 2048]))
    n_live = int(rng.integers(0, n_bs + 1))
    per = int(rng.integers(1, 17))
    kind = seed % 4
    if kind == 0:
        s = rng.random((n_bs, 15))
    elif kind == 1:
        s = rng.beta(0.4, 0.4, (n_bs, 15))
    elif kind == 2:      # heavy ties: few distinct values
        s = rng.integers(0, 5, (n_bs, 15)) / 4.0
    else:                # sorted, near-threshold sums
        s = np.sort(rng.random((n_bs, 15)), axis=1)[:, ::-1] * 1.02
    s = s.astype(np.float32)
    g, o, ws = _run(s, n_live, per, 16 * n_bs, seed=seed)
    _assert_same(g, o)
    assert ws.read_status() == 0


@pytest.mark.parametrize("w", [2, 5, 16])
@pytest.mark.parametrize("n", [20, 40])   # a quarter block and a full block of threads
def test_widths_and_extremes(w, n):
    rng = np.random.default_rng(w)
    for s in (np.ones((n, w - 1)), np.zeros((n, w - 1)), rng.random((n, w - 1))):
        for per in sorted({1, max(1, w // 2), w}):
            g, o, ws = _run(s.astype(np.float32), n, per, w * n + 5, seed=w)
            _assert_same(g, o)


@pytest.mark.parametrize("n_bs", [1, 2, 17, 31, 32, 33])
def test_small_batch_sizes(n_bs):
    """Small batches (fewer requests than a warp, about one warp, one more): the kernel
    agrees with the reference on growing, shrinking and tie-heavy batches, with all, some
    or none of the requests live."""
    rng = np.random.default_rng(500 + n_bs)
    for kind in range(3):
        if kind == 0:
            s = rng.random((n_bs, 15))
        elif kind == 1:
            s = rng.integers(0, 3, (n_bs, 15)) / 2.0      # few distinct values: many ties
        else:
            s = rng.beta(0.3, 0.3, (n_bs, 15))
        s = s.astype(np.float32)
        for n_live in sorted({n_bs, max(0, n_bs - 3), 0}):
            for per in (1, 4, 16):
                g, o, ws = _run(s, n_live, per, 16 * n_bs + 2, seed=kind)
                _assert_same(g, o)
                assert ws.read_status() == 0


def test_no_fields_and_bad_live_count():
    s = np.random.default_rng(3).random((16, 15)).astype(np.float32)
    g, o, ws = _run(s, 10, 8, 160, fields=False)
    _assert_same(g, o, fields=False)
    assert ws.read_status() == 0
    # more live requests than the bucket holds: status bit, everything inactive
    g, _, ws = _run(s, 17, 8, 160, fields=True, reference=False)
    assert ws.read_status() == svp.DEV_BAD_SLOTS
    assert g["k"].cpu().tolist() == [0] * 16
    assert g["cu_slots"].cpu().tolist() == [0] * 17
    assert g["tokens"].cpu().tolist() == [0] * 160
    # budget beyond m_cap
    g, _, ws = _run(s, 10, 8, 79, fields=False, reference=False)
    assert ws.read_status() == svp.DEV_BAD_SLOTS


def test_gather_rows_single_and_multi():
    """Row-mapped packing of wide fields: dst[r] = src[idx[r]] for ids in range, zeros
    otherwise (the packer's placeholder reference -1 and ids past the source), for one field
    and for four fields of different widths in one launch."""
    g = torch.Generator().manual_seed(3)
    src_rows, rows = 37, 29
    idx = torch.randint(-1, src_rows + 3, (rows,), generator=g, dtype=torch.int32)
    idx[0], idx[1], idx[2] = -1, src_rows, src_rows - 1
    fields = [torch.randn(src_rows, 8, 16, generator=g).to(torch.bfloat16),
              torch.randn(src_rows, 2, 16, generator=g).to(torch.bfloat16),
              torch.randint(0, 1 << 20, (src_rows, 4), generator=g, dtype=torch.int32),
              torch.randn(src_rows, 1000, generator=g)]

    def expect(src):
        out = torch.zeros((rows,) + tuple(src.shape[1:]), dtype=src.dtype)
        for r in range(rows):
            if 0 <= int(idx[r]) < src_rows:
                out[r] = src[int(idx[r])]
        return out

    d_idx = idx.cuda()
    one = svp.gather_rows(fields[0].cuda(), d_idx)
    outs = svp.gather_rows_multi([f.cuda() for f in fields], d_idx)
    torch.cuda.synchronize()
    assert torch.equal(one.cpu(), expect(fields[0]))
    for f, o in zip(fields, outs):
        assert torch.equal(o.cpu(), expect(f))
    with pytest.raises(ValueError):
        svp.gather_rows_multi([fields[0].cuda()] * (svp.GATHER_MAX_FIELDS + 1), d_idx)

"""GPU parity of svp_draft_features / svp_act_truncate against oracle/features.py
("DScale" SIII-C Acceptance predictor; DFlash-Mini-Lab DFlash7-ACT).  The top logit is a
stored value (bit-exact); the gaps are fp32 differences of stored values (within one fp32
rounding of the fp64 reference); log-probability and entropy come from fp32 sums (bars
below).  ACT decisions are bit-exact given the same margins."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_packed_gb300 as svp
from oracle import features as ft

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [(0, 40, 300, torch.bfloat16, 0), (1, 17, 1001, torch.float32, 0),
                                  (2, 12, 10000, torch.bfloat16, 8), (3, 9, 248320, torch.bfloat16, 0),
                                  (4, 6, 40007, torch.float32, 3)])
def test_features_match_reference(case):
    seed, rows, V, dtype, pad = case
    g = torch.Generator().manual_seed(seed)
    z = (torch.randn(rows, V + pad, generator=g) * 2.0).to(dtype)
    z[1, 7] = z[1].max() + 1.0
    z[1, 70] = z[1, 7]                    # repeated maximum: gap 2 = 0
    ref = ft.draft_features(z.float().numpy()[:, :V].astype(np.float64))
    ws = svp.Workspace(svp.draft_features_workspace_size(rows, V))
    out = svp.draft_features(z.cuda(), vocab=V, ws=ws).cpu().numpy().astype(np.float64)
    assert out[:, 0].tolist() == ref[:, 0].tolist()
    assert np.all(np.abs(out[:, 1:16] - ref[:, 1:16]) <= 6e-8 * np.maximum(np.abs(ref[:, 1:16]), np.abs(ref[:, :1])))
    assert out[1, 1] == 0.0
    assert np.abs(out[:, 16] - ref[:, 16]).max() <= 1e-4
    assert np.abs(out[:, 17] - ref[:, 17]).max() <= 1e-4 * max(1.0, np.log(V))
    # the workspace tickets are back at zero: a second call on the same workspace agrees
    out2 = svp.draft_features(z.cuda(), vocab=V, ws=ws).cpu().numpy().astype(np.float64)
    assert np.array_equal(out, out2)


def test_act_truncation():
    rng = np.random.default_rng(5)
    n, w, V = 32, 16, 4096
    z = (torch.randn(n * (w - 1), V) * 2.0).to(torch.bfloat16)
    feats = svp.draft_features(z.cuda())
    margins = feats[:, 1].contiguous()
    mg = margins.cpu().numpy().reshape(n, w - 1)
    for thr in (0.0, 0.25, 0.5, 1.0, 1.5, 2.0, 1e9):
        # stride 18 with the margin column: pass a view starting at column 1
        k = svp.act_truncate(feats.view(-1)[1:].contiguous(), n=n, w=w, threshold=thr, stride=18)
        k1 = svp.act_truncate(margins, n=n, w=w, threshold=thr, stride=1)
        expect = ft.act_truncate(mg, thr)
        assert k.cpu().tolist() == expect.tolist()
        assert k1.cpu().tolist() == expect.tolist()
    assert svp.act_truncate(margins, n=n, w=w, threshold=0.0).cpu().tolist() == [w] * n


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_features_adversarial_layouts(dtype):
    """Rows whose top values share one lane position (every 256th element, so a kernel that
    keeps a few values per lane stream must notice and recover), a row of equal values, a
    row with -inf entries and fewer than 16 finite values, and a row whose top-16 sits in
    one contiguous run."""
    V = 20000
    g = torch.Generator().manual_seed(9)
    z = torch.randn(5, V, generator=g) * 2.0
    idx = 5 + 256 * torch.arange(20)
    z[0, idx] = 20.0 + torch.arange(20, dtype=torch.float32) * 0.25
    z[1] = 1.5
    z[2] = -float("inf")
    z[2, torch.tensor([3, 700, 9000, 19999])] = torch.tensor([1.0, 4.0, -2.0, 0.5])
    z[3, 1000:1016] = 30.0 - torch.arange(16, dtype=torch.float32)
    z[4, idx[:6]] = 25.0
    z = z.to(dtype)
    ref = ft.draft_features(z.float().numpy().astype(np.float64))
    out = svp.draft_features(z.cuda()).cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref[:, 1:16])
    assert out[:, 0].tolist() == ref[:, 0].tolist()
    assert np.array_equal(np.isfinite(out[:, 1:16]), fin)
    d = np.abs(np.where(fin, out[:, 1:16], 0.0) - np.where(fin, ref[:, 1:16], 0.0))
    assert np.all(d <= 6e-8 * np.maximum(np.abs(np.where(fin, ref[:, 1:16], 0.0)), np.abs(ref[:, :1])))
    assert np.abs(out[:, 16] - ref[:, 16]).max() <= 1e-4
    assert np.abs(out[:, 17] - ref[:, 17]).max() <= 1e-4 * np.log(V)


def test_full_size_wide_gqa_sampled_rows():
    """The launch the bench times: 192 draft rows x 248,320 bf16; sampled rows against the
    oracle."""
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    b = wl.make_batch("wide_gqa_bf16", seed=0, device="cuda")
    z = b.draft_logits
    rows, V = z.shape
    ws = svp.Workspace(svp.draft_features_workspace_size(rows, V))
    out = svp.draft_features(z, ws=ws).cpu().numpy().astype(np.float64)
    pick = [0, 1, 63, 64, 127, 150, rows - 1]
    ref = ft.draft_features(z[pick].float().cpu().numpy().astype(np.float64))
    o = out[pick]
    assert o[:, 0].tolist() == ref[:, 0].tolist()
    assert np.all(np.abs(o[:, 1:16] - ref[:, 1:16]) <= 6e-8 * np.maximum(np.abs(ref[:, 1:16]), np.abs(ref[:, :1])))
    assert np.abs(o[:, 16] - ref[:, 16]).max() <= 1e-4
    assert np.abs(o[:, 17] - ref[:, 17]).max() <= 1e-4 * np.log(V)
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("rows,V,pad", [(4000, 1000, 0), (4500, 2999, 1)])
def test_features_several_units_per_warp(rows, V, pad):
    """More rows than resident warps: warps take several (row, chunk) units in turn, each
    chunk ending in a partial batch (and, for V = 2999, a tail of fewer than 8 values)."""
    g = torch.Generator().manual_seed(rows)
    z = (torch.randn(rows, V + pad, generator=g) * 3.0).to(torch.bfloat16)
    ref = ft.draft_features(z.float().numpy()[:, :V].astype(np.float64))
    ws = svp.Workspace(svp.draft_features_workspace_size(rows, V))
    out = svp.draft_features(z.cuda(), vocab=V, ws=ws).cpu().numpy().astype(np.float64)
    assert out[:, 0].tolist() == ref[:, 0].tolist()
    assert np.all(np.abs(out[:, 1:16] - ref[:, 1:16]) <= 6e-8 * np.maximum(np.abs(ref[:, 1:16]), np.abs(ref[:, :1])))
    assert np.abs(out[:, 16] - ref[:, 16]).max() <= 1e-4
    assert np.abs(out[:, 17] - ref[:, 17]).max() <= 1e-4 * np.log(V)


def test_workspace_reused_across_sizes():
    """One workspace, sized for the largest call, serves calls with other row counts and
    vocabularies: every call leaves it zeroed, so no stale partial list lands in a later
    call's row tickets (the layout moves with the row count)."""
    shapes = [(232, 60000, torch.bfloat16), (270, 4099, torch.float32), (17, 1001, torch.float32),
              (300, 20000, torch.bfloat16), (40, 248320, torch.bfloat16)]
    ws = svp.Workspace(max(svp.draft_features_workspace_size(r, V) for r, V, _ in shapes))
    for i, (rows, V, dtype) in enumerate(shapes):
        g = torch.Generator().manual_seed(50 + i)
        z = (torch.randn(rows, V, generator=g) * 2.0).to(dtype)
        ref = ft.draft_features(z.float().numpy().astype(np.float64))
        out = svp.draft_features(z.cuda(), ws=ws).cpu().numpy().astype(np.float64)
        assert out[:, 0].tolist() == ref[:, 0].tolist(), (rows, V)
        assert np.all(np.abs(out[:, 1:16] - ref[:, 1:16]) <= 6e-8 * np.maximum(np.abs(ref[:, 1:16]), np.abs(ref[:, :1])))
        assert np.abs(out[:, 16] - ref[:, 16]).max() <= 1e-4
        assert np.abs(out[:, 17] - ref[:, 17]).max() <= 1e-4 * np.log(V)
    assert torch.count_nonzero(ws.buf[256:]).item() == 0   # all zero again past the header

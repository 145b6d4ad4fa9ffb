"""Shared helpers for the GPU parity tests: run the CUDA path through the binding and
the fp64 oracle on the same seeded batch, and compare."""
import numpy as np
import torch

import oracle
import speculative_decoding_verification_packed_gb300 as svp

BF16_MAX_ABS = 2e-2     # attention bars for bf16 inputs with fp32 accumulation
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-4      # attention bar for fp32 inputs
# lse for bf16 inputs: the row sum l is accumulated from P rounded to bf16 (the same
# weights O uses), so |d l / l| <= 2^-9 and |d lse| <= ln(1 + 2^-9) ~ 1.95e-3; bar 2x that.
BF16_LSE_ABS = 4e-3


def to_dev(b, device="cuda"):
    """Copy every tensor field of a workloads.Batch to the device (new object)."""
    import copy
    d = copy.copy(b)
    for name, val in vars(b).items():
        if isinstance(val, torch.Tensor):
            setattr(d, name, val.to(device))
    d.full = {}
    return d


def gpu_verify(bd, tile_mode=svp.TILE_AUTO, w=None, out=None, lse=None, expect_status=0):
    """Run the CUDA path with a fresh workspace; check the device status word."""
    kw = {}
    if bd.paged:
        kw = dict(k_cache=bd.k_cache, v_cache=bd.v_cache, block_table=bd.block_table)
    else:
        kw = dict(k_ctx=bd.k_ctx, v_ctx=bd.v_ctx, cu_ctx=bd.cu_ctx)
    w = w or bd.W
    ws = svp.Workspace(svp.verify_attn_workspace_size(bd.n, bd.m_cap, w, bd.hq, bd.hkv, bd.d,
                                                      bd.q.dtype, tile_mode))
    out, lse = svp.verify_attn_packed(bd.q, bd.k_new, bd.v_new, bd.ctx_len, bd.cu_slots,
                                      w=w, tile_mode=tile_mode, out=out, lse=lse, ws=ws, **kw)
    torch.cuda.synchronize()
    st = ws.read_status()
    assert st == expect_status, f"device status {st:#x}"
    return out, lse


def oracle_verify(b, requests=None, threads=16):
    """b: CPU batch."""
    if b.paged:
        return oracle.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv,
                                scale=b.scale, k_cache=b.k_cache, v_cache=b.v_cache,
                                block_table=b.block_table, cache_strides=b.cache_strides,
                                requests=requests, threads=threads)
    return oracle.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv,
                            scale=b.scale, k_ctx=b.k_ctx, v_ctx=b.v_ctx, cu_ctx=b.cu_ctx,
                            requests=requests, threads=threads)


def rows_of(b, requests=None):
    cu = b.cu_slots.tolist()
    reqs = range(b.n) if requests is None else requests
    rows = []
    for i in reqs:
        rows.extend(range(cu[i], cu[i + 1]))
    return np.array(rows, dtype=np.int64)


def compare_attention(out_gpu, lse_gpu, ref_o, ref_l, rows, dtype):
    """Element-wise comparison on the given packed rows; returns error stats."""
    o = out_gpu.float().cpu().numpy()[rows]
    r = ref_o[rows]
    bad_g = np.argwhere(~np.isfinite(o))
    bad_r = np.argwhere(~np.isfinite(r))
    assert bad_g.size == 0 and bad_r.size == 0, (
        f"non-finite: gpu {len(bad_g)} (first {bad_g[:4].tolist()}), "
        f"oracle {len(bad_r)} (first {bad_r[:4].tolist()}), rows {rows[:3].tolist()}...")
    err = np.abs(o.astype(np.float64) - r)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()),
                 max_rel=float((err / np.maximum(np.abs(r), 1e-3)).max()))
    if lse_gpu is not None:
        le = np.abs(lse_gpu.cpu().numpy()[rows].astype(np.float64) - ref_l[rows])
        stats["lse_max_abs"] = float(le.max())
    if dtype == torch.float32:
        assert stats["max_abs"] <= F32_MAX_ABS, stats
        if lse_gpu is not None:
            assert stats["lse_max_abs"] <= F32_MAX_ABS, stats
    else:
        assert stats["max_abs"] <= BF16_MAX_ABS, stats
        assert stats["mean_abs"] <= BF16_MEAN_ABS, stats
        if lse_gpu is not None:
            assert stats["lse_max_abs"] <= BF16_LSE_ABS, stats
    assert np.isfinite(o).all()
    return stats


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.int32)


def check_margin_rows(logits_cpu, outs, rows=None):
    """Row top-1 index, top-1, top-2 and margin bit for bit against the oracle's scalar
    scan (NaN margins must match as NaN); returns the oracle's argmax indices."""
    idx, t1, t2, mg = (o.cpu().numpy() for o in outs[:4])
    r_idx, r_t1, r_t2, r_mg = oracle.row_top2(logits_cpu)
    sel = slice(None) if rows is None else rows
    assert np.array_equal(idx[sel], r_idx[sel])
    assert np.array_equal(_bits(t1[sel]), _bits(r_t1[sel]))
    assert np.array_equal(_bits(t2[sel]), _bits(r_t2[sel]))
    ok = (_bits(mg[sel]) == _bits(r_mg[sel])) | (np.isnan(mg[sel]) & np.isnan(r_mg[sel]))
    assert ok.all()
    return r_idx

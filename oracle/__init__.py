"""fp64 CPU oracle for packed speculative verification -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library never imports, links or calls it, and it
shares no code with the CUDA library: the arithmetic lives in ``svp_oracle.c`` (plain
C, fp64), compiled here with gcc, and in the two small pure-Python functions below.

What it computes, with the passages it follows:

* ``attention``       -- masked softmax attention of every packed candidate row over its
  request's KV context followed by its own candidates 0..j, straight from the
  definition in fp64 ("DScale: Scaling Block-Diffusion Speculative Decoding with
  Adaptive Verification", SIII-D: valid rows read offset_i + j with request-local
  causal masking; SIII-B: each block handles one request's query tile for one head).
* ``row_top2``        -- per-row top-1 value/index, top-2 value and fp32 margin
  (DFlash-Mini-Lab README, DFlash7-ACT top-1/top-2 margin; DScale SII-B, Fig. 4).
* ``greedy_accept``   -- longest matching draft prefix and the successor token
  (DScale SIII-D, Prefix verifier at temperature 0; DFlash-Mini-Lab "accept exact
  prefix").
* ``offsets``         -- exclusive prefix sum of slot counts (DScale SIII-C, Flat-buffer
  packer, Fig. 6).
* ``inactive_row_fraction`` -- query-row capacity and idle fraction of a tile of height
  B for a request of length l (DScale SIII-B; the equation itself is missing from the
  page text, the reading capacity = B*ceil(l/B) is pinned by 112 of 128 rows at l=16,
  B=128 in SII-A).

* ``dvl`` (oracle/dvl.py) -- the DVL budget allocator and flat-buffer packer of
  Algorithm 1 (DScale SIII-C): prefix scores, initial lengths, grow / shrink to the
  budget, offsets, row-mapped packing with tail placeholders, and the retention measure
  of SIV.

* ``stochastic`` (oracle/stochastic.py) -- the stochastic prefix verifier at temperature
  T > 0 (DScale SIII-D, Prefix verifier): deterministic draft candidates accepted with the
  target probability, the successor drawn from the target with the rejected candidate
  removed (or unmodified after a full accept), random numbers given as inputs; plus the
  exact output law of one request.

* ``features`` (oracle/features.py) -- the 18 draft-signal values per draft-logit row
  (DScale SIII-C, Acceptance predictor) and DFlash7-ACT margin-threshold truncation
  (DFlash-Mini-Lab README).

Pins (tests/test_oracle_*.py): brute force on tiny inputs, closed forms, the packed vs
alone / relayout / paged vs contiguous / permutation invariants, numpy argmax and sort
on planted ties, exhaustive accept patterns, and the worked examples the pages print
(tests/golden/).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sysconfig
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "svp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liborc.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile svp_oracle.c with gcc into oracle/liborc.so (a checker, not the product)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.orc_attention.restype = ctypes.c_int
        lib.orc_attention.argtypes = [
            ctypes.c_int, i32, i32, i32, i32, f64,
            vp, vp, vp,
            ctypes.c_int, vp, vp, vp,
            vp, i32, i32, i64, i64, i64,
            vp, vp, vp,
            i32, vp, vp]
        lib.orc_row_top2.restype = None
        lib.orc_row_top2.argtypes = [ctypes.c_int, vp, i64, i32, i32, vp, vp, vp, vp]
        lib.orc_greedy_accept.restype = None
        lib.orc_greedy_accept.argtypes = [vp, vp, vp, i32, vp, vp]
        lib.orc_offsets.restype = None
        lib.orc_offsets.argtypes = [vp, i32, vp]
        _lib = lib
    return _lib


def _raw(t, dtype_code: Optional[int] = None):
    """numpy view of a CPU torch tensor / numpy array holding fp32 or bf16 storage."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().contiguous()
            if t.device.type != "cpu":
                raise ValueError("oracle inputs must live on the CPU")
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), BF16
            if t.dtype == torch.float32:
                return t.numpy(), F32
            if t.dtype == torch.int32:
                return t.numpy(), None
            if t.dtype == torch.int64:
                return t.numpy(), None
            if t.dtype == torch.uint8 or t.dtype == torch.bool:
                return t.to(torch.uint8).numpy(), None
            raise TypeError(f"unsupported tensor dtype {t.dtype}")
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    return a, None


def _ptr(a) -> int:
    return 0 if a is None else a.ctypes.data


def attention(q, k_new, v_new, ctx_len, cu_slots, *, hkv: int, scale: float,
              k_ctx=None, v_ctx=None, cu_ctx=None,
              k_cache=None, v_cache=None, block_table=None, page_size: int = 16,
              cache_strides: Optional[Sequence[int]] = None,
              requests: Optional[Sequence[int]] = None, threads: int = 1):
    """fp64 attention of every packed candidate row (see module docstring).

    q: [m_cap, hq, d]; k_new, v_new: [m_cap, hkv, d]; all fp32 or all bf16.
    Contiguous context: k_ctx, v_ctx [sum L, hkv, d] with cu_ctx [n+1] (int64).
    Paged context: k_cache, v_cache with cache_strides = (page, head, token) in
    elements and block_table [n, max_pages] (int32).
    Returns (out [m_cap, hq, d] float64, lse [m_cap, hq] float64); rows outside every
    request, and rows of requests not listed in ``requests``, are NaN.
    """
    lib = _load()
    qa, dt = _raw(q)
    kna, dt2 = _raw(k_new)
    vna, dt3 = _raw(v_new)
    if not (dt == dt2 == dt3) or dt is None:
        raise TypeError("q, k_new, v_new must share one float dtype (fp32 or bf16)")
    m_cap, hq, d = qa.shape
    ctx_len_a = np.ascontiguousarray(_raw(ctx_len)[0], dtype=np.int32)
    cu_a = np.ascontiguousarray(_raw(cu_slots)[0], dtype=np.int32)
    n = ctx_len_a.shape[0]
    paged = k_cache is not None
    if paged:
        kca, _ = _raw(k_cache)
        vca, _ = _raw(v_cache)
        bta = np.ascontiguousarray(_raw(block_table)[0], dtype=np.int32)
        max_pages = bta.shape[1] if bta.ndim == 2 else 0
        s_page, s_head, s_tok = cache_strides
        kc, vc, cuc = kca, vca, None
    else:
        kc, _ = _raw(k_ctx)
        vc, _ = _raw(v_ctx)
        cuc = np.ascontiguousarray(_raw(cu_ctx)[0], dtype=np.int64)
        bta, max_pages, s_page, s_head, s_tok = None, 0, 0, 0, 0
    want = None
    if requests is not None:
        want = np.zeros(max(n, 1), dtype=np.uint8)
        want[np.asarray(list(requests), dtype=np.int64)] = 1
    out = np.full((m_cap, hq, d), np.nan, dtype=np.float64)
    lse = np.full((m_cap, hq), np.nan, dtype=np.float64)
    rc = lib.orc_attention(dt, n, hq, hkv, d, float(scale),
                           _ptr(qa), _ptr(kna), _ptr(vna),
                           int(paged), _ptr(kc), _ptr(vc), _ptr(cuc),
                           _ptr(bta), int(max_pages), int(page_size),
                           int(s_page), int(s_head), int(s_tok),
                           _ptr(ctx_len_a), _ptr(cu_a), _ptr(want),
                           int(threads), _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle attention failed (rc={rc})")
    return out, lse


def row_top2(logits, row_stride: Optional[int] = None):
    """Per-row (top1_idx int32, top1 f32, top2 f32, margin f32) of a [rows, V] array."""
    lib = _load()
    la, dt = _raw(logits)
    if dt is None:
        raise TypeError("logits must be fp32 or bf16")
    rows, vocab = la.shape
    stride = vocab if row_stride is None else row_stride
    idx = np.zeros(rows, dtype=np.int32)
    t1 = np.zeros(rows, dtype=np.float32)
    t2 = np.zeros(rows, dtype=np.float32)
    mg = np.zeros(rows, dtype=np.float32)
    lib.orc_row_top2(dt, _ptr(la), int(stride), int(rows), int(vocab),
                     _ptr(idx), _ptr(t1), _ptr(t2), _ptr(mg))
    return idx, t1, t2, mg


def greedy_accept(target_argmax, tokens, cu_slots):
    """(accept_len [n] int32, next_token [n] int32) -- see module docstring."""
    lib = _load()
    am = np.ascontiguousarray(_raw(target_argmax)[0], dtype=np.int32)
    tk = np.ascontiguousarray(_raw(tokens)[0], dtype=np.int32)
    cu = np.ascontiguousarray(_raw(cu_slots)[0], dtype=np.int32)
    n = cu.shape[0] - 1
    acc = np.zeros(max(n, 0), dtype=np.int32)
    nxt = np.zeros(max(n, 0), dtype=np.int32)
    lib.orc_greedy_accept(_ptr(am), _ptr(tk), _ptr(cu), int(n), _ptr(acc), _ptr(nxt))
    return acc, nxt


def offsets(k) -> np.ndarray:
    """cu_slots [n+1] = exclusive prefix sum of the slot counts k [n]."""
    lib = _load()
    ka = np.ascontiguousarray(np.asarray(k), dtype=np.int32)
    cu = np.zeros(ka.shape[0] + 1, dtype=np.int32)
    lib.orc_offsets(_ptr(ka), int(ka.shape[0]), _ptr(cu))
    return cu


def inactive_row_fraction(ell: int, B: int):
    """(capacity, idle fraction) of a height-B tile for a request of length ell > 0."""
    cap = B * math.ceil(ell / B)
    return cap, 1.0 - ell / cap

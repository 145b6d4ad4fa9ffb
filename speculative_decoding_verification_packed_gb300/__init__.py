"""Packed speculative-verification attention and margin/accept for GB300 (sm_103a).

A thin Python binding over the C ABI of ``include/svp.h`` (``libsvp.so``, built in-tree
by ``build.py``).  The functions here only marshal torch CUDA tensors into pointers,
sizes and the current stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing or the tensors are
not on a CUDA device, the call raises.

Entry points (same names as the C ABI, without the ``svp_`` prefix):
  verify_attn_packed   attention of packed candidate rows over their request's KV
                       context and their own earlier candidates (contiguous or paged KV,
                       GQA); ``tile_mode`` selects the contrast tiles
  prefill_attn         wide-tile causal prefill attention
  draft_margin         per-row top-1 index/value, top-2 value and fp32 margin
  greedy_accept        longest matching draft prefix and successor token per request
  margin_accept        draft_margin over packed target rows fused with greedy_accept
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsvp.so")

SVP_OK, SVP_EINVAL, SVP_EUNSUPPORTED, SVP_EWORKSPACE, SVP_ECUDA = 0, 1, 2, 3, 4
SVP_F32, SVP_BF16 = 0, 1
TILE_AUTO, TILE_SHORT, TILE_FIXED128, TILE_WIDE, TILE_SHORT_UNPACKED = 0, 1, 2, 3, 4
DEV_BAD_SLOTS, DEV_BAD_CONTEXT, DEV_TIMEOUT, DEV_WORKSPACE = 0x1, 0x2, 0x4, 0x8


class SvpError(RuntimeError):
    """A library call returned a non-OK status."""

    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class svp_heads(ctypes.Structure):
    _fields_ = [("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class svp_kv(ctypes.Structure):
    _fields_ = [("paged", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("cu_ctx", ctypes.c_void_p), ("total_tokens", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int64),
                ("stride_page", ctypes.c_int64), ("stride_head", ctypes.c_int64),
                ("stride_tok", ctypes.c_int64)]


class svp_gather_field(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("src_rows", ctypes.c_int64),
                ("row_bytes", ctypes.c_int64), ("dst", ctypes.c_void_p)]


GATHER_MAX_FIELDS = 8

_lib = None

_SIGS = {
    "svp_version": (ctypes.c_int32, []),
    "svp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "svp_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "svp_read_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.POINTER(ctypes.c_int32)]),
    "svp_verify_attn_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(svp_heads), ctypes.c_int,
        ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "svp_verify_attn_packed": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(svp_kv),
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(svp_heads), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "svp_verify_attn_packed_ex": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(svp_kv),
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(svp_heads), ctypes.c_int, ctypes.c_int32, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "svp_prefill_attn_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(svp_heads), ctypes.c_int,
        ctypes.POINTER(ctypes.c_size_t)]),
    "svp_prefill_attn": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(svp_heads), ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "svp_draft_margin_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "svp_draft_margin": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]),
    "svp_greedy_accept": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "svp_margin_accept_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "svp_dvl_allocate_pack": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]),
    "svp_gather_rows": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p]),
    "svp_gather_rows_multi": (ctypes.c_int, [
        ctypes.POINTER(svp_gather_field), ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p]),
    "svp_stochastic_accept_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "svp_stochastic_accept": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]),
    "svp_draft_features_workspace_size": (ctypes.c_int, [
        ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "svp_draft_features": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "svp_act_truncate": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
        ctypes.c_void_p, ctypes.c_void_p]),
    "svp_margin_accept": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]),
}


def lib() -> ctypes.CDLL:
    """The loaded libsvp.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libsvp.so is not built ({LIB_PATH}); run "
                "`python -m speculative_decoding_verification_packed_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().svp_status_string(int(status)).decode()
    except Exception:  # library missing: still produce a message
        return f"status {status}"


def _check(status: int, what: str) -> None:
    if status != SVP_OK:
        raise SvpError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SVP_BF16
    if t.dtype == torch.float32:
        return SVP_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _dev(t: Optional[torch.Tensor], name: str, dtype=None) -> int:
    if t is None:
        return 0
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Workspace:
    """Device scratch for one entry point, zeroed once at creation (svp_workspace_init).

    The clear is enqueued on ``stream`` (default: the current stream).  A call on another
    stream must be ordered after it (the same stream, a synchronize, or an event): torch's
    side streams do not wait for the default stream."""

    def __init__(self, nbytes: int, device=None, stream=None):
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check(lib().svp_workspace_init(self.ptr, self.nbytes, _stream(stream)),
               "svp_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def read_status(self, stream=None) -> int:
        """Device status bits since the last read (synchronises the stream)."""
        v = ctypes.c_int32(0)
        _check(lib().svp_read_status(self.ptr, _stream(stream), ctypes.byref(v)),
               "svp_read_status")
        return int(v.value)


_ws_cache: dict = {}


def _workspace(key, nbytes: int, device, stream) -> Workspace:
    ws = _ws_cache.get((key, device))
    if ws is None or ws.nbytes < nbytes:
        ws = Workspace(nbytes, device, stream)
        _ws_cache[(key, device)] = ws
    return ws


def _heads(hq: int, hkv: int, d: int, scale: float) -> svp_heads:
    return svp_heads(int(hq), int(hkv), int(d), float(scale))


# ----------------------------------------------------------------- attention
def verify_attn_workspace_size(n: int, m_cap: int, w: int, hq: int, hkv: int, d: int,
                               dtype=torch.bfloat16, tile_mode: int = TILE_AUTO) -> int:
    out = ctypes.c_size_t(0)
    code = SVP_BF16 if dtype == torch.bfloat16 else SVP_F32
    h = _heads(hq, hkv, d, 0.0)
    _check(lib().svp_verify_attn_workspace_size(n, m_cap, w, ctypes.byref(h), code, tile_mode,
                                                ctypes.byref(out)),
           "svp_verify_attn_workspace_size")
    return int(out.value)


def make_kv(*, k_ctx=None, v_ctx=None, cu_ctx=None, k_cache=None, v_cache=None,
            block_table=None, page_size: int = 16) -> svp_kv:
    """svp_kv for contiguous (k_ctx, v_ctx, cu_ctx) or paged (k_cache, v_cache,
    block_table) committed context; None for both means no context."""
    kv = svp_kv()
    if k_cache is not None:
        if k_cache.stride() != v_cache.stride() or k_cache.stride(-1) != 1:
            raise ValueError("k_cache and v_cache need identical strides, last dim contiguous")
        kv.paged = 1
        kv.k = k_cache.data_ptr()
        kv.v = v_cache.data_ptr()
        _dev(block_table, "block_table", torch.int32)
        kv.block_table = block_table.data_ptr()
        kv.max_pages = block_table.shape[1]
        kv.page_size = page_size
        kv.num_pages = k_cache.shape[0]
        s = k_cache.stride()
        kv.stride_page, kv.stride_head, kv.stride_tok = s[0], s[1], s[2]
        if k_cache.device.type != "cuda" or v_cache.device.type != "cuda":
            raise ValueError("KV cache must be on a CUDA device")
    elif k_ctx is not None:
        kv.paged = 0
        kv.k = _dev(k_ctx, "k_ctx")
        kv.v = _dev(v_ctx, "v_ctx")
        kv.cu_ctx = _dev(cu_ctx, "cu_ctx", torch.int64)
        kv.total_tokens = k_ctx.shape[0]
    return kv


def verify_attn_packed(q, k_new, v_new, ctx_len, cu_slots, *, w: int, hkv: Optional[int] = None,
                       kv: Optional[svp_kv] = None, out=None, lse=None, want_lse: bool = True,
                       scale: float = 0.0, tile_mode: int = TILE_AUTO, ws: Optional[Workspace] = None,
                       stream=None, **kv_tensors):
    """Verification attention; returns (out [m_cap, hq, d], lse [m_cap, hq] or None).

    q [m_cap, hq, d]; k_new, v_new [m_cap, hkv, d]; ctx_len [n] int32; cu_slots [n+1]
    int32; context via ``kv`` (see make_kv) or the make_kv keyword tensors.
    """
    m_cap, hq, d = q.shape
    hkv = hkv if hkv is not None else k_new.shape[1]
    n = cu_slots.shape[0] - 1
    code = _dtype_code(q)
    if kv is None:
        kv = make_kv(**kv_tensors)
    if out is None:
        out = torch.full_like(q, float("nan"))
    if lse is None and want_lse:
        lse = torch.full((m_cap, hq), float("nan"), dtype=torch.float32, device=q.device)
    nbytes = verify_attn_workspace_size(n, m_cap, w, hq, hkv, d, q.dtype, tile_mode)
    if ws is None:
        ws = _workspace(("verify", tile_mode, code, d), nbytes, q.device, stream)
    h = _heads(hq, hkv, d, scale)
    _check(lib().svp_verify_attn_packed_ex(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), ctypes.byref(kv),
        _dev(ctx_len, "ctx_len", torch.int32), _dev(cu_slots, "cu_slots", torch.int32),
        n, m_cap, int(w), ctypes.byref(h), code, int(tile_mode), _dev(out, "out"),
        _dev(lse, "lse", torch.float32), ws.ptr, ws.nbytes, _stream(stream)),
        "svp_verify_attn_packed")
    return out, lse


def prefill_attn_workspace_size(n: int, max_s: int, hq: int, hkv: int, d: int) -> int:
    out = ctypes.c_size_t(0)
    h = _heads(hq, hkv, d, 0.0)
    _check(lib().svp_prefill_attn_workspace_size(n, max_s, ctypes.byref(h), SVP_BF16,
                                                 ctypes.byref(out)),
           "svp_prefill_attn_workspace_size")
    return int(out.value)


def prefill_attn(q, k, v, cu_seqlens, *, max_s: int, out=None, lse=None, want_lse=True,
                 scale: float = 0.0, ws: Optional[Workspace] = None, stream=None):
    """Causal prefill attention of packed sequences; returns (out, lse)."""
    total_s, hq, d = q.shape
    hkv = k.shape[1]
    n = cu_seqlens.shape[0] - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((total_s, hq), dtype=torch.float32, device=q.device)
    nbytes = prefill_attn_workspace_size(n, max_s, hq, hkv, d)
    if ws is None:
        ws = _workspace(("prefill", d), nbytes, q.device, stream)
    h = _heads(hq, hkv, d, scale)
    _check(lib().svp_prefill_attn(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(cu_seqlens, "cu_seqlens", torch.int32),
        n, int(max_s), int(total_s), 1, ctypes.byref(h), _dtype_code(q), _dev(out, "out"),
        _dev(lse, "lse", torch.float32), ws.ptr, ws.nbytes, _stream(stream)),
        "svp_prefill_attn")
    return out, lse


# ----------------------------------------------------------------- margin / accept
def draft_margin_workspace_size(rows: int, vocab: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().svp_draft_margin_workspace_size(rows, vocab, ctypes.byref(out)),
           "svp_draft_margin_workspace_size")
    return int(out.value)


def draft_margin(logits, *, vocab: Optional[int] = None, ws: Optional[Workspace] = None,
                 outs=None, stream=None):
    """(top1_idx int32, top1 f32, top2 f32, margin f32) per row of logits [rows, V]."""
    rows, stride = logits.shape
    vocab = stride if vocab is None else vocab
    dev = logits.device
    if outs is None:
        outs = (torch.empty(rows, dtype=torch.int32, device=dev),
                torch.empty(rows, dtype=torch.float32, device=dev),
                torch.empty(rows, dtype=torch.float32, device=dev),
                torch.empty(rows, dtype=torch.float32, device=dev))
    idx, t1, t2, mg = outs
    if ws is None:
        ws = _workspace(("margin",), draft_margin_workspace_size(rows, vocab), dev, stream)
    _check(lib().svp_draft_margin(
        _dev(logits, "logits"), stride, rows, vocab, _dtype_code(logits),
        _dev(idx, "top1_idx", torch.int32), _dev(t1, "top1", torch.float32),
        _dev(t2, "top2", torch.float32), _dev(mg, "margin", torch.float32),
        ws.ptr, ws.nbytes, _stream(stream)), "svp_draft_margin")
    return outs


def greedy_accept(target_argmax, tokens, cu_slots, *, outs=None, stream=None):
    """(accept_len [n] int32, next_token [n] int32)."""
    n = cu_slots.shape[0] - 1
    m_cap = tokens.shape[0]
    dev = tokens.device
    if outs is None:
        outs = (torch.empty(n, dtype=torch.int32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev))
    acc, nxt = outs
    _check(lib().svp_greedy_accept(
        _dev(target_argmax, "target_argmax", torch.int32), _dev(tokens, "tokens", torch.int32),
        _dev(cu_slots, "cu_slots", torch.int32), n, m_cap, _dev(acc, "accept_len", torch.int32),
        _dev(nxt, "next_token", torch.int32), _stream(stream)), "svp_greedy_accept")
    return outs


def margin_accept_workspace_size(n: int, m_cap: int, vocab: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().svp_margin_accept_workspace_size(n, m_cap, vocab, ctypes.byref(out)),
           "svp_margin_accept_workspace_size")
    return int(out.value)


def margin_accept(logits, tokens, cu_slots, *, vocab: Optional[int] = None,
                  ws: Optional[Workspace] = None, outs=None, stream=None):
    """Fused row margin over packed target logits [m_cap, V] + greedy acceptance.

    Returns (top1_idx, top1, top2, margin) per row and (accept_len, next_token) per
    request.  Rows >= cu_slots[n] are neither read nor written."""
    m_cap, stride = logits.shape
    vocab = stride if vocab is None else vocab
    n = cu_slots.shape[0] - 1
    dev = logits.device
    if outs is None:
        outs = (torch.full((m_cap,), -1, dtype=torch.int32, device=dev),
                torch.full((m_cap,), float("nan"), dtype=torch.float32, device=dev),
                torch.full((m_cap,), float("nan"), dtype=torch.float32, device=dev),
                torch.full((m_cap,), float("nan"), dtype=torch.float32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev))
    idx, t1, t2, mg, acc, nxt = outs
    if ws is None:
        ws = _workspace(("margin_accept",), margin_accept_workspace_size(n, m_cap, vocab), dev,
                        stream)
    _check(lib().svp_margin_accept(
        _dev(logits, "logits"), stride, m_cap, vocab, _dtype_code(logits),
        _dev(tokens, "tokens", torch.int32), _dev(cu_slots, "cu_slots", torch.int32), n,
        _dev(idx, "top1_idx", torch.int32), _dev(t1, "top1", torch.float32),
        _dev(t2, "top2", torch.float32), _dev(mg, "margin", torch.float32),
        _dev(acc, "accept_len", torch.int32), _dev(nxt, "next_token", torch.int32),
        ws.ptr, ws.nbytes, _stream(stream)), "svp_margin_accept")
    return outs


def dvl_allocate_pack(scores, *, n_live=None, budget_per_req: int = 8, m_cap: Optional[int] = None,
                      tokens=None, positions=None, kv_refs=None, fill_token: int = 0,
                      fill_pos: int = 0, fill_ref: int = -1, ws: Optional[Workspace] = None,
                      stream=None) -> Dict[str, torch.Tensor]:
    """DVL budget allocator + flat-buffer packer (svp_dvl_allocate_pack).

    scores [n_bs, w-1] fp32 acceptance scores; n_live: device int32 scalar tensor or None
    (all live); tokens / positions / kv_refs [n_bs, w] int32 or None.  Returns k_init,
    k, cu_slots, n_adjust and the packed fields that were given.
    """
    if scores.dim() != 2:
        raise SvpError("scores must be [n_bs, w-1]")
    n_bs, wm1 = scores.shape
    w = wm1 + 1
    dev = scores.device
    if m_cap is None:
        m_cap = w * n_bs
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(k_init=torch.empty(n_bs, **i32), k=torch.empty(n_bs, **i32),
               cu_slots=torch.empty(n_bs + 1, **i32), n_adjust=torch.empty(1, **i32))
    for name, f in (("tokens", tokens), ("positions", positions), ("kv_refs", kv_refs)):
        if f is not None:
            if tuple(f.shape) != (n_bs, w):
                raise SvpError(f"{name} must be [n_bs, w]")
            out[name] = torch.empty(m_cap, **i32)
    if ws is None:
        ws = _workspace(("dvl",), 256, dev, stream)
    st = lib().svp_dvl_allocate_pack(
        _dev(scores, "scores", torch.float32), n_bs, w,
        _dev(n_live, "n_live", torch.int32) if n_live is not None else None, budget_per_req,
        _dev(tokens, "tokens", torch.int32) if tokens is not None else None,
        _dev(positions, "positions", torch.int32) if positions is not None else None,
        _dev(kv_refs, "kv_refs", torch.int32) if kv_refs is not None else None,
        m_cap, fill_token, fill_pos, fill_ref,
        out["k_init"].data_ptr(), out["k"].data_ptr(), out["cu_slots"].data_ptr(),
        out["tokens"].data_ptr() if "tokens" in out else None,
        out["positions"].data_ptr() if "positions" in out else None,
        out["kv_refs"].data_ptr() if "kv_refs" in out else None,
        out["n_adjust"].data_ptr(), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "svp_dvl_allocate_pack")
    out["ws"] = ws
    return out


def gather_rows_multi(srcs, idx, *, outs=None, stream=None):
    """svp_gather_rows_multi: the packed copy of several wide per-row fields sharing the row
    map idx, in one launch; returns the list of outputs."""
    rows = idx.shape[0]
    if not 1 <= len(srcs) <= GATHER_MAX_FIELDS:
        raise ValueError(f"gather_rows_multi takes 1..{GATHER_MAX_FIELDS} fields")
    if outs is None:
        outs = [torch.empty((rows,) + tuple(s.shape[1:]), dtype=s.dtype, device=s.device) for s in srcs]
    fields = (svp_gather_field * len(srcs))()
    for f, (s, o) in enumerate(zip(srcs, outs)):
        rb = s[0].numel() * s.element_size() if s.shape[0] else o[0].numel() * o.element_size()
        fields[f] = svp_gather_field(_dev(s, f"srcs[{f}]"), s.shape[0], rb, _dev(o, f"outs[{f}]"))
    _check(lib().svp_gather_rows_multi(fields, len(srcs), _dev(idx, "idx", torch.int32), rows,
                                       _stream(stream)), "svp_gather_rows_multi")
    return outs


def gather_rows(src, idx, *, out=None, stream=None):
    """Packed copy of a wide per-row field (svp_gather_rows): out[r] = src[idx[r]] for
    in-range ids, zeros otherwise.  src [src_rows, ...] contiguous; idx [rows] int32."""
    rows = idx.shape[0]
    if out is None:
        out = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else out[0].numel() * out.element_size()
    _check(lib().svp_gather_rows(_dev(src, "src"), src.shape[0], row_bytes,
                                 _dev(idx, "idx", torch.int32), rows, _dev(out, "out"),
                                 _stream(stream)), "svp_gather_rows")
    return out


def stochastic_accept_workspace_size(m_cap: int, vocab: int) -> int:
    nb = ctypes.c_size_t(0)
    _check(lib().svp_stochastic_accept_workspace_size(m_cap, vocab, ctypes.byref(nb)),
           "svp_stochastic_accept_workspace_size")
    return int(nb.value)


def stochastic_accept(logits, tokens, cu_slots, u_accept, u_next, *, temperature: float,
                      vocab: Optional[int] = None, ws: Optional[Workspace] = None, outs=None,
                      stream=None):
    """Stochastic prefix verifier (svp_stochastic_accept); returns (accept_len [n],
    next_token [n], p_draft [m_cap])."""
    m_cap, stride = logits.shape
    vocab = stride if vocab is None else vocab
    n = cu_slots.shape[0] - 1
    dev = logits.device
    if outs is None:
        outs = (torch.empty(n, dtype=torch.int32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev),
                torch.full((m_cap,), float("nan"), dtype=torch.float32, device=dev))
    acc, nxt, pd = outs
    if ws is None:
        ws = _workspace(("stochastic",), stochastic_accept_workspace_size(m_cap, vocab), dev, stream)
    _check(lib().svp_stochastic_accept(
        _dev(logits, "logits"), stride, m_cap, vocab, _dtype_code(logits),
        _dev(tokens, "tokens", torch.int32), _dev(cu_slots, "cu_slots", torch.int32), n,
        float(temperature), _dev(u_accept, "u_accept", torch.float32),
        _dev(u_next, "u_next", torch.float32), _dev(acc, "accept_len", torch.int32),
        _dev(nxt, "next_token", torch.int32), _dev(pd, "p_draft", torch.float32) if pd is not None else None,
        ws.ptr, ws.nbytes, _stream(stream)), "svp_stochastic_accept")
    return outs


def draft_features_workspace_size(rows: int, vocab: int) -> int:
    nb = ctypes.c_size_t(0)
    _check(lib().svp_draft_features_workspace_size(rows, vocab, ctypes.byref(nb)),
           "svp_draft_features_workspace_size")
    return int(nb.value)


def draft_features(logits, *, vocab: Optional[int] = None, out=None, ws: Optional[Workspace] = None,
                   stream=None):
    """[rows, 18] fp32 draft-signal features of every logit row (svp_draft_features)."""
    rows, stride = logits.shape
    vocab = stride if vocab is None else vocab
    if out is None:
        out = torch.empty(rows, 18, dtype=torch.float32, device=logits.device)
    if ws is None:
        ws = _workspace(("features",), draft_features_workspace_size(rows, vocab), logits.device, stream)
    _check(lib().svp_draft_features(_dev(logits, "logits"), stride, rows, vocab, _dtype_code(logits),
                                    _dev(out, "features", torch.float32), ws.ptr, ws.nbytes,
                                    _stream(stream)), "svp_draft_features")
    return out


def act_truncate(margins, *, n: int, w: int, threshold: float, stride: int = 1, out=None, stream=None):
    """k [n] int32 after ACT truncation of margins laid out per request and position."""
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=margins.device)
    _check(lib().svp_act_truncate(_dev(margins, "margins", torch.float32), stride, n, w,
                                  float(threshold), _dev(out, "k", torch.int32), _stream(stream)),
           "svp_act_truncate")
    return out

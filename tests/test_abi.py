"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports
every function include/svp.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_packed_gb300 as svp
from speculative_decoding_verification_packed_gb300 import build as svp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    svp_build.build()
    return svp.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "svp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(svp_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert "svp_verify_attn_packed" in names and "svp_margin_accept" in names
    for name in names:
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.svp_version() == 1
    assert svp.status_string(svp.SVP_OK) == "ok"
    assert "workspace" in svp.status_string(svp.SVP_EWORKSPACE)


def test_workspace_size_queries():
    a = svp.verify_attn_workspace_size(8, 128, 16, 32, 8, 128)
    b = svp.verify_attn_workspace_size(64, 512, 16, 32, 8, 128)
    assert 0 < a <= b
    assert svp.verify_attn_workspace_size(3, 24, 16, 4, 2, 64, dtype=__import__("torch").float32) >= 256
    assert svp.draft_margin_workspace_size(224, 248320) > 224 * 16 * 12
    assert svp.margin_accept_workspace_size(32, 224, 248320) >= svp.draft_margin_workspace_size(224, 248320)
    assert svp.prefill_attn_workspace_size(1, 4096, 32, 8, 128) > 0


def test_invalid_arguments_rejected_on_host(L):
    h = svp.svp_heads(32, 7, 128, 0.0)      # hq % hkv != 0
    out = ctypes.c_size_t(0)
    assert L.svp_verify_attn_workspace_size(8, 128, 16, ctypes.byref(h), 1, 0,
                                            ctypes.byref(out)) == svp.SVP_EINVAL
    h = svp.svp_heads(32, 8, 96, 0.0)       # unsupported head_dim
    assert L.svp_verify_attn_workspace_size(8, 128, 16, ctypes.byref(h), 1, 0,
                                            ctypes.byref(out)) == svp.SVP_EUNSUPPORTED
    h = svp.svp_heads(32, 8, 128, 0.0)
    kv = svp.svp_kv()
    # missing workspace
    assert L.svp_verify_attn_packed(1, 1, 1, ctypes.byref(kv), 1, 1, 8, 128, 16, ctypes.byref(h),
                                    1, 1, None, None, 0, None) == svp.SVP_EWORKSPACE
    # null q with a workspace
    assert L.svp_verify_attn_packed(None, 1, 1, ctypes.byref(kv), 1, 1, 8, 128, 16,
                                    ctypes.byref(h), 1, 1, None, 1, 1 << 30, None) == svp.SVP_EINVAL
    # vocab < 2
    assert L.svp_draft_margin(1, 1, 4, 1, 1, None, None, None, None, 1, 1 << 20,
                              None) == svp.SVP_EINVAL
    # prefill without causal
    assert L.svp_prefill_attn(1, 1, 1, 1, 1, 16, 16, 0, ctypes.byref(h), 1, 1, None, 1, 1 << 20,
                              None) == svp.SVP_EUNSUPPORTED
    # empty batch is a no-op
    assert L.svp_verify_attn_packed(None, None, None, ctypes.byref(kv), None, None, 0, 0, 16,
                                    ctypes.byref(h), 1, None, None, 1, 1 << 20, None) == svp.SVP_OK
    # multi-field gather: field count, row width and alignment are checked on the host
    fields = (svp.svp_gather_field * 9)()
    for f in range(9):
        fields[f] = svp.svp_gather_field(1 << 12, 4, 64, 1 << 16)
    assert L.svp_gather_rows_multi(fields, 0, 1 << 20, 4, None) == svp.SVP_EINVAL
    assert L.svp_gather_rows_multi(fields, 9, 1 << 20, 4, None) == svp.SVP_EINVAL
    assert L.svp_gather_rows_multi(fields, 2, None, 4, None) == svp.SVP_EINVAL
    fields[1] = svp.svp_gather_field(1 << 12, 4, 8, 1 << 16)       # row narrower than 16 bytes
    assert L.svp_gather_rows_multi(fields, 2, 1 << 20, 4, None) == svp.SVP_EINVAL
    fields[1] = svp.svp_gather_field(1 << 12, 4, 24, 1 << 16)      # not a multiple of 16
    assert L.svp_gather_rows_multi(fields, 2, 1 << 20, 4, None) == svp.SVP_EUNSUPPORTED
    fields[1] = svp.svp_gather_field(1 << 12, 4, 64, 1 << 16)
    assert L.svp_gather_rows_multi(fields, 8, 1 << 20, 0, None) == svp.SVP_OK   # no rows


def test_gather_binding_field_count():
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        svp.gather_rows_multi([x] * (svp.GATHER_MAX_FIELDS + 1), torch.zeros(4, dtype=torch.int32))


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(4, 2, 64)
    with pytest.raises((ValueError, RuntimeError)):
        svp.verify_attn_packed(q, q[:, :1], q[:, :1], torch.zeros(1, dtype=torch.int32),
                               torch.tensor([0, 4], dtype=torch.int32), w=16,
                               k_ctx=q[:0, :1], v_ctx=q[:0, :1],
                               cu_ctx=torch.zeros(2, dtype=torch.int64))


def test_host_checks_of_the_logit_and_allocator_calls(L):
    """The stochastic verifier, draft features, ACT truncation, the DVL allocator, greedy
    accept and both fused margin calls reject bad arguments (and empty calls return OK)
    on the host, before any CUDA call."""
    OK, INV, UNS, WSP = svp.SVP_OK, svp.SVP_EINVAL, svp.SVP_EUNSUPPORTED, svp.SVP_EWORKSPACE
    big = 1 << 30
    nb = ctypes.c_size_t(0)
    # stochastic prefix verifier
    assert L.svp_stochastic_accept_workspace_size(224, 1, ctypes.byref(nb)) == INV     # vocab < 2
    assert L.svp_stochastic_accept_workspace_size(224, 248320, ctypes.byref(nb)) == OK
    need = nb.value
    st = lambda T=1.0, vocab=1000, stride=1000, dtype=1, ws=1, wsb=big, n=4, logits=1: \
        L.svp_stochastic_accept(logits, stride, 16, vocab, dtype, 1, 1, n, T, 1, 1, 1, 1, None, ws, wsb, None)
    assert st(T=0.0) == INV and st(T=-1.0) == INV and st(T=float("nan")) == INV
    assert st(logits=None) == INV and st(vocab=1) == INV and st(stride=999) == INV
    assert st(ws=None) == WSP and st(n=-1) == INV
    assert st(dtype=7) == UNS
    assert st(wsb=16) == WSP
    assert st(n=0) == OK                                                              # nothing to do
    assert need > 0
    # draft features
    assert L.svp_draft_features_workspace_size(8, 15, ctypes.byref(nb)) == INV          # vocab < 16
    ft = lambda rows=8, vocab=1000, stride=1000, dtype=1, ws=1, wsb=big, out=1: \
        L.svp_draft_features(1, stride, rows, vocab, dtype, out, ws, wsb, None)
    assert ft(vocab=15) == INV and ft(rows=-1) == INV and ft(stride=999) == INV and ft(out=None) == INV
    assert ft(dtype=7) == UNS and ft(wsb=16) == WSP and ft(ws=None) == WSP and ft(rows=0) == OK
    # ACT truncation
    assert L.svp_act_truncate(1, 1, 4, 0, 0.5, 1, None) == INV                         # w < 1
    assert L.svp_act_truncate(1, 0, 4, 8, 0.5, 1, None) == INV                         # stride < 1
    assert L.svp_act_truncate(None, 1, 4, 8, 0.5, 1, None) == INV
    assert L.svp_act_truncate(1, 1, 0, 8, 0.5, 1, None) == OK
    # DVL allocator / packer
    dv = lambda n_bs=8, w=16, per=8, m_cap=128, ws=1, wsb=256, scores=1: L.svp_dvl_allocate_pack(
        scores, n_bs, w, None, per, None, None, None, m_cap, 0, 0, -1, None, 1, 1, None, None, None,
        None, ws, wsb, None)
    assert dv(scores=None) == INV and dv(n_bs=0) == INV and dv(w=1) == INV and dv(per=17) == INV
    assert dv(per=0) == INV and dv(m_cap=0) == INV
    assert dv(n_bs=4096) == UNS and dv(w=17, per=8) == UNS
    assert dv(wsb=16) == WSP and dv(ws=None) == WSP
    # greedy accept and the fused margin calls
    assert L.svp_greedy_accept(1, 1, 1, -1, 8, 1, 1, None) == INV
    assert L.svp_greedy_accept(None, 1, 1, 4, 8, 1, 1, None) == INV
    assert L.svp_greedy_accept(1, 1, 1, 0, 8, 1, 1, None) == OK
    assert L.svp_margin_accept(1, 1000, 16, 1000, 1, 1, None, 4, None, None, None, None, 1, 1, 1, big,
                               None) == INV                                           # no cu_slots
    # every call below breaks one documented rule, so none reaches a CUDA call
    ma = lambda logits=1, stride=1000, rows=16, vocab=1000, dtype=1, tokens=1, n=4, acc=1, nxt=1, \
        ws=1, wsb=big: L.svp_margin_accept(logits, stride, rows, vocab, dtype, tokens, 1, n, None, None,
                                           None, None, acc, nxt, ws, wsb, None)
    assert ma(tokens=None) == INV and ma(acc=None) == INV and ma(nxt=None) == INV
    assert ma(n=-1) == INV and ma(vocab=1) == INV and ma(stride=999) == INV and ma(rows=-1) == INV
    assert ma(logits=None) == INV
    assert ma(dtype=7) == UNS
    assert ma(ws=None) == WSP and ma(wsb=16) == WSP
    na = L.svp_margin_accept_noalloc
    na.restype = ctypes.c_int
    na.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32] + [ctypes.c_void_p] * 7
    assert na(1, 1000, 16, 1000, 1, 1, None, 4, None, None, None, None, 1, 1, None) == INV
    # sizes whose workspace exceeds the fixed 2 MiB scratch (8192 rows of V = 248,320)
    assert L.svp_margin_accept_workspace_size(512, 8192, 248320, ctypes.byref(nb)) == OK
    assert nb.value > (2 << 20)
    assert na(1, 248320, 8192, 248320, 1, 1, 1, 512, None, None, None, None, 1, 1, None) == WSP

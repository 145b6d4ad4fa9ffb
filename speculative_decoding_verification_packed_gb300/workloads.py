"""Seeded synthetic workloads for packed speculative verification.

This module only draws random inputs and lays them out; it holds none of the method's
arithmetic (no attention, no argmax, no acceptance).  Both the CUDA path and the CPU
oracle are fed from the tensors it returns.

Layout ("DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive
Verification", SIII-C Flat-buffer packer): request i owns packed rows
cu_slots[i] .. cu_slots[i+1]-1; row cu_slots[i] + j holds candidate j, j = 0 being the
anchor.  Every per-row field (q, k_new, v_new, tokens, target logits) is generated for
the full block width W first and then packed, so that the same data can be re-packed
under other lengths (truncation and relayout invariants).

Target-logit rows get a planted argmax: values are N(0, std) clamped to +-6 std and one
planted entry per row is set to 6.5 std, so that the generator knows the argmax without
computing it.  Draft token j of request i copies the planted argmax of target row j-1
with the workload's match probability, otherwise it is a uniform token different from
it.  Draft-logit rows (when present) plant their argmax at the draft token.

Workloads (sizes and distributions of the five synthetic configurations):
  tiny_fp32        N=3, k=[4,12,8] (relayout [10,8,6]) in 24 slots, 4q/2kv, d=64,
                   contiguous ctx [37,100,250], fp32, vocab 512, logits N(0,1),
                   each draft matches with probability 0.5.
  full_width_bf16  N=8, k=16 each (128 slots), 32q/8kv, d=128, ctx ~ U[512,8192],
                   contiguous, bf16.
  budget8n_bf16    N=8, 64 slots: k_i = 1 + min(Geom0(0.1555), 15), then grown
                   (smallest first) or shrunk (largest first) to exactly 64; otherwise
                   as full_width_bf16.
  paged_n64_bf16   N=64, 512 slots (lengths as budget8n), 32q/8kv, d=128,
                   ctx ~ U[4096,32768] in 16-token pages through a shuffled block table.
  prefill_4096     one request, 4096 query rows, causal, 32q/8kv, d=128, bf16.
  wide_gqa_bf16    N=32, k=7 (224 slots), 24q/2kv, d=256, ctx ~ U[1024,8192], target
                   logits [224, 248320] and draft logits [192, 248320] ~ N(0,2) bf16,
                   draft j matches with probability 0.8**j.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

PAGE_SIZE = 16

WORKLOADS: Dict[str, dict] = {
    "tiny_fp32": dict(n=3, W=16, lengths=[4, 12, 8], relayout=[10, 8, 6], m_cap=24,
                      hq=4, hkv=2, d=64, ctx=[37, 100, 250], dtype="f32", paged=False,
                      vocab=512, logit_std=1.0, match="half", draft_logits=False),
    "full_width_bf16": dict(n=8, W=16, lengths="full", m_cap=128, hq=32, hkv=8, d=128,
                            ctx=(512, 8192), dtype="bf16", paged=False, vocab=0),
    "budget8n_bf16": dict(n=8, W=16, lengths="budget", m_cap=64, hq=32, hkv=8, d=128,
                          ctx=(512, 8192), dtype="bf16", paged=False, vocab=0),
    "paged_n64_bf16": dict(n=64, W=16, lengths="budget", m_cap=512, hq=32, hkv=8, d=128,
                           ctx=(4096, 32768), dtype="bf16", paged=True, vocab=0),
    "prefill_4096": dict(n=1, W=4096, lengths="full", m_cap=4096, hq=32, hkv=8, d=128,
                         ctx=[0], dtype="bf16", paged=False, vocab=0),
    "wide_gqa_bf16": dict(n=32, W=7, lengths="full", m_cap=224, hq=24, hkv=2, d=256,
                          ctx=(1024, 8192), dtype="bf16", paged=False, vocab=248320,
                          logit_std=2.0, match="decay0.8", draft_logits=True),
}

GEOM_P = 0.1555   # truncated Geom0 draft count: mean progress 1 + E[min(G, 15)] = 6.00


@dataclass
class Batch:
    """One verification step's inputs (all tensors on ``device``)."""
    name: str
    n: int
    W: int
    m_cap: int
    hq: int
    hkv: int
    d: int
    scale: float
    dtype: torch.dtype
    lengths: torch.Tensor          # [n] int32 slot counts k_i (anchor included)
    cu_slots: torch.Tensor         # [n+1] int32
    ctx_len: torch.Tensor          # [n] int32
    q: torch.Tensor                # [m_cap, hq, d]
    k_new: torch.Tensor            # [m_cap, hkv, d]
    v_new: torch.Tensor            # [m_cap, hkv, d]
    paged: bool = False
    k_ctx: Optional[torch.Tensor] = None      # [sum L, hkv, d]
    v_ctx: Optional[torch.Tensor] = None
    cu_ctx: Optional[torch.Tensor] = None     # [n+1] int64
    k_cache: Optional[torch.Tensor] = None    # [pages, hkv, 16, d]
    v_cache: Optional[torch.Tensor] = None
    block_table: Optional[torch.Tensor] = None  # [n, max_pages] int32, -1 = unused
    tokens: Optional[torch.Tensor] = None       # [m_cap] int32 (anchor, drafts)
    target_logits: Optional[torch.Tensor] = None  # [m_cap, V]
    draft_logits: Optional[torch.Tensor] = None   # [n*(W-1), V]
    planted_argmax: Optional[torch.Tensor] = None  # [m_cap] int32, generator's record
    full: dict = field(default_factory=dict)      # full-width per-request fields

    @property
    def m_live(self) -> int:
        return int(self.cu_slots[-1])

    @property
    def cache_strides(self):
        """(page, head, token) element strides of k_cache / v_cache."""
        s = self.k_cache.stride()
        return (s[0], s[1], s[2])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, dtype, std=1.0):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def budget_lengths(n: int, budget: int, W: int, g: torch.Generator) -> List[int]:
    """Truncated-geometric draft counts, then greedy fill to exactly ``budget`` slots.

    k_i = 1 + min(Geom0(p), W-1).  While sum(k) < budget the smallest k_i < W grows by
    one (ties: lowest i); while sum(k) > budget the largest k_i > 1 shrinks by one
    (ties: highest i).  A score-free stand-in for the budget allocator.
    """
    u = torch.rand(n, generator=g, dtype=torch.float64).clamp_min(1e-300)
    draws = torch.floor(torch.log(u) / math.log(1.0 - GEOM_P)).to(torch.int64)
    k = [1 + min(int(x), W - 1) for x in draws]
    if not (n <= budget <= n * W):
        raise ValueError("budget must lie in [n, n*W]")
    while sum(k) < budget:
        cand = [i for i in range(n) if k[i] < W]
        i = min(cand, key=lambda j: (k[j], j))
        k[i] += 1
    while sum(k) > budget:
        cand = [i for i in range(n) if k[i] > 1]
        i = max(cand, key=lambda j: (k[j], j))
        k[i] -= 1
    return k


def prefix_offsets(lengths) -> torch.Tensor:
    """Row offsets of a packed layout, as the caller (the packer) supplies them."""
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + int(x))
    return torch.tensor(cu, dtype=torch.int32)


def pack_rows(full: torch.Tensor, lengths, m_cap: int, fill=0.0) -> torch.Tensor:
    """Pack per-request full-width rows full[i, :k_i] into an [m_cap, ...] buffer."""
    out = torch.full((m_cap,) + tuple(full.shape[2:]), fill, dtype=full.dtype,
                     device=full.device)
    r = 0
    for i, k in enumerate(lengths):
        k = int(k)
        out[r:r + k] = full[i, :k]
        r += k
    return out


def _ctx_lengths(spec, n, g) -> List[int]:
    c = spec["ctx"]
    if isinstance(c, list):
        return list(c)
    lo, hi = c
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def make_batch(name: str, seed: int = 0, device="cpu", *, lengths=None,
               ctx_lengths=None, n: Optional[int] = None, paged: Optional[bool] = None,
               poison: bool = False, with_logits: bool = True,
               dtype: Optional[str] = None, hq=None, hkv=None, d=None, W=None,
               m_cap=None, vocab=None) -> Batch:
    """Build one seeded batch of workload ``name`` (overrides allow smaller variants).

    poison=True fills every storage slot that the method must not read (packed tail
    rows, unused slots of the last page of each request) with NaN.
    """
    spec = dict(WORKLOADS[name])
    for key, val in (("hq", hq), ("hkv", hkv), ("d", d), ("W", W), ("vocab", vocab)):
        if val is not None:
            spec[key] = val
    if n is not None:
        spec["n"] = n
    if paged is not None:
        spec["paged"] = paged
    if dtype is not None:
        spec["dtype"] = dtype
    N, Wd, HQ, HKV, D = spec["n"], spec["W"], spec["hq"], spec["hkv"], spec["d"]
    tdtype = torch.float32 if spec["dtype"] == "f32" else torch.bfloat16
    g_host = _gen(seed, "cpu")           # small integer draws: always on the host
    g_dev = _gen(seed + 1_000_003, device)

    # slot counts
    if lengths is None:
        if spec["lengths"] == "full":
            lengths = [Wd] * N
        elif spec["lengths"] == "budget":
            lengths = budget_lengths(N, spec["m_cap"] if n is None else 8 * N, Wd, g_host)
        else:
            lengths = list(spec["lengths"])
    lengths = [int(x) for x in lengths]
    if len(lengths) != N:
        raise ValueError("lengths must have one entry per request")
    cu = prefix_offsets(lengths)
    mcap = m_cap if m_cap is not None else (spec["m_cap"] if n is None else max(sum(lengths), 1))
    mcap = max(mcap, int(cu[-1]))

    # context lengths
    if ctx_lengths is None:
        ctx_lengths = _ctx_lengths(spec, N, g_host)
        if len(ctx_lengths) != N:
            ctx_lengths = (ctx_lengths * N)[:N]
    ctx_lengths = [int(x) for x in ctx_lengths]

    nanv = float("nan")
    fill = nanv if poison else 0.0
    q_full = _randn((N, Wd, HQ, D), g_dev, device, tdtype)
    kn_full = _randn((N, Wd, HKV, D), g_dev, device, tdtype)
    vn_full = _randn((N, Wd, HKV, D), g_dev, device, tdtype)
    b = Batch(name=name, n=N, W=Wd, m_cap=mcap, hq=HQ, hkv=HKV, d=D,
              scale=1.0 / math.sqrt(D), dtype=tdtype,
              lengths=torch.tensor(lengths, dtype=torch.int32, device=device),
              cu_slots=cu.to(device),
              ctx_len=torch.tensor(ctx_lengths, dtype=torch.int32, device=device),
              q=pack_rows(q_full, lengths, mcap, fill),
              k_new=pack_rows(kn_full, lengths, mcap, fill),
              v_new=pack_rows(vn_full, lengths, mcap, fill),
              paged=bool(spec["paged"]))
    b.full = dict(q=q_full, k_new=kn_full, v_new=vn_full)

    # KV context
    if not b.paged:
        total = sum(ctx_lengths)
        cu_ctx = [0]
        for L in ctx_lengths:
            cu_ctx.append(cu_ctx[-1] + L)
        b.k_ctx = torch.empty((total, HKV, D), dtype=tdtype, device=device)
        b.v_ctx = torch.empty((total, HKV, D), dtype=tdtype, device=device)
        for i, L in enumerate(ctx_lengths):
            s = cu_ctx[i]
            b.k_ctx[s:s + L] = _randn((L, HKV, D), g_dev, device, tdtype)
            b.v_ctx[s:s + L] = _randn((L, HKV, D), g_dev, device, tdtype)
        b.cu_ctx = torch.tensor(cu_ctx, dtype=torch.int64, device=device)
    else:
        pages_per = [(L + PAGE_SIZE - 1) // PAGE_SIZE for L in ctx_lengths]
        n_pages = max(sum(pages_per), 1)
        max_pages = max(max(pages_per), 1)
        perm = torch.randperm(n_pages, generator=g_host).to(torch.int32)
        bt = torch.full((N, max_pages), -1, dtype=torch.int32)
        p = 0
        for i, np_i in enumerate(pages_per):
            bt[i, :np_i] = perm[p:p + np_i]
            p += np_i
        b.block_table = bt.to(device)
        b.k_cache = torch.empty((n_pages, HKV, PAGE_SIZE, D), dtype=tdtype, device=device)
        b.v_cache = torch.empty((n_pages, HKV, PAGE_SIZE, D), dtype=tdtype, device=device)
        # fill page by page in request order so the data does not depend on the shuffle
        for i, L in enumerate(ctx_lengths):
            for t0 in range(0, pages_per[i] * PAGE_SIZE, 4096):
                cnt = min(4096, pages_per[i] * PAGE_SIZE - t0)
                kk = _randn((cnt // PAGE_SIZE, HKV, PAGE_SIZE, D), g_dev, device, tdtype)
                vv = _randn((cnt // PAGE_SIZE, HKV, PAGE_SIZE, D), g_dev, device, tdtype)
                ids = b.block_table[i, t0 // PAGE_SIZE:(t0 + cnt) // PAGE_SIZE].long()
                b.k_cache[ids] = kk
                b.v_cache[ids] = vv
            if poison and L % PAGE_SIZE:
                last = int(bt[i, pages_per[i] - 1])
                b.k_cache[last, :, L % PAGE_SIZE:] = nanv
                b.v_cache[last, :, L % PAGE_SIZE:] = nanv

    # tokens and logits
    V = spec.get("vocab", 0)
    if V and with_logits:
        std = spec["logit_std"]
        planted = torch.randint(0, V, (N, Wd), generator=g_host, dtype=torch.int64)
        tok_full = torch.empty((N, Wd), dtype=torch.int64)
        tok_full[:, 0] = torch.randint(0, V, (N,), generator=g_host)
        u = torch.rand((N, Wd), generator=g_host, dtype=torch.float64)
        other = torch.randint(0, V - 1, (N, Wd), generator=g_host, dtype=torch.int64)
        for j in range(1, Wd):
            p_match = 0.5 if spec["match"] == "half" else 0.8 ** j
            prev = planted[:, j - 1]
            alt = other[:, j] + (other[:, j] >= prev).to(torch.int64)
            tok_full[:, j] = torch.where(u[:, j] < p_match, prev, alt)
        tl_full = _planted_logits((N, Wd, V), planted.to(device), std, g_dev, device, tdtype)
        b.target_logits = pack_rows(tl_full, lengths, mcap, fill)
        b.tokens = pack_rows(tok_full.to(torch.int32), lengths, mcap, -1).to(device)
        b.planted_argmax = pack_rows(planted.to(torch.int32), lengths, mcap, -1).to(device)
        b.full.update(tokens=tok_full.to(torch.int32), planted=planted.to(torch.int32))
        del tl_full
        if spec.get("draft_logits"):
            dl = _planted_logits((N, Wd - 1, V), tok_full[:, 1:].to(device), std, g_dev,
                                 device, tdtype)
            b.draft_logits = dl.reshape(N * (Wd - 1), V)
    return b


def _planted_logits(shape, planted, std, g, device, dtype):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    x.clamp_(-6.0 * std, 6.0 * std)
    x.scatter_(-1, planted.reshape(shape[:-1] + (1,)).to(torch.int64),
               torch.full(shape[:-1] + (1,), 6.5 * std, device=device))
    return x.to(dtype)


def make_prefill(seed: int = 0, device="cpu", s: int = 4096, hq: int = 32, hkv: int = 8,
                 d: int = 128, dtype=torch.bfloat16):
    """One causal prefill sequence: q [s, hq, d], k, v [s, hkv, d]."""
    g = _gen(seed + 7, device)
    q = _randn((s, hq, d), g, device, dtype)
    k = _randn((s, hkv, d), g, device, dtype)
    v = _randn((s, hkv, d), g, device, dtype)
    return q, k, v

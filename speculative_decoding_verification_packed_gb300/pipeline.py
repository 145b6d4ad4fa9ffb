"""Fixed-address verification step captured once as a CUDA graph.

"DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-D
(Graph integration, Algorithm 2, Fig. 5): the step's tensors keep their addresses and
shapes from step to step, boundaries change only through device values, and the whole
step (allocate and pack, verify, accept) is captured once per request bucket and replayed
with no host readback.

This module only orders calls into the library (svp_dvl_allocate_pack,
svp_gather_rows_multi, svp_verify_attn_packed, svp_margin_accept); every step of the computation runs in the
library's kernels.  The wide per-slot fields a target model would produce for the packed
rows (query / key / value rows, target logits) are given here at full block width,
[n_bs * w, ...], and packed by the row references the packer writes (row i * w + j for
slot j of request i), so that one row map serves every buffer of the step.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (dvl_allocate_pack, gather_rows_multi, margin_accept, margin_accept_workspace_size,
               verify_attn_packed, verify_attn_workspace_size, Workspace, make_kv)


class VerifyPipeline:
    """One request bucket: n_bs requests of up to w slots, budget_per_req * n_live live
    slots out of a captured capacity m_cap = budget_per_req * n_bs.

    Inputs (fixed addresses; write them in place before step()):
      scores [n_bs, w-1] fp32, n_live [1] int32, tokens [n_bs, w] int32,
      positions [n_bs, w] int32, q_full [n_bs*w, hq, d], k_full / v_full [n_bs*w, hkv, d],
      logits_full [n_bs*w, vocab], ctx_len [n_bs] int32 and the context storage (kv).
    Outputs (fixed addresses): k, cu_slots, tokens_packed, positions_packed, refs_packed,
      out [m_cap, hq, d], lse [m_cap, hq], top1_idx / top1 / top2 / margin [m_cap],
      accept_len / next_token [n_bs].
    """

    def __init__(self, n_bs: int, *, hq: int, hkv: int, d: int, vocab: int, ctx_len: torch.Tensor,
                 kv_tensors: dict, w: int = 16, budget_per_req: int = 8,
                 dtype: torch.dtype = torch.bfloat16, device="cuda"):
        self.n_bs, self.w, self.per = n_bs, w, budget_per_req
        self.m_cap = budget_per_req * n_bs
        self.hq, self.hkv, self.d, self.vocab = hq, hkv, d, vocab
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        rows = n_bs * w
        self.scores = torch.zeros(n_bs, w - 1, dtype=torch.float32, device=dev)
        self.n_live = torch.full((1,), n_bs, **i32)
        self.tokens = torch.zeros(n_bs, w, **i32)
        self.positions = torch.zeros(n_bs, w, **i32)
        self.row_ids = torch.arange(rows, **i32).view(n_bs, w)
        self.q_full = torch.zeros(rows, hq, d, dtype=dtype, device=dev)
        self.k_full = torch.zeros(rows, hkv, d, dtype=dtype, device=dev)
        self.v_full = torch.zeros(rows, hkv, d, dtype=dtype, device=dev)
        self.logits_full = torch.zeros(rows, vocab, dtype=dtype, device=dev)
        self.ctx_len = ctx_len
        self.kv = make_kv(**kv_tensors)
        self._kv_tensors = kv_tensors   # keep the context storage alive
        # packed buffers
        m = self.m_cap
        self.q = torch.zeros(m, hq, d, dtype=dtype, device=dev)
        self.k_new = torch.zeros(m, hkv, d, dtype=dtype, device=dev)
        self.v_new = torch.zeros(m, hkv, d, dtype=dtype, device=dev)
        self.logits = torch.zeros(m, vocab, dtype=dtype, device=dev)
        self.out = torch.zeros(m, hq, d, dtype=dtype, device=dev)
        self.lse = torch.zeros(m, hq, dtype=torch.float32, device=dev)
        self.margin_outs = (torch.zeros(m, **i32), torch.zeros(m, dtype=torch.float32, device=dev),
                            torch.zeros(m, dtype=torch.float32, device=dev),
                            torch.zeros(m, dtype=torch.float32, device=dev),
                            torch.zeros(n_bs, **i32), torch.zeros(n_bs, **i32))
        self.ws_dvl = Workspace(256, dev)
        self.ws_attn = Workspace(verify_attn_workspace_size(n_bs, m, w, hq, hkv, d, dtype, 0), dev)
        self.ws_margin = Workspace(margin_accept_workspace_size(n_bs, m, vocab), dev)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.alloc = None

    def _enqueue(self, stream=None):
        a = dvl_allocate_pack(self.scores, n_live=self.n_live, budget_per_req=self.per,
                              m_cap=self.m_cap, tokens=self.tokens, positions=self.positions,
                              kv_refs=self.row_ids, fill_token=0, fill_pos=0, fill_ref=-1,
                              ws=self.ws_dvl, stream=stream)
        gather_rows_multi([self.q_full, self.k_full, self.v_full, self.logits_full], a["kv_refs"],
                          outs=[self.q, self.k_new, self.v_new, self.logits], stream=stream)
        verify_attn_packed(self.q, self.k_new, self.v_new, self.ctx_len, a["cu_slots"], w=self.w,
                           hkv=self.hkv, kv=self.kv, out=self.out, lse=self.lse, ws=self.ws_attn,
                           stream=stream)
        margin_accept(self.logits, a["tokens"], a["cu_slots"], vocab=self.vocab, ws=self.ws_margin,
                      outs=self.margin_outs, stream=stream)
        return a

    def capture(self):
        """Run the step once eagerly, then capture it (fixed addresses from here on)."""
        self._enqueue()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.alloc = self._enqueue(stream=torch.cuda.current_stream())
        return self

    def step(self):
        """Replay the captured step on the current inputs (no host readback)."""
        self.graph.replay()

    @property
    def accept_len(self):
        return self.margin_outs[4]

    @property
    def next_token(self):
        return self.margin_outs[5]

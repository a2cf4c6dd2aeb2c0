"""One draft-verify cycle on device buffers, in C-ABI call order.

Allocation of the caller-owned workspaces and outputs, then the sequence
tree_init -> expand x D -> rerank -> build_tree -> tree_attention -> verify ->
kv_compact. Every step runs in libeagle's kernels; this module only holds
buffers and passes pointers.
"""
from __future__ import annotations

import torch

from . import eagle as E


def torch_dtype(code: int) -> torch.dtype:
    return torch.float32 if code == E.EAGLE_F32 else torch.bfloat16


class DeviceCycle:
    """Buffers for one cycle of a (TreeCfg, KvCfg) problem on one device."""

    def __init__(self, cfg: E.TreeCfg, kv: E.KvCfg, device="cuda", fused_head: bool = False):
        self.cfg, self.kv = cfg, kv
        self.fused_head = fused_head
        dev = torch.device(device)
        B, D, k, T, W = cfg.batch, cfg.depth, cfg.top_k, cfg.T, cfg.W
        i32 = dict(dtype=torch.int32, device=dev)
        self.ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg), dev)
        self.attn_ws = E.alloc_workspace(E.eagle_attention_workspace_bytes(kv, T), dev)
        self.row_lse = torch.empty(B, D, k, dtype=torch.float32, device=dev)
        self.ftok = torch.empty(B, k, **i32)
        self.fcount = torch.empty(B, **i32)
        self.tokens = torch.empty(B, T, **i32)
        self.parent = torch.empty(B, T, **i32)
        self.depth = torch.empty(B, T, **i32)
        self.pos = torch.empty(B, T, **i32)
        self.mask = torch.empty(B, T, W, **i32)  # uint32 bit rows
        self.n_tree = torch.empty(B, **i32)
        self.attn_out = torch.empty(B, T, kv.n_q_heads, kv.head_dim, dtype=torch_dtype(kv.dtype), device=dev)
        self.accept_len = torch.empty(B, **i32)
        self.slots = torch.empty(B, D + 1, **i32)
        self.out_tokens = torch.empty(B, D + 1, **i32)
        self.new_len = torch.empty(B, **i32)
        if fused_head:  # stage 1 in the LM head's epilogue: per-CTA partials and the merged top-k
            self.lm_scratch = E.alloc_workspace(E.eagle_lmhead_topk_scratch_bytes(cfg), dev)
            self.lm_lse = torch.empty(B * k, dtype=torch.float32, device=dev)
            self.lm_ids = torch.empty(B * k, k, **i32)
            self.lm_vals = torch.empty(B * k, k, dtype=torch.float32, device=dev)

    # ---- stages -----------------------------------------------------------
    def draft(self, draft_logits: torch.Tensor, stream=None, steps=None, lse_in=None, head=None):
        """Stages 1-3. draft_logits: [D, B, k, V] (one contiguous block per step);
        lse_in: optional [D, B, k] row log-sum-exp supplied from upstream.
        head: optional (weight [V, H], hidden [D, B*k, H]), both bf16: each
        step's rows are then first written into draft_logits[s] by the LM head,
        or, with fused_head, reduced to their lse and top-k in the LM head's
        epilogue and expanded from those (draft_logits unused)."""
        cfg = self.cfg
        E.eagle_tree_init(cfg, self.ws, stream)
        for s in range(cfg.depth if steps is None else steps):
            if head is not None and self.fused_head:
                weight, hidden = head
                self.head_topk(weight, hidden[s], stream)
                E.eagle_expand_topk(cfg, self.ws, s, self.lm_ids, self.lm_vals, self.lm_lse, self.row_lse, self.ftok,
                                    self.fcount, stream)
                continue
            if head is not None:
                weight, hidden = head
                E.eagle_lmhead(cfg, self.ws, hidden.shape[-1], hidden[s], weight, draft_logits[s], stream)
            E.eagle_expand(cfg, self.ws, s, draft_logits[s], None if lse_in is None else lse_in[s], self.row_lse,
                           self.ftok, self.fcount, stream)
        if steps is None:
            E.eagle_rerank(cfg, self.ws, stream)

    def head_topk(self, weight, hidden_s, stream=None):
        """LM head of one step with stage 1 in its epilogue (fused_head)."""
        E.eagle_lmhead_topk(self.cfg, self.ws, hidden_s.shape[-1], hidden_s, weight, self.lm_scratch, self.lm_lse,
                            self.lm_ids, self.lm_vals, stream)

    def build(self, prefix_len, root_token, stream=None):
        E.eagle_build_tree(self.cfg, self.ws, prefix_len, root_token, self.tokens, self.parent, self.depth, self.pos,
                           self.mask, self.n_tree, stream)

    def attention(self, q, cache, layer, prefix_len, stream=None):
        E.eagle_tree_attention(self.kv, self.cfg.T, q, cache, layer, prefix_len, self.mask, self.n_tree,
                               self.attn_out, self.attn_ws, stream)

    def verify(self, mode, temperature, target, seed, cycle, stream=None):
        """Stage 6; lossless uniforms are Philox words of (seed, cycle) drawn on the device."""
        E.eagle_verify(self.cfg, self.ws, mode, temperature, seed, cycle, target, self.tokens, self.parent,
                       self.n_tree, self.accept_len, self.slots, self.out_tokens, stream=stream)

    def compact(self, cache, prefix_len, stream=None):
        E.eagle_kv_compact(self.kv, cache, prefix_len, self.accept_len, self.slots, self.cfg.depth + 1, self.new_len,
                           self.ws, stream)

    def run(self, draft_logits, prefix_len, root_token, q, cache, layer, target, seed, cycle, mode, temperature=1.0,
            compact=True, stream=None, head=None):
        """The whole cycle (all stages) enqueued on `stream`."""
        self.draft(draft_logits, stream, head=head)
        self.build(prefix_len, root_token, stream)
        self.attention(q, cache, layer, prefix_len, stream)
        self.verify(mode, temperature, target, seed, cycle, stream)
        if compact:
            self.compact(cache, prefix_len, stream)

    def status(self, stream=None) -> int:
        a = E.eagle_status_fetch(self.ws, stream)
        b = E.eagle_status_fetch(self.attn_ws, stream)
        return a or b


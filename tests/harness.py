"""Shared helpers of the parity tests: seeded inputs -> oracle and device.

Every expected value comes from the oracle run on the generator's inputs;
nothing computed by the CUDA library is ever fed to the oracle.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth
from synth import workloads as WL


# ------------------------------------------------------------- host inputs ---

class Inputs:
    """Host (numpy) inputs of one cycle of a workload."""

    def __init__(self, w: WL.Workload, seed: int = 42, planted: bool = False, attn_layer: int = 0):
        self.w, self.seed, self.planted = w, seed, planted
        self.draft = WL.draft_logits(w, seed, planted=planted)  # [D, B, k, V]
        self.target = WL.target_logits(w, seed)  # [B, T, V]
        self.prefix_len = w.prefix_lengths(seed)
        self.root = WL.root_tokens(w, seed)
        self.uniforms = WL.uniforms(w, seed, 0)
        self.attn_layer = attn_layer

    def oracle_tree(self, lse_in=None, policy: int = 0):
        """Stages 1-4 in the oracle; lse_in: [D, B, k] or None (own lse)."""
        w = self.w
        cfg = oracle.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, policy)
        t = oracle.Tree(cfg)
        fronts = []
        for s in range(w.depth):
            ft, fc = t.expand(s, self.draft[s], None if lse_in is None else lse_in[s])
            fronts.append((ft.copy(), fc.copy()))
        t.rerank()
        tr = t.build_tree(self.prefix_len, self.root)
        return t, tr, fronts

    def oracle_lse(self) -> np.ndarray:
        """Row lse (fp64 rounded to fp32) of every draft row, [D, B, k]."""
        w = self.w
        out = np.zeros((w.depth, w.batch, w.top_k), np.float32)
        for s in range(w.depth):
            for b in range(w.batch):
                for f in range(w.top_k):
                    _, out[s, b, f], _ = oracle.row_stats(self.draft[s, b, f], 1)
        return out

    def align_target(self, tr: dict, frac: float = 1.0, value: float | None = None) -> None:
        """Make the target favour the first kept child of each slot (from the given
        oracle tree) so that acceptance happens; value defaults to a 0.9-mass plant."""
        w = self.w
        rng = np.random.default_rng(self.seed + 1)
        v = value if value is not None else WL.plant_value(w, float(np.mean(w.sharpness_per_seq(self.seed))))
        for b in range(w.batch):
            n = int(tr["n_tree"][b])
            for t in range(n):
                kids = [c for c in range(n) if tr["parent"][b, c] == t]
                if kids and rng.random() < frac:
                    tok = int(tr["tokens"][b, kids[0]])
                    if self.target.dtype == np.uint16:
                        self.target[b, t, tok] = np.float32(v).view(np.uint32) >> 16
                    else:
                        self.target[b, t, tok] = v


# ------------------------------------------------------------ device side ---

def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    if a.dtype == np.uint8:
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(a).cuda()


def to_host(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def device_cycle(w: WL.Workload):
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E
    return C, E


def make_cfgs(w: WL.Workload, geo: dict, policy: int = 0):
    from speculative_decoding_dynamic_gb300 import eagle as E
    cfg = E.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, w.dtype, policy)
    kv = E.KvCfg(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, geo["layers"], geo["max_len"], w.dtype,
                 geo["seq_stride"], geo["layer_stride"], geo["kv_stride"], geo["pos_stride"])
    return cfg, kv


class DeviceKV:
    """Device KV cache of a workload: the attention layer is filled for
    positions [0, L_b + T); every other layer only on its tree region
    [L_b, L_b + T) (the only part compaction reads or writes)."""

    def __init__(self, inp: Inputs, layers: int):
        import torch
        w = inp.w
        self.geo = WL.kv_geometry(w, inp.seed, layers)
        g = self.geo
        n = w.batch * g["seq_stride"]
        dt = torch.float32 if w.dtype == synth.F32 else torch.bfloat16
        self.cache = torch.empty(n, dtype=dt, device="cuda")
        npdt = np.float32 if w.dtype == synth.F32 else np.uint16
        T = w.T
        for b in range(w.batch):
            L = int(inp.prefix_len[b])
            for layer in range(layers):
                for which in range(2):
                    p0 = 0 if layer == inp.attn_layer else L
                    p1 = L + T
                    host = np.zeros((p1 - p0) * g["pos_stride"], npdt)
                    base = b * g["seq_stride"] + layer * g["layer_stride"] + which * g["kv_stride"]
                    WL.kv_fill(host, w, g, b, layer, which, p0, p1, inp.seed, offset=base + p0 * g["pos_stride"])
                    lo = base + p0 * g["pos_stride"]
                    self.cache[lo:lo + host.size].copy_(to_dev(host).view(-1))
        self.inp = inp

    def host_layer(self, layer: int):
        """Host copies (K, V) of one layer as [B, max_len, Hkv, d] (unfilled positions zero)."""
        w, g = self.inp.w, self.geo
        npdt = np.float32 if w.dtype == synth.F32 else np.uint16
        shape = (w.batch, g["max_len"], w.n_kv_heads, w.head_dim)
        K = np.zeros(shape, npdt)
        V = np.zeros(shape, npdt)
        for b in range(w.batch):
            L = int(self.inp.prefix_len[b])
            p0 = 0 if layer == self.inp.attn_layer else L
            for which, arr in ((0, K), (1, V)):
                WL.kv_fill(arr, w, g, b, layer, which, p0, L + w.T, self.inp.seed,
                           offset=b * g["seq_stride"] + layer * g["layer_stride"] + which * g["kv_stride"]
                           - b * g["max_len"] * g["pos_stride"])
        return K, V

    def tree_regions(self) -> np.ndarray:
        """Device tree regions [B, layers, 2, T, Hkv, d] (host copy)."""
        w, g = self.inp.w, self.geo
        c = self.cache.view(w.batch, g["layers"], 2, g["max_len"], w.n_kv_heads, w.head_dim)
        out = []
        for b in range(w.batch):
            L = int(self.inp.prefix_len[b])
            out.append(to_host(c[b, :, :, L:L + w.T].contiguous()))
        return np.stack(out)


def tree_region_host(inp: Inputs, layers: int) -> np.ndarray:
    """Generator values of the tree regions [B, layers, 2, T, Hkv, d] before any compaction."""
    w = inp.w
    geo = WL.kv_geometry(w, inp.seed, layers)
    npdt = np.float32 if w.dtype == synth.F32 else np.uint16
    out = np.zeros((w.batch, layers, 2, w.T, w.n_kv_heads, w.head_dim), npdt)
    for b in range(w.batch):
        L = int(inp.prefix_len[b])
        for layer in range(layers):
            for which in range(2):
                sub = np.zeros(w.T * geo["pos_stride"], npdt)
                base = b * geo["seq_stride"] + layer * geo["layer_stride"] + which * geo["kv_stride"]
                WL.kv_fill(sub, w, geo, b, layer, which, L, L + w.T, inp.seed, offset=base + L * geo["pos_stride"])
                out[b, layer, which] = sub.reshape(w.T, w.n_kv_heads, w.head_dim)
    return out


def f32(a: np.ndarray) -> np.ndarray:
    return a.astype(np.float64) if a.dtype != np.uint16 else synth.bf16_to_f32(a).astype(np.float64)


def near_tie_tol(depth: int) -> float:
    """Largest |logv| difference that a 1e-5-accurate lse can flip, summed over a path."""
    return 2e-5 * max(1, depth)


def isclose_bits(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and (a.view(np.uint32) == b.view(np.uint32)).all()


def log_thr(thr: float) -> float:
    return -math.inf if thr <= 0 else float(np.float32(math.log(thr)))

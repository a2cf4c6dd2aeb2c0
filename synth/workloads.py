"""The five synthetic workloads of the draft-tree cycle and their seeded inputs.

Shapes follow the models the pages name (Llama-3.1-8B, Vicuna-13B,
Llama-3.3-70B; "EAGLE-2: Faster Inference ..." summary App. A for depth 6 /
10 expansion nodes) and the sharpness knob of the dynamic-trees tutorial's
widget. Logits are sharpness * N(0,1) (the public benchmark suites the pages
measure on are not reproduced; these synthetic rows stand in for them).
Nothing here computes any part of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import BF16, F32, STREAM_DRAFT, STREAM_HIDDEN, STREAM_K, STREAM_LMHEAD, STREAM_Q, STREAM_TARGET, STREAM_V, \
    kv_region, normal4, plant, seq_params, words


@dataclass
class Workload:
    name: str
    batch: int
    vocab: int
    top_k: int
    depth: int
    node_budget: int
    threshold: float
    dtype: int  # F32 / BF16 for logits and q/k/v
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    prefix: int | tuple[int, int]  # fixed length or (lmin, lspan) drawn per sequence
    sharpness: float | tuple[float, float]  # fixed or (smin, sspan) drawn per sequence
    verify: str  # "greedy" | "lossless"
    layers: int  # layers moved by compaction (memory-capped for 70B)
    model_layers: int
    temperature: float = 1.0
    hidden_size: int = 0  # LM-head input width of the model
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.node_budget + 1

    @property
    def W(self) -> int:
        return (self.T + 31) // 32

    @property
    def C(self) -> int:
        return self.top_k + (self.depth - 1) * self.top_k * self.top_k

    @property
    def esize(self) -> int:
        return 4 if self.dtype == F32 else 2

    def prefix_lengths(self, seed: int) -> np.ndarray:
        if isinstance(self.prefix, tuple):
            L, _ = seq_params(self.batch, self.prefix[0], self.prefix[1], 0.0, 0.0, seed)
            return L
        return np.full(self.batch, self.prefix, np.int32)

    def sharpness_per_seq(self, seed: int) -> np.ndarray:
        if isinstance(self.sharpness, tuple):
            _, s = seq_params(self.batch, 0, 0, self.sharpness[0], self.sharpness[1], seed)
            return s
        return np.full(self.batch, self.sharpness, np.float32)

    def max_len(self, seed: int) -> int:
        """Positions per (sequence, layer, K|V) region: longest prefix + T, rounded up to 64."""
        return int((int(self.prefix_lengths(seed).max()) + self.T + 63) // 64 * 64)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", batch=1, vocab=1024, top_k=2, depth=3, node_budget=8, threshold=0.1, dtype=F32,
                     n_q_heads=4, n_kv_heads=4, head_dim=16, prefix=32, sharpness=2.5, verify="greedy", layers=1,
                     model_layers=1, hidden_size=64,
                     notes="CPU-checkable cycle; threshold 0.1, k 2, N 8 as in the EAGLE notes' figure"),
    "llama8b_b1": Workload("llama8b_b1", batch=1, vocab=128256, top_k=10, depth=6, node_budget=60, threshold=0.0,
                           dtype=BF16, n_q_heads=32, n_kv_heads=8, head_dim=128, prefix=2048, sharpness=2.5,
                           verify="lossless", layers=32, model_layers=32, hidden_size=4096,
                           notes="Llama-3.1-8B shape, batch 1 (sharpness 0.8 and 2.5; greedy and lossless)"),
    "vicuna13b_b1": Workload("vicuna13b_b1", batch=1, vocab=32000, top_k=10, depth=6, node_budget=60, threshold=0.0,
                             dtype=BF16, n_q_heads=40, n_kv_heads=40, head_dim=128, prefix=4096, sharpness=2.5,
                             verify="lossless", layers=40, model_layers=40, hidden_size=5120,
                             notes="Vicuna-13B shape, batch 1, MHA, lossless at temperature 1"),
    "llama8b_b64": Workload("llama8b_b64", batch=64, vocab=128256, top_k=10, depth=6, node_budget=60, threshold=0.0,
                            dtype=BF16, n_q_heads=32, n_kv_heads=8, head_dim=128, prefix=(256, 1793),
                            sharpness=(0.8, 1.7), verify="greedy", layers=32, model_layers=32, hidden_size=4096,
                            notes="Llama-3.1-8B shape, batch 64, prefix U[256,2048], sharpness U[0.8,2.5]"),
    "llama70b_b8": Workload("llama70b_b8", batch=8, vocab=128256, top_k=8, depth=8, node_budget=64, threshold=0.0,
                            dtype=BF16, n_q_heads=64, n_kv_heads=8, head_dim=128, prefix=32768, sharpness=1.5,
                            verify="lossless", layers=16, model_layers=80, hidden_size=8192,
                            notes="Llama-3.3-70B shape, batch 8, 32K prefix; compaction capped at 16 of 80 layers"),
}


def plant_value(w: Workload, s: float) -> float:
    """Logit that gives a planted token about 0.9 of the softmax mass in a row of
    V - 1 draws of s*N(0,1): E[sum exp] = (V-1) exp(s^2/2), so ln(9 (V-1)) + s^2/2."""
    return math.log(9.0 * (w.vocab - 1)) + 0.5 * s * s


def draft_logits(w: Workload, seed: int, planted: bool = False) -> np.ndarray:
    """[D, B, k, V] (one contiguous [B, k, V] block per draft step): element
    (s, b, f, x) drawn at counter (x, f, b, s), stream 1."""
    s = w.sharpness_per_seq(seed)
    out = normal4((w.depth, w.batch, w.top_k, w.vocab), w.dtype, s, seed, STREAM_DRAFT, scale_axis=2)
    if planted:
        # one planted token per row, same value for the batch (uses the mean sharpness)
        plant(out, w.dtype, plant_value(w, float(np.mean(s))), seed, STREAM_DRAFT)
    return out


LMHEAD_STD = 0.02  # weight scale of the synthetic LM head


def lmhead_weight(w: Workload, seed: int) -> np.ndarray:
    """[V, H] bf16 LM-head weights, 0.02 * N(0,1): element (v, h) at counter (h, v, 0, 0), stream 9."""
    return normal4((w.vocab, w.hidden_size), BF16, LMHEAD_STD, seed, STREAM_LMHEAD)


def hidden_states(w: Workload, seed: int) -> np.ndarray:
    """[D, B*k, H] bf16 draft hidden states of the frontier rows, one block per
    draft step, scaled so that logits through ``lmhead_weight`` have standard
    deviation about the workload's (mean) sharpness: element (s, r, h) at
    counter (h, r, s, 0), stream 8."""
    s = float(np.mean(w.sharpness_per_seq(seed)))
    scale = s / (LMHEAD_STD * math.sqrt(w.hidden_size))
    return normal4((w.depth, w.batch * w.top_k, w.hidden_size), BF16, scale, seed, STREAM_HIDDEN)


def target_logits(w: Workload, seed: int) -> np.ndarray:
    """[B, T, V]: element (b, t, x) drawn at counter (x, t, b, 0), stream 2."""
    s = w.sharpness_per_seq(seed)
    return normal4((1, w.batch, w.T, w.vocab), w.dtype, s, seed, STREAM_TARGET, scale_axis=2).reshape(
        w.batch, w.T, w.vocab)


def queries(w: Workload, seed: int) -> np.ndarray:
    """[B, T, Hq, d] N(0,1), element counter (index, 0, 0, 0), stream 3."""
    n = w.batch * w.T * w.n_q_heads * w.head_dim
    return normal4((n,), w.dtype, 1.0, seed, STREAM_Q).reshape(w.batch, w.T, w.n_q_heads, w.head_dim)


def kv_geometry(w: Workload, seed: int, layers: int) -> dict:
    """Contiguous per-sequence cache [B][layers][2][max_len][Hkv][d] (element strides)."""
    Lmax = w.max_len(seed)
    pos_stride = w.n_kv_heads * w.head_dim
    kv_stride = Lmax * pos_stride
    layer_stride = 2 * kv_stride
    seq_stride = layers * layer_stride
    return dict(max_len=Lmax, pos_stride=pos_stride, kv_stride=kv_stride, layer_stride=layer_stride,
                seq_stride=seq_stride, layers=layers)


def kv_fill(buf: np.ndarray, w: Workload, geo: dict, b: int, layer: int, which: int, pos0: int, pos1: int,
            seed: int, offset: int = 0) -> None:
    """Fill positions [pos0, pos1) of (b, layer, K|V) of a cache laid out by kv_geometry.

    ``offset`` is subtracted from the element offset (for buffers that hold a sub-range)."""
    off = b * geo["seq_stride"] + layer * geo["layer_stride"] + which * geo["kv_stride"] - offset
    kv_region(buf, w.dtype, off, geo["pos_stride"], w.n_kv_heads, w.head_dim, pos0, pos1, layer, b, seed,
              STREAM_K + which)


def uniforms(w: Workload, seed: int, cycle: int = 0) -> np.ndarray:
    """[B, T+2] raw 32-bit words at counter (j, b, cycle, 0), stream 7."""
    return words(w.batch, w.T + 2, cycle, seed)


def root_tokens(w: Workload, seed: int) -> np.ndarray:
    return (words(1, w.batch, 0xABCD, seed, stream=6)[0] % np.uint32(w.vocab)).astype(np.int32)

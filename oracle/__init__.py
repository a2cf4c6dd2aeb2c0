"""CPU oracle of the EAGLE-2 draft-tree cycle (ctypes over oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and by
bench.py's cpu_baseline / reference leg, never by the product path. Shares no
code with the CUDA library. Arrays are numpy; bf16 data are uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp (g++ -O2 -ffp-contract=off) into _oracle.so next to it."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o",
                    _LIB_PATH + ".tmp"], check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    p, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.oracle_row_stats.argtypes = [p, i32, i32, i32, p, p, p]
    lib.oracle_dexp.argtypes = [f32]
    lib.oracle_dexp.restype = f32
    lib.oracle_tree_init.argtypes = [i32, i32, i32, p, p, p, p, p, p, p]
    lib.oracle_expand.argtypes = [i32, i32, i32, i32, i32, f32, i32, p, p, i32, p, p, p, p, p, p, p, p, p, p, p]
    lib.oracle_rerank.argtypes = [i32, i32, i32, i32, i32, i32, p, p, p, p, p, p]
    lib.oracle_build_tree.argtypes = [i32, i32, i32, i32, p, p, p, p, p, p, p, p, p, p, p, p, p]
    lib.oracle_value_sum.argtypes = [i32, p, p]
    lib.oracle_value_sum.restype = f64
    lib.oracle_attention.argtypes = [i32, i32, i32, i32, i32, i32, p, p, p, i64, i64, p, p, p, i32, p]
    lib.oracle_attention_rows.argtypes = [i32, p, i32, i32, i32, i32, i32, p, p, p, i64, i64, p, p, p, i32, p]
    lib.oracle_verify_greedy.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, p, p, p, p]
    lib.oracle_verify_lossless.argtypes = [i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p, p, p]
    lib.oracle_kv_compact.argtypes = [i32, i32, i32, i32, i32, p, i64, i64, i64, i64, p, p, p, i32, p]
    lib.oracle_lmhead_logits.argtypes = [i32, i32, i32, p, p, p]
    lib.oracle_expand_sampled.argtypes = [i32, i32, i32, i32, i32, f32, i32, p, p, p, i32, p, p, p, p, p, p, p, p,
                                          p, p, p]
    lib.oracle_dlog.argtypes = [i32, p, p]
    lib.oracle_gumbel.argtypes = [i32, p, p]
    lib.oracle_verify_draft.argtypes = [i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p, p, p]
    _lib = lib
    return lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle needs C-contiguous numpy arrays"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError(f"logits/qkv must be float32 or bf16-as-uint16, got {a.dtype}")


def capacity(k: int, depth: int) -> int:
    """Candidate capacity C = k + (D-1) k^2 (step 0 expands the root only)."""
    return k + (depth - 1) * k * k


def step_base(s: int, k: int) -> int:
    return 0 if s == 0 else k + (s - 1) * k * k


def log_threshold(thr: float) -> np.float32:
    """Threshold on the path value, in the log domain (thr = 0 -> -inf: off)."""
    return np.float32(-np.inf) if thr <= 0 else np.float32(math.log(thr))


def dexp(z: float) -> float:
    return float(_load().oracle_dexp(ctypes.c_float(z)))


def row_stats(row: np.ndarray, k: int):
    """(lse64, lse32, topk ids) of one vocabulary row."""
    row = np.ascontiguousarray(row)
    lse64 = np.zeros(1, np.float64)
    lse32 = np.zeros(1, np.float32)
    top = np.zeros(k, np.int32)
    _load().oracle_row_stats(_p(row), _dtype_code(row), row.shape[-1], k, _p(lse64), _p(lse32), _p(top))
    return float(lse64[0]), np.float32(lse32[0]), top


@dataclass
class TreeCfg:
    batch: int
    vocab: int
    top_k: int
    depth: int
    node_budget: int
    threshold: float = 0.0
    policy: int = 0  # 0 EAGLE-2, 1 confidence-based expansion, 2 without reranking, 3 static shape

    @property
    def C(self) -> int:
        return capacity(self.top_k, self.depth)

    @property
    def T(self) -> int:
        return self.node_budget + 1

    @property
    def W(self) -> int:
        return (self.T + 31) // 32


class Tree:
    """Per-cycle draft-tree state held by the oracle (one batch of sequences)."""

    def __init__(self, cfg: TreeCfg):
        self.cfg = cfg
        B, C, k = cfg.batch, cfg.C, cfg.top_k
        self.token = np.zeros((B, C), np.int32)
        self.parent = np.zeros((B, C), np.int32)
        self.depth = np.zeros((B, C), np.int32)
        self.logv = np.zeros((B, C), np.float32)
        self.valid = np.zeros((B, C), np.uint8)
        self.fnode = np.zeros((B, k), np.int32)
        self.fcount = np.zeros(B, np.int32)
        self.kept = np.zeros((B, C), np.uint8)
        self.n_kept = np.zeros(B, np.int32)
        self.lp = np.full((B, C), -np.inf, np.float32)               # each node's own confidence (log)
        self.fhist = np.full((cfg.depth + 1, B, k), -1, np.int32)   # frontier node ids of every step
        self.row_lse = np.full((B, cfg.depth, k), np.nan, np.float32)
        _load().oracle_tree_init(B, C, k, _p(self.token), _p(self.parent), _p(self.depth), _p(self.logv),
                                 _p(self.valid), _p(self.fnode), _p(self.fcount))

    def expand(self, step: int, logits_s: np.ndarray, lse_in: np.ndarray | None = None,
               words: np.ndarray | None = None):
        """Stages 1+2 for step ``step``; logits_s is [B, k, V]. Returns (frontier tokens [B,k], count [B]).
        words: optional uint32 [B, k, V]; the children are then drawn from the row's softmax
        without replacement (Gumbel-top-k) instead of being its top-k."""
        cfg = self.cfg
        B, k, V = cfg.batch, cfg.top_k, cfg.vocab
        logits_s = np.ascontiguousarray(logits_s)
        assert logits_s.shape == (B, k, V), logits_s.shape
        if lse_in is not None:
            lse_in = np.ascontiguousarray(lse_in, dtype=np.float32).reshape(B, k)
        lse_out = np.full((B, k), np.nan, np.float32)
        ftok = np.zeros((B, k), np.int32)
        fcnt = np.zeros(B, np.int32)
        if words is None:
            rc = _load().oracle_expand(B, V, k, step, _dtype_code(logits_s), log_threshold(cfg.threshold),
                                       cfg.policy, _p(logits_s), _p(lse_in), cfg.C, _p(self.token), _p(self.parent),
                                       _p(self.depth), _p(self.logv), _p(self.lp), _p(self.valid), _p(self.fnode),
                                       _p(self.fcount), _p(lse_out), _p(ftok), _p(fcnt))
        else:
            words = np.ascontiguousarray(words, np.uint32)
            assert words.shape == (B, k, V), words.shape
            rc = _load().oracle_expand_sampled(B, V, k, step, _dtype_code(logits_s), log_threshold(cfg.threshold),
                                               cfg.policy, _p(logits_s), _p(lse_in), _p(words), cfg.C,
                                               _p(self.token), _p(self.parent), _p(self.depth), _p(self.logv),
                                               _p(self.lp), _p(self.valid), _p(self.fnode), _p(self.fcount),
                                               _p(lse_out), _p(ftok), _p(fcnt))
        if rc != 0:
            raise RuntimeError(f"oracle_expand failed: {rc}")
        self.fhist[step + 1] = self.fnode
        self.row_lse[:, step, :] = lse_out
        return ftok, fcnt

    def rerank(self):
        cfg = self.cfg
        _load().oracle_rerank(cfg.batch, cfg.C, cfg.node_budget, cfg.policy, cfg.depth, cfg.top_k,
                              _p(self.fhist), _p(self.depth), _p(self.logv), _p(self.valid), _p(self.kept),
                              _p(self.n_kept))
        return self.kept, self.n_kept

    def build_tree(self, prefix_len: np.ndarray, root_token: np.ndarray):
        """Stage 4. Returns dict of tokens/parent/depth/pos [B,T], mask [B,T,W], n_tree [B], slot_of [B,C]."""
        cfg = self.cfg
        B, T, W, C = cfg.batch, cfg.T, cfg.W, cfg.C
        out = {
            "tokens": np.zeros((B, T), np.int32), "parent": np.zeros((B, T), np.int32),
            "depth": np.zeros((B, T), np.int32), "pos": np.zeros((B, T), np.int32),
            "mask": np.zeros((B, T, W), np.uint32), "n_tree": np.zeros(B, np.int32),
            "slot_of": np.zeros((B, C), np.int32),
        }
        pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
        rt = np.ascontiguousarray(root_token, dtype=np.int32)
        rc = _load().oracle_build_tree(B, C, T, W, _p(pl), _p(rt), _p(self.token), _p(self.parent), _p(self.depth),
                                       _p(self.kept), _p(out["tokens"]), _p(out["parent"]), _p(out["depth"]),
                                       _p(out["pos"]), _p(out["mask"]), _p(out["n_tree"]), _p(out["slot_of"]))
        if rc != 0:
            raise RuntimeError(f"oracle_build_tree failed: {rc}")
        return out

    def draft_rows(self, slot_of: np.ndarray, n_tree: np.ndarray) -> np.ndarray:
        """[B, T] int64: for each tree slot, the row of the draft logits [D, B, k, V]
        (flattened to [D*B*k, V]) its children were drawn from, -1 if never expanded."""
        cfg = self.cfg
        B, T, k, D = cfg.batch, cfg.T, cfg.top_k, cfg.depth
        out = np.full((B, T), -1, np.int64)
        for b in range(B):
            out[b, 0] = (0 * B + b) * k + 0  # the root: step 0, row 0
            for st in range(1, D):
                for f in range(k):
                    nid = int(self.fhist[st, b, f])
                    if nid >= 0 and self.kept[b, nid]:
                        sl = int(slot_of[b, nid])
                        if 0 <= sl < int(n_tree[b]):
                            out[b, sl] = (st * B + b) * k + f
        return out

    def value_sum(self, b: int) -> float:
        """Summed path value of the kept nodes of sequence b (expected accepted tokens)."""
        return float(_load().oracle_value_sum(self.cfg.C, _p(np.ascontiguousarray(self.logv[b])),
                                              _p(np.ascontiguousarray(self.kept[b]))))


def attention(q: np.ndarray, k_base: np.ndarray, v_base: np.ndarray, seq_stride: int, pos_stride: int,
              prefix_len, mask, n_tree, Hkv: int) -> np.ndarray:
    """Stage 5 over all rows; q [B,T,Hq,d]; returns float64 [B,T,Hq,d]."""
    B, T, Hq, d = q.shape
    W = mask.shape[-1]
    out = np.zeros((B, T, Hq, d), np.float64)
    _load().oracle_attention(B, T, Hq, Hkv, d, _dtype_code(q), _p(q), _p(k_base), _p(v_base), seq_stride,
                             pos_stride, _p(np.ascontiguousarray(prefix_len, np.int32)),
                             _p(np.ascontiguousarray(mask, np.uint32)), _p(np.ascontiguousarray(n_tree, np.int32)),
                             W, _p(out))
    return out


def attention_rows(rows: np.ndarray, q: np.ndarray, k_base: np.ndarray, v_base: np.ndarray, seq_stride: int,
                   pos_stride: int, prefix_len, mask, n_tree, Hkv: int) -> np.ndarray:
    """Stage 5 for selected (b, i, h) rows; returns float64 [n_rows, d]."""
    B, T, Hq, d = q.shape
    W = mask.shape[-1]
    rows = np.ascontiguousarray(rows, np.int32)
    out = np.zeros((rows.shape[0], d), np.float64)
    _load().oracle_attention_rows(rows.shape[0], _p(rows), T, Hq, Hkv, d, _dtype_code(q), _p(q), _p(k_base),
                                  _p(v_base), seq_stride, pos_stride,
                                  _p(np.ascontiguousarray(prefix_len, np.int32)),
                                  _p(np.ascontiguousarray(mask, np.uint32)),
                                  _p(np.ascontiguousarray(n_tree, np.int32)), W, _p(out))
    return out


def verify_greedy(target: np.ndarray, tokens, parent, n_tree, depth: int):
    """Stage 6, greedy. target [B,T,V]. Returns (accept_len, accepted_slots, out_tokens, argmax)."""
    B, T, V = target.shape
    Dp1 = depth + 1
    a = np.zeros(B, np.int32)
    slots = np.zeros((B, Dp1), np.int32)
    toks = np.zeros((B, Dp1), np.int32)
    am = np.zeros((B, T), np.int32)
    _load().oracle_verify_greedy(B, T, V, Dp1, _dtype_code(target), _p(np.ascontiguousarray(target)),
                                 _p(np.ascontiguousarray(tokens, np.int32)),
                                 _p(np.ascontiguousarray(parent, np.int32)),
                                 _p(np.ascontiguousarray(n_tree, np.int32)), _p(a), _p(slots), _p(toks), _p(am))
    return a, slots, toks, am


def verify_lossless(target: np.ndarray, tokens, parent, n_tree, uniforms, depth: int, inv_temp: float = 1.0,
                    row_stats_out: bool = False):
    """Stage 6, lossless. uniforms [B, T+2] uint32. Returns (accept_len, slots, out_tokens[, row_max, row_mass])."""
    B, T, V = target.shape
    Dp1 = depth + 1
    a = np.zeros(B, np.int32)
    slots = np.zeros((B, Dp1), np.int32)
    toks = np.zeros((B, Dp1), np.int32)
    rmax = np.zeros((B, T), np.float32) if row_stats_out else None
    rmass = np.zeros((B, T), np.uint64) if row_stats_out else None
    u = np.ascontiguousarray(uniforms, np.uint32)
    assert u.shape == (B, T + 2)
    _load().oracle_verify_lossless(B, T, V, Dp1, _dtype_code(target), ctypes.c_float(inv_temp),
                                   _p(np.ascontiguousarray(target)), _p(np.ascontiguousarray(tokens, np.int32)),
                                   _p(np.ascontiguousarray(parent, np.int32)),
                                   _p(np.ascontiguousarray(n_tree, np.int32)), _p(u), _p(a), _p(slots), _p(toks),
                                   _p(rmax), _p(rmass))
    if row_stats_out:
        return a, slots, toks, rmax, rmass
    return a, slots, toks


def kv_compact(cache: np.ndarray, B: int, layers: int, Hkv: int, d: int, seq_stride: int, layer_stride: int,
               kv_stride: int, pos_stride: int, prefix_len, accept_len, accepted_slots) -> np.ndarray:
    """Stage 6b in place on ``cache`` (element strides). Returns new_len [B]."""
    new_len = np.zeros(B, np.int32)
    Dp1 = accepted_slots.shape[-1]
    _load().oracle_kv_compact(B, layers, Hkv, d, cache.itemsize, _p(cache), seq_stride, layer_stride, kv_stride,
                              pos_stride, _p(np.ascontiguousarray(prefix_len, np.int32)),
                              _p(np.ascontiguousarray(accept_len, np.int32)),
                              _p(np.ascontiguousarray(accepted_slots, np.int32)), Dp1, _p(new_len))
    return new_len


def lmhead_logits(hidden: np.ndarray, W: np.ndarray) -> np.ndarray:
    """LM-head logits of frontier rows: hidden [M, H] and W [V, H] as bf16 bits (uint16);
    returns fp32 [M, V] (exact dot products rounded once to fp32)."""
    hidden = np.ascontiguousarray(hidden, np.uint16)
    W = np.ascontiguousarray(W, np.uint16)
    M, H = hidden.shape
    V, H2 = W.shape
    assert H == H2
    out = np.empty((M, V), np.float32)
    rc = _load().oracle_lmhead_logits(M, V, H, _p(hidden), _p(W), _p(out))
    if rc != 0:
        raise RuntimeError(f"oracle_lmhead_logits failed: {rc}")
    return out


def dlog(y: np.ndarray) -> np.ndarray:
    """The oracle's fixed-order fp32 logarithm (positive normal inputs)."""
    y = np.ascontiguousarray(y, np.float32)
    out = np.empty_like(y)
    _load().oracle_dlog(y.size, _p(y), _p(out))
    return out


def gumbel(words: np.ndarray) -> np.ndarray:
    """Gumbel noise -ln(-ln u) of uint32 words (u = ((w >> 9) + 1/2) 2^-23), fp32."""
    w = np.ascontiguousarray(words, np.uint32)
    out = np.empty(w.shape, np.float32)
    _load().oracle_gumbel(w.size, _p(w), _p(out))
    return out


def verify_draft(target: np.ndarray, draft: np.ndarray, draft_row: np.ndarray, tokens, parent, n_tree, uniforms,
                 depth: int, inv_temp: float = 1.0):
    """Stage 6 with the draft-probability rule (children drawn from the draft rows).
    target [B,T,V]; draft [R,V] (same dtype); draft_row [B,T] int64. Returns (accept_len, slots, out_tokens)."""
    B, T, V = target.shape
    Dp1 = depth + 1
    a = np.zeros(B, np.int32)
    slots = np.zeros((B, Dp1), np.int32)
    toks = np.zeros((B, Dp1), np.int32)
    u = np.ascontiguousarray(uniforms, np.uint32)
    assert u.shape == (B, T + 2)
    draft = np.ascontiguousarray(draft)
    assert draft.dtype == target.dtype and draft.shape[-1] == V
    rc = _load().oracle_verify_draft(B, T, V, Dp1, _dtype_code(target), ctypes.c_float(inv_temp),
                                     _p(np.ascontiguousarray(target)), _p(draft),
                                     _p(np.ascontiguousarray(draft_row, np.int64)),
                                     _p(np.ascontiguousarray(tokens, np.int32)),
                                     _p(np.ascontiguousarray(parent, np.int32)),
                                     _p(np.ascontiguousarray(n_tree, np.int32)), _p(u), _p(a), _p(slots), _p(toks))
    if rc != 0:
        raise RuntimeError(f"oracle_verify_draft failed: {rc}")
    return a, slots, toks

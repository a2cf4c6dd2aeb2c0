"""Python binding of libeagle (ctypes). Argument marshalling only.

Every function has the name of the C entry point it calls (see
include/eagle.h for the contract). Tensors are torch CUDA tensors; their data
pointers and the current CUDA stream are passed through. Importing this module
fails loudly if the CUDA library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# EAGLE_DEBUG=1: the checked library (each launching call waits and returns
# its own kernels' device status; internal indices range-checked)
DEBUG = os.environ.get("EAGLE_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libeagle_debug.so" if DEBUG else "libeagle.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{os.path.basename(LIB_PATH)} is missing ({LIB_PATH}); build it with "
                      "`python -m speculative_decoding_dynamic_gb300.build" + (" --debug" if DEBUG else "") +
                      "` (nvcc, sm_103a)")
_lib = ctypes.CDLL(LIB_PATH)

EAGLE_OK = 0
EAGLE_F32, EAGLE_BF16 = 0, 1
GREEDY, LOSSLESS, DRAFT = 0, 1, 2
MAX_TOPK, MAX_DEPTH, MAX_SLOTS, MAX_CANDIDATES = 16, 16, 256, 1024


class EagleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.eagle_status_string(code).decode()
        if code == -3:  # EAGLE_ERR_LAUNCH: add the CUDA error
            cmsg = ctypes.c_char_p()
            cerr = _lib.eagle_last_cuda_error(ctypes.byref(cmsg))
            msg += f"; CUDA error {cerr}: {cmsg.value.decode() if cmsg.value else ''}"
        super().__init__(f"{fn} -> {code} ({msg})")
        self.code = code


class TreeCfg(ctypes.Structure):
    """eagle_tree_cfg."""
    _fields_ = [("batch", ctypes.c_int), ("vocab", ctypes.c_int), ("top_k", ctypes.c_int), ("depth", ctypes.c_int),
                ("node_budget", ctypes.c_int), ("threshold", ctypes.c_float), ("logit_dtype", ctypes.c_int),
                ("policy", ctypes.c_int)]

    @property
    def T(self) -> int:
        return self.node_budget + 1

    @property
    def W(self) -> int:
        return (self.T + 31) // 32

    @property
    def C(self) -> int:
        return self.top_k + (self.depth - 1) * self.top_k * self.top_k


class KvCfg(ctypes.Structure):
    """eagle_kv_cfg (strides in elements)."""
    _fields_ = [("batch", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("layers", ctypes.c_int), ("max_len", ctypes.c_int),
                ("dtype", ctypes.c_int), ("seq_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("kv_stride", ctypes.c_int64), ("pos_stride", ctypes.c_int64)]


_p = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_TP = ctypes.POINTER(TreeCfg)
_KP = ctypes.POINTER(KvCfg)

_lib.eagle_workspace_bytes.argtypes = [_TP]
_lib.eagle_workspace_bytes.restype = _sz
_lib.eagle_tree_init.argtypes = [_TP, _p, _sz, _p]
_lib.eagle_expand.argtypes = [_TP, _p, _sz, _i, _p, _p, _p, _p, _p, _p]
_lib.eagle_expand_sampled.argtypes = [_TP, _p, _sz, _i, _p, _p, ctypes.c_uint64, ctypes.c_uint64, _p, _p, _p, _p]
_lib.eagle_test_expand_starved.argtypes = [_TP, _p, _sz, _i, _p, _p, _p, _p, _p]
_lib.eagle_lmhead.argtypes = [_TP, _p, _sz, _i, _p, _p, _p, _p]
_lib.eagle_lmhead_topk_scratch_bytes.argtypes = [_TP]
_lib.eagle_lmhead_topk_scratch_bytes.restype = _sz
_lib.eagle_lmhead_topk.argtypes = [_TP, _p, _sz, _i, _p, _p, _p, _sz, _p, _p, _p, _p]
_lib.eagle_rerank.argtypes = [_TP, _p, _sz, _p]
_lib.eagle_tree_value.argtypes = [_TP, _p, _sz, _p, _p]
_lib.eagle_build_tree.argtypes = [_TP, _p, _sz, _p, _p, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_attention_workspace_bytes.argtypes = [_KP, _i]
_lib.eagle_attention_workspace_bytes.restype = _sz
_lib.eagle_tree_attention.argtypes = [_KP, _i, _p, _p, _i, _p, _p, _p, _p, _p, _sz, _p]
_u64 = ctypes.c_uint64
_lib.eagle_verify.argtypes = [_TP, _p, _sz, _i, ctypes.c_float, _u64, _u64, _p, _p, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_shard_partials.argtypes = [_TP, _p, _sz, _i, _i, _i, _p, _p, _p, _p]
_lib.eagle_shard_merge.argtypes = [_TP, _p, _sz, _i, _i, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_expand_topk.argtypes = [_TP, _p, _sz, _i, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_verify_argmax.argtypes = [_TP, _p, _sz, _p, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_kv_compact.argtypes = [_KP, _p, _p, _p, _p, _i, _p, _p, _p]
_lib.eagle_verify_static.argtypes = [_TP, _i, ctypes.c_float, _u64, _u64, _p, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_status_fetch.argtypes = [_p, ctypes.POINTER(ctypes.c_int), _p]
_lib.eagle_tree_export.argtypes = [_TP, _p, _sz, _p, _p, _p, _p, _p, _p, _p, _p]
_lib.eagle_verify_export.argtypes = [_TP, _p, _sz, _p, _p, _p, _p]
_lib.eagle_test_sampling.argtypes = [_p, _p, _i, _p, _p, _p]
_lib.eagle_kernel_launches.restype = ctypes.c_uint64
_lib.eagle_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
_lib.eagle_last_cuda_error.restype = _i
_lib.eagle_status_string.argtypes = [_i]
_lib.eagle_status_string.restype = ctypes.c_char_p


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != EAGLE_OK:
        raise EagleError(fn, rc)


def _ws(ws) -> tuple[int, int]:
    return ws.data_ptr(), ws.numel() * ws.element_size()


def eagle_workspace_bytes(cfg: TreeCfg) -> int:
    return int(_lib.eagle_workspace_bytes(ctypes.byref(cfg)))


def eagle_attention_workspace_bytes(kv: KvCfg, T: int) -> int:
    return int(_lib.eagle_attention_workspace_bytes(ctypes.byref(kv), T))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned uint8 device tensor (torch allocations are 512-byte aligned)."""
    if nbytes <= 0:
        raise ValueError("invalid configuration (workspace size 0)")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def eagle_tree_init(cfg, ws, stream=None):
    _check("eagle_tree_init", _lib.eagle_tree_init(ctypes.byref(cfg), *_ws(ws), _stream(stream)))


def eagle_expand(cfg, ws, step, draft_logits, row_lse_in, row_lse, frontier_tokens, frontier_count, stream=None):
    _check("eagle_expand", _lib.eagle_expand(ctypes.byref(cfg), *_ws(ws), step, _ptr(draft_logits),
                                             _ptr(row_lse_in), _ptr(row_lse), _ptr(frontier_tokens),
                                             _ptr(frontier_count), _stream(stream)))


def eagle_expand_sampled(cfg, ws, step, draft_logits, row_lse_in, seed, cycle, row_lse, frontier_tokens,
                         frontier_count, stream=None):
    """Stages 1+2 with the children drawn from each row's softmax without replacement (Gumbel-top-k)."""
    _check("eagle_expand_sampled", _lib.eagle_expand_sampled(ctypes.byref(cfg), *_ws(ws), step, _ptr(draft_logits),
                                                             _ptr(row_lse_in), int(seed), int(cycle), _ptr(row_lse),
                                                             _ptr(frontier_tokens), _ptr(frontier_count),
                                                             _stream(stream)))


def eagle_test_expand_starved(cfg, ws, step, draft_logits, row_lse, frontier_tokens, frontier_count, stream=None):
    """Failure-path test hook: expansion whose row ring receives no copies (status 2 expected)."""
    _check("eagle_test_expand_starved", _lib.eagle_test_expand_starved(ctypes.byref(cfg), *_ws(ws), step,
                                                                       _ptr(draft_logits), _ptr(row_lse),
                                                                       _ptr(frontier_tokens), _ptr(frontier_count),
                                                                       _stream(stream)))


def eagle_lmhead(cfg, ws, hidden_dim, hidden, weight, draft_logits, stream=None):
    _check("eagle_lmhead", _lib.eagle_lmhead(ctypes.byref(cfg), *_ws(ws), hidden_dim, _ptr(hidden), _ptr(weight),
                                             _ptr(draft_logits), _stream(stream)))


def eagle_lmhead_topk_scratch_bytes(cfg: TreeCfg) -> int:
    return int(_lib.eagle_lmhead_topk_scratch_bytes(ctypes.byref(cfg)))


def eagle_lmhead_topk(cfg, ws, hidden_dim, hidden, weight, scratch, row_lse, topk_ids, topk_logits, stream=None):
    _check("eagle_lmhead_topk", _lib.eagle_lmhead_topk(ctypes.byref(cfg), *_ws(ws), hidden_dim, _ptr(hidden),
                                                       _ptr(weight), *_ws(scratch), _ptr(row_lse), _ptr(topk_ids),
                                                       _ptr(topk_logits), _stream(stream)))


def eagle_rerank(cfg, ws, stream=None):
    _check("eagle_rerank", _lib.eagle_rerank(ctypes.byref(cfg), *_ws(ws), _stream(stream)))


def eagle_tree_value(cfg, ws, value_sum, stream=None):
    _check("eagle_tree_value", _lib.eagle_tree_value(ctypes.byref(cfg), *_ws(ws), _ptr(value_sum), _stream(stream)))


def eagle_build_tree(cfg, ws, prefix_len, root_token, tokens, parent, depth, pos_ids, mask, n_tree, stream=None):
    _check("eagle_build_tree", _lib.eagle_build_tree(ctypes.byref(cfg), *_ws(ws), _ptr(prefix_len), _ptr(root_token),
                                                     _ptr(tokens), _ptr(parent), _ptr(depth), _ptr(pos_ids),
                                                     _ptr(mask), _ptr(n_tree), _stream(stream)))


def eagle_tree_attention(kv, T, q, kv_cache, layer, prefix_len, mask, n_tree, out, ws, stream=None):
    _check("eagle_tree_attention", _lib.eagle_tree_attention(ctypes.byref(kv), T, _ptr(q), _ptr(kv_cache), layer,
                                                             _ptr(prefix_len), _ptr(mask), _ptr(n_tree), _ptr(out),
                                                             *_ws(ws), _stream(stream)))


def eagle_verify(cfg, ws, mode, temperature, seed, cycle, target_logits, tokens, parent, n_tree, accept_len,
                 accepted_slots, out_tokens, draft_logits=None, stream=None):
    _check("eagle_verify", _lib.eagle_verify(ctypes.byref(cfg), *_ws(ws), mode, float(temperature), int(seed),
                                             int(cycle), _ptr(target_logits), _ptr(draft_logits), _ptr(tokens),
                                             _ptr(parent), _ptr(n_tree), _ptr(accept_len), _ptr(accepted_slots),
                                             _ptr(out_tokens), _stream(stream)))


def eagle_verify_static(cfg, mode, temperature, seed, cycle, target_logits, tokens, parent, n_tree, accept_len,
                        accepted_slots, out_tokens, stream=None):
    """eagle_verify for callers that may not allocate: scratch lives in a fixed device array of the library."""
    _check("eagle_verify_static", _lib.eagle_verify_static(ctypes.byref(cfg), mode, float(temperature), int(seed),
                                                           int(cycle), _ptr(target_logits), _ptr(tokens),
                                                           _ptr(parent), _ptr(n_tree), _ptr(accept_len),
                                                           _ptr(accepted_slots), _ptr(out_tokens), _stream(stream)))


def eagle_shard_partials(cfg, ws, rows, shard_vocab, vocab_offset, logits, part_max_sum, part_keys, stream=None):
    _check("eagle_shard_partials", _lib.eagle_shard_partials(ctypes.byref(cfg), *_ws(ws), rows, shard_vocab,
                                                             vocab_offset, _ptr(logits), _ptr(part_max_sum),
                                                             _ptr(part_keys), _stream(stream)))


def eagle_shard_merge(cfg, ws, n_shards, rows, part_max_sum, part_keys, row_lse, topk_ids, topk_logits, row_argmax,
                      stream=None):
    _check("eagle_shard_merge", _lib.eagle_shard_merge(ctypes.byref(cfg), *_ws(ws), n_shards, rows,
                                                       _ptr(part_max_sum), _ptr(part_keys), _ptr(row_lse),
                                                       _ptr(topk_ids), _ptr(topk_logits), _ptr(row_argmax),
                                                       _stream(stream)))


def eagle_expand_topk(cfg, ws, step, topk_ids, topk_logits, row_lse_in, row_lse, frontier_tokens, frontier_count,
                      stream=None):
    _check("eagle_expand_topk", _lib.eagle_expand_topk(ctypes.byref(cfg), *_ws(ws), step, _ptr(topk_ids),
                                                       _ptr(topk_logits), _ptr(row_lse_in), _ptr(row_lse),
                                                       _ptr(frontier_tokens), _ptr(frontier_count), _stream(stream)))


def eagle_verify_argmax(cfg, ws, row_argmax, tokens, parent, n_tree, accept_len, accepted_slots, out_tokens,
                        stream=None):
    _check("eagle_verify_argmax", _lib.eagle_verify_argmax(ctypes.byref(cfg), *_ws(ws), _ptr(row_argmax),
                                                           _ptr(tokens), _ptr(parent), _ptr(n_tree),
                                                           _ptr(accept_len), _ptr(accepted_slots), _ptr(out_tokens),
                                                           _stream(stream)))


def eagle_kv_compact(kv, kv_cache, prefix_len, accept_len, accepted_slots, slots_stride, new_len, ws=None,
                     stream=None):
    _check("eagle_kv_compact", _lib.eagle_kv_compact(ctypes.byref(kv), _ptr(kv_cache), _ptr(prefix_len),
                                                     _ptr(accept_len), _ptr(accepted_slots), slots_stride,
                                                     _ptr(new_len), _ptr(ws), _stream(stream)))


def eagle_status_fetch(ws, stream=None) -> int:
    """Synchronises the stream; returns the device status code (0 = no fault) and clears it."""
    st = ctypes.c_int(0)
    _lib.eagle_status_fetch(_ptr(ws), ctypes.byref(st), _stream(stream))
    return int(st.value)


def eagle_tree_export(cfg, ws, cand_token=None, cand_parent=None, cand_depth=None, cand_logv=None, cand_valid=None,
                      kept=None, n_kept=None, stream=None):
    _check("eagle_tree_export", _lib.eagle_tree_export(ctypes.byref(cfg), *_ws(ws), _ptr(cand_token),
                                                       _ptr(cand_parent), _ptr(cand_depth), _ptr(cand_logv),
                                                       _ptr(cand_valid), _ptr(kept), _ptr(n_kept), _stream(stream)))


def eagle_verify_export(cfg, ws, row_max=None, row_argmax=None, row_mass=None, stream=None):
    _check("eagle_verify_export", _lib.eagle_verify_export(ctypes.byref(cfg), *_ws(ws), _ptr(row_max),
                                                           _ptr(row_argmax), _ptr(row_mass), _stream(stream)))


def eagle_test_sampling(words, ys, n, gumbel_out, log_out, stream=None):
    _check("eagle_test_sampling", _lib.eagle_test_sampling(_ptr(words), _ptr(ys), n, _ptr(gumbel_out), _ptr(log_out),
                                                           _stream(stream)))


def eagle_kernel_launches() -> int:
    return int(_lib.eagle_kernel_launches())


def raw_call(name: str, *args) -> int:
    """Call an entry point with raw ctypes arguments and return its status (host-side checks in tests)."""
    return int(getattr(_lib, name)(*args))

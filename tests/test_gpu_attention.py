"""Tree attention on the GPU against the fp64 oracle, on every row.

Shapes cover GQA group sizes 1, 4 and 8, ragged prefixes (partial key tiles),
several key tiles per CTA and split-KV merges, trees with padded slots, and
NaN bit patterns planted in cache rows no query may see (positions past the
last used tree slot), which must not leak into the output.
"""
import numpy as np
import pytest

import oracle
import synth

import harness as H

pytestmark = pytest.mark.gpu


def _case(B, Hq, Hkv, d, k, D, N, L, max_len, dtype, seed, nan_tail=True, threshold=0.0, with_vmax=False):
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E

    V = 64
    cfg_o = oracle.TreeCfg(B, V, k, D, N, threshold)
    logits = synth.normal4((D, B, k, V), synth.F32, 2.0, seed, synth.STREAM_DRAFT)
    t = oracle.Tree(cfg_o)
    for s in range(D):
        t.expand(s, logits[s])
    t.rerank()
    L = np.asarray(L, np.int32)
    tr = t.build_tree(L, np.zeros(B, np.int32))
    T = N + 1
    npdt = np.float32 if dtype == synth.F32 else np.uint16
    pos_stride = Hkv * d
    kv_stride = max_len * pos_stride
    layers = 2
    seq_stride = layers * 2 * kv_stride
    layer = 1
    cache = np.zeros(B * seq_stride, npdt)
    if nan_tail:
        cache[:] = 0x7FC0 if dtype == synth.BF16 else np.float32(np.nan)
    for b in range(B):
        for which in range(2):
            off = b * seq_stride + layer * 2 * kv_stride + which * kv_stride
            synth.kv_region(cache, dtype, off, pos_stride, Hkv, d, 0, int(L[b]) + int(tr["n_tree"][b]), layer, b, seed,
                            synth.STREAM_K + which)
    q = synth.normal4((B * T * Hq * d,), dtype, 1.0, seed, synth.STREAM_Q).reshape(B, T, Hq, d)
    c5 = cache.reshape(B, layers, 2, max_len, Hkv, d)
    kh = np.ascontiguousarray(c5[:, layer, 0])
    vh = np.ascontiguousarray(c5[:, layer, 1])
    want = oracle.attention(q, kh, vh, max_len * pos_stride, pos_stride, L, tr["mask"], tr["n_tree"], Hkv)

    kv = E.KvCfg(B, Hq, Hkv, d, layers, max_len, dtype, seq_stride, 2 * kv_stride, kv_stride, pos_stride)
    ws = E.alloc_workspace(E.eagle_attention_workspace_bytes(kv, T))
    out = torch.full((B, T, Hq, d), float("nan"), dtype=torch.float32 if dtype == synth.F32 else torch.bfloat16,
                     device="cuda")
    E.eagle_tree_attention(kv, T, H.to_dev(q), H.to_dev(cache), layer, H.to_dev(L), H.to_dev(tr["mask"]),
                           H.to_dev(tr["n_tree"]), out, ws)
    torch.cuda.synchronize()
    assert E.eagle_status_fetch(ws) == 0
    got = H.f32(H.to_host(out))
    if with_vmax:
        return got, want, tr, float(np.nanmax(np.abs(H.f32(vh))))  # (tails past the keys hold NaN)
    return got, want, tr


@pytest.mark.parametrize("B,Hq,Hkv,N,k,D,L,max_len", [
    (2, 8, 2, 60, 10, 6, [100, 300], 384),      # G=4, 2 row blocks, partial tiles
    (1, 4, 4, 60, 10, 6, [1000], 1088),         # G=1 (MHA), one row block of 61 rows, split-KV
    (3, 16, 2, 64, 8, 8, [5, 130, 777], 896),   # G=8, 5 row blocks, tiny and ragged prefixes
    (1, 32, 8, 60, 10, 6, [2048], 2112),        # the Llama-3.1-8B b1 shape
    (2, 8, 8, 20, 4, 3, [0, 129], 192),         # empty prefix, many padded slots? (N small)
])
def test_tensor_core_attention_matches_oracle(B, Hq, Hkv, N, k, D, L, max_len):
    got, want, tr = _case(B, Hq, Hkv, 128, k, D, N, L, max_len, synth.BF16, seed=5)
    assert np.isfinite(got).all()
    err = np.abs(got - want).max()
    assert err <= 1e-2, err
    # unused slots are zero rows
    for b in range(B):
        assert (got[b, tr["n_tree"][b]:] == 0).all()


def test_tensor_core_attention_with_threshold_padding():
    # threshold prunes the tree below N: many padded slots, their keys never visible
    got, want, tr = _case(2, 8, 2, 128, 4, 4, 40, [64, 200], 320, synth.BF16, seed=9, threshold=0.2)
    assert (tr["n_tree"] < 41).any()
    assert np.abs(got - want).max() <= 1e-2


@pytest.mark.parametrize("d", [16, 64, 128])
def test_fp32_attention_matches_oracle(d):
    got, want, _ = _case(2, 4, 2, d, 2, 3, 8, [32, 7], 64, synth.F32, seed=3, nan_tail=False)
    assert np.abs(got - want).max() <= 1e-4


# Shapes whose (sequence, KV head, row block) items fill two CTAs on every SM
# run on the persistent pipeline kernel (64-key tiles, two CTAs per SM,
# sequences longest first). Bound, element by element, from the arithmetic:
# each weight p_k enters PV as bf16 (relative error <= 2^-9), which moves
# sum_k p_k v_k / l by at most 2^-9 max|V|; the row sum l is taken from the
# unrounded p and the output is rounded to bf16, each <= 2^-9 |o|; 1e-4
# covers the fp32 sums. Rows that see only a few keys (prefix 0 or 1) reach
# |o| > 2, where a bf16 step is 2^-6, so a flat 1e-2 would not follow.
@pytest.mark.parametrize("B,Hq,Hkv,N,k,D,lmax,seed,threshold", [
    (20, 32, 8, 60, 10, 6, 700, 21, 0.0),   # G=4, two row blocks: 320 items
    (40, 8, 8, 60, 10, 6, 400, 22, 0.0),    # G=1, one row block of 61 rows: 320 items
    (24, 32, 8, 40, 4, 4, 300, 23, 0.2),    # threshold-pruned trees: padded slots
])
def test_persistent_pipeline_matches_oracle(B, Hq, Hkv, N, k, D, lmax, seed, threshold):
    rng = np.random.default_rng(seed)
    L = rng.integers(0, lmax, B)
    L[:4] = [0, 1, 63, 64]  # empty prefix, tile edges
    max_len = int((L.max() + N + 1 + 63) // 64 * 64)
    got, want, tr, vmax = _case(B, Hq, Hkv, 128, k, D, N, list(L), max_len, synth.BF16, seed=seed,
                                threshold=threshold, with_vmax=True)
    assert np.isfinite(got).all()
    bound = 2.0 ** -8 * np.abs(want) + 2.0 ** -9 * vmax + 1e-4
    excess = np.abs(got - want) - bound
    assert excess.max() <= 0.0, (float(excess.max()), float(np.abs(got - want).max()))
    for b in range(B):
        assert (got[b, tr["n_tree"][b]:] == 0).all()

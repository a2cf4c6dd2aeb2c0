"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: the
tutorial's worked chain, library routines (scipy logsumexp, numpy sorts),
closed forms, brute-force enumeration on tiny trees, an independent
sequence-based attention, and exact probabilities of the acceptance rule.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run_tree(cfg, logits, prefix_len=None, root_token=None):
    """Oracle stages 1-4 on draft logits [B, D, k, V]."""
    t = oracle.Tree(cfg)
    for s in range(cfg.depth):
        t.expand(s, np.ascontiguousarray(logits[:, s]))
    t.rerank()
    B = cfg.batch
    pl = np.zeros(B, np.int32) if prefix_len is None else prefix_len
    rt = np.zeros(B, np.int32) if root_token is None else root_token
    return t, t.build_tree(pl, rt)


# ------------------------------------------------------------ worked chain ---

def test_worked_chain_sum_of_values():
    g = json.load(open(os.path.join(GOLDEN, "worked_chain.json")))
    vals = g["path_values"]
    D = len(vals)
    conf = [vals[0]] + [vals[i] / vals[i - 1] for i in range(1, D)]
    V, k = 2, 1
    cfg = oracle.TreeCfg(batch=1, vocab=V, top_k=k, depth=D, node_budget=D)
    logits = np.zeros((1, D, k, V), np.float32)
    for s, c in enumerate(conf):
        logits[0, s, 0] = [math.log(c), math.log(1.0 - c)]
    t, tr = _run_tree(cfg, logits)
    kept_vals = np.exp(t.logv[0][t.kept[0] == 1].astype(np.float64))
    np.testing.assert_allclose(np.sort(kept_vals)[::-1], vals, atol=1e-6)
    assert abs(t.value_sum(0) - g["expected_accepted"]) < 1e-6
    assert tr["n_tree"][0] == D + 1
    assert list(tr["parent"][0]) == [-1, 0, 1, 2, 3]


# ----------------------------------------------------------------- stage 1 ---

@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_row_lse_matches_scipy(dtype):
    V = 4099
    rows = synth.normal4((6, V), dtype, 2.5, seed=3, stream=synth.STREAM_DRAFT)
    for r in range(rows.shape[0]):
        row = rows[r]
        x = row.astype(np.float64) if dtype == synth.F32 else synth.bf16_to_f32(row).astype(np.float64)
        lse64, lse32, _ = oracle.row_stats(row, 5)
        assert abs(lse64 - logsumexp(x)) <= 1e-12 * abs(lse64) + 1e-12
        assert lse32 == np.float32(lse64)


def test_row_lse_closed_forms():
    V = 1000
    row = np.full(V, 0.75, np.float32)
    lse64, _, top = oracle.row_stats(row, 4)
    assert abs(lse64 - (0.75 + math.log(V))) < 1e-12
    assert list(top) == [0, 1, 2, 3]  # all equal: lowest ids first
    row = np.full(V, -300.0, np.float32)
    row[417] = 5.0
    lse64, lse32, top = oracle.row_stats(row, 1)
    assert lse32 == np.float32(5.0) and top[0] == 417


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_topk_matches_lexsort_with_ties(dtype):
    V, k = 2048, 10
    rows = synth.normal4((8, V), dtype, 1.0, seed=11, stream=synth.STREAM_DRAFT)
    # plant exact ties at the top of some rows
    rows[0, [5, 900, 77]] = rows[0].max() if dtype == synth.F32 else rows[0, np.argmax(synth.bf16_to_f32(rows[0]))]
    rows[1, :] = rows[1, 0]
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        x = row if dtype == synth.F32 else synth.bf16_to_f32(row)
        want = np.lexsort((np.arange(V), -x.astype(np.float64)))[:k]
        _, _, top = oracle.row_stats(row, k)
        assert list(top) == list(want)


def test_dexp_accuracy():
    z = np.concatenate([np.linspace(-32.0, 0.0, 200001, dtype=np.float32),
                        np.array([0.0, -1e-8, -0.5, -0.34657359, -0.34657360, -31.999, -32.0], np.float32)])
    worst = 0.0
    for v in z[::7]:
        got = oracle.dexp(float(v))
        ref = math.exp(float(v))
        worst = max(worst, abs(got - ref) / ref)
    assert worst < 4 * 2.0 ** -23, worst
    assert oracle.dexp(0.0) == 1.0
    assert oracle.dexp(-32.5) == 0.0


# ------------------------------------------------------- stage 2: threshold ---

def test_threshold_stops_expansion():
    V, k = 4, 2
    cfg = oracle.TreeCfg(batch=1, vocab=V, top_k=k, depth=3, node_budget=6, threshold=0.4)
    logits = np.full((1, 3, k, V), -30.0, np.float32)
    logits[0, 0, 0] = np.log([0.5, 0.3, 0.15, 0.05])
    logits[0, 1, 0] = np.log([0.9, 0.05, 0.03, 0.02])
    logits[0, 2, 0] = np.log([0.25, 0.25, 0.25, 0.25])
    t = oracle.Tree(cfg)
    tok0, cnt0 = t.expand(0, np.ascontiguousarray(logits[:, 0]))
    assert cnt0[0] == 1 and tok0[0, 0] == 0 and tok0[0, 1] == -1  # 0.3 < 0.4 is not expanded
    tok1, cnt1 = t.expand(1, np.ascontiguousarray(logits[:, 1]))
    assert cnt1[0] == 1 and tok1[0, 0] == 0  # 0.45 >= 0.4, 0.025 < 0.4
    vals = np.exp(t.logv[0, :k + k * k].astype(np.float64))
    np.testing.assert_allclose(vals[:2], [0.5, 0.3], rtol=1e-6)
    np.testing.assert_allclose(vals[2:4], [0.45, 0.025], rtol=1e-6)
    assert not t.valid[0, 4:6].any()  # frontier slot 1 of step 1 did not exist
    t.expand(2, np.ascontiguousarray(logits[:, 2]))
    t.rerank()
    # nodes below the threshold stay candidates for the rerank
    kept_vals = sorted(np.exp(t.logv[0][t.kept[0] == 1].astype(np.float64)), reverse=True)
    np.testing.assert_allclose(kept_vals[:3], [0.5, 0.45, 0.3], rtol=1e-6)


def test_figure_parameters_config():
    g = json.load(open(os.path.join(GOLDEN, "expand_rerank_params.json")))
    k, N, thr = g["top_k"], g["node_budget"], g["threshold"]
    cfg = oracle.TreeCfg(batch=16, vocab=64, top_k=k, depth=3, node_budget=N, threshold=thr)
    logits = synth.normal4((16, 3, k, 64), synth.F32, 2.5, seed=5, stream=synth.STREAM_DRAFT)
    t = oracle.Tree(cfg)
    for s in range(3):
        base = oracle.step_base(s, k)
        F = t.fcount.copy()
        t.expand(s, np.ascontiguousarray(logits[:, s]))
        for b in range(16):
            ids = np.arange(base, base + F[b] * k)
            v = t.logv[b, ids]
            elig = ids[v >= np.float32(math.log(thr))]
            order = elig[np.lexsort((elig, -t.logv[b, elig].astype(np.float64)))][:k]
            assert t.fcount[b] == len(order)
            assert list(t.fnode[b, :len(order)]) == list(order)
    t.rerank()
    tr = t.build_tree(np.zeros(16, np.int32), np.zeros(16, np.int32))
    assert (tr["n_tree"] <= N + 1).all()


# ---------------------------------------------------- stage 3: brute force ---

def _ancestor_closed(sub, parent):
    s = set(sub)
    return all(parent[i] < 0 or parent[i] in s for i in sub)


@pytest.mark.parametrize("k,D,N", [(2, 3, 3), (2, 3, 5), (3, 2, 4), (3, 2, 7), (2, 2, 2)])
def test_rerank_maximises_value_over_connected_subtrees(k, D, N):
    V = 16
    B = 12
    cfg = oracle.TreeCfg(batch=B, vocab=V, top_k=k, depth=D, node_budget=N)
    logits = synth.normal4((B, D, k, V), synth.F32, 1.7, seed=100 + k * 10 + D + N, stream=synth.STREAM_DRAFT)
    t, tr = _run_tree(cfg, logits)
    for b in range(B):
        valid = [i for i in range(cfg.C) if t.valid[b, i]]
        val = np.exp(t.logv[b].astype(np.float64))
        n = min(N, len(valid))
        best = -1.0
        best_set = None
        for sub in itertools.combinations(valid, n):
            if not _ancestor_closed(sub, t.parent[b]):
                continue
            s = float(sum(val[list(sub)]))
            if s > best:
                best, best_set = s, set(sub)
        kept = set(np.nonzero(t.kept[b])[0].tolist())
        assert _ancestor_closed(kept, t.parent[b])
        assert abs(sum(val[list(kept)]) - best) <= 1e-12 * best
        assert kept == best_set


def test_rerank_tie_keeps_shallower():
    # A child with confidence exactly 1 in fp32 (lp == 0) ties with its parent.
    V, k = 8, 1
    cfg = oracle.TreeCfg(batch=1, vocab=V, top_k=k, depth=2, node_budget=1)
    logits = np.full((1, 2, k, V), -200.0, np.float32)
    logits[0, 0, 0, 3] = 1.0
    logits[0, 0, 0, 4] = 0.5
    logits[0, 1, 0, 6] = 0.0
    t, tr = _run_tree(cfg, logits)
    assert t.logv[0, 0] == t.logv[0, 1]
    assert t.kept[0].tolist() == [1, 0]
    assert tr["tokens"][0, :2].tolist() == [0, 3]


# ----------------------------------------------------- stage 4: emission ---

def test_mask_positions_closed_form():
    B, V, k, D, N = 10, 32, 3, 4, 12
    cfg = oracle.TreeCfg(batch=B, vocab=V, top_k=k, depth=D, node_budget=N)
    logits = synth.normal4((B, D, k, V), synth.F32, 2.0, seed=9, stream=synth.STREAM_DRAFT)
    L = np.arange(B, dtype=np.int32) * 7 + 3
    t, tr = _run_tree(cfg, logits, prefix_len=L, root_token=np.arange(B, dtype=np.int32) + 100)
    for b in range(B):
        n = tr["n_tree"][b]
        assert n == 1 + t.n_kept[b]
        assert tr["tokens"][b, 0] == 100 + b
        for i in range(cfg.T):
            bits = {j for j in range(cfg.T) if tr["mask"][b, i, j // 32] >> (j % 32) & 1}
            if i >= n:
                assert not bits and tr["tokens"][b, i] == -1 and tr["parent"][b, i] == -1
                continue
            anc, j = {i}, i
            while tr["parent"][b, j] >= 0:
                assert tr["parent"][b, j] < j
                j = tr["parent"][b, j]
                anc.add(j)
            assert bits == anc
            assert tr["depth"][b, i] == len(anc) - 1
            assert tr["pos"][b, i] == L[b] + tr["depth"][b, i]
        ids = np.nonzero(t.kept[b])[0]
        assert list(tr["tokens"][b, 1:n]) == list(t.token[b, ids])  # id (BFS) order


# --------------------------------------------------- stage 5: attention ---

def _tiny_attention_case(dtype, B=2, T=9, Hq=4, Hkv=2, d=16, seed=21):
    V, k, D = 32, 2, 3
    cfg = oracle.TreeCfg(batch=B, vocab=V, top_k=k, depth=D, node_budget=T - 1)
    logits = synth.normal4((B, D, k, V), synth.F32, 2.0, seed=seed, stream=synth.STREAM_DRAFT)
    L = np.array([5, 12][:B], np.int32)
    _, tr = _run_tree(cfg, logits, prefix_len=L)
    Lmax = int(L.max()) + T
    q = synth.normal4((B, T, Hq, d), dtype, 1.0, seed=seed, stream=synth.STREAM_Q)
    npdt = np.float32 if dtype == synth.F32 else np.uint16
    kc = np.zeros((B, Lmax, Hkv, d), npdt)
    vc = np.zeros((B, Lmax, Hkv, d), npdt)
    for b in range(B):
        synth.kv_region(kc, dtype, b * Lmax * Hkv * d, Hkv * d, Hkv, d, 0, int(L[b]) + T, 0, b, seed, synth.STREAM_K)
        synth.kv_region(vc, dtype, b * Lmax * Hkv * d, Hkv * d, Hkv, d, 0, int(L[b]) + T, 0, b, seed, synth.STREAM_V)
    return tr, L, q, kc, vc, Lmax


def _widen(a, dtype):
    return a.astype(np.float64) if dtype == synth.F32 else synth.bf16_to_f32(a).astype(np.float64)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_tree_attention_equals_per_path_causal(dtype):
    B, T, Hq, Hkv, d = 2, 9, 4, 2, 16
    tr, L, q, kc, vc, Lmax = _tiny_attention_case(dtype, B, T, Hq, Hkv, d)
    out = oracle.attention(q, kc, vc, Lmax * Hkv * d, Hkv * d, L, tr["mask"], tr["n_tree"], Hkv)
    qf, kf, vf = _widen(q, dtype), _widen(kc, dtype), _widen(vc, dtype)
    for b in range(B):
        for i in range(T):
            if i >= tr["n_tree"][b]:
                assert not out[b, i].any()
                continue
            path, j = [], i
            while j >= 0:
                path.append(j)
                j = tr["parent"][b, j]
            seq_pos = list(range(L[b])) + [L[b] + s for s in reversed(path)]  # prefix ++ root..i
            for h in range(Hq):
                g = h // (Hq // Hkv)
                K = kf[b, seq_pos, g]
                Vv = vf[b, seq_pos, g]
                # causal attention of the last position of the sequence
                s = K @ qf[b, i, h] / math.sqrt(d)
                w = np.exp(s - s.max())
                want = (w / w.sum()) @ Vv
                np.testing.assert_allclose(out[b, i, h], want, rtol=1e-10, atol=1e-12)


def test_chain_tree_attention_is_causal_attention():
    # k = 1: the tree is a chain, the mask is lower-triangular; textbook causal attention.
    B, V, D, d, Hq = 1, 16, 5, 8, 2
    T = D + 1
    cfg = oracle.TreeCfg(batch=B, vocab=V, top_k=1, depth=D, node_budget=D)
    logits = synth.normal4((B, D, 1, V), synth.F32, 1.0, seed=2, stream=synth.STREAM_DRAFT)
    L = np.array([4], np.int32)
    _, tr = _run_tree(cfg, logits, prefix_len=L)
    S = int(L[0]) + T
    q = synth.normal4((B, T, Hq, d), synth.F32, 1.0, seed=2, stream=synth.STREAM_Q)
    kc = synth.normal4((B, S, Hq, d), synth.F32, 1.0, seed=2, stream=synth.STREAM_K)
    vc = synth.normal4((B, S, Hq, d), synth.F32, 1.0, seed=2, stream=synth.STREAM_V)
    out = oracle.attention(q, kc, vc, S * Hq * d, Hq * d, L, tr["mask"], tr["n_tree"], Hq)
    # full causal attention over S positions; queries are the last T positions
    for h in range(Hq):
        Qf = np.zeros((S, d))
        Qf[L[0]:] = q[0, :, h]
        scores = Qf @ kc[0, :, h].T.astype(np.float64) / math.sqrt(d)
        scores = np.where(np.tril(np.ones((S, S), bool)), scores, -np.inf)
        w = np.exp(scores - scores.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        want = w @ vc[0, :, h].astype(np.float64)
        np.testing.assert_allclose(out[0, :, h], want[L[0]:], rtol=1e-10, atol=1e-12)


# ------------------------------------------------------ stage 6: verify ---

def _tree_and_target(B, V, k, D, N, seed, plant_frac=0.8):
    cfg = oracle.TreeCfg(batch=B, vocab=V, top_k=k, depth=D, node_budget=N)
    logits = synth.normal4((B, D, k, V), synth.F32, 2.0, seed=seed, stream=synth.STREAM_DRAFT)
    _, tr = _run_tree(cfg, logits)
    T = cfg.T
    target = synth.normal4((B, T, V), synth.F32, 1.0, seed=seed, stream=synth.STREAM_TARGET)
    # make the target agree with some child of each slot so paths get accepted
    rng = np.random.default_rng(seed)
    for b in range(B):
        for t in range(tr["n_tree"][b]):
            kids = [c for c in range(T) if tr["parent"][b, c] == t]
            if kids and rng.random() < plant_frac:
                target[b, t, tr["tokens"][b, rng.choice(kids)]] = 50.0
    return cfg, tr, target


def test_greedy_verify_bruteforce():
    B, V, k, D, N = 24, 16, 3, 4, 10
    cfg, tr, target = _tree_and_target(B, V, k, D, N, seed=31)
    a, slots, toks, am = oracle.verify_greedy(target, tr["tokens"], tr["parent"], tr["n_tree"], D)
    assert (a > 0).any() and (a >= 2).any()
    for b in range(B):
        n = tr["n_tree"][b]
        g = [int(np.argmax(target[b, t])) for t in range(n)]
        path, cur = [0], 0
        while True:
            nxt = [c for c in range(n) if tr["parent"][b, c] == cur and tr["tokens"][b, c] == g[cur]]
            assert len(nxt) <= 1
            if not nxt:
                break
            cur = nxt[0]
            path.append(cur)
        assert a[b] == len(path) - 1
        assert list(slots[b, :a[b] + 1]) == path
        assert list(toks[b, :a[b] + 1]) == [tr["tokens"][b, s] for s in path[1:]] + [g[cur]]
        assert (slots[b, a[b] + 1:] == -1).all() and (toks[b, a[b] + 1:] == -1).all()


def test_greedy_chain_equals_chain_speculative_decoding():
    # k = 1 chain: accept draft token j while it equals the target's greedy choice at j-1.
    B, V, D = 40, 8, 5
    cfg, tr, target = _tree_and_target(B, V, 1, D, D, seed=7, plant_frac=0.7)
    a, _, toks, _ = oracle.verify_greedy(target, tr["tokens"], tr["parent"], tr["n_tree"], D)
    for b in range(B):
        draft = tr["tokens"][b, 1:tr["n_tree"][b]]
        tgt = target[b].argmax(axis=1)
        n_acc = 0
        while n_acc < len(draft) and draft[n_acc] == tgt[n_acc]:
            n_acc += 1
        assert a[b] == n_acc
        assert list(toks[b, :n_acc + 1]) == list(draft[:n_acc]) + [tgt[n_acc]]


def _softmax(x):
    x = x.astype(np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def test_lossless_single_child_accept_probability_is_p():
    # The proposal of a deterministic top-k child is a point mass, so min(1, p/q) = p(x).
    V, T = 8, 2
    row = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.0, 0.7, 0.1], np.float32)
    target = np.zeros((1, T, V), np.float32)
    target[0, 0] = row
    tokens = np.array([[0, 6]], np.int32)
    parent = np.array([[-1, 0]], np.int32)
    p = _softmax(row)[6]
    n = 4096
    U = np.zeros((n, T + 2), np.uint32)
    U[:, 1] = (np.arange(n, dtype=np.uint64) * (2 ** 32 // n)).astype(np.uint32)
    a, _, _ = oracle.verify_lossless(np.repeat(target, n, 0), np.repeat(tokens, n, 0), np.repeat(parent, n, 0),
                                     np.full(n, 2, np.int32), U, depth=1)
    assert abs(a.mean() - p) <= 1.0 / n + 1e-6


def test_lossless_output_distribution_equals_target():
    # Root with 3 kept children (two of them with kept children). The first two
    # emitted tokens must follow the target's own autoregressive distribution.
    V, T = 6, 6
    tokens = np.array([[9, 2, 0, 5, 1, 4]], np.int32)
    parent = np.array([[-1, 0, 0, 0, 1, 2]], np.int32)
    rows = np.array([[0.3, -0.2, 1.1, 0.0, -1.0, 0.6],
                     [1.5, 0.1, -0.3, 0.2, 0.9, -2.0],
                     [0.0, 0.4, 0.1, -0.5, 1.2, 0.3],
                     [0.2, 0.2, 0.2, 0.2, 0.2, 0.2],
                     [-1.0, 0.0, 1.0, 0.5, 0.5, 0.1],
                     [0.3, 0.1, 0.0, 2.0, -0.4, 0.2]], np.float32)
    n = 200000
    target = np.repeat(rows[None], n, 0)
    U = synth.words(n, T + 2, c2=0, seed=77)
    a, slots, toks = oracle.verify_lossless(target, np.repeat(tokens, n, 0), np.repeat(parent, n, 0),
                                            np.full(n, T, np.int32), U, depth=2)
    p0 = _softmax(rows[0])
    emp0 = np.bincount(toks[:, 0], minlength=V) / n
    sigma = np.sqrt(p0 * (1 - p0) / n)
    assert (np.abs(emp0 - p0) < 5 * sigma + 1e-9).all(), (emp0, p0)
    # joint of the first two tokens where the first lands on a tree node
    slot_of_tok = {int(tokens[0, c]): c for c in range(1, T) if parent[0, c] == 0}
    for x, c in slot_of_tok.items():
        pc = _softmax(rows[c])
        sel = toks[:, 0] == x
        emp = np.bincount(toks[sel, 1], minlength=V) / sel.sum()
        sig = np.sqrt(pc * (1 - pc) / sel.sum())
        assert (np.abs(emp - pc) < 5 * sig + 1e-9).all(), (x, emp, pc)
    assert (a <= 2).all() and (a >= 0).all()


def test_lossless_row_mass_is_exact_integer_sum():
    V, T = 300, 3
    target = synth.normal4((1, T, V), synth.BF16, 2.5, seed=4, stream=synth.STREAM_TARGET)
    U = synth.words(1, T + 2, c2=0, seed=4)
    tokens = np.array([[1, 2, 3]], np.int32)
    parent = np.array([[-1, 0, 0]], np.int32)
    _, _, _, rmax, rmass = oracle.verify_lossless(target, tokens, parent, np.array([T], np.int32), U, depth=1,
                                                  row_stats_out=True)
    for t in range(T):
        x = synth.bf16_to_f32(target[0, t])
        assert rmax[0, t] == x.max()
        want = sum(int(np.float32(oracle.dexp(float(np.float32(v - x.max())))) * np.float32(2.0 ** 40)) for v in x)
        assert int(rmass[0, t]) == want
        # and the integer masses follow softmax to fp32 precision
        assert abs(want / 2.0 ** 40 - np.exp(x.astype(np.float64) - x.max()).sum()) < 1e-5 * want / 2.0 ** 40


# ------------------------------------------------------ stage 6b: compact ---

def test_kv_compact_moves_path_kv():
    B, layers, Hkv, d, Lmax, D = 3, 2, 2, 8, 40, 4
    L = np.array([5, 17, 0], np.int32)
    a = np.array([3, 0, 4], np.int32)
    slots = np.array([[0, 2, 5, 7, -1], [0, -1, -1, -1, -1], [0, 1, 3, 4, 8]], np.int32)
    pos_stride = Hkv * d
    kv_stride = Lmax * pos_stride
    layer_stride = 2 * kv_stride
    seq_stride = layers * layer_stride
    cache = np.zeros(B * seq_stride, np.uint16)
    for b in range(B):
        for l in range(layers):
            for kv in range(2):
                synth.kv_region(cache, synth.BF16, b * seq_stride + l * layer_stride + kv * kv_stride, pos_stride,
                                Hkv, d, 0, Lmax, l, b, 13, synth.STREAM_K + kv)
    before = cache.copy()
    new_len = oracle.kv_compact(cache, B, layers, Hkv, d, seq_stride, layer_stride, kv_stride, pos_stride, L, a,
                                slots)
    assert list(new_len) == list(L + a + 1)
    c4 = cache.reshape(B, layers, 2, Lmax, Hkv, d)
    b4 = before.reshape(B, layers, 2, Lmax, Hkv, d)
    for b in range(B):
        for l in range(layers):
            for kv in range(2):
                # destination L+j holds what the generator wrote for position L+s_j
                for j in range(1, a[b] + 1):
                    regen = np.zeros(Lmax * pos_stride, np.uint16)
                    synth.kv_region(regen, synth.BF16, 0, pos_stride, Hkv, d, L[b] + slots[b, j],
                                    L[b] + slots[b, j] + 1, l, b, 13, synth.STREAM_K + kv)
                    want = regen.reshape(Lmax, Hkv, d)[L[b] + slots[b, j]]
                    assert (c4[b, l, kv, L[b] + j] == want).all()
                # everything else is untouched
                others = [p for p in range(Lmax) if not (L[b] + 1 <= p <= L[b] + a[b])]
                assert (c4[b, l, kv, others] == b4[b, l, kv, others]).all()


# ------------------------------------------------- ablation policies (§5.2) ---

def _rows(*probs, V=8):
    """fp32 logit rows log(p) padded with equal small mass (sums to 1)."""
    out = []
    for p in probs:
        rest = (1.0 - sum(p)) / (V - len(p))
        out.append(np.log(np.array(list(p) + [rest] * (V - len(p)), np.float64)).astype(np.float32))
    return np.array(out, np.float32)


def _landscape():
    """Hand-built k = 2, D = 3 landscape (values by hand):
    root -> A 0.69, B 0.30; A -> A1 .5, A2 .44; B -> B1 .95, B2 .04;
    A1 -> A1a .9; A2 -> A2a .9. Node ids: A 0, B 1, A1 2, A2 3, B1 4, B2 5,
    A1a 6, A1b 7, A2a 8, A2b 9."""
    s0 = np.zeros((1, 2, 8), np.float32)
    s0[0, 0] = _rows((0.69, 0.30))[0]
    s1 = _rows((0.5, 0.44), (0.95, 0.04))[None]
    s2 = _rows((0.9, 0.09), (0.9, 0.09))[None]
    return [s0, s1, s2]


def _run(policy, N, steps):
    t = oracle.Tree(oracle.TreeCfg(1, 8, 2, 3, N, 0.0, policy))
    fronts = [t.expand(s, logits) for s, logits in enumerate(steps)]
    t.rerank()
    return t, fronts


def test_confidence_expansion_ranks_the_frontier_by_own_confidence():
    # value-based: A1 (.345) and A2 (.3036) lead depth 2; confidence-based:
    # B1 (.95) and A1 (.5) lead, although B1's value (.285) is lower
    steps = _landscape()[:2]
    tv, fv = _run(0, 6, steps)
    tc, fc = _run(1, 6, steps)
    assert list(tv.fhist[2, 0]) == [2, 3]
    assert list(tc.fhist[2, 0]) == [4, 2]
    assert list(fc[1][0][0]) == [0, 0]  # B1 and A1 are both token 0 of their rows
    # the threshold and the values themselves do not depend on the policy
    assert np.array_equal(tv.logv, tc.logv)


def test_without_rerank_keeps_the_expanded_nodes():
    steps = _landscape()
    t2, _ = _run(2, 6, steps)
    t0, _ = _run(0, 6, steps)
    kept2 = set(np.flatnonzero(t2.kept[0]))
    kept0 = set(np.flatnonzero(t0.kept[0]))
    assert kept2 == {0, 1, 2, 3, 6, 8}  # the frontier of every step (k per depth)
    assert kept0 == {0, 1, 2, 3, 4, 6}  # top-6 by value: B1 (.285) beats A2a (.2732)
    # reranking improves the expected acceptance length [EAGLE-2 summary 5.2.2]
    v0, v2 = t0.value_sum(0), t2.value_sum(0)
    assert abs(v0 - (0.69 + 0.345 + 0.3036 + 0.30 + 0.3105 + 0.285)) < 1e-3
    assert abs(v2 - (0.69 + 0.30 + 0.345 + 0.3036 + 0.3105 + 0.27324)) < 1e-3
    assert v0 > v2


def test_rerank_value_never_below_expansion_only_tree():
    # rerank keeps the N most valuable candidates, a connected set; the nodes
    # of the expansion phase are one of the connected sets it chooses among
    for seed in range(6):
        B, V, k, D, N = 3, 64, 3, 4, 9
        logits = synth.normal4((D, B, k, V), synth.F32, 2.5, seed=seed, stream=synth.STREAM_DRAFT)
        t0 = oracle.Tree(oracle.TreeCfg(B, V, k, D, N, 0.0, 0))
        t2 = oracle.Tree(oracle.TreeCfg(B, V, k, D, N, 0.0, 2))
        for s in range(D):
            t0.expand(s, logits[s])
            t2.expand(s, logits[s])
        t0.rerank()
        t2.rerank()
        for b in range(B):
            assert t0.value_sum(b) >= t2.value_sum(b) - 1e-9
            # the expansion-only tree is connected: every kept node's parent is kept or the root
            kept = np.flatnonzero(t2.kept[b])
            assert all(t2.parent[b, i] < 0 or t2.kept[b, t2.parent[b, i]] for i in kept)


def test_static_shape_is_the_same_for_every_landscape():
    # policy 3: frontier by position (f + r, then id), kept = the frontiers,
    # first N by depth then id. k = 3, D = 3, N = 9: step 1 frontier {0, 1, 2};
    # step 2 children 3 + 3f + r, positions (0,0) (0,1) (1,0) -> {3, 4, 6};
    # step 3 children 12 + 3f + r -> {12, 13, 15}.
    B, V, k, D, N = 2, 64, 3, 3, 9
    shapes = []
    for seed, sharp in [(0, 2.5), (1, 0.8), (5, 4.0)]:
        logits = synth.normal4((D, B, k, V), synth.F32, sharp, seed=seed, stream=synth.STREAM_DRAFT)
        t = oracle.Tree(oracle.TreeCfg(B, V, k, D, N, 0.0, 3))
        for s in range(D):
            t.expand(s, logits[s])
        t.rerank()
        assert [list(t.fhist[s, 0]) for s in (1, 2, 3)] == [[0, 1, 2], [3, 4, 6], [12, 13, 15]]
        for b in range(B):
            kept = np.flatnonzero(t.kept[b])
            assert list(kept) == [0, 1, 2, 3, 4, 6, 12, 13, 15]
            shapes.append(tuple(int(t.parent[b, i]) for i in kept))
    assert len(set(shapes)) == 1
    assert shapes[0] == (-1, -1, -1, 0, 0, 1, 3, 3, 4)


def test_dynamic_tree_gains_over_static_shape_on_sharp_landscapes():
    # the tutorial's widget: on a sharp landscape the dynamic tree commits to
    # deep chains and its summed path value (expected accepted tokens) exceeds
    # the static shape's; on a flat one the two come close
    def mean_values(sharp):
        B, V, k, D, N = 8, 256, 4, 5, 16
        vs = {0: [], 3: []}
        for seed in range(4):
            logits = synth.normal4((D, B, k, V), synth.F32, sharp, seed=seed, stream=synth.STREAM_DRAFT)
            for pol in (0, 3):
                t = oracle.Tree(oracle.TreeCfg(B, V, k, D, N, 0.0, pol))
                for s in range(D):
                    t.expand(s, logits[s])
                t.rerank()
                vs[pol] += [t.value_sum(b) for b in range(B)]
        return np.mean(vs[0]), np.mean(vs[3])
    d_sharp, s_sharp = mean_values(4.0)
    d_flat, s_flat = mean_values(0.8)
    assert d_sharp > 1.08 * s_sharp  # 1.67 vs 1.49 at these seeds
    assert d_flat >= s_flat
    assert (d_flat - s_flat) / s_flat < (d_sharp - s_sharp) / s_sharp


# ------------------------------------------------- LM-head logits (f1) ---
# The draft reuses the target's LM head ("EAGLE" notes, EAGLE 方法): logits of a
# frontier row are its hidden state times the head's weight rows.

def _lmhead_case(M, V, H, seed):
    h = synth.normal4((M, H), synth.BF16, 1.0, seed, synth.STREAM_HIDDEN)
    W = synth.normal4((V, H), synth.BF16, 0.05, seed, synth.STREAM_LMHEAD)
    return h, W


def _f32_ulp(x):
    x = np.abs(x.astype(np.float32))
    return np.spacing(x).astype(np.float64)


def test_lmhead_one_hot_rows_select_weight_columns():
    # hidden row m = c_m * e_{h_m} with c_m a power of two: logits row m is
    # exactly c_m * W[:, h_m] (one exact product per entry)
    M, V, H = 6, 37, 24
    _, W = _lmhead_case(M, V, H, 3)
    h = np.zeros((M, H), np.uint16)
    cols = [0, 5, 23, 11, 5, 17]
    scales = [1.0, 2.0, 0.5, -4.0, 0.125, 1.0]
    for m, (c, s) in enumerate(zip(cols, scales)):
        h[m, c] = np.array([s], np.float32).view(np.uint32)[0] >> 16
    got = oracle.lmhead_logits(h, W)
    Wf = synth.bf16_to_f32(W)
    for m, (c, s) in enumerate(zip(cols, scales)):
        assert np.array_equal(got[m], (Wf[:, c] * np.float32(s)).astype(np.float32))


def test_lmhead_matches_float64_matmul():
    # non-square M, V, H so that a transposed operand cannot pass; the double
    # sums differ from numpy's only in summation order, far below fp32 ulp
    M, V, H = 5, 203, 96
    h, W = _lmhead_case(M, V, H, 7)
    got = oracle.lmhead_logits(h, W)
    ref = synth.bf16_to_f32(h).astype(np.float64) @ synth.bf16_to_f32(W).astype(np.float64).T
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= 0.5 * _f32_ulp(ref) + 1e-30)
    assert np.mean(got == ref.astype(np.float32)) > 0.99


def test_lmhead_linear_and_order_free():
    M, V, H = 4, 64, 48
    h, W = _lmhead_case(M, V, H, 11)
    base = oracle.lmhead_logits(h, W)
    # doubling (exponent + 1) and negation (sign bit) are exact on bf16 inputs
    h2 = (synth.bf16_to_f32(h) * 2).view(np.uint32) >> 16
    assert np.array_equal(oracle.lmhead_logits(h2.astype(np.uint16), W), 2 * base)
    hn = h ^ np.uint16(0x8000)
    assert np.array_equal(oracle.lmhead_logits(hn, W), -base)
    # permuting the hidden dimension of both operands leaves each sum within rounding
    perm = np.random.default_rng(0).permutation(H)
    pp = oracle.lmhead_logits(np.ascontiguousarray(h[:, perm]), np.ascontiguousarray(W[:, perm]))
    assert np.all(np.abs(pp.astype(np.float64) - base) <= _f32_ulp(base) + 1e-30)
    # one weight row zeroed: that vocabulary column becomes 0, the others stay
    Wz = W.copy()
    Wz[9] = 0
    z = oracle.lmhead_logits(h, Wz)
    assert np.all(z[:, 9] == 0) and np.array_equal(np.delete(z, 9, 1), np.delete(base, 9, 1))


# ------------------------------------- which verification rule is lossless ---
# Exact enumeration on one node with two sampled children (no Monte Carlo):
# children c1, c2 drawn from the draft distribution q without replacement
# (sequential draws), first emitted token under three tree/verify choices.

def _draws_without_replacement(q):
    V = len(q)
    for a in range(V):
        for b in range(V):
            if a != b:
                yield a, b, q[a] * q[b] / (1.0 - q[a])


def _residual(p, q):
    r = np.maximum(p - q, 0.0)
    return r / r.sum()


def _draft_rule_tests(p, q, children):
    """Emitted-token distribution of min(1, p/q) tests along `children` (the
    draft distribution loses each rejected child; the target becomes the
    residual), then a draw from the last residual."""
    out = np.zeros_like(p)
    stay = 1.0
    p_cur, q_cur = p.copy(), q.copy()
    for x in children:
        acc = min(1.0, p_cur[x] / q_cur[x])
        out[x] += stay * acc
        stay *= 1.0 - acc
        p_cur = _residual(p_cur, q_cur)
        q_cur = q_cur.copy()
        q_cur[x] = 0.0
        q_cur /= q_cur.sum()
    return out + stay * p_cur


def _onehot_rule_tests(p, children):
    """Emitted-token distribution of the built rule: accept x with p_cur(x),
    on rejection remove x from the target and renormalise."""
    out = np.zeros_like(p)
    stay = 1.0
    p_cur = p.copy()
    for x in children:
        out[x] += stay * p_cur[x]
        stay *= 1.0 - p_cur[x]
        p_cur = p_cur.copy()
        p_cur[x] = 0.0
        p_cur /= p_cur.sum()
    return out + stay * p_cur


def test_draft_rule_lossless_only_for_token_independent_shapes():
    p = np.array([0.1, 0.45, 0.3, 0.15])
    q = np.array([0.5, 0.2, 0.2, 0.1])
    both = np.zeros(4)      # every sampled child tested, in sampling order
    by_value = np.zeros(4)  # only the child of higher draft probability kept (a value-ranked budget of one)
    onehot = np.zeros(4)    # the same value-ranked child under the built rule
    for a, b, w in _draws_without_replacement(q):
        keep = a if (q[a], -a) > (q[b], -b) else b
        both += w * _draft_rule_tests(p, q, [a, b])
        by_value += w * _draft_rule_tests(p, q, [keep])
        onehot += w * _onehot_rule_tests(p, [keep])
    assert np.allclose(both, p, atol=1e-12)
    assert np.allclose(onehot, p, atol=1e-12)
    # the draft-probability rule on a value-selected child is biased
    assert np.abs(by_value - p).max() > 0.02


def test_lmhead_parity_bound_catches_planted_mistakes():
    """The GPU parity bound for the LM head (H * 2^-23 * sum_h |h w| plus half a
    bf16 ulp) is tight enough to flag the mistakes a tiled kernel could make:
    a dropped 64-wide hidden block, a block counted twice, a neighbouring
    vocabulary row, or operands read transposed. Mistakes are planted in
    copies of the inputs fed to the oracle."""
    M, V, Hd = 6, 300, 256
    h, W = _lmhead_case(M, V, Hd, 13)
    ref = oracle.lmhead_logits(h, W).astype(np.float64)
    a = np.abs(synth.bf16_to_f32(h)).astype(np.float64)
    b = np.abs(synth.bf16_to_f32(W)).astype(np.float64)
    tol = Hd * 2.0 ** -23 * (a @ b.T)
    tol = tol + 2.0 ** -8 * (np.abs(ref) + tol)

    def flagged(got):
        return bool(np.any(np.abs(got.astype(np.float64) - ref) > tol))

    assert not flagged(ref)
    dropped = h.copy()
    dropped[:, 64:128] = 0
    assert flagged(oracle.lmhead_logits(dropped, W))
    twice = np.concatenate([h, h[:, 128:192]], axis=1)
    assert flagged(oracle.lmhead_logits(twice, np.concatenate([W, W[:, 128:192]], axis=1)))
    assert flagged(oracle.lmhead_logits(h, np.roll(W, 1, axis=0)))
    Wt = np.ascontiguousarray(W.reshape(-1)[: V * Hd].reshape(Hd, V).T)  # the weight read as [H, V]
    assert flagged(oracle.lmhead_logits(h, Wt))


# ------------------------------------------- sampled drafting (next row f4) ---

def test_dlog_within_three_ulp_of_log():
    rng = np.random.default_rng(0)
    y = np.exp2(rng.uniform(-24, 12, 100000)).astype(np.float32)
    near_one = (1 + rng.uniform(-0.01, 0.01, 50000)).astype(np.float32)
    edges = np.float32([2.0, 0.5, 1 + 2 ** -23, 1 - 2 ** -24, 2 ** -24, 1.4142135, 1.4142137, 0.70710677, 4096.0])
    y = np.concatenate([y, near_one, edges])
    got = oracle.dlog(y).astype(np.float64)
    ref = np.log(y.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 3 * ulp)
    assert oracle.dlog(np.float32([1.0]))[0] == 0.0


def test_gumbel_noise_quantiles():
    # g = -ln(-ln u): P(g <= t) = exp(-exp(-t)); u is the word's top 23 bits + 1/2
    w = np.arange(0, 1 << 32, 1 << 12, dtype=np.uint64).astype(np.uint32)  # 2^20 evenly spaced words
    g = oracle.gumbel(w).astype(np.float64)
    for t in (-1.5, -0.5, 0.0, 0.5, 1.0, 2.0, 4.0):
        assert abs(np.mean(g <= t) - math.exp(-math.exp(-t))) < 1e-5
    assert np.all(np.diff(g) >= 0)  # monotone in the word


def _chi2_sf(counts, probs):
    from scipy.stats import chi2
    n = counts.sum()
    exp = n * probs
    stat = float(((counts - exp) ** 2 / exp).sum())
    return chi2.sf(stat, len(probs) - 1)


def test_gumbel_topk_draws_without_replacement():
    """Children of a row drawn by the oracle's sampled expansion: the first is
    distributed as q = softmax(row), the ordered pair as q(a) q(b) / (1 - q(a))."""
    V, k, B = 5, 2, 60000
    x = np.array([1.2, 0.3, -0.5, 0.9, -1.4], np.float32)
    q = np.exp(x.astype(np.float64) - x.max())
    q /= q.sum()
    logits = np.ascontiguousarray(np.broadcast_to(x, (B, k, V)))
    words = synth.words(B, k * V, 0, 31, synth.STREAM_GUMBEL).reshape(B, k, V)
    t = oracle.Tree(oracle.TreeCfg(B, V, k, 1, k, 0.0, 0))
    t.expand(0, logits, words=words)
    first, second = t.token[:, 0], t.token[:, 1]
    assert np.all(first != second)
    assert _chi2_sf(np.bincount(first, minlength=V).astype(float), q) > 1e-4
    pair = np.zeros((V, V))
    np.add.at(pair, (first, second), 1.0)
    probs = np.array([[q[a] * q[b] / (1 - q[a]) if a != b else 0.0 for b in range(V)] for a in range(V)])
    m = probs > 0
    assert _chi2_sf(pair[m], probs[m]) > 1e-4
    # the values stay the unperturbed log-probabilities
    lse = np.log(np.exp(x.astype(np.float64)).sum())
    assert np.allclose(t.lp[:, 0], x[first] - lse, atol=1e-6)


def _sampled_tree_first_tokens(policy, N, xp, xq, B, seed, draft_equals_target=False, both=False):
    """One sampled-drafting cycle per sequence (k 2, depth 2, V 6) verified with
    the draft-probability rule; returns (first emitted tokens, accept lengths)
    (with both=True, all emitted tokens instead of the first)."""
    V, k, D = xp.shape[-1], 2, 2
    cfg = oracle.TreeCfg(B, V, k, D, N, 0.0, policy)
    draft = np.empty((D, B, k, V), np.float32)
    draft[0] = xq[0]
    draft[1] = xq[1]
    t = oracle.Tree(cfg)
    for s in range(D):
        w = synth.words(B, k * V, s, seed, synth.STREAM_GUMBEL).reshape(B, k, V)
        t.expand(s, np.ascontiguousarray(draft[s]), words=w)
    t.rerank()
    tr = t.build_tree(np.zeros(B, np.int32), np.zeros(B, np.int32))
    T = cfg.T
    target = np.empty((B, T, V), np.float32)
    target[:, 0] = xp[0]
    target[:, 1:] = xp[1]
    rows = t.draft_rows(tr["slot_of"], tr["n_tree"])
    uni = synth.words(B, T + 2, 0, seed, synth.STREAM_VERIFY)
    if draft_equals_target:  # every node's draft row is its own target row
        flat = np.empty((D * B * k, V), np.float32)
        flat[:] = xp[1]
        flat[rows[:, 0]] = xp[0]
    else:
        flat = draft.reshape(D * B * k, V)
    a, _, toks = oracle.verify_draft(target, flat, rows, tr["tokens"], tr["parent"], tr["n_tree"], uni, D)
    return (toks if both else toks[:, 0]), a


XP = np.array([[0.2, 1.5, 1.1, 0.4, -0.3, 0.9], [0.5, -0.2, 1.0, 0.1, 0.7, -1.0]], np.float32)
XQ = np.array([[1.4, 0.2, 0.9, 1.0, -0.8, 0.3], [-0.4, 0.6, 0.8, 1.1, 0.0, 0.2]], np.float32)


def _softmax64(x):
    e = np.exp(x.astype(np.float64) - x.max())
    return e / e.sum()


def test_draft_rule_with_drawn_children_is_lossless_on_a_static_tree():
    toks, a = _sampled_tree_first_tokens(3, 6, XP, XQ, B=40000, seed=5, both=True)
    assert _chi2_sf(np.bincount(toks[:, 0], minlength=6).astype(float), _softmax64(XP[0])) > 1e-4
    # after an accepted first-level child, the next token follows that child's target row
    moved = a >= 1
    assert 0.2 < moved.mean() < 0.95  # both accepts and rejections are exercised
    assert _chi2_sf(np.bincount(toks[moved, 1], minlength=6).astype(float), _softmax64(XP[1])) > 1e-4


def test_draft_rule_on_a_value_ranked_tree_is_biased():
    # budget 1: the rerank keeps the drawn first-level child of higher draft value
    first, _ = _sampled_tree_first_tokens(0, 1, XP, XQ, B=40000, seed=6)
    assert _chi2_sf(np.bincount(first, minlength=6).astype(float), _softmax64(XP[0])) < 1e-9


def test_draft_rule_accepts_every_first_child_when_draft_equals_target():
    _, a = _sampled_tree_first_tokens(3, 6, XP, XQ, B=2000, seed=7, draft_equals_target=True)
    assert np.all(a == 2)

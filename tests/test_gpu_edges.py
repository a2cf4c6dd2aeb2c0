"""Edge cases of the CUDA cycle against the oracle, and device status codes.

Degenerate and boundary inputs: a threshold that empties the frontier, odd
vocabulary sizes whose rows split unevenly over a cluster, k = 1 and the
maximum k = 16, one draft step, a budget of one node and the largest tree
(T = 256, eight mask words), rows of equal logits (every element ties at the
top), verification of a root-only tree and of a chain accepted to full
depth, compaction of zero and of the maximum number of tokens. Device-side
faults (a NaN row, a token out of range, an accept length past the limit)
are reported through the status word without touching memory out of range.
"""
import numpy as np
import pytest

import oracle
import synth

import harness as H

pytestmark = pytest.mark.gpu


def _E():
    from speculative_decoding_dynamic_gb300 import eagle as E
    return E


def _tables(E, cfg, ws):
    import torch
    B, C = cfg.batch, cfg.C
    t = {k: torch.empty(B, C, dtype=dt, device="cuda") for k, dt in
         [("token", torch.int32), ("parent", torch.int32), ("depth", torch.int32), ("logv", torch.float32),
          ("valid", torch.uint8), ("kept", torch.uint8)]}
    E.eagle_tree_export(cfg, ws, t["token"], t["parent"], t["depth"], t["logv"], t["valid"], t["kept"])
    torch.cuda.synchronize()
    return {k: H.to_host(v) for k, v in t.items()}


def _run_tree(logits, B, V, k, D, N, thr, dtype, L=None, root=None, policy=0):
    """Stages 1-4 on both sides with identical log-prob inputs (the oracle's lse)."""
    import torch
    E = _E()
    cfg_o = oracle.TreeCfg(B, V, k, D, N, thr, policy)
    t = oracle.Tree(cfg_o)
    fronts = []
    for s in range(D):
        fronts.append(t.expand(s, logits[s]))
    t.rerank()
    L = np.zeros(B, np.int32) if L is None else L
    root = np.zeros(B, np.int32) if root is None else root
    tr = t.build_tree(L, root)
    lse = np.zeros((D, B, k), np.float32)
    for s in range(D):
        for b in range(B):
            for f in range(k):
                _, lse[s, b, f], _ = oracle.row_stats(np.ascontiguousarray(logits[s, b, f]), 1)
    cfg = E.TreeCfg(B, V, k, D, N, thr, dtype, policy)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    dl, dlse = H.to_dev(logits), H.to_dev(lse)
    E.eagle_tree_init(cfg, ws)
    for s in range(D):
        E.eagle_expand(cfg, ws, s, dl[s], dlse[s], row_lse, ftok, fcnt)
        torch.cuda.synchronize()
        assert (H.to_host(fcnt) == fronts[s][1]).all(), f"frontier count step {s}"
        assert (H.to_host(ftok) == fronts[s][0]).all(), f"frontier tokens step {s}"
    E.eagle_rerank(cfg, ws)
    T, W = cfg.T, cfg.W
    out = {n: torch.empty(B, T, **i32) for n in ("tokens", "parent", "depth", "pos")}
    mask = torch.empty(B, T, W, **i32)
    n_tree = torch.empty(B, **i32)
    E.eagle_build_tree(cfg, ws, H.to_dev(L), H.to_dev(root), out["tokens"], out["parent"], out["depth"], out["pos"],
                       mask, n_tree)
    torch.cuda.synchronize()
    g = _tables(E, cfg, ws)
    v = t.valid.astype(bool)
    assert (g["valid"] == t.valid).all()
    assert (g["token"][v] == t.token[v]).all() and (g["parent"][v] == t.parent[v]).all()
    assert H.isclose_bits(g["logv"][v], t.logv[v])
    assert (g["kept"] == t.kept).all()
    for key in ("tokens", "parent", "depth", "pos"):
        assert (H.to_host(out[key]) == tr[key]).all(), key
    assert (H.to_host(mask).view(np.uint32) == tr["mask"]).all()
    assert (H.to_host(n_tree) == tr["n_tree"]).all()
    assert E.eagle_status_fetch(ws) == 0
    return t, tr


@pytest.mark.parametrize("B,V,k,D,N,thr,dtype", [
    (2, 1000, 2, 3, 8, 0.95, synth.F32),        # threshold empties the frontier after step 0
    (3, 4104, 3, 4, 20, 0.0, synth.BF16),       # odd vocabulary: uneven chunks
    (2, 40000, 5, 3, 30, 0.0, synth.BF16),      # several CTAs per row, ragged last chunk
    (1, 128256, 1, 5, 5, 0.0, synth.BF16),      # k = 1: a chain
    (2, 2048, 16, 4, 255, 0.0, synth.F32),      # k = 16, T = 256: eight mask words
    (4, 1032, 4, 1, 1, 0.0, synth.BF16),        # one step, one node
    (2, 32000, 10, 6, 60, 0.3, synth.BF16),     # threshold prunes part of every layer
])
def test_tree_edges(B, V, k, D, N, thr, dtype):
    logits = synth.normal4((D, B, k, V), dtype, 2.5, seed=V + k, stream=synth.STREAM_DRAFT)
    synth.plant(logits, dtype, float(np.log(9.0 * V)) + 3.0, seed=V + k, stream=synth.STREAM_DRAFT, frac=0.7)
    t, tr = _run_tree(logits, B, V, k, D, N, thr, dtype)
    if thr > 0.9:
        assert (t.fcount == 0).all() or (tr["n_tree"] <= 1 + k).all()


@pytest.mark.parametrize("policy", [1, 2, 3])
@pytest.mark.parametrize("B,V,k,D,N,thr,dtype", [
    (2, 1000, 2, 3, 8, 0.95, synth.F32),        # threshold empties the frontier after step 0
    (1, 128256, 1, 5, 5, 0.0, synth.BF16),      # k = 1: a chain
    (2, 2048, 16, 4, 255, 0.0, synth.F32),      # k = 16, T = 256
    (2, 32000, 10, 6, 60, 0.3, synth.BF16),     # threshold prunes part of every layer
    (3, 4104, 3, 4, 5, 0.0, synth.BF16),        # budget below the expanded nodes
])
def test_policy_edges(B, V, k, D, N, thr, dtype, policy):
    """The ablation policies (confidence frontier, no rerank, static shape)
    on the same degenerate inputs: bit-exact tables, kept sets and trees."""
    logits = synth.normal4((D, B, k, V), dtype, 2.5, seed=V + k + policy, stream=synth.STREAM_DRAFT)
    synth.plant(logits, dtype, float(np.log(9.0 * V)) + 3.0, seed=V + k, stream=synth.STREAM_DRAFT, frac=0.7)
    t, tr = _run_tree(logits, B, V, k, D, N, thr, dtype, policy=policy)
    kept = t.kept.astype(bool)
    assert (t.n_kept <= N).all() and (kept.sum(1) == t.n_kept).all()
    if policy in (2, 3):  # only expanded nodes (frontiers) can be kept
        for b in range(B):
            fr = set(int(x) for x in t.fhist[1:, b].ravel() if x >= 0)
            assert set(np.flatnonzero(kept[b])) <= fr


def test_equal_logit_rows_use_exact_fallback():
    # every element of some rows is equal: all elements tie at the top
    B, V, k, D, N = 2, 8192, 10, 2, 12
    logits = synth.normal4((D, B, k, V), synth.BF16, 1.0, seed=3, stream=synth.STREAM_DRAFT)
    logits[0, 0, 0, :] = logits[0, 0, 0, 0]
    logits[1, 1, :, :] = logits[1, 1, 0, 0]
    logits[1, 0, 3, 100:4000] = 0x4120  # bf16 10.0 on a wide range
    _run_tree(logits, B, V, k, D, N, 0.0, synth.BF16)


def _verify_both(target, tokens, parent, n_tree, depth, mode, seed=0, cycle=0):
    import torch
    E = _E()
    B, T, V = target.shape
    cfg = E.TreeCfg(B, V, 2, depth, T - 1, 0.0, synth.BF16 if target.dtype == np.uint16 else synth.F32)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    a, sl, tk = torch.empty(B, **i32), torch.empty(B, depth + 1, **i32), torch.empty(B, depth + 1, **i32)
    E.eagle_verify(cfg, ws, mode, 1.0, seed, cycle, H.to_dev(target), H.to_dev(tokens), H.to_dev(parent),
                   H.to_dev(n_tree), a, sl, tk)
    torch.cuda.synchronize()
    if mode == E.GREEDY:
        ra, rs, rt, _ = oracle.verify_greedy(target, tokens, parent, n_tree, depth)
    else:
        uniforms = synth.words(B, T + 2, cycle, seed=seed, stream=synth.STREAM_VERIFY)
        ra, rs, rt = oracle.verify_lossless(target, tokens, parent, n_tree, uniforms, depth)
    assert (H.to_host(a) == ra).all() and (H.to_host(sl) == rs).all() and (H.to_host(tk) == rt).all()
    assert E.eagle_status_fetch(ws) == 0
    return ra


@pytest.mark.parametrize("mode", [0, 1])
def test_verify_root_only_and_full_chain(mode):
    V, D = 4096, 5
    T = D + 1
    target = synth.normal4((2, T, V), synth.BF16, 2.0, seed=5, stream=synth.STREAM_TARGET)
    tokens = np.full((2, T), -1, np.int32)
    parent = np.full((2, T), -1, np.int32)
    tokens[:, 0] = 7
    # sequence 0: root only; sequence 1: a chain root -> 1 -> ... -> D whose tokens
    # the target prefers overwhelmingly, so it is accepted to full depth
    n_tree = np.array([1, T], np.int32)
    for c in range(1, T):
        tokens[1, c] = 100 + c
        parent[1, c] = c - 1
        target[1, c - 1, 100 + c] = np.float32(60.0).view(np.uint32) >> 16
    a = _verify_both(target, tokens, parent, n_tree, D, mode, seed=9, cycle=0)
    assert a[0] == 0 and a[1] == D


@pytest.mark.parametrize("a_max", [0, 6])
def test_compact_zero_and_full(a_max):
    import torch
    E = _E()
    B, layers, Hkv, d, Lmax, D = 3, 3, 2, 64, 96, 6
    pos_stride = Hkv * d
    kv_stride = Lmax * pos_stride
    layer_stride = 2 * kv_stride
    seq_stride = layers * layer_stride
    cache = np.zeros(B * seq_stride, np.uint16)
    for b in range(B):
        for l in range(layers):
            for kv in range(2):
                synth.kv_region(cache, synth.BF16, b * seq_stride + l * layer_stride + kv * kv_stride, pos_stride, Hkv,
                                d, 0, Lmax, l, b, 4, synth.STREAM_K + kv)
    L = np.array([10, 0, 50], np.int32)
    a = np.full(B, a_max, np.int32)
    stride = D + 3
    slots = np.full((B, stride), -1, np.int32)
    for b in range(B):
        slots[b, 0] = 0
        for j in range(1, a_max + 1):
            slots[b, j] = j + (j // 2) + b  # increasing, s_j >= j, sources overlap destinations
    ref = cache.copy()
    want_len = oracle.kv_compact(ref, B, layers, Hkv, d, seq_stride, layer_stride, kv_stride, pos_stride, L, a, slots)
    kv = E.KvCfg(B, 4, Hkv, d, layers, Lmax, synth.BF16, seq_stride, layer_stride, kv_stride, pos_stride)
    dc = H.to_dev(cache)
    nl = torch.empty(B, dtype=torch.int32, device="cuda")
    E.eagle_kv_compact(kv, dc, H.to_dev(L), H.to_dev(a), H.to_dev(slots), stride, nl)
    torch.cuda.synchronize()
    assert (H.to_host(dc) == ref).all()
    assert (H.to_host(nl) == want_len).all()


# ------------------------------------------------------- device status ---

def test_status_nonfinite_row():
    import torch
    E = _E()
    B, V, k, D, N = 1, 2048, 4, 2, 6
    cfg = E.TreeCfg(B, V, k, D, N, 0.0, synth.F32)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    logits = synth.normal4((D, B, k, V), synth.F32, 1.0, seed=1, stream=synth.STREAM_DRAFT)
    logits[0, 0, 0, 77] = np.nan
    dl = H.to_dev(logits)
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, dtype=torch.int32, device="cuda"), torch.empty(B, dtype=torch.int32, device="cuda")
    E.eagle_tree_init(cfg, ws)
    E.eagle_expand(cfg, ws, 0, dl[0], None, row_lse, ftok, fcnt)
    assert E.eagle_status_fetch(ws) == 1
    assert E.eagle_status_fetch(ws) == 0  # fetching clears the word


def test_status_token_out_of_range_in_verify():
    E = _E()
    V, T = 512, 3
    target = synth.normal4((1, T, V), synth.F32, 1.0, seed=2, stream=synth.STREAM_TARGET)
    tokens = np.array([[3, V + 5, 4]], np.int32)  # slot 1 carries an invalid token
    parent = np.array([[-1, 0, 0]], np.int32)
    import torch
    cfg = E.TreeCfg(1, V, 2, 2, T - 1, 0.0, synth.F32)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    a, sl, tk = torch.empty(1, **i32), torch.empty(1, 3, **i32), torch.empty(1, 3, **i32)
    E.eagle_verify(cfg, ws, E.LOSSLESS, 1.0, 1, 0, H.to_dev(target), H.to_dev(tokens), H.to_dev(parent),
                   H.to_dev(np.array([T], np.int32)), a, sl, tk)
    assert E.eagle_status_fetch(ws) == 3


def test_status_accept_length_past_limit_leaves_cache():
    import torch
    E = _E()
    B, layers, Hkv, d, Lmax = 1, 2, 1, 64, 64
    pos_stride = Hkv * d
    kv_stride = Lmax * pos_stride
    cache = np.arange(B * layers * 2 * kv_stride, dtype=np.uint16)
    kv = E.KvCfg(B, 1, Hkv, d, layers, Lmax, synth.BF16, layers * 2 * kv_stride, 2 * kv_stride, kv_stride,
                 pos_stride)
    ws = E.alloc_workspace(256)
    dc = H.to_dev(cache)
    slots = np.arange(20, dtype=np.int32)[None, :]
    nl = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    E.eagle_kv_compact(kv, dc, H.to_dev(np.array([3], np.int32)), H.to_dev(np.array([17], np.int32)),
                       H.to_dev(slots), 20, nl, ws)
    assert E.eagle_status_fetch(ws) == 3
    assert (H.to_host(dc) == cache).all() and int(nl.item()) == -9


# --------------------------------------- rows of -inf, short and constant rows ---

def _edge_rows(shape, dtype, seed, k):
    """Logit rows of four kinds, chosen by the row's flat index mod 4:
    0 ordinary (2.5 N(0, 1)); 1 mostly -inf (512 finite entries at seeded
    positions); 2 fewer than k finite entries (k // 3 + 1); 3 constant (every
    entry equal). No row is entirely -inf (its log-sum-exp would be NaN)."""
    x = synth.normal4(shape, dtype, 2.5, seed=seed, stream=synth.STREAM_DRAFT)
    V = shape[-1]
    rows = x.reshape(-1, V)
    ninf = np.uint16(0xFF80) if dtype == synth.BF16 else np.float32(-np.inf)
    rng = np.random.default_rng(seed)
    for i in range(rows.shape[0]):
        kind = i % 4
        if kind in (1, 2):
            keep = rng.choice(V, 512 if kind == 1 else k // 3 + 1, replace=False)
            vals = rows[i, keep].copy()
            rows[i, :] = ninf
            rows[i, keep] = vals
        elif kind == 3:
            rows[i, :] = rows[i, 7]
    return x


@pytest.mark.parametrize("V,dtype", [(128256, synth.BF16), (1024, synth.F32)])
def test_expand_rows_of_neg_inf_few_finite_and_constant(V, dtype):
    """Stage 1+2 on rows that are mostly -inf, hold fewer than k finite entries
    (their last children are -inf entries, lowest ids first) or are constant:
    the kernel's exact paths for few lanes holding values and for ties at the
    top, bit-exact against the oracle through stages 2-4."""
    B, k, D, N = 2, 10, 3, 40
    logits = _edge_rows((D, B, k, V), dtype, seed=V + 11, k=k)
    t, tr = _run_tree(logits, B, V, k, D, N, 0.0, dtype)
    assert np.isneginf(t.logv[t.valid == 1]).any(), "some children should be -inf entries"


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("V,dtype", [(128256, synth.BF16), (1024, synth.F32)])
def test_verify_rows_of_neg_inf_few_finite_and_constant(V, dtype, mode):
    """Stage 6 on target rows of the same four kinds (argmax over -inf entries
    and over ties; integer masses of -inf entries are zero), on a tree built
    from ordinary draft rows; accepted paths and bonus tokens bit-exact."""
    B, k, D, N = 2, 4, 3, 12
    draft = synth.normal4((D, B, k, V), dtype, 2.5, seed=5, stream=synth.STREAM_DRAFT)
    synth.plant(draft, dtype, float(np.log(9.0 * V)) + 3.0, seed=5, stream=synth.STREAM_DRAFT, frac=0.8)
    _, tr = _run_tree(draft, B, V, k, D, N, 0.0, dtype)
    T = N + 1
    target = _edge_rows((1, B, T, V), dtype, seed=V + 17, k=k)[0]
    # favour first children on the ordinary rows so that a path is accepted there
    for b in range(B):
        for t in range(int(tr["n_tree"][b])):
            kids = [c for c in range(int(tr["n_tree"][b])) if tr["parent"][b, c] == t]
            if kids and (b * T + t) % 4 == 0:
                val = np.float32(40.0)
                target[b, t, tr["tokens"][b, kids[0]]] = (val.view(np.uint32) >> 16) if dtype == synth.BF16 else val
    tokens = np.ascontiguousarray(tr["tokens"])
    parent = np.ascontiguousarray(tr["parent"])
    for seed in (3, 4):
        _verify_both(np.ascontiguousarray(target), tokens, parent, tr["n_tree"], D, mode, seed=seed, cycle=seed)


def test_status_ring_wait_timeout_then_recovers():
    """A row-kernel wait that runs out: the expansion's chunk ring receives no
    copies (test hook), every consumer's bounded wait gives up, the status word
    reads 2, and the same workspace then serves a normal, oracle-exact draft."""
    import torch
    E = _E()
    B, V, k, D, N = 1, 4096, 2, 2, 4
    cfg = E.TreeCfg(B, V, k, D, N, 0.0, synth.BF16)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    logits = synth.normal4((D, B, k, V), synth.BF16, 2.0, seed=8, stream=synth.STREAM_DRAFT)
    dl = H.to_dev(logits)
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, dtype=torch.int32, device="cuda"), torch.empty(B, dtype=torch.int32, device="cuda")
    E.eagle_tree_init(cfg, ws)
    E.eagle_test_expand_starved(cfg, ws, 0, dl[0], row_lse, ftok, fcnt)
    assert E.eagle_status_fetch(ws) == 2
    assert E.eagle_status_fetch(ws) == 0
    _run_tree(logits, B, V, k, D, N, 0.0, synth.BF16)

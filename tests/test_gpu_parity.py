"""Parity of the CUDA cycle with the CPU oracle at the five workloads.

For each workload, on the same seeded inputs:
  stage 1   top-k token ids bit-exact; the kernel's own row lse within 1e-5.
  stage 2-4 given identical fp32 log-prob inputs (the oracle's lse passed to
            both sides), candidate table, frontiers, kept set, tokens,
            parents, depths, positions, mask and n_tree bit-exact.
  end-to-end with the kernel's own lse: trees equal except at near-ties
            (keys closer than the lse tolerance), which are counted.
  stage 5   tree attention within 1e-2 max-abs (bf16) / 1e-4 (fp32) of the
            fp64 oracle on sampled (b, slot, head) rows.
  stage 6   accept lengths, accepted slots and output tokens bit-exact;
            per-row max / argmax / integer mass bit-exact.
  stage 6b  compacted KV bytewise equal to the oracle's compaction.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL

import harness as H

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", {}, False),
    ("tiny", {"threshold": 0.0}, True),
    ("llama8b_b1", {}, True),
    ("llama8b_b1", {"sharpness": 0.8, "verify": "greedy"}, False),
    ("vicuna13b_b1", {}, True),
    ("vicuna13b_b1", {"sharpness": 0.8}, False),
    ("llama8b_b64", {}, True),
    ("llama70b_b8", {}, True),
]


def _ids(case):
    name, kw, planted = case
    return name + "".join(f"-{k}{v}" for k, v in kw.items()) + ("-planted" if planted else "")


def _gpu_tree_tables(E, cfg, dc):
    import torch
    B, C = cfg.batch, cfg.C
    t = {k: torch.empty(B, C, dtype=dt, device="cuda") for k, dt in
         [("token", torch.int32), ("parent", torch.int32), ("depth", torch.int32), ("logv", torch.float32),
          ("valid", torch.uint8), ("kept", torch.uint8)]}
    nk = torch.empty(B, dtype=torch.int32, device="cuda")
    E.eagle_tree_export(cfg, dc.ws, t["token"], t["parent"], t["depth"], t["logv"], t["valid"], t["kept"], nk)
    torch.cuda.synchronize()
    out = {k: H.to_host(v) for k, v in t.items()}
    out["n_kept"] = H.to_host(nk)
    return out


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_cycle_parity(case):
    import torch
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E

    name, kw, planted = case
    w = WL.WORKLOADS[name].with_(**kw)
    inp = H.Inputs(w, seed=42, planted=planted)
    lse_o = inp.oracle_lse()
    ot, otr, ofronts = inp.oracle_tree()
    inp.align_target(otr, frac=0.9)

    kvd = H.DeviceKV(inp, layers=w.layers)
    cfg, kv = H.make_cfgs(w, kvd.geo)
    dc = C.DeviceCycle(cfg, kv)
    draft = H.to_dev(inp.draft)
    prefix = H.to_dev(inp.prefix_len)
    root = H.to_dev(inp.root)

    # ---- stages 1-2 with identical log-prob inputs, step by step ----
    lse_dev = H.to_dev(lse_o)
    E.eagle_tree_init(cfg, dc.ws)
    for s in range(w.depth):
        E.eagle_expand(cfg, dc.ws, s, draft[s], lse_dev[s], dc.row_lse, dc.ftok, dc.fcount)
        torch.cuda.synchronize()
        ft, fc = ofronts[s]
        assert (H.to_host(dc.fcount) == fc).all(), f"frontier count, step {s}"
        assert (H.to_host(dc.ftok) == ft).all(), f"frontier tokens, step {s}"
    g = _gpu_tree_tables(E, cfg, dc)
    assert (g["valid"] == ot.valid).all()
    v = ot.valid.astype(bool)
    assert (g["token"][v] == ot.token[v]).all()
    assert (g["parent"][v] == ot.parent[v]).all()
    assert (g["depth"][v] == ot.depth[v]).all()
    assert H.isclose_bits(g["logv"][v], ot.logv[v]), "child values differ in bits"

    # ---- stage 3 + 4 ----
    E.eagle_rerank(cfg, dc.ws)
    dc.build(prefix, root)
    g = _gpu_tree_tables(E, cfg, dc)
    assert (g["kept"] == ot.kept).all() and (g["n_kept"] == ot.n_kept).all()
    for key in ("tokens", "parent", "depth", "pos", "n_tree"):
        assert (H.to_host(getattr(dc, key)) == otr[key]).all(), key
    assert (H.to_host(dc.mask).view(np.uint32) == otr["mask"]).all(), "mask"

    # ---- stage 5 on sampled rows ----
    q = H.to_dev(H.WL.queries(w, inp.seed))
    dc.attention(q, kvd.cache, inp.attn_layer, prefix)
    torch.cuda.synchronize()
    got = H.f32(H.to_host(dc.attn_out))
    Kh, Vh = kvd.host_layer(inp.attn_layer)
    qh = H.WL.queries(w, inp.seed)
    rng = np.random.default_rng(0)
    nrows = w.batch * w.T * w.n_q_heads
    pick = np.arange(nrows) if nrows <= 4096 else rng.choice(nrows, 512, replace=False)
    rows = np.stack([pick // (w.T * w.n_q_heads), (pick // w.n_q_heads) % w.T, pick % w.n_q_heads], 1)
    pos_stride = w.n_kv_heads * w.head_dim
    want = oracle.attention_rows(rows, qh, Kh, Vh, kvd.geo["max_len"] * pos_stride, pos_stride, inp.prefix_len,
                                 otr["mask"], otr["n_tree"], w.n_kv_heads)
    gsel = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    tol = 1e-2 if w.dtype == synth.BF16 else 1e-4
    err = np.abs(gsel - want).max()
    assert err <= tol, f"attention max-abs {err}"

    # ---- stage 6: both modes, lossless at temperature 1 ----
    target = H.to_dev(inp.target)
    for mode in (E.GREEDY, E.LOSSLESS):
        dc.verify(mode, w.temperature, target, inp.seed, 0)
        torch.cuda.synchronize()
        if mode == E.GREEDY:
            a, sl, tk, am = oracle.verify_greedy(inp.target, otr["tokens"], otr["parent"], otr["n_tree"], w.depth)
        else:
            a, sl, tk, rmax, rmass = oracle.verify_lossless(inp.target, otr["tokens"], otr["parent"], otr["n_tree"],
                                                            inp.uniforms, w.depth, np.float32(1.0 / w.temperature),
                                                            row_stats_out=True)
        assert (H.to_host(dc.accept_len) == a).all(), f"accept_len mode {mode}"
        assert (H.to_host(dc.slots) == sl).all(), f"slots mode {mode}"
        assert (H.to_host(dc.out_tokens) == tk).all(), f"tokens mode {mode}"
        rm = torch.empty(w.batch, w.T, dtype=torch.float32, device="cuda")
        ra = torch.empty(w.batch, w.T, dtype=torch.int32, device="cuda")
        rs = torch.empty(w.batch, w.T, dtype=torch.int64, device="cuda")
        E.eagle_verify_export(cfg, dc.ws, rm, ra, rs)
        torch.cuda.synchronize()
        live = np.arange(w.T)[None, :] < otr["n_tree"][:, None]
        if mode == E.GREEDY:
            assert (H.to_host(ra)[live] == am[live]).all(), "row argmax"
        else:
            assert H.isclose_bits(H.to_host(rm)[live], rmax[live]), "row max"
            # integer masses: summed for the rows of the nodes the walk visited, 0 elsewhere
            got_mass = H.to_host(rs).view(np.uint64)
            visited = np.zeros_like(live)
            for b_ in range(w.batch):
                visited[b_, sl[b_, :a[b_] + 1]] = True
            assert (got_mass[visited] == rmass[visited]).all(), "row integer mass"
            assert (got_mass[live & ~visited] == 0).all(), "rows not visited"
        if mode == (E.GREEDY if w.verify == "greedy" else E.LOSSLESS):
            acc = a.copy()
            acc_slots = sl.copy()
    if planted:
        assert acc.max() >= 2, "planted case should accept a path"

    # ---- stage 6b ----
    before = H.tree_region_host(inp, w.layers)
    E.eagle_verify(cfg, dc.ws, E.GREEDY if w.verify == "greedy" else E.LOSSLESS, w.temperature, inp.seed, 0, target,
                   dc.tokens, dc.parent, dc.n_tree, dc.accept_len, dc.slots, dc.out_tokens)
    dc.compact(kvd.cache, prefix)
    torch.cuda.synchronize()
    after = kvd.tree_regions()
    ref = before.copy()
    g_ = kvd.geo
    Lsub = w.T
    pos_stride = w.n_kv_heads * w.head_dim
    new_len = oracle.kv_compact(ref.reshape(-1), w.batch, w.layers, w.n_kv_heads, w.head_dim,
                                w.layers * 2 * Lsub * pos_stride, 2 * Lsub * pos_stride, Lsub * pos_stride,
                                pos_stride, np.zeros(w.batch, np.int32), acc, acc_slots)
    assert (after == ref).all(), "compacted KV differs"
    assert (H.to_host(dc.new_len) == inp.prefix_len + acc + 1).all()
    assert (new_len == acc + 1).all()
    assert dc.status() == 0


def _first_divergence(ot, b, step, ft_d, fc_d, ft_o, fc_o, log_thr, tol):
    """Where the device's frontier of sequence b after `step` first differs
    from the oracle's, the two oracle values that decide the place must be a
    near-tie (closer than `tol`). Returns a description of the tie."""
    k = ot.cfg.top_k
    base = 0 if step == 0 else k + (step - 1) * k * k
    ids = np.arange(base, base + k * k)
    ids = ids[ids < ot.cfg.C]
    vals = ot.logv[b, ids]
    elig = (ot.valid[b, ids] == 1) & (vals >= log_thr)
    order = sorted(ids[elig], key=lambda i: (-float(ot.logv[b, i]), int(i)))
    n_o, n_d = int(fc_o[b]), int(fc_d[b])
    f = next((j for j in range(min(n_o, n_d)) if ft_d[b, j] != ft_o[b, j]), min(n_o, n_d))
    if f < min(n_o, n_d):
        # the device ranked at f a child that the oracle ranks after its own pick at f
        later = [i for i in order[f + 1:] if ot.token[b, i] == ft_d[b, f]]
        assert later, f"sequence {b} step {step}: device frontier token {ft_d[b, f]} is no eligible child"
        gap = float(ot.logv[b, order[f]]) - float(ot.logv[b, later[0]])
        assert 0.0 <= gap <= tol, f"sequence {b} step {step} slot {f}: values {gap:.3g} apart, not a near-tie"
        return f"step {step} slot {f}: gap {gap:.2e}"
    # one side has more frontier nodes: a child whose value sits at the threshold
    nearest = np.abs(vals[ot.valid[b, ids] == 1] - log_thr).min() if (ot.valid[b, ids] == 1).any() else np.inf
    assert np.isfinite(log_thr) and nearest <= tol, f"sequence {b} step {step}: frontier counts {n_d} vs {n_o}"
    return f"step {step}: threshold tie {nearest:.2e}"


OWN_LSE_CASES = CASES + [("llama8b_b64", {"sharpness": 0.8}, False)]


@pytest.mark.parametrize("case", OWN_LSE_CASES, ids=_ids)
def test_own_lse_end_to_end(case):
    """Stages 1-4 driven by the kernel's own fp32 lse (within 1e-5 of the
    oracle's fp64 value) against the oracle driven by its own lse. Every
    step's frontier, the candidate table, the kept set and the emitted tree
    must be identical for every sequence, at every batch size. The one
    allowed difference is a near-tie: where a sequence first diverges, the
    two oracle values that decide the place differ by at most the lse
    tolerance summed over the path (that sequence is not compared further)."""
    import torch
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E

    name, kw, planted = case
    w = WL.WORKLOADS[name].with_(**kw)
    inp = H.Inputs(w, seed=7, planted=planted)
    lse_o = inp.oracle_lse()
    geo = WL.kv_geometry(w, inp.seed, 1)
    cfg, kv = H.make_cfgs(w, geo)
    dc = C.DeviceCycle(cfg, kv)
    draft = H.to_dev(inp.draft)
    ot = oracle.Tree(oracle.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold))
    tol = H.near_tie_tol(w.depth)
    lthr = H.log_thr(w.threshold)
    B = w.batch
    diverged = {}
    E.eagle_tree_init(cfg, dc.ws)
    for s in range(w.depth):
        ft_o, fc_o = ot.expand(s, inp.draft[s])  # the oracle's own fp64-rounded lse
        E.eagle_expand(cfg, dc.ws, s, draft[s], None, dc.row_lse, dc.ftok, dc.fcount)
        torch.cuda.synchronize()
        ft_d, fc_d = H.to_host(dc.ftok), H.to_host(dc.fcount)
        g = _gpu_tree_tables(E, cfg, dc)
        for b in range(B):
            if b in diverged:
                continue
            v = ot.valid[b].astype(bool)
            # this step's children come from the same frontier: same tokens, parents, depths
            assert (g["valid"][b] == ot.valid[b]).all(), f"sequence {b} step {s}: valid"
            assert (g["token"][b][v] == ot.token[b][v]).all(), f"sequence {b} step {s}: child tokens"
            assert (g["parent"][b][v] == ot.parent[b][v]).all() and (g["depth"][b][v] == ot.depth[b][v]).all()
            assert np.abs(g["logv"][b][v].astype(np.float64) - ot.logv[b][v]).max(initial=0.0) <= tol / 2
            if fc_d[b] != fc_o[b] or (ft_d[b] != ft_o[b]).any():
                diverged[b] = _first_divergence(ot, b, s, ft_d, fc_d, ft_o, fc_o, lthr, tol)
    lse_g = H.to_host(dc.row_lse)  # [B, D, k]
    read = ~np.isnan(lse_g)
    ref = np.transpose(lse_o, (1, 0, 2))
    live = np.array([[b not in diverged] for b in range(B)])[:, :, None] & read
    err = np.abs(lse_g - ref)[live].max(initial=0.0)
    assert err <= 1e-5, f"lse abs err {err}"

    E.eagle_rerank(cfg, dc.ws)
    dc.build(H.to_dev(inp.prefix_len), H.to_dev(inp.root))
    ot.rerank()
    otr = ot.build_tree(inp.prefix_len, inp.root)
    g = _gpu_tree_tables(E, cfg, dc)
    out = {key: H.to_host(getattr(dc, key)) for key in ("tokens", "parent", "depth", "pos", "n_tree")}
    mask = H.to_host(dc.mask).view(np.uint32)
    for b in range(B):
        if b in diverged:
            continue
        kd, ko = g["kept"][b].astype(bool), ot.kept[b].astype(bool)
        if (kd != ko).any():
            # the budget's boundary fell between near-tied values
            only_d, only_o = np.flatnonzero(kd & ~ko), np.flatnonzero(ko & ~kd)
            assert len(only_d) == len(only_o), f"sequence {b}: kept counts differ"
            gap = np.abs(ot.logv[b, only_d][:, None].astype(np.float64) - ot.logv[b, only_o][None, :]).max()
            assert gap <= tol, f"sequence {b}: kept sets differ by values {gap:.3g} apart"
            diverged[b] = f"rerank boundary: gap {gap:.2e}"
            continue
        for key in ("tokens", "parent", "depth", "pos", "n_tree"):
            assert (out[key][b] == otr[key][b]).all(), f"sequence {b}: {key}"
        assert (mask[b] == otr["mask"][b]).all(), f"sequence {b}: mask"
    print(f"{name}: {B - len(diverged)}/{B} trees identical; near-ties {diverged}; lse max err {err:.2e}")
    assert dc.status() == 0


POLICY_CASES = [(name, pol) for name in ("tiny", "llama8b_b1", "llama8b_b64") for pol in (0, 1, 2, 3)]


@pytest.mark.parametrize("case", POLICY_CASES, ids=[f"{n}-policy{p}" for n, p in POLICY_CASES])
def test_policy_parity(case):
    """Stages 2-4 under each tree policy (EAGLE-2, confidence-ranked
    frontier, no rerank, static shape) with identical log-prob inputs: frontiers,
    candidate tables, kept sets and the emitted tree bit-exact; the summed
    path value of the kept nodes within fp32 rounding of the oracle's."""
    import torch
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E

    name, policy = case
    w = WL.WORKLOADS[name]
    inp = H.Inputs(w, seed=11, planted=True)
    lse_o = inp.oracle_lse()
    ot, otr, ofronts = inp.oracle_tree(lse_o, policy=policy)
    geo = WL.kv_geometry(w, inp.seed, 1)
    cfg, kv = H.make_cfgs(w, geo, policy=policy)
    dc = C.DeviceCycle(cfg, kv)
    draft = H.to_dev(inp.draft)
    lse_dev = H.to_dev(lse_o)
    E.eagle_tree_init(cfg, dc.ws)
    for s in range(w.depth):
        E.eagle_expand(cfg, dc.ws, s, draft[s], lse_dev[s], dc.row_lse, dc.ftok, dc.fcount)
        torch.cuda.synchronize()
        ft, fc = ofronts[s]
        assert (H.to_host(dc.fcount) == fc).all(), f"frontier count, step {s}"
        assert (H.to_host(dc.ftok) == ft).all(), f"frontier tokens, step {s}"
    E.eagle_rerank(cfg, dc.ws)
    dc.build(H.to_dev(inp.prefix_len), H.to_dev(inp.root))
    vs = torch.empty(w.batch, dtype=torch.float32, device="cuda")
    E.eagle_tree_value(cfg, dc.ws, vs)
    g = _gpu_tree_tables(E, cfg, dc)
    v = ot.valid.astype(bool)
    assert (g["valid"] == ot.valid).all()
    assert (g["token"][v] == ot.token[v]).all() and (g["parent"][v] == ot.parent[v]).all()
    assert H.isclose_bits(g["logv"][v], ot.logv[v])
    assert (g["kept"] == ot.kept).all() and (g["n_kept"] == ot.n_kept).all()
    for key in ("tokens", "parent", "depth", "pos", "n_tree"):
        assert (H.to_host(getattr(dc, key)) == otr[key]).all(), key
    assert (H.to_host(dc.mask).view(np.uint32) == otr["mask"]).all(), "mask"
    want = np.array([ot.value_sum(b) for b in range(w.batch)])
    got = H.to_host(vs).astype(np.float64)
    # fp32 terms each within 2 ulp of exp, summed in fp32: relative 1e-5 of the sum
    assert np.allclose(got, want, rtol=1e-5, atol=1e-6), np.abs(got - want).max()
    assert dc.status() == 0

"""Sampled drafting on the GPU against the oracle.

The device's Gumbel noise and fixed-order logarithm equal the oracle's bit for
bit (they decide which children are drawn). Stages 1-4 with the children drawn
from each row's softmax without replacement (Gumbel-top-k over the words of
the input generator, the same words on both sides; the oracle's lse passed
to both sides): frontiers, candidate tables, kept sets and trees bit-exact,
under the EAGLE-2 policy and the static shape, on fp32 and bf16 rows.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as WL

import harness as H

pytestmark = pytest.mark.gpu


def test_device_gumbel_and_log_equal_the_oracle_bit_for_bit():
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = np.concatenate([np.arange(0, 1 << 32, 1 << 14, dtype=np.uint64).astype(np.uint32),
                        synth.words(1, 1 << 16, 3, 5, synth.STREAM_GUMBEL)[0],
                        np.array([0, 1, 511, 512, 0xFFFFFFFF, 0xFFFFFE00, 0x80000000], np.uint32)])
    y = np.concatenate([np.geomspace(2.0 ** -24, 2.0 ** 12, 50000).astype(np.float32),
                        np.linspace(0.5, 2.0, 20001, dtype=np.float32), np.float32([1.0, np.sqrt(2.0)])])
    n = max(len(w), len(y))
    wd = H.to_dev(np.resize(w, n))
    yd = H.to_dev(np.resize(y, n).astype(np.float32))
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    lg = torch.empty(n, dtype=torch.float32, device="cuda")
    E.eagle_test_sampling(wd, yd, n, g, lg)
    torch.cuda.synchronize()
    assert H.isclose_bits(H.to_host(g)[:len(w)], oracle.gumbel(w)), "Gumbel noise differs"
    assert H.isclose_bits(H.to_host(lg)[:len(y)], oracle.dlog(y)), "fixed-order logarithm differs"


CASES = [("tiny", 0), ("tiny", 3), ("llama8b_b1", 0), ("llama8b_b1", 3), ("vicuna13b_b1", 0), ("llama8b_b64", 3)]


@pytest.mark.parametrize("name,policy", CASES, ids=[f"{n}-policy{p}" for n, p in CASES])
def test_sampled_expansion_parity(name, policy):
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = WL.WORKLOADS[name].with_(batch=min(WL.WORKLOADS[name].batch, 8))
    seed, cycle = 21, 3
    inp = H.Inputs(w, seed=seed)
    lse_o = inp.oracle_lse()
    B, k, D, V = w.batch, w.top_k, w.depth, w.vocab
    words = [synth.gumbel_words(B, k, V, s, cycle, seed) for s in range(D)]
    ot = oracle.Tree(oracle.TreeCfg(B, V, k, D, w.node_budget, w.threshold, policy))
    cfg = E.TreeCfg(B, V, k, D, w.node_budget, w.threshold, w.dtype, policy)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    draft, lse_dev = H.to_dev(inp.draft), H.to_dev(lse_o)
    E.eagle_tree_init(cfg, ws)
    differs_from_topk = 0
    for s in range(D):
        ft, fc = ot.expand(s, inp.draft[s], lse_o[s], words=words[s])
        E.eagle_expand_sampled(cfg, ws, s, draft[s], lse_dev[s], seed, cycle, row_lse, ftok, fcnt)
        torch.cuda.synchronize()
        assert (H.to_host(fcnt) == fc).all(), f"frontier count, step {s}"
        assert (H.to_host(ftok) == ft).all(), f"frontier tokens, step {s}"
    ot.rerank()
    tr = ot.build_tree(inp.prefix_len, inp.root)
    E.eagle_rerank(cfg, ws)
    T = w.T
    out = {n_: torch.empty(B, T, **i32) for n_ in ("tokens", "parent", "depth", "pos")}
    mask = torch.empty(B, T, cfg.W, **i32)
    n_tree = torch.empty(B, **i32)
    E.eagle_build_tree(cfg, ws, H.to_dev(inp.prefix_len), H.to_dev(inp.root), out["tokens"], out["parent"],
                       out["depth"], out["pos"], mask, n_tree)
    tab = {kk: torch.empty(B, cfg.C, dtype=dt, device="cuda") for kk, dt in
           [("token", torch.int32), ("parent", torch.int32), ("logv", torch.float32), ("valid", torch.uint8),
            ("kept", torch.uint8)]}
    E.eagle_tree_export(cfg, ws, tab["token"], tab["parent"], None, tab["logv"], tab["valid"], tab["kept"])
    torch.cuda.synchronize()
    g = {kk: H.to_host(v) for kk, v in tab.items()}
    v = ot.valid.astype(bool)
    assert (g["valid"] == ot.valid).all() and (g["token"][v] == ot.token[v]).all()
    assert (g["parent"][v] == ot.parent[v]).all() and H.isclose_bits(g["logv"][v], ot.logv[v])
    assert (g["kept"] == ot.kept).all()
    for key in ("tokens", "parent", "depth", "pos"):
        assert (H.to_host(out[key]) == tr[key]).all(), key
    assert (H.to_host(mask).view(np.uint32) == tr["mask"]).all()
    # the draw is not the top-k: some root child is not among the root row's k largest logits
    for b in range(B):
        _, _, top = oracle.row_stats(np.ascontiguousarray(inp.draft[0, b, 0]), k)
        differs_from_topk += not set(ot.token[b, :k][ot.valid[b, :k] == 1]) <= set(top)
    assert differs_from_topk > 0 or w.vocab <= 1024
    assert E.eagle_status_fetch(ws) == 0


DRAFT_CASES = [("tiny", 3, 0.0), ("tiny", 0, 0.9), ("llama8b_b1", 3, 0.9), ("llama8b_b1", 0, 0.0),
               ("vicuna13b_b1", 3, 0.5)]


@pytest.mark.parametrize("name,policy,align", DRAFT_CASES, ids=[f"{n}-policy{p}-align{a}" for n, p, a in DRAFT_CASES])
def test_draft_probability_verification_parity(name, policy, align):
    """A sampled-drafting cycle (the oracle's lse on both sides), then stage 6
    with the draft-probability rule against the oracle's verify_draft: accept
    lengths, accepted slots and output tokens bit-exact, for two cycles of
    uniforms; targets partly aligned with the first drawn children so that
    paths are accepted as well as rejected."""
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = WL.WORKLOADS[name].with_(batch=2)
    seed = 33
    inp = H.Inputs(w, seed=seed)
    lse_o = inp.oracle_lse()
    B, k, D, V, T = w.batch, w.top_k, w.depth, w.vocab, w.T
    words = [synth.gumbel_words(B, k, V, s, 0, seed) for s in range(D)]
    ot = oracle.Tree(oracle.TreeCfg(B, V, k, D, w.node_budget, w.threshold, policy))
    for s in range(D):
        ot.expand(s, inp.draft[s], lse_o[s], words=words[s])
    ot.rerank()
    tr = ot.build_tree(inp.prefix_len, inp.root)
    if align > 0:
        inp.align_target(tr, frac=align)
    cfg = E.TreeCfg(B, V, k, D, w.node_budget, w.threshold, w.dtype, policy)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    draft, lse_dev = H.to_dev(inp.draft), H.to_dev(lse_o)
    E.eagle_tree_init(cfg, ws)
    for s in range(D):
        E.eagle_expand_sampled(cfg, ws, s, draft[s], lse_dev[s], seed, 0, row_lse, ftok, fcnt)
    E.eagle_rerank(cfg, ws)
    out = {n_: torch.empty(B, T, **i32) for n_ in ("tokens", "parent", "depth", "pos")}
    mask = torch.empty(B, T, cfg.W, **i32)
    n_tree = torch.empty(B, **i32)
    E.eagle_build_tree(cfg, ws, H.to_dev(inp.prefix_len), H.to_dev(inp.root), out["tokens"], out["parent"],
                       out["depth"], out["pos"], mask, n_tree)
    torch.cuda.synchronize()
    assert (H.to_host(out["tokens"]) == tr["tokens"]).all() and (H.to_host(n_tree) == tr["n_tree"]).all()
    target = H.to_dev(inp.target)
    flat = np.ascontiguousarray(inp.draft.reshape(-1, V))
    rows = ot.draft_rows(tr["slot_of"], tr["n_tree"])
    accepted = 0
    for cycle in (0, 1):
        a, sl, tk = torch.empty(B, **i32), torch.empty(B, D + 1, **i32), torch.empty(B, D + 1, **i32)
        E.eagle_verify(cfg, ws, E.DRAFT, 1.0, seed, cycle, target, out["tokens"], out["parent"], n_tree, a, sl, tk,
                       draft_logits=draft)
        torch.cuda.synchronize()
        ra, rs, rt = oracle.verify_draft(inp.target, flat, rows, tr["tokens"], tr["parent"], tr["n_tree"],
                                         WL.uniforms(w, seed, cycle), D)
        assert (H.to_host(a) == ra).all(), (cycle, H.to_host(a), ra)
        assert (H.to_host(sl) == rs).all() and (H.to_host(tk) == rt).all(), cycle
        accepted += int(ra.sum())
    if align >= 0.9:
        assert accepted > 0, "aligned targets should accept drawn children"
    assert E.eagle_status_fetch(ws) == 0

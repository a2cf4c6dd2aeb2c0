"""Stage 1 and greedy verification over a vocabulary split into slices.

CPU (gloo, world size 2): the exchange moves every rank's partials (its
slice's maximum, exp-sum and top-k keys) to every rank in rank order, and a
merge of the gathered partials reproduces the oracle's stage 1 of the whole
row (top-k ids exactly, lse in fp64). GPU: the slice partial and merge
kernels on 1, 2, 3, 4 and 8 slices of the same rows give the oracle's top-k
ids and argmax exactly and its lse within 1e-5; stage 2 from the merged top-k
(with the oracle's lse, the stage-chained reading of "identical log-prob
inputs") and the greedy walk from the merged argmax are bit-exact with the
oracle's tree and accepted path.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import synth
from synth import workloads as WL

import harness as H


def _f2o(v: np.ndarray) -> np.ndarray:
    """Order-preserving bits of float32 values (-0 and +0 one value)."""
    b = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    b = np.where((b & 0x7FFFFFFF) == 0, 0, b)
    return np.where(b & 0x80000000, (~b) & 0xFFFFFFFF, b | 0x80000000)


def _keys(values: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """The partials' 64-bit keys: (ordered value bits) << 32 | (0xFFFFFFFF - id)."""
    return (_f2o(values) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ids.astype(np.uint64))


def _host_partial(row: np.ndarray, offset: int, k: int):
    """A slice's partial on the host (fp64 statistics; ties: lower id first)."""
    x = row.astype(np.float64)
    m = x.max()
    s = np.exp(x - m).sum()
    order = np.lexsort((np.arange(len(x)), -x))[:k]
    keys = np.zeros(16, np.uint64)
    keys[:len(order)] = _keys(row[order].astype(np.float32), order + offset)
    return np.array([m, s]), keys


def _host_merge(ms_all: np.ndarray, keys_all: np.ndarray, k: int):
    m = ms_all[:, 0].max()
    lse = m + np.log((ms_all[:, 1] * np.exp(ms_all[:, 0] - m)).sum())
    keys = np.sort(keys_all.ravel())[::-1][:k]
    return lse, (np.uint64(0xFFFFFFFF) - (keys & np.uint64(0xFFFFFFFF))).astype(np.int64)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gather_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from speculative_decoding_dynamic_gb300 import shard
    rows, V, k = 3, 1000, 5
    full = synth.normal4((rows, V), synth.F32, 2.0, seed=12, stream=synth.STREAM_DRAFT)
    lo, n = shard.slice_bounds(V, world, 4)[rank]
    ms = np.zeros((rows, 2))
    keys = np.zeros((rows, 16), np.uint64)
    for r in range(rows):
        ms[r], keys[r] = _host_partial(full[r, lo:lo + n], lo, k)
    ms_all, keys_all = shard.all_gather_partials(torch.from_numpy(ms), torch.from_numpy(keys.view(np.int64)))
    out[rank] = (ms_all.numpy(), keys_all.numpy().view(np.uint64), ms, keys)
    dist.barrier()
    dist.destroy_process_group()


def test_slice_bounds_are_aligned_and_cover_the_vocabulary():
    from speculative_decoding_dynamic_gb300 import shard
    for V, S, es in ((128256, 8, 2), (128256, 3, 2), (32000, 4, 2), (1000, 2, 4), (1024, 8, 4)):
        b = shard.slice_bounds(V, S, es)
        assert len(b) == S and b[0][0] == 0 and sum(n for _, n in b) == V
        assert all(off * es % 16 == 0 and n > 0 for off, n in b)
        assert all(b[i][0] + b[i][1] == b[i + 1][0] for i in range(S - 1))
    with pytest.raises(ValueError):
        shard.slice_bounds(10, 20, 4)


def test_two_gloo_ranks_exchange_partials_and_the_merge_is_the_whole_row():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_gather_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    rows, V, k = 3, 1000, 5
    full = synth.normal4((rows, V), synth.F32, 2.0, seed=12, stream=synth.STREAM_DRAFT)
    for rank in range(world):
        ms_all, keys_all, _, _ = out[rank]
        for src in range(world):  # rank order, the sender's own partials
            assert np.array_equal(ms_all[src], out[src][2]) and np.array_equal(keys_all[src], out[src][3])
        for r in range(rows):
            lse, ids = _host_merge(ms_all[:, r], keys_all[:, r], k)
            lse64, _, top = oracle.row_stats(np.ascontiguousarray(full[r]), k)
            assert np.array_equal(ids, top)
            assert abs(lse - lse64) < 1e-9


# ------------------------------------------------------------------ GPU ---

def _slices(E, rows_host: np.ndarray, S: int):
    """Device copies of the S slices of host rows [R, V] and their offsets."""
    from speculative_decoding_dynamic_gb300 import shard
    V = rows_host.shape[-1]
    es = 2 if rows_host.dtype == np.uint16 else 4
    out = []
    for off, n in shard.slice_bounds(V, S, es):
        out.append((off, n, H.to_dev(np.ascontiguousarray(rows_host[..., off:off + n]))))
    return out


def _merged(E, cfg, ws, rows_host: np.ndarray, S: int):
    import torch
    R = rows_host.shape[0]
    parts = _slices(E, rows_host, S)
    ms = torch.empty(S, R, 2, dtype=torch.float32, device="cuda")
    keys = torch.empty(S, R, 16, dtype=torch.int64, device="cuda")
    for i, (off, n, dev) in enumerate(parts):
        E.eagle_shard_partials(cfg, ws, R, n, off, dev, ms[i], keys[i])
    k = cfg.top_k
    lse = torch.empty(R, dtype=torch.float32, device="cuda")
    ids = torch.empty(R, k, dtype=torch.int32, device="cuda")
    vals = torch.empty(R, k, dtype=torch.float32, device="cuda")
    arg = torch.empty(R, dtype=torch.int32, device="cuda")
    E.eagle_shard_merge(cfg, ws, S, R, ms, keys, lse, ids, vals, arg)
    torch.cuda.synchronize()
    return H.to_host(lse), H.to_host(ids), H.to_host(vals), H.to_host(arg)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "llama8b_b1", "vicuna13b_b1"])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
def test_shard_merge_equals_the_whole_row(name, S):
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = WL.WORKLOADS[name].with_(batch=2)
    draft = WL.draft_logits(w, 9, planted=True)  # [D, B, k, V]
    rows = np.ascontiguousarray(draft[1].reshape(-1, w.vocab))
    rows[3] = rows[3, 0]  # a constant row: every entry ties
    cfg = E.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, w.dtype)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    lse, ids, vals, arg = _merged(E, cfg, ws, rows, S)
    for r in range(rows.shape[0]):
        lse64, _, top = oracle.row_stats(np.ascontiguousarray(rows[r]), w.top_k)
        assert (ids[r] == top).all(), (r, ids[r], top)
        assert arg[r] == top[0]
        assert abs(float(lse[r]) - lse64) <= 1e-5, (r, float(lse[r]), lse64)
        assert (vals[r] == H.f32(rows[r])[top]).all()
    assert E.eagle_status_fetch(ws) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("name,S", [("tiny", 2), ("llama8b_b1", 4), ("llama8b_b1", 8)])
def test_sharded_expansion_and_greedy_verify_match_the_oracle(name, S):
    """Stages 1-2 of every step from slice partials (merged top-k; the oracle's
    lse), rerank and emission, then greedy verification from the merged argmax
    of the target rows: tree and accepted path bit-exact with the oracle."""
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = WL.WORKLOADS[name].with_(batch=2)
    inp = H.Inputs(w, seed=13, planted=True)
    lse_o = inp.oracle_lse()
    ot, otr, ofronts = inp.oracle_tree(lse_o)
    inp.align_target(otr, frac=0.9)
    cfg = E.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, w.dtype)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    B, k, D, T = w.batch, w.top_k, w.depth, w.T
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    E.eagle_tree_init(cfg, ws)
    for s in range(D):
        rows = np.ascontiguousarray(inp.draft[s].reshape(B * k, w.vocab))
        _, ids, vals, _ = _merged(E, cfg, ws, rows, S)
        E.eagle_expand_topk(cfg, ws, s, H.to_dev(ids), H.to_dev(vals), H.to_dev(lse_o[s]), row_lse, ftok, fcnt)
        torch.cuda.synchronize()
        assert (H.to_host(fcnt) == ofronts[s][1]).all() and (H.to_host(ftok) == ofronts[s][0]).all(), s
    E.eagle_rerank(cfg, ws)
    out = {n: torch.empty(B, T, **i32) for n in ("tokens", "parent", "depth", "pos")}
    mask = torch.empty(B, T, cfg.W, **i32)
    n_tree = torch.empty(B, **i32)
    E.eagle_build_tree(cfg, ws, H.to_dev(inp.prefix_len), H.to_dev(inp.root), out["tokens"], out["parent"],
                       out["depth"], out["pos"], mask, n_tree)
    torch.cuda.synchronize()
    for key in ("tokens", "parent", "depth", "pos"):
        assert (H.to_host(out[key]) == otr[key]).all(), key
    assert (H.to_host(n_tree) == otr["n_tree"]).all()
    # greedy verification from the merged argmax of the target rows
    _, _, _, arg = _merged(E, cfg, ws, np.ascontiguousarray(inp.target.reshape(B * T, w.vocab)), S)
    a, sl, tk = torch.empty(B, **i32), torch.empty(B, D + 1, **i32), torch.empty(B, D + 1, **i32)
    E.eagle_verify_argmax(cfg, ws, H.to_dev(arg.reshape(B, T)), out["tokens"], out["parent"], n_tree, a, sl, tk)
    torch.cuda.synchronize()
    ra, rs, rt, _ = oracle.verify_greedy(inp.target, otr["tokens"], otr["parent"], otr["n_tree"], D)
    assert (H.to_host(a) == ra).all() and (H.to_host(sl) == rs).all() and (H.to_host(tk) == rt).all()
    assert ra.max() >= 1, "aligned targets should accept a path"
    assert E.eagle_status_fetch(ws) == 0

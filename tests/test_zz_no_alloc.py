"""eagle_verify_static: verification for callers that may not allocate.

Some callers cannot give the library a workspace: an engine plugin whose host
plans all device memory up front, or a decode loop that must never wait on
the allocator. eagle_verify_static keeps its scratch in a fixed array inside
the library instead. These tests call it through the C ABI on real device
buffers only and check its results against eagle_verify (the workspace
version) on the same inputs, for two calls in a row, in greedy and lossless
mode, and against the oracle on the small cases; the large cases sit near the
array's row limit, in bf16 and fp32 and both modes. (Its size checks, which
reject a call before any CUDA work, are tested without a GPU in test_abi.py.) The file is collected last so that a run
stopping at the first failure has already run the rest.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as WL

import harness as H

pytestmark = pytest.mark.gpu


def _outs(B, Dp1):
    import torch
    return (torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, Dp1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, Dp1), -7, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("name,batch", [("tiny", 3), ("llama8b_b1", 2)])
def test_static_scratch_verify_matches_workspace_verify(name, batch):
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E

    w = WL.WORKLOADS[name].with_(batch=batch, prefix=64)
    inp = H.Inputs(w, seed=11, planted=True)
    _, tr, _ = inp.oracle_tree()
    inp.align_target(tr, frac=0.8)
    cfg = E.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, w.dtype)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    target = H.to_dev(inp.target)
    tokens, parent, n_tree = H.to_dev(tr["tokens"]), H.to_dev(tr["parent"]), H.to_dev(tr["n_tree"])
    B, Dp1 = w.batch, w.depth + 1

    for mode in (E.GREEDY, E.LOSSLESS):
        for call in range(2):
            ref = _outs(B, Dp1)
            E.eagle_verify(cfg, ws, mode, 1.0, inp.seed, call, target, tokens, parent, n_tree, *ref)
            got = _outs(B, Dp1)
            E.eagle_verify_static(cfg, mode, 1.0, inp.seed, call, target, tokens, parent, n_tree, *got)
            torch.cuda.synchronize()
            for r, g in zip(ref, got):
                assert (H.to_host(r) == H.to_host(g)).all(), (mode, call)
            if mode == E.GREEDY:
                a, sl, tk, _ = oracle.verify_greedy(inp.target, tr["tokens"], tr["parent"], tr["n_tree"], w.depth)
            else:
                a, sl, tk = oracle.verify_lossless(inp.target, tr["tokens"], tr["parent"], tr["n_tree"],
                                                   WL.uniforms(w, inp.seed, call), w.depth)
            assert (H.to_host(got[0]) == a).all() and (H.to_host(got[1]) == sl).all()
            assert (H.to_host(got[2]) == tk).all()
    assert E.eagle_status_fetch(ws) == 0


@pytest.mark.parametrize("mode,B,N,esize", [
    (1, 64, 60, 2),   # lossless bf16: 3904 rows, near the 4096-row limit
    (1, 34, 60, 4),   # lossless fp32: 2074 rows of 128256 entries
    (0, 34, 60, 4),   # greedy fp32
])
def test_static_scratch_verify_near_its_limits(mode, B, N, esize):
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E

    V, k, D = 128256, 4, 3
    T = N + 1
    dt = torch.bfloat16 if esize == 2 else torch.float32
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + mode)
    target = (2.0 * torch.randn(B, T, V, generator=g, device="cuda")).to(dt)
    # a complete k-ary tree in slot order (parents precede children, at most k
    # children per node, depth 3 at 61 slots)
    tokens = torch.randint(0, V, (B, T), generator=g, device="cuda", dtype=torch.int32)
    par = np.full((B, T), -1, np.int32)
    for c in range(1, T):
        par[:, c] = (c - 1) // k
    parent = H.to_dev(par)
    n_tree = torch.full((B,), T, dtype=torch.int32, device="cuda")
    cfg = E.TreeCfg(B, V, k, D, N, 0.0, E.EAGLE_BF16 if esize == 2 else E.EAGLE_F32)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    for call in range(2):
        ref = _outs(B, D + 1)
        E.eagle_verify(cfg, ws, mode, 1.0, 5, call, target, tokens, parent, n_tree, *ref)
        got = _outs(B, D + 1)
        E.eagle_verify_static(cfg, mode, 1.0, 5, call, target, tokens, parent, n_tree, *got)
        torch.cuda.synchronize()
        for r, g_ in zip(ref, got):
            assert (H.to_host(r) == H.to_host(g_)).all(), call
        assert (H.to_host(got[0]) >= 0).all()
    assert E.eagle_status_fetch(ws) == 0

"""eagle_verify_static: verification for callers that may not allocate.

Some callers cannot give the library a workspace: an engine plugin whose host
plans all device memory up front, or a decode loop that must never wait on
the allocator. eagle_verify_static keeps its scratch in a fixed array inside
the library instead. This test calls it through the C ABI and checks that its
results equal those of eagle_verify (the workspace version) on the same
inputs, for two calls in a row, in greedy and lossless mode. It is collected
last so that a run stopping at the first failure has already run the rest.
"""
import numpy as np
import pytest

from synth import workloads as WL

import harness as H

pytestmark = pytest.mark.gpu


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

    def outs():
        return (torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                torch.full((B, Dp1), -7, dtype=torch.int32, device="cuda"),
                torch.full((B, Dp1), -7, dtype=torch.int32, device="cuda"))

    for mode in (E.GREEDY, E.LOSSLESS):
        for call in range(2):
            uni = H.to_dev(WL.uniforms(w, inp.seed, call))
            ref = outs()
            E.eagle_verify(cfg, ws, mode, 1.0, target, tokens, parent, n_tree, uni, *ref)
            got = outs()
            E.eagle_verify_static(cfg, mode, 1.0, target, tokens, parent, n_tree, uni, *got)
            torch.cuda.synchronize()
            for r, g in zip(ref, got):
                assert (H.to_host(r) == H.to_host(g)).all(), (mode, call)
            assert (H.to_host(ref[0]) >= 0).all()
    assert E.eagle_status_fetch(ws) == 0


def test_static_scratch_verify_rejects_oversized_batches():
    from speculative_decoding_dynamic_gb300 import eagle as E

    cfg = E.TreeCfg(80, 1024, 4, 3, 60, 0.0, E.EAGLE_F32)  # 80 * 61 rows > 4096
    p = 1 << 20
    rc = E.raw_call("eagle_verify_static", cfg, 0, 1.0, p, p, p, p, None, p, p, p, None)
    assert rc == -2

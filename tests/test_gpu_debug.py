"""Checked library and canary-padded outputs (failure detection without a sanitizer).

The checked build (EAGLE_DEBUG) makes every launching call wait for its work
and return the device status its own kernels raised, so the first faulty
call is the one that reports it; the release library reports the same fault
only at eagle_status_fetch. The faults are made on the host side of the data
(a NaN logit, a token id past the vocabulary): no kernel traps or hangs.

Canary-padded outputs: every output of one whole cycle (and of the LM-head
calls) is a view into a larger buffer whose margins hold a byte pattern; the
margins must come back unchanged and the results equal those of a run into
plain buffers.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from synth import workloads as WL

import harness as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

_CHECKED_SCRIPT = r'''
import sys
import numpy as np
import torch
sys.path[:0] = [ROOT, TESTS]
from speculative_decoding_dynamic_gb300 import eagle as E
import synth
import harness as H
assert E.DEBUG and E.LIB_PATH.endswith("libeagle_debug.so")

B, V, k, D, N = 1, 2048, 4, 2, 6
cfg = E.TreeCfg(B, V, k, D, N, 0.0, synth.F32)
ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
i32 = dict(dtype=torch.int32, device="cuda")
row_lse = torch.empty(B, D, k, dtype=torch.float32, device="cuda")
ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
T, W = cfg.T, cfg.W
out = [torch.empty(B, T, **i32) for _ in range(4)]
mask, n_tree = torch.empty(B, T, W, **i32), torch.empty(B, **i32)
prefix = H.to_dev(np.array([7], np.int32))

# a clean draft: every call returns EAGLE_OK
logits = synth.normal4((D, B, k, V), synth.F32, 1.0, seed=1, stream=synth.STREAM_DRAFT)
dl = H.to_dev(logits)
E.eagle_tree_init(cfg, ws)
for s in range(D):
    E.eagle_expand(cfg, ws, s, dl[s], None, row_lse, ftok, fcnt)
E.eagle_rerank(cfg, ws)
E.eagle_build_tree(cfg, ws, prefix, H.to_dev(np.array([5], np.int32)), *out, mask, n_tree)
assert E.eagle_status_fetch(ws) == 0

# a root token past the vocabulary: eagle_build_tree itself fails
try:
    E.eagle_build_tree(cfg, ws, prefix, H.to_dev(np.array([V + 3], np.int32)), *out, mask, n_tree)
    raise SystemExit("build_tree: no error from the checked library")
except E.EagleError as e:
    assert e.code == -5, e
assert E.eagle_status_fetch(ws) == 3  # the word stays set for the fetch, which clears it

# a non-finite logit in the root row: the expansion of step 0 fails at once
logits[0, 0, 0, 77] = np.nan
dl = H.to_dev(logits)
E.eagle_tree_init(cfg, ws)
try:
    E.eagle_expand(cfg, ws, 0, dl[0], None, row_lse, ftok, fcnt)
    raise SystemExit("expand: no error from the checked library")
except E.EagleError as e:
    assert e.code == -5, e
print("CHECKED-OK")
'''


def test_checked_library_reports_a_fault_at_the_faulty_call():
    from speculative_decoding_dynamic_gb300 import build as Bd
    Bd.build(debug=True)
    env = dict(os.environ, EAGLE_DEBUG="1")
    script = f"ROOT = {ROOT!r}\nTESTS = {TESTS!r}\n" + _CHECKED_SCRIPT
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "CHECKED-OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


def test_release_library_reports_the_same_fault_at_status_fetch():
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    assert not E.DEBUG
    B, V, k, D, N = 1, 2048, 4, 2, 6
    cfg = E.TreeCfg(B, V, k, D, N, 0.0, synth.F32)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    T, W = cfg.T, cfg.W
    out = [torch.empty(B, T, **i32) for _ in range(4)]
    mask, n_tree = torch.empty(B, T, W, **i32), torch.empty(B, **i32)
    E.eagle_tree_init(cfg, ws)
    E.eagle_rerank(cfg, ws)  # no candidates: the tree is the root alone
    E.eagle_build_tree(cfg, ws, H.to_dev(np.array([7], np.int32)), H.to_dev(np.array([V + 3], np.int32)), *out,
                       mask, n_tree)  # returns 0: the fault is found on the device
    assert E.eagle_status_fetch(ws) == 3


# ------------------------------------------------------------- canaries ---

PAD = 4096           # bytes of margin on each side (keeps 256-byte alignment)
CANARY = 0xA5


def _padded(shape, dtype):
    import torch
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((n + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")
    return raw, raw[PAD:PAD + n].view(dtype).view(*shape)


def _margins_intact(raw) -> bool:
    h = raw.cpu().numpy()
    return bool((h[:PAD] == CANARY).all() and (h[-PAD:] == CANARY).all())


@pytest.mark.parametrize("name,verify", [("tiny", "lossless"), ("llama8b_b1", "lossless"), ("llama8b_b1", "greedy")])
def test_cycle_outputs_stay_inside_their_buffers(name, verify):
    import torch
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E
    w = WL.WORKLOADS[name].with_(batch=2, verify=verify)
    inp = H.Inputs(w, seed=31, planted=True)
    ot, otr, _ = inp.oracle_tree()
    inp.align_target(otr, frac=0.9)
    mode = E.GREEDY if verify == "greedy" else E.LOSSLESS
    results = []
    for padded in (False, True):
        kvd = H.DeviceKV(inp, layers=w.layers)
        cfg, kv = H.make_cfgs(w, kvd.geo)
        dc = C.DeviceCycle(cfg, kv)
        raws = {}
        if padded:
            for attr in ("row_lse", "ftok", "fcount", "tokens", "parent", "depth", "pos", "mask", "n_tree",
                         "attn_out", "accept_len", "slots", "out_tokens", "new_len"):
                t = getattr(dc, attr)
                raws[attr], v = _padded(tuple(t.shape), t.dtype)
                setattr(dc, attr, v)
        q = H.to_dev(WL.queries(w, 31))
        dc.run(H.to_dev(inp.draft), H.to_dev(inp.prefix_len), H.to_dev(inp.root), q, kvd.cache, inp.attn_layer,
               H.to_dev(inp.target), 7, 3, mode, w.temperature)
        torch.cuda.synchronize()
        assert dc.status() == 0
        for attr, raw in raws.items():
            assert _margins_intact(raw), f"{attr} written outside its buffer"
        res = {a: H.to_host(getattr(dc, a)) for a in ("tokens", "parent", "mask", "n_tree", "accept_len", "slots",
                                                       "out_tokens", "new_len")}
        att = H.to_host(dc.attn_out)  # rows past a tree's slots are not outputs
        res["attn_out"] = [att[b, :res["n_tree"][b]] for b in range(w.batch)]
        res["cache"] = kvd.tree_regions()  # the positions compaction reads and writes
        results.append(res)
    for a in results[0]:
        if a == "attn_out":
            # the split-KV merge adds the splits' partials starting from the last
            # CTA's own: the fp32 order may differ between runs, so a bf16 output
            # may round to a neighbour (one bf16 step: at most 2^-7 |o|; 2^-8 near 0)
            for x, y in zip(results[0][a], results[1][a]):
                xf, yf = H.f32(x), H.f32(y)
                big = np.maximum(np.abs(xf), np.abs(yf))
                tol = np.maximum(2.0 ** -8, 2.0 ** -7 * big) if x.dtype == np.uint16 else 1e-6 + 1e-6 * big
                assert (np.abs(xf - yf) <= tol).all(), a
        else:
            assert np.array_equal(results[0][a], results[1][a]), a


def test_lmhead_outputs_stay_inside_their_buffers():
    import torch
    from speculative_decoding_dynamic_gb300 import eagle as E
    B, k, V, Hd = 3, 10, 4104, 256
    cfg = E.TreeCfg(B, V, k, 1, 4, 0.0, synth.BF16, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h = synth.normal4((B * k, Hd), synth.BF16, 1.0, 3, synth.STREAM_HIDDEN)
    W = synth.normal4((V, Hd), synth.BF16, 0.05, 3, synth.STREAM_LMHEAD)
    dh, dW = H.to_dev(h), H.to_dev(W)
    raw_lg, lg = _padded((B, k, V), torch.bfloat16)
    E.eagle_lmhead(cfg, ws, Hd, dh, dW, lg)
    sc = E.alloc_workspace(E.eagle_lmhead_topk_scratch_bytes(cfg))
    raws = [_padded((B * k,), torch.float32), _padded((B * k, k), torch.int32), _padded((B * k, k), torch.float32)]
    E.eagle_lmhead_topk(cfg, ws, Hd, dh, dW, sc, *(v for _, v in raws))
    torch.cuda.synchronize()
    assert E.eagle_status_fetch(ws) == 0
    assert _margins_intact(raw_lg)
    for raw, _ in raws:
        assert _margins_intact(raw)

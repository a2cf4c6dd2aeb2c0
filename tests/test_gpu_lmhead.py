"""LM-head logits on the tensor cores against the oracle, a draft step fed by
them, and the LM head with stage 1 in its epilogue.

The draft model reuses the target's LM head ("EAGLE" notes, EAGLE 方法). The
oracle sums the exact bf16 products in double and rounds once; the kernel
accumulates in fp32 on the tensor cores in an unspecified order and rounding,
so each entry must lie within H * 2^-23 * sum_h |hidden[h] W[v, h]| of the
exact sum (recursive fp32 summation of H terms, round-toward-zero allowed),
plus half a bf16 ulp when the output is bf16. A dropped or repeated 64-wide
hidden block, a transposed operand or a wrong vocabulary tile misses that
bound by orders of magnitude.

The fused call (eagle_lmhead_topk) rounds the same fp32 sums to the logit
type and reduces them on chip, so its top-k ids and logits must equal the
oracle's stage 1 on the rows eagle_lmhead writes (whose entries the check
above pins to the oracle's exact sums) bit for bit, and its lse the oracle's
fp64 lse of those rows within 1e-5.
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


def _inputs(M, V, Hd, seed):
    h = synth.normal4((M, Hd), synth.BF16, 1.0, seed, synth.STREAM_HIDDEN)
    W = synth.normal4((V, Hd), synth.BF16, 0.05, seed, synth.STREAM_LMHEAD)
    return h, W


def _check(got, h, W, dtype):
    ref = oracle.lmhead_logits(h, W).astype(np.float64)
    a = np.abs(synth.bf16_to_f32(h)).astype(np.float64)
    b = np.abs(synth.bf16_to_f32(W)).astype(np.float64)
    tol = h.shape[1] * 2.0 ** -23 * (a @ b.T) + np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    if dtype == synth.BF16:
        tol = tol + 2.0 ** -8 * (np.abs(ref) + tol)
        g = synth.bf16_to_f32(got).astype(np.float64)
    else:
        g = got.astype(np.float64)
    err = np.abs(g - ref)
    assert np.all(err <= tol), f"max err {err.max()} at {np.unravel_index(np.argmax(err - tol), err.shape)}"
    return g


def _lmhead(E, cfg, ws, Hd, dh, dW):
    import torch
    B, k, V = cfg.batch, cfg.top_k, cfg.vocab
    dt = torch.float32 if cfg.logit_dtype == synth.F32 else torch.bfloat16
    out = torch.full((B, k, V), float("nan"), dtype=dt, device="cuda")
    E.eagle_lmhead(cfg, ws, Hd, dh, dW, out)
    torch.cuda.synchronize()
    assert E.eagle_status_fetch(ws) == 0
    return H.to_host(out).reshape(B * k, V)


@pytest.mark.parametrize("B,k,V,Hd,dtype", [
    (1, 10, 1000, 256, synth.F32),     # 10 rows (one 16-column MMA), ragged last vocabulary tile
    (1, 10, 1000, 200, synth.BF16),    # hidden size not a multiple of 64: zero-filled last block
    (30, 10, 2056, 512, synth.F32),    # 300 rows: two row chunks of 160
    (1, 1, 136, 64, synth.F32),        # one row, one hidden block, 8-row last tile
    (64, 10, 4096, 128, synth.BF16),   # 640 rows: three chunks of 224 (the last one 192 live)
    (2, 16, 384, 1024, synth.BF16),    # 32 rows, 16 hidden blocks (the ring wraps)
    (8, 8, 2056, 8192, synth.BF16),    # 70B shape: 64 rows, 128 hidden blocks
    (1, 10, 32000, 5120, synth.BF16),  # 13B shape: 250 vocabulary tiles, 80 hidden blocks
])
def test_lmhead_matches_oracle(B, k, V, Hd, dtype):
    E = _E()
    cfg = E.TreeCfg(B, V, k, 1, 1, 0.0, dtype, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h, W = _inputs(B * k, V, Hd, seed=V + Hd)
    got = _lmhead(E, cfg, ws, Hd, H.to_dev(h), H.to_dev(W))
    _check(got, h, W, dtype)


@pytest.fixture(scope="module")
def llama8b_head():
    """Llama-8B-shaped LM head (V = 128256, H = 4096), bf16, on the device."""
    V, Hd = 128256, 4096
    W = synth.normal4((V, Hd), synth.BF16, 0.02, 8, synth.STREAM_LMHEAD)
    return V, Hd, W, H.to_dev(W)


@pytest.mark.parametrize("B", [1, 64])
def test_lmhead_full_size_sampled(llama8b_head, B):
    """Full vocabulary and hidden size at batch 1 and 64 (k = 10): sampled
    vocabulary columns (every tile boundary of a few tiles, the last entries
    and a seeded spread) against the oracle."""
    E = _E()
    V, Hd, W, dW = llama8b_head
    k = 10
    cfg = E.TreeCfg(B, V, k, 6, 60, 0.0, synth.BF16, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h = synth.normal4((B * k, Hd), synth.BF16, 1.0, B, synth.STREAM_HIDDEN)
    got = _lmhead(E, cfg, ws, Hd, H.to_dev(h), dW)
    rng = np.random.default_rng(B)
    cols = np.unique(np.concatenate([[0, 1, 127, 128, 129, 255, 256, 1001 * 128 - 1, 1001 * 128, V - 2, V - 1],
                                     rng.integers(0, V, 53)]))
    _check(np.ascontiguousarray(got[:, cols]), h, np.ascontiguousarray(W[cols]), synth.BF16)
    assert np.isfinite(synth.bf16_to_f32(got)).all()


def test_lmhead_feeds_expand():
    """One draft step on device logits: the expansion equals the oracle's on
    the same (device-written) rows and log-sum-exps."""
    import torch
    E = _E()
    B, k, V, Hd = 2, 4, 4104, 256
    cfg = E.TreeCfg(B, V, k, 1, 4, 0.0, synth.BF16, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h, W = _inputs(B * k, V, Hd, seed=5)
    E.eagle_tree_init(cfg, ws)
    out = torch.empty(B, k, V, dtype=torch.bfloat16, device="cuda")
    E.eagle_lmhead(cfg, ws, Hd, H.to_dev(h), H.to_dev(W), out)
    torch.cuda.synchronize()
    lg = H.to_host(out)
    _check(lg.reshape(B * k, V), h, W, synth.BF16)
    lse = np.zeros((B, k), np.float32)
    for b in range(B):
        for f in range(k):
            _, lse[b, f], _ = oracle.row_stats(np.ascontiguousarray(lg[b, f]), 1)
    t = oracle.Tree(oracle.TreeCfg(B, V, k, 1, 4, 0.0, 0))
    ftok_o, fcnt_o = t.expand(0, lg)[:2]
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, 1, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    E.eagle_expand(cfg, ws, 0, out, H.to_dev(lse), row_lse, ftok, fcnt)
    torch.cuda.synchronize()
    assert (H.to_host(fcnt) == fcnt_o).all()
    assert (H.to_host(ftok) == ftok_o).all()
    assert E.eagle_status_fetch(ws) == 0


def _fused(E, cfg, ws, Hd, dh, dW):
    import torch
    M, k = cfg.batch * cfg.top_k, cfg.top_k
    scratch = E.alloc_workspace(E.eagle_lmhead_topk_scratch_bytes(cfg))
    scratch.fill_(0xA5)  # stale partials must never be read
    lse = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((M, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda")
    E.eagle_lmhead_topk(cfg, ws, Hd, dh, dW, scratch, lse, ids, vals)
    torch.cuda.synchronize()
    assert E.eagle_status_fetch(ws) == 0
    return H.to_host(lse), H.to_host(ids), H.to_host(vals)


def _check_fused(logits, lse, ids, vals, k, rows=None):
    """Stage 1 of every (or each listed) row of the unfused kernel's logits."""
    lg = synth.bf16_to_f32(logits) if logits.dtype == np.uint16 else logits
    for r in (range(logits.shape[0]) if rows is None else rows):
        lse64, _, top = oracle.row_stats(np.ascontiguousarray(logits[r]), k)
        assert (ids[r] == top).all(), (r, ids[r], top)
        assert (vals[r] == lg[r][top]).all(), r
        assert abs(float(lse[r]) - lse64) <= 1e-5, (r, float(lse[r]), lse64)


@pytest.mark.parametrize("B,k,V,Hd,dtype", [
    (1, 10, 1000, 256, synth.F32),     # ragged last vocabulary tile (104 live entries)
    (1, 10, 1000, 200, synth.BF16),
    (30, 10, 2056, 512, synth.F32),    # three row blocks of 128, the last 44 rows live
    (2, 10, 40000, 64, synth.F32),     # 313 vocabulary tiles: two or three per CTA (64-bit list keys)
    (1, 1, 136, 64, synth.F32),        # k = 1, 8-entry last tile
    (64, 10, 4096, 128, synth.BF16),   # 640 rows: three chunks of 224
    (2, 16, 384, 1024, synth.BF16),    # k = 16
    (8, 8, 2056, 8192, synth.BF16),    # 70B shape
    (1, 10, 32000, 5120, synth.BF16),  # 13B shape
    (1, 16, 24, 64, synth.BF16),       # vocabulary barely above k: one partial tile
])
def test_fused_stage1_matches_oracle(B, k, V, Hd, dtype):
    E = _E()
    cfg = E.TreeCfg(B, V, k, 1, 1, 0.0, dtype, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h, W = _inputs(B * k, V, Hd, seed=V + Hd + 1)
    dh, dW = H.to_dev(h), H.to_dev(W)
    got = _lmhead(E, cfg, ws, Hd, dh, dW)
    _check(got, h, W, dtype)
    lse, ids, vals = _fused(E, cfg, ws, Hd, dh, dW)
    _check_fused(got, lse, ids, vals, k)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_fused_stage1_ties_and_constant_rows(dtype):
    """Equal logits in different tiles, warps and CTAs (duplicated weight rows
    scaled to the top) resolve to the lower id; a zero hidden row makes every
    logit 0 (top-k = ids 0..k-1, lse = log V)."""
    E = _E()
    B, k, V, Hd = 3, 8, 9000, 128
    cfg = E.TreeCfg(B, V, k, 1, 1, 0.0, dtype, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h, W = _inputs(B * k, V, Hd, seed=77)
    h[1] = 0                                  # a constant row
    dup = [8999, 17, 4200, 130, 96, 5000]     # one weight row repeated across tiles and CTAs
    for d in dup[1:]:
        W[d] = W[dup[0]]
    # times 4, exact in bf16: the top entries of about half the rows
    W[dup] = ((synth.bf16_to_f32(W[dup]) * np.float32(4.0)).view(np.uint32) >> 16).astype(np.uint16)
    dh, dW = H.to_dev(h), H.to_dev(W)
    got = _lmhead(E, cfg, ws, Hd, dh, dW)
    _check(got, h, W, dtype)
    lse, ids, vals = _fused(E, cfg, ws, Hd, dh, dW)
    _check_fused(got, lse, ids, vals, k)
    assert (ids[1] == np.arange(k)).all() and abs(float(lse[1]) - np.log(V)) <= 1e-5


@pytest.mark.parametrize("B", [1, 64])
def test_fused_stage1_full_size(llama8b_head, B):
    """Llama-8B head (V = 128256, H = 4096, k = 10) at batch 1 and 64: every
    row's stage 1 against the oracle on the unfused kernel's logits."""
    E = _E()
    V, Hd, W, dW = llama8b_head
    k = 10
    cfg = E.TreeCfg(B, V, k, 6, 60, 0.0, synth.BF16, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h = synth.normal4((B * k, Hd), synth.BF16, 1.0, B + 100, synth.STREAM_HIDDEN)
    dh = H.to_dev(h)
    got = _lmhead(E, cfg, ws, Hd, dh, dW)
    cols = np.unique(np.concatenate([[0, 127, 128, V - 1], np.random.default_rng(B).integers(0, V, 29)]))
    _check(np.ascontiguousarray(got[:, cols]), h, np.ascontiguousarray(W[cols]), synth.BF16)
    lse, ids, vals = _fused(E, cfg, ws, Hd, dh, dW)
    _check_fused(got, lse, ids, vals, k)


def test_fused_head_feeds_expand_topk():
    """A draft step from the fused head: eagle_expand_topk on its outputs
    equals the oracle's expansion of the unfused logits with the same lse."""
    import torch
    E = _E()
    B, k, V, Hd = 2, 4, 4104, 256
    cfg = E.TreeCfg(B, V, k, 1, 4, 0.0, synth.BF16, 0)
    ws = E.alloc_workspace(E.eagle_workspace_bytes(cfg))
    h, W = _inputs(B * k, V, Hd, seed=6)
    dh, dW = H.to_dev(h), H.to_dev(W)
    E.eagle_tree_init(cfg, ws)
    lg = _lmhead(E, cfg, ws, Hd, dh, dW).reshape(B, k, V)
    lse, ids, vals = _fused(E, cfg, ws, Hd, dh, dW)
    t = oracle.Tree(oracle.TreeCfg(B, V, k, 1, 4, 0.0, 0))
    ftok_o, fcnt_o = t.expand(0, lg, lse_in=lse.reshape(B, k))[:2]
    i32 = dict(dtype=torch.int32, device="cuda")
    row_lse = torch.empty(B, 1, k, dtype=torch.float32, device="cuda")
    ftok, fcnt = torch.empty(B, k, **i32), torch.empty(B, **i32)
    E.eagle_expand_topk(cfg, ws, 0, H.to_dev(ids), H.to_dev(vals), H.to_dev(lse), row_lse, ftok, fcnt)
    torch.cuda.synchronize()
    assert (H.to_host(fcnt) == fcnt_o).all()
    assert (H.to_host(ftok) == ftok_o).all()
    assert E.eagle_status_fetch(ws) == 0

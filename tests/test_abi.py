"""The C-ABI library: it loads, exports every entry point include/eagle.h
declares, and its host-side argument checks reject bad calls before any
launch (no GPU needed: a rejected call touches no CUDA API)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def E():
    from speculative_decoding_dynamic_gb300 import build
    build.build()
    from speculative_decoding_dynamic_gb300 import eagle
    return eagle


def test_header_declares_the_six_stage_calls():
    names = _declared()
    for n in ("eagle_expand", "eagle_rerank", "eagle_build_tree", "eagle_tree_attention", "eagle_verify",
              "eagle_kv_compact"):
        assert n in names


def test_library_exports_every_declared_symbol(E):
    lib = ctypes.CDLL(E.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(E, **kw):
    base = dict(batch=2, vocab=1024, top_k=4, depth=3, node_budget=10, threshold=0.0, logit_dtype=E.EAGLE_F32)
    base.update(kw)
    return E.TreeCfg(**base)


def test_workspace_bytes_and_invalid_configs(E):
    assert E.eagle_workspace_bytes(_cfg(E)) > 0
    assert E.eagle_workspace_bytes(_cfg(E, top_k=0)) == 0
    assert E.eagle_workspace_bytes(_cfg(E, top_k=17)) == 0
    assert E.eagle_workspace_bytes(_cfg(E, depth=17)) == 0
    assert E.eagle_workspace_bytes(_cfg(E, node_budget=256)) == 0  # T = 257 > 256
    assert E.eagle_workspace_bytes(_cfg(E, node_budget=255)) > 0
    assert E.eagle_workspace_bytes(_cfg(E, top_k=16, depth=5)) == 0  # C = 16 + 4*256 > 1024
    assert E.eagle_workspace_bytes(_cfg(E, vocab=1001)) == 0  # row not 16-byte aligned in fp32
    assert E.eagle_workspace_bytes(_cfg(E, vocab=1000)) > 0
    assert E.eagle_workspace_bytes(_cfg(E, vocab=3, top_k=4)) == 0
    assert E.eagle_workspace_bytes(_cfg(E, logit_dtype=7)) == 0
    for pol in (0, 1, 2, 3):
        assert E.eagle_workspace_bytes(_cfg(E, policy=pol)) > 0
    assert E.eagle_workspace_bytes(_cfg(E, policy=4)) == 0
    assert E.eagle_workspace_bytes(_cfg(E, policy=-1)) == 0


def test_calls_reject_bad_arguments_before_launch(E):
    cfg = _cfg(E)
    P = ctypes.c_void_p
    ws_bytes = E.eagle_workspace_bytes(cfg)
    fake_ws = P(1 << 20)  # aligned, never dereferenced: every call below fails its checks first
    bad_ws = P((1 << 20) + 16)
    ptr = P(1 << 21)
    r = E.raw_call
    assert r("eagle_tree_init", ctypes.byref(cfg), None, ws_bytes, None) == -4
    assert r("eagle_tree_init", ctypes.byref(cfg), bad_ws, ws_bytes, None) == -4
    assert r("eagle_tree_init", ctypes.byref(cfg), fake_ws, ws_bytes - 1, None) == -4
    assert r("eagle_expand", ctypes.byref(cfg), fake_ws, ws_bytes, 3, ptr, None, ptr, ptr, ptr, None) == -1
    assert r("eagle_expand", ctypes.byref(cfg), fake_ws, ws_bytes, -1, ptr, None, ptr, ptr, ptr, None) == -1
    assert r("eagle_expand", ctypes.byref(cfg), fake_ws, ws_bytes, 0, None, None, ptr, ptr, ptr, None) == -1
    assert r("eagle_expand", ctypes.byref(cfg), fake_ws, ws_bytes, 0, P((1 << 21) + 4), None, ptr, ptr, ptr,
             None) == -2
    u64 = ctypes.c_uint64
    one = ctypes.c_float(1.0)
    assert r("eagle_verify", ctypes.byref(cfg), fake_ws, ws_bytes, 5, one, u64(1), u64(0), ptr, None, ptr, ptr, ptr,
             ptr, ptr, ptr, None) == -1
    assert r("eagle_verify", ctypes.byref(cfg), fake_ws, ws_bytes, 1, ctypes.c_float(0.0), u64(1), u64(0), ptr, None,
             ptr, ptr, ptr, ptr, ptr, ptr, None) == -1
    assert r("eagle_verify", ctypes.byref(cfg), fake_ws, ws_bytes, 0, one, u64(1), u64(0), None, None, ptr, ptr, ptr,
             ptr, ptr, ptr, None) == -1
    assert r("eagle_verify", ctypes.byref(cfg), fake_ws, ws_bytes, 0, one, u64(1), u64(0), P((1 << 21) + 4), None,
             ptr, ptr, ptr, ptr, ptr, ptr, None) == -2
    assert r("eagle_test_expand_starved", ctypes.byref(cfg), fake_ws, ws_bytes, 3, ptr, ptr, ptr, ptr, None) == -1
    assert r("eagle_lmhead", ctypes.byref(cfg), fake_ws, ws_bytes, 4096, None, ptr, ptr, None) == -1
    assert r("eagle_lmhead", ctypes.byref(cfg), fake_ws, ws_bytes, 0, ptr, ptr, ptr, None) == -1
    assert r("eagle_lmhead", ctypes.byref(cfg), fake_ws, ws_bytes, 4100, ptr, ptr, ptr, None) == -2  # H % 8
    assert r("eagle_lmhead", ctypes.byref(cfg), fake_ws, ws_bytes, 4096, ptr, P((1 << 21) + 8), ptr, None) == -2
    assert r("eagle_lmhead", ctypes.byref(cfg), None, ws_bytes, 4096, ptr, ptr, ptr, None) == -4
    sb = E.eagle_lmhead_topk_scratch_bytes(cfg)
    assert sb > 0
    fake_sc = P(1 << 22)
    lm = lambda ws_, H_, hid, sc, sbytes: r("eagle_lmhead_topk", ctypes.byref(cfg), ws_, ws_bytes, H_, hid, ptr, sc,
                                            sbytes, ptr, ptr, ptr, None)
    assert lm(fake_ws, 4096, None, fake_sc, sb) == -1
    assert lm(fake_ws, 0, ptr, fake_sc, sb) == -1
    assert lm(fake_ws, 4100, ptr, fake_sc, sb) == -2  # H % 8
    assert lm(fake_ws, 4096, P((1 << 21) + 8), fake_sc, sb) == -2
    assert lm(fake_ws, 4096, ptr, None, sb) == -4
    assert lm(fake_ws, 4096, ptr, P((1 << 22) + 128), sb) == -4
    assert lm(fake_ws, 4096, ptr, fake_sc, sb - 1) == -4
    assert lm(None, 4096, ptr, fake_sc, sb) == -4
    big = E.TreeCfg(2048, 32000, 16, 4, 60, 0.0, E.EAGLE_BF16, 0)  # B*k = 32768 rows
    assert r("eagle_lmhead_topk", ctypes.byref(big), fake_ws, E.eagle_workspace_bytes(big), 4096, ptr, ptr, fake_sc,
             E.eagle_lmhead_topk_scratch_bytes(big), ptr, ptr, ptr, None) == -2
    kv = E.KvCfg(2, 8, 3, 64, 4, 100, E.EAGLE_BF16, 0, 0, 0, 192)  # 8 % 3 != 0
    assert r("eagle_tree_attention", ctypes.byref(kv), 9, ptr, ptr, 0, ptr, ptr, ptr, ptr, fake_ws, 4096, None) == -1
    kv = E.KvCfg(2, 8, 2, 64, 4, 100, E.EAGLE_BF16, 4 * 2 * 100 * 128, 2 * 100 * 128, 100 * 128, 128)
    assert r("eagle_tree_attention", ctypes.byref(kv), 300, ptr, ptr, 0, ptr, ptr, ptr, ptr, fake_ws, 4096,
             None) == -1
    assert r("eagle_tree_attention", ctypes.byref(kv), 9, ptr, ptr, 0, ptr, ptr, ptr, ptr, None, 4096, None) == -4
    kv_odd = E.KvCfg(2, 8, 2, 60, 4, 100, E.EAGLE_BF16, 4 * 2 * 100 * 120, 2 * 100 * 120, 100 * 120, 121)
    assert r("eagle_kv_compact", ctypes.byref(kv_odd), ptr, ptr, ptr, ptr, 7, ptr, None, None) == -2
    assert r("eagle_kv_compact", ctypes.byref(kv), ptr, ptr, ptr, ptr, 0, ptr, None, None) == -1


def test_status_strings(E):
    for code in range(-6, 1):
        assert E._lib.eagle_status_string(code)


def test_static_verify_rejects_what_its_fixed_scratch_cannot_hold(E):
    """eagle_verify_static's size limits, checked before any CUDA call (the
    pointers are never dereferenced: every call here is rejected first)."""
    P = ctypes.c_void_p
    p = P(1 << 20)
    u64 = ctypes.c_uint64
    one = ctypes.c_float(1.0)

    def call(cfg, mode):
        return E.raw_call("eagle_verify_static", ctypes.byref(cfg), mode, one, u64(1), u64(0), p, p, p, p, p, p, p,
                          None)

    assert call(E.TreeCfg(80, 1024, 4, 3, 60, 0.0, E.EAGLE_F32), 0) == -2  # 80 * 61 rows > 4096
    assert call(E.TreeCfg(1025, 1024, 4, 3, 1, 0.0, E.EAGLE_F32), 0) == -2  # batch > 1024
    assert call(E.TreeCfg(80, 128256, 4, 3, 60, 0.0, E.EAGLE_BF16), 1) == -2  # lossless: the same row limit
    assert call(E.TreeCfg(2, 1024, 4, 3, 10, 0.0, E.EAGLE_F32), 7) == -1  # unknown mode
    assert call(E.TreeCfg(2, 1024, 0, 3, 10, 0.0, E.EAGLE_F32), 0) == -1  # invalid tree
    assert E.raw_call("eagle_verify_static", ctypes.byref(E.TreeCfg(2, 1024, 4, 3, 10, 0.0, E.EAGLE_F32)), 1,
                      ctypes.c_float(0.0), u64(1), u64(0), p, p, p, p, p, p, p, None) == -1  # temperature 0

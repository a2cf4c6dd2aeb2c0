"""Host-side models of selection rules the CUDA kernels rely on (CPU only).

The expansion kernel finds a row segment's top-k without ranking every
element: it admits only the lane groups (32 elements) whose maximum reaches
an admission key tau (the largest over warps of the warp's k-th largest lane
maximum), and for bf16 rows it keeps just the top 16 order bits of each group
maximum. This models that rule on the kernel's data layout and checks that
the admitted keys always contain the exact top-k (value descending, equal
values by lower id), on random rows, heavy ties, negative rows, -inf entries
and a ragged tail. It does not run or import any CUDA code. The end of the
file models two rules of the LM head with stage 1 in its epilogue (its
32-bit list keys and its merge's candidate bound).
"""
import numpy as np
import pytest

import synth

CHUNK = 8192          # bf16 elements per 16 KB chunk
WARPS, J, LANES, E = 8, 4, 32, 8


def _f2o(x):
    b = x.astype(np.float32).view(np.uint32).copy()
    b[(b & 0x7FFFFFFF) == 0] = 0
    neg = (b & 0x80000000) != 0
    return np.where(neg, ~b, b | 0x80000000).astype(np.uint32)


def _keys(o, ids):
    return (o.astype(np.uint64) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ids.astype(np.uint64))


def _admitted_topk(bits, k):
    """The kernel's rule on one segment of bf16 bit patterns (uint16)."""
    n = bits.size
    nch = (n + CHUNK - 1) // CHUNK
    x = np.full(nch * CHUNK, -np.inf, np.float32)
    x[:n] = synth.bf16_to_f32(bits)
    ids = np.arange(nch * CHUNK, dtype=np.int64)
    real = ids < n
    xv = x.reshape(nch, WARPS, J, LANES, E)
    group_max = xv.max(axis=(2, 4))                          # [chunk, warp, lane]
    first_vec = (np.arange(WARPS)[:, None] * (J * LANES) + np.arange(LANES)[None, :]) * E
    has = (np.arange(nch)[:, None, None] * CHUNK + first_vec[None]) < n
    gm_o = np.where(has, _f2o(group_max), 0).astype(np.uint32)
    gm16 = (gm_o >> 16).astype(np.uint32)                   # bf16 rows keep 16 bits
    lane_max = group_max.max(axis=0)                          # [warp, lane]
    lane_has = has.any(axis=0)
    lane_o = np.where(lane_has, _f2o(lane_max), 0).astype(np.uint32)
    kth = np.sort(lane_o, axis=1)[:, ::-1][:, k - 1]           # warp's k-th largest lane maximum
    tau = int(kth.max())
    if tau == 0:
        hot = gm16 != 0
    else:
        hot = (gm16 != 0) & ((gm16 << 16) >= (tau & 0xFFFF0000))
    hot_el = np.broadcast_to(hot[:, :, None, :, None], xv.shape).reshape(-1)
    keys = _keys(_f2o(x), ids)
    ok = hot_el & real & ~np.isnan(x) & (keys >= (np.uint64(tau) << np.uint64(32)))
    cand = np.sort(keys[ok])[::-1][:k]
    return cand, int(ok.sum())


def _true_topk(bits, k):
    x = synth.bf16_to_f32(bits)
    ids = np.arange(bits.size)
    keys = _keys(_f2o(x), ids)
    return np.sort(keys[~np.isnan(x)])[::-1][:k]


def _bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("n", [16 * CHUNK, 128256, 9 * CHUNK + 1000])
@pytest.mark.parametrize("k", [1, 10, 16])
def test_admission_key_keeps_the_exact_topk(n, k):
    rng = np.random.default_rng(n + k)
    cases = [
        _bf16(rng.normal(0, 2.5, n)),                            # the workloads' rows
        _bf16(rng.integers(-3, 3, n).astype(np.float32)),        # six distinct values: ties everywhere
        _bf16(-np.abs(rng.normal(0, 1, n)) - 1.0),               # every value negative
        _bf16(np.where(rng.random(n) < 0.9, -np.inf, rng.normal(0, 1, n))),  # mostly -inf
        _bf16(np.full(n, 0.5, np.float32)),                      # one value
    ]
    for bits in cases:
        got, admitted = _admitted_topk(bits, k)
        want = _true_topk(bits, k)
        assert np.array_equal(got, want)
        assert admitted >= min(k, int((~np.isnan(synth.bf16_to_f32(bits))).sum()))


def test_input_generator_philox_known_answers():
    """The seeded input generator's Philox4x32-10 against the known-answer
    vectors published with the Random123 library (counter, key -> output)."""
    kat = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, out in kat:
        assert list(synth.philox(ctr, key)) == out


# Device arithmetic of sampled drafting, compiled for the host from the same
# header (every operation an explicit round-to-nearest step, so the host twin
# reaches the device's bits): bit-exact against the oracle's own logarithm and
# Gumbel noise, and against the input generator's Philox.

_SHIM = r"""
#include "sampling.cuh"
extern "C" void t_log(int n, const float* y, float* o) { for (int i = 0; i < n; ++i) o[i] = eagle::sampling::fixed_log(y[i]); }
extern "C" void t_gumbel(int n, const unsigned* w, float* o) { for (int i = 0; i < n; ++i) o[i] = eagle::sampling::gumbel_of_word(w[i]); }
extern "C" void t_philox(const unsigned* c, const unsigned* k, unsigned* o) { eagle::sampling::philox4x32_10(c, k[0], k[1], o); }
"""


@pytest.fixture(scope="module")
def sampling_host(tmp_path_factory):
    import ctypes
    import os
    import subprocess
    d = tmp_path_factory.mktemp("sampling")
    src = d / "shim.cpp"
    src.write_text(_SHIM)
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "speculative_decoding_dynamic_gb300", "csrc")
    lib = d / "shim.so"
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-I", csrc, str(src), "-o",
                    str(lib)], check=True)
    return ctypes.CDLL(str(lib))


def test_sampling_arithmetic_matches_the_oracle_bit_for_bit(sampling_host):
    import ctypes
    import oracle
    rng = np.random.default_rng(3)
    y = np.concatenate([np.exp2(rng.uniform(-24, 12, 50000)), 1 + rng.uniform(-0.01, 0.01, 20000)]).astype(np.float32)
    got = np.empty_like(y)
    sampling_host.t_log(y.size, y.ctypes.data_as(ctypes.c_void_p), got.ctypes.data_as(ctypes.c_void_p))
    assert np.array_equal(got.view(np.uint32), oracle.dlog(y).view(np.uint32))
    w = synth.words(1, 100000, 0, 9, synth.STREAM_GUMBEL).reshape(-1)
    w = np.concatenate([w, np.uint32([0, 1, 511, 512, 0xFFFFFFFF, 0x80000000])])
    g = np.empty(w.size, np.float32)
    sampling_host.t_gumbel(w.size, w.ctypes.data_as(ctypes.c_void_p), g.ctypes.data_as(ctypes.c_void_p))
    assert np.array_equal(g.view(np.uint32), oracle.gumbel(w).view(np.uint32))


def test_sampling_philox_matches_the_input_generator(sampling_host):
    import ctypes
    rng = np.random.default_rng(4)
    for _ in range(200):
        c = rng.integers(0, 1 << 32, 4, dtype=np.uint64).astype(np.uint32)
        k = rng.integers(0, 1 << 32, 2, dtype=np.uint64).astype(np.uint32)
        o = np.zeros(4, np.uint32)
        sampling_host.t_philox(c.ctypes.data_as(ctypes.c_void_p), k.ctypes.data_as(ctypes.c_void_p),
                               o.ctypes.data_as(ctypes.c_void_p))
        assert np.array_equal(o, synth.philox(c, k))


# ----------------------------------------------- LM head with stage 1 ---
#
# Models of two rules of eagle_lmhead_topk. (1) An epilogue thread keeps its
# row's best keys as 32-bit words for bf16 logits: the top 16 order bits of
# the value, then 0xFFFF minus the entry's position in the CTA's scan (which
# grows with the token id), so a larger word is a larger value, then a lower
# id, and the value decodes exactly. (2) The merge keeps, among the CTAs'
# sorted k-key lists, the keys at or above max(largest k-th key, k-th largest
# first key); that set must hold the row's whole top-k.

def _list_key(bits16, pos):
    o = _f2o(synth.bf16_to_f32(bits16))
    return (o & np.uint32(0xFFFF0000)) | (np.uint32(0xFFFF) - pos.astype(np.uint32))


def _list_val(word):
    hi = word & np.uint32(0xFFFF0000)
    o = hi | np.where((hi & np.uint32(0x80000000)) != 0, np.uint32(0), np.uint32(0xFFFF))
    b = np.where((o & np.uint32(0x80000000)) != 0, o & np.uint32(0x7FFFFFFF), ~o).astype(np.uint32)
    return b.view(np.float32)


def test_bf16_list_keys_order_like_value_then_lower_id_and_decode_exactly():
    rng = np.random.default_rng(3)
    special = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x3F80, 0xBF80, 0x0001, 0x8001, 0x7F7F, 0xFF7F],
                       np.uint16)  # +0, -0, +inf, -inf, +1, -1, denormals, max finite
    bits = np.concatenate([special, rng.integers(0, 1 << 16, 3000).astype(np.uint16),
                           np.repeat(np.uint16(0x4100), 40)])  # runs of equal values
    bits = bits[((bits & 0x7F80) != 0x7F80) | ((bits & 0x007F) == 0)]  # no NaN patterns
    pos = rng.permutation(bits.size).astype(np.int64)  # distinct scan positions < 2^16
    words = _list_key(bits, pos)
    x = synth.bf16_to_f32(bits).astype(np.float64)
    x[x == 0] = 0.0  # -0 and +0 are one value
    order_words = np.argsort(-words.astype(np.int64), kind="stable")
    order_ref = np.lexsort((pos, -x))  # value descending, then lower position
    assert (order_words == order_ref).all()
    dec = _list_val(words)
    same = (dec == synth.bf16_to_f32(bits)) | ((dec == 0) & (synth.bf16_to_f32(bits) == 0))
    assert same.all()


def _merge_candidates(lists, k):
    """Keys the merge kernel ranks: >= max(largest k-th key, k-th largest first key)."""
    kth = max(int(l[k - 1]) for l in lists)
    firsts = sorted((int(l[0]) for l in lists), reverse=True)
    kth_first = firsts[k - 1] if len(firsts) >= k and firsts[k - 1] != 0 else 0
    th = max(kth, kth_first)
    return [int(x) for l in lists for x in l if x != 0 and x >= th]


@pytest.mark.parametrize("case", ["random", "one_partial_holds_all", "identical_partials", "sparse", "few_keys"])
@pytest.mark.parametrize("S,k", [(152, 10), (30, 16), (4, 8), (3, 1)])
def test_merge_bound_keeps_the_whole_topk(case, S, k):
    rng = np.random.default_rng(S * 100 + k)
    n_per = 200
    vals = rng.normal(size=(S, n_per)).astype(np.float32)
    if case == "one_partial_holds_all":
        vals[0] += 10.0
    elif case == "identical_partials":
        vals[:] = vals[0]
    elif case == "sparse":
        vals[rng.random(vals.shape) < 0.97] = -np.inf
    ids = np.arange(S * n_per).reshape(S, n_per)
    keys = _keys(_f2o(vals.reshape(-1)), ids.reshape(-1)).reshape(S, n_per)
    if case == "few_keys":  # partials with fewer than k entries (zero padding)
        keys[:, max(1, k // 2):] = 0
    lists = [np.concatenate([np.sort(r[r != 0])[::-1], np.zeros(k, np.uint64)])[:k] for r in keys]
    everything = np.sort(keys[keys != 0].reshape(-1))[::-1][:k]
    cand = np.sort(np.array(_merge_candidates(lists, k), np.uint64))[::-1][:k]
    assert np.array_equal(cand, everything)

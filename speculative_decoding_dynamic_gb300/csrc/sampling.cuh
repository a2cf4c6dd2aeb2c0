// Counter-based uniforms and Gumbel keys for sampled drafting: children of a
// draft row drawn from its softmax without replacement (the Gumbel-top-k
// identity: perturb each logit by independent Gumbel noise, keep the k
// largest; their order is the order of sequential draws). Device code for
// sm_103a with a host twin of the same operations, so that the host can
// check the device arithmetic bit for bit. Not part of the public ABI.
//
// Philox4x32-10 is written from its published definition (Salmon, Moraes,
// Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): per
// round, two 32x32->64 multiplies by 0xD2511F53 (word 0) and 0xCD9E8D57
// (word 2), new words (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0), then the key
// bumped by 0x9E3779B9 / 0xBB67AE85; ten rounds.
//
// fixed_log is the natural logarithm of a positive normal float as a fixed
// sequence of correctly rounded fp32 operations: y = m 2^e with m in
// [sqrt(1/2), sqrt(2)) (bit operations), s = (m - 1) / (m + 1), ln m =
// 2 atanh(s) = 2 s (1 + s^2/3 + s^4/5 + s^6/7 + s^8/9 + s^10/11) by Horner
// steps in s^2 (fused multiply-adds), ln y = e ln2_hi + (e ln2_lo + ln m)
// with ln 2 = 0x1.62e4p-1 + 0x1.7f7d1cp-20 (e ln2_hi exact). Every operation
// is an explicit round-to-nearest intrinsic, so the compiler contracts
// nothing and the host twin (std::fma, IEEE division) reaches the same bits.

#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define EAGLE_SAMPLING_FN __host__ __device__ __forceinline__
#else
#define EAGLE_SAMPLING_FN inline
#endif

namespace eagle {
namespace sampling {

EAGLE_SAMPLING_FN float rn_fma(float a, float b, float c) {
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fma(a, b, c);
#endif
}
EAGLE_SAMPLING_FN float rn_mul(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
EAGLE_SAMPLING_FN float rn_add(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}
EAGLE_SAMPLING_FN float rn_sub(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}
EAGLE_SAMPLING_FN float rn_div(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fdiv_rn(a, b);
#else
    return a / b;
#endif
}
EAGLE_SAMPLING_FN uint32_t bits_of(float x) {
#if defined(__CUDA_ARCH__)
    return __float_as_uint(x);
#else
    uint32_t b;
    std::memcpy(&b, &x, 4);
    return b;
#endif
}
EAGLE_SAMPLING_FN float float_of(uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __uint_as_float(b);
#else
    float x;
    std::memcpy(&x, &b, 4);
    return x;
#endif
}

// out = Philox4x32-10(counter c, key (k0, k1)).
EAGLE_SAMPLING_FN void philox4x32_10(const uint32_t c_in[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
    uint32_t c0 = c_in[0], c1 = c_in[1], c2 = c_in[2], c3 = c_in[3];
#if defined(__CUDA_ARCH__)
#pragma unroll
#endif
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
        const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
        const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
        c0 = n0;
        c1 = static_cast<uint32_t>(p1);
        c2 = n2;
        c3 = static_cast<uint32_t>(p0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// Natural logarithm of a positive normal float (see the file comment).
EAGLE_SAMPLING_FN float fixed_log(float y) {
    const uint32_t b = bits_of(y);
    int e = static_cast<int>((b >> 23) & 0xffu) - 127;
    float m = float_of((b & 0x7fffffu) | 0x3f800000u);  // [1, 2)
    if (m > 1.41421353816986083984375f) {               // fp32 below sqrt(2): halve (exact)
        m = rn_mul(m, 0.5f);
        e += 1;
    }
    const float s = rn_div(rn_sub(m, 1.0f), rn_add(m, 1.0f));
    const float z = rn_mul(s, s);
    float p = 1.0f / 11.0f;
    p = rn_fma(p, z, 1.0f / 9.0f);
    p = rn_fma(p, z, 1.0f / 7.0f);
    p = rn_fma(p, z, 1.0f / 5.0f);
    p = rn_fma(p, z, 1.0f / 3.0f);
    p = rn_fma(p, z, 1.0f);
    float t = rn_mul(s, p);
    t = rn_add(t, t);
    const float ef = static_cast<float>(e);
    return rn_fma(ef, 0x1.62e4p-1f, rn_fma(ef, 0x1.7f7d1cp-20f, t));
}

// Gumbel noise of a uniform word: u = ((w >> 9) + 1/2) 2^-23, exact and
// strictly inside (0, 1); g = -ln(-ln u).
EAGLE_SAMPLING_FN float gumbel_of_word(uint32_t w) {
    const float u = rn_mul(rn_add(static_cast<float>(w >> 9), 0.5f), 0x1p-23f);
    return -fixed_log(-fixed_log(u));
}

}  // namespace sampling
}  // namespace eagle

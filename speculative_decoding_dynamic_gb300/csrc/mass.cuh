// Exact integer probability masses of lossless verification (device code for
// sm_103a; not part of the public ABI). A mass is floor(dexp((x - m) / T)
// 2^40) with dexp the fixed-order exp of the contract in eagle.h.
#pragma once

#include <cstdint>

#include "eagle_internal.cuh"

namespace eagle {

// Fixed-order exp for lossless verification (contract in eagle.h): Cody-Waite
// reduction with ln2 = 0x1.62e4p-1 + 0x1.7f7d1cp-20, degree-7 Taylor series of
// exp(r) in Horner form, exact scaling by 2^n. Every step is one correctly
// rounded fp32 operation: n = z log2(e) rounded to nearest-even by one fused
// multiply-add with 1.5 * 2^23, then fused multiply-adds for the reduction and
// each Horner step. z <= 0. Returns p and the exponent n (value p * 2^n),
// p = 0 below -32.
__device__ __forceinline__ float dexp_parts(float z, int& n_out) {
    if (!(z >= -32.0f)) {
        n_out = 0;
        return 0.0f;
    }
    const float t = __fmaf_rn(z, 0x1.715476p+0f, 12582912.0f);  // 1.5 * 2^23 + nearest integer
    const float n = __fsub_rn(t, 12582912.0f);
    n_out = __float_as_int(t) - 0x4B400000;
    float r = __fmaf_rn(-n, 0x1.62e4p-1f, z);
    r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
    float p = 0x1.a01a02p-13f;              // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
    p = __fmaf_rn(p, r, 0.5f);             // 1/2!
    p = __fmaf_rn(p, r, 1.0f);             // 1/1!
    p = __fmaf_rn(p, r, 1.0f);             // 1/0!
    return p;
}

// Integer mass floor(dexp((x - m) * inv_t) * 2^40) = floor(p * 2^(n + 40)):
// p's 24-bit significand shifted by (its exponent + n + 17), an exact
// integer operation (the float product would be exact as well).
__device__ __forceinline__ uint64_t fixed_mass(float x, float m, float inv_t) {
    int n;
    const float p = dexp_parts(__fmul_rn(__fsub_rn(x, m), inv_t), n);
    const uint32_t bits = __float_as_uint(p);
    const uint32_t sig = (bits & 0x7FFFFFu) | 0x800000u;
    const int sh = static_cast<int>(bits >> 23) - 127 + n + 17;
    if (p == 0.0f || sh <= -24) return 0ull;
    return sh >= 0 ? static_cast<uint64_t>(sig) << sh : static_cast<uint64_t>(sig >> (-sh));
}

__device__ __forceinline__ uint64_t f2_add_rz(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The masses of two elements at once, in two parts. The fixed-order exp's
// fp32 operations run as packed pairs (each lane of a pair rounds exactly as
// the scalar operation). Per element the mass is floor(f), f = p * 2^(n + 40)
// < 2^41: n + 40 added to p's exponent field (exact: a normal float for
// every argument in [-32, 0]); then hi = rz(f + 2^46) - 2^46 = floor(f / 2^23)
// 2^23 and b = f - hi (both exact), lo = rz(b + 2^23) - 2^23 = floor(b), so
// floor(f) = floor(f / 2^23) 2^23 + floor(b). The two parts of both elements
// are added to *ahi (in units of 2^23, the float bits of rz(f + 2^46)
// minus those of 2^46) and *alo (the bits of rz(b + 2^23) minus those of
// 2^23). Arguments below -32 are clamped to -32, whose mass exp(-32) 2^40 < 1
// is 0 as the definition's is for them. Equal to fixed_mass of each element.
__device__ __forceinline__ void pair_mass_parts(float x0, float x1, uint64_t neg_m2, uint64_t inv_t2, uint32_t& ahi,
                                                uint32_t& alo) {
    uint64_t z = f2_mul(f2_add(f2_pack(x0, x1), neg_m2), inv_t2);
    z = f2_pack(fmaxf(f2_lo(z), -32.0f), fmaxf(f2_hi(z), -32.0f));
    const uint64_t t = f2_fma(z, f2_pack(0x1.715476p+0f, 0x1.715476p+0f), f2_pack(12582912.0f, 12582912.0f));
    const uint64_t n = f2_add(t, f2_pack(-12582912.0f, -12582912.0f));
    uint64_t r = f2_fma(n, f2_pack(-0x1.62e4p-1f, -0x1.62e4p-1f), z);
    r = f2_fma(n, f2_pack(-0x1.7f7d1cp-20f, -0x1.7f7d1cp-20f), r);
    uint64_t p = f2_fma(f2_pack(0x1.a01a02p-13f, 0x1.a01a02p-13f), r, f2_pack(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = f2_fma(p, r, f2_pack(0x1.111112p-7f, 0x1.111112p-7f));
    p = f2_fma(p, r, f2_pack(0x1.555556p-5f, 0x1.555556p-5f));
    p = f2_fma(p, r, f2_pack(0x1.555556p-3f, 0x1.555556p-3f));
    p = f2_fma(p, r, f2_pack(0.5f, 0.5f));
    p = f2_fma(p, r, f2_pack(1.0f, 1.0f));
    p = f2_fma(p, r, f2_pack(1.0f, 1.0f));
    // t's low word is n (t = 1.5 * 2^23 + n, exact), so t << 23 = n << 23 modulo 2^32
    const uint32_t f0 = static_cast<uint32_t>(p) + (static_cast<uint32_t>(t) << 23) + (40u << 23);
    const uint32_t f1 = static_cast<uint32_t>(p >> 32) + (static_cast<uint32_t>(t >> 32) << 23) + (40u << 23);
    const uint64_t f = (static_cast<uint64_t>(f1) << 32) | f0;
    const uint64_t k46 = f2_pack(0x1p46f, 0x1p46f), k23 = f2_pack(0x1p23f, 0x1p23f);
    const uint64_t x46 = f2_add_rz(f, k46);                                  // 2^46 + floor(f / 2^23) 2^23
    const uint64_t b = f2_add(f, f2_add(k46, x46 ^ 0x8000000080000000ull));  // f - (x46 - 2^46), exact
    const uint64_t x23 = f2_add_rz(b, k23);                                  // 2^23 + floor(b)
    ahi += (static_cast<uint32_t>(x46) - 0x56800000u) + (static_cast<uint32_t>(x46 >> 32) - 0x56800000u);
    alo += (static_cast<uint32_t>(x23) - 0x4B000000u) + (static_cast<uint32_t>(x23 >> 32) - 0x4B000000u);
}

// The integer mass of the parts: ahi 2^23 + alo.
__device__ __forceinline__ uint64_t mass_of_parts(uint32_t ahi, uint32_t alo) {
    return (static_cast<uint64_t>(ahi) << 23) + alo;
}

// The masses of two elements, each on its own.
__device__ __forceinline__ void pair_mass2(float x0, float x1, uint64_t neg_m2, uint64_t inv_t2, uint64_t& m0,
                                           uint64_t& m1) {
    uint32_t h0 = 0, l0 = 0, h1 = 0, l1 = 0;
    pair_mass_parts(x0, -INFINITY, neg_m2, inv_t2, h0, l0);
    pair_mass_parts(x1, -INFINITY, neg_m2, inv_t2, h1, l1);
    m0 = mass_of_parts(h0, l0);
    m1 = mass_of_parts(h1, l1);
}

}  // namespace eagle

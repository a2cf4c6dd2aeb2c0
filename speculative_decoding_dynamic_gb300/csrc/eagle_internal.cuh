// Internal device helpers of libeagle (sm_103a). Not part of the public ABI.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_runtime.h>

namespace eagle {

namespace cg = cooperative_groups;

// ------------------------------------------- programmatic dependent launch ---
// Every kernel of the cycle is launched with programmatic stream
// serialisation: it lets the next kernel launch at once and waits for the
// previous one only where it first reads that kernel's results. Both are
// no-ops for a launch without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- status word ---
// Device-detected faults: the first error of a cycle wins (atomicCAS on 0).
enum DeviceError : int {
    kDevOk = 0,
    kDevNonFinite = 1,   // a logit row has a non-finite log-sum-exp / maximum
    kDevTimeout = 2,     // a bounded wait on an mbarrier gave up
    kDevBadIndex = 3,    // a token / slot / length out of range
    kDevOverflow = 4,    // a candidate or tree table would overflow
};

__device__ __forceinline__ void raise_status(int* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// Checked builds (EAGLE_DEBUG): an index that the release kernels take on
// trust from an earlier kernel (a node id read from the workspace, a slot
// from a scan) is tested before use; out of range, the status word gets
// kDevBadIndex and the caller skips the access. Release builds: always true.
__device__ __forceinline__ bool checked_index(bool ok, int* status) {
    if (!ok) raise_status(status, kDevBadIndex);
    return ok;
}
#ifdef EAGLE_DEBUG
#define EAGLE_CHECKED(cond, status) (::eagle::checked_index((cond), (status)))
#else
#define EAGLE_CHECKED(cond, status) (true)
#endif

// --------------------------------------------------------------- sort keys ---
// Float -> unsigned with the same order (-0 and +0 are one value).
__device__ __forceinline__ uint32_t f2o(float f) {
    uint32_t b = __float_as_uint(f);
    if ((b & 0x7fffffffu) == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float o2f(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
// 64-bit key: larger value first, then lower id. Unique per id.
__device__ __forceinline__ uint64_t make_key(float v, uint32_t id) {
    return (static_cast<uint64_t>(f2o(v)) << 32) | static_cast<uint32_t>(0xffffffffu - id);
}
__device__ __forceinline__ uint32_t key_id(uint64_t k) { return 0xffffffffu - static_cast<uint32_t>(k); }
__device__ __forceinline__ float key_val(uint64_t k) { return o2f(static_cast<uint32_t>(k >> 32)); }

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    lo = __shfl_xor_sync(0xffffffffu, lo, m);
    hi = __shfl_xor_sync(0xffffffffu, hi, m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    uint32_t lo = static_cast<uint32_t>(v), hi = static_cast<uint32_t>(v >> 32);
    lo = __shfl_sync(0xffffffffu, lo, src);
    hi = __shfl_sync(0xffffffffu, hi, src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        uint64_t o = shfl_xor_u64(v, m);
        v = o > v ? o : v;
    }
    return v;
}
// Bits of the lanes below this one.
__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += shfl_xor_u64(v, m);
    return v;
}

// Top-k of n unique keys held in shared memory, by one warp: k rounds of warp
// argmax, each round taking the largest key below the previous one. Writes
// out[0..k) (0 = no key). Cost O(k * n / 32) per lane; used for n <= a few
// hundred.
__device__ __forceinline__ void warp_topk_smem(const uint64_t* keys, int n, int k, uint64_t* out) {
    const int lane = threadIdx.x & 31;
    uint64_t prev = ~0ull;
    for (int r = 0; r < k; ++r) {
        uint64_t best = 0;
        for (int i = lane; i < n; i += 32) {
            uint64_t v = keys[i];
            if (v < prev && v > best) best = v;
        }
        best = warp_max_u64(best);
        if (lane == 0) out[r] = best;
        prev = best;
        if (best == 0) {
            for (int q = r + 1 + lane; q < k; q += 32) out[q] = 0;
            break;
        }
    }
    __syncwarp();
}

// -------------------------------------------------------------- fast exp2 ---
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs: (lo, hi) in one 64-bit register; two correctly rounded
// results per instruction, each equal to the scalar operation's.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// --------------------------------------------------- mbarrier + bulk copies ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase. Returns false after ~max_iter polls
// (each poll may suspend the thread for a hardware-chosen time).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter = (1u << 21)) {
    for (uint32_t i = 0; i < max_iter; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Bounded wait that lets the hardware suspend the thread (up to `hint_ns` per
// poll, woken early when the phase completes) instead of spinning: for
// waits that may be long, so that idle warps leave issue slots to the others.
// Returns false after max_iter polls.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t max_iter = (1u << 16),
                                                uint32_t hint_ns = 20000u) {
    for (uint32_t i = 0; i < max_iter; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// Bulk (non-tensor) copy global -> this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes. Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Hint: bring [src, src + bytes) into L2 (16-byte aligned, bytes a multiple
// of 16). Reads nothing into the CTA, so it may be issued before the
// programmatic-dependency wait: L2 is the point of coherence, a later write
// by the previous kernel still lands before the copy issued after the wait.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// The head of a row segment (at most its first two 16 KB chunks: enough to
// hide the first copies' latency without crowding L2 when many CTAs are in
// flight), one hint per 16 KB.
__device__ __forceinline__ void prefetch_l2_segment(const char* src, int bytes) {
    bytes = min(bytes, 2 * 16384);
    for (int off = 0; off < bytes; off += 16384) prefetch_l2(src + off, static_cast<uint32_t>(min(16384, bytes - off)));
}

// Global loads that bypass L1 (data written by other CTAs of the same launch).
__device__ __forceinline__ int ld_cg_i32(const int* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_cg_f32(const float* p) { return __ldcg(p); }

// Per-sequence ticket: add one at device scope with acquire-release
// semantics. The release covers the caller's writes and, being cumulative,
// the writes it observed through earlier barriers (its CTA's, its cluster's);
// the returned count acquires every earlier arrival's. Threads of the CTA
// that read those writes after a barrier following the call observe them.
__device__ __forceinline__ int ticket_add(int* p) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(p) : "memory");
    return prev;
}

// ------------------------------------------------------------- host side ---
// Dynamic shared memory opt-in and launch helpers live in the launcher files.

}  // namespace eagle

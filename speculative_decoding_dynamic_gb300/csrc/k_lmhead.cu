// LM-head logits of the frontier rows on the tensor cores (sm_103a): the
// projection that feeds stages 1+2 of each draft step.
//
// The draft model reuses the target's LM head ["EAGLE" notes, EAGLE 方法]:
// logits[m, v] = sum_h hidden[m, h] * W[v, h] for the M = B*k frontier rows of
// a step (hidden [M, H] bf16) and the whole vocabulary (W [V, H] bf16, one row
// per vocabulary entry). With M a few rows and W a gigabyte, the product is
// computed as D = W hidden^T so that the vocabulary fills the 128 rows of a
// tcgen05 MMA and the frontier rows its N columns (16..256):
//   tile (vt, rc)   vocabulary rows 128 vt .. 128 vt + 127 against frontier
//                   rows Nr rc .. Nr rc + Nr - 1, summed over H in 64-element
//                   stages (128-byte rows, 128B swizzle)
//   TMA             one lane streams the W and hidden boxes of each stage
//                   into a ring of shared-memory stages (full/empty mbarriers)
//   MMA             one lane issues four K=16 MMAs per stage into an fp32
//                   accumulator in tensor memory, double buffered across tiles
//   epilogue        four warps (TMEM lane = vocabulary row) read the
//                   accumulator and store fp32 (or bf16, round to nearest
//                   even) logits rows; one warp store covers 32 consecutive
//                   vocabulary entries of a frontier row
// The grid is persistent (one CTA per SM); tile t takes row chunk t % nrc
// and vocabulary tile t / nrc, so CTAs that run together share W tiles in L2
// and W is read from HBM about once. Out-of-range vocabulary rows, frontier
// rows and hidden columns arrive as zeros from TMA and are not stored.
//
// With stage 1 in the epilogue (TopK drafting reads the LM head's
// distribution, ["EAGLE" notes, EAGLE 方法]) the product is not swapped: the
// frontier rows fill the 128 TMEM lanes (M) and Nv vocabulary entries the
// columns (N = 128 or 256), so each epilogue thread holds one frontier row.
// CTA c serves row block c % nrb and the vocabulary tiles c / nrb,
// c / nrb + cpb, ... (the CTAs of one slot share each W tile in L2); a
// thread folds the logits of its row, rounded to the logit type, into a
// running maximum and sum of exp(x - max) and a sorted list (registers) of
// its largest keys (value, then lower token id), taking a group of 4 entries
// into the list only when its maximum beats the list's last key. The thread writes
// its row's partial once, after its last tile, and a merge kernel (one CTA
// per row) combines the cpb partials of a row: lse = M + log(sum_c S_c
// exp(M_c - M)), and the k largest keys among those at least the largest of
// the partials' k-th keys (every key of the row's top-k is one of them). The
// logits never leave the SM.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "eagle_ws.h"
#include "tc_ptx.cuh"

namespace eagle {
namespace {

constexpr int kVT = 128;                   // vocabulary rows per tile (MMA M)
constexpr int kKC = 64;                    // hidden elements per stage
constexpr int kMaxNr = 256;                // frontier rows per tile (MMA N)
constexpr int kMaxStages = 8;
constexpr int kLmThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kWBox = kVT * kKC * 2;       // 16 KB of W per stage
constexpr int kSmemBudget = 226 * 1024;    // ring bytes (+1 KB alignment slack: within 227 KB)

struct LmParams {
    int M, V, H;
    int Nr;      // frontier rows per tile (multiple of 16)
    int nrc;     // row chunks
    int ntiles;  // nrc * ceil(V / 128)
    int nkc;     // ceil(H / 64)
    int stages;
    int stage_bytes;
    int out_bf16;
    uint32_t acc_stride;  // TMEM columns between the two accumulator buffers (power of two >= 32)
    uint32_t tmem_cols;
    void* out;
    int* status;
};

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                  const LmParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages], bar_acc_full[2], bar_acc_empty[2];
    __shared__ uint32_t tmem_holder;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_acc_full[s], 1);
            mbar_init(&bar_acc_empty[s], kLmThreads - 64);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    // hidden is written by the draft forward, the logits buffer read by the
    // previous expand step
    pdl_wait_prior();

    if (warp == 0) {
        // ------------------------------------------------- TMA producer ---
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x) {
                const int rc = t % p.nrc, vt = t / p.nrc;
                for (int kc = 0; kc < p.nkc; ++kc, ++it) {
                    const uint32_t st = it % p.stages;
                    if (it >= static_cast<uint32_t>(p.stages) &&
                        !mbar_wait_sleep(&bar_empty[st], ((it / p.stages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    unsigned char* dst = smem + st * p.stage_bytes;
                    mbar_arrive_expect_tx(&bar_full[st], p.stage_bytes);
                    tma_load_2d(dst, &tm_w, kc * kKC, vt * kVT, &bar_full[st]);
                    tma_load_2d(dst + kWBox, &tm_h, kc * kKC, rc * p.Nr, &bar_full[st]);
                }
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer ---
        // D[v, m] (TMEM lane v, column m of buffer lt & 1) = sum over the
        // stages of W box (A, K-major) times hidden box (B, K-major).
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kVT, p.Nr, 0);
            uint32_t it = 0;
            bool ok = true;
            int lt = 0;
            for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x, ++lt) {
                const int buf = lt & 1;
                if (lt >= 2 && !mbar_wait_sleep(&bar_acc_empty[buf], ((lt >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * p.acc_stride;
                for (int kc = 0; kc < p.nkc; ++kc, ++it) {
                    const uint32_t st = it % p.stages;
                    if (!mbar_wait_sleep(&bar_full[st], (it / p.stages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t aW = smem_u32(smem + st * p.stage_bytes);
                    const uint32_t aH = aW + kWBox;
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled row
                        mma_bf16(d, smem_desc(aW + kk * 32, 16, 1024), smem_desc(aH + kk * 32, 16, 1024), idesc,
                                 (kc > 0 || kk > 0) ? 1 : 0);
                    mma_commit(&bar_empty[st]);
                }
                if (ok) mma_commit(&bar_acc_full[buf]);
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- epilogue ---
        // Warp w reads TMEM lanes 32 (w % 4) .. + 31: vocabulary rows of the tile.
        const int q4 = warp & 3;
        const int vl = (q4 << 5) | lane;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        int lt = 0;
        for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++lt) {
            const int rc = t % p.nrc, vt = t / p.nrc;
            const int buf = lt & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&bar_acc_full[buf], (lt >> 1) & 1))) {
                raise_status(p.status, kDevTimeout);
                break;
            }
            tc_fence_after();
            const int v = vt * kVT + vl;
            const int m0 = rc * p.Nr;
            const int mn = min(p.Nr, p.M - m0);  // live rows of the chunk (uniform)
            const uint32_t cols = tmem + lane_off + buf * p.acc_stride;
            const bool vlive = v < p.V;
            int c = 0;
            for (; c + 32 <= mn; c += 32) {
                float x[32];
                tmem_ld32(cols + c, x);
                if (vlive) {
                    if (p.out_bf16) {
                        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(m0 + c) * p.V + v;
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[static_cast<size_t>(j) * p.V] = __float2bfloat16_rn(x[j]);
                    } else {
                        float* o = static_cast<float*>(p.out) + static_cast<size_t>(m0 + c) * p.V + v;
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[static_cast<size_t>(j) * p.V] = x[j];
                    }
                }
            }
            for (; c < mn; c += 16) {
                float x[16];
                tmem_ld16(cols + c, x);
                if (vlive) {
                    const int jn = min(16, mn - c);
                    if (p.out_bf16) {
                        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(m0 + c) * p.V + v;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < jn) o[static_cast<size_t>(j) * p.V] = __float2bfloat16_rn(x[j]);
                    } else {
                        float* o = static_cast<float*>(p.out) + static_cast<size_t>(m0 + c) * p.V + v;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < jn) o[static_cast<size_t>(j) * p.V] = x[j];
                    }
                }
            }
            // the accumulator buffer may take the tile after next
            tc_fence_before();
            mbar_arrive(&bar_acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols) : "memory");
}

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer) {
    auto fn = tensor_map_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

// ---------------------------------------------- stage 1 in the epilogue ---

constexpr int kTkRows = 128;  // frontier rows per tile (MMA M, TMEM lanes)
constexpr int kTkMaxStages = 12;
constexpr float kLog2eLm = 1.4426950408889634f;

struct TkParams {
    int M, V, H, k;
    int Nv;     // vocabulary entries per tile (MMA N)
    int nrb;    // row blocks of 128 frontier rows
    int cpb;    // CTAs per row block = partials per row
    int nvt;    // vocabulary tiles
    int nkc;    // hidden stages per tile
    int stages, stage_bytes;
    int a_bytes;  // hidden box of a stage (the W box follows it)
    int cb_warps; // epilogue warps with live rows: each has a candidate buffer after the ring
    int bf16;   // logits rounded to bf16 (else fp32)
    uint32_t tmem_cols;
    float2* part_ms;      // [cpb, M]
    uint64_t* part_keys;  // [cpb, M, k]
    int* status;
};

// A list key: the logit's order-preserving bits, then the entry's position in
// the CTA's scan (lower position = lower token id) inverted; 0 = none. bf16
// logits fit 16 + 16 bits, fp32 logits take 32 + 32.
template <typename KeyT>
__device__ __forceinline__ KeyT list_key(float y, uint32_t pos);
template <>
__device__ __forceinline__ uint32_t list_key<uint32_t>(float y, uint32_t pos) {
    return (f2o(y) & 0xffff0000u) | (0xffffu - pos);
}
template <>
__device__ __forceinline__ uint64_t list_key<uint64_t>(float y, uint32_t pos) {
    return (static_cast<uint64_t>(f2o(y)) << 32) | (0xffffffffu - pos);
}
__device__ __forceinline__ float list_val(uint32_t key, uint32_t* pos) {
    *pos = 0xffffu - (key & 0xffffu);
    const uint32_t hi = key & 0xffff0000u;
    return o2f(hi | ((hi & 0x80000000u) ? 0u : 0xffffu));
}
__device__ __forceinline__ float list_val(uint64_t key, uint32_t* pos) {
    *pos = 0xffffffffu - static_cast<uint32_t>(key);
    return o2f(static_cast<uint32_t>(key >> 32));
}

// Insert into a list sorted best first (the last key drops out).
template <typename KeyT, int KL>
__device__ __forceinline__ void list_insert(KeyT (&top)[KL], KeyT key) {
#pragma unroll
    for (int i = KL - 1; i > 0; --i) top[i] = key > top[i - 1] ? top[i - 1] : (key > top[i] ? key : top[i]);
    top[0] = key > top[0] ? key : top[0];
}

template <typename KeyT, int KL>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_topk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                       const TkParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_full[kTkMaxStages], bar_empty[kTkMaxStages], bar_acc_full[2],
        bar_acc_empty[2];
    __shared__ uint32_t tmem_holder;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x % p.nrb, slot = blockIdx.x / p.nrb;

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_acc_full[s], 1);
            mbar_init(&bar_acc_empty[s], kLmThreads - 64);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    // hidden is written by the draft forward; the partials were read by the
    // previous merge
    pdl_wait_prior();

    if (warp == 0) {
        // ------------------------------------------------- TMA producer ---
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int vt = slot; ok && vt < p.nvt; vt += p.cpb) {
                for (int kc = 0; kc < p.nkc; ++kc, ++it) {
                    const uint32_t st = it % p.stages;
                    if (it >= static_cast<uint32_t>(p.stages) &&
                        !mbar_wait_sleep(&bar_empty[st], ((it / p.stages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    unsigned char* dst = smem + st * p.stage_bytes;
                    mbar_arrive_expect_tx(&bar_full[st], p.stage_bytes);
                    tma_load_2d(dst, &tm_h, kc * kKC, rb * kTkRows, &bar_full[st]);
                    tma_load_2d(dst + p.a_bytes, &tm_w, kc * kKC, vt * p.Nv, &bar_full[st]);
                }
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer ---
        // D[m, v] (TMEM lane m, column v of buffer ts & 1) = sum over the
        // stages of hidden box (A, K-major) times W box (B, K-major).
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTkRows, p.Nv, 0);
            uint32_t it = 0;
            bool ok = true;
            int ts = 0;
            for (int vt = slot; ok && vt < p.nvt; vt += p.cpb, ++ts) {
                const int buf = ts & 1;
                if (ts >= 2 && !mbar_wait_sleep(&bar_acc_empty[buf], ((ts >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * p.Nv;
                for (int kc = 0; kc < p.nkc; ++kc, ++it) {
                    const uint32_t st = it % p.stages;
                    if (!mbar_wait_sleep(&bar_full[st], (it / p.stages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t aA = smem_u32(smem + st * p.stage_bytes);
                    const uint32_t aB = aA + p.a_bytes;
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk)
                        mma_bf16(d, smem_desc(aA + kk * 32, 16, 1024), smem_desc(aB + kk * 32, 16, 1024), idesc,
                                 (kc > 0 || kk > 0) ? 1 : 0);
                    mma_commit(&bar_empty[st]);
                }
                if (ok) mma_commit(&bar_acc_full[buf]);
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- epilogue ---
        // Warp w reads TMEM lanes 32 (w % 4) .. + 31: thread = frontier row.
        // Lanes past the hidden box hold sums of stale shared memory: a warp
        // with no live row skips its chunks, dead lanes never take keys.
        const int q4 = warp & 3;
        const int row = rb * kTkRows + q4 * 32 + lane;
        const bool live = row < p.M;
        const bool warp_live = rb * kTkRows + q4 * 32 < p.M;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        float m = -INFINITY, s = 0.0f;
        // this lane's candidate buffer: slot t at cb[t * 32] (32 slots, one chunk)
        KeyT* const cb = reinterpret_cast<KeyT*>(smem + p.stages * p.stage_bytes) + q4 * 32 * 32 + lane;
        KeyT top[KL];  // the KL >= k largest keys so far, best first (0 = none)
#pragma unroll
        for (int i = 0; i < KL; ++i) top[i] = KeyT(0);
        int ts = 0;
        for (int vt = slot; vt < p.nvt; vt += p.cpb, ++ts) {
            const int buf = ts & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&bar_acc_full[buf], (ts >> 1) & 1))) {
                raise_status(p.status, kDevTimeout);
                break;
            }
            tc_fence_after();
            const uint32_t base = tmem + lane_off + buf * p.Nv;
            for (int c = 0; warp_live && c < p.Nv; c += 32) {
                const int nv = min(32, p.V - (vt * p.Nv + c));  // live entries of the chunk (uniform)
                if (nv <= 0) break;
                float x[32];
                tmem_ld32(base + c, x);
                // the logits as the logits buffer would hold them; dead entries -inf
                float gm[8];  // maxima of the groups of 4 entries
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = i < nv ? (p.bf16 ? __bfloat162float(__float2bfloat16_rn(x[i])) : x[i]) : -INFINITY;
                    gm[i >> 2] = (i & 3) ? fmaxf(gm[i >> 2], x[i]) : x[i];
                }
                const float cm = fmaxf(fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3])),
                                       fmaxf(fmaxf(gm[4], gm[5]), fmaxf(gm[6], gm[7])));
                // running maximum and sum of exp(x - max)
                if (cm > m) {
                    if (s != 0.0f) s *= ex2_approx((m - cm) * kLog2eLm);
                    m = cm;
                }
                if (m > -INFINITY) {
                    const float mb = m * kLog2eLm;
                    float t0 = 0.0f, t1 = 0.0f, t2 = 0.0f, t3 = 0.0f;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        t0 += ex2_approx(fmaf(x[i], kLog2eLm, -mb));
                        t1 += ex2_approx(fmaf(x[i + 1], kLog2eLm, -mb));
                        t2 += ex2_approx(fmaf(x[i + 2], kLog2eLm, -mb));
                        t3 += ex2_approx(fmaf(x[i + 3], kLog2eLm, -mb));
                    }
                    s += (t0 + t1) + (t2 + t3);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (x[i] != x[i]) s = x[i];  // a NaN among -inf entries: the sum turns NaN
                }
                // keys of the chunk that may enter the list
                const uint32_t pos0 = static_cast<uint32_t>(ts * p.Nv + c);
                // (a group's best possible key: its maximum at its first position)
                // Candidates: each lane first stages the keys of its groups
                // that may enter its list (against the list's last key before
                // the chunk), then inserts its own; the warp runs the
                // insertion network for the largest count among its lanes,
                // not for every entry any lane has.
                const KeyT thr = top[KL - 1];
                const bool cand = live && (list_key<KeyT>(cm, pos0) > thr || cm != cm);
                if (__any_sync(0xffffffffu, cand)) {
                    int nc = 0;
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        if (cand && (list_key<KeyT>(gm[g], pos0 + 4 * g) > thr || gm[g] != gm[g])) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int i = 4 * g + j;
                                const KeyT key = i < nv ? list_key<KeyT>(x[i], pos0 + i) : KeyT(0);
                                if (key > thr) cb[(nc++) * 32] = key;
                            }
                        }
                    }
                    for (int t = 0; t < nc; ++t) {
                        const KeyT key = cb[t * 32];
                        if (key > top[KL - 1]) list_insert(top, key);
                    }
                }
            }
            // the accumulator buffer may take the tile after next
            tc_fence_before();
            mbar_arrive(&bar_acc_empty[buf]);
        }
        if (live) {
            p.part_ms[static_cast<size_t>(slot) * p.M + row] = make_float2(m, s);
            uint64_t* dst = p.part_keys + (static_cast<size_t>(slot) * p.M + row) * p.k;
#pragma unroll
            for (int i = 0; i < KL; ++i) {
                if (i >= p.k) break;
                const KeyT key = top[i];
                uint64_t out = 0ull;
                if (key != KeyT(0)) {
                    uint32_t pos;
                    const float val = list_val(key, &pos);
                    const uint32_t tsq = pos / static_cast<uint32_t>(p.Nv), col = pos % static_cast<uint32_t>(p.Nv);
                    const uint32_t id = (static_cast<uint32_t>(slot) + tsq * static_cast<uint32_t>(p.cpb)) *
                                            static_cast<uint32_t>(p.Nv) + col;
                    out = make_key(val, id);
                }
                dst[i] = out;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols) : "memory");
}

// Merge of a row's partials, one CTA per row (see the file comment). The
// bound on the candidates is the larger of the partials' largest k-th key
// and the k-th largest of the partials' first keys: the k partials holding
// those first keys give k keys at least that large, so every key of the
// row's top-k is at or above either bound.
constexpr int kLmMergeThreads = 256;
static_assert(kLmShards <= kLmMergeThreads, "one partial per merge thread");
__global__ void __launch_bounds__(kLmMergeThreads) lm_merge_kernel(int S, int M, int k,
                                                                   const float2* __restrict__ part_ms,
                                                                   const uint64_t* __restrict__ part_keys,
                                                                   float* __restrict__ lse_out,
                                                                   int32_t* __restrict__ topk_id,
                                                                   float* __restrict__ topk_val, int* status) {
    __shared__ uint64_t keys[kLmShards * kMaxTopK];
    __shared__ uint64_t cand[kLmShards * kMaxTopK];
    __shared__ uint64_t red_key[kLmMergeThreads / 32];
    __shared__ float red_f[kLmMergeThreads / 32];
    __shared__ uint64_t kth_first;
    __shared__ int ncand;
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nw = kLmMergeThreads / 32;
    pdl_launch_dependents();
    pdl_wait_prior();
    if (tid == 0) {
        ncand = 0;
        kth_first = 0ull;
    }
    for (int i = tid; i < S * k; i += kLmMergeThreads) {
        const int c = i / k, r = i - c * k;
        keys[i] = __ldcg(&part_keys[(static_cast<size_t>(c) * M + row) * k + r]);
    }
    // thread c < S holds partial c (S <= kLmShards < threads)
    float2 ms = make_float2(-INFINITY, 0.0f);
    if (tid < S) ms = __ldcg(&part_ms[static_cast<size_t>(tid) * M + row]);
    __syncthreads();
    uint64_t th = 0ull;
    float m = ms.x;
    if (tid < S) {
        const uint64_t first = keys[tid * k];
        th = keys[tid * k + k - 1];
        int r = 0;
        for (int c = 0; c < S; ++c) r += keys[c * k] > first;
        if (r == k - 1 && first != 0ull) kth_first = first;  // keys are unique: one thread at most
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        th = max(th, shfl_xor_u64(th, o));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    if (lane == 0) {
        red_key[warp] = th;
        red_f[warp] = m;
    }
    __syncthreads();
    th = max(red_key[0], kth_first);
    m = red_f[0];
#pragma unroll
    for (int w = 1; w < nw; ++w) {
        th = max(th, red_key[w]);
        m = fmaxf(m, red_f[w]);
    }
    // sum of S_c exp(M_c - M), summed in a fixed order (threads, then warps)
    float t = 0.0f;
    if (tid < S && ms.y != 0.0f) t = ms.y * ex2_approx((ms.x - m) * kLog2eLm);  // a NaN sum stays NaN
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    // candidates: the keys at or above the bound
    for (int i = tid; i < S * k; i += kLmMergeThreads) {
        const uint64_t key = keys[i];
        if (key != 0ull && key >= th) cand[atomicAdd(&ncand, 1)] = key;
    }
    __syncthreads();  // every thread has read red_f before it takes the warp sums
    if (lane == 0) red_f[warp] = t;
    __syncthreads();
    const int nc = ncand;
    for (int i = tid; i < nc; i += kLmMergeThreads) {
        const uint64_t key = cand[i];
        int r = 0;
        for (int j = 0; j < nc; ++j) r += cand[j] > key;
        if (r < k) {
            topk_id[static_cast<size_t>(row) * k + r] = static_cast<int32_t>(key_id(key));
            topk_val[static_cast<size_t>(row) * k + r] = key_val(key);
        }
    }
    for (int r = nc + tid; r < k; r += kLmMergeThreads) {
        topk_id[static_cast<size_t>(row) * k + r] = -1;
        topk_val[static_cast<size_t>(row) * k + r] = -INFINITY;
    }
    if (tid == 0) {
        float sum = 0.0f;
        for (int w = 0; w < nw; ++w) sum += red_f[w];
        const float lse = m + logf(sum);
        lse_out[row] = lse;
        if (!isfinite(lse)) raise_status(status, kDevNonFinite);
    }
}

template <typename KeyT, int KL>
cudaError_t launch_topk_gemm(const TkParams& p, const CUtensorMap& tw, const CUtensorMap& th, cudaStream_t stream) {
    const int smem = p.stages * p.stage_bytes + p.cb_warps * 32 * 32 * static_cast<int>(sizeof(KeyT)) + 1024;
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(lmhead_topk_kernel<KeyT, KL>), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(lmhead_topk_kernel<KeyT, KL>, dim3(p.nrb * p.cpb), dim3(kLmThreads), static_cast<size_t>(smem),
                      stream, tw, th, p);
}

}  // namespace

cudaError_t launch_lmhead(int M, int V, int H, const void* hidden, const void* weight, int out_dtype, void* out,
                          int* status, cudaStream_t stream) {
    if (M < 1 || V < 1 || H < 8 || (H % 8) != 0) return cudaErrorInvalidValue;
    LmParams p{};
    p.M = M;
    p.V = V;
    p.H = H;
    p.nrc = (M + kMaxNr - 1) / kMaxNr;
    const int per = (M + p.nrc - 1) / p.nrc;
    p.Nr = (per + 15) & ~15;
    p.ntiles = p.nrc * ((V + kVT - 1) / kVT);
    p.nkc = (H + kKC - 1) / kKC;
    p.stage_bytes = kWBox + p.Nr * kKC * 2;
    p.stages = kSmemBudget / p.stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages > p.nkc) p.stages = p.nkc < 2 ? 2 : p.nkc;
    p.out_bf16 = out_dtype == 1;
    uint32_t stride = 32;
    while (stride < static_cast<uint32_t>(p.Nr)) stride <<= 1;
    p.acc_stride = stride;
    p.tmem_cols = 2 * stride;
    p.out = out;
    p.status = status;
    CUtensorMap tw, th;
    if (!make_map_2d(&tw, weight, static_cast<uint64_t>(H), static_cast<uint64_t>(V), kKC, kVT))
        return cudaErrorInvalidValue;
    if (!make_map_2d(&th, hidden, static_cast<uint64_t>(H), static_cast<uint64_t>(M), kKC,
                     static_cast<uint32_t>(p.Nr)))
        return cudaErrorInvalidValue;
    const int smem = p.stages * p.stage_bytes + 1024;
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(lmhead_kernel), smem);
    if (e != cudaSuccess) return e;
    const int grid = p.ntiles < sm_count() ? p.ntiles : sm_count();
    return launch_pdl(lmhead_kernel, dim3(grid), dim3(kLmThreads), static_cast<size_t>(smem), stream, tw, th, p);
}

size_t lmhead_topk_scratch_bytes(long M, int k) {
    const size_t ms = align_up(static_cast<size_t>(kLmShards) * M * sizeof(float2), 256);
    return ms + align_up(static_cast<size_t>(kLmShards) * M * k * sizeof(uint64_t), 256);
}

cudaError_t launch_lmhead_topk(int M, int V, int H, int k, const void* hidden, const void* weight, int out_dtype,
                               void* scratch, float* row_lse, int32_t* topk_id, float* topk_val, int* status,
                               cudaStream_t stream) {
    if (M < 1 || V < k || H < 8 || (H % 8) != 0 || k < 1 || k > kMaxTopK) return cudaErrorInvalidValue;
    TkParams p{};
    p.M = M;
    p.V = V;
    p.H = H;
    p.k = k;
    p.nrb = (M + kTkRows - 1) / kTkRows;
    // 256 vocabulary entries per tile when several row blocks make the GEMM
    // compute-bound (fewer hidden re-reads), else 128 (more tiles to spread)
    p.Nv = p.nrb > 1 ? 256 : 128;
    p.nvt = (V + p.Nv - 1) / p.Nv;
    const int ctas = sm_count() < kLmShards ? sm_count() : kLmShards;
    p.cpb = ctas / p.nrb;
    if (p.cpb > p.nvt) p.cpb = p.nvt;
    if (p.cpb < 1) return cudaErrorInvalidValue;
    p.bf16 = out_dtype == 1;
    // bf16 keys carry a 16-bit scan position
    if (p.bf16 && static_cast<long>((p.nvt + p.cpb - 1) / p.cpb) * p.Nv > 65536) return cudaErrorInvalidValue;
    p.nkc = (H + kKC - 1) / kKC;
    // one row block: the hidden box covers the live rows only (16-row steps),
    // so no zero rows cross from L2 and more W fits in the ring; the MMA's
    // A operand (128 rows) then runs on into the stage's W box, whose rows
    // land in TMEM lanes of dead rows
    const int hbox = p.nrb == 1 ? (M + 15) & ~15 : kTkRows;
    p.a_bytes = hbox * kKC * 2;
    p.stage_bytes = p.a_bytes + p.Nv * kKC * 2;
    // candidate buffers (32 keys per lane) for the epilogue warps with live rows
    p.cb_warps = p.nrb > 1 ? 4 : (M + 31) / 32;
    const int cb_bytes = p.cb_warps * 32 * 32 * (p.bf16 ? 4 : 8);
    p.stages = (kSmemBudget - 1024 - cb_bytes) / p.stage_bytes;  // (1 KB left for the static barriers)
    if (p.stages > kTkMaxStages) p.stages = kTkMaxStages;
    if (p.stages > p.nkc) p.stages = p.nkc < 2 ? 2 : p.nkc;
    p.tmem_cols = 2 * static_cast<uint32_t>(p.Nv);
    p.status = status;
    p.part_ms = static_cast<float2*>(scratch);
    p.part_keys = reinterpret_cast<uint64_t*>(static_cast<char*>(scratch) +
                                              align_up(static_cast<size_t>(kLmShards) * M * sizeof(float2), 256));
    CUtensorMap tw, th;
    if (!make_map_2d(&tw, weight, static_cast<uint64_t>(H), static_cast<uint64_t>(V), kKC,
                     static_cast<uint32_t>(p.Nv)))
        return cudaErrorInvalidValue;
    if (!make_map_2d(&th, hidden, static_cast<uint64_t>(H), static_cast<uint64_t>(M), kKC,
                     static_cast<uint32_t>(hbox)))
        return cudaErrorInvalidValue;
    // list length: the smallest of 4, 8, 12, 16 that holds k keys
    cudaError_t e;
    if (!p.bf16)
        e = launch_topk_gemm<uint64_t, kMaxTopK>(p, tw, th, stream);
    else if (k <= 4)
        e = launch_topk_gemm<uint32_t, 4>(p, tw, th, stream);
    else if (k <= 8)
        e = launch_topk_gemm<uint32_t, 8>(p, tw, th, stream);
    else if (k <= 12)
        e = launch_topk_gemm<uint32_t, 12>(p, tw, th, stream);
    else
        e = launch_topk_gemm<uint32_t, kMaxTopK>(p, tw, th, stream);
    if (e != cudaSuccess) return e;
    return launch_pdl(lm_merge_kernel, dim3(M), dim3(kLmMergeThreads), 0, stream, p.cpb, M, k,
                      static_cast<const float2*>(p.part_ms), static_cast<const uint64_t*>(p.part_keys), row_lse,
                      topk_id, topk_val, status);
}

}  // namespace eagle

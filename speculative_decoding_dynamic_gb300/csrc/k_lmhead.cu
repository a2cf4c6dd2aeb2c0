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

}  // namespace eagle

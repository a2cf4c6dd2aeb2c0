// Stage 5, CUDA-core path (sm_103a): tree-masked GQA attention for fp32
// inputs (any head_dim <= 128) and small problems. One CTA per (slot, query
// head, sequence); its warps stride over the keys, each lane holding d/32
// elements of q, the running output and the current key/value row; online
// softmax in the log2 domain; warps merged through shared memory.
//
// Keys of slot i: prefix positions [0, L_b) and tree slots j with bit j of
// mask row i (position L_b + j) ["EAGLE" notes, EAGLE 方法: Medusa-style tree
// attention; "EAGLE-2: Faster Inference ..." summary 4.2].

#include <cuda_bf16.h>

#include <cmath>

#include "eagle_internal.cuh"
#include "eagle_ws.h"

namespace eagle {

constexpr int kSimtWarps = 4;

template <int DT>
__device__ __forceinline__ float ld_elem(const void* base, int64_t idx) {
    if (DT == 1) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

template <int DT, int EPL>
__global__ void __launch_bounds__(kSimtWarps * 32) attn_simt_kernel(KvDims kv, int T, const void* __restrict__ q,
                                                                     const void* __restrict__ cache, int layer,
                                                                     const int32_t* __restrict__ prefix_len,
                                                                     const uint32_t* __restrict__ mask,
                                                                     const int32_t* __restrict__ n_tree,
                                                                     void* __restrict__ out, float scale_log2,
                                                                     int* status) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int d = kv.d;
    const int W = (T + 31) / 32;
    const int64_t orow = ((static_cast<int64_t>(b) * T + i) * kv.Hq + h) * d;
    const int n = n_tree[b];
    const int L = prefix_len[b];
    if (i >= n || L < 0 || L + T > kv.max_len) {
        if (i < n && threadIdx.x == 0) raise_status(status, kDevBadIndex);
        for (int e = threadIdx.x; e < d; e += blockDim.x) {
            if (DT == 1)
                reinterpret_cast<__nv_bfloat16*>(out)[orow + e] = __float2bfloat16_rn(0.0f);
            else
                reinterpret_cast<float*>(out)[orow + e] = 0.0f;
        }
        return;
    }
    const int hk = h / (kv.Hq / kv.Hkv);
    const int64_t kbase = static_cast<int64_t>(b) * kv.seq_stride + static_cast<int64_t>(layer) * kv.layer_stride +
                          static_cast<int64_t>(hk) * d;
    const int64_t vbase = kbase + kv.kv_stride;
    const uint32_t* mrow = mask + (static_cast<int64_t>(b) * T + i) * W;

    float qr[EPL], acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int c = lane + 32 * e;
        qr[e] = c < d ? ld_elem<DT>(q, orow + c) * scale_log2 : 0.0f;
        acc[e] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;
    const int nkeys = L + T;
    for (int kk = warp; kk < nkeys; kk += kSimtWarps) {
        if (kk >= L) {
            const int j = kk - L;
            if (!((mrow[j >> 5] >> (j & 31)) & 1u)) continue;
        }
        const int64_t ko = kbase + static_cast<int64_t>(kk) * kv.pos_stride;
        const int64_t vo = vbase + static_cast<int64_t>(kk) * kv.pos_stride;
        float s = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int c = lane + 32 * e;
            if (c < d) s = fmaf(qr[e], ld_elem<DT>(cache, ko + c), s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float mn = fmaxf(m, s);
        const float corr = ex2_approx(m - mn);
        const float p = ex2_approx(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int c = lane + 32 * e;
            const float v = c < d ? ld_elem<DT>(cache, vo + c) : 0.0f;
            acc[e] = fmaf(p, v, acc[e] * corr);
        }
        m = mn;
    }
    __shared__ float sm_m[kSimtWarps], sm_l[kSimtWarps];
    __shared__ float sm_acc[kSimtWarps][32 * 4];
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_acc[warp][lane + 32 * e] = acc[e];
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, sm_m[w]);
    float Lsum = 0.0f;
    float o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
    for (int w = 0; w < kSimtWarps; ++w) {
        if (sm_m[w] == -INFINITY) continue;
        const float c = ex2_approx(sm_m[w] - M);
        Lsum += sm_l[w] * c;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] += sm_acc[w][lane + 32 * e] * c;
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int c = lane + 32 * e;
        if (c >= d) continue;
        if (DT == 1)
            reinterpret_cast<__nv_bfloat16*>(out)[orow + c] = __float2bfloat16_rn(o[e] * inv);
        else
            reinterpret_cast<float*>(out)[orow + c] = o[e] * inv;
    }
}

cudaError_t launch_attention_simt(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream) {
    dim3 grid(T, kv.Hq, kv.B);
    const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kv.d)));
    const int epl = kv.d <= 32 ? 1 : (kv.d <= 64 ? 2 : 4);
#define EAGLE_SIMT_LAUNCH(DT, E)                                                                               \
    return launch_pdl(attn_simt_kernel<DT, E>, grid, dim3(kSimtWarps * 32), 0, stream, kv, T, q, cache, layer, \
                      prefix_len, mask, n_tree, out, scale_log2, status)
    if (kv.dtype == 1) {
        if (epl == 1) EAGLE_SIMT_LAUNCH(1, 1);
        if (epl == 2) EAGLE_SIMT_LAUNCH(1, 2);
        EAGLE_SIMT_LAUNCH(1, 4);
    }
    if (epl == 1) EAGLE_SIMT_LAUNCH(0, 1);
    if (epl == 2) EAGLE_SIMT_LAUNCH(0, 2);
    EAGLE_SIMT_LAUNCH(0, 4);
#undef EAGLE_SIMT_LAUNCH
}

}  // namespace eagle

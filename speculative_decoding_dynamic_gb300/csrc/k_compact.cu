// Stage 6b: accepted-path KV compaction (sm_103a).
//
// For sequence b, layer l, K|V and j = 1..a_b:
//   cache[L_b + j] <- cache[L_b + s_j]      (s_j = accepted slot j)
// Accepted slots are increasing and s_j >= j, but a destination can be the
// source of a later j, so every source is read before any destination is
// written. Each thread owns one 16-byte column of the (Hkv * d)-element
// position row and moves that column for all j: it loads every source into
// registers first, then stores, so no barrier is needed.
//
// Not on the pages; the plain reading of moving the accepted nodes' KV into
// the contiguous cache.

#include "eagle_internal.cuh"
#include "eagle_ws.h"

namespace eagle {

constexpr int kCompactThreads = 128;
constexpr int kMaxAccept = kMaxDepth;  // a_b <= D <= 16

__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(KvDims kv, char* __restrict__ cache, int esize,
                                                                      const int32_t* __restrict__ prefix_len,
                                                                      const int32_t* __restrict__ accept_len,
                                                                      const int32_t* __restrict__ slots,
                                                                      int slots_stride, int32_t* __restrict__ new_len,
                                                                      int* status) {
    const int b = blockIdx.z;
    const int lk = blockIdx.y;  // layer * 2 + kv
    const int layer = lk >> 1, which = lk & 1;
    const int col = blockIdx.x * kCompactThreads + threadIdx.x;  // 16-byte column
    pdl_launch_dependents();
    pdl_wait_prior();
    const int ncol = kv.Hkv * kv.d * esize / 16;
    const int L = prefix_len[b];
    const int a = accept_len[b];
    const bool ok = a >= 0 && a <= kMaxAccept && a < slots_stride && L >= 0 && L + a < kv.max_len;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        if (ok)
            new_len[b] = L + a + 1;
        else
            raise_status(status, kDevBadIndex);
    }
    if (!ok || col >= ncol) return;
    const int32_t* s = slots + static_cast<size_t>(b) * slots_stride;
    char* region = cache + (static_cast<int64_t>(b) * kv.seq_stride + layer * kv.layer_stride + which * kv.kv_stride) *
                               static_cast<int64_t>(esize);
    const int64_t prow = kv.pos_stride * esize;
    uint4 v[kMaxAccept];
#pragma unroll
    for (int j = 1; j <= kMaxAccept; ++j) {
        if (j <= a) {
            const int sj = s[j];
            if (sj < j || L + sj >= kv.max_len) {
                raise_status(status, kDevBadIndex);
                return;
            }
            v[j - 1] = __ldcs(reinterpret_cast<const uint4*>(region + (L + sj) * prow) + col);
        }
    }
#pragma unroll
    for (int j = 1; j <= kMaxAccept; ++j)
        if (j <= a) __stcs(reinterpret_cast<uint4*>(region + (L + j) * prow) + col, v[j - 1]);
}

cudaError_t launch_kv_compact(const KvDims& kv, void* cache, const int32_t* prefix_len, const int32_t* accept_len,
                              const int32_t* slots, int slots_stride, int32_t* new_len, int* status,
                              cudaStream_t stream) {
    const int esize = kv.dtype == 1 ? 2 : 4;
    const int ncol = kv.Hkv * kv.d * esize / 16;
    dim3 grid((ncol + kCompactThreads - 1) / kCompactThreads, kv.layers * 2, kv.B);
    return launch_pdl(kv_compact_kernel, grid, dim3(kCompactThreads), 0, stream, kv, static_cast<char*>(cache), esize,
                      prefix_len, accept_len, slots, slots_stride, new_len, status);
}

}  // namespace eagle

// Per-sequence tree kernels (sm_103a): state reset, stage 3 (global top-N
// rerank) and stage 4 (flattening with ancestor mask). One CTA per sequence;
// the candidate table (C <= 1024) lives in shared memory.
//
// Sources (page title and section): "EAGLE-2: Faster Inference ..." summary,
// 4.2 Reranking Phase (keep the top m tokens by value, flatten them with a
// branch-separating mask); "EAGLE" notes (garden.houmin.site), EAGLE 2 方法,
// ReRank (equal values keep the shallower node); "EAGLE-2: Dynamic Draft
// Trees" tutorial (a node's ancestors always outscore it, so the kept set is a
// connected tree).

#include <cmath>

#include "eagle_internal.cuh"
#include "eagle_ws.h"

namespace eagle {

// ------------------------------------------------------------ tree init ---

__global__ void tree_init_kernel(TreeDims d, TreeWs w) {
    pdl_launch_dependents();
    pdl_wait_prior();
    const size_t BC = static_cast<size_t>(d.B) * d.C;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < BC; i += stride) {
        w.cand_token[i] = -1;
        w.cand_parent[i] = -1;
        w.cand_depth[i] = -1;
        w.cand_logv[i] = -INFINITY;
        w.cand_lp[i] = -INFINITY;
        w.cand_valid[i] = 0;
        w.kept[i] = 0;
        w.slot_of[i] = -1;
    }
    const size_t F = static_cast<size_t>(d.D + 1) * d.B * d.k;
    for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < F; i += stride) w.fnode[i] = -1;
    const size_t S = static_cast<size_t>(d.D + 1) * d.B;
    for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < S; i += stride)
        w.fcount[i] = i < static_cast<size_t>(d.B) ? 1 : 0;  // step 0: the root
    for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < static_cast<size_t>(d.B); i += stride) {
        w.expand_ticket[i] = 0;
        w.verify_ticket[i] = 0;
        w.n_kept[i] = 0;
    }
}

// ---------------------------------------------------------------- rerank ---

constexpr int kSortThreads = 512;

// Key of a candidate: value first (larger), then lower node id. Node ids are
// depth-major, so for equal values the lower id is also the shallower node.
// Invalid candidates get key 0 and sort last. Without rerank (policy 2) only
// the nodes the expansion chose (the frontier of steps 1..D) are candidates;
// the static shape (policy 3) takes the same candidates keyed by depth
// (shallower first), then lower id, so the kept shape ignores the values.
__global__ void __launch_bounds__(kSortThreads) rerank_kernel(TreeDims d, TreeWs w, int P) {
    __shared__ uint64_t keys[kMaxCandidates];
    __shared__ uint8_t chosen[kMaxCandidates];
    __shared__ int n_valid;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait_prior();
    if (tid == 0) n_valid = 0;
    const bool frontiers_only = d.policy == 2 || d.policy == 3;
    if (frontiers_only) {
        for (int i = tid; i < d.C; i += kSortThreads) chosen[i] = 0;
        __syncthreads();
        for (int q = tid; q < d.D * d.k; q += kSortThreads) {
            const int id = w.fnode[((1 + q / d.k) * d.B + b) * d.k + q % d.k];
            if (id >= 0 && id < d.C) chosen[id] = 1;
        }
    }
    __syncthreads();
    int local = 0;
    for (int i = tid; i < P; i += kSortThreads) {
        uint64_t key = 0;
        if (i < d.C) {
            const size_t at = static_cast<size_t>(b) * d.C + i;
            if (w.cand_valid[at] && (!frontiers_only || chosen[i])) {
                // static shape: by depth (shallower first), not by value
                const float v = d.policy == 3 ? -static_cast<float>(w.cand_depth[at]) : w.cand_logv[at];
                key = make_key(v, static_cast<uint32_t>(i));
                ++local;
            }
            w.kept[at] = 0;
        }
        keys[i] = key;
    }
    if (local) atomicAdd(&n_valid, local);
    if (P <= kSortThreads) {
        // Bitonic sort, descending, one key per thread in a register: pairs
        // closer than 32 meet by warp shuffles, farther ones through shared
        // memory (two buffers alternate, one barrier per such stage).
        __syncthreads();
        uint64_t v = tid < P ? keys[tid] : 0ull;
        int sm_stage = 0;
        for (int size = 2; size <= kSortThreads; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                uint64_t o;
                if (stride >= 32) {
                    uint64_t* buf = keys + (sm_stage & 1) * kSortThreads;
                    buf[tid] = v;
                    __syncthreads();
                    o = buf[tid ^ stride];
                    ++sm_stage;
                } else {
                    o = shfl_xor_u64(v, stride);
                }
                const bool desc = (tid & size) == 0;
                const bool lower = (tid & stride) == 0;
                v = (lower == desc) ? (o > v ? o : v) : (o < v ? o : v);
            }
        }
        const int keep = min(d.N, n_valid);
        if (tid < keep && EAGLE_CHECKED(key_id(v) < static_cast<uint32_t>(d.C), w.status))
            w.kept[static_cast<size_t>(b) * d.C + key_id(v)] = 1;
        if (tid == 0) w.n_kept[b] = keep;
        return;
    }
    // Bitonic sort, descending (more than 512 keys: in shared memory).
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int t = tid; t < P / 2; t += kSortThreads) {
                const int i = 2 * t - (t & (stride - 1));
                const int j = i + stride;
                const bool desc = (i & size) == 0;
                const uint64_t a = keys[i], c = keys[j];
                if ((a < c) == desc) {
                    keys[i] = c;
                    keys[j] = a;
                }
            }
        }
    }
    __syncthreads();
    const int keep = min(d.N, n_valid);
    for (int r = tid; r < keep; r += kSortThreads) {
        const uint32_t id = key_id(keys[r]);
        if (EAGLE_CHECKED(id < static_cast<uint32_t>(d.C), w.status)) w.kept[static_cast<size_t>(b) * d.C + id] = 1;
    }
    if (tid == 0) w.n_kept[b] = keep;
}

// ------------------------------------------------------------ build tree ---

constexpr int kBuildThreads = 1024;

__global__ void __launch_bounds__(kBuildThreads) build_tree_kernel(TreeDims d, TreeWs w,
                                                                    const int32_t* __restrict__ prefix_len,
                                                                    const int32_t* __restrict__ root_token,
                                                                    int32_t* __restrict__ tokens,
                                                                    int32_t* __restrict__ parent,
                                                                    int32_t* __restrict__ depth,
                                                                    int32_t* __restrict__ pos,
                                                                    uint32_t* __restrict__ mask,
                                                                    int32_t* __restrict__ n_tree) {
    __shared__ int slot_of[kMaxCandidates];
    __shared__ int par_node[kMaxCandidates];
    __shared__ int tok_of[kMaxCandidates];  // token and depth of every candidate, loaded with the flags
    __shared__ int dep_of[kMaxCandidates];
    __shared__ int warp_sum[kBuildThreads / 32];
    __shared__ int node_at[kMaxSlots];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = d.T, W = d.W;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int L = prefix_len[b];
    if (tid == 0 && L < 0) raise_status(w.status, kDevBadIndex);
#ifdef EAGLE_DEBUG
    for (int i = tid; i < kMaxSlots; i += kBuildThreads) node_at[i] = -1;  // slots no kept node fills stay -1
    __syncthreads();
#endif

    // Exclusive scan of the kept flags in node-id order gives each kept node its slot.
    const size_t base = static_cast<size_t>(b) * d.C;
    const int flag = (tid < d.C) ? (w.kept[base + tid] != 0) : 0;
    if (tid < d.C) {
        par_node[tid] = w.cand_parent[base + tid];
        tok_of[tid] = w.cand_token[base + tid];
        dep_of[tid] = w.cand_depth[base + tid];
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, flag);
    const int before_in_warp = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) warp_sum[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
        const int v = lane < kBuildThreads / 32 ? warp_sum[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < kBuildThreads / 32) warp_sum[lane] = incl - v;
    }
    __syncthreads();
    const int slot = flag ? 1 + warp_sum[warp] + before_in_warp : -1;
    if (tid < d.C) {
        slot_of[tid] = slot;
        w.slot_of[base + tid] = slot;
        if (flag && slot < T) node_at[slot] = tid;
    }
    __syncthreads();
    const int n = 1 + w.n_kept[b];
    if (tid == 0 && n > T) raise_status(w.status, kDevOverflow);

    // One thread per slot writes its row.
    for (int i = tid; i < T; i += kBuildThreads) {
        const size_t r = static_cast<size_t>(b) * T + i;
        uint32_t* mrow = mask + r * W;
        if (i >= n) {
            tokens[r] = parent[r] = depth[r] = pos[r] = -1;
            for (int q = 0; q < W; ++q) mrow[q] = 0u;
            continue;
        }
        for (int q = 0; q < W; ++q) mrow[q] = 0u;
        uint32_t m0 = 1u;  // the root is an ancestor of every slot
        if (i == 0) {
            const int rt = root_token[b];
            if (rt < 0 || rt >= d.V) raise_status(w.status, kDevBadIndex);
            tokens[r] = rt;
            parent[r] = -1;
            depth[r] = 0;
            pos[r] = L;
        } else {
            const int id = node_at[i];
            if (!EAGLE_CHECKED(id >= 0 && id < d.C, w.status)) continue;
            const int pn = par_node[id];
            if (!EAGLE_CHECKED(pn >= -1 && pn < d.C, w.status)) continue;
            const int ps = pn < 0 ? 0 : slot_of[pn];
            if (ps < 0) raise_status(w.status, kDevOverflow);  // parent not kept: cannot happen
            const int dep = dep_of[id];
            tokens[r] = tok_of[id];
            parent[r] = ps;
            depth[r] = dep;
            pos[r] = L + dep;
            // ancestors-or-self: walk up the parent chain (at most D steps)
            int cur = id;
            int sl = i;
            for (int guard = 0; guard <= kMaxDepth && sl > 0; ++guard) {
                if (sl / 32 == 0)
                    m0 |= 1u << sl;
                else
                    mrow[sl / 32] |= 1u << (sl % 32);
                const int p = par_node[cur];
                if (p < 0) break;
                if (!EAGLE_CHECKED(p < d.C && slot_of[p] >= 0 && slot_of[p] < sl, w.status)) break;
                cur = p;
                sl = slot_of[p];
            }
        }
        mrow[0] |= m0;
    }
    if (tid == 0) n_tree[b] = n;
}

// ------------------------------------------------------------- tree value ---

// Sum of exp(log value) over the kept nodes of a sequence, in node-id order
// (one warp per sequence: lane-strided partial sums combined in lane order).
__global__ void __launch_bounds__(32) tree_value_kernel(TreeDims d, TreeWs w, float* __restrict__ value_sum) {
    const int b = blockIdx.x, lane = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait_prior();
    float s = 0.0f;
    for (int i = lane; i < d.C; i += 32) {
        const size_t at = static_cast<size_t>(b) * d.C + i;
        if (w.kept[at]) s += expf(w.cand_logv[at]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) value_sum[b] = s;
}

// -------------------------------------------------------------- launchers ---

cudaError_t launch_tree_init(const TreeDims& d, const TreeWs& ws, cudaStream_t stream) {
    const size_t work = static_cast<size_t>(d.B) * d.C;
    int blocks = static_cast<int>((work + 255) / 256);
    blocks = blocks < 1 ? 1 : (blocks > 1216 ? 1216 : blocks);
    return launch_pdl(tree_init_kernel, dim3(blocks), dim3(256), 0, stream, d, ws);
}

cudaError_t launch_rerank(const TreeDims& d, const TreeWs& ws, cudaStream_t stream) {
    int P = 2;
    while (P < d.C) P <<= 1;
    return launch_pdl(rerank_kernel, dim3(d.B), dim3(kSortThreads), 0, stream, d, ws, P);
}

cudaError_t launch_tree_value(const TreeDims& d, const TreeWs& ws, float* value_sum, cudaStream_t stream) {
    return launch_pdl(tree_value_kernel, dim3(d.B), dim3(32), 0, stream, d, ws, value_sum);
}

cudaError_t launch_build_tree(const TreeDims& d, const TreeWs& ws, const int32_t* prefix_len,
                              const int32_t* root_token, int32_t* tokens, int32_t* parent, int32_t* depth,
                              int32_t* pos, uint32_t* mask, int32_t* n_tree, cudaStream_t stream) {
    return launch_pdl(build_tree_kernel, dim3(d.B), dim3(kBuildThreads), 0, stream, d, ws, prefix_len, root_token,
                      tokens, parent, depth, pos, mask, n_tree);
}

}  // namespace eagle

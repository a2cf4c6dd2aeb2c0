// Vocabulary-row kernels of the draft-tree cycle (sm_103a):
//   expand_kernel  stages 1+2: per frontier row softmax statistics + top-k,
//                  child values, then (last row of a sequence) the next frontier.
//   verify_kernel  stage 6: per target row max/argmax (+ integer mass), then
//                  (last row of a sequence) the acceptance walk.
//
// Layout of the work: one logit row is split over a thread-block cluster of
// `cpr` CTAs. Each CTA stages its contiguous chunk of the row in shared memory
// with one bulk asynchronous copy (TMA engine, completion on an mbarrier), so
// HBM is read exactly once; each warp then owns a contiguous part of the
// chunk and reduces it without block-wide barriers. Partial results are
// pushed into the cluster leader's shared memory with remote stores before a
// single cluster barrier. The per-sequence tail (frontier selection /
// acceptance walk) runs in the cluster leader that arrives last on a
// per-sequence ticket: an atomic add after a device-scope fence, no spin-wait.
//
// Top-k of a warp's part: with key = (value, -id) unique per element, let tau
// be the k-th largest of the 32 lane maxima. The k lane maxima >= tau are k
// distinct elements, so every element of the part's top-k has key >= tau; the
// few elements >= tau are gathered and sorted. The union of the warps' top-k
// contains the chunk's top-k, and so on up the cluster.
//
// Sources (page title and section): "EAGLE" notes (garden.houmin.site),
// EAGLE 方法 (TopK drafting) and EAGLE 2 方法 (Expand, threshold);
// "EAGLE-2: Faster Inference ..." summary, 2.1 Speculative Sampling and 4.1
// Expansion Phase; "EAGLE-2: Dynamic Draft Trees" tutorial, "Value of a Node =
// Its Path Product".

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "eagle_internal.cuh"
#include "eagle_ws.h"

namespace eagle {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kWarpCand = 64;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ helpers ---

struct RowChunk {
    int c0;  // first token id of this CTA's chunk
    int n;   // tokens in the chunk (may be 0)
};

template <int DT>
__device__ __forceinline__ void unpack16(const uint4& u, float* x) {
    if (DT == 1) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        x[0] = __uint_as_float(u.x);
        x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z);
        x[3] = __uint_as_float(u.w);
    }
}

// Largest element of a 16-byte vector (NaN elements are ignored).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& u) {
    if (DT == 1) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&u.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&u.w);
        const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return fmaxf(__low2float(m), __high2float(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                     fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
    }
}

// Descending bitonic sort of 32 unsigned values, one per lane.
__device__ __forceinline__ uint32_t warp_sort_desc_u32(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int s = size >> 1; s > 0; s >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, s);
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & s) == 0;
            v = (lower == desc) ? max(o, v) : min(o, v);
        }
    }
    return v;
}

// Issue the bulk copy of this CTA's chunk into `buf` and wait for it.
__device__ __forceinline__ bool stage_chunk(void* buf, const char* row_base, const RowChunk& ch, int esize,
                                            uint64_t* bar, int* status) {
    const uint32_t bytes = static_cast<uint32_t>(ch.n) * esize;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (bytes == 0) return true;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(buf, row_base + static_cast<size_t>(ch.c0) * esize, bytes, bar);
    }
    if (!mbar_wait(bar, 0)) {
        raise_status(status, kDevTimeout);
        return false;
    }
    return true;
}

// Descending bitonic sort of 32*E keys held by one warp, E per lane
// (element e = lane*E + j).
template <int E>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&v)[E]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32 * E; size <<= 1) {
#pragma unroll
        for (int s = size >> 1; s > 0; s >>= 1) {
            if (s < E) {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int pj = j ^ s;
                    if (pj > j) {
                        const int e = lane * E + j;
                        const bool desc = (e & size) == 0;
                        const uint64_t a = v[j], c = v[pj];
                        if ((a < c) == desc) {
                            v[j] = c;
                            v[pj] = a;
                        }
                    }
                }
            } else {
                const int ls = s / E;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const uint64_t o = shfl_xor_u64(v[j], ls);
                    const int e = lane * E + j;
                    const bool desc = (e & size) == 0;
                    const bool lower = (e & s) == 0;
                    const bool keep_max = lower == desc;
                    v[j] = keep_max ? (o > v[j] ? o : v[j]) : (o < v[j] ? o : v[j]);
                }
            }
        }
    }
}

// Top-k (k <= 16) of n <= 32*E keys in shared memory by one warp; writes
// out[0..k), 0 = no key.
template <int E>
__device__ __forceinline__ void warp_topk_sorted(const uint64_t* keys, int n, int k, uint64_t* out) {
    const int lane = threadIdx.x & 31;
    uint64_t v[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int e = lane * E + j;
        v[j] = e < n ? keys[e] : 0ull;
    }
    warp_sort_desc<E>(v);
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int e = lane * E + j;
        if (e < k) out[e] = v[j];
    }
    __syncwarp();
}

// ------------------------------------------------------------ expand kernel ---

struct ExpandSmem {
    uint64_t bar;
    uint64_t wcand[kRowWarps][kWarpCand];
    int wcount[kRowWarps];
    uint64_t wtop[kRowWarps * kMaxTopK];
    float wm[kRowWarps];
    float ws[kRowWarps];
    // filled by every CTA of the cluster in the leader's copy (remote stores)
    uint64_t rtop[kMaxChunks * kMaxTopK];
    float rm[kMaxChunks];
    float rs[kMaxChunks];
    uint64_t top[kMaxTopK];
    uint64_t sel[kMaxTopK * kMaxTopK];
    int last;
};

template <int DT>
__global__ void __launch_bounds__(kRowThreads) expand_kernel(TreeDims d, TreeWs w, int step, int chunk,
                                                              const void* __restrict__ logits,
                                                              const float* __restrict__ lse_in,
                                                              float* __restrict__ row_lse,
                                                              int32_t* __restrict__ ftok_out,
                                                              int32_t* __restrict__ fcount_out) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ ExpandSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cpr = static_cast<int>(cluster.num_blocks());
    const int row = blockIdx.y;
    const int b = row / d.k, f = row % d.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int F = w.fcount[step * d.B + b];
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int EPV = 16 / ES;
    const int k = d.k;

    if (f >= F) {  // this frontier slot holds no node in this step
        if (rank == 0 && tid == 0) {
            row_lse[(static_cast<size_t>(b) * d.D + step) * d.k + f] = __int_as_float(0x7fc00000);
            if (f == 0) {  // F == 0: nothing to expand, the next frontier is empty
                fcount_out[b] = 0;
                for (int j = 0; j < d.k; ++j) ftok_out[b * d.k + j] = -1;
            }
        }
        return;
    }

    RowChunk ch;
    ch.c0 = rank * chunk;
    ch.n = max(0, min(chunk, d.V - ch.c0));
    const char* row_base = static_cast<const char*>(logits) + static_cast<size_t>(b * d.k + f) * d.V * ES;
    const uint4* buf = reinterpret_cast<const uint4*>(dyn_smem);
    if (tid < kRowWarps) sm.wcount[tid] = 0;
    stage_chunk(dyn_smem, row_base, ch, ES, &sm.bar, w.status);

    // ---- per warp: a contiguous part of the chunk ----
    const int nvec = ch.n / EPV;
    const int vpw = (nvec + kRowWarps - 1) / kRowWarps;
    const int v0 = warp * vpw, v1 = min(nvec, v0 + vpw);
    // pass 1: lane maximum (packed compares for bf16)
    float lmax = -INFINITY;
    bool lhas = false;
    for (int v = v0 + lane; v < v1; v += 32) {
        lmax = fmaxf(lmax, vec_max<DT>(buf[v]));
        lhas = true;
    }
    // tau = k-th largest lane maximum: at least k elements of the part are
    // >= tau, so its top-k all are (0 bits: fewer than k lanes with elements)
    const uint32_t lo = warp_sort_desc_u32(lhas ? f2o(lmax) : 0u);
    const uint32_t tau_o = __shfl_sync(0xffffffffu, lo, k - 1);
    const uint32_t wmax_o = __shfl_sync(0xffffffffu, lo, 0);
    const bool take_all = tau_o == 0u;
    const float tau = o2f(tau_o);
    const float wmax = wmax_o ? o2f(wmax_o) : -INFINITY;
    // pass 2: exp-sum (fp32) and candidates >= tau
    float s = 0.0f;
    const bool do_sum = lse_in == nullptr && wmax > -INFINITY;
    const float mb = wmax * kLog2e;
    for (int v = v0 + lane; v < v1; v += 32) {
        const uint4 u = buf[v];
        float x[EPV];
        unpack16<DT>(u, x);
        if (do_sum) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) s += ex2_approx(fmaf(x[e], kLog2e, -mb));
        }
        if (take_all || vec_max<DT>(u) >= tau) {
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                if (take_all || x[e] >= tau) {
                    const int at = atomicAdd(&sm.wcount[warp], 1);
                    if (at < kWarpCand) sm.wcand[warp][at] = make_key(x[e], static_cast<uint32_t>(ch.c0 + v * EPV + e));
                }
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    __syncwarp();
    const int cnt = sm.wcount[warp];
    if (cnt <= kWarpCand) {
        warp_topk_sorted<2>(sm.wcand[warp], cnt, k, &sm.wtop[warp * kMaxTopK]);
    } else {
        // Many equal values at the top: k exact rounds over the warp's part.
        uint64_t prev = ~0ull;
        for (int r = 0; r < k; ++r) {
            uint64_t best = 0;
            for (int v = v0 + lane; v < v1; v += 32) {
                float x[EPV];
                unpack16<DT>(buf[v], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const uint64_t key = make_key(x[e], static_cast<uint32_t>(ch.c0 + v * EPV + e));
                    if (key < prev && key > best) best = key;
                }
            }
            best = warp_max_u64(best);
            if (lane == 0) sm.wtop[warp * kMaxTopK + r] = best;
            prev = best;
        }
        __syncwarp();
    }
    if (lane == 0) {
        sm.wm[warp] = wmax;
        sm.ws[warp] = s;
    }
    __syncthreads();

    // ---- CTA: merge the warps, push to the cluster leader ----
    ExpandSmem* leader = cluster.map_shared_rank(&sm, 0);
    if (warp == 0) {
        // the 8 warps' top-k: k <= 16, so 8 * 16 = 128 slots, 4 per lane
        uint64_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = lane * 4 + j;  // e = warp_index * 16 + r
            const int wi = e >> 4, r = e & 15;
            v[j] = r < k ? sm.wtop[wi * kMaxTopK + r] : 0ull;
        }
        warp_sort_desc<4>(v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = lane * 4 + j;
            if (e < k) leader->rtop[rank * kMaxTopK + e] = v[j];
        }
        if (lane == 0) {
            float M = -INFINITY;
            for (int i = 0; i < kRowWarps; ++i) M = fmaxf(M, sm.wm[i]);
            float S = 0.0f;
            if (M > -INFINITY)
                for (int i = 0; i < kRowWarps; ++i)
                    if (sm.wm[i] > -INFINITY) S += sm.ws[i] * ex2_approx((sm.wm[i] - M) * kLog2e);
            leader->rm[rank] = M;
            leader->rs[rank] = S;
        }
    }
    cluster.sync();
    if (rank != 0) return;

    // ---- leader: row top-k and lse ----
    if (warp == 0) {
        uint64_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = lane * 4 + j;  // e = rank_index * 16 + r
            const int ri = e >> 4, r = e & 15;
            v[j] = (ri < cpr && r < k) ? sm.rtop[ri * kMaxTopK + r] : 0ull;
        }
        warp_sort_desc<4>(v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = lane * 4 + j;
            if (e < k) sm.top[e] = v[j];
        }
        if (lane == 0) {
            float M = -INFINITY;
            for (int r = 0; r < cpr; ++r) M = fmaxf(M, sm.rm[r]);
            float S = 0.0f;
            if (M > -INFINITY)
                for (int r = 0; r < cpr; ++r)
                    if (sm.rm[r] > -INFINITY) S += sm.rs[r] * ex2_approx((sm.rm[r] - M) * kLog2e);
            sm.wm[0] = M;
            sm.ws[0] = S;
        }
    }
    __syncthreads();

    // Children of this frontier node.
    const float lse = lse_in != nullptr ? lse_in[b * d.k + f] : sm.wm[0] + logf(sm.ws[0]);
    const int parent = w.fnode[(step * d.B + b) * d.k + f];
    const float plogv = parent < 0 ? 0.0f : w.cand_logv[static_cast<size_t>(b) * d.C + parent];
    const int base = step == 0 ? 0 : d.k + (step - 1) * d.k * d.k;
    if (tid < d.k) {
        const uint64_t key = sm.top[tid];
        const int id = base + f * d.k + tid;
        const size_t at = static_cast<size_t>(b) * d.C + id;
        if (key != 0) {
            const float x = key_val(key);
            const float lp = __fsub_rn(x, lse);
            w.cand_token[at] = static_cast<int32_t>(key_id(key));
            w.cand_parent[at] = parent;
            w.cand_depth[at] = step + 1;
            w.cand_logv[at] = __fadd_rn(plogv, lp);
            w.cand_valid[at] = 1;
        }
    }
    if (tid == 0) {
        row_lse[(static_cast<size_t>(b) * d.D + step) * d.k + f] = lse;
        if (!isfinite(lse)) raise_status(w.status, kDevNonFinite);
    }
    __syncthreads();

    // Per-sequence ticket: the last row of this sequence picks the next frontier.
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(&w.expand_ticket[b], 1);
        sm.last = (prev == F - 1);
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    if (warp == 0) {
        const int n = F * d.k;
        for (int i = lane; i < n; i += 32) {
            const int id = base + i;
            const size_t at = static_cast<size_t>(b) * d.C + id;
            const bool valid = __ldcg(reinterpret_cast<const unsigned char*>(&w.cand_valid[at])) != 0;
            const float lv = __ldcg(&w.cand_logv[at]);
            sm.sel[i] = (valid && lv >= d.log_thr) ? make_key(lv, static_cast<uint32_t>(id)) : 0ull;
        }
        __syncwarp();
        warp_topk_smem(sm.sel, n, d.k, sm.top);
        int cnt = 0;
        for (int j = 0; j < d.k; ++j) cnt += sm.top[j] != 0;
        if (lane < d.k) {
            const uint64_t key = sm.top[lane];
            const int id = key ? static_cast<int>(key_id(key)) : -1;
            w.fnode[((step + 1) * d.B + b) * d.k + lane] = id;
            ftok_out[b * d.k + lane] = id >= 0 ? __ldcg(&w.cand_token[static_cast<size_t>(b) * d.C + id]) : -1;
        }
        if (lane == 0) {
            w.fcount[(step + 1) * d.B + b] = cnt;
            fcount_out[b] = cnt;
            w.expand_ticket[b] = 0;
        }
    }
}

// ------------------------------------------------------------ verify kernel ---

// Fixed-order exp for lossless verification (contract in eagle.h): Cody-Waite
// reduction with ln2 = 0x1.62e4p-1 + 0x1.7f7d1cp-20, degree-7 Taylor series of
// exp(r) in Horner form, exact scaling by 2^n; every step one correctly
// rounded fp32 multiply or add. z <= 0; returns 0 below -32.
__device__ __forceinline__ float dexp_fixed(float z) {
    if (!(z >= -32.0f)) return 0.0f;
    const float n = rintf(__fmul_rn(z, 0x1.715476p+0f));
    float r = __fsub_rn(z, __fmul_rn(n, 0x1.62e4p-1f));
    r = __fsub_rn(r, __fmul_rn(n, 0x1.7f7d1cp-20f));
    float p = 0x1.a01a02p-13f;                           // 1/7!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);     // 1/6!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);      // 1/5!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);      // 1/4!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);      // 1/3!
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);                // 1/2!
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);                // 1/1!
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);                // 1/0!
    const float scale = __int_as_float((static_cast<int>(n) + 127) << 23);
    return __fmul_rn(p, scale);
}

// Integer mass floor(dexp((x - m) * inv_t) * 2^40).
__device__ __forceinline__ uint64_t fixed_mass(float x, float m, float inv_t) {
    const float e = dexp_fixed(__fmul_rn(__fsub_rn(x, m), inv_t));
    return __float2ull_rz(__fmul_rn(e, 0x1p40f));
}

struct VerifySmem {
    uint64_t bar;
    uint64_t wkey[kRowWarps];
    uint64_t wmass[kRowWarps];
    uint64_t rkey[kMaxChunks];   // every rank's chunk maximum (pushed to every rank)
    uint64_t rmass[kMaxChunks];  // every rank's chunk mass (pushed to the leader)
    int last;
    // walk state (last-arriving CTA of a sequence)
    int tok[kMaxSlots];
    int par[kMaxSlots];
    int arg[kMaxSlots];
    float rmax[kMaxSlots];
    unsigned long long rowmass[kMaxSlots];
    unsigned long long pmass[kMaxSlots];  // mass of slot c's token in its parent's row
    uint32_t uni[kMaxSlots + 2];
    int path[kMaxDepth + 1];
    int removed_tok[kMaxSlots];
    unsigned long long removed_mass[kMaxSlots];
    unsigned long long wscan[kRowWarps];
    int n_removed, a, cur, sample_chunk, bonus, bad, found;
    unsigned long long sample_t;
};

template <int DT>
__global__ void __launch_bounds__(kRowThreads) verify_kernel(TreeDims d, TreeWs w, int mode, float inv_t, int chunk,
                                                              const void* __restrict__ target,
                                                              const int32_t* __restrict__ tokens,
                                                              const int32_t* __restrict__ parent,
                                                              const int32_t* __restrict__ n_tree,
                                                              const uint32_t* __restrict__ uniforms,
                                                              int32_t* __restrict__ accept_len,
                                                              int32_t* __restrict__ slots_out,
                                                              int32_t* __restrict__ tokens_out) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ VerifySmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cpr = static_cast<int>(cluster.num_blocks());
    const int row = blockIdx.y;
    const int b = row / d.T, t = row % d.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int EPV = 16 / ES;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int n = n_tree[b];
    if (n < 1 || n > d.T) {
        if (rank == 0 && t == 0 && tid == 0) raise_status(w.status, kDevBadIndex);
        return;
    }
    if (t >= n) return;

    RowChunk ch;
    ch.c0 = rank * chunk;
    ch.n = max(0, min(chunk, d.V - ch.c0));
    const char* row_base = static_cast<const char*>(target) + static_cast<size_t>(b * d.T + t) * d.V * ES;
    const uint4* buf = reinterpret_cast<const uint4*>(dyn_smem);
    stage_chunk(dyn_smem, row_base, ch, ES, &sm.bar, w.status);

    // ---- pass 1: maximum (lowest id among equal values) ----
    const int nvec = ch.n / EPV;
    const int vpw = (nvec + kRowWarps - 1) / kRowWarps;
    const int v0 = warp * vpw, v1 = min(nvec, v0 + vpw);
    float lmax = -INFINITY;
    int larg = -1;
    for (int v = v0 + lane; v < v1; v += 32) {
        const uint4 u = buf[v];
        const float m8 = vec_max<DT>(u);
        if (larg < 0 || m8 > lmax) {  // first element equal to the vector maximum: lowest id
            float x[EPV];
            unpack16<DT>(u, x);
            int e0 = 0;
#pragma unroll
            for (int e = EPV - 1; e >= 0; --e)
                if (x[e] == m8) e0 = e;
            lmax = m8;
            larg = ch.c0 + v * EPV + e0;
        }
    }
    uint64_t key = larg < 0 ? 0ull : make_key(lmax, static_cast<uint32_t>(larg));
    key = warp_max_u64(key);
    if (lane == 0) sm.wkey[warp] = key;
    __syncthreads();
    if (warp == 0) {
        uint64_t m = lane < kRowWarps ? sm.wkey[lane] : 0ull;
        m = warp_max_u64(m);
        if (lane < cpr) cluster.map_shared_rank(&sm, lane)->rkey[rank] = m;  // to every rank
    }
    cluster.sync();
    uint64_t gkey = 0;
    for (int r = 0; r < cpr; ++r) gkey = sm.rkey[r] > gkey ? sm.rkey[r] : gkey;
    const float M = key_val(gkey);
    const size_t rt = static_cast<size_t>(b) * d.T + t;
    if (mode == 1) {
        // ---- pass 2: integer mass of the chunk ----
        uint64_t s = 0;
        for (int v = v0 + lane; v < v1; v += 32) {
            float x[EPV];
            unpack16<DT>(buf[v], x);
#pragma unroll
            for (int e = 0; e < EPV; ++e) s += fixed_mass(x[e], M, inv_t);
        }
        s = warp_sum_u64(s);
        if (lane == 0) sm.wmass[warp] = s;
        __syncthreads();
        if (warp == 0) {
            uint64_t tot = lane < kRowWarps ? sm.wmass[lane] : 0ull;
            tot = warp_sum_u64(tot);
            if (lane == 0) {
                w.chunk_mass[rt * kMaxChunks + rank] = tot;
                cluster.map_shared_rank(&sm, 0)->rmass[rank] = tot;
            }
        }
        cluster.sync();
    }
    if (rank != 0) return;
    if (tid == 0) {
        uint64_t mass = 0;
        if (mode == 1)
            for (int r = 0; r < cpr; ++r) mass += sm.rmass[r];
        w.row_max[rt] = M;
        w.row_arg[rt] = static_cast<int32_t>(key_id(gkey));
        w.row_mass[rt] = mass;
        if (!isfinite(M)) raise_status(w.status, kDevNonFinite);
        __threadfence();
        const int prev = atomicAdd(&w.verify_ticket[b], 1);
        sm.last = (prev == n - 1);
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    // ---- acceptance walk for sequence b (one CTA) ----
    const int T = d.T;
    if (tid == 0) sm.bad = 0;
    for (int c = tid; c < T; c += kRowThreads) {
        sm.tok[c] = c < n ? tokens[static_cast<size_t>(b) * T + c] : -1;
        sm.par[c] = c < n ? parent[static_cast<size_t>(b) * T + c] : -1;
        if (c < n) {
            sm.arg[c] = __ldcg(&w.row_arg[static_cast<size_t>(b) * T + c]);
            sm.rmax[c] = __ldcg(&w.row_max[static_cast<size_t>(b) * T + c]);
            sm.rowmass[c] = __ldcg(&w.row_mass[static_cast<size_t>(b) * T + c]);
        }
    }
    // chunk masses of every row of the sequence, in the (now idle) chunk buffer
    unsigned long long* cmass = reinterpret_cast<unsigned long long*>(dyn_smem);
    if (mode == 1) {
        for (int c = tid; c < T + 2; c += kRowThreads) sm.uni[c] = uniforms[static_cast<size_t>(b) * (T + 2) + c];
        for (int q = tid; q < n * cpr; q += kRowThreads)
            cmass[q] = __ldcg(&w.chunk_mass[(static_cast<size_t>(b) * T + q / cpr) * kMaxChunks + q % cpr]);
    }
    __syncthreads();
    for (int c = 1 + tid; c < n; c += kRowThreads) {
        const int tk = sm.tok[c], p = sm.par[c];
        sm.pmass[c] = 0;
        if (tk < 0 || tk >= d.V || p < 0 || p >= c) {
            sm.bad = 1;
            continue;
        }
        if (mode == 1) {
            const char* prow = static_cast<const char*>(target) + (static_cast<size_t>(b) * T + p) * d.V * ES;
            float x;
            if (DT == 1)
                x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(prow)[tk]) << 16);
            else
                x = reinterpret_cast<const float*>(prow)[tk];
            sm.pmass[c] = fixed_mass(x, sm.rmax[p], inv_t);
        }
    }
    __syncthreads();
    if (tid == 0 && sm.bad) raise_status(w.status, kDevBadIndex);

    if (tid == 0) {
        int cur = 0, a = 0;
        sm.path[0] = 0;
        sm.n_removed = 0;
        unsigned long long S = mode == 1 ? sm.rowmass[0] : 0ull;
        for (;;) {
            int next = -1;
            if (a < d.D) {
                for (int c = cur + 1; c < n; ++c) {
                    if (sm.par[c] != cur) continue;
                    if (mode == 0) {
                        if (sm.tok[c] == sm.arg[cur]) {
                            next = c;
                            break;
                        }
                    } else {
                        const unsigned __int128 lhs = static_cast<unsigned __int128>(sm.uni[c] >> 8) * S;
                        const unsigned __int128 rhs = static_cast<unsigned __int128>(sm.pmass[c]) << 24;
                        if (lhs < rhs) {
                            next = c;
                            break;
                        }
                        S -= sm.pmass[c];
                        sm.removed_tok[sm.n_removed] = sm.tok[c];
                        sm.removed_mass[sm.n_removed] = sm.pmass[c];
                        sm.n_removed++;
                    }
                }
            }
            if (next < 0) break;
            sm.path[++a] = next;
            cur = next;
            if (mode == 1) {
                S = sm.rowmass[cur];
                sm.n_removed = 0;
            }
        }
        sm.a = a;
        sm.cur = cur;
        sm.bonus = mode == 0 ? sm.arg[cur] : -1;
        if (mode == 1) {
            // choose the chunk of row `cur` that holds the draw
            const uint64_t U64 = (static_cast<uint64_t>(sm.uni[T + 1]) << 32) | sm.uni[T];
            const unsigned long long tdraw =
                static_cast<unsigned long long>((static_cast<unsigned __int128>(U64) * S) >> 64);
            unsigned long long run = 0;
            int chosen = cpr - 1;
            unsigned long long tin = 0;
            for (int r = 0; r < cpr; ++r) {
                unsigned long long cm = cmass[cur * cpr + r];
                const int lo = r * chunk, hi = min(d.V, lo + chunk);
                for (int q = 0; q < sm.n_removed; ++q)
                    if (sm.removed_tok[q] >= lo && sm.removed_tok[q] < hi) cm -= sm.removed_mass[q];
                if (run + cm > tdraw) {
                    chosen = r;
                    tin = tdraw - run;
                    break;
                }
                run += cm;
            }
            sm.sample_chunk = chosen;
            sm.sample_t = tin;
        }
    }
    __syncthreads();

    if (mode == 1) {
        // Smallest y (not removed) of the chosen chunk of row `cur` whose
        // running mass exceeds the draw. The chunk is staged in shared memory
        // (second phase of the CTA's mbarrier) and walked in id order in
        // rounds of 256 vectors, one vector per thread, with a block scan per
        // round.
        const int cur = sm.cur;
        const int lo = sm.sample_chunk * chunk, hi = min(d.V, lo + chunk);
        const int len = max(0, hi - lo);
        const char* crow = static_cast<const char*>(target) + (static_cast<size_t>(b) * T + cur) * d.V * ES;
        fence_proxy_async_smem();  // earlier generic reads of the buffer before the async-proxy rewrite
        __syncthreads();
        if (tid == 0) {
            sm.found = 0;
            if (len > 0) {
                mbar_arrive_expect_tx(&sm.bar, static_cast<uint32_t>(len) * ES);
                bulk_g2s(dyn_smem, crow + static_cast<size_t>(lo) * ES, static_cast<uint32_t>(len) * ES, &sm.bar);
            }
        }
        if (len > 0 && !mbar_wait(&sm.bar, 1)) raise_status(w.status, kDevTimeout);
        __syncthreads();
        const float m = sm.rmax[cur];
        const int nrem = sm.n_removed;
        const int nv = len / EPV;
        unsigned long long tin = sm.sample_t;
        for (int base = 0; base < nv; base += kRowThreads) {
            const int v = base + tid;
            unsigned long long em[EPV];
            unsigned long long mv = 0;
            if (v < nv) {
                float x[EPV];
                unpack16<DT>(buf[v], x);
                const int y0 = lo + v * EPV;
                bool has_removed = false;
                for (int q = 0; q < nrem; ++q)
                    has_removed |= static_cast<unsigned>(sm.removed_tok[q] - y0) < static_cast<unsigned>(EPV);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    em[e] = fixed_mass(x[e], m, inv_t);
                    if (has_removed)
                        for (int q = 0; q < nrem; ++q)
                            if (sm.removed_tok[q] == y0 + e) em[e] = 0;
                    mv += em[e];
                }
            }
            // block exclusive scan of mv
            unsigned long long incl = mv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t lo32 = __shfl_up_sync(0xffffffffu, static_cast<uint32_t>(incl), o);
                const uint32_t hi32 = __shfl_up_sync(0xffffffffu, static_cast<uint32_t>(incl >> 32), o);
                if (lane >= o) incl += (static_cast<unsigned long long>(hi32) << 32) | lo32;
            }
            if (lane == 31) sm.wscan[warp] = incl;
            __syncthreads();
            unsigned long long wbase = 0, total = 0;
            for (int i = 0; i < kRowWarps; ++i) {
                if (i < warp) wbase += sm.wscan[i];
                total += sm.wscan[i];
            }
            const unsigned long long ex = wbase + incl - mv;
            if (mv > 0 && ex <= tin && tin < ex + mv) {
                unsigned long long run = ex;
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    run += em[e];
                    if (run > tin) {
                        sm.bonus = lo + v * EPV + e;
                        break;
                    }
                }
                sm.found = 1;
            }
            __syncthreads();
            if (sm.found) break;
            tin -= total;
        }
        __syncthreads();
    }

    if (tid == 0) {
        const int a = sm.a;
        const int Dp1 = d.D + 1;
        accept_len[b] = a;
        for (int j = 0; j < Dp1; ++j) {
            slots_out[b * Dp1 + j] = j <= a ? sm.path[j] : -1;
            tokens_out[b * Dp1 + j] = j < a ? sm.tok[sm.path[j + 1]] : (j == a ? sm.bonus : -1);
        }
        if (sm.bonus < 0) raise_status(w.status, kDevBadIndex);
        w.verify_ticket[b] = 0;
    }
}

// -------------------------------------------------------------- launchers ---

RowSplit choose_row_split(int V, int esize) {
    RowSplit s;
    const long row_bytes = static_cast<long>(V) * esize;
    int cpr = 1;
    while (cpr < kMaxChunks && row_bytes > static_cast<long>(cpr) * 32 * 1024) cpr *= 2;
    const int epv = 16 / esize;
    int chunk = (V + cpr - 1) / cpr;
    chunk = (chunk + epv - 1) / epv * epv;
    s.cpr = cpr;
    s.chunk = chunk;
    s.smem_bytes = static_cast<int>(align_up(static_cast<size_t>(chunk) * esize, 128));
    return s;
}

cudaError_t ensure_dyn_smem(const void* kernel, int smem) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const std::pair<const void*, int> key(kernel, dev);
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) done[key] = smem;
    return e;
}

template <typename K>
static cudaError_t launch_rows(K kernel, dim3 grid, int cpr, int smem, cudaStream_t stream, void** args) {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cpr;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
}

cudaError_t launch_expand(const TreeDims& d, const TreeWs& ws, int step, const void* logits, const float* lse_in,
                          float* row_lse, int32_t* ftok, int32_t* fcount_out, cudaStream_t stream) {
    const RowSplit s = choose_row_split(d.V, d.dtype == 1 ? 2 : 4);
    dim3 grid(s.cpr, d.B * d.k, 1);
    TreeDims dd = d;
    TreeWs ww = ws;
    int chunk = s.chunk;
    void* args[] = {&dd,      &ww,   &step,       &chunk, const_cast<void**>(&logits), const_cast<float**>(&lse_in),
                    &row_lse, &ftok, &fcount_out};
    return d.dtype == 1 ? launch_rows(expand_kernel<1>, grid, s.cpr, s.smem_bytes, stream, args)
                        : launch_rows(expand_kernel<0>, grid, s.cpr, s.smem_bytes, stream, args);
}

cudaError_t launch_verify(const TreeDims& d, const TreeWs& ws, int mode, float inv_temp, const void* target,
                          const int32_t* tokens, const int32_t* parent, const int32_t* n_tree,
                          const uint32_t* uniforms, int32_t* accept_len, int32_t* slots, int32_t* out_tokens,
                          cudaStream_t stream) {
    const RowSplit s = choose_row_split(d.V, d.dtype == 1 ? 2 : 4);
    dim3 grid(s.cpr, d.B * d.T, 1);
    // the acceptance walk keeps the chunk masses of all T rows in the chunk buffer
    const int smem = static_cast<int>(std::max<size_t>(s.smem_bytes, align_up(static_cast<size_t>(d.T) * s.cpr * 8, 128)));
    TreeDims dd = d;
    TreeWs ww = ws;
    int chunk = s.chunk;
    void* args[] = {&dd,
                    &ww,
                    &mode,
                    &inv_temp,
                    &chunk,
                    const_cast<void**>(&target),
                    const_cast<int32_t**>(&tokens),
                    const_cast<int32_t**>(&parent),
                    const_cast<int32_t**>(&n_tree),
                    const_cast<uint32_t**>(&uniforms),
                    &accept_len,
                    &slots,
                    &out_tokens};
    return d.dtype == 1 ? launch_rows(verify_kernel<1>, grid, s.cpr, smem, stream, args)
                        : launch_rows(verify_kernel<0>, grid, s.cpr, smem, stream, args);
}

}  // namespace eagle

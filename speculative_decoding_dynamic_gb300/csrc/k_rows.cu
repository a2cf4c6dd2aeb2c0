// Vocabulary-row kernels of the draft-tree cycle (sm_103a):
//   expand_kernel  stages 1+2: per frontier row softmax statistics + top-k,
//                  child values, then (last row of a sequence) the next frontier.
//   verify_kernel  stage 6: per target row max/argmax (+ integer mass), then
//                  (last row of a sequence) the acceptance walk.
//
// Layout of the work. A logit row is split into `cpr` contiguous segments,
// one per CTA of a thread-block cluster; cpr (1..8) is chosen per launch so
// that the grid holds about two waves of CTAs. Each CTA runs eight consumer
// warps and one producer warp. The producer streams the segment through a
// ring of 16 KB shared-memory stages with bulk asynchronous copies (TMA
// engine): a "full" mbarrier per stage counts the bytes, an "empty" mbarrier
// counts the consumer warps that are done with it, so HBM is read once and
// the copies of later chunks overlap the arithmetic on earlier ones. Within a
// chunk every consumer warp owns 128 consecutive 16-byte vectors, four per
// lane, and keeps its running statistics in registers across chunks.
//
// Expansion, one pass over the data: per lane a running maximum and a
// rescaled exp-sum (online normaliser), and the maximum of each lane group
// (the lane's four vectors of one chunk). After the pass, the admission key
// tau = the k-th largest lane maximum of the CTA's segment (k distinct
// elements reach it, so every element of the segment's top-k does, and lies
// in a group whose maximum reaches it). Only those groups are
// read again (from the stages when the segment stayed resident, else from
// L2) and their keys >= tau ranked. Keys are (value, -id): unique, so ties go
// to the lower token id. CTA and cluster results are merged by rank
// selection (each key counts the keys above it). Partial results are pushed
// into the cluster leader's shared memory before one cluster barrier. The
// per-sequence tail (frontier selection / acceptance walk) runs in the
// cluster leader that arrives last on a per-sequence ticket: an atomic add
// after a device-scope fence, no spin-wait.
//
// Sources (page title and section): "EAGLE" notes (garden.houmin.site),
// EAGLE 方法 (TopK drafting) and EAGLE 2 方法 (Expand, threshold);
// "EAGLE-2: Faster Inference ..." summary, 2.1 Speculative Sampling and 4.1
// Expansion Phase; "EAGLE-2: Dynamic Draft Trees" tutorial, "Value of a Node =
// Its Path Product".

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>

#include "eagle_internal.cuh"
#include "eagle_ws.h"
#include "mass.cuh"
#include "sampling.cuh"

namespace eagle {

constexpr int kConsumerWarps = kRowWarpsPerCta;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kRowThreads = (kConsumerWarps + 1) * 32;
constexpr int kVecPerLane = 4;
constexpr int kVecPerWarp = 32 * kVecPerLane;
static_assert(kVecPerWarp * kConsumerWarps * 16 == kRowChunkBytes, "chunk geometry");
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kMaxSegChunks = 8;  // chunks of one CTA's row segment in expansion (fp32 rows)
// bf16 rows: group maxima are bf16 values, whose order-preserving bits are
// decided by their top half, so 16 bits per group and twice the chunks fit
constexpr int kMaxSegChunksBf16 = 2 * kMaxSegChunks;
template <int DT>
__host__ __device__ constexpr int max_seg_chunks() { return DT == 1 ? kMaxSegChunksBf16 : kMaxSegChunks; }
constexpr int kExpandStages = 2;  // five CTAs per SM (40 registers, ~43 KB shared memory each)
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ helpers ---

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

// A vector of -inf elements (fills the lanes past the end of a chunk).
template <int DT>
__device__ __forceinline__ uint4 neg_inf_vec() {
    const uint32_t w = DT == 1 ? 0xff80ff80u : 0xff800000u;
    return make_uint4(w, w, w, w);
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); }

// Largest element of a 16-byte vector (NaN elements are ignored).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& u) {
    if (DT == 1) {
        const __nv_bfloat162 m = __hmax2(__hmax2(as_bf2(u.x), as_bf2(u.y)), __hmax2(as_bf2(u.z), as_bf2(u.w)));
        return fmaxf(__low2float(m), __high2float(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                     fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
    }
}

// Largest element of a lane's four vectors (packed compares for bf16).
template <int DT>
__device__ __forceinline__ float lane_max4(const uint4 (&u)[kVecPerLane]) {
    if (DT == 1) {
        __nv_bfloat162 m[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j)
            m[j] = __hmax2(__hmax2(as_bf2(u[j].x), as_bf2(u[j].y)), __hmax2(as_bf2(u[j].z), as_bf2(u[j].w)));
        const __nv_bfloat162 a = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
        return fmaxf(__low2float(a), __high2float(a));
    } else {
        return fmaxf(fmaxf(vec_max<DT>(u[0]), vec_max<DT>(u[1])), fmaxf(vec_max<DT>(u[2]), vec_max<DT>(u[3])));
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

__device__ __forceinline__ uint32_t shfl_xor_key(uint32_t v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ uint64_t shfl_xor_key(uint64_t v, int m) { return shfl_xor_u64(v, m); }

// Descending bitonic sort of 32*E keys held by one warp, E per lane
// (element e = lane*E + j).
template <int E, typename K>
__device__ __forceinline__ void warp_sort_desc(K (&v)[E]) {
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
                        const K a = v[j], c = v[pj];
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
                    const K o = shfl_xor_key(v[j], ls);
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


// Rank of `key` among the first n of kMaxChunks lists of kMaxTopK keys
// (zeros = empty): how many keys are larger. Every list is read whole (zero
// padding counts nothing); all kMaxChunks lists are read, so that the loads
// are issued back to back, and the ones past n are not counted.
__device__ __forceinline__ int rank_in_lists(const uint64_t* lists, int n, uint64_t key) {
    int r = 0;
#pragma unroll
    for (int l = 0; l < kMaxChunks; ++l) {
        const ulonglong2* p = reinterpret_cast<const ulonglong2*>(lists + l * kMaxTopK);
        int rl = 0;
#pragma unroll
        for (int q = 0; q < kMaxTopK / 2; ++q) {
            const ulonglong2 a = p[q];
            rl += (a.x > key) + (a.y > key);
        }
        r += l < n ? rl : 0;
    }
    return r;
}

// Rank of `key` among n keys (a 16-byte aligned list zero-padded to a
// multiple of 8): how many are larger. Eight keys per step, loads first.
__device__ __forceinline__ int rank_in_list(const uint64_t* list, int n, uint64_t key) {
    const ulonglong2* p = reinterpret_cast<const ulonglong2*>(list);
    int r = 0;
    for (int q = 0; q < (n + 7) / 8 * 4; q += 4) {
        ulonglong2 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = p[q + u];
#pragma unroll
        for (int u = 0; u < 4; ++u) r += (a[u].x > key) + (a[u].y > key);
    }
    return r;
}

// --------------------------------------------------------- the chunk ring ---

struct RowRing {
    uint64_t full[kRowStages];
    uint64_t empty[kRowStages];
};

__device__ __forceinline__ void ring_init(RowRing& r, int ns) {
    for (int s = 0; s < ns; ++s) {
        mbar_init(&r.full[s], 1);
        mbar_init(&r.empty[s], kConsumerWarps);
    }
    fence_mbar_init();
}

// Producer (one thread): chunk c of the segment goes to stage c % ns once the
// consumers have released that stage's previous chunk.
__device__ __forceinline__ void ring_produce(RowRing& r, unsigned char* stages, const char* src, int seg_bytes,
                                             int nch, int ns, int* status) {
    for (int c = 0; c < nch; ++c) {
        const int s = c % ns;
        if (c >= ns && !mbar_wait_sleep(&r.empty[s], ((c / ns) - 1) & 1)) {
            raise_status(status, kDevTimeout);
            return;
        }
        const uint32_t bytes = static_cast<uint32_t>(min(kRowChunkBytes, seg_bytes - c * kRowChunkBytes));
        mbar_arrive_expect_tx(&r.full[s], bytes);
        bulk_g2s(stages + s * kRowChunkBytes, src + static_cast<size_t>(c) * kRowChunkBytes, bytes, &r.full[s]);
    }
}

// Consumer warp: wait (bounded) until chunk c has landed. After a first
// timeout later waits are short, so a failed launch still ends promptly.
__device__ __forceinline__ bool ring_wait(RowRing& r, int c, int ns, bool& failed, int* status) {
    bool ok = mbar_wait_sleep(&r.full[c % ns], (c / ns) & 1, failed ? 16u : (1u << 16));
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        failed = true;
        if ((threadIdx.x & 31) == 0) raise_status(status, kDevTimeout);
    }
    return ok;
}

// Consumer warp: done reading chunk c (its vectors are in registers).
__device__ __forceinline__ void ring_release(RowRing& r, int c, int ns) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[c % ns]);
}

// This lane's four vectors of a chunk (-inf past the end of the chunk).
template <int DT>
__device__ __forceinline__ void load_lane(const unsigned char* stage, int nvec, int warp, int lane,
                                          uint4 (&u)[kVecPerLane]) {
    const uint4* vb = reinterpret_cast<const uint4*>(stage) + warp * kVecPerWarp + lane;
    if (nvec == kVecPerWarp * kConsumerWarps) {  // a full chunk
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) u[j] = vb[j * 32];
        return;
    }
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
        const int v = warp * kVecPerWarp + j * 32 + lane;
        u[j] = v < nvec ? vb[j * 32] : neg_inf_vec<DT>();
    }
}

// ------------------------------------------------------------ expand kernel ---

// Barrier of the eight consumer warps only (the producer warp keeps streaming).
__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

struct ExpandSmem {
    RowRing ring;
    unsigned long long tau;                       // segment admission key
    alignas(16) uint32_t wtop[kConsumerWarps][kMaxTopK];  // each warp's k largest lane maxima (ordered bits)
    uint32_t gmax[kMaxSegChunks][kConsumers];     // maximum of each lane group (ordered bits; see gmax_put)
    int ngroups, nkeys;
    int F, parent;                                // this step's frontier count; the row's parent node
    float plogv;                                  // the parent's log path value
    float wm[kConsumerWarps];
    float ws[kConsumerWarps];
    uint64_t ctop[kMaxTopK];
    // filled by every CTA of the cluster in the leader's copy (remote stores)
    alignas(16) uint64_t rtop[kMaxChunks * kMaxTopK];
    float rm[kMaxChunks];
    float rs[kMaxChunks];
    uint64_t top[kMaxTopK];
    int last;
};

// Group maximum of lane group (chunk c, consumer thread t), as ordered bits.
// bf16 rows keep the top 16 bits only (exact for bf16 values: equal top
// halves mean equal values), read back as (top << 16); compare them with
// gmax_floor(tau). 0 marks a group without elements.
template <int DT>
__device__ __forceinline__ void gmax_put(ExpandSmem& sm, int c, int t, uint32_t o) {
    if (DT == 1)
        reinterpret_cast<uint16_t*>(&sm.gmax[0][0])[c * kConsumers + t] = static_cast<uint16_t>(o >> 16);
    else
        sm.gmax[c][t] = o;
}
template <int DT>
__device__ __forceinline__ uint32_t gmax_get(const ExpandSmem& sm, int c, int t) {
    if (DT == 1) return static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(&sm.gmax[0][0])[c * kConsumers + t]) << 16;
    return sm.gmax[c][t];
}
template <int DT>
__device__ __forceinline__ uint32_t gmax_floor(uint32_t o) { return DT == 1 ? (o & 0xFFFF0000u) : o; }

// Sampled drafting: the children of a row are drawn from its softmax without
// replacement by the Gumbel-top-k identity, keys kappa = fl(x + g), g the
// Gumbel noise of one uniform word per element ("EAGLE-2: Faster Inference
// ..." summary, 2.1 Speculative Sampling: the draft proposes tokens sampled
// from its distribution; the perturbed-key form of the draw is the reading
// taken here). The words of row r (= b * k + f) of a step come from
// Philox4x32-10 at counter (x / 4, r, step, cycle), word x % 4.
struct GumbelRng {
    uint32_t k0, k1;  // key (seed_lo ^ 10, seed_hi)
    uint32_t c2, c3;  // step, cycle
};

// The perturbed keys of one 16-byte vector whose first element is element id0
// (a multiple of 4) of row `row`.
template <int DT>
__device__ __forceinline__ void gumbel_keys(const float (&x)[16 / (DT == 1 ? 2 : 4)], int id0, uint32_t row,
                                            const GumbelRng& g, float (&kap)[16 / (DT == 1 ? 2 : 4)]) {
    constexpr int EPV = 16 / (DT == 1 ? 2 : 4);
#pragma unroll
    for (int q = 0; q < EPV; q += 4) {
        const uint32_t ctr[4] = {static_cast<uint32_t>((id0 + q) >> 2), row, g.c2, g.c3};
        uint32_t wd[4];
        sampling::philox4x32_10(ctr, g.k0, g.k1, wd);
#pragma unroll
        for (int i = 0; i < 4; ++i) kap[q + i] = __fadd_rn(x[q + i], sampling::gumbel_of_word(wd[i]));
    }
}

// Top-k keys of a CTA's row segment, after the streaming pass (consumer
// threads only). A lane group is one lane's four vectors of one chunk, and
// gmax holds each group's maximum. tau = the k-th largest lane maximum of the
// whole segment as a key with zero id bits (0: fewer than k lanes hold
// elements): k distinct elements reach it, so every element of the segment's
// top-k does, and lies in a group whose maximum reaches it; and key(x) >= tau
// exactly when x >= the value of tau. Those groups are read again (from the
// stages, or from L2: the row was just streamed), their elements >= tau
// collected, and the k largest keys found by rank selection into ctop. When the keys do not fit the scratch
// (many equal values at the top), k block-wide rounds over the candidate
// groups pick the keys one by one instead.
template <int DT, bool SAMP>
__device__ __forceinline__ void segment_topk(ExpandSmem& sm, const unsigned char* stages, bool resident,
                                             unsigned char* scratch, int scratch_bytes, const char* row_base, int c0,
                                             int n, int nch, int k, int id_base, uint32_t grow, const GumbelRng& g) {
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int EPV = 16 / ES;
    constexpr int CE = kRowChunkBytes / ES;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t tau = sm.tau;  // zero id bits: key(x) >= tau exactly when x >= tv
    const float tv = key_val(tau);
    const bool all = tau == 0ull;
    const uint32_t tau_o = static_cast<uint32_t>(tau >> 32);
    uint32_t* glist = reinterpret_cast<uint32_t*>(scratch);
    const int gcap = nch * kConsumers;
    uint64_t* keys = reinterpret_cast<uint64_t*>(scratch + gcap * sizeof(uint32_t));
    const int kcap = (scratch_bytes - gcap * static_cast<int>(sizeof(uint32_t))) / static_cast<int>(sizeof(uint64_t));
    // candidate groups: this thread's own lane groups, appended warp by warp
    for (int c = 0; c < nch; ++c) {
        const uint32_t gm = gmax_get<DT>(sm, c, tid);
        const bool hot = gm != 0u && (all || gm >= gmax_floor<DT>(tau_o));
        const unsigned bal = __ballot_sync(0xffffffffu, hot);
        if (bal == 0u) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(&sm.ngroups, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (hot) glist[base + __popc(bal & lanemask_lt())] = static_cast<uint32_t>(c * kConsumers + tid);
    }
    consumer_bar();
    const int ng = sm.ngroups;
    // element id of vector j of candidate group q
    auto group_vec = [&](uint32_t q, int j) -> int {
        const int c = static_cast<int>(q) / kConsumers, l = static_cast<int>(q) % kConsumers;
        return c0 + c * CE + ((l / 32) * kVecPerWarp + j * 32 + (l % 32)) * EPV;
    };
    // keys >= tau: one 16-byte vector of a candidate group per thread
    for (int p = tid; p < ng * kVecPerLane; p += kConsumers) {
        const uint32_t q = glist[p / kVecPerLane];
        const int id0 = group_vec(q, p % kVecPerLane);
        if (id0 >= c0 + n) continue;
        float x[EPV];
        // a resident segment is still in the stages (chunk c in stage c); else read it back from L2
        const uint4 u = resident ? reinterpret_cast<const uint4*>(stages)[(id0 - c0) / EPV]
                                 : __ldcg(reinterpret_cast<const uint4*>(row_base + static_cast<size_t>(id0) * ES));
        unpack16<DT>(u, x);
        if (SAMP) {  // the keys are the perturbed values
            float kap[EPV];
            gumbel_keys<DT>(x, id0, grow, g, kap);
#pragma unroll
            for (int e = 0; e < EPV; ++e) x[e] = kap[e];
        }
        uint32_t mask = 0;  // bit e: element e is a key >= tau (NaN never is)
#pragma unroll
        for (int e = 0; e < EPV; ++e) mask |= static_cast<uint32_t>(all ? x[e] == x[e] : x[e] >= tv) << e;
        if (mask == 0u) continue;
        int at = atomicAdd(&sm.nkeys, __popc(mask));
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            if ((mask >> e) & 1u) {
                if (at < kcap) keys[at] = make_key(x[e], static_cast<uint32_t>(id_base + id0 + e));
                ++at;
            }
    }
    consumer_bar();
    const int nk = sm.nkeys;
    if (nk <= kcap) {
        // rank = keys above; two keys per 16-byte load (the keys start 16-byte aligned)
        const ulonglong2* kp = reinterpret_cast<const ulonglong2*>(keys);
        for (int i = tid; i < nk; i += kConsumers) {
            const uint64_t key = keys[i];
            int r = 0;
            for (int j = 0; j < nk / 2; ++j) {
                const ulonglong2 q = kp[j];
                r += (q.x > key) + (q.y > key);
            }
            if (nk & 1) r += keys[nk - 1] > key;
            if (r < k) sm.ctop[r] = key;
        }
        return;
    }
    // many equal values: k rounds, each the largest key below the previous one
    uint64_t* red = keys;  // one slot per consumer warp
    uint64_t prev = ~0ull;
    for (int r = 0; r < k; ++r) {
        uint64_t best = 0;
        for (int p = tid; p < ng * kVecPerLane; p += kConsumers) {
            const int id0 = group_vec(glist[p / kVecPerLane], p % kVecPerLane);
            if (id0 >= c0 + n) continue;
            float x[EPV];
            unpack16<DT>(__ldcg(reinterpret_cast<const uint4*>(row_base + static_cast<size_t>(id0) * ES)), x);
            if (SAMP) {
                float kap[EPV];
                gumbel_keys<DT>(x, id0, grow, g, kap);
#pragma unroll
                for (int e = 0; e < EPV; ++e) x[e] = kap[e];
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                if (x[e] != x[e]) continue;
                const uint64_t key = make_key(x[e], static_cast<uint32_t>(id_base + id0 + e));
                if (key < prev && key > best) best = key;
            }
        }
        best = warp_max_u64(best);
        consumer_bar();
        if (lane == 0) red[warp] = best;
        consumer_bar();
        best = 0;
        for (int i = 0; i < kConsumerWarps; ++i) best = red[i] > best ? red[i] : best;
        if (tid == 0) sm.ctop[r] = best;
        prev = best;
        if (best == 0) break;
    }
}

// The consumer warps' part of one CTA's row segment (expansion and vocabulary
// shards): one pass over the streamed chunks for the lane maxima, the online
// exp-sum (when do_sum) and the group maxima; then tau and the segment's top-k
// keys into sm.ctop (token ids id_base + element index in the row), and the
// warps' (max, sum) into sm.wm / sm.ws.
template <int DT, bool SAMP>
__device__ __forceinline__ void segment_consume(ExpandSmem& sm, unsigned char* dyn_smem, int smem_bytes, int ns,
                                                const char* row_base, int c0, int n, int nch, int k, bool do_sum,
                                                int id_base, int* status, uint32_t grow, const GumbelRng& g) {
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int EPV = 16 / ES;
    constexpr int CE = kRowChunkBytes / ES;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // ---- one pass: lane maxima, online exp-sum, group maxima ----
    // (sampled drafting: the lane and group maxima are those of the perturbed
    // keys, kappa_l; the exp-sum stays that of the logits)
    float m_l = -INFINITY, s_l = 0.0f;  // lane: running max and sum of exp(x - m_l)
    float kappa_l = -INFINITY;
    bool failed = false;
    for (int c = 0; c < nch; ++c) {
        const bool ok = ring_wait(sm.ring, c, ns, failed, status);
        const int nvec = ok ? min(CE, n - c * CE) / EPV : 0;
        uint4 u[kVecPerLane];
        load_lane<DT>(dyn_smem + (c % ns) * kRowChunkBytes, nvec, warp, lane, u);
        ring_release(sm.ring, c, ns);
        const float cm = lane_max4<DT>(u);
        if (SAMP) {
            float km = -INFINITY;
#pragma unroll
            for (int j = 0; j < kVecPerLane; ++j) {
                float x[EPV], kap[EPV];
                unpack16<DT>(u[j], x);
                gumbel_keys<DT>(x, c0 + c * CE + (warp * kVecPerWarp + j * 32 + lane) * EPV, grow, g, kap);
#pragma unroll
                for (int e = 0; e < EPV; ++e) km = fmaxf(km, kap[e]);
            }
            gmax_put<DT>(sm, c, tid, warp * kVecPerWarp + lane < nvec ? f2o(km) : 0u);
            kappa_l = fmaxf(kappa_l, km);
        } else {
            gmax_put<DT>(sm, c, tid, warp * kVecPerWarp + lane < nvec ? f2o(cm) : 0u);
        }
        if (cm > m_l) {
            s_l = (do_sum && m_l > -INFINITY) ? s_l * ex2_approx((m_l - cm) * kLog2e) : 0.0f;
            m_l = cm;
        }
        if (do_sum && m_l > -INFINITY) {
            // even and odd elements summed apart, as packed fp32 pairs (one
            // multiply-add and one add per two elements, each lane's result
            // the scalar operation's)
            const float mb = m_l * kLog2e;
            const uint64_t l2 = f2_pack(kLog2e, kLog2e), nmb = f2_pack(-mb, -mb);
            uint64_t sab = 0ull;  // (even sum, odd sum)
#pragma unroll
            for (int j = 0; j < kVecPerLane; ++j) {
                float x[EPV];
                unpack16<DT>(u[j], x);
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const uint64_t z = f2_fma(f2_pack(x[e], x[e + 1]), l2, nmb);
                    sab = f2_add(sab, f2_pack(ex2_approx(f2_lo(z)), ex2_approx(f2_hi(z))));
                }
            }
            s_l += f2_lo(sab) + f2_hi(sab);
        }
    }
    // each warp's k largest lane maxima (0 bits: a lane without elements)
    const float lane_key = SAMP ? kappa_l : m_l;
    const uint32_t lo = warp_sort_desc_u32(lane_key > -INFINITY || (nch > 0 && warp * kVecPerWarp + lane < n / EPV)
                                               ? f2o(lane_key) : 0u);
    if (lane < kMaxTopK) sm.wtop[warp][lane] = lane < k ? lo : 0u;
    // the warp's (max, sum)
    float sw = do_sum ? s_l : 0.0f, mw = m_l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, mw, o);
        const float so = __shfl_xor_sync(0xffffffffu, sw, o);
        const float M = fmaxf(mw, mo);
        float sum = 0.0f;
        if (mw > -INFINITY) sum += sw * ex2_approx((mw - M) * kLog2e);
        if (mo > -INFINITY) sum += so * ex2_approx((mo - M) * kLog2e);
        mw = M;
        sw = sum;
    }
    if (lane == 0) {
        sm.wm[warp] = mw;
        sm.ws[warp] = sw;
    }
    consumer_bar();
    // tau: the k-th largest of the warps' lists (each zero-padded): entry t
    // ranks by the entries above it (larger, or equal and earlier)
    if (tid < kConsumerWarps * kMaxTopK) {
        const uint32_t v = (&sm.wtop[0][0])[tid];
        if (v != 0u) {
            const uint4* p = reinterpret_cast<const uint4*>(&sm.wtop[0][0]);
            int r = 0;
#pragma unroll
            for (int q = 0; q < kConsumerWarps * kMaxTopK / 4; ++q) {
                const uint4 a = p[q];
                r += (a.x > v || (a.x == v && 4 * q + 0 < tid)) + (a.y > v || (a.y == v && 4 * q + 1 < tid)) +
                     (a.z > v || (a.z == v && 4 * q + 2 < tid)) + (a.w > v || (a.w == v && 4 * q + 3 < tid));
            }
            if (r == k - 1) sm.tau = static_cast<unsigned long long>(v) << 32;
        }
    }
    consumer_bar();
    // a segment of at most ns chunks stays in the stages; the scratch then follows them
    const bool resident = nch <= ns;
    const int scratch_off = resident ? ns * kRowChunkBytes : 0;
    segment_topk<DT, SAMP>(sm, dyn_smem, resident, dyn_smem + scratch_off, smem_bytes - scratch_off, row_base, c0, n,
                           nch, k, id_base, grow, g);
}

// Merge of the CTAs of one row's cluster: every CTA pushes its top-k keys and
// (max, sum) into the leader's shared memory, then the leader (rank 0) ranks
// the keys into sm.top and combines (max, sum) into (sm.wm[0], sm.ws[0]).
// Returns true in the leader, after a block barrier.
__device__ __forceinline__ bool cluster_row_merge(ExpandSmem& sm, cg::cluster_group& cluster, int rank, int cpr, int k) {
    const int tid = threadIdx.x;
    ExpandSmem* leader = cluster.map_shared_rank(&sm, 0);
    if (tid < kMaxTopK) leader->rtop[rank * kMaxTopK + tid] = sm.ctop[tid];
    if (tid == 0) {
        float M = -INFINITY;
        for (int i = 0; i < kConsumerWarps; ++i) M = fmaxf(M, sm.wm[i]);
        float S = 0.0f;
        if (M > -INFINITY)
            for (int i = 0; i < kConsumerWarps; ++i)
                if (sm.wm[i] > -INFINITY) S += sm.ws[i] * ex2_approx((sm.wm[i] - M) * kLog2e);
        leader->rm[rank] = M;
        leader->rs[rank] = S;
    }
    cluster.sync();
    if (rank != 0) return false;
    if (tid < cpr * k) {
        const uint64_t key = sm.rtop[(tid / k) * kMaxTopK + tid % k];
        if (key != 0ull) {
            const int r = rank_in_lists(sm.rtop, cpr, key);
            if (r < k) sm.top[r] = key;
        }
    }
    if (tid == kRowThreads - 1) {
        float M = -INFINITY;
        for (int r = 0; r < cpr; ++r) M = fmaxf(M, sm.rm[r]);
        float S = 0.0f;
        if (M > -INFINITY)
            for (int r = 0; r < cpr; ++r)
                if (sm.rm[r] > -INFINITY) S += sm.rs[r] * ex2_approx((sm.rm[r] - M) * kLog2e);
        sm.wm[0] = M;
        sm.ws[0] = S;
    }
    __syncthreads();
    return true;
}

template <int DT, bool SAMP>
__global__ void __launch_bounds__(kRowThreads, SAMP ? 3 : 5) expand_kernel(TreeDims d, TreeWs w, int step, int seg, int ns,
                                                                 int smem_bytes, const void* __restrict__ logits,
                                                                 const float* __restrict__ lse_in,
                                                                 float* __restrict__ row_lse,
                                                                 int32_t* __restrict__ ftok_out,
                                                                 int32_t* __restrict__ fcount_out, int starve,
                                                                 GumbelRng grng) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ ExpandSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cpr = static_cast<int>(cluster.num_blocks());
    const int row = blockIdx.y;
    const int rps = step == 0 ? 1 : d.k;  // step 0 expands the root only: one row per sequence
    const int b = row / rps, f = row % rps;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int ES = DT == 1 ? 2 : 4;
    const int k = d.k;
    const int c0 = rank * seg;
    const int n = max(0, min(seg, d.V - c0));
    const int nch = min(max_seg_chunks<DT>(), (n * ES + kRowChunkBytes - 1) / kRowChunkBytes);  // the launcher keeps within
    const char* row_base = static_cast<const char*>(logits) + static_cast<size_t>(b * d.k + f) * d.V * ES;
    pdl_launch_dependents();
    // Before the dependency wait: the head of the segment into L2 (a hint; a
    // later write by the previous kernel still lands first), and every piece
    // of state that does not depend on the previous kernel.
    if (tid == kProducerWarp * 32) prefetch_l2_segment(row_base + static_cast<size_t>(c0) * ES, n * ES);
    if (tid == 0) {
        ring_init(sm.ring, ns);
        sm.tau = 0ull;
        sm.ngroups = 0;
        sm.nkeys = 0;
    }
    if (tid < kMaxTopK) {
        sm.ctop[tid] = 0ull;
        sm.top[tid] = 0ull;
    }
    __syncthreads();
    pdl_wait_prior();

    if (warp == kProducerWarp) {
        // The copies start before the frontier count is known: a row past the
        // count is streamed and dropped (all its copies land before the CTA
        // exits). (starve: the failure-path test hook, no copy is issued and
        // every ring wait gives up.)
        if (lane == 0 && nch > 0 && !starve) {
            ring_produce(sm.ring, dyn_smem, row_base + static_cast<size_t>(c0) * ES, n * ES, nch, ns, w.status);
        } else if (lane == 1) {
            // the frontier count and this row's parent, read while the row streams
            const int F = w.fcount[step * d.B + b];
            int parent = -1;
            float plogv = 0.0f;
            if (rank == 0 && f < F) {
                parent = w.fnode[(step * d.B + b) * d.k + f];
                if (parent >= 0 && EAGLE_CHECKED(parent < d.C, w.status))
                    plogv = w.cand_logv[static_cast<size_t>(b) * d.C + parent];
            }
            sm.F = F;
            sm.parent = parent;
            sm.plogv = plogv;
        }
        __syncwarp();
    } else {
        segment_consume<DT, SAMP>(sm, dyn_smem, smem_bytes, ns, row_base, c0, n, nch, k, lse_in == nullptr, 0, w.status,
                                  static_cast<uint32_t>(b * d.k + f), grng);
    }
    __syncthreads();
    const int F = sm.F;
    if (f >= F) {  // this frontier slot holds no node in this step (every CTA of the cluster leaves here)
        if (rank == 0 && tid == 0) {
            row_lse[(static_cast<size_t>(b) * d.D + step) * d.k + f] = __int_as_float(0x7fc00000);
            if (f == 0) {  // F == 0: nothing to expand, the next frontier is empty
                fcount_out[b] = 0;
                for (int j = 0; j < d.k; ++j) ftok_out[b * d.k + j] = -1;
            }
        }
        return;
    }
    __syncthreads();
    if (!cluster_row_merge(sm, cluster, rank, cpr, k)) return;

    // Children of this frontier node.
    const float lse = lse_in != nullptr ? lse_in[b * d.k + f] : sm.wm[0] + logf(sm.ws[0]);
    const int parent = sm.parent;
    const float plogv = sm.plogv;
    const int base = step == 0 ? 0 : d.k + (step - 1) * d.k * d.k;
    if (tid < d.k) {
        const uint64_t key = sm.top[tid];
        const int id = base + f * d.k + tid;
        const size_t at = static_cast<size_t>(b) * d.C + id;
        if (key != 0 && EAGLE_CHECKED(id < d.C && key_id(key) < static_cast<uint32_t>(d.V), w.status)) {
            // the child's logit (sampled drafting: the key holds the perturbed value)
            const float x = SAMP ? (DT == 1 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(
                                                                   row_base)[key_id(key)]) << 16)
                                            : reinterpret_cast<const float*>(row_base)[key_id(key)])
                                 : key_val(key);
            const float lp = __fsub_rn(x, lse);
            w.cand_token[at] = static_cast<int32_t>(key_id(key));
            w.cand_parent[at] = parent;
            w.cand_depth[at] = step + 1;
            w.cand_logv[at] = __fadd_rn(plogv, lp);
            w.cand_lp[at] = lp;
            w.cand_valid[at] = 1;
        }
    }
    if (tid == 0) {
        row_lse[(static_cast<size_t>(b) * d.D + step) * d.k + f] = lse;
        if (!isfinite(lse)) raise_status(w.status, kDevNonFinite);
    }
    if (step == 0 && tid > 0 && tid < d.k)  // rows 1.. of step 0 are not read (not launched)
        row_lse[static_cast<size_t>(b) * d.D * d.k + tid] = __int_as_float(0x7fc00000);
    __syncthreads();

    // Per-sequence ticket: the last row of this sequence picks the next frontier.
    if (tid == 0) {
        const int prev = ticket_add(&w.expand_ticket[b]);
        sm.last = (prev == F - 1);
    }
    __syncthreads();
    if (!sm.last) return;
    const int nsel = F * d.k;
    // the ring is idle now: candidate keys (zero-padded to a multiple of 8),
    // their tokens, the chosen tokens
    uint64_t* sel = reinterpret_cast<uint64_t*>(dyn_smem);
    int32_t* sel_tok = reinterpret_cast<int32_t*>(dyn_smem + kMaxTopK * kMaxTopK * sizeof(uint64_t));
    int32_t* top_tok = sel_tok + kMaxTopK * kMaxTopK;
    for (int i = tid; i < nsel; i += kRowThreads) {
        const int id = base + i;
        const size_t at = static_cast<size_t>(b) * d.C + id;
        const bool valid = __ldcg(reinterpret_cast<const unsigned char*>(&w.cand_valid[at])) != 0;
        const float lv = __ldcg(&w.cand_logv[at]);
        // ranked by value (EAGLE-2), by the child's own confidence (policy 1),
        // or by position f + r within the step (static shape, policy 3)
        const float rank_by = d.policy == 1   ? __ldcg(&w.cand_lp[at])
                              : d.policy == 3 ? -static_cast<float>(i / d.k + i % d.k)
                                              : lv;
        sel_tok[i] = __ldcg(&w.cand_token[at]);
        sel[i] = (valid && lv >= d.log_thr) ? make_key(rank_by, static_cast<uint32_t>(id)) : 0ull;
    }
    if (tid >= nsel && tid < (nsel + 7) / 8 * 8) sel[tid] = 0ull;  // padding
    if (tid < kMaxTopK) sm.top[tid] = 0ull;
    __syncthreads();
    for (int i = tid; i < nsel; i += kRowThreads) {
        const uint64_t key = sel[i];
        if (key == 0ull) continue;
        const int r = rank_in_list(sel, nsel, key);
        if (r < d.k) {
            sm.top[r] = key;
            top_tok[r] = sel_tok[i];
        }
    }
    __syncthreads();
    if (tid < d.k) {
        const uint64_t key = sm.top[tid];
        const int id = key ? static_cast<int>(key_id(key)) : -1;
        w.fnode[((step + 1) * d.B + b) * d.k + tid] = id;
        ftok_out[b * d.k + tid] = id >= 0 ? top_tok[tid] : -1;
    }
    if (tid == 0) {
        int cnt = 0;
        for (int j = 0; j < d.k; ++j) cnt += sm.top[j] != 0ull;
        w.fcount[(step + 1) * d.B + b] = cnt;
        fcount_out[b] = cnt;
        w.expand_ticket[b] = 0;
    }
}

// ------------------------------------------------------------ verify kernel ---

struct VerifySmem {
    RowRing ring;
    int tok[kMaxSlots];
    int par[kMaxSlots];
    // lossless: this row's children (slot, token logit in this row), read while the row streams
    int kid_c[kMaxTopK];
    float kid_x[kMaxTopK];
    int kid_n;
    uint64_t wkey[kConsumerWarps];
    uint64_t rkey[kMaxChunks];  // every rank's segment maximum (pushed to the leader)
    int last;
};

// Greedy-walk state of the last-arriving CTA of a sequence; it lives in the
// (then idle) dynamic shared memory of the chunk ring.
struct WalkSmem {
    int arg[kMaxSlots];
    int path[kMaxDepth + 1];
    int child[kMaxTopK];
    int a, bonus, bad;
};

// Stage 6 over the target rows: every row's maximum and argmax (lowest id
// among equal values). MODE 0 (greedy): the last row of a sequence to finish
// walks its tree. MODE 1 (lossless): the statistics only, the walk is
// verify_lossless_walk_kernel.
template <int DT, int MODE>
__global__ void __launch_bounds__(kRowThreads) verify_kernel(TreeDims d, TreeWs w, float inv_t, int seg, int ns,
                                                              const void* __restrict__ target,
                                                              const int32_t* __restrict__ tokens,
                                                              const int32_t* __restrict__ parent,
                                                              const int32_t* __restrict__ n_tree,
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
    constexpr int CE = kRowChunkBytes / ES;
    pdl_launch_dependents();
    if (tid == kProducerWarp * 32) {  // the segment's head into L2 while the previous kernel finishes
        const int cp = rank * seg;
        const int np = max(0, min(seg, d.V - cp));
        prefetch_l2_segment(static_cast<const char*>(target) + (static_cast<size_t>(row) * d.V + cp) * ES, np * ES);
    }
    pdl_wait_prior();
    const int n = n_tree[b];
    if (n < 1 || n > d.T) {
        if (rank == 0 && t == 0 && tid == 0) raise_status(w.status, kDevBadIndex);
        return;
    }
    if (t >= n) return;

    const int c0 = rank * seg;
    const int len = max(0, min(seg, d.V - c0));
    const int nch = (len * ES + kRowChunkBytes - 1) / kRowChunkBytes;
    const char* row_base = static_cast<const char*>(target) + static_cast<size_t>(b * d.T + t) * d.V * ES;
    if (tid == 0) {
        ring_init(sm.ring, ns);
        sm.kid_n = 0;
    }
    __syncthreads();

    bool failed = false;
    if (warp == kProducerWarp) {
        if (lane == 0 && nch > 0) {
            ring_produce(sm.ring, dyn_smem, row_base + static_cast<size_t>(c0) * ES, len * ES, nch, ns, w.status);
        } else if (MODE == 1 && rank == 0 && lane > 0) {
            // lossless: the token logits of this row's children, read while the
            // row streams (their masses need the row maximum, known at the end)
            for (int c = t + lane; c < n; c += 31) {
                if (parent[static_cast<size_t>(b) * d.T + c] != t) continue;
                const int tk = tokens[static_cast<size_t>(b) * d.T + c];
                if (tk < 0 || tk >= d.V) continue;  // the walk flags it
                const int at = atomicAdd(&sm.kid_n, 1);
                if (at >= kMaxTopK) continue;
                sm.kid_c[at] = c;
                sm.kid_x[at] = DT == 1 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(
                                                             row_base)[tk]) << 16)
                                       : reinterpret_cast<const float*>(row_base)[tk];
            }
        }
        __syncwarp();
    } else {
        // ---- pass 1: maximum, lowest id among equal values ----
        float lm = -INFINITY;
        int larg = -1;
        for (int c = 0; c < nch; ++c) {
            if (!ring_wait(sm.ring, c, ns, failed, w.status)) {
                ring_release(sm.ring, c, ns);
                continue;
            }
            const int nvec = min(CE, len - c * CE) / EPV;
            uint4 u[kVecPerLane];
            load_lane<DT>(dyn_smem + (c % ns) * kRowChunkBytes, nvec, warp, lane, u);
            ring_release(sm.ring, c, ns);
            if (larg >= 0 && !(lane_max4<DT>(u) > lm)) continue;  // nothing above the lane maximum
#pragma unroll
            for (int j = 0; j < kVecPerLane; ++j) {
                const int v = warp * kVecPerWarp + j * 32 + lane;
                if (v >= nvec) continue;
                const float m8 = vec_max<DT>(u[j]);
                if (larg < 0 || m8 > lm) {  // first element equal to the vector maximum: lowest id
                    float x[EPV];
                    unpack16<DT>(u[j], x);
                    int e0 = 0;
#pragma unroll
                    for (int e = EPV - 1; e >= 0; --e)
                        if (x[e] == m8) e0 = e;
                    lm = m8;
                    larg = c0 + c * CE + v * EPV + e0;
                }
            }
        }
        uint64_t key = larg < 0 ? 0ull : make_key(lm, static_cast<uint32_t>(larg));
        key = warp_max_u64(key);
        if (lane == 0) sm.wkey[warp] = key;
    }
    __syncthreads();
    if (warp == 0) {
        uint64_t m = lane < kConsumerWarps ? sm.wkey[lane] : 0ull;
        m = warp_max_u64(m);
        if (lane == 0) cluster.map_shared_rank(&sm, 0)->rkey[rank] = m;
    }
    cluster.sync();
    if (rank != 0) return;
    uint64_t gkey = 0;
    for (int r = 0; r < cpr; ++r) gkey = sm.rkey[r] > gkey ? sm.rkey[r] : gkey;
    const float M = key_val(gkey);
    const size_t rt = static_cast<size_t>(b) * d.T + t;
    if (MODE == 1 && tid < min(sm.kid_n, kMaxTopK))  // the children's masses in this row
        w.pmass[static_cast<size_t>(b) * d.T + sm.kid_c[tid]] = fixed_mass(sm.kid_x[tid], M, inv_t);
    if (tid == 0) {
        w.row_max[rt] = M;
        w.row_arg[rt] = static_cast<int32_t>(key_id(gkey));
        w.row_mass[rt] = 0;  // lossless: written by the walk for the rows it visits
        if (!isfinite(M)) raise_status(w.status, kDevNonFinite);
        if (MODE == 0) {
            const int prev = ticket_add(&w.verify_ticket[b]);
            sm.last = (prev == n - 1);
        }
    }
    // lossless: the walk is its own kernel (verify_lossless_walk_kernel)
    if (MODE == 1) return;
    __syncthreads();
    if (!sm.last) return;

    // ---- greedy acceptance walk for sequence b (one CTA) ----
    WalkSmem& ws = *reinterpret_cast<WalkSmem*>(dyn_smem);
    const int T = d.T;
    if (tid == 0) ws.bad = 0;
    for (int c = tid; c < n; c += kRowThreads) {
        sm.tok[c] = tokens[static_cast<size_t>(b) * T + c];
        sm.par[c] = parent[static_cast<size_t>(b) * T + c];
        ws.arg[c] = __ldcg(&w.row_arg[static_cast<size_t>(b) * T + c]);
    }
    __syncthreads();
    for (int c = 1 + tid; c < n; c += kRowThreads) {
        const int tk = sm.tok[c], p = sm.par[c];
        if (tk < 0 || tk >= d.V || p < 0 || p >= c) ws.bad = 1;
    }
    __syncthreads();
    const bool bad = ws.bad != 0;
    if (tid == 0 && bad) raise_status(w.status, kDevBadIndex);

    if (warp == 0) {
        // One warp walks the tree; at each node its children (contiguous in
        // slot order) are tested together, lane j on child j.
        int cur = 0, a = 0;
        if (lane == 0) ws.path[0] = 0;
        while (a < d.D && !bad) {
            int nchild = 0;
            for (int c0w = cur + 1; c0w < n; c0w += 32) {
                const int c = c0w + lane;
                const bool is = c < n && sm.par[c] == cur;
                const unsigned bal = __ballot_sync(0xffffffffu, is);
                if (is) {
                    const int pos = nchild + __popc(bal & lanemask_lt());
                    if (pos < kMaxTopK) ws.child[pos] = c;
                }
                nchild += __popc(bal);
            }
            __syncwarp();
            nchild = min(nchild, kMaxTopK);
            if (nchild == 0) break;
            const int c = lane < nchild ? ws.child[lane] : -1;
            int next = -1;
            const unsigned bal = __ballot_sync(0xffffffffu, c >= 0 && sm.tok[c] == ws.arg[cur]);
            if (bal) next = ws.child[__ffs(bal) - 1];
            if (next < 0) break;
            ++a;
            if (lane == 0) ws.path[a] = next;
            cur = next;
        }
        __syncwarp();
        if (lane == 0) {
            ws.a = a;
            ws.bonus = ws.arg[cur];
        }
    }
    __syncthreads();

    if (tid == 0) {
        const int a = ws.a;
        const int Dp1 = d.D + 1;
        accept_len[b] = a;
        for (int j = 0; j < Dp1; ++j) {
            slots_out[b * Dp1 + j] = j <= a ? ws.path[j] : -1;
            tokens_out[b * Dp1 + j] = j < a ? sm.tok[ws.path[j + 1]] : (j == a ? ws.bonus : -1);
        }
        if (ws.bonus < 0) raise_status(w.status, kDevBadIndex);
        w.verify_ticket[b] = 0;
    }
}

// ------------------------------------------------------ vocabulary shards ---
//
// When the LM head is split over GPUs by vocabulary rows, each GPU holds a
// slice [offset, offset + Vs) of every logit row. Stage 1 and the greedy
// verify then run per slice into small partials, the partials of all slices
// meet in one exchange (k keys and two floats per row), and a merge gives the
// results of the whole row ["EAGLE" notes, EAGLE 方法: TopK over the
// vocabulary; the split itself is not on the pages]. Partials: (max, sum of
// exp(x - max)) in fp32 and the slice's top-k keys (value desc, then lower
// token id, ids of the whole vocabulary); the top-1 key is the slice's argmax.

// Stage-1 partials of one vocabulary slice: grid (cpr, rows), a cluster per row.
template <int DT>
__global__ void __launch_bounds__(kRowThreads, 5) shard_partial_kernel(int Vs, int k, int seg, int ns, int smem_bytes,
                                                                        const void* __restrict__ logits, int id_base,
                                                                        float2* __restrict__ part_ms,
                                                                        uint64_t* __restrict__ part_keys,
                                                                        int* status) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ ExpandSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cpr = static_cast<int>(cluster.num_blocks());
    const int row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int ES = DT == 1 ? 2 : 4;
    const int c0 = rank * seg;
    const int n = max(0, min(seg, Vs - c0));
    const int nch = min(max_seg_chunks<DT>(), (n * ES + kRowChunkBytes - 1) / kRowChunkBytes);
    const char* row_base = static_cast<const char*>(logits) + static_cast<size_t>(row) * Vs * ES;
    pdl_launch_dependents();
    if (tid == kProducerWarp * 32) prefetch_l2_segment(row_base + static_cast<size_t>(c0) * ES, n * ES);
    if (tid == 0) {
        ring_init(sm.ring, ns);
        sm.tau = 0ull;
        sm.ngroups = 0;
        sm.nkeys = 0;
    }
    if (tid < kMaxTopK) {
        sm.ctop[tid] = 0ull;
        sm.top[tid] = 0ull;
    }
    __syncthreads();
    pdl_wait_prior();
    if (warp == kProducerWarp) {
        if (lane == 0 && nch > 0)
            ring_produce(sm.ring, dyn_smem, row_base + static_cast<size_t>(c0) * ES, n * ES, nch, ns, status);
        __syncwarp();
    } else {
        segment_consume<DT, false>(sm, dyn_smem, smem_bytes, ns, row_base, c0, n, nch, k, true, id_base, status, 0u,
                                   GumbelRng{});
    }
    __syncthreads();
    if (!cluster_row_merge(sm, cluster, rank, cpr, k)) return;
    if (tid < kMaxTopK) part_keys[static_cast<size_t>(row) * kMaxTopK + tid] = tid < k ? sm.top[tid] : 0ull;
    if (tid == 0) part_ms[row] = make_float2(sm.wm[0], sm.ws[0]);
}

// Merge of S slices' partials, one warp per row: lse = M + log(sum S_s
// 2^((M_s - M) log2 e)), M = max M_s; the top-k of the union of the slices'
// top-k (rank among them); the argmax = the largest key.
constexpr int kMaxShards = 16;
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeWarps * 32) shard_merge_kernel(int S, int rows, int k,
                                                                       const float2* __restrict__ part_ms,
                                                                       const uint64_t* __restrict__ part_keys,
                                                                       float* __restrict__ lse_out,
                                                                       int32_t* __restrict__ topk_id,
                                                                       float* __restrict__ topk_val,
                                                                       int32_t* __restrict__ argmax_out, int* status) {
    __shared__ alignas(16) uint64_t keys[kMergeWarps][kMaxShards * kMaxTopK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kMergeWarps + warp;
    pdl_launch_dependents();
    pdl_wait_prior();
    if (row >= rows) return;
    uint64_t* kl = keys[warp];
    for (int i = lane; i < S * kMaxTopK; i += 32)
        kl[i] = part_keys[(static_cast<size_t>(i / kMaxTopK) * rows + row) * kMaxTopK + i % kMaxTopK];
    float m = -INFINITY, s = 0.0f;
    if (lane < S) {
        const float2 ms = part_ms[static_cast<size_t>(lane) * rows + row];
        m = ms.x;
        s = ms.y;
    }
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float t = (lane < S && m > -INFINITY) ? s * ex2_approx((m - M) * kLog2e) : 0.0f;
    // the slices' terms in slice order (one fixed order: lane 0 first)
    float sum = 0.0f;
    for (int i = 0; i < S; ++i) sum += __shfl_sync(0xffffffffu, t, i);
    __syncwarp();
    for (int i = lane; i < S * kMaxTopK; i += 32) {
        const uint64_t key = kl[i];
        if (key == 0ull || i % kMaxTopK >= k) continue;
        int r = 0;
        for (int j = 0; j < S * kMaxTopK; ++j) r += (j % kMaxTopK < k) && kl[j] > key;
        if (r < k) {
            topk_id[static_cast<size_t>(row) * k + r] = static_cast<int32_t>(key_id(key));
            topk_val[static_cast<size_t>(row) * k + r] = key_val(key);
        }
        if (r == 0) argmax_out[row] = static_cast<int32_t>(key_id(key));
    }
    // ranks past the union's key count: none
    int have = 0;
    for (int j = lane; j < S * kMaxTopK; j += 32) have += (j % kMaxTopK < k) && kl[j] != 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) have += __shfl_xor_sync(0xffffffffu, have, o);
    if (lane >= have && lane < k) {
        topk_id[static_cast<size_t>(row) * k + lane] = -1;
        topk_val[static_cast<size_t>(row) * k + lane] = -INFINITY;
    }
    if (lane == 0) {
        const float lse = M + logf(sum);
        lse_out[row] = lse;
        if (!isfinite(lse)) raise_status(status, kDevNonFinite);
        if (have == 0) argmax_out[row] = -1;
    }
}

// Stage 2 from merged top-k, one CTA per sequence: the children of the F
// frontier rows of step `step` (row f's top-k ids and logits, its lse) and
// the next frontier, exactly as the expansion's last CTA does.
__global__ void __launch_bounds__(kRowThreads) expand_topk_kernel(TreeDims d, TreeWs w, int step,
                                                                  const int32_t* __restrict__ topk_id,
                                                                  const float* __restrict__ topk_val,
                                                                  const float* __restrict__ lse_in,
                                                                  float* __restrict__ row_lse,
                                                                  int32_t* __restrict__ ftok_out,
                                                                  int32_t* __restrict__ fcount_out) {
    __shared__ alignas(16) uint64_t sel[kMaxTopK * kMaxTopK];
    __shared__ int32_t sel_tok[kMaxTopK * kMaxTopK];
    __shared__ uint64_t top[kMaxTopK];
    __shared__ int32_t top_tok[kMaxTopK];
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int F = w.fcount[step * d.B + b];
    const int base = step == 0 ? 0 : d.k + (step - 1) * d.k * d.k;
    const int nsel = F * d.k;
    for (int i = tid; i < d.k; i += kRowThreads)
        row_lse[(static_cast<size_t>(b) * d.D + step) * d.k + i] =
            i < F ? lse_in[b * d.k + i] : __int_as_float(0x7fc00000);
    for (int i = tid; i < nsel; i += kRowThreads) {
        const int fr = i / d.k, r = i % d.k;
        const size_t src = (static_cast<size_t>(b) * d.k + fr) * d.k + r;
        const int tok = topk_id[src];
        uint64_t sk = 0ull;
        const int parent = w.fnode[(step * d.B + b) * d.k + fr];
        if (tok >= 0 && tok < d.V && EAGLE_CHECKED(parent < d.C && base + i < d.C, w.status)) {
            const float plogv = parent < 0 ? 0.0f : __ldcg(&w.cand_logv[static_cast<size_t>(b) * d.C + parent]);
            const float lse = lse_in[b * d.k + fr];
            const float lp = __fsub_rn(topk_val[src], lse);
            const float lv = __fadd_rn(plogv, lp);
            const int id = base + i;
            const size_t at = static_cast<size_t>(b) * d.C + id;
            w.cand_token[at] = tok;
            w.cand_parent[at] = parent;
            w.cand_depth[at] = step + 1;
            w.cand_logv[at] = lv;
            w.cand_lp[at] = lp;
            w.cand_valid[at] = 1;
            if (!isfinite(lse)) raise_status(w.status, kDevNonFinite);
            const float rank_by = d.policy == 1 ? lp : d.policy == 3 ? -static_cast<float>(fr + r) : lv;
            if (lv >= d.log_thr) sk = make_key(rank_by, static_cast<uint32_t>(id));
        } else if (tok >= d.V) {
            raise_status(w.status, kDevBadIndex);
        }
        sel[i] = sk;
        sel_tok[i] = tok;
    }
    if (tid >= nsel && tid < (nsel + 7) / 8 * 8) sel[tid] = 0ull;
    if (tid < kMaxTopK) top[tid] = 0ull;
    __syncthreads();
    for (int i = tid; i < nsel; i += kRowThreads) {
        const uint64_t key = sel[i];
        if (key == 0ull) continue;
        const int r = rank_in_list(sel, nsel, key);
        if (r < d.k) {
            top[r] = key;
            top_tok[r] = sel_tok[i];
        }
    }
    __syncthreads();
    if (tid < d.k) {
        const uint64_t key = top[tid];
        const int id = key ? static_cast<int>(key_id(key)) : -1;
        w.fnode[((step + 1) * d.B + b) * d.k + tid] = id;
        ftok_out[b * d.k + tid] = id >= 0 ? top_tok[tid] : -1;
    }
    if (tid == 0) {
        int cnt = 0;
        for (int j = 0; j < d.k; ++j) cnt += top[j] != 0ull;
        w.fcount[(step + 1) * d.B + b] = cnt;
        fcount_out[b] = cnt;
    }
}

// Greedy verification from the target's argmax of every slot (merged over the
// vocabulary slices), one warp per sequence: the walk of verify_kernel.
__global__ void __launch_bounds__(32) verify_argmax_kernel(TreeDims d, TreeWs w, const int32_t* __restrict__ row_argmax,
                                                          const int32_t* __restrict__ tokens,
                                                          const int32_t* __restrict__ parent,
                                                          const int32_t* __restrict__ n_tree,
                                                          int32_t* __restrict__ accept_len,
                                                          int32_t* __restrict__ slots_out,
                                                          int32_t* __restrict__ tokens_out) {
    __shared__ int par[kMaxSlots], tok[kMaxSlots], path[kMaxDepth + 1];
    const int b = blockIdx.x, lane = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait_prior();
    const int n = n_tree[b];
    const int T = d.T;
    if (n < 1 || n > T) {
        if (lane == 0) raise_status(w.status, kDevBadIndex);
        return;
    }
    bool bad = false;
    for (int c = lane; c < n; c += 32) {
        par[c] = parent[static_cast<size_t>(b) * T + c];
        tok[c] = tokens[static_cast<size_t>(b) * T + c];
        if (c > 0 && (par[c] < 0 || par[c] >= c || tok[c] < 0 || tok[c] >= d.V)) bad = true;
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    int cur = 0, a = 0;
    path[0] = 0;
    while (a < d.D && !bad) {
        const int want = row_argmax[static_cast<size_t>(b) * T + cur];
        int next = -1;
        for (int c0 = cur + 1; c0 < n && next < 0; c0 += 32) {
            const int c = c0 + lane;
            const unsigned bal = __ballot_sync(0xffffffffu, c < n && par[c] == cur && tok[c] == want);
            if (bal) next = c0 + __ffs(bal) - 1;
        }
        if (next < 0) break;
        ++a;
        if (lane == 0) path[a] = next;
        cur = next;
    }
    __syncwarp();
    if (lane == 0) {
        const int bonus = bad ? -1 : row_argmax[static_cast<size_t>(b) * T + cur];
        if (bad || bonus < 0 || bonus >= d.V) raise_status(w.status, kDevBadIndex);
        const int Dp1 = d.D + 1;
        accept_len[b] = a;
        for (int j = 0; j < Dp1; ++j) {
            slots_out[b * Dp1 + j] = j <= a ? path[j] : -1;
            tokens_out[b * Dp1 + j] = j < a ? tok[path[j + 1]] : (j == a ? bonus : -1);
        }
    }
}

// Inspection: the device's Gumbel noise of words and fixed-order logarithm of
// values, element by element (checked bit for bit against the oracle's).
__global__ void sampling_probe_kernel(const uint32_t* __restrict__ words, const float* __restrict__ ys, int n,
                                      float* __restrict__ gumbel_out, float* __restrict__ log_out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    if (words != nullptr) gumbel_out[i] = sampling::gumbel_of_word(words[i]);
    if (ys != nullptr) log_out[i] = sampling::fixed_log(ys[i]);
}

// -------------------------------------------------------------- launchers ---

static int sm_count() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev] = n;
    return n;
}

RowPlan plan_rows(int V, int esize, long rows, int max_stages, int max_seg_chunks) {
    // about two waves of CTAs (three to five resident per SM)
    const long target = 2L * 3 * sm_count();
    int cpr = 1;
    while (cpr < kMaxChunks &&
           (rows * cpr < target || row_chunks(row_seg_elems(V, esize, cpr), esize) > max_seg_chunks))
        cpr *= 2;
    RowPlan p;
    p.cpr = cpr;
    p.seg = row_seg_elems(V, esize, cpr);
    p.nch = row_chunks(p.seg, esize);
    p.stages = std::min(p.nch, max_stages);
    p.smem = p.nch <= 1 ? static_cast<int>(align_up(static_cast<size_t>(p.seg) * esize, 128))
                        : p.stages * kRowChunkBytes;
    return p;
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
                          float* row_lse, int32_t* ftok, int32_t* fcount_out, cudaStream_t stream, bool starve_ring,
                          const uint64_t* sample_seed_cycle) {
    const int esize = d.dtype == 1 ? 2 : 4;
    const long rows = static_cast<long>(d.B) * (step == 0 ? 1 : d.k);  // step 0 reads the root rows only
    const int max_seg = esize == 2 ? kMaxSegChunksBf16 : kMaxSegChunks;
    RowPlan p = plan_rows(d.V, esize, rows, kExpandStages, kMaxSegChunks);
    // Rows enough to fill every CTA slot once (three to five per SM, five
    // resident): one CTA per row in a single wave, no cluster merge, instead
    // of about two waves of half rows whose per-CTA tails leave HBM idle.
    if (p.cpr > 1 && rows >= 3L * sm_count() && rows <= 5L * sm_count()) {
        const int seg1 = row_seg_elems(d.V, esize, 1);
        const int nch1 = row_chunks(seg1, esize);
        if (nch1 <= max_seg) {
            p.cpr = 1;
            p.seg = seg1;
            p.nch = nch1;
            p.stages = std::min(nch1, kExpandStages);
            p.smem = nch1 <= 1 ? static_cast<int>(align_up(static_cast<size_t>(seg1) * esize, 128))
                               : p.stages * kRowChunkBytes;
        }
    }
    // With enough rows to fill the SMs at four CTAs per row, four larger
    // resident segments beat eight small ones (fewer tails and cluster
    // members per row; 70B b8: 14.4 -> 13.0 us per step). Few rows keep eight.
    if (p.cpr > 4 && rows * 4 >= sm_count()) {
        const int seg4 = row_seg_elems(d.V, esize, 4);
        const int nch4 = row_chunks(seg4, esize);
        if (nch4 <= kRowStages) {
            p.cpr = 4;
            p.seg = seg4;
            p.nch = nch4;
            p.stages = nch4;
            p.smem = nch4 * kRowChunkBytes;
        }
    }
    if (p.nch > max_seg) return cudaErrorInvalidValue;
    dim3 grid(p.cpr, step == 0 ? d.B : d.B * d.k, 1);  // step 0: the root row of each sequence
    TreeDims dd = d;
    TreeWs ww = ws;
    // after the pass the stage memory holds the candidate groups and keys of
    // the segment's top-k and, in the last CTA of a sequence, the frontier
    // candidates (keys and tokens)
    const int scratch = p.nch * kConsumers * 4 + 512 * 8;  // candidate groups + keys
    const int pick = kMaxTopK * kMaxTopK * (8 + 4) + kMaxTopK * 4 + 16;
    const int smem = std::max(pick, p.nch <= p.stages ? p.stages * kRowChunkBytes + scratch : std::max(p.smem, scratch));
    int seg = p.seg, ns = p.stages, smem_bytes = smem, starve = starve_ring ? 1 : 0;
    GumbelRng grng{};
    if (sample_seed_cycle != nullptr) {
        const uint64_t seed = sample_seed_cycle[0], cycle = sample_seed_cycle[1];
        grng = GumbelRng{static_cast<uint32_t>(seed) ^ 10u, static_cast<uint32_t>(seed >> 32),
                         static_cast<uint32_t>(step), static_cast<uint32_t>(cycle)};
    }
    void* args[] = {&dd,
                    &ww,
                    &step,
                    &seg,
                    &ns,
                    &smem_bytes,
                    const_cast<void**>(&logits),
                    const_cast<float**>(&lse_in),
                    &row_lse,
                    &ftok,
                    &fcount_out,
                    &starve,
                    &grng};
    if (sample_seed_cycle != nullptr)
        return d.dtype == 1 ? launch_rows(expand_kernel<1, true>, grid, p.cpr, smem, stream, args)
                            : launch_rows(expand_kernel<0, true>, grid, p.cpr, smem, stream, args);
    return d.dtype == 1 ? launch_rows(expand_kernel<1, false>, grid, p.cpr, smem, stream, args)
                        : launch_rows(expand_kernel<0, false>, grid, p.cpr, smem, stream, args);
}

cudaError_t launch_verify(const TreeDims& d, const TreeWs& ws, int mode, float inv_temp, const void* target,
                          const int32_t* tokens, const int32_t* parent, const int32_t* n_tree, VerifyRng rng,
                          int32_t* accept_len, int32_t* slots, int32_t* out_tokens, cudaStream_t stream) {
    const int esize = d.dtype == 1 ? 2 : 4;
    const long rows = static_cast<long>(d.B) * d.T;
    RowPlan p = plan_rows(d.V, esize, rows, kRowStages, 1 << 20);
    // Rows enough to fill three to five CTA slots per SM: one CTA per row in
    // a single wave (no cluster merge, no second wave of tails), as expansion;
    // a three-stage ring keeps four CTAs resident per SM.
    if (p.cpr > 1 && rows >= 3L * sm_count() && rows <= 5L * sm_count()) {
        p.cpr = 1;
        p.seg = row_seg_elems(d.V, esize, 1);
        p.nch = row_chunks(p.seg, esize);
        p.stages = std::min(p.nch, 3);
        p.smem = p.nch <= 1 ? static_cast<int>(align_up(static_cast<size_t>(p.seg) * esize, 128))
                            : p.stages * kRowChunkBytes;
    }
    dim3 grid(p.cpr, d.B * d.T, 1);
    // the greedy walk keeps its state in the (then idle) stage memory
    const int smem = static_cast<int>(std::max<size_t>(p.smem, align_up(sizeof(WalkSmem), 128)));
    TreeDims dd = d;
    TreeWs ww = ws;
    int seg = p.seg, ns = p.stages;
    void* args[] = {&dd,
                    &ww,
                    &inv_temp,
                    &seg,
                    &ns,
                    const_cast<void**>(&target),
                    const_cast<int32_t**>(&tokens),
                    const_cast<int32_t**>(&parent),
                    const_cast<int32_t**>(&n_tree),
                    &accept_len,
                    &slots,
                    &out_tokens};
    cudaError_t e;
    if (d.dtype == 1)
        e = mode == 1 ? launch_rows(verify_kernel<1, 1>, grid, p.cpr, smem, stream, args)
                      : launch_rows(verify_kernel<1, 0>, grid, p.cpr, smem, stream, args);
    else
        e = mode == 1 ? launch_rows(verify_kernel<0, 1>, grid, p.cpr, smem, stream, args)
                      : launch_rows(verify_kernel<0, 0>, grid, p.cpr, smem, stream, args);
    if (e != cudaSuccess || mode != 1) return e;
    // lossless: one cluster per sequence walks the tree, summing only the rows it visits
    return launch_verify_walk(d, ws, inv_temp, rng, target, tokens, parent, n_tree, accept_len, slots, out_tokens,
                              stream);
}

cudaError_t launch_shard_partials(int Vs, int k, int rows, int dtype, const void* logits, int id_base, float2* part_ms,
                                  uint64_t* part_keys, int* status, cudaStream_t stream) {
    const int esize = dtype == 1 ? 2 : 4;
    const int max_seg = esize == 2 ? kMaxSegChunksBf16 : kMaxSegChunks;
    const RowPlan p = plan_rows(Vs, esize, rows, kExpandStages, kMaxSegChunks);
    if (p.nch > max_seg) return cudaErrorInvalidValue;
    const int scratch = p.nch * kConsumers * 4 + 512 * 8;
    const int smem = p.nch <= p.stages ? p.stages * kRowChunkBytes + scratch : std::max(p.smem, scratch);
    dim3 grid(p.cpr, rows, 1);
    int seg = p.seg, ns = p.stages, smem_bytes = smem;
    void* args[] = {&Vs, &k, &seg, &ns, &smem_bytes, const_cast<void**>(&logits), &id_base, &part_ms, &part_keys,
                    &status};
    return dtype == 1 ? launch_rows(shard_partial_kernel<1>, grid, p.cpr, smem, stream, args)
                      : launch_rows(shard_partial_kernel<0>, grid, p.cpr, smem, stream, args);
}

cudaError_t launch_shard_merge(int S, int rows, int k, const float2* part_ms, const uint64_t* part_keys, float* lse,
                               int32_t* topk_id, float* topk_val, int32_t* argmax, int* status, cudaStream_t stream) {
    const int blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    return launch_pdl(shard_merge_kernel, dim3(blocks), dim3(kMergeWarps * 32), 0, stream, S, rows, k, part_ms,
                      part_keys, lse, topk_id, topk_val, argmax, status);
}

cudaError_t launch_expand_topk(const TreeDims& d, const TreeWs& ws, int step, const int32_t* topk_id,
                               const float* topk_val, const float* lse_in, float* row_lse, int32_t* ftok,
                               int32_t* fcount_out, cudaStream_t stream) {
    return launch_pdl(expand_topk_kernel, dim3(d.B), dim3(kRowThreads), 0, stream, d, ws, step, topk_id, topk_val,
                      lse_in, row_lse, ftok, fcount_out);
}

cudaError_t launch_verify_argmax(const TreeDims& d, const TreeWs& ws, const int32_t* row_argmax, const int32_t* tokens,
                                 const int32_t* parent, const int32_t* n_tree, int32_t* accept_len, int32_t* slots,
                                 int32_t* out_tokens, cudaStream_t stream) {
    return launch_pdl(verify_argmax_kernel, dim3(d.B), dim3(32), 0, stream, d, ws, row_argmax, tokens, parent, n_tree,
                      accept_len, slots, out_tokens);
}

cudaError_t launch_sampling_probe(const uint32_t* words, const float* ys, int n, float* gumbel_out, float* log_out,
                                  cudaStream_t stream) {
    count_launch();
    sampling_probe_kernel<<<(n + 255) / 256, 256, 0, stream>>>(words, ys, n, gumbel_out, log_out);
    return cudaGetLastError();
}

}  // namespace eagle

// Stage 6 walks that run on one cluster of CTAs per sequence, sm_103a: the
// draft-probability rule (sampled drafting) and the lossless rule with
// deterministic candidates (further down).
//
// "EAGLE-2: Faster Inference ..." summary, 2.1 Speculative Sampling: the
// target accepts the draft's tokens one after another with probability
// min(1, p/q), and on a rejection continues from the residual distribution.
// Here the children of a node were drawn from the draft distribution q of the
// node's draft row without replacement (eagle_expand_sampled) and are tested
// in drawing (slot) order: child x is accepted iff U24 Q[x] SA < 2^24 A[x] SQ,
// with A the target residual and Q the remaining draft masses (integer masses
// floor(dexp((x - max) / T) 2^40) of the rows), SA, SQ their sums. A rejection
// replaces A by r(y) = max(0, A[y] SQ - Q[y] SA) scaled down by the smallest
// shift that brings max r to 2^40 or below (A kept when every r is 0), then
// removes x from Q. With no child accepted the bonus token is the smallest y
// whose running sum of A exceeds floor(U64 SA / 2^64).
//
// Layout of the work: one cluster of kDraftCtas CTAs per sequence walks its
// tree. CTA r owns a contiguous slice of the vocabulary; every pass over a
// row (maxima, mass sums, the residual's maximum, the residual itself, the
// bonus draw) runs on the slices in parallel and its partial results meet
// through distributed shared memory, so that every CTA holds the same totals
// and takes the same decisions. The residual A lives in the workspace once
// the first child of a node is rejected.

#include <cuda_bf16.h>

#include "eagle_internal.cuh"
#include "eagle_ws.h"
#include "mass.cuh"
#include "sampling.cuh"

namespace eagle {
namespace {

constexpr int kDraftCtas = 8;
constexpr int kDraftThreads = 256;
constexpr int kDraftWarps = kDraftThreads / 32;

typedef unsigned __int128 u128;

struct DraftSmem {
    // all-reduce slots, two alternating sets: CTA r's partial in slot r of every CTA
    u128 rmax[2][kDraftCtas];
    unsigned long long rsum[2][kDraftCtas];
    unsigned long long rsum2[2][kDraftCtas];
    float rm[2][kDraftCtas][2];
    // block reduction scratch
    u128 wmax[kDraftWarps];
    unsigned long long wsum[kDraftWarps], wsum2[kDraftWarps];
    float wm[kDraftWarps][2];
    // the tree of the sequence
    int tok[kMaxSlots], par[kMaxSlots];
    long long drow[kMaxSlots];  // flat draft row [D * B * k, V] of each slot, -1 = never expanded
    uint32_t uni[kMaxSlots + 2];
    int removed[kMaxTopK];
    int path[kMaxDepth + 1];
    unsigned long long part[kDraftCtas];  // each CTA's share of A (the bonus draw)
    unsigned long long tscan[kDraftThreads];
    int bonus;
    int bad;
};

__device__ __forceinline__ float load_logit(const char* row, int dt, int y) {
    return dt == 1 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[y]) << 16)
                   : reinterpret_cast<const float*>(row)[y];
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int m) {
    const uint64_t lo = shfl_xor_u64(static_cast<uint64_t>(v), m);
    const uint64_t hi = shfl_xor_u64(static_cast<uint64_t>(v >> 64), m);
    return (static_cast<u128>(hi) << 64) | lo;
}

// Cluster-wide totals. Each block reduces its threads' values; thread 0
// writes the CTA's result into slot `rank` of every CTA of the cluster; after
// the cluster barrier every thread combines the slots in rank order, so every
// CTA holds the same result. The slot set alternates between calls (a CTA
// reads call i's set before it arrives at call i + 1's barrier, so call
// i + 2 may overwrite it).
struct ClusterReduce {
    cg::cluster_group cluster;
    DraftSmem* sm;
    int rank, parity;

    __device__ u128 max_u128(u128 v) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const u128 w = shfl_xor_u128(v, o);
            v = w > v ? w : v;
        }
        if (lane == 0) sm->wmax[warp] = v;
        __syncthreads();
        if (threadIdx.x == 0) {
            u128 m = 0;
            for (int i = 0; i < kDraftWarps; ++i) m = sm->wmax[i] > m ? sm->wmax[i] : m;
            for (int r = 0; r < kDraftCtas; ++r) cluster.map_shared_rank(sm, r)->rmax[parity][rank] = m;
        }
        cluster.sync();
        u128 m = 0;
        for (int r = 0; r < kDraftCtas; ++r) m = sm->rmax[parity][r] > m ? sm->rmax[parity][r] : m;
        parity ^= 1;
        return m;
    }

    // sums of two values; the CTA's own parts are left in part1 / part2
    __device__ void sum2(unsigned long long a, unsigned long long b, unsigned long long& ta, unsigned long long& tb,
                         unsigned long long* parts_a) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        a = warp_sum_u64(a);
        b = warp_sum_u64(b);
        if (lane == 0) {
            sm->wsum[warp] = a;
            sm->wsum2[warp] = b;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long x = 0, y = 0;
            for (int i = 0; i < kDraftWarps; ++i) {
                x += sm->wsum[i];
                y += sm->wsum2[i];
            }
            for (int r = 0; r < kDraftCtas; ++r) {
                DraftSmem* o = cluster.map_shared_rank(sm, r);
                o->rsum[parity][rank] = x;
                o->rsum2[parity][rank] = y;
            }
        }
        cluster.sync();
        ta = 0;
        tb = 0;
        for (int r = 0; r < kDraftCtas; ++r) {
            ta += sm->rsum[parity][r];
            tb += sm->rsum2[parity][r];
            if (parts_a != nullptr && threadIdx.x == 0) parts_a[r] = sm->rsum[parity][r];
        }
        parity ^= 1;
    }

    __device__ void max2(float a, float b, float& ma, float& mb) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
        }
        if (lane == 0) {
            sm->wm[warp][0] = a;
            sm->wm[warp][1] = b;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float x = -INFINITY, y = -INFINITY;
            for (int i = 0; i < kDraftWarps; ++i) {
                x = fmaxf(x, sm->wm[i][0]);
                y = fmaxf(y, sm->wm[i][1]);
            }
            for (int r = 0; r < kDraftCtas; ++r) {
                DraftSmem* o = cluster.map_shared_rank(sm, r);
                o->rm[parity][rank][0] = x;
                o->rm[parity][rank][1] = y;
            }
        }
        cluster.sync();
        ma = -INFINITY;
        mb = -INFINITY;
        for (int r = 0; r < kDraftCtas; ++r) {
            ma = fmaxf(ma, sm->rm[parity][r][0]);
            mb = fmaxf(mb, sm->rm[parity][r][1]);
        }
        parity ^= 1;
    }
};

template <int DT>
__global__ void __launch_bounds__(kDraftThreads) verify_draft_kernel(TreeDims d, TreeWs w, float inv_t, VerifyRng rng,
                                                                     const void* __restrict__ target,
                                                                     const void* __restrict__ draft,
                                                                     const int32_t* __restrict__ tokens,
                                                                     const int32_t* __restrict__ parent,
                                                                     const int32_t* __restrict__ n_tree,
                                                                     int32_t* __restrict__ accept_len,
                                                                     int32_t* __restrict__ slots_out,
                                                                     int32_t* __restrict__ tokens_out) {
    __shared__ DraftSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    constexpr int ES = DT == 1 ? 2 : 4;
    const int V = d.V, T = d.T;
    // this CTA's slice of the vocabulary
    const int seg = (V + kDraftCtas - 1) / kDraftCtas;
    const int lo = min(V, rank * seg), hi = min(V, lo + seg);
    uint64_t* A = w.resid + static_cast<size_t>(b) * V;
    ClusterReduce red{cluster, &sm, rank, 0};
    pdl_launch_dependents();
    pdl_wait_prior();

    const int n = n_tree[b];
    if (tid == 0) {
        sm.bad = (n < 1 || n > T) ? 1 : 0;
        sm.bonus = -1;
    }
    for (int c = tid; c < T; c += kDraftThreads) {
        sm.tok[c] = c < n ? tokens[static_cast<size_t>(b) * T + c] : -1;
        sm.par[c] = c < n ? parent[static_cast<size_t>(b) * T + c] : -1;
        sm.drow[c] = -1;
    }
    // uniform word c of sequence b: Philox4x32-10 at counter (c, b, cycle), word 0
    for (int c = tid; c < T + 2; c += kDraftThreads) {
        const uint32_t ctr[4] = {static_cast<uint32_t>(c), static_cast<uint32_t>(b), rng.c2, rng.c3};
        uint32_t out[4];
        sampling::philox4x32_10(ctr, rng.k0, rng.k1, out);
        sm.uni[c] = out[0];
    }
    __syncthreads();
    // the draft row of every kept node that was expanded: the root's is row 0
    // of step 0; node f of step s's frontier (s >= 1) owns row f of step s
    if (tid == 0) sm.drow[0] = static_cast<long long>(b) * d.k;
    for (int i = tid; i < (d.D - 1) * d.k; i += kDraftThreads) {
        const int s = 1 + i / d.k, f = i % d.k;
        const int nid = w.fnode[(s * d.B + b) * d.k + f];
        if (nid < 0) continue;
        const int slot = w.slot_of[static_cast<size_t>(b) * d.C + nid];
        if (slot > 0 && slot < n && slot < T) sm.drow[slot] = (static_cast<long long>(s) * d.B + b) * d.k + f;
    }
    for (int c = 1 + tid; c < n; c += kDraftThreads) {
        const int tk = sm.tok[c], p = sm.par[c];
        if (tk < 0 || tk >= V || p < 0 || p >= c) sm.bad = 1;
    }
    __syncthreads();
    if (sm.bad) {
        if (tid == 0 && rank == 0) raise_status(w.status, kDevBadIndex);
        cluster.sync();
        return;
    }

    int cur = 0, a = 0;
    if (tid == 0) sm.path[0] = 0;
    int outcome_bonus = -1;
    while (true) {
        const char* trow = static_cast<const char*>(target) + (static_cast<size_t>(b) * T + cur) * V * ES;
        const long long dr = sm.drow[cur];
        const char* qrow = dr >= 0 ? static_cast<const char*>(draft) + static_cast<size_t>(dr) * V * ES : nullptr;
        // children of cur in slot order (the walk stops at depth D)
        int child[kMaxTopK];
        int nchild = 0;
        if (a < d.D)
            for (int c = cur + 1; c < n && nchild < kMaxTopK; ++c)
                if (sm.par[c] == cur) child[nchild++] = c;
        if (nchild > 0 && qrow == nullptr) {  // a kept child of a node that was never expanded
            if (tid == 0 && rank == 0) raise_status(w.status, kDevBadIndex);
            break;
        }
        // maxima of the target row and the draft row
        float lm_t = -INFINITY, lm_q = -INFINITY;
        for (int y = lo + tid; y < hi; y += kDraftThreads) {
            lm_t = fmaxf(lm_t, load_logit(trow, DT, y));
            if (qrow) lm_q = fmaxf(lm_q, load_logit(qrow, DT, y));
        }
        float Mt, Mq;
        red.max2(lm_t, lm_q, Mt, Mq);
        // sums of the masses
        unsigned long long st = 0, sq = 0;
        for (int y = lo + tid; y < hi; y += kDraftThreads) {
            st += fixed_mass(load_logit(trow, DT, y), Mt, inv_t);
            if (qrow && nchild > 0) sq += fixed_mass(load_logit(qrow, DT, y), Mq, inv_t);
        }
        unsigned long long SA, SQ;
        red.sum2(st, sq, SA, SQ, sm.part);
        bool materialized = false;  // A in the workspace (after a rejection) or the target row's masses
        int nrem = 0;
        int next = -1;
        for (int j = 0; j < nchild; ++j) {
            const int c = child[j];
            const int x = sm.tok[c];
            const uint64_t Ax = materialized ? __ldcg(A + x) : fixed_mass(load_logit(trow, DT, x), Mt, inv_t);
            const uint64_t Qx = fixed_mass(load_logit(qrow, DT, x), Mq, inv_t);
            const u128 lhs = static_cast<u128>(static_cast<uint64_t>(sm.uni[c] >> 8) * Qx) * SA;
            const u128 rhs = (static_cast<u128>(Ax) * SQ) << 24;
            if (lhs < rhs) {
                next = c;
                break;
            }
            // rejected: the residual r(y) = max(0, A[y] SQ - Q[y] SA) (x still in Q)
            auto resid = [&](int y) -> u128 {
                const uint64_t Ay = materialized ? __ldcg(A + y) : fixed_mass(load_logit(trow, DT, y), Mt, inv_t);
                bool rem = false;
                for (int i = 0; i < nrem; ++i) rem |= sm.removed[i] == y;
                const uint64_t Qy = rem ? 0ull : fixed_mass(load_logit(qrow, DT, y), Mq, inv_t);
                const u128 pa = static_cast<u128>(Ay) * SQ, qa = static_cast<u128>(Qy) * SA;
                return pa > qa ? pa - qa : 0;
            };
            u128 lmax = 0;
            for (int y = lo + tid; y < hi; y += kDraftThreads) {
                const u128 r = resid(y);
                lmax = r > lmax ? r : lmax;
            }
            const u128 mx = red.max_u128(lmax);
            if (mx > 0) {
                int sh = 0;
                while ((mx >> sh) > (static_cast<u128>(1) << 40)) ++sh;
                // every CTA reads its slice of the old A before any writes the new one
                unsigned long long s_new = 0;
                uint64_t vals[8];
                for (int y0 = lo + tid; y0 < hi; y0 += 8 * kDraftThreads) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int y = y0 + u * kDraftThreads;
                        vals[u] = y < hi ? static_cast<uint64_t>(resid(y) >> sh) : 0ull;
                    }
                    // (the slice of this thread's elements is its own: reads and writes of A[y] for
                    // one y are by the same thread)
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int y = y0 + u * kDraftThreads;
                        if (y < hi) {
                            A[y] = vals[u];
                            s_new += vals[u];
                        }
                    }
                }
                unsigned long long unused;
                red.sum2(s_new, 0ull, SA, unused, sm.part);
                materialized = true;
            }
            SQ -= Qx;
            if (tid == 0) sm.removed[nrem] = x;
            ++nrem;
            __syncthreads();
        }
        if (next >= 0) {
            ++a;
            if (tid == 0) sm.path[a] = next;
            cur = next;
            continue;
        }
        // the bonus: the smallest y whose running sum of A exceeds t = floor(U64 SA / 2^64);
        // sm.part holds the CTAs' shares of A (from the last cluster sum)
        __syncthreads();
        const uint64_t U64 = (static_cast<uint64_t>(sm.uni[T + 1]) << 32) | sm.uni[T];
        const unsigned long long tdraw = static_cast<unsigned long long>((static_cast<u128>(U64) * SA) >> 64);
        unsigned long long before = 0;
        for (int r = 0; r < rank; ++r) before += sm.part[r];
        const unsigned long long mine = sm.part[rank];
        if (tdraw >= before && tdraw < before + mine) {
            // this CTA's slice holds the draw: thread i sums a contiguous run of it
            const int per = (hi - lo + kDraftThreads - 1) / kDraftThreads;
            const int y0 = lo + tid * per, y1 = min(hi, y0 + per);
            unsigned long long s = 0;
            for (int y = y0; y < y1; ++y)
                s += materialized ? __ldcg(A + y) : fixed_mass(load_logit(trow, DT, y), Mt, inv_t);
            sm.tscan[tid] = s;
            __syncthreads();
            if (tid == 0) {
                unsigned long long run = before;
                for (int i = 0; i < kDraftThreads; ++i) {
                    const unsigned long long nx = run + sm.tscan[i];
                    sm.tscan[i] = run;  // exclusive prefix
                    run = nx;
                }
            }
            __syncthreads();
            unsigned long long run = sm.tscan[tid];
            if (tdraw >= run && tdraw < run + s) {
                for (int y = y0; y < y1; ++y) {
                    run += materialized ? __ldcg(A + y) : fixed_mass(load_logit(trow, DT, y), Mt, inv_t);
                    if (run > tdraw) {
                        sm.bonus = y;
                        break;
                    }
                }
            }
            __syncthreads();
            outcome_bonus = sm.bonus;
            if (tid == 0) {
                const int Dp1 = d.D + 1;
                accept_len[b] = a;
                for (int j = 0; j < Dp1; ++j) {
                    slots_out[b * Dp1 + j] = j <= a ? sm.path[j] : -1;
                    tokens_out[b * Dp1 + j] = j < a ? sm.tok[sm.path[j + 1]] : (j == a ? outcome_bonus : -1);
                }
            }
        }
        break;
    }
    cluster.sync();  // no CTA leaves while another may still write to its shared memory
}

// ------------------------------------------------ lossless acceptance walk ---
//
// Stage 6, lossless rule with deterministic candidates ("EAGLE-2: Faster
// Inference ..." summary, 2.1 Speculative Sampling: accept a drafted token
// with probability min(1, p/q); with the draft's top-k children q is a point
// mass, so child x of node u is accepted with probability P_u(x) / S, S the
// mass left after the earlier children's removal; with every child rejected
// the bonus token is drawn from the residual). The integer masses are those of
// the row kernel's definition, floor(dexp((x - M_t) / T) 2^40), M_t the row
// maximum the row kernel wrote. Only the rows of nodes the walk visits are
// summed: one cluster of kWalkCtas CTAs per sequence, CTA r summing its slice
// of the vocabulary (one 16-byte vector per thread and round, all loads of a
// round in flight together) and keeping a sum per (round, warp) piece for the
// bonus draw; the slices' sums meet through distributed shared memory, so
// every CTA takes the same decisions.

constexpr int kWalkCtas = 8;  // CTAs per sequence (a 16-CTA cluster measured slower: longer cluster barriers)
constexpr int kWalkThreads = 256;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kWalkMaxRounds = 4;  // V <= 262144 bf16 or fp32

struct LosslessSmem {
    unsigned long long rsum[2][kWalkCtas];  // all-reduce slots, two alternating sets
    unsigned long long wsum[kWalkWarps];
    unsigned long long piece[kWalkMaxRounds * kWalkWarps];  // this CTA's mass per (round, warp) of the current row
    unsigned long long part[kWalkCtas];                  // every CTA's share of the current row's mass
    int tok[kMaxSlots], par[kMaxSlots];
    float rmax[kMaxSlots];
    unsigned long long pmass[kMaxSlots];  // mass of slot c's token in its parent's row
    uint32_t uni[kMaxSlots + 2];
    int path[kMaxDepth + 1];
    int removed_tok[kMaxTopK];
    unsigned long long removed_mass[kMaxTopK];
    int child[kMaxTopK];
    unsigned long long s_left;
    int next, nrem;
    int bad, bonus, holder;
};

// u24 * S < P * 2^24 for u24 < 2^24, S < 2^64, P < 2^41, in 64-bit halves.
__device__ __forceinline__ bool accept_u24(uint32_t u24, unsigned long long S, unsigned long long P) {
    const unsigned long long lh = __umul64hi(u24, S), ll = static_cast<unsigned long long>(u24) * S;
    const unsigned long long rh = P >> 40, rl = P << 24;
    return lh < rh || (lh == rh && ll < rl);
}

template <int DT>
__device__ __forceinline__ void unpack_vec(const uint4& u, float (&x)[16 / (DT == 1 ? 2 : 4)]) {
    if (DT == 1) {
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(wv[i] << 16);
            x[2 * i + 1] = __uint_as_float(wv[i] & 0xffff0000u);
        }
    } else {
        x[0] = __uint_as_float(u.x);
        x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z);
        x[3] = __uint_as_float(u.w);
    }
}

template <int DT>
__global__ void __launch_bounds__(kWalkThreads) verify_lossless_walk_kernel(TreeDims d, TreeWs w, float inv_t,
                                                                            VerifyRng rng,
                                                                            const void* __restrict__ target,
                                                                            const int32_t* __restrict__ tokens,
                                                                            const int32_t* __restrict__ parent,
                                                                            const int32_t* __restrict__ n_tree,
                                                                            int32_t* __restrict__ accept_len,
                                                                            int32_t* __restrict__ slots_out,
                                                                            int32_t* __restrict__ tokens_out) {
    __shared__ LosslessSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int ES = DT == 1 ? 2 : 4;
    constexpr int EPV = 16 / ES;
    constexpr int kWalkVec = 8;  // 16-byte vectors per thread and round
    const int V = d.V, T = d.T;
    // this CTA's slice [lo, hi) of the vocabulary, whole 16-byte vectors
    const int seg = (V / EPV + kWalkCtas - 1) / kWalkCtas * EPV;
    const int lo = min(V, rank * seg), hi = min(V, lo + seg);
    const int nvec = (hi - lo) / EPV;
    // rounds of kWalkVec vectors per thread, the same in every CTA (their control flow must agree)
    const int rounds = (seg / EPV + kWalkThreads * kWalkVec - 1) / (kWalkThreads * kWalkVec);
    pdl_launch_dependents();
    pdl_wait_prior();

    const int n = n_tree[b];
    const size_t tb = static_cast<size_t>(b) * T;
    if (tid == 0) {
        sm.bad = (n < 1 || n > T || rounds > kWalkMaxRounds) ? 1 : 0;
        sm.bonus = -1;
    }
    __syncthreads();
    const int nn = sm.bad ? 1 : n;
    for (int c = tid; c < nn; c += kWalkThreads) {
        sm.tok[c] = tokens[tb + c];
        sm.par[c] = parent[tb + c];
        sm.rmax[c] = __ldcg(&w.row_max[tb + c]);
        // the mass of slot c's token in its parent's row, from the row kernel (which had the parent row streaming)
        sm.pmass[c] = c > 0 ? __ldcg(&w.pmass[tb + c]) : 0ull;
    }
    // uniform word c of sequence b: Philox4x32-10 at counter (c, b, cycle), word 0
    for (int c = tid; c < T + 2; c += kWalkThreads) {
        const uint32_t ctr[4] = {static_cast<uint32_t>(c), static_cast<uint32_t>(b), rng.c2, rng.c3};
        uint32_t out[4];
        sampling::philox4x32_10(ctr, rng.k0, rng.k1, out);
        sm.uni[c] = out[0];
    }
    __syncthreads();
    for (int c = 1 + tid; c < nn; c += kWalkThreads) {
        const int tk = sm.tok[c], p = sm.par[c];
        if (tk < 0 || tk >= V || p < 0 || p >= c) sm.bad = 1;
    }
    __syncthreads();
    const bool bad = sm.bad != 0;
    int parity = 0;
    // Integer mass of row `cur` summed over the cluster: every CTA returns the
    // total and keeps its pieces (sm.piece) and every CTA's share (sm.part).
    auto row_mass = [&](int cur) -> unsigned long long {
        const char* row = static_cast<const char*>(target) + (tb + cur) * V * ES;
        const float M = sm.rmax[cur];
        const uint64_t neg_m2 = f2_pack(-M, -M), inv_t2 = f2_pack(inv_t, inv_t);
        for (int rd = 0; rd < rounds; ++rd) {
            const int vb = rd * kWalkThreads * kWalkVec + warp * 32 * kWalkVec + lane;
            uint4 u[kWalkVec];
#pragma unroll
            for (int j = 0; j < kWalkVec; ++j)
                if (vb + j * 32 < nvec)
                    u[j] = __ldcg(reinterpret_cast<const uint4*>(row + (static_cast<size_t>(lo) + (vb + j * 32) * EPV) * ES));
            uint32_t ahi = 0, alo = 0;  // at most 64 elements: no overflow
#pragma unroll
            for (int j = 0; j < kWalkVec; ++j) {
                if (vb + j * 32 >= nvec) continue;
                float x[EPV];
                unpack_vec<DT>(u[j], x);
#pragma unroll
                for (int e = 0; e < EPV; e += 2) pair_mass_parts(x[e], x[e + 1], neg_m2, inv_t2, ahi, alo);
            }
            const unsigned long long ws = warp_sum_u64(mass_of_parts(ahi, alo));
            if (lane == 0) sm.piece[rd * kWalkWarps + warp] = ws;
        }
        __syncthreads();
        if (warp == 0) {
            unsigned long long mine = lane < rounds * kWalkWarps ? sm.piece[lane] : 0ull;
            mine = warp_sum_u64(mine);
            if (lane < kWalkCtas) cluster.map_shared_rank(&sm, lane)->rsum[parity][rank] = mine;
        }
        cluster.sync();
        const unsigned long long pr = lane < kWalkCtas ? sm.rsum[parity][lane] : 0ull;
        if (warp == 0 && lane < kWalkCtas) sm.part[lane] = pr;
        parity ^= 1;
        return warp_sum_u64(pr);
    };

    int cur = 0, a = 0, nrem = 0;
    unsigned long long S = 0;
    if (tid == 0) sm.path[0] = 0;
    while (!bad) {
        S = row_mass(cur);
        if (tid == 0 && rank == 0) w.row_mass[tb + cur] = S;
        // children of cur (contiguous in slot order) tested in order by warp
        // 0, lane j on child j: accepted iff u24 S_j < P 2^24, S_j the mass
        // left after the earlier children's removal
        if (warp == 0) {
            int nchild = 0;
            if (a < d.D) {
                for (int c0w = cur + 1; c0w < n && nchild < kMaxTopK; c0w += 32) {
                    const int c = c0w + lane;
                    const bool is = c < n && sm.par[c] == cur;
                    const unsigned bal = __ballot_sync(0xffffffffu, is);
                    const int pos = nchild + __popc(bal & lanemask_lt());
                    if (is && pos < kMaxTopK) sm.child[pos] = c;
                    nchild += __popc(bal);
                }
                nchild = min(nchild, kMaxTopK);
            }
            __syncwarp();
            const int c = lane < nchild ? sm.child[lane] : -1;
            const unsigned long long P = c >= 0 ? sm.pmass[c] : 0ull;
            unsigned long long incl = P;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = shfl_u64(incl, max(lane - o, 0));
                if (lane >= o) incl += y;
            }
            const bool acc = c >= 0 && accept_u24(sm.uni[c] >> 8, S - (incl - P), P);
            const unsigned bal = __ballot_sync(0xffffffffu, acc);
            const int first = bal ? __ffs(bal) - 1 : nchild;  // children before it were rejected
            if (lane < first && c >= 0) {
                sm.removed_tok[lane] = sm.tok[c];
                sm.removed_mass[lane] = P;
            }
            const unsigned long long rej = first > 0 ? shfl_u64(incl, first - 1) : 0ull;
            if (lane == 0) {
                sm.next = bal ? sm.child[first] : -1;
                sm.nrem = first;
                sm.s_left = S - rej;
            }
        }
        __syncthreads();
        const int next = sm.next;
        nrem = sm.nrem;
        S = sm.s_left;
        if (next < 0) break;
        ++a;
        if (tid == 0) sm.path[a] = next;
        cur = next;
        __syncthreads();
    }
    __syncthreads();
    if (!bad) {
        // The bonus: the smallest y of row cur (removed tokens excluded) whose
        // running mass exceeds t = floor(U64 S / 2^64). The CTA whose slice
        // holds the draw finds its piece, then the element (one vector per
        // thread, block scan).
        int rtok[kMaxTopK];
        unsigned long long rmass[kMaxTopK];
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i) {
            rtok[i] = i < nrem ? sm.removed_tok[i] : -1;
            rmass[i] = i < nrem ? sm.removed_mass[i] : 0ull;
        }
        auto removed_in = [&](int y0, int y1) -> unsigned long long {
            unsigned long long m = 0;
#pragma unroll
            for (int i = 0; i < kMaxTopK; ++i)
                if (rtok[i] >= y0 && rtok[i] < y1) m += rmass[i];
            return m;
        };
        const uint64_t U64 = (static_cast<uint64_t>(sm.uni[T + 1]) << 32) | sm.uni[T];
        const unsigned long long tdraw = __umul64hi(U64, S);
        // every CTA knows which slice holds the draw (the same shares everywhere)
        int holder = -1;
        unsigned long long before = 0, upto = 0;  // this CTA's prefix; the running prefix over all CTAs
        for (int r = 0; r < kWalkCtas; ++r) {
            const unsigned long long share = sm.part[r] - removed_in(min(V, r * seg), min(V, r * seg + seg));
            if (holder < 0 && share > 0 && tdraw >= upto && tdraw < upto + share) holder = r;
            if (r < rank) before += share;
            upto += share;
        }
        if (tid == 0) sm.holder = holder;
        if (holder == rank) {
            // the piece: (round, warp) ranges in element order
            int pq = -1;
            unsigned long long run = before;
            for (int q = 0; q < rounds * kWalkWarps; ++q) {
                const int v0 = (q / kWalkWarps) * kWalkThreads * kWalkVec + (q % kWalkWarps) * 32 * kWalkVec;
                const int y0 = lo + v0 * EPV, y1 = min(hi, y0 + 32 * kWalkVec * EPV);
                const unsigned long long m = y0 < hi ? sm.piece[q] - removed_in(y0, y1) : 0ull;
                if (m > 0 && tdraw < run + m) {
                    pq = q;
                    break;
                }
                run += m;
            }
            // thread (warp j < kWalkVec, lane l) takes vector v0 + 32 j + l of the piece (element order)
            const int v0 = pq < 0 ? 0 : (pq / kWalkWarps) * kWalkThreads * kWalkVec + (pq % kWalkWarps) * 32 * kWalkVec;
            const int v = v0 + warp * 32 + lane;
            const int y0 = lo + v * EPV;
            uint64_t em[EPV];
            unsigned long long vm = 0;
            if (pq >= 0 && warp < kWalkVec && v < nvec) {
                const char* row = static_cast<const char*>(target) + (tb + cur) * V * ES;
                const uint4 u = __ldcg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(y0) * ES));
                const float M = sm.rmax[cur];
                const uint64_t neg_m2 = f2_pack(-M, -M), inv_t2 = f2_pack(inv_t, inv_t);
                float x[EPV];
                unpack_vec<DT>(u, x);
#pragma unroll
                for (int e = 0; e < EPV; e += 2) pair_mass2(x[e], x[e + 1], neg_m2, inv_t2, em[e], em[e + 1]);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
#pragma unroll
                    for (int i = 0; i < kMaxTopK; ++i)
                        if (rtok[i] == y0 + e) em[e] = 0;
                    vm += em[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPV; ++e) em[e] = 0;
            }
            unsigned long long incl = vm;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = shfl_u64(incl, max(lane - o, 0));
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.wsum[warp] = incl;
            __syncthreads();
            unsigned long long ex = run + incl - vm;
            for (int i = 0; i < warp; ++i) ex += sm.wsum[i];
            if (vm > 0 && tdraw >= ex && tdraw < ex + vm) {
                unsigned long long rr = ex;
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    rr += em[e];
                    if (rr > tdraw) {
                        sm.bonus = y0 + e;
                        break;
                    }
                }
            }
        }
    }
    // The outputs: written by the CTA that holds the draw (rank 0 when none
    // does). After the last cluster barrier of the walk no CTA touches
    // another's shared memory, so the CTAs leave without a final barrier.
    __syncthreads();
    if (tid == 0 && (bad ? rank == 0 : (sm.holder == rank || (sm.holder < 0 && rank == 0)))) {
        const int bonus = sm.bonus;
        const int Dp1 = d.D + 1;
        accept_len[b] = a;
        for (int j = 0; j < Dp1; ++j) {
            slots_out[b * Dp1 + j] = j <= a ? sm.path[j] : -1;
            tokens_out[b * Dp1 + j] = j < a ? sm.tok[sm.path[j + 1]] : (j == a ? bonus : -1);
        }
        if (bad || bonus < 0) raise_status(w.status, kDevBadIndex);
    }
}

}  // namespace

cudaError_t launch_verify_draft(const TreeDims& d, const TreeWs& ws, float inv_temp, VerifyRng rng,
                                const void* target, const void* draft, const int32_t* tokens, const int32_t* parent,
                                const int32_t* n_tree, int32_t* accept_len, int32_t* slots, int32_t* out_tokens,
                                cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kDraftCtas, d.B, 1);
    cfg.blockDim = dim3(kDraftThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kDraftCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    TreeDims dd = d;
    TreeWs ww = ws;
    void* args[] = {&dd,
                    &ww,
                    &inv_temp,
                    &rng,
                    const_cast<void**>(&target),
                    const_cast<void**>(&draft),
                    const_cast<int32_t**>(&tokens),
                    const_cast<int32_t**>(&parent),
                    const_cast<int32_t**>(&n_tree),
                    &accept_len,
                    &slots,
                    &out_tokens};
    const void* k = d.dtype == 1 ? reinterpret_cast<const void*>(verify_draft_kernel<1>)
                                 : reinterpret_cast<const void*>(verify_draft_kernel<0>);
    return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch_verify_walk(const TreeDims& d, const TreeWs& ws, float inv_temp, VerifyRng rng, const void* target,
                               const int32_t* tokens, const int32_t* parent, const int32_t* n_tree,
                               int32_t* accept_len, int32_t* slots, int32_t* out_tokens, cudaStream_t stream) {
    constexpr int nc = kWalkCtas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nc, d.B, 1);
    cfg.blockDim = dim3(kWalkThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    TreeDims dd = d;
    TreeWs ww = ws;
    void* args[] = {&dd, &ww, &inv_temp, &rng, const_cast<void**>(&target), const_cast<int32_t**>(&tokens),
                    const_cast<int32_t**>(&parent), const_cast<int32_t**>(&n_tree), &accept_len, &slots,
                    &out_tokens};
    const void* fn = d.dtype == 1 ? reinterpret_cast<const void*>(verify_lossless_walk_kernel<1>)
                                  : reinterpret_cast<const void*>(verify_lossless_walk_kernel<0>);
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace eagle

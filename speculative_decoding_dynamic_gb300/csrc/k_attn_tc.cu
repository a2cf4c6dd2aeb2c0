// Stage 5, tensor-core path (sm_103a): tree-masked GQA attention.
//
// For sequence b, KV head hk, the G = Hq/Hkv query heads of every tree slot
// form M = G*T query rows (row r <-> slot r / G, head hk*G + r % G, matching
// the [B, T, Hq, d] layout of Q). One CTA owns a 128-row block of them and a
// range of 128-key tiles of the sequence's keys (prefix [0, L_b) then the
// tree slots at L_b + j), and runs, per key tile j:
//   S = Q K^T        tcgen05.mma kind::f16, bf16 operands from shared memory,
//                    fp32 accumulator in tensor memory, double buffered
//                    (TMEM columns 128 (j & 1) ..), so QK^T of tile j+1 runs
//                    while the softmax works on tile j
//   P = softmax part four threads per row (TMEM lane = row, 32 key columns
//                    each; row maxima exchanged in shared memory): scale,
//                    tree mask, exponentials in the log2 domain against a
//                    reference maximum, P written as bf16 pairs into tensor
//                    memory (double buffered, columns 384 + 64 (j & 1) ..)
//   O += P V         tcgen05.mma with A = P read from tensor memory, V from
//                    shared memory (MN-major), accumulating in TMEM columns
//                    256..383; the reference maximum is raised (O and the row
//                    sum rescaled in place) only when a tile's maximum exceeds
//                    it by more than 2^8, so exponentials stay below 256
// K and V tiles arrive by TMA (cp.async.bulk.tensor, 128B swizzle) into
// their own rings (a K stage frees after QK^T, a V stage after PV), issued
// by two lanes of warp 0; one thread of warp 1 issues every MMA; warps 2..17
// do the softmax. mbarriers order them, every wait is bounded. Key ranges of
// one (b, hk, row block) may be split over CTAs (split-KV): each writes
// (O, max, sum) partials and the last CTA to arrive on a per-unit counter
// merges them (log-sum-exp combine).
//
// Keys of slot i: every prefix position and the tree slots set in mask row i
// ["EAGLE" notes, EAGLE 方法: Medusa-style tree attention verifies every
// branch in one pass; "EAGLE-2: Faster Inference ..." summary 4.2].

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "attn_common.cuh"
#include "eagle_internal.cuh"
#include "eagle_ws.h"
#include "tc_ptx.cuh"

namespace eagle {

cudaError_t launch_attention_simt(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream);

namespace {

constexpr int kBM = 128;                   // query rows per CTA (one MMA M)
constexpr int kBN = 128;                   // keys per tile (MMA N of QK^T, K of PV)
constexpr int kHD = 128;                   // head dim (MMA K of QK^T, N of PV)
constexpr int kTile = kBM * kHD * 2;       // 32 KB: a 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;           // 16 KB: 128 rows x 64 columns (one swizzle-128B column block)
constexpr int kKStages = 3;  // K tiles in flight (a stage frees after QK^T)
constexpr int kVStages = 2;  // V tiles in flight (a stage frees after PV)
constexpr int kSoftmaxThreads = 512;
constexpr int kGroupThreads = kSoftmaxThreads / 2;  // one softmax group: alternate key tiles
constexpr int kThreads = 64 + kSoftmaxThreads;  // warp 0 TMA, warp 1 MMA, warps 2..17 softmax (four column quarters)
constexpr int kSmemQ = 0;
constexpr int kSmemK = kTile;                      // K stage s at kSmemK + s * kTile
constexpr int kSmemV = kSmemK + kKStages * kTile;  // V stage s at kSmemV + s * kTile
constexpr int kSmemBytes = kSmemV + kVStages * kTile;  // 192 KB
constexpr int kTmemCols = 512;  // S double buffer (2 x 128 columns; P over S), O per softmax group (2 x 128)
constexpr int kMaxW = kMaxSlots / 32;

struct TcParams {
    int B, T, Hq, Hkv, G, n_rb, nsplit, tps, max_len, W;
    const int32_t* prefix_len;
    const uint32_t* mask;
    const int32_t* n_tree;
    __nv_bfloat16* out;
    float* part_o;   // [units * nsplit, 128, 128]
    float* part_ml;  // [units * nsplit, 128, 2]
    int* tickets;    // [units]
    int* status;
    float scale_log2;
};

// ---------------------------------------------------------------- PTX ---
// TMA, tcgen05 MMA and tensor-memory helpers: tc_ptx.cuh.

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory"); }
// The two warps of softmax group g that serve one TMEM lane quarter (the
// rows 32 q4 .. 32 q4 + 31, one warp per column half) meet on barrier
// 2 + 4 g + q4.
__device__ __forceinline__ void named_sync_pair(int g, int q4) {
    asm volatile("bar.sync %0, 64;" ::"r"(2 + 4 * g + q4) : "memory");
}

// ------------------------------------------------------------- kernel ---

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_q, bar_k_full[kKStages], bar_k_empty[kKStages], bar_v_full[kVStages], bar_v_empty[kVStages],
        bar_s_full[2], bar_p_full[2], bar_o_full[2], bar_comb;
    __shared__ uint32_t tmem_holder;
    __shared__ uint32_t mask_sm[kBM][kMaxW];
    __shared__ int sh_last;
    __shared__ float xch[2][2][2][kBM];  // [group][tile parity][column half][row]: per-tile row maxima
    __shared__ float gm[2][kBM];         // [group][row]: reference maximum (-inf: the group saw no key)
    __shared__ float gl[2][2][kBM];      // [group][column half][row]: row sums

    const int rb = blockIdx.x, split = blockIdx.y;
    const int b = blockIdx.z / p.Hkv, hk = blockIdx.z % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    // Q and the first K/V tiles of this CTA's key range into L2 while the
    // previous kernel finishes (hints only; a tile past the sequence's keys
    // is simply not used)
    if (warp == 0 && lane < 2) {
        const int key0 = split * p.tps * kBN;
        if (lane == 0) {
            tma_prefetch_4d(&tm_q, 0, hk * p.G, rb * (kBM / p.G), b);
            tma_prefetch_4d(&tm_q, 64, hk * p.G, rb * (kBM / p.G), b);
        }
        const CUtensorMap* map = lane == 0 ? &tm_k : &tm_v;
        for (int jj = 0; jj < 2 && key0 + jj * kBN < p.max_len; ++jj) {
            tma_prefetch_4d(map, 0, hk, key0 + jj * kBN, b);
            tma_prefetch_4d(map, 64, hk, key0 + jj * kBN, b);
        }
    }
    pdl_wait_prior();
    const int L = p.prefix_len[b];
    const int n = p.n_tree[b];
    const bool bad = L < 0 || L + p.T > p.max_len || n < 1 || n > p.T;
    const int nkeys = bad ? 0 : L + n;
    const int ntiles = (nkeys + kBN - 1) / kBN;
    const int nsplit_b = bad ? 1 : (ntiles + p.tps - 1) / p.tps;
    if (split >= nsplit_b) return;  // uniform over the CTA
    const int t_begin = split * p.tps, t_end = min(ntiles, t_begin + p.tps);
    const int n_local = bad ? 0 : t_end - t_begin;
    const int unit = (b * p.Hkv + hk) * p.n_rb + rb;
    const int i0 = rb * (kBM / p.G);  // first slot of this row block

    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bar_k_full[s], 1);
            mbar_init(&bar_k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bar_v_full[s], 1);
            mbar_init(&bar_v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_s_full[s], 1);
            mbar_init(&bar_p_full[s], kGroupThreads);
            mbar_init(&bar_o_full[s], 1);
        }
        mbar_init(&bar_comb, 1);
        fence_mbar_init();

        if (bad) raise_status(p.status, kDevBadIndex);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp >= 2 && warp < 6) {  // this row's mask words
        const int r = ((warp & 3) << 5) | lane;
        const int i = i0 + r / p.G;
        for (int w = 0; w < kMaxW; ++w)
            mask_sm[r][w] = (w < p.W && i < p.T && !bad) ? p.mask[(static_cast<size_t>(b) * p.T + i) * p.W + w] : 0u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    const uint32_t tmem_s = tmem;        // S(j) at tmem_s + 128 (j & 1); P(j) over its first 64 columns
    const uint32_t tmem_o = tmem + 256;  // O of group g at tmem_o + 128 g

    unsigned char* sQ = smem + kSmemQ;

    if (warp == 0) {
        // ------------------------------------------------ TMA producers ---
        // Lane 0 loads Q and the K tiles, lane 1 the V tiles: a K stage is
        // free once QK^T of its tile is done, a V stage once PV is, so the K
        // of the next tiles does not wait behind V.
        if (lane < 2 && n_local > 0) {
            const bool is_k = lane == 0;
            if (is_k) {
                mbar_arrive_expect_tx(&bar_q, kTile);
                tma_load_4d(sQ, &tm_q, 0, hk * p.G, i0, b, &bar_q);
                tma_load_4d(sQ + kHalf, &tm_q, 64, hk * p.G, i0, b, &bar_q);
            }
            uint64_t* full = is_k ? bar_k_full : bar_v_full;
            uint64_t* empty = is_k ? bar_k_empty : bar_v_empty;
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            const int ns = is_k ? kKStages : kVStages;
            for (int jj = 0; jj < n_local; ++jj) {
                const int st = jj % ns;
                if (jj >= ns && !mbar_wait_sleep(&empty[st], ((jj / ns) - 1) & 1)) {
                    raise_status(p.status, kDevTimeout);
                    break;
                }
                unsigned char* dst = smem + (is_k ? kSmemK : kSmemV) + st * kTile;
                const int key0 = (t_begin + jj) * kBN;
                mbar_arrive_expect_tx(&full[st], kTile);
                tma_load_4d(dst, map, 0, hk, key0, b, &full[st]);
                tma_load_4d(dst + kHalf, map, 64, hk, key0, b, &full[st]);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ---
        // Tile j belongs to softmax group j & 1. QK(j) goes into S buffer
        // j & 1, whose previous content P(j-2) was read by PV(j-2), issued
        // earlier (tcgen05.mma of one thread execute in issue order). PV(j)
        // reads P(j) from that buffer and accumulates into O of group j & 1.
        // Issue order QK(0) QK(1) PV(0) QK(2) PV(1) QK(3) ...: while one
        // group computes its softmax, the tensor pipe serves the other.
        if (lane == 0 && n_local > 0) {
            constexpr uint32_t id_qk = idesc_bf16(kBM, kBN, 0);
            constexpr uint32_t id_pv = idesc_bf16(kBM, kHD, 1);
            const uint32_t aQ = smem_u32(sQ);
            bool ok = mbar_wait_sleep(&bar_q, 0);
            auto issue_pv = [&](int jp) -> bool {
                const int g = jp & 1, sp = jp % kVStages;
                if (!mbar_wait_sleep(&bar_p_full[g], (jp >> 1) & 1) ||
                    !mbar_wait_sleep(&bar_v_full[sp], (jp / kVStages) & 1))
                    return false;
                tc_fence_after();
                const uint32_t aV = smem_u32(smem + kSmemV + sp * kTile);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)  // A = P from TMEM: 16 keys = 8 columns per MMA
                    mma_bf16_ts(tmem_o + g * kHD, tmem_s + g * kBN + kk * 8, smem_desc(aV + kk * 2048, kHalf, 1024),
                                id_pv, (jp >= 2 || kk > 0) ? 1 : 0);
                mma_commit(&bar_v_empty[sp]);
                mma_commit(&bar_o_full[g]);
                return true;
            };
            for (int jj = 0; ok && jj < n_local; ++jj) {
                const int sb = jj & 1, sk = jj % kKStages;
                ok = mbar_wait_sleep(&bar_k_full[sk], (jj / kKStages) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t aK = smem_u32(smem + kSmemK + sk * kTile);
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16(tmem_s + sb * kBN, smem_desc(aQ + off, 16, 1024), smem_desc(aK + off, 16, 1024), id_qk,
                             kk > 0);
                }
                mma_commit(&bar_k_empty[sk]);
                mma_commit(&bar_s_full[sb]);
                if (jj > 0) ok = issue_pv(jj - 1);
            }
            if (ok) ok = issue_pv(n_local - 1);
            if (!ok) raise_status(p.status, kDevTimeout);
        }
    } else {
        // ------------------------------------------------------ softmax ---
        // Two groups of eight warps take alternate key tiles (group g: tiles
        // g, g + 2, ...), each with its own reference maximum, row sum and O
        // accumulator; they are combined at the end. In a group, two threads
        // serve a query row (TMEM lane): warp w serves lane quarter w % 4 and
        // key / output columns 64 h onwards, h the warp's column half. The
        // two halves exchange row maxima through shared memory. The
        // exponentials use a reference maximum m_use raised (O_g, l rescaled)
        // only when a tile's maximum exceeds it by more than 2^8.
        const int gidx = (warp - 2) >> 3;                // softmax group
        const int ch = ((warp - 2) >> 2) & 1;            // column half
        const int cb = ch * 64;                          // first key / output column of the half
        const int q4 = warp & 3;
        const int r = (q4 << 5) | lane;                  // row of the block = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const int grow = rb * kBM + r;                   // row within the (b, hk) problem
        const int i = i0 + r / p.G;                      // tree slot of the row
        const int g = r % p.G;
        const float sc = p.scale_log2;
        // a lane quarter whose 32 rows are all past the problem's rows does no
        // arithmetic (it still takes part in every barrier and V clearing)
        const bool quarter_live = rb * kBM + q4 * 32 < p.G * p.T;
        const uint32_t s_cols = tmem_s + gidx * kBN;
        const uint32_t o_cols = tmem_o + gidx * kHD;
        float m_use = 0.0f, lh = 0.0f;                   // lh: this half's share of the group's row sum
        bool seen = false;
        bool ok = true;
        for (int jj = gidx; jj < n_local; jj += 2) {
            const int u = jj >> 1;  // the group's own tile count
            const int key0 = (t_begin + jj) * kBN;
            // After a timed-out wait a warp skips the work of the remaining tiles
            // but still takes every named barrier, so the others never wait for
            // it without bound.
            if (ok && !__all_sync(0xffffffffu, mbar_wait_sleep(&bar_s_full[gidx], u & 1))) ok = false;
            tc_fence_after();
            float sv[2][32];
            if (ok && quarter_live) {
                tmem_ld32(s_cols + lane_off + cb, sv[0]);
                tmem_ld32(s_cols + lane_off + cb + 32, sv[1]);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) sv[0][e] = sv[1][e] = -INFINITY;
            }
            // visibility of the half's keys, 32 at a time: prefix keys, then tree slots in mask row i
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const int kb = key0 + cb + 32 * hq;
                const int npre = L - kb;  // keys of the 32 inside the prefix
                if (npre < 32) {
                    const uint32_t pre = npre > 0 ? (1u << npre) - 1u : 0u;
                    const int j0 = kb - L;  // slot of the first key (may be negative)
                    const int lo = j0 < 0 ? 0 : j0;
                    const int w0 = lo >> 5, sh = lo & 31;
                    uint32_t win = mask_sm[r][w0 & (kMaxW - 1)] >> sh;
                    if (sh && w0 + 1 < kMaxW) win |= mask_sm[r][w0 + 1] << (32 - sh);
                    if (w0 >= kMaxW) win = 0u;
                    const int limit = n - lo;  // slots j >= n are never visible
                    if (limit <= 0) win = 0u;
                    else if (limit < 32) win &= (1u << limit) - 1u;
                    uint32_t tree = j0 < 0 ? (win << (-j0)) : win;
                    if (j0 <= -32) tree = 0u;
                    const uint32_t vis = pre | tree;
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[hq][e] = ((vis >> e) & 1u) ? sv[hq][e] : -INFINITY;
                }
            }
            float mx = fmaxf(max32(sv[0]), max32(sv[1])) * sc;  // the scale is positive
            if (quarter_live) {
                xch[gidx][u & 1][ch][r] = mx;
                tc_fence_before();
                named_sync_pair(gidx, q4);  // also: both halves have read S, so P may overwrite it
                tc_fence_after();
                mx = fmaxf(xch[gidx][u & 1][0][r], xch[gidx][u & 1][1][r]);
            }
            bool rescale = false;
            float alpha = 1.0f;
            if (mx > -INFINITY) {
                if (!seen) {
                    m_use = mx;  // O and l are still zero
                    seen = true;
                } else if (mx > m_use + 8.0f) {
                    alpha = ex2_approx(m_use - mx);
                    m_use = mx;
                    rescale = true;
                    lh *= alpha;
                }
            }
            if (!ok) continue;
            if (quarter_live) {
                // p = 2^(s sc - m_use), two per packed multiply-add; packed partial sums.
                // P(j) as bf16 pairs over S columns 32 h .. 32 h + 31 of this buffer.
                const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc[2] = {0ull, 0ull};
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint64_t z = f2_fma(f2_pack(sv[hq][e], sv[hq][e + 1]), sc2, nm2);
                        const float p0 = ex2_approx(f2_lo(z));
                        const float p1 = ex2_approx(f2_hi(z));
                        acc[(e >> 1) & 1] = f2_add(acc[(e >> 1) & 1], f2_pack(p0, p1));
                        pk[e >> 1] = pack_bf16(p0, p1);
                    }
                    tmem_st16(s_cols + lane_off + (cb >> 1) + 16 * hq, pk);
                }
                const uint64_t s2 = f2_add(acc[0], acc[1]);
                lh += f2_lo(s2) + f2_hi(s2);
            }
            // O_g is stable: its last update PV(j-2) preceded QK(j) on the tensor
            // pipe, and PV(j) waits for this thread's arrival below. tcgen05.ld/st
            // are warp-collective: rescale if any row of the warp needs it
            // (alpha = 1 for the others).
            if (quarter_live && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    float o[32];
                    tmem_ld32(o_cols + lane_off + cb + 32 * hq, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(o_cols + lane_off + cb + 32 * hq, o);
                }
            }
            // V rows of keys that no row can see may hold anything (even NaN):
            // zero them so that 0 * V stays 0 in the MMA (a V row is two 128-byte
            // halves; thread (row r, column half h) clears half h of row r).
            if (key0 + kBN > nkeys) {
                const int sv_st = jj % kVStages;
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_v_full[sv_st], (jj / kVStages) & 1))) {
                    ok = false;
                    continue;
                }
                if (key0 + r >= nkeys) {
                    uint4* z = reinterpret_cast<uint4*>(smem + kSmemV + sv_st * kTile + ch * kHalf + r * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) z[q] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();  // the MMA reads V through the async proxy
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_p_full[gidx]);
        }
        // both groups' last PV done: O_0 and O_1 final
        const int last0 = (n_local + 1) / 2 - 1, last1 = n_local / 2 - 1;  // group tile counts - 1
        if (ok && last0 >= 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_full[0], last0 & 1));
        if (ok && last1 >= 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_full[1], last1 & 1));
        tc_fence_after();
        if (!ok) raise_status(p.status, kDevTimeout);
        // per-row statistics of both groups
        if (ch == 0) gm[gidx][r] = (seen && quarter_live) ? m_use : -INFINITY;
        gl[gidx][ch][r] = lh;
        named_sync_softmax();
        // ------------------------------------------------------- epilogue ---
        // Every softmax warp now serves output columns 32 cq .. 32 cq + 31 of
        // its lane quarter: O = (2^(m0 - M) O_0 + 2^(m1 - M) O_1) with M the
        // larger reference maximum, l likewise.
        const int cq = (warp - 2) >> 2;  // output column quarter
        const int oc = cq * 32;
        const float m0 = gm[0][r], m1 = gm[1][r];
        const float M = fmaxf(m0, m1);
        const float a0 = m0 > -INFINITY ? ex2_approx(m0 - M) : 0.0f;
        const float a1 = m1 > -INFINITY ? ex2_approx(m1 - M) : 0.0f;
        const float l = a0 * (gl[0][0][r] + gl[0][1][r]) + a1 * (gl[1][0][r] + gl[1][1][r]);
        float o[32];
        // a group that saw no key has weight 0 and its O may be unset: select, not multiply
        if (last0 >= 0) tmem_ld32(tmem_o + lane_off + oc, o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = (last0 >= 0 && a0 > 0.0f) ? a0 * o[e] : 0.0f;
        if (last1 >= 0 && __any_sync(0xffffffffu, a1 > 0.0f)) {
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                float o1[16];
                tmem_ld16(tmem_o + kHD + lane_off + oc + 16 * hq, o1);
#pragma unroll
                for (int e = 0; e < 16; ++e) o[16 * hq + e] += a1 > 0.0f ? a1 * o1[e] : 0.0f;
            }
        }
        const bool row_live = grow < p.G * p.T;
        __nv_bfloat16* orow =
            p.out + ((static_cast<size_t>(b) * p.T + i) * p.Hq + static_cast<size_t>(hk) * p.G + g) * kHD;
        if (nsplit_b == 1) {
            const bool live = row_live && i < n && l > 0.0f && ok;  // rows of unused slots are zeros
            const float inv = live ? 1.0f / l : 0.0f;
            if (row_live) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 uo = make_uint4(0u, 0u, 0u, 0u);
                    if (live)
                        uo = make_uint4(pack_bf16(o[8 * q] * inv, o[8 * q + 1] * inv),
                                        pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                        pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                        pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                    *reinterpret_cast<uint4*>(orow + oc + 8 * q) = uo;
                }
            }
        } else {
            // Split partial: unnormalised O row (float4 q of each 32-column
            // chunk stored at position q ^ (row & 7)), reference max and sum.
            const size_t s0 = static_cast<size_t>(unit) * p.nsplit;
            float* po = p.part_o + ((s0 + split) * kBM + r) * kHD;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4*>(po + oc + ((q ^ (r & 7)) << 2)) =
                    make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            const float m_own = (M > -INFINITY && l > 0.0f) ? M : -INFINITY;
            if (cq == 0) {
                p.part_ml[((s0 + split) * kBM + r) * 2] = m_own;
                p.part_ml[((s0 + split) * kBM + r) * 2 + 1] = l;
            }
            __threadfence();
            named_sync_softmax();
            if (r == 0 && cq == 0) {
                const int prev = atomicAdd(&p.tickets[unit], 1);
                sh_last = prev == nsplit_b - 1;
            }
            named_sync_softmax();
            if (sh_last) {
                // Merge: O = sum_s 2^(m_s - Mx) O_s / sum_s 2^(m_s - Mx) l_s, accumulated
                // in registers; the other splits' partials are bulk-copied into the
                // idle K/V buffers, two per round.
                __threadfence();
                float Mx = -INFINITY;
                for (int s = 0; s < nsplit_b; ++s) Mx = fmaxf(Mx, __ldcg(&p.part_ml[((s0 + s) * kBM + r) * 2]));
                float Ls = 0.0f;
                for (int s = 0; s < nsplit_b; ++s) {
                    const float ms = __ldcg(&p.part_ml[((s0 + s) * kBM + r) * 2]);
                    if (ms > -INFINITY) Ls += __ldcg(&p.part_ml[((s0 + s) * kBM + r) * 2 + 1]) * ex2_approx(ms - Mx);
                }
                const bool live = row_live && i < n && Ls > 0.0f;
                const float inv = live ? 1.0f / Ls : 0.0f;
                const float w_own = m_own > -INFINITY ? ex2_approx(m_own - Mx) * inv : 0.0f;
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = w_own > 0.0f ? o[e] * w_own : 0.0f;
                constexpr int kPart = kBM * kHD * 4;  // 64 KB: one split's partial block
                unsigned char* area = smem + kSmemK;  // 160 KB of K/V stages, idle now
                int round = 0;
                for (int s = 0; s < nsplit_b;) {
                    int lst[2];
                    int cnt = 0;
                    while (s < nsplit_b && cnt < 2) {
                        if (s != split) lst[cnt++] = s;
                        ++s;
                    }
                    if (cnt == 0) break;
                    if (r == 0 && cq == 0) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&bar_comb, cnt * kPart);
                        for (int q = 0; q < cnt; ++q)
                            bulk_g2s(area + q * kPart, p.part_o + (s0 + lst[q]) * kBM * kHD, kPart, &bar_comb);
                    }
                    // on a timeout keep taking part in the named barrier below (no early exit)
                    const bool landed = __all_sync(0xffffffffu, mbar_wait(&bar_comb, round & 1));
                    if (!landed) raise_status(p.status, kDevTimeout);
                    for (int q = 0; landed && q < cnt; ++q) {
                        const float ms = __ldcg(&p.part_ml[((s0 + lst[q]) * kBM + r) * 2]);
                        const float wq = ms > -INFINITY ? ex2_approx(ms - Mx) * inv : 0.0f;
                        if (wq == 0.0f) continue;
                        const float* rowp = reinterpret_cast<const float*>(area + q * kPart) + r * kHD + oc;
#pragma unroll
                        for (int q4b = 0; q4b < 8; ++q4b) {
                            const float4 v = *reinterpret_cast<const float4*>(rowp + ((q4b ^ (r & 7)) << 2));
                            o[4 * q4b] += wq * v.x;
                            o[4 * q4b + 1] += wq * v.y;
                            o[4 * q4b + 2] += wq * v.z;
                            o[4 * q4b + 3] += wq * v.w;
                        }
                    }
                    named_sync_softmax();  // every row has read the slots before they are refilled
                    ++round;
                }
                if (row_live) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 uo = make_uint4(0u, 0u, 0u, 0u);
                        if (live)
                            uo = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                                            pack_bf16(o[8 * q + 4], o[8 * q + 5]),
                                            pack_bf16(o[8 * q + 6], o[8 * q + 7]));
                        *reinterpret_cast<uint4*>(orow + oc + 8 * q) = uo;
                    }
                }
                if (r == 0 && cq == 0) p.tickets[unit] = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------- host side ---

struct Plan {
    int G, n_rb, nsplit, tps, units;
    double cost;  // the cost model's estimate, in 128-key tile times of one SM
    size_t off_tickets, off_ml, off_o, bytes;
};

Plan make_plan(const KvDims& kv, int T) {
    Plan pl{};
    pl.G = kv.Hq / kv.Hkv;
    const int rows = pl.G * T;
    pl.n_rb = (rows + kBM - 1) / kBM;
    pl.units = kv.B * kv.Hkv * pl.n_rb;
    const int max_tiles = (kv.max_len + kBN - 1) / kBN;
    // Keys of a unit may be split over CTAs (one CTA per SM). Cost model, in
    // tile times: waves of CTAs x (tiles per CTA + a fixed eight for the
    // prologue, epilogue and partial store of a CTA) + 1.5 per extra split
    // (the merge). Fitted on GB300: 70B b8 best at 3-4 splits (6 before),
    // 8B b1 at 3-4, 8B b64 at 1.
    const int sms = 152;
    int nsplit = 1;
    double best = 1e30;
    for (int ns = 1; ns <= std::max(1, max_tiles / 2); ++ns) {
        const int tps = (max_tiles + ns - 1) / ns;
        const double waves = std::ceil(static_cast<double>(pl.units) * ns / sms);
        const double cost = waves * (tps + 8.0) + 1.5 * (ns - 1);
        if (cost < best - 1e-9) {
            best = cost;
            nsplit = ns;
        }
    }
    pl.tps = (max_tiles + nsplit - 1) / nsplit;
    pl.nsplit = (max_tiles + pl.tps - 1) / pl.tps;
    pl.cost = best;
    pl.off_tickets = 256;
    pl.off_ml = align_up(pl.off_tickets + static_cast<size_t>(pl.units) * sizeof(int), 256);
    const size_t slots = pl.nsplit > 1 ? static_cast<size_t>(pl.units) * pl.nsplit : 0;
    pl.off_o = align_up(pl.off_ml + slots * kBM * 2 * sizeof(float), 256);
    pl.bytes = align_up(pl.off_o + slots * kBM * kHD * sizeof(float), 256);
    return pl;
}

bool tc_supported(const KvDims& kv, int T) {
    const int G = kv.Hq / kv.Hkv;
    return kv.dtype == 1 && kv.d == kHD && G >= 1 && G <= kBM && (kBM % G) == 0 && T <= kMaxSlots &&
           (kv.pos_stride * 2) % 16 == 0 && (kv.seq_stride * 2) % 16 == 0 && (kv.layer_stride * 2) % 16 == 0 &&
           (kv.kv_stride * 2) % 16 == 0;
}

// The persistent pipeline (k_attn_pipe.cu) when its estimated time is the
// lower one. Both estimates take every unit at the longest length; measured
// on GB300 at 8B b64: about 1.15 us per 128-key tile of a CTA here, 1.1 us
// per 64-key tile of each of the pipeline's two CTAs per SM, whose items are
// never split (so a few very long ones leave SMs idle: 70B b8).
bool use_pipeline(const KvDims& kv, int T) {
    if (!attention_pipe_fits(kv, T)) return false;
    const Plan pl = make_plan(kv, T);
    const int tiles64 = (kv.max_len + 63) / 64;
    const double pipe_us = std::ceil(static_cast<double>(pl.units) / (2.0 * 152)) * (tiles64 + 4.0) * 1.1;
    return pipe_us < pl.cost * 1.15;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

size_t attention_ws_bytes(const KvDims& kv, int T) {
    if (!tc_supported(kv, T) || use_pipeline(kv, T)) return 256;
    return make_plan(kv, T).bytes;
}

cudaError_t launch_attention(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                             const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                             void* ws, size_t ws_bytes, int* status, cudaStream_t stream) {
    if (!tc_supported(kv, T))
        return launch_attention_simt(kv, T, q, cache, layer, prefix_len, mask, n_tree, out, status, stream);
    // many (sequence, KV head, row block) items of moderate length: the
    // persistent pipeline (k_attn_pipe.cu); else one CTA per item and key
    // split, two softmax groups each
    if (use_pipeline(kv, T))
        return launch_attention_pipe(kv, T, q, cache, layer, prefix_len, mask, n_tree, out, status, stream);
    const Plan pl = make_plan(kv, T);
    if (ws_bytes < pl.bytes) return cudaErrorInvalidValue;
    char* w = static_cast<char*>(ws);
    const char* kbase = static_cast<const char*>(cache) + static_cast<int64_t>(layer) * kv.layer_stride * 2;
    const char* vbase = kbase + kv.kv_stride * 2;
    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(kv.Hq),
                                    static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(kv.B)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHD) * 2, static_cast<cuuint64_t>(kv.Hq) * kHD * 2,
                                       static_cast<cuuint64_t>(T) * kv.Hq * kHD * 2};
        const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(pl.G), static_cast<cuuint32_t>(kBM / pl.G), 1};
        if (!make_map_bf16_4d(&tq, q, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(kv.Hkv),
                                    static_cast<cuuint64_t>(kv.max_len), static_cast<cuuint64_t>(kv.B)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHD) * 2, static_cast<cuuint64_t>(kv.pos_stride) * 2,
                                       static_cast<cuuint64_t>(kv.seq_stride) * 2};
        const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kBN), 1};
        if (!make_map_bf16_4d(&tk, kbase, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_map_bf16_4d(&tv, vbase, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams prm{};
    prm.B = kv.B;
    prm.T = T;
    prm.Hq = kv.Hq;
    prm.Hkv = kv.Hkv;
    prm.G = pl.G;
    prm.n_rb = pl.n_rb;
    prm.nsplit = pl.nsplit;
    prm.tps = pl.tps;
    prm.max_len = kv.max_len;
    prm.W = (T + 31) / 32;
    prm.prefix_len = prefix_len;
    prm.mask = mask;
    prm.n_tree = n_tree;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.tickets = reinterpret_cast<int*>(w + pl.off_tickets);
    prm.part_ml = reinterpret_cast<float*>(w + pl.off_ml);
    prm.part_o = reinterpret_cast<float*>(w + pl.off_o);
    prm.status = status;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHD)));
    if (pl.nsplit > 1) {
        cudaError_t e = cudaMemsetAsync(prm.tickets, 0, static_cast<size_t>(pl.units) * sizeof(int), stream);
        if (e != cudaSuccess) return e;
    }
    cudaError_t ae = ensure_dyn_smem(reinterpret_cast<const void*>(attn_tc_kernel), kSmemBytes + 1024);
    if (ae != cudaSuccess) return ae;
    dim3 grid(pl.n_rb, pl.nsplit, kv.B * kv.Hkv);
    return launch_pdl(attn_tc_kernel, grid, dim3(kThreads), kSmemBytes + 1024, stream, tq, tk, tv, prm);
}

}  // namespace eagle

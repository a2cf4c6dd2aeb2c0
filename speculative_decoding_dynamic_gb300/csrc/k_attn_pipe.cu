// Stage 5, tensor-core path (sm_103a): tree-masked GQA attention.
//
// For sequence b, KV head hk, the G = Hq/Hkv query heads of every tree slot
// form M = G*T query rows (row r <-> slot r / G, head hk*G + r % G, matching
// the [B, T, Hq, d] layout of Q). A work item is a 128-row block of them
// with all of the sequence's keys (prefix [0, L_b) then the tree slots at
// L_b + j) in tiles of 64. This kernel serves shapes whose items fill two
// CTAs per SM without splitting keys (k_attn_tc.cu picks it); it is
// persistent, two CTAs per SM, each walking a list of items (longest
// first); per CTA and key tile j:
//   S = Q K^T        tcgen05.mma kind::f16, bf16 operands from shared memory,
//                    fp32 accumulator in tensor memory, double buffered
//                    (TMEM columns 64 (j & 1) ..), so QK^T of tile j+1 runs
//                    while the softmax works on tile j
//   P = softmax part eight warps, two threads per row (TMEM lane = row, 32
//                    key columns each; row maxima exchanged in shared
//                    memory): scale, tree mask, exponentials in the log2
//                    domain against a reference maximum, P written as bf16
//                    pairs into tensor memory over the S buffer it came from
//   O += P V         tcgen05.mma with A = P read from tensor memory, V from
//                    shared memory (MN-major), accumulating in TMEM columns
//                    128..255; the reference maximum is raised (O and the
//                    row sum rescaled in place) only when a tile's maximum
//                    exceeds it by more than 2^8, so exponentials stay below 256
// One softmax group per CTA processes the tiles back to back; the second CTA
// on the SM fills the tensor pipe while this one is in its epilogue or waits.
// K and V tiles arrive by TMA (cp.async.bulk.tensor, 128B swizzle) into
// their own rings (a K stage frees after QK^T, a V stage after PV), Q once
// per item; three lanes of warp 0 issue them, one thread of warp 1 every MMA;
// mbarriers order them, their phases run on across items, and every wait is
// bounded.
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
namespace {

constexpr int kBM = 128;                   // query rows per item (one MMA M)
constexpr int kBN = 64;                    // keys per tile (MMA N of QK^T, K of PV)
constexpr int kHD = 128;                   // head dim (MMA K of QK^T, N of PV)
constexpr int kTileQ = kBM * kHD * 2;      // 32 KB: Q of an item
constexpr int kHalfQ = kTileQ / 2;         // 16 KB: 128 rows x 64 columns (one swizzle-128B column block)
constexpr int kTileKV = kBN * kHD * 2;     // 16 KB: a K or V tile
constexpr int kHalfKV = kTileKV / 2;       // 8 KB: 64 keys x 64 columns
constexpr int kKStages = 2;  // K tiles in flight (a stage frees after QK^T)
constexpr int kVStages = 2;  // V tiles in flight (a stage frees after PV)
constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = 64 + kSoftmaxThreads;  // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int kCtasPerSm = 2;
constexpr int kSmemQ = 0;
constexpr int kSmemK = kTileQ;                       // K stage s at kSmemK + s * kTileKV
constexpr int kSmemV = kSmemK + kKStages * kTileKV;  // V stage s at kSmemV + s * kTileKV
constexpr int kSmemBytes = kSmemV + kVStages * kTileKV;  // 96 KB
constexpr int kTmemCols = 256;  // S double buffer (2 x 64 columns; P over S), O (128)
constexpr uint32_t kTmemO = 128;
constexpr int kMaxW = kMaxSlots / 32;
constexpr int kSms = 152;

struct PipeParams {
    int B, T, Hq, Hkv, G, n_rb, max_len, W;
    int n_items;  // B * Hkv * n_rb
    const int32_t* prefix_len;
    const uint32_t* mask;
    const int32_t* n_tree;
    __nv_bfloat16* out;
    int* status;
    float scale_log2;
};

// ---------------------------------------------------------------- PTX ---
// TMA, tcgen05 MMA and tensor-memory helpers: tc_ptx.cuh.

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory"); }
// The two warps that serve one TMEM lane quarter (the rows 32 q4 ..
// 32 q4 + 31, one warp per column half) meet on barrier 2 + q4.
__device__ __forceinline__ void named_sync_pair(int q4) { asm volatile("bar.sync %0, 64;" ::"r"(2 + q4) : "memory"); }

// One work item: row block rb of (sequence b, KV head hk), key tiles
// [0, n_local) (0 when the sequence's lengths are out of range).
struct Item {
    int b, hk, rb, L, n, nkeys, n_local;
};

struct Order {
    int seq[kPipeMaxSeqs];  // sequence at each sorted position
    int L[kPipeMaxSeqs];    // its prefix length and tree size
    int n[kPipeMaxSeqs];
};

__device__ __forceinline__ void seq_range(const PipeParams& p, int L, int n, Item& it) {
    it.L = L;
    it.n = n;
    const bool bad = L < 0 || L + p.T > p.max_len || n < 1 || n > p.T;
    it.nkeys = bad ? 0 : L + n;
    it.n_local = (it.nkeys + kBN - 1) / kBN;
}

// Item at sorted position pos: sequences longest first, within a sequence
// KV head then row block (the row blocks of one head read the same K/V
// tiles and sit at neighbouring positions, so they run at about the same
// time).
__device__ __forceinline__ Item item_at(const PipeParams& p, const Order& ord, int pos) {
    const int per_seq = p.Hkv * p.n_rb;
    const int sp = pos / per_seq, rem = pos - sp * per_seq;
    Item it;
    it.b = ord.seq[sp];
    it.hk = rem / p.n_rb;
    it.rb = rem - it.hk * p.n_rb;
    seq_range(p, ord.L[sp], ord.n[sp], it);
    return it;
}

// Sorted position of this CTA's r-th item (snake order over the CTAs).
__device__ __forceinline__ int item_pos(int r) {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// ------------------------------------------------------------- kernel ---

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    attn_pipe_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, PipeParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_q, bar_q_empty, bar_k_full[kKStages], bar_k_empty[kKStages], bar_v_full[kVStages],
        bar_v_empty[kVStages], bar_s_full[2], bar_p_full[2], bar_pv_done, bar_o_full, bar_o_free;
    __shared__ uint32_t tmem_holder;
    __shared__ Order ord;
    __shared__ float xch[2][2][kBM];             // [tile parity][column half][row]: per-tile row maxima
    __shared__ float lsum[2][2][kBM];            // [item parity][column half][row]: row sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        mbar_init(&bar_q_empty, 1);
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
            mbar_init(&bar_p_full[s], kSoftmaxThreads);
        }
        mbar_init(&bar_pv_done, 1);
        mbar_init(&bar_o_full, 1);
        mbar_init(&bar_o_free, kSoftmaxThreads);
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Q and the first K/V tiles of this CTA's item in natural order into L2
    // while the previous kernel finishes (hints only: the item actually taken
    // depends on the lengths, and every item's tiles are read by some CTA)
    if (warp == 0 && lane < 2 && static_cast<int>(blockIdx.x) < p.n_items) {
        const int per_seq = p.Hkv * p.n_rb;
        const int b = blockIdx.x / per_seq, rem = blockIdx.x - b * per_seq;
        const int hk = rem / p.n_rb, rb = rem - hk * p.n_rb;
        const int key0 = 0;
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
    // Sequences ordered by key tiles, most first (equal: lower sequence
    // first): rank by counting.
    {
        int* keys = reinterpret_cast<int*>(smem + kSmemK);  // K stages are idle until the loads start
        for (int b = threadIdx.x; b < p.B; b += kThreads) {
            Item it;
            seq_range(p, __ldcg(&p.prefix_len[b]), __ldcg(&p.n_tree[b]), it);
            keys[b] = it.n_local;
            if (it.nkeys == 0 && blockIdx.x == 0) raise_status(p.status, kDevBadIndex);
        }
        __syncthreads();
        for (int b = threadIdx.x; b < p.B; b += kThreads) {
            const int kb = keys[b];
            int rank = 0;
            for (int o = 0; o < p.B; ++o) {
                const int ko = keys[o];
                rank += (ko > kb || (ko == kb && o < b)) ? 1 : 0;
            }
            ord.seq[rank] = b;
            ord.L[rank] = __ldcg(&p.prefix_len[b]);
            ord.n[rank] = __ldcg(&p.n_tree[b]);
        }
        fence_proxy_async_smem();  // TMA overwrites the keys' stage later
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;
    const uint32_t tmem_s = tmem;           // S(j) at tmem_s + 64 (j & 1); P(j) over its first 32 columns
    const uint32_t tmem_o = tmem + kTmemO;  // O
    const int n_items = p.n_items;

    unsigned char* sQ = smem + kSmemQ;
    // [item parity][row][W]: mask words of each row's tree slot
    uint32_t* mask_sm = reinterpret_cast<uint32_t*>(smem + kSmemBytes);

    if (warp == 0) {
        // ------------------------------------------------ TMA producers ---
        // Lane 0 loads the K tiles, lane 1 the V tiles, lane 2 Q: a K stage
        // is free once QK^T of its tile is done, a V stage once PV is, and Q
        // once QK^T of the item's last tile is done, so no stream waits
        // behind another.
        if (lane == 2) {
            int qi = 0;
            bool ok = true;
            for (int r = 0;; ++r) {
                const int pos = item_pos(r);
                if (pos >= n_items) break;
                const Item it = item_at(p, ord, pos);
                if (it.n_local == 0) continue;
                if (qi > 0 && !mbar_wait_sleep(&bar_q_empty, (qi - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int i0 = it.rb * (kBM / p.G);
                mbar_arrive_expect_tx(&bar_q, kTileQ);
                tma_load_4d(sQ, &tm_q, 0, it.hk * p.G, i0, it.b, &bar_q);
                tma_load_4d(sQ + kHalfQ, &tm_q, 64, it.hk * p.G, i0, it.b, &bar_q);
                ++qi;
                // the next item's Q into L2 while this item streams
                for (int r2 = r + 1;; ++r2) {
                    const int pos2 = item_pos(r2);
                    if (pos2 >= n_items) break;
                    const Item nx = item_at(p, ord, pos2);
                    if (nx.n_local == 0) continue;
                    tma_prefetch_4d(&tm_q, 0, nx.hk * p.G, nx.rb * (kBM / p.G), nx.b);
                    tma_prefetch_4d(&tm_q, 64, nx.hk * p.G, nx.rb * (kBM / p.G), nx.b);
                    break;
                }
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        } else if (lane < 2) {
            const bool is_k = lane == 0;
            uint64_t* full = is_k ? bar_k_full : bar_v_full;
            uint64_t* empty = is_k ? bar_k_empty : bar_v_empty;
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            const int ns = is_k ? kKStages : kVStages;
            int t = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int pos = item_pos(r);
                if (pos >= n_items) break;
                const Item it = item_at(p, ord, pos);
                if (it.n_local == 0) continue;
                for (int jj = 0; jj < it.n_local; ++jj, ++t) {
                    const int st = t % ns;
                    if (t >= ns && !mbar_wait_sleep(&empty[st], ((t / ns) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    unsigned char* dst = smem + (is_k ? kSmemK : kSmemV) + st * kTileKV;
                    const int key0 = jj * kBN;
                    mbar_arrive_expect_tx(&full[st], kTileKV);
                    tma_load_4d(dst, map, 0, it.hk, key0, it.b, &full[st]);
                    tma_load_4d(dst + kHalfKV, map, 64, it.hk, key0, it.b, &full[st]);
                }
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer ---
        // Tiles are numbered t over all of the CTA's items. QK(t) goes into S
        // buffer t & 1, whose previous content P(t-2) was read by PV(t-2),
        // issued earlier (tcgen05.mma of one thread execute in issue order).
        // Issue order QK(0) QK(1) PV(0) QK(2) PV(1) ...: QK^T of the next
        // tile runs while the softmax works on the current one. An item's
        // first PV overwrites O, so it waits until the previous item's
        // epilogue has read O out of tensor memory.
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(kBM, kBN, 0);
            constexpr uint32_t id_pv = idesc_bf16(kBM, kHD, 1);
            const uint32_t aQ = smem_u32(sQ);
            int t = 0, qi = 0;
            bool ok = true;
            auto issue_pv = [&](int tp, bool first, bool last) -> bool {
                const int sb = tp & 1, sv = tp % kVStages;
                if (!mbar_wait_sleep(&bar_p_full[sb], (tp >> 1) & 1)) return false;
                if (first && qi > 0 && !mbar_wait_sleep(&bar_o_free, (qi - 1) & 1)) return false;
                if (!mbar_wait_sleep(&bar_v_full[sv], (tp / kVStages) & 1)) return false;
                tc_fence_after();
                const uint32_t aV = smem_u32(smem + kSmemV + sv * kTileKV);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)  // A = P from TMEM: 16 keys = 8 columns per MMA
                    mma_bf16_ts(tmem_o, tmem_s + sb * kBN + kk * 8, smem_desc(aV + kk * 2048, kHalfKV, 1024), id_pv,
                                (!first || kk > 0) ? 1 : 0);
                mma_commit(&bar_v_empty[sv]);
                mma_commit(&bar_pv_done);
                if (last) mma_commit(&bar_o_full);
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int pos = item_pos(r);
                if (pos >= n_items) break;
                const Item it = item_at(p, ord, pos);
                if (it.n_local == 0) continue;
                if (!mbar_wait_sleep(&bar_q, qi & 1)) {
                    ok = false;
                    break;
                }
                for (int jj = 0; ok && jj < it.n_local; ++jj, ++t) {
                    const int sb = t & 1, sk = t % kKStages;
                    ok = mbar_wait_sleep(&bar_k_full[sk], (t / kKStages) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t aK = smem_u32(smem + kSmemK + sk * kTileKV);
#pragma unroll
                    for (int kk = 0; kk < kHD / 16; ++kk)
                        mma_bf16(tmem_s + sb * kBN, smem_desc(aQ + (kk >> 2) * kHalfQ + (kk & 3) * 32, 16, 1024),
                                 smem_desc(aK + (kk >> 2) * kHalfKV + (kk & 3) * 32, 16, 1024), id_qk, kk > 0);
                    mma_commit(&bar_k_empty[sk]);
                    mma_commit(&bar_s_full[sb]);
                    if (jj == it.n_local - 1) mma_commit(&bar_q_empty);
                    if (jj > 0) ok = issue_pv(t - 1, jj == 1, false);
                }
                if (ok) ok = issue_pv(t - 1, it.n_local == 1, true);
                ++qi;
            }
            if (!ok) raise_status(p.status, kDevTimeout);
        }
    } else {
        // ------------------------------------------------------ softmax ---
        // Warp w serves TMEM lane quarter w % 4 (rows 32 q4 ..) and key
        // columns 32 h .. 32 h + 31 of each tile, h the warp's column half;
        // the two threads of a row exchange row maxima through shared
        // memory. The exponentials use a reference maximum m_use raised (O,
        // l rescaled) only when a tile's maximum exceeds it by more than 2^8.
        const int h = (warp - 2) >> 2;        // column half
        const int q4 = warp & 3;
        const int r = (q4 << 5) | lane;       // row of the block = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const float sc = p.scale_log2;
        int t = 0;   // tiles so far (S, P phases)
        int qi = 0;  // items with tiles so far (O phases, mask and sum parity)
        bool ok = true;
        // Mask rows of an item's tree slots: the four warps of column half 0
        // copy them into mask_sm[item parity]; the first item's before the
        // loop, each next item's while the current item's last PV runs
        // (published by the barrier of the current item's epilogue).
        auto next_with_tiles = [&](int r0) -> int {
            for (int r2 = r0;; ++r2) {
                const int pos2 = item_pos(r2);
                if (pos2 >= n_items) return -1;
                if (item_at(p, ord, pos2).n_local > 0) return pos2;
            }
        };
        auto load_mask = [&](int pos2, int buf) {
            const Item nx = item_at(p, ord, pos2);
            const int i = nx.rb * (kBM / p.G) + r / p.G;
            uint32_t w4[kMaxW];
#pragma unroll
            for (int w = 0; w < kMaxW; ++w)
                w4[w] = (w < p.W && i < p.T) ? __ldcg(&p.mask[(static_cast<size_t>(nx.b) * p.T + i) * p.W + w]) : 0u;
#pragma unroll
            for (int w = 0; w < kMaxW; ++w)
                if (w < p.W) mask_sm[(buf * kBM + r) * p.W + w] = w4[w];
        };
        if (h == 0) {
            const int f = next_with_tiles(0);
            if (f >= 0) load_mask(f, 0);
        }
        named_sync_softmax();
        for (int rr = 0;; ++rr) {
            const int pos = item_pos(rr);
            if (pos >= n_items) break;
            const Item it = item_at(p, ord, pos);
            if (it.n_local == 0) {  // a sequence whose lengths are out of range: zero rows
                const int i = it.rb * (kBM / p.G) + r / p.G;
                __nv_bfloat16* orow = p.out + ((static_cast<size_t>(it.b) * p.T + i) * p.Hq +
                                               static_cast<size_t>(it.hk) * p.G + r % p.G) * kHD;
                if (it.rb * kBM + r < p.G * p.T)
#pragma unroll
                    for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(orow + 64 * h + 8 * q) = make_uint4(0, 0, 0, 0);
                continue;
            }
            // a lane quarter whose 32 rows are all past the problem's rows does no
            // arithmetic (it still takes part in every barrier and V clearing)
            const bool quarter_live = it.rb * kBM + q4 * 32 < p.G * p.T;
            const uint32_t* mrow = mask_sm + ((qi & 1) * kBM + r) * p.W;
            const int L = it.L, n = it.n, nkeys = it.nkeys;
            float m_use = 0.0f, lh = 0.0f;  // lh: this half's share of the row sum
            bool seen = false;
            for (int jj = 0; jj < it.n_local; ++jj, ++t) {
                const int sb = t & 1;
                const int key0 = jj * kBN;
                const uint32_t s_cols = tmem_s + sb * kBN;
                // After a timed-out wait a warp skips the work of the remaining tiles
                // but still takes every named barrier, so the others never wait for
                // it without bound.
                if (ok && !__all_sync(0xffffffffu, mbar_wait_sleep(&bar_s_full[sb], (t >> 1) & 1))) ok = false;
                tc_fence_after();
                float sv[32];
                if (ok && quarter_live) {
                    tmem_ld32(s_cols + lane_off + 32 * h, sv);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[e] = -INFINITY;
                }
                // visibility of the half's 32 keys: prefix keys, then tree slots in mask row i
                {
                    const int kb = key0 + 32 * h;
                    const int npre = L - kb;  // keys of the 32 inside the prefix
                    if (npre < 32) {
                        const uint32_t pre = npre > 0 ? (1u << npre) - 1u : 0u;
                        const int j0 = kb - L;  // slot of the first key (may be negative)
                        const int lo = j0 < 0 ? 0 : j0;
                        const int w0 = lo >> 5, sh = lo & 31;
                        uint32_t win = w0 < p.W ? mrow[w0] >> sh : 0u;
                        if (sh && w0 + 1 < p.W) win |= mrow[w0 + 1] << (32 - sh);
                        const int limit = n - lo;  // slots j >= n are never visible
                        if (limit <= 0) win = 0u;
                        else if (limit < 32) win &= (1u << limit) - 1u;
                        uint32_t tree = j0 < 0 ? (win << (-j0)) : win;
                        if (j0 <= -32) tree = 0u;
                        const uint32_t vis = pre | tree;
#pragma unroll
                        for (int e = 0; e < 32; ++e) sv[e] = ((vis >> e) & 1u) ? sv[e] : -INFINITY;
                    }
                }
                float mx = max32(sv) * sc;  // the scale is positive
                if (quarter_live) {
                    xch[t & 1][h][r] = mx;
                    tc_fence_before();
                    named_sync_pair(q4);  // also: both halves have read S, so P may overwrite it
                    tc_fence_after();
                    mx = fmaxf(xch[t & 1][0][r], xch[t & 1][1][r]);
                }
                bool rescale = false;
                float alpha = 1.0f;
                if (mx > -INFINITY) {
                    if (!seen) {
                        m_use = mx;  // O and l are still zero for this item
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
                    // P(t) as bf16 pairs over S columns 16 h .. 16 h + 15 of this buffer.
                    const uint64_t sc2 = f2_pack(sc, sc), nm2 = f2_pack(-m_use, -m_use);
                    uint64_t acc[2] = {0ull, 0ull};
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint64_t z = f2_fma(f2_pack(sv[e], sv[e + 1]), sc2, nm2);
                        const float p0 = ex2_approx(f2_lo(z));
                        const float p1 = ex2_approx(f2_hi(z));
                        acc[(e >> 1) & 1] = f2_add(acc[(e >> 1) & 1], f2_pack(p0, p1));
                        pk[e >> 1] = pack_bf16(p0, p1);
                    }
                    tmem_st16(s_cols + lane_off + 16 * h, pk);
                    const uint64_t s2 = f2_add(acc[0], acc[1]);
                    lh += f2_lo(s2) + f2_hi(s2);
                }
                // Rescaling O needs PV(t-1) done (it may still run: PV(t-1) is
                // issued after QK(t)); PV(t) waits for this thread's arrival
                // below. tcgen05.ld/st are warp-collective: rescale if any row
                // of the warp needs it (alpha = 1 for the others).
                if (quarter_live && __any_sync(0xffffffffu, rescale)) {
                    if (!__all_sync(0xffffffffu, mbar_wait_sleep(&bar_pv_done, (t - 1) & 1))) {
                        ok = false;
                    } else {
                        tc_fence_after();
#pragma unroll
                        for (int hq = 0; hq < 2; ++hq) {
                            float o[32];
                            tmem_ld32(tmem_o + lane_off + 64 * h + 32 * hq, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= alpha;
                            tmem_st32(tmem_o + lane_off + 64 * h + 32 * hq, o);
                        }
                    }
                }
                // V rows of keys that no row can see may hold anything (even NaN):
                // zero them so that 0 * V stays 0 in the MMA (a V row is two 128-byte
                // halves; thread (row r < 64, column half h) clears half h of row r).
                if (key0 + kBN > nkeys) {
                    const int sv_st = t % kVStages;
                    if (!__all_sync(0xffffffffu, mbar_wait(&bar_v_full[sv_st], (t / kVStages) & 1))) {
                        ok = false;
                        continue;
                    }
                    if (r < kBN && key0 + r >= nkeys) {
                        uint4* z = reinterpret_cast<uint4*>(smem + kSmemV + sv_st * kTileKV + h * kHalfKV + r * 128);
#pragma unroll
                        for (int q = 0; q < 8; ++q) z[q] = make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();  // the MMA reads V through the async proxy
                    }
                }
                tc_fence_before();
                mbar_arrive(&bar_p_full[sb]);
            }
            if (h == 0) {  // the next item's mask rows (other parity: nobody reads them now)
                const int f = next_with_tiles(rr + 1);
                if (f >= 0) load_mask(f, (qi + 1) & 1);
            }
            // the item's last PV done: O final
            if (ok && !__all_sync(0xffffffffu, mbar_wait_sleep(&bar_o_full, qi & 1))) ok = false;
            if (!ok) raise_status(p.status, kDevTimeout);
            // ----------------------------------------------------- epilogue ---
            // Thread (row r, half h) owns output columns 64 h .. 64 h + 63 of its row.
            const int pb = qi & 1;
            lsum[pb][h][r] = lh;
            tc_fence_before();
            named_sync_softmax();  // row sums of both halves; the next item's mask published
            tc_fence_after();
            const float l = lsum[pb][0][r] + lsum[pb][1][r];
            uint32_t ov[64];
            tmem_ld64(tmem_o + lane_off + 64 * h, ov);
            tc_fence_before();
            mbar_arrive(&bar_o_free);
            ++qi;
            const int i = it.rb * (kBM / p.G) + r / p.G;  // tree slot of the row
            const bool row_live = it.rb * kBM + r < p.G * p.T;
            __nv_bfloat16* orow = p.out + ((static_cast<size_t>(it.b) * p.T + i) * p.Hq +
                                           static_cast<size_t>(it.hk) * p.G + r % p.G) * kHD + 64 * h;
            const bool live = row_live && i < n && seen && quarter_live && l > 0.0f && ok;  // unused slots: zeros
            const float inv = live ? 1.0f / l : 0.0f;
            if (row_live) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint4 uo = make_uint4(0u, 0u, 0u, 0u);
                    if (live)
                        uo = make_uint4(
                            pack_bf16(__uint_as_float(ov[8 * q]) * inv, __uint_as_float(ov[8 * q + 1]) * inv),
                            pack_bf16(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv),
                            pack_bf16(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv),
                            pack_bf16(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv));
                    *reinterpret_cast<uint4*>(orow + 8 * q) = uo;
                }
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

}  // namespace

bool attention_pipe_fits(const KvDims& kv, int T) {
    const int G = kv.Hq / kv.Hkv;
    const int rows = G * T;
    const int n_rb = (rows + kBM - 1) / kBM;
    const long long items = static_cast<long long>(kv.B) * kv.Hkv * n_rb;
    return kv.B <= kPipeMaxSeqs && items >= static_cast<long long>(kSms) * kCtasPerSm;
}

cudaError_t launch_attention_pipe(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream) {
    const int G = kv.Hq / kv.Hkv;
    const char* kbase = static_cast<const char*>(cache) + static_cast<int64_t>(layer) * kv.layer_stride * 2;
    const char* vbase = kbase + kv.kv_stride * 2;
    CUtensorMap tq, tk, tv;
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(kv.Hq),
                                    static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(kv.B)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHD) * 2, static_cast<cuuint64_t>(kv.Hq) * kHD * 2,
                                       static_cast<cuuint64_t>(T) * kv.Hq * kHD * 2};
        const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kBM / G), 1};
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
    PipeParams prm{};
    prm.B = kv.B;
    prm.T = T;
    prm.Hq = kv.Hq;
    prm.Hkv = kv.Hkv;
    prm.G = G;
    prm.n_rb = (G * T + kBM - 1) / kBM;
    prm.max_len = kv.max_len;
    prm.W = (T + 31) / 32;
    prm.n_items = kv.B * kv.Hkv * prm.n_rb;
    prm.prefix_len = prefix_len;
    prm.mask = mask;
    prm.n_tree = n_tree;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.status = status;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHD)));
    const int dyn = kSmemBytes + 2 * kBM * prm.W * 4 + 1024;  // stages, mask rows, alignment slack
    cudaError_t ae = ensure_dyn_smem(reinterpret_cast<const void*>(attn_pipe_kernel), dyn);
    if (ae != cudaSuccess) return ae;
    // two CTAs per SM need the largest shared-memory carveout
    static std::once_flag carve;
    std::call_once(carve, [] {
        cudaFuncSetAttribute(reinterpret_cast<const void*>(attn_pipe_kernel),
                             cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    });
    dim3 grid(std::min(prm.n_items, kSms * kCtasPerSm));
    return launch_pdl(attn_pipe_kernel, grid, dim3(kThreads), dyn, stream, tq, tk, tv, prm);
}

}  // namespace eagle

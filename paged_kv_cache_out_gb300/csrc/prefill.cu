// prefill.cu -- ragged causal prefill attention over a paged KV cache, with
// the QK^T and PV contractions on the tcgen05 tensor cores.
//
// miniVLLM "Engine Architecture", prepare_prefill: the new tokens of every
// request are concatenated (the num_cached_tokens prefix of each sequence is
// skipped) with cumulative offsets cu_seqlens_q; slot_mapping and
// block_tables address the paged pool.  New token i of request r sits at
// absolute position c_r + i (c_r = cached prefix) and attends to keys
// 0 .. c_r + i (causal, aligned at the bottom right).  Grouped-query
// attention shares one KV head among num_q_heads / num_kv_heads query heads.
//
// Work item: two 128-row query tiles, A and B, of one request and one KV
// head; a tile holds 128/G consecutive new tokens x the G query heads of that
// KV head, so every K/V tile staged in shared memory serves 2 x 128 rows.
// The kernel is persistent: one block per SM takes items in order of
// decreasing work, heaviest first (its first item by block index, the rest
// from a queue counter in the caller's workspace), so the last items to
// finish are light ones, and the next item's Q and first K/V tiles load while
// the current item finishes.  Roles (384 threads):
//   warp 8      producer: takes the next item and publishes it to the other
//               roles through a 2-slot ring, and loads the Q tiles A and B.
//   warps 8, 10, 11  loaders: 128-key K and V tiles through a 2-stage K ring
//               and a 3-stage V ring, K one tile ahead of V, each warp
//               copying its share of a tile's pages.  Pages of >= 8 tokens
//               come in as TMA boxes (one per page and 64-column block,
//               128-byte swizzle, straight into the layout the tensor core
//               reads); smaller pages are gathered by the lanes with 16-byte
//               loads and swizzled stores.  Page ids are read in warp-wide
//               windows, one window ahead.
//   warp 9      allocates all 512 TMEM columns (per query tile: a 128x128
//               fp32 score buffer S, whose first 64 columns then hold P as
//               bf16 pairs, and a 128 x head_dim fp32 output accumulator O)
//               and one of its lanes issues every MMA of both tiles, in this
//               order per key tile j:
//                 O_A += P_A(j) V_j,  S_A(j+1) = Q_A K_(j+1)^T,
//                 O_B += P_B(j) V_j,  S_B(j+1) = Q_B K_(j+1)^T,
//               with S from Q and K in shared memory (M=128, N=128,
//               K=head_dim) and PV reading P from tensor memory and V from
//               shared memory (M=128, N=head_dim, K=128).  The tensor core
//               runs one thread's MMAs in order, so the commit of S(j+1) also
//               tells that PV(j) has read P(j) and written O.  (A single
//               issuing thread keeps the tensor core at its full rate; two
//               threads issuing at the same time slow each other down.)
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: thread i of a
//               warpgroup owns row i (TMEM lane i): reads its scores, applies
//               the causal mask by selection, keeps a running max and sum in
//               the log2 domain, rescales its TMEM output row when the running
//               max grew by more than 2^8 (exact: every term shares the
//               reference), writes P into tensor memory, and at the end of the
//               item reads O out of tensor memory (then frees it for the next
//               item), normalises and stores the row.  A warp whose 32 rows
//               are all past the request's last token does no arithmetic.
// While one tile's softmax runs, the tensor core works on the other tile's PV
// and QK^T, so the two tiles take turns on the tensor core.
//
// Shared-prefix mode (pkv_paged_prefill_attn_shared): requests that share the
// first S cached keys form a group, and an item is a block of the group's
// new tokens packed densely over its requests.  The item first runs the S
// shared keys (read through the first member's page row) for all its rows,
// unmasked, then each member's private keys S .. L_r - 1, causal for that
// member's rows and masked out for the rest; the online softmax carries
// every row across both phases.  A shared K/V tile is thus read once per
// item instead of once per request.
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace pkv {
namespace prefill {

constexpr int kThreads = 384;
constexpr int BM = 128;  // rows of a query tile: (token, head) pairs
constexpr int NQ = 2;    // query tiles per item
constexpr int BN = 128;  // keys per KV tile
constexpr int kKStages = 2, kVStages = 3;
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // warps 10 and 11 load K/V tiles with warp 8
constexpr int kLoaders = 3;              // warps issuing the K/V copies (8, 10, 11)
constexpr int kItemSlots = 2;            // items published ahead of the consumers
constexpr int kItemBytes = 128;          // shared memory per published item (>= sizeof(Item))
constexpr int kItemConsumers = 1 + 8 + (kLoaders - 1);  // MMA, softmax and loader warps
constexpr int kRankGroups = 256;         // up to this many (token block, request) groups
                                         // are ranked by work in the kernel
constexpr size_t kWorkspaceBytes = 256;  // queue counters (three used, the rest reserved)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
constexpr uint32_t kTmemCols = 512;
// Registers per thread: the block launches with kRegsLaunch for all 384
// threads; then warpgroup 2 (producer, MMA issuer, loaders) gives up all but
// regs_low and the two softmax warpgroups take regs_high each, so that a row's
// 128 scores and the softmax's temporaries fit without spilling.  Pages of
// fewer than 8 tokens are gathered by the loaders with per-key copies, which
// need more of their registers.  256 x regs_high + 128 x regs_low must not
// exceed 384 x kRegsLaunch.
constexpr int kRegsLaunch = 168;
template <bool SMALL, int MODE>
struct RegSplit {
    // (measured: 200/104 runs the 128-key pipeline faster than 208/88, whose
    // loader warps spill; pages of fewer than 8 tokens need still more in the
    // loaders)
    static constexpr int high = SMALL ? 176 : 200;
    static constexpr int low = SMALL ? 152 : 104;
    static_assert(8 * 32 * high + 4 * 32 * low <= kThreads * kRegsLaunch,
                  "register split exceeds the block's registers");
};

template <int D>
struct Layout {
    static constexpr int BLK = BM * 128;              // one 64-column swizzled block, 128 rows
    static constexpr int KBLK = BN * 128;             // one 64-column block of a K/V tile
    static constexpr int Q_BYTES = (D / 64) * BLK;    // one query tile
    static constexpr int KV_BYTES = (D / 64) * KBLK;  // one K or V tile (128 keys)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + kKStages * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + kVStages * KV_BYTES;
    // qfull, qempty, kfull/kempty[kKStages], vfull/vempty[kVStages],
    // per query tile: sfull, pfull, odone, ofree; item full/empty[kItemSlots]
    static constexpr int NBARS = 2 + 2 * kKStages + 2 * kVStages + NQ * 4 + 2 * kItemSlots;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int OFF_ITEMS = OFF_MISC + 64;     // decoded items, kItemSlots x kItemBytes
    static constexpr int OFF_RANK = OFF_ITEMS + kItemSlots * kItemBytes;  // int order[kRankGroups], weight[kRankGroups]
    static constexpr int TOTAL = OFF_RANK + 2 * kRankGroups * 4;
    // at least 116 KB: one block per SM (it holds all 512 TMEM columns)
    static constexpr size_t bytes() { return TOTAL > 118784 ? TOTAL : 118784; }
};

// tcgen05 shared-memory matrix descriptor: 128-byte swizzle, fixed version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, A K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte column chunk `chunk16` of row `row` in a tile stored
// as 64-column blocks of `rows` x 128 B with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk16, int rows) {
    const int blk = chunk16 >> 3, c = chunk16 & 7;
    return static_cast<uint32_t>(blk * rows * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}

// Forms of the kernel.  kCausal: each work item is a token block of one
// request against that request's keys, causally (the plain prefill).
// kFused (the shared-prefix form): a prefix group is a run of consecutive
// requests whose first S keys are the same pages; an item is a token block
// of the group's new tokens, packed back to back across its requests, and
// its key tiles are first the S shared keys (read once for all the packed
// rows, no mask: every new token comes after the prefix), then for each
// request of the block its own keys from S on, with that request's rows
// causal and the other requests' rows masked.  Each row's online softmax
// runs over both ranges, so no partial state leaves the block.
enum Mode : int { kCausal = 0, kFused = 1 };

// The prefix groups of a shared-prefix call (unused by kCausal).
struct Groups {
    const int32_t *start;   // [n + 1]: group g is requests start[g] .. start[g+1]-1
    const int32_t *len;     // [n]: keys shared by the group's requests
    int n;
    int nreq;               // requests in the call (the groups cover them all)
};

// One work item: query tiles A and B of token block mt of request r (of
// prefix group r in kFused), KV head g.  kCausal: key tiles 0 .. n_kt-1.
// kFused: the ns shared tiles (row of request pr, whose length is L0), then
// the private tiles of requests rlo .. rhi from klo = S on.
struct Item {
    int r, g, mt;
    int cu0, n, L, c;
    int tbeg[NQ], tend[NQ], nkt[NQ];
    int n_kt, klo, pr;
    int rlo, rhi, ns, L0;
};
static_assert(sizeof(Item) <= kItemBytes, "an item must fit its shared-memory slot");

// A role's position in a kFused item's key tiles: the request whose row
// holds the current tile (-1 while in the shared tiles), the tile, one past
// the last tile of its segment, and the number of keys in that row.
struct Steps {
    int r, kt, end, L;
};
// From request c.r on, the first request of the block with new tokens.
__device__ __forceinline__ void steps_seek(Steps &c, const Item &it, const int32_t *cu,
                                           const int32_t *seq_lens) {
    for (; c.r <= it.rhi; ++c.r) {
        const int nr = cu[c.r + 1] - cu[c.r];
        c.L = seq_lens[c.r];
        c.kt = it.klo / BN;
        c.end = nr > 0 ? (c.L + BN - 1) / BN : c.kt;
        if (c.end > c.kt) return;
    }
}
__device__ __forceinline__ void steps_begin(Steps &c, const Item &it, const int32_t *cu,
                                            const int32_t *seq_lens) {
    if (it.ns > 0) {
        c.r = -1;
        c.kt = 0;
        c.end = it.ns;
        c.L = it.L0;
    } else {
        c.r = it.rlo;
        steps_seek(c, it, cu, seq_lens);
    }
}
__device__ __forceinline__ void steps_next(Steps &c, const Item &it, const int32_t *cu,
                                           const int32_t *seq_lens) {
    if (++c.kt < c.end) return;
    c.r = c.r < 0 ? it.rlo : c.r + 1;
    steps_seek(c, it, cu, seq_lens);
}

template <int G, int MODE>
__device__ __forceinline__ void decode_item(int p, int Hkv, int B, int mtiles, const int *order,
                                            bool ranked, const int32_t *cu_seqlens,
                                            const int32_t *seq_lens, const Groups &gr, Item &it) {
    constexpr int TOK = BM / G;
    const int grank = p / Hkv;
    it.g = p % Hkv;
    const int grp = ranked ? order[grank] : grank;
    it.mt = mtiles - 1 - grp / B;
    it.r = grp % B;
    it.klo = 0;
    it.pr = it.r;
    it.ns = 0;
    if constexpr (MODE == kFused) {
        // the group's new tokens, packed; its shared keys; the requests of the
        // token block (rlo .. rhi) and the private tiles are set by the producer
        const int r0 = gr.start[it.r], r1 = gr.start[it.r + 1];
        it.pr = r0;
        it.cu0 = cu_seqlens[r0];
        it.n = cu_seqlens[r1] - it.cu0;
        it.klo = gr.len[it.r];
        it.L = it.klo;
        it.c = 0;
        it.ns = (it.klo + BN - 1) / BN;
        it.L0 = seq_lens[r0];
        it.rlo = r0;
        it.rhi = r1 - 1;
    } else {
        it.cu0 = cu_seqlens[it.r];
        it.n = cu_seqlens[it.r + 1] - it.cu0;
        it.L = seq_lens[it.r];
        it.c = it.L - it.n;
    }
    const int blk_tok0 = it.mt * NQ * TOK;
#pragma unroll
    for (int qt = 0; qt < NQ; ++qt) {
        it.tbeg[qt] = blk_tok0 + qt * TOK;
        it.tend[qt] = min(it.n, it.tbeg[qt] + TOK);
        it.nkt[qt] = it.tend[qt] > it.tbeg[qt] ? (it.c + it.tend[qt] + BN - 1) / BN : 0;
    }
    it.n_kt = it.nkt[0] > it.nkt[1] ? it.nkt[0] : it.nkt[1];
}

// Work of a (token block, request) group in key tiles (a (token block,
// prefix group) one in kFused, its private tiles estimated from the group's
// last request): 0 for no tokens, 1 for invalid offsets or lengths (the
// producer only flags those).
template <int G, int MODE>
__device__ __forceinline__ int group_weight(int grp, int B, int mtiles, int64_t Tq, int max_q_len,
                                            int64_t cap, const int32_t *cu_seqlens,
                                            const int32_t *seq_lens, const Groups &gr) {
    constexpr int TOK = BM / G;
    const int mt = mtiles - 1 - grp / B, r = grp % B;
    const int t0 = mt * NQ * TOK;
    if constexpr (MODE == kFused) {
        const int r0 = gr.start[r], r1 = gr.start[r + 1], S = gr.len[r];
        if (r0 < 0 || r1 <= r0 || r1 > gr.nreq) return 1;
        const int n = cu_seqlens[r1] - cu_seqlens[r0];
        if (t0 >= n) return 0;
        const int Ll = seq_lens[r1 - 1];
        if (S < 0 || S > cap || Ll < S || Ll > cap) return 1;
        return (S + BN - 1) / BN + (Ll + BN - 1) / BN - S / BN;
    } else {
        const int cu0 = cu_seqlens[r], cu1 = cu_seqlens[r + 1];
        const int n = cu1 - cu0, L = seq_lens[r];
        if (cu0 < 0 || n < 0 || cu1 > Tq || (r == 0 && cu0 != 0) || n > max_q_len) return 1;
        if (t0 >= n) return 0;
        if (L - n < 0 || L > cap) return 1;
        return (L - n + min(n, t0 + NQ * TOK) + BN - 1) / BN;
    }
}

// SMALL: pages of fewer than 8 tokens (gathered key by key); otherwise every
// page of a tile comes in as TMA boxes.
template <int D, int G, bool SMALL, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __nv_bfloat16 *__restrict__ k_cache,
                   const __nv_bfloat16 *__restrict__ v_cache, const int32_t *__restrict__ cu_seqlens,
                   const int32_t *__restrict__ page_table, int64_t pt_stride,
                   const int32_t *__restrict__ seq_lens, int B, int64_t Tq, int max_q_len, int Hkv,
                   int ps_log2, int box_rows, int64_t num_pages, float scale_log2, int mtiles,
                   const Groups gr, unsigned int *sched, int32_t *dev_status,
                   __nv_bfloat16 *__restrict__ out) {
    using Lo = Layout<D>;
    constexpr int TOK = BM / G;  // new tokens per query tile
    const int Hq = Hkv * G;
    const int64_t cap = pt_stride << ps_log2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    volatile int *misc = reinterpret_cast<volatile int *>(smem + Lo::OFF_MISC);
    volatile int *abort_flag = misc + 0;
    volatile int *item_ring = misc + 1;  // [kItemSlots]: published item, -1 = no more
    volatile int *bad_flag = misc + 3;   // [kItemSlots]: a page id of that item was invalid
    volatile int *n_items_s = misc + 5;
    volatile int *taken_s = misc + 6;    // items this block took from the queue (producer)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lo::OFF_MISC + 32);
    int *order = reinterpret_cast<int *>(smem + Lo::OFF_RANK);
    // the published items, decoded: slot s at OFF_ITEMS + s * kItemBytes
    auto item_at = [&](int s) -> Item & { return *reinterpret_cast<Item *>(smem + Lo::OFF_ITEMS + s * kItemBytes); };
    int *weight = order + kRankGroups;

    const uint32_t bar0 = smem_u32(smem + Lo::OFF_BAR);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
    constexpr int B_QFULL = 0, B_QEMPTY = 1;
    auto B_KFULL = [](int s) { return 2 + s; };
    auto B_KEMPTY = [](int s) { return 2 + kKStages + s; };
    auto B_VFULL = [](int s) { return 2 + 2 * kKStages + s; };
    auto B_VEMPTY = [](int s) { return 2 + 2 * kKStages + kVStages + s; };
    constexpr int kTileBar0 = 2 + 2 * kKStages + 2 * kVStages;
    auto B_SFULL = [](int qt) { return kTileBar0 + qt * 4; };
    auto B_PFULL = [](int qt) { return kTileBar0 + qt * 4 + 1; };
    auto B_ODONE = [](int qt) { return kTileBar0 + qt * 4 + 2; };
    auto B_OFREE = [](int qt) { return kTileBar0 + qt * 4 + 3; };
    constexpr int kItemBar0 = kTileBar0 + NQ * 4;
    auto B_IFULL = [](int s) { return kItemBar0 + s; };
    auto B_IEMPTY = [](int s) { return kItemBar0 + kItemSlots + s; };

    if (smem_u32(smem) & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
        if (tid == 0 && dev_status) atomicOr(dev_status, PKV_DEV_TIMEOUT);
        return;  // uniform for the whole block, before any barrier or counter is touched
    }
    if (tid == 0) {
        mbar_init(BAR(B_QFULL), 1);
        mbar_init(BAR(B_QEMPTY), 1);  // MMA commits
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(BAR(B_KFULL(s)), kLoaders);  // one arrival per loader warp (+ tx bytes)
            mbar_init(BAR(B_KEMPTY(s)), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(BAR(B_VFULL(s)), kLoaders);
            mbar_init(BAR(B_VEMPTY(s)), 1);
        }
        for (int qt = 0; qt < NQ; ++qt) {
            mbar_init(BAR(B_SFULL(qt)), 1);
            mbar_init(BAR(B_PFULL(qt)), 4);
            mbar_init(BAR(B_ODONE(qt)), 1);
            mbar_init(BAR(B_OFREE(qt)), 4);
        }
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(BAR(B_IFULL(s)), 1);
            mbar_init(BAR(B_IEMPTY(s)), kItemConsumers);
        }
        *abort_flag = 0;
        *n_items_s = 0;
        *taken_s = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // Rank the (token block, request) groups by work, heaviest first, when
    // there are few enough of them; all blocks compute the same order.
    const int n_groups = mtiles * B;
    const bool ranked = n_groups <= kRankGroups;
    __syncthreads();  // n_items_s zeroed
    if (ranked) {
        if (tid < n_groups) {
            const int w = group_weight<G, MODE>(tid, B, mtiles, Tq, max_q_len, cap, cu_seqlens, seq_lens, gr);
            weight[tid] = w;
            if (w > 0) atomicAdd(const_cast<int *>(n_items_s), 1);
        }
        __syncthreads();
        if (tid < n_groups) {
            const int w = weight[tid];
            int rank = 0;
            for (int u = 0; u < n_groups; ++u) {
                const int wu = weight[u];
                rank += (wu > w) || (wu == w && u < tid);
            }
            order[rank] = tid;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // groups of weight 0 are ranked last and never handed out
    const int n_items = (ranked ? *n_items_s : n_groups) * Hkv;
    // TMEM columns: S (then P over its first 64 columns) of tile qt at 128 qt,
    // O of tile qt at 256 + 128 qt
    auto tm_s = [&](int qt) -> uint32_t { return tmem + qt * BN; };
    auto tm_o = [&](int qt) -> uint32_t { return tmem + NQ * BN + qt * 128; };

    const uint32_t sQ = smem_u32(smem + Lo::OFF_Q);
    const uint32_t sK = smem_u32(smem + Lo::OFF_K);
    const uint32_t sV = smem_u32(smem + Lo::OFF_V);

    if (warp >= kProducerWarp) {
    regs_decrease<RegSplit<SMALL, MODE>::low>();
    if (warp != kMmaWarp) {
        // ================================================================ producer and loaders
        // Warp 8 takes the items and publishes them, and loads the Q tiles;
        // warps 8, 10 and 11 share the copies of every K and V tile (loader
        // li issues boxes li, li + 3, li + 6, ...): a warp's TMA issue rate,
        // not the copy engine, limits small boxes, so three warps issuing
        // keep the tensor core fed where one could not.
        const int li = warp == kProducerWarp ? 0 : warp - kMmaWarp;  // 0, 1, 2
        const uint64_t pol_kv = l2_evict_last_policy();  // K/V tiles are re-read by other blocks
        const uint64_t pol_q = l2_evict_first_policy();
        if (lane == 0) {
            if (li == 0) prefetch_tmap(&qmap);
            if (!SMALL) {
                prefetch_tmap(&kmap);
                prefetch_tmap(&vmap);
            }
        }
        const int ps_mask = (1 << ps_log2) - 1;
        const int bpt = !SMALL ? BN / box_rows : 1;  // page boxes per tile (<= 16)
        constexpr int NBLK = D / 64;                        // 64-column blocks of a row
        uint32_t kt = 0, vt = 0;  // K and V tiles loaded so far (ring position)
        bool ok = true;
        bool first = true;        // the first item of a block is its block index
        Item itm;
        // small pages: the full barrier of this warp's last gathered tile, whose
        // copies may still be in flight (0: none).  flush_gather waits for them
        // (all but the newest group when keep_one), makes them visible to the
        // tensor core and arrives on that barrier.
        uint32_t gather_pending = 0;
        // small pages: a step of the copy loop moves KPI = 4 whole key rows,
        // 8 lanes per row, each lane its 16-byte piece of every 64-column
        // block of the row; each 32-key block of a tile takes IPB steps, and
        // loader li takes steps li, li + 3, ... of every block.  So the block,
        // the key offsets and the swizzle terms are compile-time but for a
        // per-lane base, and a step costs a shuffle for its pool row, the
        // address arithmetic and one copy per 64-column block.
        constexpr int KPI = 4;                    // keys per step
        constexpr int IPB = 32 / KPI;             // steps per 32-key block
        constexpr int UPB = (IPB + kLoaders - 1) / kLoaders;  // of them per loader, at most
        static_assert(BN == 128, "the page ids of a tile's keys are held 4 per lane");
        const int ch = lane % 8;                            // this lane's piece of a 128-byte block row
        const int key_lane = li * KPI + lane / 8;           // its key in the block, u = 0
        const uint32_t dst_lane = static_cast<uint32_t>(key_lane * 128);
        const int64_t row_elems = static_cast<int64_t>(Hkv) * D;  // pool row stride (elements)
        // pool rows (slots) of keys lane + 32 r of this tile, -1 where a key has
        // none (past the row's keys, or a page id outside the pool); gpg_next
        // holds the next tile's page ids as read, converted when it is issued
        int gpg[4], gpg_next[4];
        auto flush_gather = [&](bool keep_one) {
            if (!gather_pending) return;
            if (keep_one)
                cp_async_wait<1>();
            else
                cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(gather_pending);
            gather_pending = 0;
        };
        for (uint32_t ii = 0; ok; ++ii) {
            const int slot = ii % kItemSlots;
            int p = -1;
            if (li == 0) {
                // next item with work; invalid ones are flagged (and for bad
                // lengths written as NaN) here and not published
                while (true) {
                    int q = static_cast<int>(blockIdx.x);
                    if (!first) {
                        if (lane == 0) q = static_cast<int>(gridDim.x + atomicAdd(sched, 1u));
                        q = __shfl_sync(0xffffffffu, q, 0);
                    }
                    first = false;
                    if (q >= n_items) break;
                    if (lane == 0) *taken_s += 1;
                    if constexpr (MODE == kFused) {
                        // the groups must be in range and cover the requests in order
                        const int grp = ranked ? order[q / Hkv] : q / Hkv;
                        const int gi = grp % B;
                        const int r0 = gr.start[gi], r1 = gr.start[gi + 1];
                        if (r0 < 0 || r1 <= r0 || r1 > gr.nreq || (gi == 0 && r0 != 0) ||
                            (gi == B - 1 && r1 != gr.nreq)) {
                            if (lane == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_SHARED);
                            continue;
                        }
                    }
                    decode_item<G, MODE>(q, Hkv, B, mtiles, order, ranked, cu_seqlens, seq_lens, gr, itm);
                    const int cu1 = itm.cu0 + itm.n;
                    if (itm.cu0 < 0 || itm.n < 0 || cu1 > Tq || (MODE != kFused && itm.r == 0 && itm.cu0 != 0) ||
                        itm.n > max_q_len) {
                        if (lane == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_CUSEQ);
                        continue;
                    }
                    const int blk_tok0 = itm.mt * NQ * TOK;
                    if (blk_tok0 >= itm.n) continue;
                    const int blk_tok1 = min(itm.n, blk_tok0 + NQ * TOK);
                    int bad = 0;  // a PKV_DEV_* bit: the block's rows are written as NaN
                    if constexpr (MODE == kFused) {
                        // the shared keys: a whole number of pages within the table;
                        // the requests of the token block, each with the shared keys
                        // inside its cached prefix and the group's shared pages first
                        // in its row (checked once per request), and their private tiles
                        const int S = itm.klo;
                        if (S < 0 || S > cap || (S & ((1 << ps_log2) - 1)) != 0 || itm.L0 > cap) {
                            bad = PKV_DEV_BAD_SHARED;
                        } else {
                            const int r0 = itm.pr, r1 = itm.rhi + 1;
                            // the request holding packed token t: the last r with cu[r] <= t
                            auto find_req = [&](int t) -> int {
                                int lo = r0, hi = r1;  // cu[lo] <= t < cu[hi]
                                while (hi - lo > 1) {
                                    const int step = (hi - lo + 31) / 32;
                                    const int cand = lo + lane * step;
                                    const bool le = cand < hi && cu_seqlens[cand] <= t;
                                    const unsigned m = __ballot_sync(0xffffffffu, le);
                                    lo += (31 - __clz(m)) * step;
                                    hi = min(hi, lo + step);
                                }
                                return lo;
                            };
                            itm.rlo = find_req(itm.cu0 + blk_tok0);
                            itm.rhi = find_req(itm.cu0 + blk_tok1 - 1);
                            int tiles = 0;
                            bool bs = false, bl = false, diff = false;
                            for (int r = itm.rlo + lane; r <= itm.rhi; r += 32) {
                                const int c0r = cu_seqlens[r], nr = cu_seqlens[r + 1] - c0r, Lr = seq_lens[r];
                                if (nr <= 0) continue;
                                if (Lr - nr < S) bs = true;
                                if (Lr > cap) bl = true;
                                if (!bs && !bl) tiles += (Lr + BN - 1) / BN - S / BN;
                            }
                            // each member's row lists the shared pages (the item of KV
                            // head 0 that holds the member's first new token checks)
                            if (itm.g == 0 && S > 0) {
                                for (int r = itm.rlo; r <= itm.rhi; ++r) {
                                    const int c0r = cu_seqlens[r];
                                    if (r == r0 || c0r < itm.cu0 + blk_tok0 || cu_seqlens[r + 1] == c0r) continue;
                                    const int32_t *rowr = page_table + (int64_t)r * pt_stride;
                                    const int32_t *row0 = page_table + (int64_t)r0 * pt_stride;
                                    for (int i = lane; i < (S >> ps_log2); i += 32) diff |= row0[i] != rowr[i];
                                }
                            }
                            if (__any_sync(0xffffffffu, diff) && lane == 0 && dev_status)
                                atomicOr(dev_status, PKV_DEV_BAD_SHARED);
                            tiles = __reduce_add_sync(0xffffffffu, tiles);
                            if (__any_sync(0xffffffffu, bs)) bad = PKV_DEV_BAD_SHARED;
                            else if (__any_sync(0xffffffffu, bl)) bad = PKV_DEV_BAD_SEQLEN;
                            itm.n_kt = itm.ns + tiles;
#pragma unroll
                            for (int qt = 0; qt < NQ; ++qt)
                                itm.nkt[qt] = itm.tend[qt] > itm.tbeg[qt] ? itm.n_kt : 0;
                            if (itm.n_kt == 0) continue;
                        }
                    } else if (itm.c < 0 || itm.L > cap) {
                        bad = PKV_DEV_BAD_SEQLEN;
                    }
                    if (bad) {
                        if (lane == 0 && dev_status) atomicOr(dev_status, bad);
                        for (int idx = lane; idx < (blk_tok1 - blk_tok0) * G * D; idx += 32) {
                            const int t = blk_tok0 + idx / (G * D);
                            const int rem = idx % (G * D);
                            out[((int64_t)(itm.cu0 + t) * Hq + (int64_t)itm.g * G) * D + rem] =
                                __float2bfloat16_rn(__int_as_float(0x7fc00000));
                        }
                        continue;
                    }
                    p = q;
                    break;
                }
                // publish it (or the end) to the other roles
                if (ii >= kItemSlots &&
                    !mbar_wait_warp(BAR(B_IEMPTY(slot)), ((ii / kItemSlots) & 1) ^ 1, abort_flag, dev_status))
                    break;
                if (lane == 0) {
                    item_ring[slot] = p;
                    bad_flag[slot] = 0;
                    if (p >= 0) item_at(slot) = itm;
                    mbar_arrive(BAR(B_IFULL(slot)));
                }
                __syncwarp();
            } else {
                if (!mbar_wait_warp(BAR(B_IFULL(slot)), (ii / kItemSlots) & 1, abort_flag, dev_status)) break;
                p = item_ring[slot];
                if (p >= 0) itm = item_at(slot);
            }
            if (p < 0) break;

            const int32_t *prow = page_table + (int64_t)itm.r * pt_stride;
            const int L = itm.L, g = itm.g;
            // kFused: the row, key tile and keys-in-row of the next K and the
            // next V tile (K tiles come one step ahead of V tiles)
            Steps ck{}, cv{};
            if constexpr (MODE == kFused) {
                steps_begin(ck, itm, cu_seqlens, seq_lens);
                cv = ck;
            }
            // page ids of tile kt's keys lane + 32 r of `row` (Lr keys), as read
            auto load_ids = [&](const int32_t *row, int Lr, int kt, int *dstp) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int kk = kt * BN + r * 32 + lane;
                    dstp[r] = kk < Lr ? row[kk >> ps_log2] : -1;
                }
            };
            // page ids of tile kt -> pool rows (slot = page x page_size +
            // offset; the host checks that every slot fits an int), -1 past
            // the row's Lr keys; true if a key's page id lies outside the pool
            auto to_slots = [&](int Lr, int kt, int *p) -> bool {
                bool bad = false;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int kk = kt * BN + r * 32 + lane;
                    const int id = p[r];
                    const bool ok_page = kk < Lr && id >= 0 && id < num_pages;
                    bad |= kk < Lr && !ok_page;
                    p[r] = ok_page ? (id << ps_log2) + (kk & ps_mask) : -1;
                }
                return bad;
            };
            // page ids in warp-wide windows of 32 page boxes, the next window
            // loaded ahead; a new row (kFused moves to another request's row)
            // reloads both windows
            auto load_window = [&](const int32_t *row, int Lr, int w) -> int {
                const int key = (32 * w + lane) * box_rows;
                return (!SMALL && key < Lr) ? row[key >> ps_log2] : 0;
            };
            const int32_t *win_row = nullptr;
            int w_cur = 0, pg_cur = 0, pg_nxt = 0;
            if constexpr (MODE != kFused) {  // one row per item: its first windows at once
                pg_cur = load_window(prow, L, 0);
                pg_nxt = load_window(prow, L, 1);
            }
            // page id of page box pb of key tile kt of `row` (lanes past the
            // tile's boxes get a neighbour's id, unused)
            auto page_of = [&](const int32_t *row, int Lr, int kt, int pb) -> int {
                const int b0 = kt * bpt;
                const int w = b0 >> 5;
                if constexpr (MODE == kFused) {
                    if (row != win_row || w < w_cur || w > w_cur + 1) {
                        win_row = row;
                        w_cur = w;
                        pg_cur = load_window(row, Lr, w);
                        pg_nxt = load_window(row, Lr, w + 1);
                    } else if (w == w_cur + 1) {
                        w_cur = w;
                        pg_cur = pg_nxt;
                        pg_nxt = load_window(row, Lr, w + 1);
                    }
                } else if (w != w_cur) {  // tiles come in order: the next window
                    w_cur = w;
                    pg_cur = pg_nxt;
                    pg_nxt = load_window(row, Lr, w + 1);
                }
                return __shfl_sync(0xffffffffu, pg_cur, (b0 + min(pb, bpt - 1)) & 31);
            };
            // one K or V tile (tile j of the item, ring position t): wait for
            // its slot, then this loader's share of the TMA boxes (or gather)
            auto load_tile = [&](int kv, int j, uint32_t t) -> bool {
                const int ns = kv ? kVStages : kKStages;
                const int s = t % ns;
                const uint32_t ph = (t / ns) & 1;
                const uint32_t full = BAR(kv ? B_VFULL(s) : B_KFULL(s));
                const uint32_t empty = BAR(kv ? B_VEMPTY(s) : B_KEMPTY(s));
                const uint32_t dst = (kv ? sV : sK) + s * Lo::KV_BYTES;
                // the tile's row, key tile and the keys of that row
                const int32_t *trow = prow;
                int tkt = j, tL = L;
                if constexpr (MODE == kFused) {
                    const Steps &c = kv ? cv : ck;
                    trow = page_table + (int64_t)(c.r < 0 ? itm.pr : c.r) * pt_stride;
                    tkt = c.kt;
                    tL = c.L;
                }
                const int key0 = tkt * BN;
                const int nkeys = min(BN, tL - key0);  // keys of this tile that exist in pages
                if (t >= static_cast<uint32_t>(ns) && !mbar_wait_warp(empty, ph ^ 1, abort_flag, dev_status))
                    return false;
                if constexpr (!SMALL) {
                    const int nbox = (nkeys + box_rows - 1) / box_rows;  // page boxes, <= 16
                    const int b = li + kLoaders * lane;                  // this lane's box
                    const int pb = b / NBLK, blk = b % NBLK;
                    const int pg = page_of(trow, tL, tkt, pb);
                    const bool mine = pb < nbox;
                    // a page id outside the pool is flagged; its box is read from
                    // a row before the pool, which the copy engine fills with zeros
                    const bool bad = mine && (pg < 0 || pg >= num_pages);
                    if (__any_sync(0xffffffffu, bad) && lane == 0) bad_flag[slot] = 1;
                    if (lane == 0) {
                        if (li == 0)
                            mbar_arrive_expect_tx(full,
                                                  static_cast<uint32_t>(nbox * NBLK * box_rows * 128));
                        else
                            mbar_arrive(full);
                    }
                    if (mine) {
                        const int kk = key0 + pb * box_rows;
                        const int row = bad ? -box_rows : (pg << ps_log2) + (kk & ps_mask);
                        tma_load_3d(dst + blk * Lo::KBLK + pb * box_rows * 128, kv ? &vmap : &kmap, full,
                                    blk * 64, g, row, pol_kv);
                    }
                    __syncwarp();
                } else {
                    // small pages: every key's row gathered with 16-byte copies
                    // straight into the swizzled layout (keys past the sequence or
                    // on a page outside the pool are zero-filled).  The copies of
                    // a tile complete while the warp issues its next tile; then
                    // the warp waits for them, orders them before the tensor
                    // core's reads and arrives (see flush_gather).
                    const __nv_bfloat16 *src_lane = (kv ? v_cache : k_cache) + static_cast<int64_t>(g) * D + ch * 8;
                    // page ids of this tile's keys: loaded for K(j) (or
                    // prefetched while V(j-1) was issued) and converted to
                    // pool rows, then reused for V(j), which prefetches those
                    // of tile j + 1
                    bool bad = false;
                    if constexpr (MODE == kFused) {
                        // (the tile's row may change between tiles: no lookahead)
                        if (kv == 0) {
                            load_ids(trow, tL, tkt, gpg);
                            bad = to_slots(tL, tkt, gpg);
                        }
                    } else if (kv == 0) {
                        if (j == 0) {
                            load_ids(prow, L, 0, gpg);
                        } else {
#pragma unroll
                            for (int r = 0; r < 4; ++r) gpg[r] = gpg_next[r];
                        }
                        bad = to_slots(L, j, gpg);
                    } else if (j + 1 < itm.n_kt) {
                        load_ids(prow, L, j + 1, gpg_next);
                    }
#pragma unroll
                    for (int b32 = 0; b32 < 4; ++b32) {
#pragma unroll
                        for (int u = 0; u < UPB; ++u) {
                            if (li + kLoaders * u >= IPB) break;  // (warp-uniform)
                            const int kl = key_lane + kLoaders * KPI * u;  // key in the block, < 32
                            const int sl = __shfl_sync(0xffffffffu, gpg[b32], kl);
                            const uint32_t d = dst + dst_lane +
                                               static_cast<uint32_t>(b32 * 32 * 128 + kLoaders * KPI * u * 128 +
                                                                     (((ch ^ kl) & 7) << 4));
                            const __nv_bfloat16 *src = src_lane + max(sl, 0) * row_elems;
                            const uint32_t nb = sl >= 0 ? 16u : 0u;
#pragma unroll
                            for (int blk = 0; blk < NBLK; ++blk)
                                cp_async16(d + blk * Lo::KBLK, src + blk * 64, nb);
                        }
                    }
                    cp_async_commit();
                    if (__any_sync(0xffffffffu, bad) && lane == 0) bad_flag[slot] = 1;
                    flush_gather(true);
                    gather_pending = full;
                }
                if constexpr (MODE == kFused) steps_next(kv ? cv : ck, itm, cu_seqlens, seq_lens);
                return true;
            };
            // K(0) first: it needs only a free K slot; the Q tiles wait until
            // the previous item's QK^T MMAs have read the Q buffer.  Until then
            // the Q tiles and the first K and V tiles are prefetched into L2.
            // (The first item's Q tiles have nothing to wait for: they are
            // loaded at once, before the page ids are read.)
            auto load_q = [&]() {
                if (lane == 0) {
                    mbar_arrive_expect_tx(BAR(B_QFULL), static_cast<uint32_t>(NQ * Lo::Q_BYTES));
#pragma unroll
                    for (int qt = 0; qt < NQ; ++qt)
#pragma unroll
                        for (int blk = 0; blk < NBLK; ++blk)
                            tma_load_3d(sQ + qt * Lo::Q_BYTES + blk * Lo::BLK, &qmap, BAR(B_QFULL),
                                        blk * 64, g * G, itm.cu0 + (qt ? itm.tbeg[1] : itm.tbeg[0]), pol_q);
                }
                __syncwarp();
            };
            if (li == 0 && ii == 0) load_q();
            if (li == 0 && ii > 0) {
                if (lane == 0) {
#pragma unroll
                    for (int qt = 0; qt < NQ; ++qt)
#pragma unroll
                        for (int blk = 0; blk < NBLK; ++blk)
                            tma_prefetch_3d(&qmap, blk * 64, g * G, itm.cu0 + itm.tbeg[qt]);
                }
                if (!SMALL) {
                    const int32_t *row0 = MODE == kFused ? page_table + (int64_t)(ck.r < 0 ? itm.pr : ck.r) * pt_stride
                                                         : prow;
                    const int kt0 = MODE == kFused ? ck.kt : 0, L0 = MODE == kFused ? ck.L : L;
                    const int nbox0 = (min(BN, L0 - kt0 * BN) + box_rows - 1) / box_rows;
                    const int pg0 = page_of(row0, L0, kt0, lane);
                    if (lane < nbox0 && pg0 >= 0 && pg0 < num_pages) {
                        const int row = (pg0 << ps_log2) + ((kt0 * BN + lane * box_rows) & ps_mask);
#pragma unroll
                        for (int blk = 0; blk < NBLK; ++blk) {
                            tma_prefetch_3d(&kmap, blk * 64, g, row);
                            tma_prefetch_3d(&vmap, blk * 64, g, row);
                        }
                    }
                }
            }
            ok = load_tile(0, 0, kt);
            if (ok && li == 0 && ii > 0) {
                ok = mbar_wait_warp(BAR(B_QEMPTY), (ii - 1) & 1, abort_flag, dev_status);
                if (ok) load_q();
            }
            if (!ok) break;
            // in the order the MMAs need them: V(j) for PV(j), then K(j+1) for
            // the QK^T that follows it (K runs one tile ahead of V)
            for (int j = 0; ok && j < itm.n_kt; ++j) {
                ok = load_tile(1, j, vt + j);
                if (ok && j + 1 < itm.n_kt) ok = load_tile(0, j + 1, kt + j + 1);
            }
            flush_gather(false);  // the item's last gathered tile is needed now
            kt += itm.n_kt;
            vt += itm.n_kt;
            if (ok && li > 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_IEMPTY(slot)));
            }
        }

    } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        // One lane issues the MMAs of both query tiles in a fixed order, so a
        // tile's PV and next QK^T run on the tensor core while the other
        // tile's softmax runs.  The K and V slots are released by commits
        // after both tiles' MMAs that read them.  The whole warp runs the
        // issue code and an elected lane issues (see elect_one).
        constexpr uint32_t idesc_s = instr_desc(BM, BN, false);
        constexpr uint32_t idesc_o = instr_desc(BM, D, true);
        auto issue_s = [&](int qt, uint32_t t) {  // S(qt) = Q(qt) K^T; K tile at ring position t
            const uint32_t kb = sK + (t % kKStages) * Lo::KV_BYTES;
            const uint32_t qb = sQ + qt * Lo::Q_BYTES;
            const uint32_t leader = elect_one();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qoff = (kk >> 2) * Lo::BLK + (kk & 3) * 32;
                const uint32_t koff = (kk >> 2) * Lo::KBLK + (kk & 3) * 32;
                umma_bf16_ss_if(tm_s(qt), smem_desc(qb + qoff, 16, 1024), smem_desc(kb + koff, 16, 1024),
                                idesc_s, kk > 0 ? 1u : 0u, leader);
            }
            umma_commit_if(BAR(B_SFULL(qt)), leader);
        };
        auto issue_pv = [&](int qt, uint32_t t, bool acc) {  // O(qt) += P(qt) V; V at ring position t
            const uint32_t vb = sV + (t % kVStages) * Lo::KV_BYTES;
            const uint32_t leader = elect_one();
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                umma_bf16_ts_if(tm_o(qt), tm_s(qt) + kk * 8, smem_desc(vb + kk * 16 * 128, Lo::KBLK, 1024),
                                idesc_o, (acc || kk > 0) ? 1u : 0u, leader);
        };
        auto commit = [&](uint32_t bar) { umma_commit_if(bar, elect_one()); };
        uint32_t kt = 0, vt = 0;        // ring positions of the current item's K(0) and V(0)
        uint32_t pc[NQ] = {0u, 0u};     // P tiles consumed per query tile (all items)
        uint32_t wk[NQ] = {0u, 0u};     // items in which the query tile had rows
        bool ok = true;
        for (uint32_t ii = 0; ok; ++ii) {
            const int slot = ii % kItemSlots;
            if (!mbar_wait_warp(BAR(B_IFULL(slot)), (ii / kItemSlots) & 1, abort_flag, dev_status)) break;
            const int p = item_ring[slot];
            if (p < 0) break;
            const Item &itm = item_at(slot);
            const int nk[NQ] = {itm.nkt[0], itm.nkt[1]};
            const int n_kt = itm.n_kt, L = itm.L;
            Steps cm{};  // kFused: the row and keys of each V tile
            if constexpr (MODE == kFused) steps_begin(cm, itm, cu_seqlens, seq_lens);
            ok = mbar_wait_warp(BAR(B_QFULL), ii & 1, abort_flag, dev_status) &&
                 mbar_wait_warp(BAR(B_KFULL(kt % kKStages)), (kt / kKStages) & 1, abort_flag, dev_status);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < NQ; ++t)
                if (nk[t] > 0) issue_s(t, kt);
            if (n_kt <= 1) commit(BAR(B_QEMPTY));  // every QK^T MMA of the item is issued
            commit(BAR(B_KEMPTY(kt % kKStages)));
            for (int j = 0; j < n_kt; ++j) {
                const uint32_t tv = vt + j;
                const int s = tv % kVStages;
                if (!mbar_wait_warp(BAR(B_VFULL(s)), (tv / kVStages) & 1, abort_flag, dev_status)) {
                    ok = false;
                    break;
                }
                const int tkt = MODE == kFused ? cm.kt : j, tL = MODE == kFused ? cm.L : L;
                if constexpr (MODE == kFused) steps_next(cm, itm, cu_seqlens, seq_lens);
                if ((tkt + 1) * BN > tL) {
                    // keys past the end of the tile's row hold stale pool data
                    // (maybe NaN): zero those V rows so that P = 0 there
                    // contributes exactly 0
                    const uint32_t vb = sV + s * Lo::KV_BYTES;
                    const int first_dead = tL - tkt * BN;
                    for (int idx = lane; idx < (BN - first_dead) * (D / 8); idx += 32) {
                        const int key = first_dead + idx / (D / 8), ch = idx % (D / 8);
                        *reinterpret_cast<uint4 *>(smem + (vb - smem_u32(smem)) +
                                                   swz_offset(key, ch, BN)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const uint32_t tk = kt + j + 1;
                bool k_ready = false;
#pragma unroll
                for (int t = 0; t < NQ; ++t) {
                    if (!ok || j >= nk[t]) continue;
                    if (!mbar_wait_warp(BAR(B_PFULL(t)), pc[t] & 1, abort_flag, dev_status)) {
                        ok = false;
                        break;
                    }
                    ++pc[t];
                    // the first PV of an item overwrites O: the previous item's
                    // output must have been read out of tensor memory
                    if (j == 0 && wk[t] > 0 &&
                        !mbar_wait_warp(BAR(B_OFREE(t)), (wk[t] - 1) & 1, abort_flag, dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(t, tv, j > 0);
                    if (j == nk[t] - 1) commit(BAR(B_ODONE(t)));
                    if (j + 1 < nk[t]) {
                        if (!k_ready) {
                            if (!mbar_wait_warp(BAR(B_KFULL(tk % kKStages)), (tk / kKStages) & 1,
                                                abort_flag, dev_status)) {
                                ok = false;
                                break;
                            }
                            k_ready = true;
                            tc_fence_after();
                        }
                        issue_s(t, tk);
                    }
                }
                if (!ok) break;
                commit(BAR(B_VEMPTY(s)));
                if (j + 1 < n_kt) {
                    if (!k_ready && !mbar_wait_warp(BAR(B_KFULL(tk % kKStages)), (tk / kKStages) & 1,
                                                    abort_flag, dev_status)) {
                        ok = false;
                        break;
                    }
                    if (j + 1 == n_kt - 1) commit(BAR(B_QEMPTY));
                    commit(BAR(B_KEMPTY(tk % kKStages)));
                }
            }
            kt += n_kt;
            vt += n_kt;
#pragma unroll
            for (int t = 0; t < NQ; ++t)
                if (nk[t] > 0) ++wk[t];
            if (ok) {
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_IEMPTY(slot)));
            }
        }
    }
    } else {
        // ================================================================ softmax
        regs_increase<RegSplit<SMALL, MODE>::high>();
        const int qt = warp >> 2;                  // query tile of this warpgroup
        const int row = tid & 127;                 // TMEM lane == tile row
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t sc = 0;                  // S tiles consumed by this warpgroup (all items)
        uint32_t od = 0;                  // items in which this tile had rows
        bool ok = true;
        for (uint32_t ii = 0; ok; ++ii) {
            const int slot = ii % kItemSlots;
            if (!mbar_wait_warp(BAR(B_IFULL(slot)), (ii / kItemSlots) & 1, abort_flag, dev_status)) break;
            const int p = item_ring[slot];
            if (p < 0) break;
            const Item &itm = item_at(slot);
            const int tok = (qt ? itm.tbeg[1] : itm.tbeg[0]) + row / G;
            const bool row_valid = tok < (qt ? itm.tend[1] : itm.tend[0]);
            const bool warp_live = __any_sync(0xffffffffu, row_valid);
            const int lim = itm.c + tok;  // kCausal: the last key this row may see
            // kFused: the row's request and the last of its keys it may see;
            // the step cursor tells whose keys each tile holds
            int r_row = -1, lim_row = 0;
            Steps cs{};
            if constexpr (MODE == kFused) {
                if (row_valid) {
                    const int t = itm.cu0 + tok;
                    int r = itm.rlo;
                    while (r < itm.rhi && cu_seqlens[r + 1] <= t) ++r;
                    r_row = r;
                    lim_row = seq_lens[r] - cu_seqlens[r + 1] + t;
                }
                steps_begin(cs, itm, cu_seqlens, seq_lens);
            }
            const int my_kt = (qt ? itm.nkt[1] : itm.nkt[0]);
            float m_ref = kNegBig, l_sum = 0.f;
            // tcgen05.ld/st are warp-collective: every wait outcome is warp-uniform
            for (int j = 0; j < my_kt; ++j) {
                // S(j) complete implies PV(j-1) complete: O is stable and P free
                ok = mbar_wait_warp(BAR(B_SFULL(qt)), (sc + j) & 1, abort_flag, dev_status);
                if (!ok) break;
                if (warp_live) {
                    tc_fence_after();
                    // all 128 scores of this row in registers (one wait for four loads)
                    uint32_t sv[BN];
#pragma unroll
                    for (int cc = 0; cc < BN / 32; ++cc)
                        tmem_ld_32cols(tm_s(qt) + lane_off + cc * 32, sv + cc * 32);
                    tmem_wait_ld();
                    // causal mask by selection (-inf), only on tiles that cross some
                    // valid row's limit (a warp-uniform branch).  Rows past the
                    // request's last token are not masked: their scores are never
                    // used (their output is not stored, and each row of P only
                    // feeds the same row of O), so a warp holding such rows does
                    // not pay for masking on every tile.
                    // nvalid: keys of the tile this row keeps from the start;
                    // nlow: kFused private tiles drop the shared keys below klo
                    int key0 = j * BN, nvalid = row_valid ? lim - key0 + 1 : BN, nlow = 0;
                    if constexpr (MODE == kFused) {
                        key0 = cs.kt * BN;
                        if (cs.r < 0) {  // shared keys: every row, no causal limit
                            nvalid = row_valid ? itm.klo - key0 : BN;
                        } else {         // request cs.r's own keys: its rows only
                            nvalid = row_valid ? (r_row == cs.r ? lim_row - key0 + 1 : 0) : BN;
                            nlow = itm.klo - key0;
                        }
                    }
                    if (__any_sync(0xffffffffu, nvalid < BN || nlow > 0)) {
#pragma unroll
                        for (int i = 0; i < BN; ++i)
                            if (i >= nvalid || i < nlow) sv[i] = __float_as_uint(-INFINITY);
                    }
                    // the row max, then p = 2^(s*scale*log2e - m_ref) on the SFU, packed
                    // to bf16 pairs and written 32 keys at a time into tensor memory
                    // over the S columns already read (keys 32cc.. -> columns 16cc..)
                    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < BN; i += 2)
                        mx4[(i >> 1) & 3] =
                            fmax3(mx4[(i >> 1) & 3], __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
                    const float mt_max = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
                    const bool need = (j > 0) && row_valid && (mt_max > m_ref + kRescaleLog2);
                    const bool warp_need = __any_sync(0xffffffffu, need);
                    float alpha = 1.f;
                    if (j == 0) {
                        m_ref = fmaxf(mt_max, kNegBig);  // stays finite for rows with no key
                        l_sum = 0.f;
                    } else if (warp_need) {
                        const float mn = fmaxf(m_ref, mt_max);
                        alpha = ex2(m_ref - mn);
                        m_ref = mn;
                    }
                    const float neg_m = -m_ref;
                    float rs[4] = {0.f, 0.f, 0.f, 0.f};  // two packed pairs of partial sums
#pragma unroll
                    for (int cc = 0; cc < BN / 32; ++cc) {
                        uint32_t pk[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int i = cc * 32 + 2 * q;
                            float x0, x1;
                            fma2(x0, x1, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]), scale_log2,
                                 scale_log2, neg_m, neg_m);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            add2(rs[2 * (q & 1)], rs[2 * (q & 1) + 1], p0, p1);
                            pk[q] = pack_bf16x2(p0, p1);
                        }
                        tmem_st_16cols(tm_s(qt) + lane_off + cc * 16, pk);
                    }
                    l_sum = l_sum * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
                    // rescale the output row to the new reference (PV(j-1) is complete)
                    if (warp_need) {
#pragma unroll
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t ov[32];
                            tmem_ld_32cols(tm_o(qt) + lane_off + cc * 32, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st_32cols(tm_o(qt) + lane_off + cc * 32, ov);
                        }
                    }
                    tmem_wait_st();  // P and O stores
                }
                if constexpr (MODE == kFused) steps_next(cs, itm, cu_seqlens, seq_lens);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_PFULL(qt)));
            }
            if (!ok) break;
            if (my_kt > 0) {
                ok = mbar_wait_warp(BAR(B_ODONE(qt)), od & 1, abort_flag, dev_status);
                ++od;
                if (!ok) break;
                tc_fence_after();
                // the output row out of tensor memory 32 columns at a time,
                // normalised, packed to bf16 and stored by its own thread in
                // 32-byte pieces (whole sectors)
                const bool poison = (bad_flag[slot] != 0) || (*abort_flag != 0);
                const float inv = row_valid ? 1.f / l_sum : 0.f;
                const int64_t out_row = ((int64_t)(itm.cu0 + tok) * Hq + (int64_t)itm.g * G + row % G) * D;
                if (warp_live) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        tmem_ld_32cols(tm_o(qt) + lane_off + cc * 32, ov);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            pk[e / 2] = poison ? 0x7fc07fc0u  // two bf16 NaNs
                                               : pack_bf16x2(__uint_as_float(ov[e]) * inv,
                                                             __uint_as_float(ov[e + 1]) * inv);
                        if (row_valid) {
                            st_global_32B(out + out_row + cc * 32, pk);
                            st_global_32B(out + out_row + cc * 32 + 16, pk + 8);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_OFREE(qt)));
                if (poison && tid == 0 && dev_status && bad_flag[slot])
                    atomicOr(dev_status, PKV_DEV_BAD_PAGE);
            }
            sc += my_kt;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_IEMPTY(slot)));
        }
    }
    // all roles meet here, then the TMEM is freed and the queue counters of
    // this call are reset by the last block to finish.  Every block adds the
    // number of items it took to a third counter before it counts itself
    // finished, so the last block sees exactly n_items there when the call
    // started from zeroed counters; anything else (items skipped or taken
    // twice) means the counters were shared or not cleared.
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0) {
        atomicAdd(sched + 2, static_cast<unsigned int>(*taken_s));
        __threadfence();
        if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
            __threadfence();
            const unsigned int taken = *reinterpret_cast<volatile unsigned int *>(sched + 2);
            if (dev_status && taken != static_cast<unsigned int>(n_items) &&
                (*reinterpret_cast<volatile int32_t *>(dev_status) & PKV_DEV_TIMEOUT) == 0)
                atomicOr(dev_status, PKV_DEV_BAD_WORKSPACE);
            sched[0] = 0;
            sched[1] = 0;
            sched[2] = 0;
            __threadfence();
        }
    }
}

template <int D, int G, int MODE>
static bool prepare(const pkv_host::DeviceInfo &dev) {
    static std::mutex mu;
    static bool ready[64] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev.device]) {
        if (Layout<D>::bytes() > static_cast<size_t>(dev.max_smem_optin)) return false;
        if (cudaFuncSetAttribute(prefill_kernel<D, G, false, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Layout<D>::bytes())) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_kernel<D, G, true, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Layout<D>::bytes())) != cudaSuccess)
            return false;
        ready[dev.device] = true;
    }
    return true;
}

// One pass over B work units (requests, or prefix groups in the shared pass)
// whose new tokens number at most max_q_len each.
template <int D, int G, int MODE>
static pkv_status launch(const pkv_bf16 *q, const int32_t *cu, const pkv_bf16 *k_cache,
                         const pkv_bf16 *v_cache, const int32_t *page_table, int64_t pt_stride,
                         const int32_t *seq_lens, int B, int64_t Tq, int max_q_len, int Hkv,
                         int page_size, int64_t num_pages, float scale, const Groups &gr,
                         unsigned int *sched, int32_t *dev_status, pkv_bf16 *out, cudaStream_t stream) {
    pkv_host::DeviceInfo dev;
    if (!pkv_host::current_device(&dev)) return PKV_ECUDA;
    if (!prepare<D, G, MODE>(dev)) return PKV_ECUDA;
    constexpr int TOK = BM / G;
    const int Hq = Hkv * G;
    const int box_rows = page_size < BN ? page_size : BN;
    CUtensorMap qmap, kmap, vmap;
    if (!pkv_host::encode_q_map(&qmap, q, Tq, Hq, D, G, TOK)) return PKV_EINVAL;
    const int64_t slots = num_pages * page_size;
    if (box_rows >= 8) {
        if (!pkv_host::encode_kv_map(&kmap, k_cache, slots, Hkv, D, 64, box_rows, true) ||
            !pkv_host::encode_kv_map(&vmap, v_cache, slots, Hkv, D, 64, box_rows, true))
            return PKV_EINVAL;
    } else {
        kmap = qmap;  // unused: small pages are gathered by the loaders' lanes
        vmap = qmap;
    }
    int ps_log2 = 0;
    while ((1 << ps_log2) < page_size) ++ps_log2;
    const int mtiles = (max_q_len + NQ * TOK - 1) / (NQ * TOK);
    const int64_t items = static_cast<int64_t>(mtiles) * B * Hkv;
    if (items == 0) return PKV_OK;
    if (items > 0x7fffffffll) return PKV_EUNSUPPORTED;
    // persistent: one block per SM (fewer when there are fewer items)
    const int grid = items < dev.sm_count ? static_cast<int>(items) : dev.sm_count;
    auto kernel = box_rows >= 8 ? prefill_kernel<D, G, false, MODE> : prefill_kernel<D, G, true, MODE>;
    kernel<<<static_cast<unsigned>(grid), kThreads, Layout<D>::bytes(), stream>>>(
        qmap, kmap, vmap, reinterpret_cast<const __nv_bfloat16 *>(k_cache),
        reinterpret_cast<const __nv_bfloat16 *>(v_cache), cu, page_table, pt_stride, seq_lens, B, Tq,
        max_q_len, Hkv, ps_log2, box_rows, num_pages, scale * kLog2e, mtiles, gr, sched, dev_status,
        reinterpret_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// Both entry points: argument checks, then the plain causal pass (no groups)
// or the shared pass followed by the private pass.
static pkv_status prefill_entry(const pkv_bf16 *q, const int32_t *cu_seqlens_q, const pkv_bf16 *k_cache,
                                const pkv_bf16 *v_cache, const int32_t *page_table,
                                int64_t page_table_stride, const int32_t *seq_lens, int batch,
                                int64_t total_q_tokens, int max_q_len, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int64_t num_pages, float softmax_scale,
                                const int32_t *group_start, const int32_t *group_len, int num_groups,
                                int max_group_tokens, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, pkv_bf16 *out, void *stream) {
    if (batch < 0 || total_q_tokens < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_pages <= 0 || page_table_stride < 0 || page_size <= 0 || num_groups < 0 ||
        max_group_tokens < 0)
        return PKV_EINVAL;
    if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
    if (!(softmax_scale == softmax_scale)) return PKV_EINVAL;
    if (batch == 0 || total_q_tokens == 0 || max_q_len == 0) return PKV_OK;
    if (!q || !cu_seqlens_q || !k_cache || !v_cache || !page_table || !seq_lens || !out ||
        !workspace)
        return PKV_EINVAL;
    const bool shared = num_groups > 0 && max_group_tokens > 0;
    if (shared && (!group_start || !group_len)) return PKV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    if (head_dim != 64 && head_dim != 128) return PKV_EUNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_EUNSUPPORTED;
    if ((page_size & (page_size - 1)) != 0 || page_size > 256) return PKV_EUNSUPPORTED;
    if (!pkv_host::aligned16(q) || !pkv_host::aligned16(k_cache) || !pkv_host::aligned16(v_cache) ||
        !pkv_host::aligned16(out) || !pkv_host::aligned16(workspace))
        return PKV_EINVAL;
    if (workspace_bytes < kWorkspaceBytes) return PKV_EINVAL;
    if (num_pages * page_size > 0x7fffffffll || total_q_tokens > 0x7fffffffll)
        return PKV_EUNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int *sched = static_cast<unsigned int *>(workspace);
    const Groups gr{group_start, group_len, shared ? num_groups : 0, batch};
#define PKV_PREFILL_CASE(DD, GG)                                                                      \
    if (head_dim == DD && G == GG) {                                                                  \
        if (!shared)                                                                                  \
            return launch<DD, GG, kCausal>(q, cu_seqlens_q, k_cache, v_cache, page_table,              \
                                           page_table_stride, seq_lens, batch, total_q_tokens,         \
                                           max_q_len, num_kv_heads, page_size, num_pages,              \
                                           softmax_scale, gr, sched, dev_status, out, st);            \
        return launch<DD, GG, kFused>(q, cu_seqlens_q, k_cache, v_cache, page_table,                   \
                                      page_table_stride, seq_lens, num_groups, total_q_tokens,         \
                                      max_group_tokens, num_kv_heads, page_size, num_pages,            \
                                      softmax_scale, gr, sched, dev_status, out, st);                 \
    }
    PKV_PREFILL_CASE(128, 1)
    PKV_PREFILL_CASE(128, 2)
    PKV_PREFILL_CASE(128, 4)
    PKV_PREFILL_CASE(128, 8)
    PKV_PREFILL_CASE(64, 1)
    PKV_PREFILL_CASE(64, 2)
    PKV_PREFILL_CASE(64, 4)
    PKV_PREFILL_CASE(64, 8)
#undef PKV_PREFILL_CASE
    return PKV_EUNSUPPORTED;
}

}  // namespace prefill
}  // namespace pkv

extern "C" size_t pkv_prefill_workspace_size(void) { return pkv::prefill::kWorkspaceBytes; }

extern "C" pkv_status pkv_paged_prefill_attn(const pkv_bf16 *q, const int32_t *cu_seqlens_q,
                                             const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                             const int32_t *page_table, int64_t page_table_stride,
                                             const int32_t *seq_lens, int batch,
                                             int64_t total_q_tokens, int max_q_len,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int page_size, int64_t num_pages, float softmax_scale,
                                             void *workspace, size_t workspace_bytes,
                                             int32_t *dev_status, pkv_bf16 *out, void *stream) {
    return pkv::prefill::prefill_entry(q, cu_seqlens_q, k_cache, v_cache, page_table, page_table_stride,
                                       seq_lens, batch, total_q_tokens, max_q_len, num_q_heads,
                                       num_kv_heads, head_dim, page_size, num_pages, softmax_scale,
                                       nullptr, nullptr, 0, 0, workspace, workspace_bytes, dev_status,
                                       out, stream);
}

extern "C" pkv_status pkv_paged_prefill_attn_shared(
    const pkv_bf16 *q, const int32_t *cu_seqlens_q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
    const int32_t *page_table, int64_t page_table_stride, const int32_t *seq_lens, int batch,
    int64_t total_q_tokens, int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int64_t num_pages, float softmax_scale, const int32_t *prefix_group_start,
    const int32_t *prefix_len, int num_prefix_groups, int max_group_tokens, void *workspace,
    size_t workspace_bytes, int32_t *dev_status, pkv_bf16 *out, void *stream) {
    return pkv::prefill::prefill_entry(q, cu_seqlens_q, k_cache, v_cache, page_table, page_table_stride,
                                       seq_lens, batch, total_q_tokens, max_q_len, num_q_heads,
                                       num_kv_heads, head_dim, page_size, num_pages, softmax_scale,
                                       prefix_group_start, prefix_len, num_prefix_groups,
                                       max_group_tokens, workspace, workspace_bytes, dev_status, out,
                                       stream);
}

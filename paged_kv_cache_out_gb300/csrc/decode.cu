// decode.cu -- paged decode attention: one query token per sequence over all
// of its cached keys, read through the page table.
//
// miniVLLM "Engine Architecture", prepare_decode: every sequence contributes
// one token; context_lens counts its keys; block_tables map each logical block
// to a physical one.  Grouped-query attention: the num_q_heads / num_kv_heads
// query heads of one KV head share its K/V rows (miniVLLM "LLMEngine":
// num_heads, num_kv_heads).
//
// Design (memory-bound: ~2 flops per byte of K/V):
//  * Work is measured in tiles of T key tokens of one (sequence, KV head)
//    "segment".  All segments are laid end to end and cut into gridDim.x equal
//    ranges, one per persistent block, so every block streams the same number
//    of bytes however unequal the sequence lengths are.  A segment cut by a
//    range boundary yields partial softmax states (max, sum, weighted values)
//    in the workspace; a second kernel merges them by log-sum-exp.
//  * One producer warp walks the block's tiles and stages each page's K and V
//    rows for this KV head into shared memory with TMA tensor copies (one box
//    of min(page_size, T) rows per page), through a ring of mbarrier-tracked
//    stages.  K/V are streamed once, so the copies carry an L2 evict-first hint.
//    Pages under 8 tokens are gathered four rows per copy (tile::gather4) by
//    four producer warps, whose issue rate limits such copies.
//  * Four consumer warps split every tile by rows: head_dim/16 lanes hold one
//    32-byte slice of a row each (head_dim/8 lanes, 16 bytes, with 8 query
//    heads per KV head); each lane keeps the G query heads' slice of q in
//    registers (pre-multiplied by scale*log2 e), reduces dot products with
//    warp shuffles, keeps its own online-softmax state per head, and
//    accumulates its slice of the output.  At the end of a segment piece the
//    row-groups' states are merged through shared memory.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace pkv {
namespace decode {

constexpr int kConsumerWarps = 4;
// warps 0-3 (warpgroup 0) consume; warp 4 produces, and with pages under 8
// tokens warps 5-7 produce too (below)
constexpr int kProducerWarps = 4;
constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
// With two blocks per SM a block launches with 128 registers per thread; the
// producers then give up all but RegSplit::producer and the consumers take
// RegSplit::consumer (128 x (176 + 80) = 256 x 128, so the increase always
// finds its registers).  With one block per SM (G = 8) nothing moves.  With
// 4 query heads per KV head the consumers keep 16 elements per lane (below)
// and take 184 (measured: long-context decode, head size 64, 71.0 -> 69.4 us
// at page size 256 and 89.3 -> 83.9 us at page size 1; head size 128,
// 64 sequences of 512-4096 keys, 119.1 -> 113.8 us at page size 16 and
// 142.6 -> 134.2 us at page size 1).
template <int D, int G>
struct RegSplit {
    static constexpr int consumer = (G == 4) ? 184 : 176;
    static constexpr int producer = 256 - consumer;
    static_assert(kConsumerWarps * 32 * consumer + kProducerWarps * 32 * producer <=
                      kThreads * (65536 / (2 * kThreads)),
                  "register split exceeds the registers of a block at two blocks per SM");
};
constexpr int kMaxBatch = 4096;
constexpr int kCtasPerSm = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;  // running-max start: finite, so 2^(m - m') never is NaN

// A consumer lane owns EPL elements of a row (EPL/8 16-byte chunks): 16 when
// there are at most 4 query heads per KV head (fewer lanes per row, so fewer
// shuffle levels to reduce the dot products), else 8, which keeps 8 heads
// within the registers of one block per SM.
template <int D, int G>
struct Shape {
    static constexpr int T = (D == 128) ? 32 : 64;  // key tokens per tile
    static constexpr int EPL = (G <= 4) ? 16 : 8;  // elements per lane
    static constexpr int NCH = EPL / 8;               // 16-byte chunks per lane
    static constexpr int R = D / EPL;                 // lanes per K/V row
    static constexpr int ROWS_PER_WARP = 32 / R;
    static constexpr int GROUPS = kConsumerWarps * ROWS_PER_WARP;
    static constexpr int U = T / GROUPS;  // rows of a tile per row-group
    static constexpr int TILE_BYTES = T * D * 2;
    static constexpr int STAGES = 4;
};

template <int D, int G>
struct Smem {
    using S = Shape<D, G>;
    static constexpr int Q_BYTES = ((G * D * 2 + 127) / 128) * 128;
    static constexpr int STAGE_BYTES = 2 * S::TILE_BYTES + Q_BYTES;
    static constexpr int RING = S::STAGES * STAGE_BYTES;
    static constexpr int RED_O = S::GROUPS * G * D * 4;
    static constexpr int RED_ML = S::GROUPS * G * 2 * 4;
    static constexpr int BARS = (2 * S::STAGES + 1) * 8;  // full, empty, fused stores done
    static constexpr int FLAGS = S::STAGES * 4 + 16;
    static constexpr int FIXED = RING + RED_O + RED_ML + BARS + FLAGS;
    // + tile offsets [batch + 1] and sequence lengths [batch], int32
    static size_t bytes(int batch) {
        return 1024 /* alignment slack */ + FIXED + static_cast<size_t>(2 * batch + 1) * 4;
    }
};

// Geometry of the balanced partition, shared by the main and merge kernels.
struct Part {
    int64_t W;   // total tiles
    int grid;    // blocks of the main kernel
    // floor(k W / grid), as k q + floor(k r / grid) with W = q grid + r: exact,
    // and k r < grid^2 fits 32 bits
    __device__ __forceinline__ int64_t start(int k) const {
        const int64_t q = W / grid;
        const int r = static_cast<int>(W - q * grid);
        return (int64_t)k * q + static_cast<int>(static_cast<unsigned>(k * r) / static_cast<unsigned>(grid));
    }
    __device__ __forceinline__ int block_of(int64_t x) const {
        return static_cast<int>(((x + 1) * grid - 1) / W);
    }
};

// Floats of one partial state in the workspace: G x D weighted sums, then a
// (max, sum) pair per head, padded to a multiple of 4 so that every state
// starts on a 16-byte boundary (the merge kernel reads it as float4).
__host__ __device__ constexpr int part_stride(int G, int D) { return ((G * D + 2 * G + 3) / 4) * 4; }

__device__ __forceinline__ int ntiles_of(int L, int64_t cap, int T) {
    return (L > 0 && L <= cap) ? (L + T - 1) / T : 0;
}

// Work units of a segment in the balanced partition: its tiles plus kLead
// units standing for the fixed cost of a segment piece (the page-id read, the
// q copy, the reduction across row groups and the output write), so that a
// block whose range holds many short segments gets fewer tiles.  A segment
// occupies [kLead lead units][its tiles]; lead units load nothing.  Empty
// segments occupy no units.
constexpr int kLead = 2;
__device__ __forceinline__ int units_of(int ntiles) { return ntiles > 0 ? ntiles + kLead : 0; }

// Largest b in [0, B) with prefix[b] <= x (x < prefix[B]).
__device__ __forceinline__ int owner_search(const int32_t *prefix, int B, int64_t x) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

struct Piece {
    int b, g;
    int t0, t1;         // tile range inside the segment (t1 <= t0: lead units only)
    int nt;             // tiles of the whole segment
    bool whole;         // covers all tiles of the segment
    bool block_first;   // first piece of this block
};

// The next piece of the block's unit range, with its units turned into tiles.
__device__ __forceinline__ bool next_piece(int64_t &pos, int64_t end, int64_t block_start,
                                           const int32_t *prefix, int B, int Hkv, Piece &p) {
    if (pos >= end) return false;
    const int b = owner_search(prefix, B, pos);
    const int nu = (prefix[b + 1] - prefix[b]) / Hkv;  // units of each segment of b
    const int64_t rel = pos - prefix[b];
    p.b = b;
    p.g = static_cast<int>(rel / nu);
    const int u0 = static_cast<int>(rel % nu);
    const int64_t seg_end = prefix[b] + (int64_t)(p.g + 1) * nu;
    const int64_t pend = end < seg_end ? end : seg_end;
    const int u1 = u0 + static_cast<int>(pend - pos);
    p.t0 = u0 > kLead ? u0 - kLead : 0;
    p.t1 = u1 - kLead;
    p.nt = nu - kLead;
    p.whole = (u0 <= kLead) && (pend == seg_end);
    p.block_first = (pos == block_start);
    pos = pend;
    return true;
}

// Block-wide exclusive scan: prefix[b] = Hkv * sum_{b' < b} units(b'); the
// lengths themselves are kept in lens[b].
__device__ void build_prefix(int32_t *prefix, int32_t *lens, const int32_t *seq_lens, int B,
                             int Hkv, int64_t cap, int T,
                             int32_t *scratch /* kThreads/32 + 1 ints */) {
    const int tid = threadIdx.x;
    const int per = (B + kThreads - 1) / kThreads;
    const int lo = tid * per;
    const int hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
        const int L = seq_lens[b];
        lens[b] = L;
        local += units_of(ntiles_of(L, cap, T)) * Hkv;
    }
    // inclusive scan of `local` over the block
    const int lane = tid & 31, warp = tid >> 5;
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            const int t = scratch[w];
            scratch[w] = acc;
            acc += t;
        }
        scratch[kThreads / 32] = acc;
    }
    __syncthreads();
    int run = scratch[warp] + v - local;  // exclusive prefix of this thread's chunk
    for (int b = lo; b < hi; ++b) {
        prefix[b] = run;
        run += units_of(ntiles_of(lens[b], cap, T)) * Hkv;
    }
    if (tid == 0) prefix[B] = scratch[kThreads / 32];
    __syncthreads();
}

// The fused store: each sequence's new K/V row (k_new/v_new [B, Hkv, D]) is
// written to pool slot out_loc[b], which must be the slot of position
// seq_lens[b] - 1.  k_new == nullptr turns it off.
struct Fuse {
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    const int32_t *out_loc;
    __nv_bfloat16 *k_cache;
    __nv_bfloat16 *v_cache;
};

// Copy one head's new K and V rows (D bf16 each) to their pool slot with the
// lanes of one warp.
template <int D>
__device__ __forceinline__ void store_new_rows(const Fuse &fz, int b, int g, int Hkv, int64_t slot,
                                               int lane) {
    constexpr int VEC = D * 2 / 16;
    const uint4 *ks = reinterpret_cast<const uint4 *>(fz.k_new + ((int64_t)b * Hkv + g) * D);
    const uint4 *vs = reinterpret_cast<const uint4 *>(fz.v_new + ((int64_t)b * Hkv + g) * D);
    uint4 *kd = reinterpret_cast<uint4 *>(fz.k_cache + (slot * Hkv + g) * D);
    uint4 *vd = reinterpret_cast<uint4 *>(fz.v_cache + (slot * Hkv + g) * D);
    for (int i = lane; i < VEC; i += 32) {
        kd[i] = __ldg(ks + i);
        vd[i] = __ldg(vs + i);
    }
}

// Fused store, run by the consumer threads of a block before its first tile:
// every segment (b, g) whose last tile lies in the block's range [t0, t1) gets
// its new K/V row written to pool slot out_loc[b], one thread per segment.
// Those segments are consecutive in (b, g) order.  Ends with a proxy fence, so
// that after the barrier that follows, the copy engine reads the stored rows.
template <int D>
__device__ void store_block_rows(const Fuse &fz, const int32_t *prefix, const int32_t *lens,
                                 const int32_t *page_table, int64_t pt_stride, int B, int Hkv,
                                 int ps_log2, int64_t num_slots, int64_t t0, int64_t t1, int ctid,
                                 int32_t *dev_status) {
    constexpr int CH = D * 2 / 16;  // 16-byte chunks of a row
    const int b0 = owner_search(prefix, B, t0);
    const int b1 = owner_search(prefix, B, t1 - 1);
    const int64_t o0 = (int64_t)b0 * Hkv + (t0 - prefix[b0]) / ((prefix[b0 + 1] - prefix[b0]) / Hkv);
    const int64_t o1 = (int64_t)b1 * Hkv + (t1 - 1 - prefix[b1]) / ((prefix[b1 + 1] - prefix[b1]) / Hkv);
    bool flag = false;
    for (int64_t o = o0 + ctid; o <= o1; o += kConsumerWarps * 32) {
        const int b = static_cast<int>(o / Hkv), g = static_cast<int>(o % Hkv);
        const int nu = (prefix[b + 1] - prefix[b]) / Hkv;
        if (nu == 0) continue;  // no keys: the merge kernel stores its row
        const int64_t last = prefix[b] + (int64_t)(g + 1) * nu - 1;  // its last tile
        if (last < t0 || last >= t1) continue;
        const int64_t slot = fz.out_loc[b];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            flag = true;  // beyond the pool: not stored
            continue;
        }
        const int L = lens[b];
        const int64_t expect =
            ((int64_t)page_table[(int64_t)b * pt_stride + ((L - 1) >> ps_log2)] << ps_log2) +
            ((L - 1) & ((1 << ps_log2) - 1));
        if (slot != expect) flag = true;
        const uint4 *ks = reinterpret_cast<const uint4 *>(fz.k_new + ((int64_t)b * Hkv + g) * D);
        const uint4 *vs = reinterpret_cast<const uint4 *>(fz.v_new + ((int64_t)b * Hkv + g) * D);
        uint4 *kd = reinterpret_cast<uint4 *>(fz.k_cache + (slot * Hkv + g) * D);
        uint4 *vd = reinterpret_cast<uint4 *>(fz.v_cache + (slot * Hkv + g) * D);
        uint4 kr[CH], vr[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            kr[c] = __ldg(ks + c);
            vr[c] = __ldg(vs + c);
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            kd[c] = kr[c];
            vd[c] = vr[c];
        }
    }
    if (flag && dev_status) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
    fence_proxy_async_global();
}

template <int D, int G, bool FUSE>
__global__ void __launch_bounds__(kThreads, G <= 4 ? kCtasPerSm : 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const __nv_bfloat16 *__restrict__ k_cache, const __nv_bfloat16 *__restrict__ v_cache,
                  const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ page_table,
                  int64_t pt_stride, const int32_t *__restrict__ seq_lens, int B, int Hkv,
                  int ps_log2, int box_rows, int64_t num_pages, float scale_log2,
                  float *__restrict__ ws_part, int32_t *__restrict__ ws_prefix,
                  int32_t *dev_status, __nv_bfloat16 *__restrict__ out, const Fuse fz) {
    using S = Shape<D, G>;
    using M = Smem<D, G>;
    constexpr int T = S::T, R = S::R, U = S::U, GROUPS = S::GROUPS, STAGES = S::STAGES;
    constexpr int NCH = S::NCH;
    const int Hq = Hkv * G;
    const int64_t cap = pt_stride << ps_log2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *ring = smem;
    float *red_o = reinterpret_cast<float *>(smem + M::RING);
    float *red_ml = reinterpret_cast<float *>(smem + M::RING + M::RED_O);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M::RING + M::RED_O + M::RED_ML);
    int *flags = reinterpret_cast<int *>(smem + M::RING + M::RED_O + M::RED_ML + M::BARS);
    volatile int *abort_flag = flags + STAGES;
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + M::FIXED);
    int32_t *lens = prefix + (B + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dependency_wait();  // the pool rows of this step are written by the kernel before
    // No early trigger for the merge kernel: its blocks would become resident
    // at once and sit on every SM until this grid ends, which keeps a
    // whole-SM kernel on another stream (the prefill of a mixed step) from
    // starting, and the standalone call measured no faster with them.  The
    // merge kernel is released as this grid's blocks exit.
    if (tid == 0) {
        // full: the producer's arrival with the tx bytes
        for (int s = 0; s < STAGES; ++s) {
            // full: each producer's arrival with its tx bytes
            mbar_init(smem_u32(&bars[s]), box_rows < 8 ? static_cast<uint32_t>(kProducerWarps) : 1u);
            mbar_init(smem_u32(&bars[STAGES + s]), kConsumerWarps);  // empty: one per consumer warp
        }
        mbar_init(smem_u32(&bars[2 * STAGES]), kConsumerWarps);  // fused stores written
        *abort_flag = 0;
        fence_mbar_init();
    }
    // red_ml doubles as the scan scratch before any piece is reduced
    build_prefix(prefix, lens, seq_lens, B, Hkv, cap, T, reinterpret_cast<int32_t *>(red_ml));
    if (blockIdx.x == 0)
        for (int b = tid; b <= B; b += kThreads) ws_prefix[b] = prefix[b];

    Part part{prefix[B], static_cast<int>(gridDim.x)};
    if (part.W == 0) return;
    const int64_t my_start = part.start(blockIdx.x);
    const int64_t my_end = part.start(blockIdx.x + 1);
    if (my_start >= my_end) return;

    if (warp >= kConsumerWarps) {
        // ------------------------------------------------------------ producers
        // Page boxes (pages of >= 8 tokens) take a few TMA copies per tile, all
        // issued by warp 4.  Pages of fewer tokens take a tile::gather4 per
        // four key rows, and a warp's TMA issue rate then limits the copy
        // rate, so warps 4 and 5 issue half of the K gathers each (warp 4 also
        // the q copy) and warps 6 and 7 those of V.  Measured on the page
        // size 1 decode workloads, one issuing warp -> two -> four: Qwen3
        // 290 -> 232 -> 233 us, long context (d 64) 135 -> 100 -> 89 us.
        // (Warps splitting the page boxes too made long-context decode at
        // page size 256 slower, 71.4 -> 73.0 us.)
        const int pw = warp - kConsumerWarps;
        if constexpr (G <= 4) regs_decrease<RegSplit<D, G>::producer>();
        if (pw > 0 && box_rows >= 8) return;
        const uint64_t policy = l2_evict_first_policy();
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
        }
        const int ps_mask = (1 << ps_log2) - 1;
        const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * D * 2;
        const bool small = box_rows < 8;  // gather key rows instead of page boxes
        int64_t pos = my_start;
        Piece p;
        uint32_t it = 0;
        bool ok = true;
        bool stores_seen = false;
        // boxes per tile; up to 32 of them page ids come in warp-wide windows
        // of 32 boxes, the next two windows loaded ahead (with pages of one
        // token a window lasts one tile)
        const int bpt = T / box_rows;
        while (ok && next_piece(pos, my_end, my_start, prefix, B, Hkv, p)) {
            if (p.t1 <= p.t0) continue;  // lead units only: nothing to load
            const int L = lens[p.b];
            const int32_t *prow = page_table + (int64_t)p.b * pt_stride;
            auto load_window = [&](int w) -> int {
                const int key = (32 * w + lane) * box_rows;
                return key < L ? prow[key >> ps_log2] : 0;
            };
            int w_cur = (p.t0 * bpt) >> 5;
            int pg_cur = 0, pg_nxt = 0, pg_nxt2 = 0;
            if (bpt <= 32) {
                pg_cur = load_window(w_cur);
                pg_nxt = load_window(w_cur + 1);
                pg_nxt2 = load_window(w_cur + 2);
            }
            auto advance = [&](int w) {
                w_cur = w;
                pg_cur = pg_nxt;
                pg_nxt = pg_nxt2;
                pg_nxt2 = load_window(w + 2);
            };
            for (int tile = p.t0; tile < p.t1; ++tile, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (it >= STAGES && !mbar_wait_warp(smem_u32(&bars[STAGES + s]), ph ^ 1, abort_flag,
                                                    dev_status)) {
                    ok = false;
                    break;
                }
                const int tok0 = tile * T;
                const int ntok = min(T, L - tok0);
                const bool first = (tile == p.t0);
                // fused store: the consumers write the new rows of the block's
                // segments first; a segment's last tile (which holds its new
                // row) is copied only after that
                if (FUSE && tile == p.nt - 1 && !stores_seen) {
                    if (!mbar_wait_warp(smem_u32(&bars[2 * STAGES]), 0, abort_flag, dev_status)) {
                        ok = false;
                        break;
                    }
                    stores_seen = true;
                }
                uint8_t *st = ring + s * M::STAGE_BYTES;
                const uint32_t full = smem_u32(&bars[s]);
                const uint32_t q_bytes = first ? static_cast<uint32_t>(G * D * 2) : 0u;
                if (!small) {
                    const int nbox = (ntok + box_rows - 1) / box_rows;
                    // page ids of this tile's boxes (at most T boxes: two per lane)
                    int pg[2] = {0, 0};
                    bool bad = false;
                    if (bpt <= 32) {
                        const int b0 = tile * bpt;
                        if ((b0 >> 5) != w_cur) advance(b0 >> 5);
                        pg[0] = __shfl_sync(0xffffffffu, pg_cur, (b0 + (lane % bpt)) & 31);
                        if (lane < nbox && (pg[0] < 0 || pg[0] >= num_pages)) bad = true;
                    } else {
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int i = lane + 32 * k;
                            if (i < nbox) {
                                pg[k] = prow[(tok0 + i * box_rows) >> ps_log2];
                                if (pg[k] < 0 || pg[k] >= num_pages) bad = true;
                            }
                        }
                    }
                    bad = __any_sync(0xffffffffu, bad);
                    const uint32_t bytes = (bad ? 0u : 2u * box_bytes * nbox) + q_bytes;
                    if (lane == 0) {
                        flags[s] = bad ? 1 : 0;
                        mbar_arrive_expect_tx(full, bytes);
                    }
                    __syncwarp();
                    if (!bad) {
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int i = lane + 32 * k;
                            if (i < nbox) {
                                const int j = tok0 + i * box_rows;
                                const int row = (pg[k] << ps_log2) + (j & ps_mask);
                                tma_load_3d(smem_u32(st + i * box_bytes), &kmap, full, 0, p.g, row,
                                            policy);
                                tma_load_3d(smem_u32(st + S::TILE_BYTES + i * box_bytes), &vmap, full,
                                            0, p.g, row, policy);
                            }
                        }
                    }
                } else {
                    // pages of fewer than 8 tokens: the tile's key rows gathered
                    // four at a time with TMA (tile::gather4 over the pool viewed
                    // as rows of one head, row = slot * Hkv + g).  Gather i < NG
                    // (rows 4i..4i+3) of K is issued by lane i % NH of warp
                    // 4 + i / NH, the same gather of V by the same lane of warp
                    // 6 + i / NH.  Keys
                    // past the sequence end take the row of the tile's first key
                    // (the consumers never use them), so every row read exists.
                    constexpr int NG = T / 4;  // gathers per tile and tensor
                    static_assert(NG % 2 == 0 && NG / 2 <= 32, "one gather per lane");
                    const int b0 = tile * bpt;
                    if (bpt <= 32 && (b0 >> 5) != w_cur) advance(b0 >> 5);
                    constexpr int NH = NG / 2;  // gathers per producer warp
                    const int gi = (pw & 1) * NH + lane % NH;
                    int rows[4];
                    bool bad = false;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int key = 4 * gi + r;
                        const int kk = key < ntok ? key : 0;
                        int pg;
                        if (bpt <= 32)
                            pg = __shfl_sync(0xffffffffu, pg_cur, (b0 + kk / box_rows) & 31);
                        else
                            pg = prow[(tok0 + kk) >> ps_log2];
                        if (key < ntok && (pg < 0 || pg >= num_pages)) bad = true;
                        const int64_t slot = ((int64_t)pg << ps_log2) + ((tok0 + kk) & ps_mask);
                        rows[r] = static_cast<int>(slot * Hkv + p.g);
                    }
                    bad = __any_sync(0xffffffffu, bad);
                    if (lane == 0) {
                        if (pw == 0) flags[s] = bad ? 1 : 0;
                        mbar_arrive_expect_tx(full, (bad ? 0u : static_cast<uint32_t>(S::TILE_BYTES / 2)) +
                                                        (pw == 0 ? q_bytes : 0u));
                    }
                    __syncwarp();
                    if (!bad && lane < NH) {
                        const uint32_t dst = smem_u32(st) + (pw < 2 ? 0u : S::TILE_BYTES) + gi * 4 * D * 2;
                        tma_gather4(dst, pw < 2 ? &kmap : &vmap, full, 0, rows[0], rows[1], rows[2], rows[3],
                                    policy);
                    }
                }
                if (first && lane == 0 && pw == 0)
                    bulk_load(smem_u32(st + 2 * S::TILE_BYTES),
                              q + ((int64_t)p.b * Hq + (int64_t)p.g * G) * D, G * D * 2, full);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    if constexpr (G <= 4) regs_increase<RegSplit<D, G>::consumer>();
    const int grp = warp * S::ROWS_PER_WARP + lane / R;  // row-group of this lane
    const int lr = lane % R;                             // slice of a row
    // the lane owns 16-byte chunks lr, lr + R, ... of each row
    const int ctid = tid;                                // 0..127
    if constexpr (FUSE) {
        // while the first tiles are in flight: store the new K/V rows of the
        // segments whose last tile is in this block, then tell the producer
        store_block_rows<D>(fz, prefix, lens, page_table, pt_stride, B, Hkv, ps_log2,
                            num_pages << ps_log2, my_start, my_end, ctid, dev_status);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[2 * STAGES]));
    }
    // q (pre-scaled by scale*log2 e) and the output slice as fp32 pairs, so the
    // dot products and the value accumulation run as packed fp32x2 FMAs
    float2 q2[G][4 * NCH];
    float m[G], l[G];
    float2 o2[G][4 * NCH];
    int64_t pos = my_start;
    Piece p;
    uint32_t it = 0;
    bool ok = true;
    while (ok && next_piece(pos, my_end, my_start, prefix, B, Hkv, p)) {
        if (p.t1 <= p.t0) continue;  // lead units only: nothing to do
        const int L = lens[p.b];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = kNegBig;
            l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 4 * NCH; ++e) o2[h][e] = make_float2(0.f, 0.f);
        }
        bool bad_piece = false;
        for (int tile = p.t0; tile < p.t1; ++tile, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait_warp(smem_u32(&bars[s]), ph, abort_flag, dev_status)) {
                ok = false;
                break;
            }
            const uint8_t *st = ring + s * M::STAGE_BYTES;
            const uint32_t kbase = smem_u32(st);
            const uint32_t vbase = kbase + S::TILE_BYTES;
            if (flags[s]) bad_piece = true;
            if (tile == p.t0) {
                const uint32_t qbase = kbase + 2 * S::TILE_BYTES;
                const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int k = 0; k < NCH; ++k) {
                        const uint4 w = lds128(qbase + (h * D + (lr + k * R) * 8) * 2);
                        q2[h][4 * k + 0] = fmul2(bf16x2_to_f2(w.x), sc2);
                        q2[h][4 * k + 1] = fmul2(bf16x2_to_f2(w.y), sc2);
                        q2[h][4 * k + 2] = fmul2(bf16x2_to_f2(w.z), sc2);
                        q2[h][4 * k + 3] = fmul2(bf16x2_to_f2(w.w), sc2);
                    }
            }
            const int tok0 = tile * T;
            const bool full_tile = tok0 + T <= L;  // same for the whole block: no row masking
            float sc[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int row = grp + u * GROUPS;
                float2 kv[4 * NCH];
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    const uint4 w = lds128(kbase + (row * D + (lr + k * R) * 8) * 2);
                    kv[4 * k + 0] = bf16x2_to_f2(w.x);
                    kv[4 * k + 1] = bf16x2_to_f2(w.y);
                    kv[4 * k + 2] = bf16x2_to_f2(w.z);
                    kv[4 * k + 3] = bf16x2_to_f2(w.w);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 acc = fmul2(q2[h][0], kv[0]);
#pragma unroll
                    for (int e = 1; e < 4 * NCH; ++e) acc = ffma2(q2[h][e], kv[e], acc);
                    sc[u][h] = acc.x + acc.y;
                }
            }
#pragma unroll
            for (int off = R / 2; off >= 1; off >>= 1) {
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        sc[u][h] += __shfl_xor_sync(0xffffffffu, sc[u][h], off);
            }
            if (!full_tile) {
                // rows past the sequence end: score -inf, so p = 0
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (tok0 + grp + u * GROUPS >= L)
#pragma unroll
                        for (int h = 0; h < G; ++h) sc[u][h] = -INFINITY;
            }
            // online softmax with a lazy reference: the running max m only moves
            // when a score exceeds it by more than 2^8, so p <= 256 and the
            // rescaling of l and o is rare (exact: every term shares m)
            float pr[U][G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mt = sc[0][h];
#pragma unroll
                for (int u = 1; u < U; ++u) mt = fmaxf(mt, sc[u][h]);
                if (mt > m[h] + 8.0f) {
                    const float alpha = ex2(m[h] - mt);
                    m[h] = mt;
                    l[h] *= alpha;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < 4 * NCH; ++e) o2[h][e] = fmul2(o2[h][e], a2);
                }
                float sum = 0.f;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    pr[u][h] = ex2(sc[u][h] - m[h]);
                    sum += pr[u][h];
                }
                l[h] += sum;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int row = grp + u * GROUPS;
                // rows past the sequence end hold stale data (maybe NaN): zero
                // them, since 0 * NaN would poison the sum
                const bool dead = !full_tile && tok0 + row >= L;
                float2 vv[4 * NCH];
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    uint4 w = lds128(vbase + (row * D + (lr + k * R) * 8) * 2);
                    if (dead) w = make_uint4(0u, 0u, 0u, 0u);
                    vv[4 * k + 0] = bf16x2_to_f2(w.x);
                    vv[4 * k + 1] = bf16x2_to_f2(w.y);
                    vv[4 * k + 2] = bf16x2_to_f2(w.z);
                    vv[4 * k + 3] = bf16x2_to_f2(w.w);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float2 p2 = make_float2(pr[u][h], pr[u][h]);
#pragma unroll
                    for (int e = 0; e < 4 * NCH; ++e) o2[h][e] = ffma2(p2, vv[e], o2[h][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[STAGES + s]));
        }
        if (!ok) break;

        // ---- merge the row-groups' states of this piece
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < NCH; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    red_o[(grp * G + h) * D + (lr + k * R) * 8 + 2 * e] = o2[h][4 * k + e].x;
                    red_o[(grp * G + h) * D + (lr + k * R) * 8 + 2 * e + 1] = o2[h][4 * k + e].y;
                }
            if (lr == 0) {
                red_ml[(grp * G + h) * 2 + 0] = m[h];
                red_ml[(grp * G + h) * 2 + 1] = l[h];
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
        const int slot = static_cast<int>(blockIdx.x) * 2 + (p.block_first ? 0 : 1);
        for (int idx = ctid; idx < G * D; idx += kConsumerWarps * 32) {
            const int h = idx / D;
            float mx = kNegBig;
#pragma unroll
            for (int g2 = 0; g2 < GROUPS; ++g2) mx = fmaxf(mx, red_ml[(g2 * G + h) * 2]);
            float sum = 0.f, acc = 0.f;
#pragma unroll
            for (int g2 = 0; g2 < GROUPS; ++g2) {
                const float w = ex2(red_ml[(g2 * G + h) * 2] - mx);
                sum = fmaf(red_ml[(g2 * G + h) * 2 + 1], w, sum);
                acc = fmaf(red_o[(g2 * G + h) * D + (idx % D)], w, acc);
            }
            if (p.whole) {
                const float v = bad_piece ? __int_as_float(0x7fc00000) : acc / sum;
                out[((int64_t)p.b * Hq + (int64_t)p.g * G) * D + idx] = __float2bfloat16_rn(v);
            } else {
                float *part_o = ws_part + (int64_t)slot * part_stride(G, D);
                part_o[idx] = acc;
                if (idx % D == 0) {
                    part_o[G * D + 2 * h] = bad_piece ? __int_as_float(0x7fc00000) : mx;
                    part_o[G * D + 2 * h + 1] = sum;
                }
            }
        }
        if (bad_piece && ctid == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_PAGE);
        named_bar_sync(1, kConsumerWarps * 32);
    }
}

// Merge of the partial states of segments that were cut across blocks, and
// the output of segments with no keys (zeros, or NaN for an invalid length).
// One block per segment; thread (v, kl) owns the 4 output values of float4 v
// and the partial states k0 + kl, k0 + kl + KL, ... of the segment, so all of
// a thread's loads are independent and the KL partial sums of a vector meet
// in warp shuffles.
constexpr int kMergeThreads = 256;
template <int D, int G>
__global__ void __launch_bounds__(kMergeThreads)
    decode_merge_kernel(const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ ws_prefix,
                        const float *__restrict__ ws_part, int B, int Hkv, int64_t cap, int grid,
                        int32_t *dev_status, __nv_bfloat16 *__restrict__ out, const Fuse fz,
                        int64_t num_slots) {
    constexpr int E = G * D;                       // output values of a segment
    constexpr int NV = E / 4;                      // float4 pieces
    constexpr int KL = kMergeThreads / NV;         // partial states per piece in parallel
    static_assert(KL >= 1 && KL <= 32 && (KL & (KL - 1)) == 0, "merge layout");
    constexpr int STRIDE = part_stride(G, D);      // floats per partial state
    grid_dependency_wait();  // partial states come from the main kernel
    const int b = blockIdx.x / Hkv, g = blockIdx.x % Hkv;
    const int Hq = Hkv * G;
    __nv_bfloat16 *orow = out + ((int64_t)b * Hq + (int64_t)g * G) * D;
    const int nu = (ws_prefix[b + 1] - ws_prefix[b]) / Hkv;  // units of the segment
    if (nu == 0) {
        const int L = seq_lens[b];
        const bool bad = (L < 0 || L > cap);
        // fused store of a sequence that attends to nothing: still store its row
        if (fz.k_new && threadIdx.x < 32) {
            const int64_t slot = fz.out_loc[b];
            if (slot >= 0 && slot < num_slots)
                store_new_rows<D>(fz, b, g, Hkv, slot, threadIdx.x);
            else if (slot >= num_slots && threadIdx.x == 0 && dev_status)
                atomicOr(dev_status, PKV_DEV_BAD_SLOT);
        }
        if (bad && g == 0 && threadIdx.x == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_SEQLEN);
        for (int idx = threadIdx.x; idx < E; idx += blockDim.x)
            orow[idx] = __float2bfloat16_rn(bad ? __int_as_float(0x7fc00000) : 0.f);
        return;
    }
    Part part{ws_prefix[B], grid};
    const int64_t s0 = ws_prefix[b] + (int64_t)g * nu;  // the segment's units, lead units first
    const int64_t s1 = s0 + nu;
    // blocks holding its tiles (blocks before k0 hold lead units only)
    const int k0 = part.block_of(s0 + kLead), k1 = part.block_of(s1 - 1);
    if (k0 == k1) return;  // written directly by the main kernel
    const int v = threadIdx.x / KL, kl = threadIdx.x % KL;
    const int h = (4 * v) / D;  // query head of this piece
    // the partial-state slot of block k, or -1 for blocks whose range is empty
    // (fewer units than blocks): they hold no state of this segment.  The
    // segment's piece is the block's first piece (slot 2k) unless the segment
    // starts after the block's range does (slot 2k + 1: its last piece).
    auto slot_of = [&](int k) -> int {
        const int64_t a = part.start(k), z = part.start(k + 1);
        if (z <= a) return -1;
        return 2 * k + ((k == k0 && s0 > a) ? 1 : 0);
    };
    float mx = kNegBig;
    bool bad = false;
    for (int k = k0 + kl; k <= k1; k += KL) {
        const int sl = slot_of(k);
        if (sl < 0) continue;
        const float mk = ws_part[(int64_t)sl * STRIDE + E + 2 * h];
        bad |= isnan(mk);
        mx = fmaxf(mx, mk);
    }
#pragma unroll
    for (int o = KL / 2; o >= 1; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        bad |= __shfl_xor_sync(0xffffffffu, bad ? 1 : 0, o) != 0;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
    for (int k = k0 + kl; k <= k1; k += KL) {
        const int sl = slot_of(k);
        if (sl < 0) continue;
        const float *pk = ws_part + (int64_t)sl * STRIDE;
        const float w = ex2(pk[E + 2 * h] - mx);
        sum = fmaf(pk[E + 2 * h + 1], w, sum);
        const float4 o4 = *reinterpret_cast<const float4 *>(pk + 4 * v);
        acc.x = fmaf(o4.x, w, acc.x);
        acc.y = fmaf(o4.y, w, acc.y);
        acc.z = fmaf(o4.z, w, acc.z);
        acc.w = fmaf(o4.w, w, acc.w);
    }
#pragma unroll
    for (int o = KL / 2; o >= 1; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (kl == 0) {
        const float inv = 1.f / sum;
        const float nan = __int_as_float(0x7fc00000);
        const uint32_t lo = pack_bf16x2(bad ? nan : acc.x * inv, bad ? nan : acc.y * inv);
        const uint32_t hi = pack_bf16x2(bad ? nan : acc.z * inv, bad ? nan : acc.w * inv);
        *reinterpret_cast<uint2 *>(orow + 4 * v) = make_uint2(lo, hi);
    }
}

// ---------------------------------------------------------------- host side
struct LaunchInfo {
    bool ready = false;
    int ctas_per_sm = 0;
};

template <int D, int G>
static bool prepare(const pkv_host::DeviceInfo &dev, int batch, int *ctas_per_sm) {
    static std::mutex mu;
    static LaunchInfo info[64];
    std::lock_guard<std::mutex> lk(mu);
    LaunchInfo &li = info[dev.device];
    const size_t max_smem = Smem<D, G>::bytes(kMaxBatch);
    if (!li.ready) {
        if (max_smem > static_cast<size_t>(dev.max_smem_optin)) return false;
        if (cudaFuncSetAttribute(decode_kernel<D, G, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(max_smem)) != cudaSuccess ||
            cudaFuncSetAttribute(decode_kernel<D, G, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(max_smem)) != cudaSuccess)
            return false;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, G, false>, kThreads,
                                                          Smem<D, G>::bytes(256)) != cudaSuccess)
            return false;
        li.ctas_per_sm = n < 1 ? 1 : (n > kCtasPerSm ? kCtasPerSm : n);
        li.ready = true;
    }
    (void)batch;
    *ctas_per_sm = li.ctas_per_sm;
    return true;
}

template <int D, int G>
static pkv_status launch(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                         const int32_t *page_table, int64_t pt_stride, const int32_t *seq_lens,
                         int B, int Hkv, int page_size, int64_t num_pages, float scale,
                         void *workspace, int32_t *dev_status, pkv_bf16 *out, const Fuse &fz,
                         cudaStream_t stream) {
    pkv_host::DeviceInfo dev;
    if (!pkv_host::current_device(&dev)) return PKV_ECUDA;
    int ctas = 0;
    if (!prepare<D, G>(dev, B, &ctas)) return PKV_ECUDA;
    const int T = Shape<D, G>::T;
    const int box_rows = page_size < T ? page_size : T;
    CUtensorMap kmap, vmap;
    const int64_t slots = num_pages * page_size;
    if (box_rows >= 8) {  // page boxes
        if (!pkv_host::encode_kv_map(&kmap, k_cache, slots, Hkv, D, D, box_rows, false) ||
            !pkv_host::encode_kv_map(&vmap, v_cache, slots, Hkv, D, D, box_rows, false))
            return PKV_EINVAL;
    } else {  // rows gathered four at a time
        if (slots * Hkv > 0x7fffffffll) return PKV_EUNSUPPORTED;
        if (!pkv_host::encode_rows_map(&kmap, k_cache, slots * Hkv, D) ||
            !pkv_host::encode_rows_map(&vmap, v_cache, slots * Hkv, D))
            return PKV_EINVAL;
    }
    int ps_log2 = 0;
    while ((1 << ps_log2) < page_size) ++ps_log2;
    const int grid = dev.sm_count * ctas;
    int32_t *ws_prefix = static_cast<int32_t *>(workspace);
    float *ws_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                               (((size_t)(B + 1) * 4 + 255) & ~size_t(255)));
    const float scale_log2 = scale * kLog2e;
    // the fused store has its own instantiation, so the plain call carries none of it
    auto kernel = fz.k_new ? decode_kernel<D, G, true> : decode_kernel<D, G, false>;
    if (pkv_host::launch_dependent(kernel, dim3(grid), dim3(kThreads),
                                   Smem<D, G>::bytes(B), stream, kmap, vmap,
                                   reinterpret_cast<const __nv_bfloat16 *>(k_cache),
                                   reinterpret_cast<const __nv_bfloat16 *>(v_cache),
                                   reinterpret_cast<const __nv_bfloat16 *>(q), page_table, pt_stride,
                                   seq_lens, B, Hkv, ps_log2, box_rows, num_pages, scale_log2,
                                   ws_part, ws_prefix, dev_status,
                                   reinterpret_cast<__nv_bfloat16 *>(out), fz) != cudaSuccess)
        return PKV_ECUDA;
    if (pkv_host::launch_dependent(decode_merge_kernel<D, G>, dim3(B * Hkv), dim3(kMergeThreads), 0, stream,
                                   seq_lens, static_cast<const int32_t *>(ws_prefix),
                                   static_cast<const float *>(ws_part), B, Hkv,
                                   pt_stride * page_size, grid, dev_status,
                                   reinterpret_cast<__nv_bfloat16 *>(out), fz, slots) != cudaSuccess)
        return PKV_ECUDA;
    return PKV_OK;
}

}  // namespace decode
}  // namespace pkv

using namespace pkv::decode;

static bool supported_gqa(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }

extern "C" size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                            int head_dim) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
        return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    pkv_host::DeviceInfo dev;
    if (!pkv_host::current_device(&dev)) return 0;
    const int G = num_q_heads / num_kv_heads;
    const size_t grid = static_cast<size_t>(dev.sm_count) * kCtasPerSm;
    const size_t prefix = ((static_cast<size_t>(batch) + 1) * 4 + 255) & ~size_t(255);
    return prefix + grid * 2 * static_cast<size_t>(part_stride(G, head_dim)) * 4;
}

// Shared argument checks and dispatch of the decode entry points.  With
// `scratch` set, the workspace arguments are ignored: after every other check
// has passed, sizes needing more than scratch->bytes are rejected with
// PKV_EUNSUPPORTED and scratch->get() supplies the workspace.
static pkv_status decode_entry(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                               const int32_t *page_table, int64_t page_table_stride,
                               const int32_t *seq_lens, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                               float softmax_scale, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, pkv_bf16 *out, const Fuse &fz, void *stream,
                               const pkv_host::Scratch *scratch) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_pages <= 0 ||
        page_table_stride < 0 || page_size <= 0)
        return PKV_EINVAL;
    if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
    if (!(softmax_scale == softmax_scale)) return PKV_EINVAL;
    if (batch == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out) return PKV_EINVAL;
    if (!scratch && !workspace) return PKV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || !supported_gqa(G)) return PKV_EUNSUPPORTED;
    if ((page_size & (page_size - 1)) != 0 || page_size > 256) return PKV_EUNSUPPORTED;
    if (batch > kMaxBatch) return PKV_EUNSUPPORTED;
    if (!pkv_host::aligned16(q) || !pkv_host::aligned16(k_cache) || !pkv_host::aligned16(v_cache) ||
        !pkv_host::aligned16(out) || (!scratch && !pkv_host::aligned16(workspace)))
        return PKV_EINVAL;
    if (fz.k_new && (!pkv_host::aligned16(fz.k_new) || !pkv_host::aligned16(fz.v_new)))
        return PKV_EINVAL;
    if (num_pages * page_size > 0x7fffffffll) return PKV_EUNSUPPORTED;
    // total tiles must fit the block's int32 prefix sums
    const int T = head_dim == 128 ? Shape<128, 1>::T : Shape<64, 1>::T;  // T depends on head_dim only
    const int64_t max_tiles = (page_table_stride * page_size + T - 1) / T + kLead;  // units
    if (static_cast<double>(batch) * num_kv_heads * max_tiles >= 2147483647.0)
        return PKV_EUNSUPPORTED;
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim);
    if (scratch) {
        if (need > scratch->bytes) return PKV_EUNSUPPORTED;
        workspace = scratch->get();
        if (!workspace) return PKV_ECUDA;
    } else if (workspace_bytes < need) {
        return PKV_EINVAL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define PKV_DECODE_CASE(DD, GG)                                                                 \
    if (head_dim == DD && G == GG)                                                              \
        return launch<DD, GG>(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, batch, \
                              num_kv_heads, page_size, num_pages, softmax_scale, workspace,     \
                              dev_status, out, fz, st);
    PKV_DECODE_CASE(128, 1)
    PKV_DECODE_CASE(128, 2)
    PKV_DECODE_CASE(128, 4)
    PKV_DECODE_CASE(128, 8)
    PKV_DECODE_CASE(64, 1)
    PKV_DECODE_CASE(64, 2)
    PKV_DECODE_CASE(64, 4)
    PKV_DECODE_CASE(64, 8)
#undef PKV_DECODE_CASE
    return PKV_EUNSUPPORTED;
}

extern "C" pkv_status pkv_paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                            const pkv_bf16 *v_cache, const int32_t *page_table,
                                            int64_t page_table_stride, const int32_t *seq_lens,
                                            int batch, int num_q_heads, int num_kv_heads,
                                            int head_dim, int page_size, int64_t num_pages,
                                            float softmax_scale, void *workspace,
                                            size_t workspace_bytes, int32_t *dev_status,
                                            pkv_bf16 *out, void *stream) {
    const Fuse none{nullptr, nullptr, nullptr, nullptr, nullptr};
    return decode_entry(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, batch,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, softmax_scale,
                        workspace, workspace_bytes, dev_status, out, none, stream, nullptr);
}

extern "C" pkv_status pkv_paged_decode_attn_store(
    const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *out_loc,
    pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *page_table, int64_t page_table_stride,
    const int32_t *seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int64_t num_pages, float softmax_scale, void *workspace,
    size_t workspace_bytes, int32_t *dev_status, pkv_bf16 *out, void *stream) {
    if (batch > 0 && (!k_new || !v_new || !out_loc)) return PKV_EINVAL;
    const Fuse fz{reinterpret_cast<const __nv_bfloat16 *>(k_new),
                  reinterpret_cast<const __nv_bfloat16 *>(v_new), out_loc,
                  reinterpret_cast<__nv_bfloat16 *>(k_cache),
                  reinterpret_cast<__nv_bfloat16 *>(v_cache)};
    return decode_entry(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, batch,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, softmax_scale,
                        workspace, workspace_bytes, dev_status, out, fz, stream, nullptr);
}

pkv_status pkv_host::decode_with_scratch(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                         const pkv_bf16 *v_cache, const int32_t *page_table,
                                         int64_t page_table_stride, const int32_t *seq_lens,
                                         int batch, int num_q_heads, int num_kv_heads,
                                         int head_dim, int page_size, int64_t num_pages,
                                         float softmax_scale, int32_t *dev_status, pkv_bf16 *out,
                                         void *stream, const Scratch &scratch) {
    const Fuse none{nullptr, nullptr, nullptr, nullptr, nullptr};
    return decode_entry(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, batch,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, softmax_scale,
                        nullptr, 0, dev_status, out, none, stream, &scratch);
}

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
// One block computes a 128-row tile of (token, query head) rows of one
// request and one KV head: 128/G consecutive new tokens x the G query heads of
// that KV head, so every K/V tile staged in shared memory serves all G heads.
// Roles (256 threads):
//   warp 0      producer: Q once, then 128-key K and V tiles through a
//               2-stage ring.  Pages of >= 8 tokens come in as TMA boxes
//               (one per page, 128-byte swizzle, straight into the layout the
//               tensor core reads); smaller pages are gathered by the warp's
//               lanes with 16-byte loads and swizzled stores.
//   warp 1      allocates 512 TMEM columns (two 128x128 fp32 score buffers and
//               the 128 x head_dim fp32 output accumulator); one lane issues
//               S = Q K^T (M=128, N=128, K=head_dim) and O += P V (M=128,
//               N=head_dim, K=128), bf16 operands from shared memory.
//   warps 4-7   softmax: thread i owns row i (TMEM lane i): reads its scores,
//               applies the causal mask by selection, keeps a running max and
//               sum in the log2 domain, writes P as bf16 into shared memory in
//               the swizzled K-major layout, and rescales the TMEM output row
//               when the running max grew by more than 2^8; at the end it
//               normalises the output row and stores it.
//   warps 2-3   idle.
// QK^T of tile j+1 and PV of tile j-1 run on the tensor cores while the
// softmax warps compute the exponentials of tile j.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace pkv {
namespace prefill {

constexpr int kThreads = 256;
constexpr int BM = 128;  // rows of a tile: (token, head) pairs
constexpr int BN = 128;  // keys per KV tile
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Layout {
    static constexpr int BLK = BM * 128;             // one 64-column swizzled block, 128 rows
    static constexpr int Q_BYTES = (D / 64) * BLK;   // Q tile
    static constexpr int KV_BYTES = (D / 64) * BLK;  // one K or V tile (128 keys)
    static constexpr int P_BYTES = (BN / 64) * BLK;  // P tile, 128 x 128 bf16
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + kStages * KV_BYTES;
    static constexpr int OFF_P = OFF_V + kStages * KV_BYTES;
    static constexpr int OFF_BAR = OFF_P + P_BYTES;
    // barriers: q_full, kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], sfree[2], pfull, odone
    static constexpr int NBARS = 1 + 4 * kStages + 2 + 2 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    // at least 116 KB so that two blocks never share an SM: each holds 512 TMEM columns
    static constexpr size_t bytes() { return (1024 + TOTAL) > 118784 ? (1024 + TOTAL) : 118784; }
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

// Byte offset of element (row, col) of a [rows x 64k] bf16 tile stored as
// 64-column blocks of `rows` x 128 B with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk16 /* 16-byte column chunk */,
                                               int rows) {
    const int blk = chunk16 >> 3, c = chunk16 & 7;
    return static_cast<uint32_t>(blk * rows * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __nv_bfloat16 *__restrict__ k_cache,
                   const __nv_bfloat16 *__restrict__ v_cache, const int32_t *__restrict__ cu_seqlens,
                   const int32_t *__restrict__ page_table, int64_t pt_stride,
                   const int32_t *__restrict__ seq_lens, int B, int64_t Tq, int max_q_len, int Hkv,
                   int ps_log2, int box_rows, int64_t num_pages, float scale_log2, int mtiles,
                   int32_t *dev_status, __nv_bfloat16 *__restrict__ out) {
    using Lo = Layout<D>;
    constexpr int TOK = BM / G;  // new tokens per tile
    const int Hq = Hkv * G;
    const int64_t cap = pt_stride << ps_log2;

    // ---- which tile: heaviest (largest mt) first over all requests and heads
    const int lin = blockIdx.x;
    const int per_mt = B * Hkv;
    const int mt = mtiles - 1 - lin / per_mt;
    const int r = (lin % per_mt) / Hkv;
    const int g = lin % Hkv;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cu0 = cu_seqlens[r], cu1 = cu_seqlens[r + 1];
    const int n = cu1 - cu0;
    const int L = seq_lens[r];
    const int c = L - n;
    const bool cu_bad = cu0 < 0 || n < 0 || cu1 > Tq || (r == 0 && cu0 != 0) || n > max_q_len;
    if (cu_bad) {
        if (tid == 0 && mt == 0 && g == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_CUSEQ);
        return;
    }
    const int tok_begin = mt * TOK;
    if (tok_begin >= n) return;
    const int tok_end = min(n, tok_begin + TOK);
    const bool len_bad = (c < 0) || (L > cap);
    if (len_bad) {
        if (tid == 0 && mt == 0 && g == 0 && dev_status) atomicOr(dev_status, PKV_DEV_BAD_SEQLEN);
        // rows are known: write NaN
        for (int idx = tid; idx < (tok_end - tok_begin) * G * D; idx += kThreads) {
            const int t = tok_begin + idx / (G * D);
            const int rem = idx % (G * D);
            out[((int64_t)(cu0 + t) * Hq + (int64_t)g * G) * D + rem] =
                __float2bfloat16_rn(__int_as_float(0x7fc00000));
        }
        return;
    }
    const int kend = c + tok_end;  // keys [0, kend) are needed by this tile
    const int n_kt = (kend + BN - 1) / BN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lo::OFF_BAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
    // barrier indices
    const int B_QFULL = 0;
    auto B_KFULL = [](int s) { return 1 + s; };
    auto B_KEMPTY = [](int s) { return 1 + kStages + s; };
    auto B_VFULL = [](int s) { return 1 + 2 * kStages + s; };
    auto B_VEMPTY = [](int s) { return 1 + 3 * kStages + s; };
    auto B_SFULL = [](int b) { return 1 + 4 * kStages + b; };
    auto B_SFREE = [](int b) { return 3 + 4 * kStages + b; };
    const int B_PFULL = 5 + 4 * kStages;
    const int B_ODONE = 6 + 4 * kStages;
    volatile int *misc = reinterpret_cast<volatile int *>(smem + Lo::OFF_MISC);
    volatile int *abort_flag = misc + 0;
    volatile int *bad_page = misc + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lo::OFF_MISC + 16);

    if (tid == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(BAR(B_KFULL(s)), 1);
            mbar_init(BAR(B_KEMPTY(s)), 1);
            mbar_init(BAR(B_VFULL(s)), 1);
            mbar_init(BAR(B_VEMPTY(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR(B_SFULL(b)), 1);
            mbar_init(BAR(B_SFREE(b)), 4);
        }
        mbar_init(BAR(B_PFULL), 4);
        mbar_init(BAR(B_ODONE), 1);
        *abort_flag = 0;
        *bad_page = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_s[2] = {tmem, tmem + 128};
    const uint32_t tm_o = tmem + 256;

    const uint32_t sQ = smem_u32(smem + Lo::OFF_Q);
    const uint32_t sK = smem_u32(smem + Lo::OFF_K);
    const uint32_t sV = smem_u32(smem + Lo::OFF_V);
    const uint32_t sP = smem_u32(smem + Lo::OFF_P);
    const int32_t *prow = page_table + (int64_t)r * pt_stride;

    if (warp == 0) {
        // ================================================================ producer
        const uint64_t pol_kv = l2_evict_last_policy();  // K/V tiles are re-read by other tiles
        if (lane == 0) {
            prefetch_tmap(&qmap);
            if (box_rows >= 8) {
                prefetch_tmap(&kmap);
                prefetch_tmap(&vmap);
            }
            mbar_arrive_expect_tx(BAR(B_QFULL), static_cast<uint32_t>(Lo::Q_BYTES));
#pragma unroll
            for (int blk = 0; blk < D / 64; ++blk)
                tma_load_3d(sQ + blk * Lo::BLK, &qmap, BAR(B_QFULL), blk * 64, g * G,
                            cu0 + tok_begin, l2_evict_first_policy());
        }
        const int ps_mask = (1 << ps_log2) - 1;
        bool ok = true;
        for (int j = 0; ok && j < n_kt; ++j) {
            const int s = j % kStages;
            const uint32_t ph = (j / kStages) & 1;
            const int key0 = j * BN;
            const int nkeys = min(BN, L - key0);  // keys of this tile that exist in pages
            for (int kv = 0; ok && kv < 2; ++kv) {
                const uint32_t full = BAR(kv ? B_VFULL(s) : B_KFULL(s));
                const uint32_t empty = BAR(kv ? B_VEMPTY(s) : B_KEMPTY(s));
                const uint32_t dst = (kv ? sV : sK) + s * Lo::KV_BYTES;
                if (j >= kStages && !mbar_wait_warp(empty, ph ^ 1, abort_flag, dev_status)) {
                    ok = false;
                    break;
                }
                if (box_rows >= 8) {
                    // one TMA box per page (or per 128-key slice of a large page) and 64-column block
                    const int nbox = (nkeys + box_rows - 1) / box_rows;  // <= 16
                    int pg = 0;
                    bool bad = false;
                    if (lane < nbox) {
                        pg = prow[(key0 + lane * box_rows) >> ps_log2];
                        bad = (pg < 0 || pg >= num_pages);
                    }
                    const unsigned badmask = __ballot_sync(0xffffffffu, bad);
                    const int nbad = __popc(badmask);
                    if (lane == 0) {
                        if (nbad) *bad_page = 1;
                        mbar_arrive_expect_tx(
                            full, static_cast<uint32_t>((nbox - nbad) * (D / 64) * box_rows * 128));
                    }
                    __syncwarp();
                    // each lane issues the boxes of its page for every column block
                    if (lane < nbox && !bad) {
                        const int kk = key0 + lane * box_rows;
                        const int row = (pg << ps_log2) + (kk & ps_mask);
#pragma unroll
                        for (int blk = 0; blk < D / 64; ++blk)
                            tma_load_3d(dst + blk * Lo::BLK + lane * box_rows * 128,
                                        kv ? &vmap : &kmap, full, blk * 64, g, row, pol_kv);
                    }
                } else {
                    // small pages: gather 16-byte chunks, swizzle, zero rows past the sequence
                    const __nv_bfloat16 *base = kv ? v_cache : k_cache;
                    bool bad = false;
                    for (int idx = lane; idx < BN * (D / 8); idx += 32) {
                        const int key = idx / (D / 8), ch = idx % (D / 8);
                        uint4 val = make_uint4(0u, 0u, 0u, 0u);
                        if (key < nkeys) {
                            const int kk = key0 + key;
                            const int pg = prow[kk >> ps_log2];
                            if (pg >= 0 && pg < num_pages) {
                                const int64_t slot = ((int64_t)pg << ps_log2) + (kk & ps_mask);
                                val = __ldg(reinterpret_cast<const uint4 *>(
                                    base + (slot * Hkv + g) * D + ch * 8));
                            } else {
                                bad = true;
                            }
                        }
                        *reinterpret_cast<uint4 *>(smem + (dst - smem_u32(smem)) +
                                                   swz_offset(key, ch, BN)) = val;
                    }
                    if (__any_sync(0xffffffffu, bad) && lane == 0) *bad_page = 1;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full);
                }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc_s = instr_desc(BM, BN, false);
        constexpr uint32_t idesc_o = instr_desc(BM, D, true);
        bool ok = mbar_wait_warp(BAR(B_QFULL), 0, abort_flag, dev_status);
        auto issue_s = [&](int j) -> bool {
            const int s = j % kStages, b = j & 1;
            if (!mbar_wait_warp(BAR(B_KFULL(s)), (j / kStages) & 1, abort_flag, dev_status)) return false;
            if (j >= 2 && !mbar_wait_warp(BAR(B_SFREE(b)), ((j - 2) >> 1) & 1, abort_flag, dev_status))
                return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kb = sK + s * Lo::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * Lo::BLK + (kk & 3) * 32;
                    umma_bf16_ss(tm_s[b], smem_desc(sQ + off, 16, 1024), smem_desc(kb + off, 16, 1024),
                                 idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(BAR(B_SFULL(b)));
                umma_commit(BAR(B_KEMPTY(s)));
            }
            __syncwarp();
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 0; ok && j < n_kt; ++j) {
            if (j + 1 < n_kt && !(ok = issue_s(j + 1))) break;
            const int s = j % kStages;
            if (!mbar_wait_warp(BAR(B_PFULL), j & 1, abort_flag, dev_status)) { ok = false; break; }
            if (!mbar_wait_warp(BAR(B_VFULL(s)), (j / kStages) & 1, abort_flag, dev_status)) { ok = false; break; }
            const uint32_t vb = sV + s * Lo::KV_BYTES;
            if (j == n_kt - 1 && (j + 1) * BN > L) {
                // keys past the sequence end hold stale pool data (maybe NaN):
                // zero those V rows so that P = 0 there contributes exactly 0
                const int first = L - j * BN;
                for (int idx = lane; idx < (BN - first) * (D / 8); idx += 32) {
                    const int key = first + idx / (D / 8), ch = idx % (D / 8);
                    *reinterpret_cast<uint4 *>(smem + (vb - smem_u32(smem)) + swz_offset(key, ch, BN)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t aoff = (kk >> 2) * Lo::BLK + (kk & 3) * 32;  // P: K-major
                    const uint32_t boff = kk * 16 * 128;                       // V: 16 keys per step
                    umma_bf16_ss(tm_o, smem_desc(sP + aoff, 16, 1024),
                                 smem_desc(vb + boff, Lo::BLK, 1024), idesc_o,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(BAR(B_ODONE));
                umma_commit(BAR(B_VEMPTY(s)));
            }
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ================================================================ softmax
        const int row = tid - 128;                 // TMEM lane == tile row
        const int wq = warp - 4;                   // TMEM lane quarter of this warp
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const int tok = tok_begin + row / G;
        const bool row_valid = tok < tok_end;
        const int lim = c + tok;                   // last key this row may see
        float m_ref = kNegBig, l_sum = 0.f;
        bool ok = true;
        // tcgen05.ld/st are warp-collective: every wait outcome is made
        // warp-uniform before the warp goes on to them.
        for (int j = 0; j < n_kt; ++j) {
            const int b = j & 1;
            ok = mbar_wait_warp(BAR(B_SFULL(b)), (j >> 1) & 1, abort_flag, dev_status);
            if (!ok) break;
            tc_fence_after();
            uint32_t sv[BN];
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) tmem_ld_32cols(tm_s[b] + lane_off + cc * 32, sv + cc * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_SFREE(b)));
            // scores in the log2 domain, masked by selection
            const int key0 = j * BN;
            float mt_max = kNegBig;
#pragma unroll
            for (int i = 0; i < BN; ++i) {
                const bool v = row_valid && (key0 + i) <= lim;
                const float x = v ? __uint_as_float(sv[i]) * scale_log2 : kNegBig;
                sv[i] = __float_as_uint(x);
                mt_max = fmaxf(mt_max, x);
            }
            const bool need = (j == 0) ? false : (mt_max > m_ref + kRescaleLog2);
            const bool warp_need = __any_sync(0xffffffffu, need);
            float alpha = 1.f;
            if (j == 0) {
                m_ref = mt_max;
            } else if (warp_need) {
                const float mn = fmaxf(m_ref, mt_max);
                alpha = ex2(m_ref - mn);
                m_ref = mn;
            }
            // probabilities, packed to bf16 pairs
            uint32_t pk[BN / 2];
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < BN; i += 2) {
                const float x0 = __uint_as_float(sv[i]), x1 = __uint_as_float(sv[i + 1]);
                const float p0 = (x0 > 0.5f * kNegBig) ? ex2(x0 - m_ref) : 0.f;
                const float p1 = (x1 > 0.5f * kNegBig) ? ex2(x1 - m_ref) : 0.f;
                rs += p0 + p1;
                pk[i / 2] = pack_bf16x2(p0, p1);
            }
            l_sum = l_sum * alpha + rs;
            // previous PV must be done before P is overwritten and O rescaled
            if (j > 0) {
                ok = mbar_wait_warp(BAR(B_ODONE), (j - 1) & 1, abort_flag, dev_status);
                if (!ok) break;
                tc_fence_after();
                if (warp_need) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        tmem_ld_32cols(tm_o + lane_off + cc * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st_32cols(tm_o + lane_off + cc * 32, ov);
                    }
                    tmem_wait_st();
                }
            }
            // P row -> shared memory, swizzled K-major (16 chunks of 8 keys)
            uint8_t *pbase = smem + Lo::OFF_P;
#pragma unroll
            for (int ch = 0; ch < BN / 8; ++ch)
                *reinterpret_cast<uint4 *>(pbase + swz_offset(row, ch, BM)) =
                    make_uint4(pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_PFULL));
        }
        if (ok) ok = mbar_wait_warp(BAR(B_ODONE), (n_kt - 1) & 1, abort_flag, dev_status);
        tc_fence_after();
        __syncthreads();
        const bool poison = (*bad_page != 0) || (*abort_flag != 0) || !ok;
        // every lane takes part in the warp-wide TMEM loads; only valid rows store
        const float inv = row_valid ? 1.f / l_sum : 0.f;
        __nv_bfloat16 *orow = out + ((int64_t)(cu0 + tok) * Hq + (int64_t)g * G + row % G) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld_32cols(tm_o + lane_off + cc * 32, ov);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float a = __uint_as_float(ov[e]) * inv, bb = __uint_as_float(ov[e + 1]) * inv;
                if (poison) a = bb = __int_as_float(0x7fc00000);
                pk[e / 2] = pack_bf16x2(a, bb);
            }
            if (row_valid) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    reinterpret_cast<uint4 *>(orow + cc * 32)[q4] =
                        make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
            }
        }
        if (poison && tid == 128 && dev_status && *bad_page) atomicOr(dev_status, PKV_DEV_BAD_PAGE);
        tc_fence_before();
        __syncthreads();
        return;
    }
    // producer, MMA and idle warps meet the softmax warps here, then free TMEM
    __syncthreads();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int G>
static bool prepare(const pkv_host::DeviceInfo &dev) {
    static std::mutex mu;
    static bool ready[64] = {};
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev.device]) {
        if (Layout<D>::bytes() > static_cast<size_t>(dev.max_smem_optin)) return false;
        if (cudaFuncSetAttribute(prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Layout<D>::bytes())) != cudaSuccess)
            return false;
        ready[dev.device] = true;
    }
    return true;
}

template <int D, int G>
static pkv_status launch(const pkv_bf16 *q, const int32_t *cu, const pkv_bf16 *k_cache,
                         const pkv_bf16 *v_cache, const int32_t *page_table, int64_t pt_stride,
                         const int32_t *seq_lens, int B, int64_t Tq, int max_q_len, int Hkv,
                         int page_size, int64_t num_pages, float scale, int32_t *dev_status,
                         pkv_bf16 *out, cudaStream_t stream) {
    pkv_host::DeviceInfo dev;
    if (!pkv_host::current_device(&dev)) return PKV_ECUDA;
    if (!prepare<D, G>(dev)) return PKV_ECUDA;
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
        kmap = qmap;  // unused: small pages are gathered by the producer's lanes
        vmap = qmap;
    }
    int ps_log2 = 0;
    while ((1 << ps_log2) < page_size) ++ps_log2;
    const int mtiles = (max_q_len + TOK - 1) / TOK;
    const int64_t grid = static_cast<int64_t>(mtiles) * B * Hkv;
    if (grid == 0) return PKV_OK;
    if (grid > 0x7fffffffll) return PKV_EUNSUPPORTED;
    prefill_kernel<D, G><<<static_cast<unsigned>(grid), kThreads, Layout<D>::bytes(), stream>>>(
        qmap, kmap, vmap, reinterpret_cast<const __nv_bfloat16 *>(k_cache),
        reinterpret_cast<const __nv_bfloat16 *>(v_cache), cu, page_table, pt_stride, seq_lens, B, Tq,
        max_q_len, Hkv, ps_log2, box_rows, num_pages, scale * kLog2e, mtiles, dev_status,
        reinterpret_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace prefill
}  // namespace pkv

extern "C" pkv_status pkv_paged_prefill_attn(const pkv_bf16 *q, const int32_t *cu_seqlens_q,
                                             const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                             const int32_t *page_table, int64_t page_table_stride,
                                             const int32_t *seq_lens, int batch,
                                             int64_t total_q_tokens, int max_q_len,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int page_size, int64_t num_pages, float softmax_scale,
                                             int32_t *dev_status, pkv_bf16 *out, void *stream) {
    using namespace pkv::prefill;
    if (batch < 0 || total_q_tokens < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_pages <= 0 || page_table_stride < 0 || page_size <= 0)
        return PKV_EINVAL;
    if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
    if (!(softmax_scale == softmax_scale)) return PKV_EINVAL;
    if (batch == 0 || total_q_tokens == 0 || max_q_len == 0) return PKV_OK;
    if (!q || !cu_seqlens_q || !k_cache || !v_cache || !page_table || !seq_lens || !out)
        return PKV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    if (head_dim != 64 && head_dim != 128) return PKV_EUNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_EUNSUPPORTED;
    if ((page_size & (page_size - 1)) != 0 || page_size > 256) return PKV_EUNSUPPORTED;
    if (!pkv_host::aligned16(q) || !pkv_host::aligned16(k_cache) || !pkv_host::aligned16(v_cache) ||
        !pkv_host::aligned16(out))
        return PKV_EINVAL;
    if (num_pages * page_size > 0x7fffffffll || total_q_tokens > 0x7fffffffll)
        return PKV_EUNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#define PKV_PREFILL_CASE(DD, GG)                                                                   \
    if (head_dim == DD && G == GG)                                                                 \
        return launch<DD, GG>(q, cu_seqlens_q, k_cache, v_cache, page_table, page_table_stride,    \
                              seq_lens, batch, total_q_tokens, max_q_len, num_kv_heads, page_size, \
                              num_pages, softmax_scale, dev_status, out, st);
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

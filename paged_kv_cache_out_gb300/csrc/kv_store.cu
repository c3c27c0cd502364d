// kv_store.cu -- scatter of this step's new K/V rows into their pool slots.
//
// mini-sglang "Engine Class" (forward_batch: the batch carries out_loc) and
// miniVLLM "Engine Architecture" (slot_mapping: the physical cache slot of
// each new token; allocate_kv_cache: pool layout [pages, page_size, kv_heads,
// head_dim]).  A row is num_kv_heads * head_dim bf16 (2 KB for 8 x 128), moved
// as 16-byte vectors: one warp per (token, K-or-V) row, every lane issuing all
// of its loads before its stores.
#include "common.cuh"

namespace pkv {

constexpr int kStoreThreads = 256;
constexpr int kStoreMaxVecPerLane = 8;  // rows up to 32 * 8 * 16 B = 4 KB in one pass

__global__ void __launch_bounds__(kStoreThreads) kv_store_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int32_t *__restrict__ out_loc, int64_t num_tokens, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, int64_t num_slots, int row_vecs, int32_t *dev_status) {
    grid_dependency_wait();  // inputs may come from the kernel before this one
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kStoreThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kStoreThreads) >> 5;
    for (int64_t w = warp; w < 2 * num_tokens; w += nwarps) {
        const int64_t t = w >> 1;
        const bool is_v = (w & 1) != 0;
        const int64_t slot = out_loc[t];
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (lane == 0 && !is_v && dev_status) atomicOr(dev_status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const uint4 *src = (is_v ? v_new : k_new) + t * row_vecs;
        uint4 *dst = (is_v ? v_cache : k_cache) + slot * row_vecs;
        for (int base = 0; base < row_vecs; base += 32 * kStoreMaxVecPerLane) {
            uint4 buf[kStoreMaxVecPerLane];
#pragma unroll
            for (int i = 0; i < kStoreMaxVecPerLane; ++i) {
                const int idx = base + i * 32 + lane;
                if (idx < row_vecs) buf[i] = __ldg(src + idx);
            }
#pragma unroll
            for (int i = 0; i < kStoreMaxVecPerLane; ++i) {
                const int idx = base + i * 32 + lane;
                if (idx < row_vecs) dst[idx] = buf[i];
            }
        }
    }
}

}  // namespace pkv

extern "C" pkv_status pkv_kv_store(const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                   const int32_t *out_loc, int64_t num_tokens,
                                   pkv_bf16 *k_cache, pkv_bf16 *v_cache, int64_t num_pages,
                                   int page_size, int num_kv_heads, int head_dim,
                                   int32_t *dev_status, void *stream) {
    if (num_tokens < 0 || num_pages < 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_EINVAL;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !out_loc || !k_cache || !v_cache) return PKV_EINVAL;
    if ((static_cast<int64_t>(num_kv_heads) * head_dim * 2) % 16 != 0) return PKV_EUNSUPPORTED;
    if (!pkv_host::aligned16(k_new) || !pkv_host::aligned16(v_new) ||
        !pkv_host::aligned16(k_cache) || !pkv_host::aligned16(v_cache))
        return PKV_EINVAL;
    pkv_host::DeviceInfo dev;
    if (!pkv_host::current_device(&dev)) return PKV_ECUDA;
    const int row_vecs = num_kv_heads * head_dim * 2 / 16;
    const int64_t warps_needed = 2 * num_tokens;
    const int64_t blocks_needed =
        (warps_needed + pkv::kStoreThreads / 32 - 1) / (pkv::kStoreThreads / 32);
    const int64_t max_blocks = static_cast<int64_t>(dev.sm_count) * 8;
    const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
    const cudaError_t err = pkv_host::launch_dependent(
        pkv::kv_store_kernel, dim3(blocks), dim3(pkv::kStoreThreads), 0,
        static_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(k_new),
        reinterpret_cast<const uint4 *>(v_new), out_loc, num_tokens,
        reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
        num_pages * page_size, row_vecs, dev_status);
    return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// decode_noalloc.cu -- decode attention whose scratch lives in a fixed device
// array owned by the library, for callers that cannot allocate a workspace.
//
// The scratch array below is declared at file scope; every GPU that loads the
// library holds PKV_NOALLOC_SCRATCH_BYTES for it until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device with that
// device current, and that address is what the kernels receive.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on error).
void *scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
    const int32_t *page_table, int64_t page_table_stride, const int32_t *seq_lens, int batch,
    int num_q_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float softmax_scale, int32_t *dev_status, pkv_bf16 *out, void *stream) {
    // every argument and shape check runs first, as in pkv_paged_decode_attn;
    // then sizes beyond the scratch array are rejected and its address looked up
    static const pkv_host::Scratch scratch{static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES),
                                           &scratch_for_current_device};
    return pkv_host::decode_with_scratch(q, k_cache, v_cache, page_table, page_table_stride,
                                         seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                                         page_size, num_pages, softmax_scale, dev_status, out,
                                         stream, scratch);
}

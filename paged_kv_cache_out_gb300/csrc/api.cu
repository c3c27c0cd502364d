// api.cu -- host-side pieces shared by every entry point: status strings,
// the cached device properties and the TMA tensor-map encoders.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_EINVAL: return "invalid argument";
        case PKV_EUNSUPPORTED: return "unsupported shape";
        case PKV_ECUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

extern "C" int pkv_version(void) { return 100; }

namespace pkv_host {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}
}  // namespace

bool current_device(DeviceInfo *info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (d.device != dev) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return false;
        d.sm_count = sms;
        d.max_smem_optin = smem;
        d.device = dev;
    }
    *info = d;
    return true;
}

bool encode_kv_map(CUtensorMap *map, const void *base, int64_t num_slots, int num_kv_heads,
                   int head_dim, int box_inner, int box_rows, bool swizzle128) {
    auto enc = encoder();
    if (!enc || num_slots <= 0 || num_slots > 0xffffffffll) return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)num_slots};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)head_dim * num_kv_heads * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    // L2 promotion no wider than one head's row: the rows of one head are
    // num_kv_heads * head_dim * 2 bytes apart, so a wider promotion would
    // fetch the neighbouring head's row, which this copy does not use
    const CUtensorMapL2promotion promo = head_dim * 2 >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                                             : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap *map, const void *base, int64_t rows, int head_dim) {
    auto enc = encoder();
    // row coordinates of a gather are 32-bit signed
    if (!enc || rows <= 0 || rows > 0x7fffffffll) return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {(cuuint32_t)head_dim, 1u};
    cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapL2promotion promo = head_dim * 2 >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                                             : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *map, const void *base, int64_t tokens, int num_q_heads,
                  int head_dim, int box_heads, int box_tokens) {
    auto enc = encoder();
    if (!enc || tokens <= 0 || tokens > 0xffffffffll) return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)head_dim * num_q_heads * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pkv_host

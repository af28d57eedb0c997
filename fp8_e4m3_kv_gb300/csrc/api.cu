// api.cu -- host-side parts of libfp8kv shared by every entry point: status
// text, the scale rules, the device gate, the device error word and the
// tensor maps over the paged cache.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace fp8kv {

// One error word per device (each device that loads the library gets its
// own copy of this variable).
__device__ uint32_t g_error_word;

namespace {
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool probed = false;
    fp8kv_status status = FP8KV_ERR_UNSUPPORTED;
    int num_sms = 0;
    uint32_t *error_word = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;
}  // namespace

static DeviceInfo *current_device_info() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_devices_mu);
    DeviceInfo &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        d.num_sms = sms;
        // The kernels are built for sm_103a only (GB300).
        d.status = (major == 10 && minor == 3) ? FP8KV_OK : FP8KV_ERR_UNSUPPORTED;
        if (d.status == FP8KV_OK) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
                cudaGetLastError();
                d.status = FP8KV_ERR_LAUNCH;
            } else {
                d.error_word = static_cast<uint32_t *>(p);
            }
        }
        d.probed = true;
    }
    return &d;
}

fp8kv_status check_device(int *num_sms) {
    DeviceInfo *d = current_device_info();
    if (!d) return FP8KV_ERR_LAUNCH;
    if (num_sms) *num_sms = d->num_sms;
    return d->status;
}

uint32_t *device_error_word() {
    DeviceInfo *d = current_device_info();
    return d ? d->error_word : nullptr;
}

bool scale_ok(float s) { return isfinite(s) && s > 0.0f; }

bool func_attrs_once(const void *func, std::atomic<uint64_t> *done, int smem_bytes,
                     bool max_carveout) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return false;
    }
    const uint64_t bit = 1ull << dev;
    if (done->load(std::memory_order_acquire) & bit) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess ||
        (max_carveout && cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                              cudaSharedmemCarveoutMaxShared) != cudaSuccess)) {
        cudaGetLastError();
        return false;
    }
    done->fetch_or(bit, std::memory_order_release);
    return true;
}

// The driver's tensor-map encoder, looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode_tiled;
}

bool make_rows_map(CUtensorMap *map, const void *base, int64_t rows, int heads, int head_dim) {
    if (!encode_tiled() || rows < 1 || rows > (1ll << 31) - 1 || heads < 1 || head_dim < 64)
        return false;
    // x[row][head][d] as (d, head, row); one box is 32 rows of one head's
    // first or second 64 values (128 bytes each)
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
    const cuuint32_t box[3] = {64u, 1u, 32u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_cache_map(CUtensorMap *map, const uint8_t *base, int64_t num_blocks, int block_size,
                    int num_kv_heads, int head_dim) {
    if (!encode_tiled()) return false;
    // The map depends only on the arguments: the last few are kept per host
    // thread, so a decode loop over the same cache encodes it once.
    struct Entry {
        const uint8_t *base;
        int64_t num_blocks;
        int block_size, num_kv_heads, head_dim;
        CUtensorMap map;
    };
    constexpr int kEntries = 4;
    thread_local Entry entries[kEntries];
    thread_local int n_entries = 0, next = 0;
    for (int i = 0; i < n_entries; ++i) {
        const Entry &e = entries[i];
        if (e.base == base && e.num_blocks == num_blocks && e.block_size == block_size &&
            e.num_kv_heads == num_kv_heads && e.head_dim == head_dim) {
            *map = e.map;
            return true;
        }
    }
    // cache[block][head][row][d] as (d, row, head, block); one box is one
    // head's block_size rows x 128 bytes, a contiguous run of the cache
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)block_size,
                                (cuuint64_t)num_kv_heads, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim, (cuuint64_t)block_size * head_dim,
                                   (cuuint64_t)num_kv_heads * block_size * head_dim};
    const cuuint32_t box[4] = {128u, (cuuint32_t)block_size, 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    Entry &e = entries[next];
    e.base = base;
    e.num_blocks = num_blocks;
    e.block_size = block_size;
    e.num_kv_heads = num_kv_heads;
    e.head_dim = head_dim;
    e.map = *map;
    next = (next + 1) % kEntries;
    if (n_entries < kEntries) ++n_entries;
    return true;
}

}  // namespace fp8kv

extern "C" {

const char *fp8kv_status_string(fp8kv_status s) {
    switch (s) {
        case FP8KV_OK: return "ok";
        case FP8KV_ERR_ARG: return "invalid argument";
        case FP8KV_ERR_SCALE: return "scale not finite and positive";
        case FP8KV_ERR_UNSUPPORTED: return "unsupported device or shape";
        case FP8KV_ERR_WORKSPACE: return "workspace missing or too small";
        case FP8KV_ERR_LAUNCH: return "CUDA launch or runtime error";
        case FP8KV_ERR_DEVICE: return "device error word set";
    }
    return "unknown status";
}

fp8kv_status fp8kv_scale_from_amax(float amax, int32_t rule, float *scale) {
    if (!scale || rule < 0 || rule > 2) return FP8KV_ERR_ARG;
    if (!(amax >= 0.0f) || !isfinite(amax)) return FP8KV_ERR_SCALE;
    float s;
    if (rule == 0) {
        s = amax / fp8kv::kE4M3Max;
    } else if (rule == 1) {
        float t = amax / fp8kv::kE4M3Max;
        uint32_t u;
        memcpy(&u, &t, sizeof u);
        if (u & 0xFFFFu) u = (u & 0xFFFF0000u) + 0x10000u;   // round up to a bf16 value
        memcpy(&s, &u, sizeof s);
    } else {
        double r = static_cast<double>(amax) * 1.3 / 448.0;
        s = static_cast<float>(r > 1.0 ? r : 1.0);
    }
    if (!fp8kv::scale_ok(s)) return FP8KV_ERR_SCALE;
    *scale = s;
    return FP8KV_OK;
}

size_t fp8kv_cache_bytes(int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim) {
    if (num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    return static_cast<size_t>(num_blocks) * block_size * num_kv_heads * head_dim;
}

fp8kv_status fp8kv_device_error(uint32_t *flags, int32_t clear) {
    if (!flags) return FP8KV_ERR_ARG;
    fp8kv_status st = fp8kv::check_device(nullptr);
    if (st != FP8KV_OK) return st;
    uint32_t *w = fp8kv::device_error_word();
    if (!w) return FP8KV_ERR_LAUNCH;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    if (cudaMemcpy(flags, w, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    if (clear && cudaMemset(w, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    return FP8KV_OK;
}

}  // extern "C"

// abi.cu -- status strings, per-thread last error, device queries and the TMA
// tensor-map encoder of libsparsepool.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace {

thread_local char g_last_error[512] = "";

constexpr int kMaxDevices = 64;
sp_host::DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices];
std::mutex g_info_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

// cuCtxGetCurrent / cuCtxGetId, for keying per-context caches (a context's id is unique
// for the life of the process, unlike its handle or the device ordinal).
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_queries()
{
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

void load_encoder()
{
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

namespace sp_host {

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_status(cudaError_t e, const char *what)
{
    if (e == cudaSuccess)
        return SPARSE_OK;
    return fail(SPARSE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(SPARSE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (!g_info_valid[dev]) {
        DeviceInfo d{dev, 0, 0};
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaDeviceGetAttribute");
        g_info[dev] = d;
        g_info_valid[dev] = true;
    }
    *out = g_info[dev];
    return SPARSE_OK;
}

int current_context_id(unsigned long long *id)
{
    std::call_once(g_ctx_once, load_ctx_queries);
    if (g_ctx_current == nullptr || g_ctx_id == nullptr)
        return fail(SPARSE_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable");
    CUcontext ctx = nullptr;
    CUresult r = g_ctx_current(&ctx);
    if (r == CUDA_SUCCESS && ctx == nullptr) {
        // no context current on this host thread yet: the runtime makes the device's
        // primary context current (a no-op call that initialises it), then look again
        const cudaError_t e = cudaFree(nullptr);
        if (e != cudaSuccess)
            return cuda_status(e, "making the primary context current");
        r = g_ctx_current(&ctx);
    }
    if (r != CUDA_SUCCESS || ctx == nullptr)
        return fail(SPARSE_ERR_CUDA, "cuCtxGetCurrent failed (CUresult %d)", static_cast<int>(r));
    unsigned long long v = 0;
    r = g_ctx_id(ctx, &v);
    if (r != CUDA_SUCCESS)
        return fail(SPARSE_ERR_CUDA, "cuCtxGetId failed (CUresult %d)", static_cast<int>(r));
    *id = v;
    return SPARSE_OK;
}

int configure_kernel(const void *func, int dyn_smem, int device, int *configured)
{
    if (device < 0 || device >= kMaxDevices)
        return fail(SPARSE_ERR_UNSUPPORTED, "device ordinal %d out of range", device);
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (configured[device] >= dyn_smem + 1)
        return SPARSE_OK;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaFuncSetAttribute");
    configured[device] = dyn_smem + 1;
    return SPARSE_OK;
}

int make_kv_tensor_map(CUtensorMap *map, const void *base, long long rows_per_pair, long long pairs)
{
    std::call_once(g_encode_once, load_encoder);
    if (g_encode == nullptr)
        return fail(SPARSE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                    cudaGetErrorString(g_encode_err));
    if (rows_per_pair <= 0 || pairs <= 0 || rows_per_pair > (1LL << 32) || pairs > (1LL << 32))
        return fail(SPARSE_ERR_UNSUPPORTED, "tensor map extent out of range");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(sp::kD), static_cast<cuuint64_t>(rows_per_pair),
                                static_cast<cuuint64_t>(pairs)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(sp::kD) * 2,
                                   static_cast<cuuint64_t>(rows_per_pair) * sp::kD * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(sp::kBlk), 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SPARSE_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return SPARSE_OK;
}

}  // namespace sp_host

extern "C" {

SPARSE_API const char *sparse_status_string(int status)
{
    switch (status) {
    case SPARSE_OK:
        return "ok";
    case SPARSE_ERR_INVALID_ARG:
        return "invalid argument";
    case SPARSE_ERR_UNSUPPORTED:
        return "unsupported size or configuration";
    case SPARSE_ERR_CUDA:
        return "CUDA runtime error";
    case SPARSE_ERR_TIMEOUT:
        return "a bounded device wait timed out";
    case SPARSE_ERR_NOT_READY:
        return "staging slot not marked ready";
    case SPARSE_ERR_BAD_INDEX:
        return "block id outside the cache (skipped)";
    default:
        return "unknown status";
    }
}

SPARSE_API const char *sparse_last_error(void)
{
    return g_last_error;
}

SPARSE_API int sparse_version(void)
{
    return 100;  // 0.1.0
}

}  // extern "C"

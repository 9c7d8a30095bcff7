// gather.cu -- stage the selected blocks of an offloaded KV cache into HBM.
//
// SparDA notes §4.5: the full KV cache lives in pinned host memory and the blocks
// chosen for the next layer are pulled into a GPU staging buffer while the current
// layer computes.  The pages use a persistent Triton kernel fed by a UVA queue; here
// the indices are already on the device (written by sparse_select_topk), so a plain
// gather kernel on a copy stream reads the mapped host memory directly with 16-byte
// loads (no host round trip, no per-block copy calls) and writes ring slot i of every
// pair.  Each CTA then publishes one release-add on the ready word.
#include "common.cuh"

namespace {

using namespace sp;

constexpr int kThreads = 256;
constexpr int kVecPerRow = kD * 2 / 16;                 // 16 x 16-byte chunks per token row
constexpr int kVecPerBlock = kBlk * kVecPerRow;         // 1024 per block per tensor
constexpr int kPerThread = kVecPerBlock / kThreads;     // 4

struct GatherParams {
    const uint16_t *k_host;
    const uint16_t *v_host;
    const int *idx;
    const int *count;
    uint16_t *k_ring;
    uint16_t *v_ring;
    unsigned *ready_flag;
    int *status;
    long long T_host;
    int k_tot;
    int n_pairs;
};

__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherParams p)
{
    const int tid = threadIdx.x;
    const long long n_items = static_cast<long long>(p.n_pairs) * p.k_tot;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int pair = static_cast<int>(item / p.k_tot);
        const int i = static_cast<int>(item - static_cast<long long>(pair) * p.k_tot);
        int cnt = p.count[pair];
        cnt = cnt < 0 ? 0 : (cnt > p.k_tot ? p.k_tot : cnt);
        if (i >= cnt)
            continue;
        const int j = p.idx[static_cast<size_t>(pair) * p.k_tot + i];
        const bool valid = j >= 0 && static_cast<long long>(j) * kBlk < p.T_host;
        if (!valid && tid == 0)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        const size_t src_row0 = static_cast<size_t>(pair) * p.T_host + (valid ? static_cast<size_t>(j) * kBlk : 0);
        const size_t dst_row0 = (static_cast<size_t>(pair) * p.k_tot + i) * kBlk;
        uint4 kv[kPerThread], vv[kPerThread];
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            const int e = tid + u * kThreads;
            const int row = e / kVecPerRow, c = e % kVecPerRow;
            const bool in = valid && static_cast<long long>(j) * kBlk + row < p.T_host;
            const size_t off = (src_row0 + row) * kD + c * 8;
            kv[u] = in ? *reinterpret_cast<const uint4 *>(p.k_host + off) : make_uint4(0, 0, 0, 0);
            vv[u] = in ? *reinterpret_cast<const uint4 *>(p.v_host + off) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            const int e = tid + u * kThreads;
            const int row = e / kVecPerRow, c = e % kVecPerRow;
            const size_t off = (dst_row0 + row) * kD + c * 8;
            *reinterpret_cast<uint4 *>(p.k_ring + off) = kv[u];
            *reinterpret_cast<uint4 *>(p.v_ring + off) = vv[u];
        }
    }
    if (p.ready_flag != nullptr) {
        __threadfence();
        __syncthreads();
        if (tid == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.ready_flag) : "memory");
    }
}

}  // namespace

extern "C" SPARSE_API int sparse_gather_offloaded(const uint16_t *k_host, const uint16_t *v_host, long long T_host,
                                                  const int *idx, const int *count, int k_tot, int B, int H_kv,
                                                  uint16_t *k_ring, uint16_t *v_ring, unsigned *ready_flag,
                                                  int n_ctas, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!k_host || !v_host || !idx || !count || !k_ring || !v_ring)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_gather_offloaded: null pointer");
    if (!aligned16(k_host) || !aligned16(v_host) || !aligned16(k_ring) || !aligned16(v_ring))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_gather_offloaded: buffers must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || k_tot < 1 || T_host < 1 || n_ctas < 0 || n_ctas > 1024)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_gather_offloaded: bad size");
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > (1LL << 30))
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_gather_offloaded: too many pairs");
    // Resolve the source pointers on the host: pinned (mapped) host memory gives its
    // device address, device or managed memory is used as is, and unregistered host
    // memory is accepted only where the GPU can read pageable memory.  Anything else
    // is rejected here rather than faulting on the device.
    const uint16_t *src[2] = {k_host, v_host};
    for (int i = 0; i < 2; ++i) {
        cudaPointerAttributes a;
        cudaError_t e = cudaPointerGetAttributes(&a, src[i]);
        if (e != cudaSuccess)
            return sp_host::cuda_status(e, "sparse_gather_offloaded: cudaPointerGetAttributes");
        if (a.type == cudaMemoryTypeHost) {
            if (a.devicePointer == nullptr)
                return fail(SPARSE_ERR_INVALID_ARG, "sparse_gather_offloaded: host buffer is not mapped");
            src[i] = static_cast<const uint16_t *>(a.devicePointer);
        } else if (a.type == cudaMemoryTypeUnregistered) {
            int dev = 0, pageable = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
                !pageable)
                return fail(SPARSE_ERR_INVALID_ARG,
                            "sparse_gather_offloaded: source is neither pinned nor device memory");
        }
    }
    if (n_ctas == 0) {
        sp_host::DeviceInfo dev;
        int rc = sp_host::device_info(&dev);
        if (rc != SPARSE_OK)
            return rc;
        n_ctas = dev.sm_count;
    }
    GatherParams p{src[0], src[1], idx, count, k_ring, v_ring, ready_flag, status, T_host, k_tot,
                   static_cast<int>(pairs)};
    {
        sp_host::DeviceInfo dinfo;
        int rc0 = sp_host::device_info(&dinfo);
        static int configured[64];
        if (rc0 == SPARSE_OK)
            rc0 = sp_host::configure_kernel(reinterpret_cast<const void *>(gather_kernel), 0, dinfo.device, configured);
        if (rc0 != SPARSE_OK)
            return rc0;
    }
    gather_kernel<<<n_ctas, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return sp_host::cuda_status(cudaGetLastError(), "sparse_gather_offloaded launch");
}

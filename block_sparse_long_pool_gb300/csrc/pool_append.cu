// pool_append.cu -- append tokens to the K/V caches and keep the compressed keys.
//
// SparDA notes §4.2 Alg.1 step 1: new K/V rows are appended and the compressed key
// cache is updated by mean pooling at O(d) cost per touched block (background
// eq.(4), one mean per 64-token block).  The running mean of block j becomes
//     ktil_j <- (n_old * ktil_j + sum of the new keys in j) / n_total.
// sparse_pool_append_kv keeps the compressed values the same way (the pooled value
// rows of NSA's compressed branch, SSV notes' NSA math step 4) and, optionally, bf16
// copies of the touched compressed key and value rows: the rows that the compressed
// branch's tensor-core attention reads.
//
// One CTA per (touched block, pair): 16 threads cover the 16 sixteen-byte chunks of
// a 256-byte token row, 16 rows per pass; each thread copies its rows of K and V
// with 16-byte loads/stores and sums its 8 key dimensions in fp32.
#include <limits.h>

#include "common.cuh"

namespace {

using namespace sp;

constexpr int kThreads = 256;

struct AppendParams {
    uint16_t *k_cache;
    uint16_t *v_cache;
    float *ktil;
    float *vtil;        // pooled values, or null
    uint16_t *khat;     // bf16 copies of the touched ktil rows, or null
    uint16_t *vhat;     // bf16 copies of the touched vtil rows, or null
    const uint16_t *k_new;
    const uint16_t *v_new;
    long long T_cap;
    long long len_before;
    int N_cap;
    int n_new;
    int first_block;
};

__global__ void __launch_bounds__(kThreads) pool_append_kernel(const AppendParams p)
{
    __shared__ float red[16][kD + 4];
    __shared__ float redv[16][kD + 4];
    griddep_wait();                // the new rows may be the preceding kernel's output
    griddep_launch_dependents();   // the next kernel may be scheduled now; it waits for this one

    const int pair = blockIdx.y;
    const int j = p.first_block + static_cast<int>(blockIdx.x);
    const long long len_after = p.len_before + p.n_new;
    const long long blk0 = static_cast<long long>(j) * kBlk;
    const long long t_begin = blk0 > p.len_before ? blk0 : p.len_before;
    const long long t_end = (blk0 + kBlk) < len_after ? (blk0 + kBlk) : len_after;
    long long n_old_ll = p.len_before - blk0;
    n_old_ll = n_old_ll < 0 ? 0 : (n_old_ll > kBlk ? kBlk : n_old_ll);
    const int n_old = static_cast<int>(n_old_ll);
    const int n_total = static_cast<int>(t_end - blk0);

    const int c = threadIdx.x & 15;   // 16-byte chunk: dims 8c .. 8c+7
    const int r0 = threadIdx.x >> 4;  // row phase 0..15

    const size_t cache_base = static_cast<size_t>(pair) * static_cast<size_t>(p.T_cap) * kD;
    const size_t new_base = static_cast<size_t>(pair) * static_cast<size_t>(p.n_new) * kD;

    float acc[8], accv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc[i] = 0.f;
        accv[i] = 0.f;
    }

    for (long long t = t_begin + r0; t < t_end; t += 16) {
        const size_t src = new_base + static_cast<size_t>(t - p.len_before) * kD + c * 8;
        const size_t dst = cache_base + static_cast<size_t>(t) * kD + c * 8;
        const uint4 kv = *reinterpret_cast<const uint4 *>(p.k_new + src);
        const uint4 vv = *reinterpret_cast<const uint4 *>(p.v_new + src);
        *reinterpret_cast<uint4 *>(p.k_cache + dst) = kv;
        *reinterpret_cast<uint4 *>(p.v_cache + dst) = vv;
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&kv);
        const __nv_bfloat162 *hv = reinterpret_cast<const __nv_bfloat162 *>(&vv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            acc[2 * i] += f.x;
            acc[2 * i + 1] += f.y;
            const float2 fv = __bfloat1622float2(hv[i]);
            accv[2 * i] += fv.x;
            accv[2 * i + 1] += fv.y;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        red[r0][c * 8 + i] = acc[i];
        redv[r0][c * 8 + i] = accv[i];
    }
    __syncthreads();

    if (threadIdx.x < kD) {
        const int d = threadIdx.x;
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            s += red[r][d];
        const size_t at = (static_cast<size_t>(pair) * p.N_cap + j) * kD + d;
        const float prev = n_old > 0 ? p.ktil[at] * static_cast<float>(n_old) : 0.f;
        const float mean = (prev + s) / static_cast<float>(n_total);
        p.ktil[at] = mean;
        if (p.khat != nullptr)
            p.khat[at] = __bfloat16_as_ushort(__float2bfloat16_rn(mean));
    } else if (p.vtil != nullptr && threadIdx.x < 2 * kD) {
        const int d = threadIdx.x - kD;
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            s += redv[r][d];
        const size_t at = (static_cast<size_t>(pair) * p.N_cap + j) * kD + d;
        const float prev = n_old > 0 ? p.vtil[at] * static_cast<float>(n_old) : 0.f;
        const float mean = (prev + s) / static_cast<float>(n_total);
        p.vtil[at] = mean;
        if (p.vhat != nullptr)
            p.vhat[at] = __bfloat16_as_ushort(__float2bfloat16_rn(mean));
    }
}

}  // namespace

namespace {

// One launch of a kThreads-thread kernel taking one parameter struct, with programmatic
// stream serialization: it may be scheduled while the kernel before it drains (it waits
// for that kernel itself), and it lets the kernel after it do the same.
template <typename Params>
cudaError_t launch_pdl(const void *kern, dim3 grid, const Params *prm, void *stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<Params *>(prm)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

int append_impl(const char *name, uint16_t *k_cache, uint16_t *v_cache, float *ktil, float *vtil,
                uint16_t *khat, uint16_t *vhat, const uint16_t *k_new, const uint16_t *v_new, int B, int H_kv,
                long long T_cap, int N_cap, long long len_before, int n_new, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!k_cache || !v_cache || !ktil || !k_new || !v_new)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(ktil) || !aligned16(k_new) ||
        !aligned16(v_new) || (vtil != nullptr && !aligned16(vtil)) || (khat != nullptr && !aligned16(khat)) ||
        (vhat != nullptr && !aligned16(vhat)))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || n_new < 1 || len_before < 0 || T_cap < 1 || N_cap < 1)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size (B=%d H_kv=%d n_new=%d len=%lld)", name,
                    B, H_kv, n_new, len_before);
    const long long len_after = len_before + n_new;
    if (len_after > T_cap)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: %lld tokens exceed T_cap=%lld", name, len_after,
                    T_cap);
    if ((len_after + kBlk - 1) / kBlk > N_cap)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: %lld tokens need more than N_cap=%d blocks", name,
                    len_after, N_cap);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: B*H_kv=%lld > 65535", name, pairs);
    const int first_block = static_cast<int>(len_before / kBlk);
    const int last_block = static_cast<int>((len_after - 1) / kBlk);
    AppendParams p{k_cache, v_cache, ktil, vtil, khat, vhat, k_new, v_new, T_cap, len_before, N_cap, n_new, first_block};
    dim3 grid(static_cast<unsigned>(last_block - first_block + 1), static_cast<unsigned>(pairs));
    {
        sp_host::DeviceInfo dinfo;
        int rc0 = sp_host::device_info(&dinfo);
        static int configured[64];
        if (rc0 == SPARSE_OK)
            rc0 = sp_host::configure_kernel(reinterpret_cast<const void *>(pool_append_kernel), 0, dinfo.device, configured);
        if (rc0 != SPARSE_OK)
            return rc0;
    }
    return sp_host::cuda_status(launch_pdl(reinterpret_cast<const void *>(pool_append_kernel), grid, &p, stream),
                                name);
}

}  // namespace

extern "C" SPARSE_API int sparse_pool_append(uint16_t *k_cache, uint16_t *v_cache, float *ktil,
                                             const uint16_t *k_new, const uint16_t *v_new, int B,
                                             int H_kv, long long T_cap, int N_cap,
                                             long long len_before, int n_new, void *stream)
{
    return append_impl("sparse_pool_append", k_cache, v_cache, ktil, nullptr, nullptr, nullptr, k_new, v_new, B,
                       H_kv, T_cap, N_cap, len_before, n_new, stream);
}

extern "C" SPARSE_API int sparse_pool_append_kv(uint16_t *k_cache, uint16_t *v_cache, float *ktil, float *vtil,
                                                uint16_t *khat, uint16_t *vhat, const uint16_t *k_new,
                                                const uint16_t *v_new, int B, int H_kv, long long T_cap, int N_cap,
                                                long long len_before, int n_new, void *stream)
{
    if (vtil == nullptr)
        return sp_host::fail(SPARSE_ERR_INVALID_ARG, "sparse_pool_append_kv: null vtil");
    return append_impl("sparse_pool_append_kv", k_cache, v_cache, ktil, vtil, khat, vhat, k_new, v_new, B, H_kv,
                       T_cap, N_cap, len_before, n_new, stream);
}

// ---------------------------------------------------------------- overlapping compression
//
// NSA's compressed rows with an overlapping kernel (SparDA notes, background eq.(4) with
// the inference kernel l = 32 and stride s = 16 of §4.4; SSV notes, "NSA" branch 1):
//     khat[p][j] = mean of K[p][s*j .. s*j + l),  vhat likewise,
// for every window completed by the tokens [len_before, len_before + n_new) (a window is
// compressed once its last token is in the cache).  One CTA per (new window, pair):
// 16 threads per 16-byte chunk of a row, 16 rows per pass, fp32 sums, the mean rounded
// once to bf16.

namespace {

struct CompressParams {
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    uint16_t *khat;
    uint16_t *vhat;
    long long T_cap;
    int n_rows_cap;
    int cmp_len;
    int cmp_stride;
    int first_row;
};

__global__ void __launch_bounds__(kThreads) compress_windows_kernel(const CompressParams p)
{
    __shared__ float red[2][16][kD + 4];
    griddep_wait();                // the cache rows may be the preceding kernel's output
    griddep_launch_dependents();   // the next kernel may be scheduled now; it waits for this one
    const int pair = blockIdx.y;
    const int j = p.first_row + static_cast<int>(blockIdx.x);
    const int c = threadIdx.x & 15;   // dims 8c .. 8c+7
    const int r0 = threadIdx.x >> 4;  // row phase
    const size_t base = static_cast<size_t>(pair) * static_cast<size_t>(p.T_cap) * kD;
    const long long t0 = static_cast<long long>(p.cmp_stride) * j;
    float ak[8], av[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        ak[i] = av[i] = 0.f;
    for (long long t = t0 + r0; t < t0 + p.cmp_len; t += 16) {
        const size_t at = base + static_cast<size_t>(t) * kD + c * 8;
        const uint4 kv = *reinterpret_cast<const uint4 *>(p.k_cache + at);
        const uint4 vv = *reinterpret_cast<const uint4 *>(p.v_cache + at);
        const __nv_bfloat162 *hk = reinterpret_cast<const __nv_bfloat162 *>(&kv);
        const __nv_bfloat162 *hv = reinterpret_cast<const __nv_bfloat162 *>(&vv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 fk = __bfloat1622float2(hk[i]);
            const float2 fv = __bfloat1622float2(hv[i]);
            ak[2 * i] += fk.x;
            ak[2 * i + 1] += fk.y;
            av[2 * i] += fv.x;
            av[2 * i + 1] += fv.y;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        red[0][r0][c * 8 + i] = ak[i];
        red[1][r0][c * 8 + i] = av[i];
    }
    __syncthreads();
    const int x = threadIdx.x / kD, d = threadIdx.x % kD;   // x = 0: keys, 1: values
    if (x < 2) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            sum += red[x][r][d];
        uint16_t *dst = x == 0 ? p.khat : p.vhat;
        dst[(static_cast<size_t>(pair) * p.n_rows_cap + j) * kD + d] =
            __bfloat16_as_ushort(__float2bfloat16_rn(sum / static_cast<float>(p.cmp_len)));
    }
}

}  // namespace

extern "C" SPARSE_API int sparse_nsa_compress(const uint16_t *k_cache, const uint16_t *v_cache, long long T_cap,
                                              int B, int H_kv, long long len_before, int n_new, int cmp_len,
                                              int cmp_stride, uint16_t *khat, uint16_t *vhat, int n_rows_cap,
                                              void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    const char *name = "sparse_nsa_compress";
    if (!k_cache || !v_cache || !khat || !vhat)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(khat) || !aligned16(vhat))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || T_cap < 1 || len_before < 0 || n_new < 0 || n_rows_cap < 1 || cmp_stride < 1 ||
        cmp_len < cmp_stride || cmp_len > 1024)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size (B=%d H_kv=%d n_new=%d l=%d s=%d)", name, B, H_kv, n_new,
                    cmp_len, cmp_stride);
    const long long len_after = len_before + n_new;
    if (len_after > T_cap)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: %lld tokens exceed T_cap=%lld", name, len_after, T_cap);
    const long long w_before = compressed_rows(len_before, cmp_len, cmp_stride);
    const long long w_after = compressed_rows(len_after, cmp_len, cmp_stride);
    if (w_after > n_rows_cap)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: %lld windows exceed n_rows_cap=%d", name, w_after, n_rows_cap);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535 || w_after - w_before > INT_MAX)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: too many pairs or windows", name);
    if (w_after == w_before)
        return SPARSE_OK;   // no window completed
    CompressParams p{k_cache, v_cache, khat, vhat, T_cap, n_rows_cap, cmp_len, cmp_stride, static_cast<int>(w_before)};
    dim3 grid(static_cast<unsigned>(w_after - w_before), static_cast<unsigned>(pairs));
    {
        sp_host::DeviceInfo dinfo;
        int rc0 = sp_host::device_info(&dinfo);
        static int configured[64];
        if (rc0 == SPARSE_OK)
            rc0 = sp_host::configure_kernel(reinterpret_cast<const void *>(compress_windows_kernel), 0, dinfo.device,
                                            configured);
        if (rc0 != SPARSE_OK)
            return rc0;
    }
    return sp_host::cuda_status(
        launch_pdl(reinterpret_cast<const void *>(compress_windows_kernel), grid, &p, stream), name);
}

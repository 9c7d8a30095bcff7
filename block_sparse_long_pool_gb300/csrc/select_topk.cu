// select_topk.cu -- Forecast scoring and exact top-k block selection.
//
// SparDA notes §4.1 eq.(6), §4.2 Alg.1 step 2, §4.3 eq.(9): one Forecast vector per
// GQA group is scored against every compressed key of the layer it selects for,
// the k best blocks outside B_init and B_local are taken, and the union
// B_init ∪ B_local ∪ top-k is written in ascending block order.
//
// GB300 design: one thread-block cluster of S CTAs per (batch, KV head) pair.  Every
// CTA scores a contiguous slice of the pair's compressed keys (a warp per 512-byte
// row, 16-byte loads, shuffle reduction) and stores each score as an order-preserving
// 32-bit key straight into CTA 0's shared memory (distributed shared memory stores).
// After one cluster barrier the other CTAs exit and CTA 0 alone finds the k-th
// largest candidate key by an MSB-first radix select over 4 byte-digits (histograms
// built with warp-aggregated shared-memory atomics), takes equal keys in ascending
// block order (ties go to the lower block index), and compacts the selection in
// block order with CTA-wide scans.  No global scratch memory.
#include <limits.h>

#include "common.cuh"

namespace {

using namespace sp;

// 256 threads and at most ~64 registers per thread (16K registers per CTA): a selection
// CTA then fits on an SM beside two attention CTAs, so the selection for layer l+1 can
// run on the SMs that stream layer l's blocks.
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kUnroll = 16;

struct SelectParams {
    const uint16_t *F;
    const float *ktil;
    const int *seq_len;
    int *idx_out;
    int *count_out;
    int *status;
    int H_kv;
    int N_cap;
    int n_init;
    int n_local;
    int k;
    int k_tot;
};

// Inclusive prefix sum over the CTA's threads (thread order); `total` receives the sum.
__device__ __forceinline__ int block_inclusive_scan(int v, int *warp_sums, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += n;
    }
    if (lane == 31)
        warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += n;
        }
        if (lane < kWarps)
            warp_sums[lane] = w;
    }
    __syncthreads();
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    total = warp_sums[kWarps - 1];
    __syncthreads();
    return v + before;
}

__global__ void __launch_bounds__(kThreads, 3) select_topk_kernel(const SelectParams p)
{
    extern __shared__ uint32_t keys[];           // CTA 0: the keys of all the pair's blocks
    __shared__ uint32_t hist[256];
    __shared__ int warp_sums[kWarps];
    __shared__ int bcast[4];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t S = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.y;
    const int b = pair / p.H_kv;

    // programmatic dependent launch: every input may come from the kernel before this
    // one on the stream
    griddep_wait();
    const long long len = p.seq_len[b];
    long long nb_ll = len <= 0 ? 0 : (len + kBlk - 1) / kBlk;
    if (nb_ll > p.N_cap) {
        if (rank == 0 && tid == 0)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        nb_ll = p.N_cap;
    }
    const int nb = static_cast<int>(nb_ll);
    const int chunk = (nb + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int j0 = min(nb, static_cast<int>(rank) * chunk);
    const int j1 = min(nb, j0 + chunk);

    // Candidates: every block that is neither init nor local (Alg.1 step 2).
    const int cand_lo = p.n_init;
    const int cand_hi = nb - p.n_local;
    const bool take_all = max(0, cand_hi - cand_lo) <= p.k;
    const bool take_none = p.k <= 0;   // only B_init and B_local

    // ---- 1. scores s_j = F . ktil_j (fp32) as order keys, stored into CTA 0
    if (!take_all && !take_none && j1 > j0) {
        uint32_t *keys0 = static_cast<uint32_t *>(__cluster_map_shared_rank(keys, 0));
        const uint2 fr = *reinterpret_cast<const uint2 *>(p.F + static_cast<size_t>(pair) * kD + 4 * lane);
        const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fr.x));
        const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fr.y));
        const float *kt = p.ktil + static_cast<size_t>(pair) * p.N_cap * kD + 4 * lane;
        for (int jb = j0 + warp; jb < j1; jb += kWarps * kUnroll) {
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = jb + u * kWarps;
                v[u] = j < j1 ? __ldg(reinterpret_cast<const float4 *>(kt + static_cast<size_t>(j) * kD))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float s = f01.x * v[u].x;
                s = fmaf(f01.y, v[u].y, s);
                s = fmaf(f23.x, v[u].z, s);
                s = fmaf(f23.y, v[u].w, s);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, o);
                const int j = jb + u * kWarps;
                if (lane == 0 && j < j1)
                    keys0[j] = order_key(s);
            }
        }
    }
    // the keys are in CTA 0 (release/acquire at cluster scope); the next kernel on the
    // stream may be scheduled, and the scoring CTAs are done
    cluster_sync();
    griddep_launch_dependents();
    if (rank != 0)
        return;

    // ---- 2. CTA 0: k-th largest candidate key by MSB-first radix select
    uint32_t prefix = 0, pmask = 0;
    int need = p.k;
    if (!take_all && !take_none) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            hist[tid] = 0;
            __syncthreads();
            for (int jb = cand_lo; jb < cand_hi; jb += kThreads) {
                const int j = jb + tid;
                uint32_t digit = 0xFFFFFFFFu;
                if (j < cand_hi) {
                    const uint32_t key = keys[j];
                    if ((key & pmask) == prefix)
                        digit = (key >> shift) & 255u;
                }
                // one atomic per distinct digit in the warp
                const uint32_t same = __match_any_sync(0xffffffffu, digit);
                if (digit != 0xFFFFFFFFu && lane == __ffs(same) - 1)
                    atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(same)));
            }
            __syncthreads();
            // thread t holds digit d = 255 - t: an inclusive scan gives the number of
            // matching keys with a digit >= d
            const int d = 255 - tid;
            const int tot = static_cast<int>(hist[d]);
            int all;
            const int at_or_above = block_inclusive_scan(tot, warp_sums, all);
            const int above = at_or_above - tot;
            if (at_or_above >= need && above < need) {
                bcast[0] = d;
                bcast[1] = need - above;
            }
            __syncthreads();
            prefix |= static_cast<uint32_t>(bcast[0]) << shift;
            pmask |= 0xFFu << shift;
            need = bcast[1];
            __syncthreads();
        }
    }
    const uint32_t thr = prefix;   // the k-th largest candidate key
    const int need_eq = need;      // keys equal to thr to take, lowest block ids first

    // ---- 3. selection in block order: this thread's contiguous run of blocks
    const int ipt = (nb + kThreads - 1) / kThreads;
    const int it0 = min(nb, tid * ipt), it1 = min(nb, it0 + ipt);
    int n_eq = 0;
    if (!take_all && !take_none)
        for (int j = it0; j < it1; ++j)
            n_eq += (j >= cand_lo && j < cand_hi && keys[j] == thr);
    int total_eq;
    const int eq_before = block_inclusive_scan(n_eq, warp_sums, total_eq) - n_eq;
    int n_sel = 0;
    int eq_rank = eq_before;
    for (int j = it0; j < it1; ++j) {
        bool sel = j < p.n_init || j >= nb - p.n_local;        // B_init and B_local
        if (!sel && !take_none && j >= cand_lo && j < cand_hi) {
            if (take_all) {
                sel = true;
            } else {
                const uint32_t key = keys[j];
                sel = key > thr || (key == thr && eq_rank++ < need_eq);
            }
        }
        n_sel += sel;
    }
    int total;
    int pos = block_inclusive_scan(n_sel, warp_sums, total) - n_sel;
    int *out = p.idx_out + static_cast<size_t>(pair) * p.k_tot;
    eq_rank = eq_before;
    bool overflow = false;
    for (int j = it0; j < it1; ++j) {
        bool sel = j < p.n_init || j >= nb - p.n_local;
        if (!sel && !take_none && j >= cand_lo && j < cand_hi) {
            if (take_all) {
                sel = true;
            } else {
                const uint32_t key = keys[j];
                sel = key > thr || (key == thr && eq_rank++ < need_eq);
            }
        }
        if (sel) {
            if (pos < p.k_tot)
                out[pos] = j;
            else
                overflow = true;
            ++pos;
        }
    }
    if (overflow)
        report(p.status, SPARSE_ERR_BAD_INDEX);
    for (int i = total + tid; i < p.k_tot; i += kThreads)
        out[i] = -1;
    if (tid == 0)
        p.count_out[pair] = min(total, p.k_tot);
}

}  // namespace

extern "C" SPARSE_API int sparse_select_topk(const uint16_t *F, const float *ktil, const int *seq_len,
                                             int B, int H_kv, int N_cap, int n_init, int n_local,
                                             int k, int *idx_out, int *count_out, int k_tot,
                                             int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!F || !ktil || !seq_len || !idx_out || !count_out)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk: null pointer");
    if (!aligned16(F) || !aligned16(ktil))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk: F and ktil must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || N_cap < 1 || n_init < 0 || n_local < 0 || k < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk: bad size");
    if (static_cast<long long>(n_init) + n_local + k > k_tot)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk: k_tot=%d < n_init+n_local+k", k_tot);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk: B*H_kv=%lld > 65535", pairs);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    // Cluster size: enough CTAs to cover the SMs twice, slices of >= 256 blocks.
    int S = 1;
    while (S < kMaxCluster && pairs * S * 2 <= 2LL * dev.sm_count && N_cap / (S * 2) >= 256)
        S *= 2;
    const size_t smem = static_cast<size_t>(N_cap) * sizeof(uint32_t);   // CTA 0 holds every key
    if (smem > static_cast<size_t>(dev.max_smem_optin) - 8192)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk: N_cap=%d too large", N_cap);
    static int configured[64];
    rc = sp_host::configure_kernel(reinterpret_cast<const void *>(select_topk_kernel), static_cast<int>(smem),
                                   dev.device, configured);
    if (rc != SPARSE_OK)
        return rc;
    SelectParams p{F, ktil, seq_len, idx_out, count_out, status, H_kv, N_cap, n_init, n_local, k, k_tot};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {&p};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(select_topk_kernel), args),
                                "sparse_select_topk launch");
}

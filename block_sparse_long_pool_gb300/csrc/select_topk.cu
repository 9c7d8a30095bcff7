// select_topk.cu -- Forecast scoring and exact top-k block selection.
//
// SparDA notes §4.1 eq.(6), §4.2 Alg.1 step 2, §4.3 eq.(9): one Forecast vector per
// GQA group is scored against every compressed key of the layer it selects for,
// the k best blocks outside B_init and B_local are taken, and the union
// B_init ∪ B_local ∪ top-k is written in ascending block order.
//
// GB300 design: one thread-block cluster of S CTAs per (batch, KV head) pair.  CTA r
// scores a contiguous slice of the pair's blocks (a warp per compressed-key row,
// 16-byte loads, shuffle reduction) into an order-preserving 32-bit key held in its
// shared memory.  The k-th largest key is found by an MSB-first radix select over 4
// byte-digits whose histograms are summed across the cluster through distributed
// shared memory; equal keys are taken in ascending block order, so ties go to the
// lower block index.  Every exchange between CTAs goes through DSMEM: the kernel
// uses no global scratch memory.
#include <limits.h>

#include "common.cuh"

namespace {

using namespace sp;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kUnroll = 4;

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

// Monotone map of a float score to an unsigned key (larger score -> larger key);
// -0 and +0 share a key.
__device__ __forceinline__ uint32_t order_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

__global__ void __launch_bounds__(kThreads) select_topk_kernel(const SelectParams p)
{
    extern __shared__ uint32_t keys[];           // keys of this CTA's block slice
    __shared__ uint32_t hist[2][256];
    __shared__ int warp_sums[kWarps];
    __shared__ int xchg[2];                      // [0] = equal-key count, [1] = sure selections
    __shared__ int bcast[4];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t S = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.y;
    const int b = pair / p.H_kv;

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
    const int my = j1 - j0;

    // Candidates: every block that is neither init nor local (Alg.1 step 2).
    const int cand_lo = p.n_init;
    const int cand_hi = nb - p.n_local;
    const int n_cand = max(0, cand_hi - cand_lo);
    const bool take_all = n_cand <= p.k;

    // ---- 1. scores s_j = F . ktil_j (fp32) as order keys
    if (!take_all && my > 0) {
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
                    keys[j - j0] = order_key(s);
            }
        }
    }
    __syncthreads();

    // ---- 2. k-th largest key by MSB-first radix select across the cluster
    uint32_t prefix = 0, pmask = 0;
    int need = p.k;
    if (!take_all) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            uint32_t *h = hist[pass & 1];
            for (int i = tid; i < 256; i += kThreads)
                h[i] = 0;
            __syncthreads();
            for (int i = tid; i < my; i += kThreads) {
                const int j = j0 + i;
                if (j >= cand_lo && j < cand_hi) {
                    const uint32_t key = keys[i];
                    if ((key & pmask) == prefix)
                        atomicAdd(&h[(key >> shift) & 255u], 1u);
                }
            }
            cluster_sync();
            // thread t holds digit d = 255 - t: an inclusive scan gives the number of
            // keys with a digit >= d.
            int tot = 0;
            const int d = 255 - tid;
            if (tid < 256) {
                const uint32_t local = smem_u32(&h[d]);
                for (uint32_t c = 0; c < S; ++c)
                    tot += static_cast<int>(dsmem_ld_u32(dsmem_addr(local, c)));
            }
            int all;
            const int at_or_above = block_inclusive_scan(tid < 256 ? tot : 0, warp_sums, all);
            if (tid < 256) {
                const int above = at_or_above - tot;
                if (at_or_above >= need && above < need) {
                    bcast[0] = d;
                    bcast[1] = need - above;
                }
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

    // ---- 3. per-thread counts over a contiguous run of this CTA's slice
    const int ipt = (my + kThreads - 1) / kThreads;
    const int it0 = min(my, tid * ipt), it1 = min(my, it0 + ipt);
    int n_eq = 0, n_sure = 0;
    for (int i = it0; i < it1; ++i) {
        const int j = j0 + i;
        const bool forced = j < p.n_init || j >= nb - p.n_local;
        if (forced) {
            ++n_sure;
        } else if (j >= cand_lo && j < cand_hi) {
            if (take_all) {
                ++n_sure;
            } else {
                const uint32_t key = keys[i];
                n_sure += key > thr;
                n_eq += key == thr;
            }
        }
    }
    int cta_eq, cta_sure;
    const int eq_incl = block_inclusive_scan(n_eq, warp_sums, cta_eq);
    block_inclusive_scan(n_sure, warp_sums, cta_sure);
    if (tid == 0) {
        xchg[0] = cta_eq;
        xchg[1] = cta_sure;
    }
    cluster_sync();
    if (tid == 0) {
        int eq_before = 0, sel_before = 0, total = 0, eq_cum = 0;
        const uint32_t a0 = smem_u32(&xchg[0]), a1 = smem_u32(&xchg[1]);
        for (uint32_t c = 0; c < S; ++c) {
            const int e = static_cast<int>(dsmem_ld_u32(dsmem_addr(a0, c)));
            const int s = static_cast<int>(dsmem_ld_u32(dsmem_addr(a1, c)));
            const int take = min(e, max(0, need_eq - eq_cum));
            if (c < rank) {
                eq_before += e;
                sel_before += s + take;
            }
            eq_cum += e;
            total += s + take;
        }
        bcast[0] = eq_before;
        bcast[1] = sel_before;
        bcast[2] = total;
    }
    __syncthreads();
    const int eq_before = bcast[0], sel_before = bcast[1], total = bcast[2];

    // ---- 4. selection flags and ascending compaction
    int eq_rank = eq_before + eq_incl - n_eq;   // global rank of this thread's first equal key
    int n_sel = 0;
    for (int i = it0; i < it1; ++i) {
        const int j = j0 + i;
        const bool forced = j < p.n_init || j >= nb - p.n_local;
        if (forced) {
            ++n_sel;
        } else if (j >= cand_lo && j < cand_hi) {
            if (take_all) {
                ++n_sel;
            } else {
                const uint32_t key = keys[i];
                if (key > thr)
                    ++n_sel;
                else if (key == thr)
                    n_sel += (eq_rank++ < need_eq);
            }
        }
    }
    int cta_sel;
    const int sel_incl = block_inclusive_scan(n_sel, warp_sums, cta_sel);
    int pos = sel_before + sel_incl - n_sel;
    eq_rank = eq_before + eq_incl - n_eq;
    int *out = p.idx_out + static_cast<size_t>(pair) * p.k_tot;
    bool overflow = false;
    for (int i = it0; i < it1; ++i) {
        const int j = j0 + i;
        const bool forced = j < p.n_init || j >= nb - p.n_local;
        bool sel = forced;
        if (!forced && j >= cand_lo && j < cand_hi) {
            if (take_all) {
                sel = true;
            } else {
                const uint32_t key = keys[i];
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
    if (rank == 0) {
        for (int i = total + tid; i < p.k_tot; i += kThreads)
            out[i] = -1;
        if (tid == 0)
            p.count_out[pair] = min(total, p.k_tot);
    }
    // peers may still be reading xchg through DSMEM
    cluster_sync();
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
    const size_t smem = static_cast<size_t>((N_cap + S - 1) / S) * sizeof(uint32_t);
    if (smem > static_cast<size_t>(dev.max_smem_optin) - 8192)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk: N_cap=%d too large", N_cap);
    static thread_local int configured_smem[64];
    if (dev.device < 64 && configured_smem[dev.device] < static_cast<int>(smem)) {
        rc = sp_host::cuda_status(cudaFuncSetAttribute(select_topk_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(smem)),
                                  "sparse_select_topk smem attribute");
        if (rc != SPARSE_OK)
            return rc;
        configured_smem[dev.device] = static_cast<int>(smem);
    }
    SelectParams p{F, ktil, seq_len, idx_out, count_out, status, H_kv, N_cap, n_init, n_local, k, k_tot};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(select_topk_kernel), args),
                                "sparse_select_topk launch");
}

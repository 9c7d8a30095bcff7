// heads.cu -- the multi-head (InfLLM-V2) block selector, the baseline the SparDA notes
// compare the Forecast selection with.
#include <math.h>

#include "attn_core.cuh"
#include "select_core.cuh"
#include "select_layout.cuh"

namespace {

// ---------------------------------------------------------------- multi-head selection
//
// The InfLLM-V2 selector that the SparDA notes compare against (§4.3 eq.(8), Figure 3):
// every one of the G query heads of a group scores the compressed keys, each head's
// scores pass through a softmax over the pair's blocks, the G distributions are summed
// and the top-k is taken as for the Forecast selection.  Same cluster layout as the
// Forecast kernel; the per-head softmax needs every block's raw scores before any sum
// can be formed, so a CTA keeps its slice's raw scores in shared memory:
//   1. stream the slice's compressed keys, raw scores a^h_j (log2 units) -> shared;
//   2. per head, the slice's max and sum of exp2 -> CTA 0, which merges them and
//      sends each CTA the head's max and 1 / sum;
//   3. s_j = sum_h exp2(a^h_j - M_h) / Z_h -> order key -> CTA 0, whose consumer
//      warps and selector warp take the top-k together: the keys in registers, the
//      bits every key shares decided at once, a binary search over the rest with
//      block-wide counts, the list written through block-wide prefix sums (a radix
//      threshold and a one-warp write past 2720 candidates).

constexpr int kMaxHeadsSel = 16;
constexpr int kCtrlStatsBar = 10;   // ctrl[10..11]
constexpr int kCtrlNormBar = 12;    // ctrl[12..13]
constexpr int kCtrlThrWords = 4;    // ctrl[4..5]: the running threshold of the top-k search
constexpr int kHeadsTopkThreads = (kConsumerWarps + 1) * 32;   // CTA 0's consumers + selector
constexpr int kHeadsKpt = 17;   // candidate keys per thread in the register top-k (2720 blocks)

struct HeadsLayout {
    int off_keys, off_q, off_raw, off_stats, off_norm, total;
};

__host__ __device__ inline HeadsLayout heads_layout(int N_cap, int rows_max, int G, int S)
{
    HeadsLayout l;
    l.off_keys = fused_off_slice();                       // after the histogram and list
    l.off_q = l.off_keys + ((N_cap * 4 + 15) & ~15);      // [G][128] fp32 queries
    l.off_raw = l.off_q + G * kD * 4;                     // [G][rows_max] raw scores (head-major)
    l.off_stats = l.off_raw + ((rows_max * G * 4 + 15) & ~15);   // CTA 0: [S][G] (max, sum)
    l.off_norm = l.off_stats + S * G * 8;                 // [G] (max, 1 / sum)
    l.total = l.off_norm + G * 8;
    return l;
}

__global__ void __launch_bounds__(kFThreads, 1) select_heads_kernel(const AttnParams p, int rows_max)
{
    griddep_wait();   // every input may be written by the kernel before this one
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const uint32_t bar_full = base_s + kOffBars;
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;
    const uint32_t bar_scored = base_s + kOffCtrl + 4 * kCtrlScoredBar;
    const uint32_t bar_stats = base_s + kOffCtrl + 4 * kCtrlStatsBar;
    const uint32_t bar_norm = base_s + kOffCtrl + 4 * kCtrlNormBar;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = static_cast<int>(gridDim.x);
    const int rank = static_cast<int>(blockIdx.x);
    const int pair = blockIdx.y;
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    const int G = p.G;
    const HeadsLayout L = heads_layout(p.N_cap, rows_max, G, S);
    uint32_t *keys = reinterpret_cast<uint32_t *>(base + L.off_keys);
    float *qf = reinterpret_cast<float *>(base + L.off_q);
    float *raw = reinterpret_cast<float *>(base + L.off_raw);
    float *stats = reinterpret_cast<float *>(base + L.off_stats);
    float *norm = reinterpret_cast<float *>(base + L.off_norm);

    const long long len = p.seq_len[b];
    long long nb_ll = len <= 0 ? 0 : (len + kBlk - 1) / kBlk;
    const bool len_bad = nb_ll > p.N_cap;
    if (len_bad)
        nb_ll = p.N_cap;
    const int nb = static_cast<int>(nb_ll);
    const bool take_all = max(0, nb - p.n_local - p.n_init) <= p.k_sel;
    const bool score = !take_all && p.k_sel > 0;
    const bool regs_topk = topk_cta_regs_fits<kHeadsKpt>(nb - p.n_local - p.n_init, kHeadsTopkThreads);
    const int chunk = (nb + S - 1) / S;
    const int r0 = score ? min(nb, rank * chunk) : 0;
    const int n_krows = score ? min(nb, r0 + chunk) - r0 : 0;
    const int n_kst = (n_krows + kKtilRowsPerStage - 1) / kKtilRowsPerStage;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_scored, S * kConsumerWarps);
        mbar_init(bar_stats, S * kConsumerWarps);
        mbar_init(bar_norm, 1);
        fence_barrier_init();
    }
    __syncthreads();
    cluster_arrive();
    griddep_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const float *kt = p.ktil + (static_cast<size_t>(pair) * p.N_cap + r0) * kD;
            for (int ks = 0; ks < n_kst; ++ks) {
                const int s = ks % kStages;
                const int use = ks / kStages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const int rows = min(kKtilRowsPerStage, n_krows - ks * kKtilRowsPerStage);
                const uint32_t bytes = static_cast<uint32_t>(rows * kKtilRowBytes);
                mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                bulk_load(base_s + s * kStageBytes, kt + static_cast<size_t>(ks) * kKtilRowsPerStage * kD, bytes,
                          bar_full + 8 * s, pol);
            }
        }
        cluster_wait();
    } else if (warp < kConsumerWarps) {
        // ------------------------------------------------------------ consumers
        if (score) {
            // the group's G query heads, fp32, scale folded in (log2 units)
            for (int i = tid; i < G * kD; i += kConsumerWarps * 32) {
                const int h = i / kD, d = i - h * kD;
                const __nv_bfloat16 q = *reinterpret_cast<const __nv_bfloat16 *>(
                    p.Q + (static_cast<size_t>(b) * p.H_q + g * G + h) * kD + d);
                qf[i] = __bfloat162float(q) * p.scale_log2;
            }
        }
        named_barrier_sync(2, kConsumerWarps * 32);
        cluster_wait();
        uint32_t *keys0 = static_cast<uint32_t *>(__cluster_map_shared_rank(keys, 0));
        float *stats0 = static_cast<float *>(__cluster_map_shared_rank(stats, 0));
        bool ok = true;
        // (1) raw scores of the slice
        for (int ks = 0; ks < n_kst; ++ks) {
            const int s = ks % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (ks / kStages) & 1, kWaitNs))) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const int rows = min(kKtilRowsPerStage, n_krows - ks * kKtilRowsPerStage);
            const int nrow = min(16, rows - warp * 16);
            if (nrow > 0) {
                const float *stage = reinterpret_cast<const float *>(base + s * kStageBytes) + warp * 16 * kD;
                float4 v[16];
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    v[r] = r < nrow ? reinterpret_cast<const float4 *>(stage + r * kD)[lane]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                for (int h = 0; h < G; ++h) {
                    const float4 q = reinterpret_cast<const float4 *>(qf + h * kD)[lane];
                    float acc[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        float sc = q.x * v[r].x;
                        sc = fmaf(q.y, v[r].y, sc);
                        sc = fmaf(q.z, v[r].z, sc);
                        sc = fmaf(q.w, v[r].w, sc);
                        acc[r] = sc;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const bool up = (lane & 16) != 0;
                        const float give = up ? acc[i] : acc[i + 8];
                        const float keep = up ? acc[i + 8] : acc[i];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const bool up = (lane & 8) != 0;
                        const float give = up ? acc[i] : acc[i + 4];
                        const float keep = up ? acc[i + 4] : acc[i];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const bool up = (lane & 4) != 0;
                        const float give = up ? acc[i] : acc[i + 2];
                        const float keep = up ? acc[i + 2] : acc[i];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
                    }
                    {
                        const bool up = (lane & 2) != 0;
                        const float give = up ? acc[0] : acc[1];
                        const float keep = up ? acc[1] : acc[0];
                        acc[0] = keep + __shfl_xor_sync(0xffffffffu, give, 2);
                    }
                    acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
                    const int r = (lane >> 1) & 15;
                    if ((lane & 1) == 0 && r < nrow)
                        raw[h * rows_max + ks * kKtilRowsPerStage + warp * 16 + r] = acc[0];
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        named_barrier_sync(2, kConsumerWarps * 32);   // every raw score of the slice is written
        // (2) per head: the slice's max and sum of exp2, merged by CTA 0
        if (score) {
            // (one warp per scheduler: four independent accumulators per lane)
            for (int h = warp; h < G; h += kConsumerWarps) {
                const float *rh = raw + h * rows_max;
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                for (int i = lane; i < n_krows; i += 128)
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {   // branch-free: clamped load, masked value
                        const float v = rh[min(i + 32 * q4, n_krows - 1)];
                        m4[q4] = fmaxf(m4[q4], i + 32 * q4 < n_krows ? v : -INFINITY);
                    }
                float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                float z4[4] = {0.f, 0.f, 0.f, 0.f};
                if (m != -INFINITY)
                    for (int i = lane; i < n_krows; i += 128)
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float e = ex2_approx(rh[min(i + 32 * q4, n_krows - 1)] - m);
                            z4[q4] += i + 32 * q4 < n_krows ? e : 0.f;
                        }
                float z = (z4[0] + z4[1]) + (z4[2] + z4[3]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    z += __shfl_xor_sync(0xffffffffu, z, o);
                if (lane == 0) {
                    stats0[(rank * G + h) * 2] = m;
                    stats0[(rank * G + h) * 2 + 1] = z;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_stats, 0));
            // (3) summed per-head distributions -> order keys in CTA 0
            const bool have_norm = __all_sync(0xffffffffu, mbar_wait_cluster(bar_norm, 0, kWaitNs));
            if (!have_norm) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
            } else {
                // heads past G read head G-1's row and add an exact 0: a branch-free body
                float nm[kMaxHeadsSel], ni[kMaxHeadsSel];
                const float *rowh[kMaxHeadsSel];
#pragma unroll
                for (int h = 0; h < kMaxHeadsSel; ++h) {
                    nm[h] = h < G ? norm[2 * h] : INFINITY;
                    ni[h] = h < G ? norm[2 * h + 1] : 0.f;
                    rowh[h] = raw + min(h, G - 1) * rows_max;
                }
                constexpr int kPass = 2, kStride = kConsumerWarps * 32;
                for (int ib = warp * 32; ib < n_krows; ib += kPass * kStride) {
                    float sum[kPass];
#pragma unroll
                    for (int q2 = 0; q2 < kPass; ++q2) {
                        const int i = min(ib + q2 * kStride + lane, n_krows - 1);
                        float acc = 0.f;
#pragma unroll
                        for (int h = 0; h < kMaxHeadsSel; ++h)
                            acc += ex2_approx(rowh[h][i] - nm[h]) * ni[h];
                        sum[q2] = acc;
                    }
#pragma unroll
                    for (int q2 = 0; q2 < kPass; ++q2) {
                        const int i = ib + q2 * kStride + lane;
                        if (ok && i < n_krows)
                            keys0[r0 + i] = order_key(sum[q2]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_scored, 0));
            if (rank == 0) {
                // CTA 0's consumers join its selector warp in the threshold search (the
                // summed probabilities share an exponent: a coarse histogram of the top
                // key bits would not narrow them)
                const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
                if (!got && lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                if (regs_topk) {
                    topk_cta_regs<kHeadsKpt>(base_s + L.off_keys, nb, p.n_init, p.n_local, p.k_sel,
                                             base_s + fused_off_hist(), tid + 32, kHeadsTopkThreads, 3, got,
                                             p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next,
                                             p.count_next + pair, p.status);
                } else {
                    uint32_t prefix;
                    int need;
                    topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel,
                                       base_s + fused_off_hist(), base_s + kOffCtrl + 4 * kCtrlThrWords, tid + 32,
                                       kHeadsTopkThreads, 3, prefix, need);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ selector (CTA 0)
        if (rank == 0) {
            if (len_bad && lane == 0)
                report(p.status, SPARSE_ERR_BAD_INDEX);
            bool ready = true;
            if (score) {
                ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_stats, 0, kWaitNs));
                // merge the slices' (max, sum) per head, then send (max, 1 / sum) to every CTA
                float *normloc = norm;
                if (ready && lane < G) {
                    float M = -INFINITY;
                    for (int c = 0; c < S; ++c)
                        M = fmaxf(M, stats[(c * G + lane) * 2]);
                    float Z = 0.f;
                    for (int c = 0; c < S; ++c) {
                        const float mc = stats[(c * G + lane) * 2];
                        if (mc != -INFINITY)
                            Z += stats[(c * G + lane) * 2 + 1] * exp2f(mc - M);
                    }
                    normloc[2 * lane] = M;
                    normloc[2 * lane + 1] = Z > 0.f ? 1.f / Z : 0.f;
                }
                __syncwarp();
                if (ready && lane < S && lane > 0) {
                    float *peer = static_cast<float *>(__cluster_map_shared_rank(norm, static_cast<unsigned>(lane)));
                    for (int i = 0; i < 2 * G; ++i)
                        peer[i] = normloc[i];
                }
                __syncwarp();
                if (ready && lane < S)
                    mbar_arrive_cluster(dsmem_addr(bar_norm, static_cast<uint32_t>(lane)));
                if (ready)
                    ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
            }
            uint32_t prefix = 0u;
            int need = 0;
            if (score && regs_topk) {
                topk_cta_regs<kHeadsKpt>(base_s + L.off_keys, nb, p.n_init, p.n_local, p.k_sel,
                                         base_s + fused_off_hist(), lane, kHeadsTopkThreads, 3, ready,
                                         p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next,
                                         p.count_next + pair, p.status);
            } else {
                if (score)
                    topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel,
                                       base_s + fused_off_hist(), base_s + kOffCtrl + 4 * kCtrlThrWords, lane,
                                       kHeadsTopkThreads, 3, prefix, need);
                if (ready) {
                    topk_write_warp(base_s + L.off_keys, 0u, 0, nb, p.n_init, p.n_local,
                                    max(0, nb - p.n_local - p.n_init) <= p.k_sel, p.k_sel <= 0, prefix, need,
                                    p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next,
                                    p.count_next + pair, p.status, lane);
                } else if (lane == 0) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                }
            }
        }
        cluster_wait();
    }
}

static_assert(4 * kCtrlNormBar + 8 <= 64, "ctrl layout");
static_assert(kCtrlThrWords >= 4 && 4 * kCtrlThrWords + 8 <= 4 * kCtrlScoredBar, "ctrl layout: threshold words");
static_assert((kHeadsTopkThreads / 32) * 256 <= kCoarseBins + kTopkList, "multi-head radix bins");


}  // namespace

extern "C" SPARSE_API int sparse_select_topk_heads(const uint16_t *Q, const float *ktil, const int *seq_len, int B,
                                                   int H_q, int H_kv, int N_cap, float scale, int n_init, int n_local,
                                                   int k, int *idx_out, int *count_out, int k_tot, int *status,
                                                   void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!Q || !ktil || !seq_len || !idx_out || !count_out)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_heads: null pointer");
    if (!aligned16(Q) || !aligned16(ktil))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_heads: Q and ktil must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || N_cap < 1 || n_init < 0 || n_local < 0 || k < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_heads: bad size");
    if (!isfinite(scale) || scale < 0.f)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_heads: scale must be finite and >= 0");
    if (static_cast<long long>(n_init) + n_local + k > k_tot)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_heads: k_tot=%d < n_init+n_local+k", k_tot);
    const int G = H_q / H_kv;
    if (G > kMaxHeadsSel)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk_heads: G=%d > %d", G, kMaxHeadsSel);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk_heads: B*H_kv=%lld > 65535", pairs);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    // one CTA per SM (the slice's raw scores stay in shared memory): CTAs <= SMs where
    // possible, at least 128 key rows per CTA, and a slice that fits
    int S = 1;
    while (S < kMaxSplit && pairs * S * 2 <= dev.sm_count && N_cap / (S * 2) >= 128)
        S *= 2;
    auto stride_for = [&](int S_) { return ((N_cap + S_ - 1) / S_ + 27) / 32 * 32 + 4; };
    HeadsLayout L = heads_layout(N_cap, stride_for(S), G, S);
    while (static_cast<size_t>(L.total) + 1024 > static_cast<size_t>(dev.max_smem_optin) && S < kMaxSplit) {
        S *= 2;
        L = heads_layout(N_cap, stride_for(S), G, S);
    }
    const size_t smem = static_cast<size_t>(L.total) + 1024;
    if (smem > static_cast<size_t>(dev.max_smem_optin))
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk_heads: N_cap=%d needs %zu bytes of shared memory",
                    N_cap, smem);
    AttnParams p = {};
    p.Q = Q;
    p.seq_len = seq_len;
    p.status = status;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.scale_log2 = scale_log2_of(scale);
    p.ktil = ktil;
    p.idx_next = idx_out;
    p.count_next = count_out;
    p.N_cap = N_cap;
    p.n_init = n_init;
    p.n_local = n_local;
    p.k_sel = k;
    p.k_tot_next = k_tot;
    // per-head stride of the raw scores: the slice's rows, = 4 mod 32 (no bank conflicts)
    const int rows_max = ((N_cap + S - 1) / S + 27) / 32 * 32 + 4;
    static int configured[64];
    rc = sp_host::configure_kernel(reinterpret_cast<const void *>(select_heads_kernel), static_cast<int>(smem),
                                   dev.device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
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
    void *args[] = {&p, const_cast<int *>(&rows_max)};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(select_heads_kernel), args),
                                "sparse_select_topk_heads launch");
}

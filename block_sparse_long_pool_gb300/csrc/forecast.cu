// forecast.cu -- Forecast block selection, alone or fused with a decode layer's attention.
//
// Two entry points share one kernel:
//   * sparse_select_topk (SparDA notes §4.1 eq.(6), §4.2 Alg.1 step 2, §4.3 eq.(9)):
//     one Forecast vector per GQA group is scored against every compressed key of the
//     layer it selects for (fp32 s_j = F . K̃_j), the k largest outside B_init and
//     B_local are taken (equal scores: the lower block index), and B_init ∪ B_local ∪
//     top-k is written in ascending block order.
//   * sparse_decode_attn_forecast: one SparDA decode layer in one launch.  The Forecast
//     vector F_l of layer l selects the blocks of layer l+1 while layer l attends over
//     the blocks chosen one layer earlier (§4.1: the decoupling; eq.(7); Alg.1 steps 2
//     and 4 of one layer).  The attention is the one of sparse_decode_attn (scale
//     1/sqrt(d), split-KV merged by the online-softmax recurrence).
//
// GB300 design.  A cluster of S CTAs per (batch, KV head) pair; 6 warps per CTA.
//   * Warp 4 (producer): one lane streams this CTA's slice of the compressed keys into
//     the ring (1-D bulk copies, 64 rows = 32 KB per stage).  In the fused launch that
//     needs nothing the preceding kernel writes, so it overlaps the preceding kernel's
//     tail under programmatic dependent launch; then the producer waits for that
//     kernel (the block list of this layer may be its output), stages the list slice,
//     and streams the selected K/V blocks with TMA tensor copies.
//   * Warps 0-3 (consumers): score every key row of a stage (fp32 dot product with F,
//     one warp per 16 rows, a transposed butterfly reduction), store the order key into
//     CTA 0's shared memory and add it to CTA 0's coarse histogram (distributed shared
//     memory); each warp then arrives on CTA 0's "scored" barrier; in the fused launch
//     they then attend as the sparse_decode_attn cluster kernel does.
//   * Warp 5 (selector) of CTA 0: waits on the "scored" barrier, finds the coarse bin
//     that holds the k-th largest key, radix-selects within it and writes the list,
//     while (in the fused launch) the consumers attend.
//   * The dependent launch is allowed at once: a following launch starts streaming its
//     key slice as SMs free up, and waits for this one before reading what it writes.
#include <string.h>

#include "attn_core.cuh"
#include "select_core.cuh"

namespace {

constexpr int kFThreads = (kConsumerWarps + 2) * 32;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;   // producer + consumers (named barrier 1)
constexpr int kKtilRowBytes = kD * 4;
constexpr int kKtilRowsPerStage = kStageBytes / kKtilRowBytes;   // 64
constexpr int kCtrlScoredBar = 8;                                 // ctrl[8..9]: the "scored" mbarrier

// Shared memory after the ring, barriers and ctrl words (offsets from the 1024-byte
// aligned base): CTA 0's coarse key histogram (reused for the radix digits), the keys
// gathered in the threshold bin, the list slice (slot, logical) and CTA 0's keys.
__host__ __device__ constexpr int fused_off_hist()
{
    return kOffList;
}
__host__ __device__ constexpr int fused_off_topk_list()
{
    return kOffList + kCoarseBins * 4;
}
__host__ __device__ constexpr int fused_off_slice()
{
    return fused_off_topk_list() + kTopkList * 4;
}
__host__ __device__ inline int fused_per_pad(int per)
{
    return (per + 3) & ~3;
}
__host__ __device__ inline int fused_off_keys(int per)
{
    return fused_off_slice() + 2 * fused_per_pad(per) * 4;
}
inline size_t fused_smem_bytes(int per, int N_cap)
{
    return static_cast<size_t>(fused_off_keys(per)) + static_cast<size_t>(N_cap) * 4 + 1024;
}

// ATTN = false: the Forecast selection alone (sparse_select_topk): no block list, no
// attention, no merge; every input may be written by the kernel before this one.
template <int NT, bool ATTN>
__global__ void __launch_bounds__(kFThreads, 2)
    decode_forecast_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const AttnParams p)
{
    if (!ATTN)
        griddep_wait();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kOffCtrl);
    const uint32_t bar_full = base_s + kOffBars;
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;
    const uint32_t bar_scored = base_s + kOffCtrl + 4 * kCtrlScoredBar;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t S = gridDim.x;       // the cluster spans gridDim.x
    const uint32_t rank = blockIdx.x;   // == %cluster_ctarank
    const int pair = blockIdx.y;
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    const int per = (p.k_tot + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int i0 = min(p.k_tot, static_cast<int>(rank) * per);
    const int cap = min(p.k_tot, i0 + per) - i0;
    int *lslot = reinterpret_cast<int *>(base + fused_off_slice());
    int *llog = lslot + fused_per_pad(per);
    uint32_t *keys = reinterpret_cast<uint32_t *>(base + fused_off_keys(per));
    uint32_t *hist = reinterpret_cast<uint32_t *>(base + fused_off_hist());

    // The next layer's rows: seq_len and its compressed keys are complete before the
    // kernel before this one finishes (the caller's promise), so they are read at once.
    const bool do_sel = p.F != nullptr;
    const long long len = p.seq_len[b];
    long long nb_ll = len <= 0 ? 0 : (len + kBlk - 1) / kBlk;
    const bool len_bad = nb_ll > p.N_cap;
    if (len_bad)
        nb_ll = p.N_cap;
    const int nb = static_cast<int>(nb_ll);
    const bool take_all = max(0, nb - p.n_local - p.n_init) <= p.k_sel;
    const bool score = do_sel && !take_all;
    const int chunk = (nb + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int r0 = score ? min(nb, static_cast<int>(rank) * chunk) : 0;
    const int n_krows = score ? min(nb, r0 + chunk) - r0 : 0;
    const int n_kst = (n_krows + kKtilRowsPerStage - 1) / kKtilRowsPerStage;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_scored, S * kConsumerWarps);
        fence_barrier_init();
    }
    if (rank == 0 && score)
        for (int i = tid; i < kCoarseBins; i += kFThreads)
            hist[i] = 0u;
    __syncthreads();
    cluster_arrive();              // every thread; waited before the first access to CTA 0
    griddep_launch_dependents();   // the next layer may start its key stream as SMs free up

    WarpState<NT> st;
    st.reset();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        int failed = 0;
        const uint64_t pol = policy_evict_first();
        int it = 0;
        if (lane == 0) {
            const float *kt = p.ktil + (static_cast<size_t>(pair) * p.N_cap + r0) * kD;
            for (int ks = 0; ks < n_kst; ++ks, ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    failed = 1;
                    break;
                }
                const int rows = min(kKtilRowsPerStage, n_krows - ks * kKtilRowsPerStage);
                const uint32_t bytes = static_cast<uint32_t>(rows * kKtilRowBytes);
                mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                bulk_load(base_s + s * kStageBytes, kt + static_cast<size_t>(ks) * kKtilRowsPerStage * kD, bytes,
                          bar_full + 8 * s, pol);
            }
        }
        failed = __shfl_sync(0xffffffffu, failed, 0);
        it = __shfl_sync(0xffffffffu, it, 0);
        // this layer's block list may be the previous kernel's output
        if (ATTN && (p.flags & SPARSE_ATTN_BLOCKS_READY) == 0u)
            griddep_wait();
        int n_run = ATTN ? producer_fetch_slice(p, pair, i0, cap, lslot, llog, ctrl, lane) : 0;
        if (failed) {
            n_run = 0;
            if (lane == 0)
                ctrl[kCtrlList] = 0;
            __syncwarp();
        }
        if (ATTN)
            named_barrier_arrive(1, kAttnThreads);
        if (ATTN && lane == 0 && n_run > 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            for (int i = 0; i < n_run; ++i, ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const int slot = lslot[i];
                const int row = slot >= 0 ? slot * kBlk : static_cast<int>(min(p.pair_stride, (long long)INT_MAX - kBlk));
                const uint32_t dst = base_s + s * kStageBytes;
                mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                tma_load_3d(dst, &kmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * s, 64, row, pair, pol);
                tma_load_3d(dst + kTileBytes, &vmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, bar_full + 8 * s, 64, row, pair, pol);
            }
        }
        cluster_wait();
    } else if (warp < kConsumerWarps) {
        // ------------------------------------------------------------ consumers
        griddep_wait();   // Q and F may be written by the kernel before this one
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (score) {
            const uint2 fr = *reinterpret_cast<const uint2 *>(p.F + static_cast<size_t>(pair) * kD + 4 * lane);
            const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fr.x));
            const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fr.y));
            f = make_float4(f01.x, f01.y, f23.x, f23.y);
        }
        QueryFrags<NT> q;
        if (ATTN)
            load_query<NT, false>(q, p, b, g, 0, p.G, lane);
        cluster_wait();   // CTA 0's "scored" barrier and key array exist
        uint32_t *keys0 = static_cast<uint32_t *>(__cluster_map_shared_rank(keys, 0));
        uint32_t *coarse0 = static_cast<uint32_t *>(__cluster_map_shared_rank(hist, 0));
        // (1) the next layer's scores, order keys into CTA 0
        int it = 0;
        bool ok = true;
        for (int ks = 0; ks < n_kst; ++ks, ++it) {
            const int s = it % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (it / kStages) & 1, kWaitNs))) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const int rows = min(kKtilRowsPerStage, n_krows - ks * kKtilRowsPerStage);
            const int nrow = min(16, rows - warp * 16);   // this warp's rows of the stage
            if (nrow > 0) {
                const float *stage = reinterpret_cast<const float *>(base + s * kStageBytes) + warp * 16 * kD;
                // lane l's partial dot product (dims 4l .. 4l+3) for each of the 16 rows
                float acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float4 v = r < nrow ? reinterpret_cast<const float4 *>(stage + r * kD)[lane]
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                    float sc = f.x * v.x;
                    sc = fmaf(f.y, v.y, sc);
                    sc = fmaf(f.z, v.z, sc);
                    sc = fmaf(f.w, v.w, sc);
                    acc[r] = sc;
                }
                // transposed butterfly: after the exchanges at distances 16, 8, 4, 2 lane l
                // holds row (l >> 1) & 15 summed over the 16 lanes that differ from it in
                // bits 1-4; distance 1 completes it (the same pairwise sums, in the same
                // tree, as a per-row xor reduction over 16, 8, 4, 2, 1)
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
                const bool own = (lane & 1) == 0 && r < nrow;
                const int j = r0 + ks * kKtilRowsPerStage + warp * 16 + r;
                const uint32_t key = order_key(acc[0]);
                if (own)
                    keys0[j] = key;
                // coarse histogram of the candidates, one atomic per distinct bin
                const bool cand = own && j >= p.n_init && j < nb - p.n_local;
                const uint32_t bin = cand ? key >> kCoarseShift : 0xFFFFFFFFu;
                const uint32_t same = __match_any_sync(0xffffffffu, bin);
                if (cand && lane == __ffs(same) - 1)
                    atomicAdd(coarse0 + bin, static_cast<uint32_t>(__popc(same)));
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive_cluster(dsmem_addr(bar_scored, 0));
        // (2) this layer's attention over the staged slice of its block list
        if (ATTN)
            named_barrier_sync(1, kAttnThreads);
        const int n_run = ATTN && ok ? ctrl[kCtrlList] : 0;
        for (int i = 0; i < n_run; ++i, ++it) {
            const int s = it % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (it / kStages) & 1, kWaitNs))) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                break;
            }
            const int logical = llog[i];
            const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
            if (logical >= 0 && tok0 < len)
                attend_block<NT, false>(st, q, base_s + s * kStageBytes, tok0, len, 0xffffffffu, p.scale_log2, warp,
                                        lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        finish_row_sums<NT>(st);
    } else {
        // ------------------------------------------------------------ selector (CTA 0)
        if (rank == 0 && do_sel) {
            if (len_bad && lane == 0)
                report(p.status, SPARSE_ERR_BAD_INDEX);
            bool ready = true;
            if (score)
                ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
            if (ready) {
                topk_warp(base_s + fused_off_keys(per), base_s + fused_off_hist(), base_s + fused_off_topk_list(), nb,
                          p.n_init, p.n_local, p.k_sel,
                          p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next, p.count_next + pair,
                          p.status, lane);
            } else if (lane == 0) {
                report(p.status, SPARSE_ERR_TIMEOUT);
            }
        }
        cluster_wait();
    }

    // ---------------------------------------------------------------- merge
    if (ATTN) {
        __syncthreads();
        cluster_merge_write<NT, false>(st, base, false, p, b, g, 0, p.G, rank, S, kFThreads);
    }
}

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
//   3. s_j = sum_h exp2(a^h_j - M_h) / Z_h -> order key -> CTA 0 (keys and coarse
//      histogram), and CTA 0's selector warp takes the top-k.

constexpr int kMaxHeadsSel = 16;
constexpr int kCtrlStatsBar = 10;   // ctrl[10..11]
constexpr int kCtrlNormBar = 12;    // ctrl[12..13]
constexpr int kCtrlThrWords = 4;    // ctrl[4..5]: the running threshold of the top-k search
constexpr int kHeadsTopkThreads = (kConsumerWarps + 1) * 32;   // CTA 0's consumers + selector

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
    uint32_t *hist = reinterpret_cast<uint32_t *>(base + fused_off_hist());
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
    if (rank == 0 && score)
        for (int i = tid; i < kCoarseBins; i += kFThreads)
            hist[i] = 0u;
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
            for (int h = warp; h < G; h += kConsumerWarps) {
                float m = -INFINITY;
                for (int i = lane; i < n_krows; i += 32)
                    m = fmaxf(m, raw[h * rows_max + i]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                float z = 0.f;
                if (m != -INFINITY)
                    for (int i = lane; i < n_krows; i += 32)
                        z += exp2f(raw[h * rows_max + i] - m);
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
            // (3) summed per-head distributions -> keys and coarse histogram in CTA 0
            const bool have_norm = __all_sync(0xffffffffu, mbar_wait_cluster(bar_norm, 0, kWaitNs));
            if (!have_norm) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
            } else {
                for (int ib = warp * 32; ib < n_krows; ib += kConsumerWarps * 32) {
                    const int i = ib + lane;
                    const bool in = ok && i < n_krows;
                    float sum = 0.f;
                    if (in)
                        for (int h = 0; h < G; ++h)
                            sum += exp2f(raw[h * rows_max + i] - norm[2 * h]) * norm[2 * h + 1];
                    const int j = r0 + i;
                    if (in)
                        keys0[j] = order_key(sum);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_scored, 0));
            if (rank == 0) {
                // CTA 0's consumers join its selector warp in the threshold search (the
                // summed probabilities share an exponent: a coarse histogram of the top
                // key bits would not narrow them)
                if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs)) && lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                uint32_t prefix;
                int need;
                topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + fused_off_hist(),
                                   base_s + kOffCtrl + 4 * kCtrlThrWords, tid + 32, kHeadsTopkThreads, 3, prefix, need);
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
            if (score)
                topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + fused_off_hist(),
                                   base_s + kOffCtrl + 4 * kCtrlThrWords, lane, kHeadsTopkThreads, 3, prefix, need);
            if (ready) {
                topk_write_warp(base_s + L.off_keys, 0u, 0, nb, p.n_init, p.n_local,
                                max(0, nb - p.n_local - p.n_init) <= p.k_sel, p.k_sel <= 0, prefix, need,
                                p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next,
                                p.count_next + pair, p.status, lane);
            } else if (lane == 0) {
                report(p.status, SPARSE_ERR_TIMEOUT);
            }
        }
        cluster_wait();
    }
}

static_assert(4 * kCtrlNormBar + 8 <= 64, "ctrl layout");
static_assert(kCtrlThrWords >= 4 && 4 * kCtrlThrWords + 8 <= 4 * kCtrlScoredBar, "ctrl layout: threshold words");
static_assert((kHeadsTopkThreads / 32) * 256 <= kCoarseBins + kTopkList, "multi-head radix bins");

// The "scored" barrier lives in the ctrl words, 8-byte aligned.
static_assert((kOffCtrl + 4 * kCtrlScoredBar) % 8 == 0 && 4 * kCtrlScoredBar + 8 <= 64, "ctrl layout");

template <int NT, bool ATTN>
int launch_fused(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int S, long long pairs,
                 size_t smem, int device, cudaStream_t stream)
{
    auto kern = decode_forecast_kernel<NT, ATTN>;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), static_cast<int>(smem), device,
                                       configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    CUtensorMap kmap = km, vmap = vm;
    AttnParams prm = p;
    void *args[] = {&kmap, &vmap, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse_decode_attn_forecast launch");
}

}  // namespace

extern "C" SPARSE_API int sparse_decode_attn_forecast(
    const uint16_t *Q, const uint16_t *k_cache, const uint16_t *v_cache, long long T_cap, const int *blk_idx,
    const int *count, int k_tot, const int *seq_len, int B, int H_q, int H_kv, float scale, uint16_t *O, float *lse,
    const uint16_t *F, const float *ktil_next, int N_cap, int n_init, int n_local, int k, int *idx_next,
    int *count_next, int k_tot_next, int n_split, unsigned flags, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!Q || !k_cache || !v_cache || !blk_idx || !count || !seq_len || !O)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: null pointer");
    if (!aligned16(Q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(O))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: Q, K, V and O must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k_tot < 1 || T_cap < 1)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: bad size (B=%d H_q=%d H_kv=%d k_tot=%d)",
                    B, H_q, H_kv, k_tot);
    if (T_cap > INT_MAX - 2 * kBlk)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: T_cap too large");
    if (!isfinite(scale))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: scale must be finite");
    const int G = H_q / H_kv;
    if (G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: G=%d > 16", G);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: B*H_kv=%lld > 65535", pairs);
    if ((flags & ~SPARSE_ATTN_BLOCKS_READY) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: unknown flags 0x%x", flags);
    const bool do_sel = F != nullptr;
    if (do_sel) {
        if (!ktil_next || !idx_next || !count_next)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: F given without ktil_next, idx_next "
                        "or count_next");
        if (!aligned16(F) || !aligned16(ktil_next))
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: F and ktil_next must be 16-byte aligned");
        if (N_cap < 1 || n_init < 0 || n_local < 0 || k < 0)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: bad selection size");
        if (static_cast<long long>(n_init) + n_local + k > k_tot_next)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_forecast: k_tot_next=%d < n_init+n_local+k",
                        k_tot_next);
    } else {
        N_cap = 0;
    }
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    int S;
    if ((rc = choose_split(n_split, pairs, k_tot, dev.sm_count, &S)) != SPARSE_OK)
        return rc;
    const int per = (k_tot + S - 1) / S;
    if (per > kMaxListCta)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: %d blocks per CTA (at most %d)", per,
                    kMaxListCta);
    const size_t smem = fused_smem_bytes(per, N_cap);
    if (smem > static_cast<size_t>(dev.max_smem_optin))
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: N_cap=%d needs %zu bytes of shared memory",
                    N_cap, smem);
    AttnParams p = {};
    p.Q = Q;
    p.O = O;
    p.lse = lse;
    p.blk_logical = blk_idx;
    p.count = count;
    p.seq_len = seq_len;
    p.status = status;
    p.pair_stride = T_cap;
    p.k_tot = k_tot;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.n_groups = 1;
    p.flags = flags;
    p.scale_log2 = scale_log2_of(scale);
    p.F = F;
    p.ktil = ktil_next;
    p.idx_next = idx_next;
    p.count_next = count_next;
    p.N_cap = N_cap;
    p.n_init = n_init;
    p.n_local = n_local;
    p.k_sel = k;
    p.k_tot_next = k_tot_next;
    CUtensorMap km, vm;
    if ((rc = sp_host::make_kv_tensor_map(&km, k_cache, T_cap, pairs)) != SPARSE_OK)
        return rc;
    if ((rc = sp_host::make_kv_tensor_map(&vm, v_cache, T_cap, pairs)) != SPARSE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return G <= 8 ? launch_fused<1, true>(p, km, vm, S, pairs, smem, dev.device, st)
                  : launch_fused<2, true>(p, km, vm, S, pairs, smem, dev.device, st);
}

extern "C" SPARSE_API int sparse_select_topk(const uint16_t *F, const float *ktil, const int *seq_len, int B,
                                             int H_kv, int N_cap, int n_init, int n_local, int k, int *idx_out,
                                             int *count_out, int k_tot, int *status, void *stream)
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
    // cluster size: enough CTAs to cover the SMs twice, at least 128 key rows per CTA
    int S = 1;
    while (S < kMaxSplit && pairs * S * 2 <= 2LL * dev.sm_count && N_cap / (S * 2) >= 128)
        S *= 2;
    const size_t smem = fused_smem_bytes(0, N_cap);
    if (smem > static_cast<size_t>(dev.max_smem_optin))
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_select_topk: N_cap=%d needs %zu bytes of shared memory", N_cap,
                    smem);
    AttnParams p = {};
    p.seq_len = seq_len;
    p.status = status;
    p.H_kv = H_kv;
    p.k_tot = 0;   // no block list of this layer: selection only
    p.F = F;
    p.ktil = ktil;
    p.idx_next = idx_out;
    p.count_next = count_out;
    p.N_cap = N_cap;
    p.n_init = n_init;
    p.n_local = n_local;
    p.k_sel = k;
    p.k_tot_next = k_tot;
    CUtensorMap unused;
    memset(&unused, 0, sizeof unused);
    return launch_fused<1, false>(p, unused, unused, S, pairs, smem, dev.device, static_cast<cudaStream_t>(stream));
}

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

// ---------------------------------------------------------------- NSA routing
//
// NSA's block selection from its compressed keys (SSV notes, "NSA three-branch math"
// steps 1-2; the per-head softmax summed over the GQA group and the max-pooling onto
// the selection grid as in the multi-head selector above):
//     a^h_j = scale * q_h . khat_j,  p_j = sum_h softmax_j(a^h),
//     s_b   = max { p_j : row j's tokens meet block b },
// then the top-k of the 64-token blocks.  The rows are bf16 (the rows the compressed
// branch attends over), so the scores run on the tensor cores exactly as that branch
// computes them: S^T = Khat Q^T, 16 rows x 8 heads per mma tile.
//
// A cluster of S CTAs per pair.  CTA r owns the selection blocks [r*bpc, (r+1)*bpc)
// and the rows that start in them; it also loads the rows before them that reach into
// its first block (the left halo of the max-pooling), so every block is pooled by one
// CTA from rows in its own shared memory.  Phases, as in the multi-head selector:
//   1. TMA ring of 64-row tiles -> raw scores (log2 units) of the CTA's rows;
//   2. per head, max and sum of exp2 over the owned rows -> CTA 0, which merges them
//      and sends every CTA the head's max and 1 / sum;
//   3. p_j for the CTA's rows and the block maxima as order keys -> CTA 0, whose
//      consumers and selector warp find the top-k threshold together (block-wide radix
//      select: the summed probabilities share an exponent, so a coarse histogram of the
//      top key bits would not narrow them), and the selector writes the list.

namespace {

constexpr int kRouteStageBytes = kTileBytes;   // 64 rows x 128 dims, bf16: two 64 x 64 boxes
constexpr int kRouteTopkThreads = (kConsumerWarps + 1) * 32;   // CTA 0's consumers + selector

struct RouteParams {
    const uint16_t *Q;
    const int *seq_len;
    int *idx;
    int *count;
    int *status;
    int H_q, H_kv, G;
    int n_rows_cap;       // rows per pair in khat
    int cmp_len;          // row geometry: [cmp_stride * j, cmp_stride * j + cmp_len)
    int cmp_stride;
    int block_rows;       // 1: the rows are the 64-token blocks (partial last block included)
    int n_blocks_cap;     // selection blocks with keys in CTA 0
    int rows_cta_max;     // raw-score rows per CTA and the per-head stride (= 4 mod 32: no bank conflicts)
    int stages;
    int n_init, n_local, k_sel, k_tot;
    float scale_log2;
};

struct RouteLayout {
    int off_bars, off_ctrl, off_hist, off_list, off_keys, off_stats, off_norm, off_raw, total;
};

__host__ __device__ inline RouteLayout route_layout(int stages, int n_blocks_cap, int rows_cta_max, int G, int S)
{
    RouteLayout l;
    l.off_bars = stages * kRouteStageBytes;                         // full[stages], empty[stages]
    l.off_ctrl = l.off_bars + 2 * stages * 8;                       // scored / stats / norm mbarriers
    l.off_hist = l.off_ctrl + 64;                                   // CTA 0: [5][256] radix digit bins
    l.off_list = l.off_hist + kCoarseBins * 4;                      // (the bins continue here)
    l.off_keys = l.off_list + kTopkList * 4;                        // CTA 0: [n_blocks_cap] keys
    l.off_stats = l.off_keys + ((n_blocks_cap * 4 + 15) & ~15);     // CTA 0: [S][G] (max, sum)
    l.off_norm = l.off_stats + ((S * G * 8 + 15) & ~15);            // [G] (max, 1 / sum)
    l.off_raw = l.off_norm + ((G * 8 + 15) & ~15);                  // [G][rows_cta_max]
    l.total = l.off_raw + ((rows_cta_max * G * 4 + 15) & ~15);
    return l;
}

// First row whose tokens reach block b (rows [s*j, s*j + l)), at least 0.
__host__ __device__ inline long long route_first_row(long long b, int l, int s)
{
    const long long x = kBlk * b - l;
    return x < 0 ? 0 : x / s + 1;
}

template <int NT>
__global__ void __launch_bounds__(kFThreads, 1) nsa_route_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                  const __grid_constant__ RouteParams p)
{
    griddep_wait();   // every input may be written by the kernel before this one
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const int S = static_cast<int>(gridDim.x);
    const int G = p.G;
    const RouteLayout L = route_layout(p.stages, p.n_blocks_cap, p.rows_cta_max, G, S);
    const uint32_t bar_full = base_s + L.off_bars;
    const uint32_t bar_empty = bar_full + 8 * p.stages;
    const uint32_t bar_scored = base_s + L.off_ctrl;
    const uint32_t bar_stats = base_s + L.off_ctrl + 8;
    const uint32_t bar_norm = base_s + L.off_ctrl + 16;
    uint32_t *keys = reinterpret_cast<uint32_t *>(base + L.off_keys);
    float *stats = reinterpret_cast<float *>(base + L.off_stats);
    float *norm = reinterpret_cast<float *>(base + L.off_norm);
    float *raw = reinterpret_cast<float *>(base + L.off_raw);
    float *prow = raw;   // p_j overwrites head 0's raw score of row j

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(blockIdx.x);
    const int pair = static_cast<int>(blockIdx.y);
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    const int l = p.block_rows ? kBlk : p.cmp_len;
    const int s = p.block_rows ? kBlk : p.cmp_stride;

    const long long len = p.seq_len[b];
    long long nb_ll = len <= 0 ? 0 : (len + kBlk - 1) / kBlk;
    long long R_ll = p.block_rows ? nb_ll : (len < l ? 0 : (len - l) / s + 1);
    const bool len_bad = nb_ll > p.n_blocks_cap || R_ll > p.n_rows_cap;
    nb_ll = nb_ll < p.n_blocks_cap ? nb_ll : p.n_blocks_cap;
    R_ll = R_ll < p.n_rows_cap ? R_ll : p.n_rows_cap;
    const int nb = static_cast<int>(nb_ll), R = static_cast<int>(R_ll);
    const bool take_all = max(0, nb - p.n_local - p.n_init) <= p.k_sel;
    const bool score = !take_all && p.k_sel > 0;
    // this CTA's blocks, its owned rows [o_lo, o_hi) and its loaded rows [j_lo, o_hi)
    const int bpc = (nb + S - 1) / S;
    const int b_lo = min(nb, rank * bpc), b_hi = min(nb, b_lo + bpc);
    const long long o_lo_ll = (static_cast<long long>(kBlk) * b_lo + s - 1) / s;
    const long long o_hi_ll = (static_cast<long long>(kBlk) * b_hi + s - 1) / s;
    const int o_lo = static_cast<int>(o_lo_ll < R ? o_lo_ll : R);
    const int o_hi = static_cast<int>(o_hi_ll < R ? o_hi_ll : R);
    const long long first_ll = route_first_row(b_lo, l, s);
    const int j_lo = static_cast<int>(first_ll < o_lo ? first_ll : o_lo);
    const int n_loc = score && b_hi > b_lo ? o_hi - j_lo : 0;
    const int n_tiles = (n_loc + kBlk - 1) / kBlk;

    if (tid == 0) {
        for (int st = 0; st < p.stages; ++st) {
            mbar_init(bar_full + 8 * st, 1);
            mbar_init(bar_empty + 8 * st, kConsumerWarps);
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
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&kmap);
            const uint64_t pol = policy_evict_first();
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % p.stages;
                const int use = t / p.stages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * st, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const uint32_t dst = base_s + st * kRouteStageBytes;
                const int row = j_lo + t * kBlk;
                mbar_arrive_expect_tx(bar_full + 8 * st, kRouteStageBytes);
                tma_load_3d(dst, &kmap, bar_full + 8 * st, 0, row, pair, pol);
                tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * st, 64, row, pair, pol);
            }
        }
        cluster_wait();
    } else if (warp < kConsumerWarps) {
        // ------------------------------------------------------------ consumers
        QueryFrags<NT> q;
        {
            AttnParams ap = {};
            ap.Q = p.Q;
            ap.H_q = p.H_q;
            ap.G = G;
            load_query<NT, false>(q, ap, b, g, 0, G, lane);
        }
        cluster_wait();
        uint32_t *keys0 = static_cast<uint32_t *>(__cluster_map_shared_rank(keys, 0));
        float *stats0 = static_cast<float *>(__cluster_map_shared_rank(stats, 0));
        const int g8 = lane >> 2, t4 = lane & 3;
        bool ok = true;
        // (1) raw scores of the loaded rows
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % p.stages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * st, (t / p.stages) & 1, kWaitNs))) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            float sacc[NT][4];
            score_rows<NT>(sacc, q, base_s + st * kRouteStageBytes, warp, lane);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int lr = t * kBlk + warp * 16 + g8 + (i >> 1) * 8;
                    const int h = nt * 8 + 2 * t4 + (i & 1);
                    if (lr < n_loc && h < G)
                        raw[h * p.rows_cta_max + lr] = sacc[nt][i] * p.scale_log2;
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * st);
        }
        named_barrier_sync(2, kConsumerWarps * 32);   // every raw score is written
        if (score) {
            // (2) per head: max and sum of exp2 over the owned rows, merged by CTA 0
            const int own0 = o_lo - j_lo, own1 = b_hi > b_lo ? o_hi - j_lo : own0;
            for (int h = warp; h < G; h += kConsumerWarps) {
                float m = -INFINITY;
                const float *rh = raw + h * p.rows_cta_max;
                float z = 0.f;
                for (int i = own0 + lane; i < own1; i += 32) {   // one pass: running max and sum
                    const float a = rh[i];
                    if (a > m) {
                        z = z * exp2f(m - a) + 1.f;
                        m = a;
                    } else {
                        z += exp2f(a - m);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
                    const float zo = __shfl_xor_sync(0xffffffffu, z, o);
                    const float mn = fmaxf(m, mo);
                    z = (m == -INFINITY ? 0.f : z * exp2f(m - mn)) + (mo == -INFINITY ? 0.f : zo * exp2f(mo - mn));
                    m = mn;
                }
                if (lane == 0) {
                    stats0[(rank * G + h) * 2] = m;
                    stats0[(rank * G + h) * 2 + 1] = z;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_stats, 0));
            const bool have_norm = __all_sync(0xffffffffu, mbar_wait_cluster(bar_norm, 0, kWaitNs));
            if (!have_norm && lane == 0)
                report(p.status, SPARSE_ERR_TIMEOUT);
            // (3) p_j of the loaded rows, then the block maxima -> keys of CTA 0 (every
            // consumer warp reaches the barrier, whatever its wait gave)
            if (have_norm)
                for (int i = tid; i < n_loc; i += kConsumerWarps * 32) {
                    float sum = 0.f;
                    for (int h = 0; h < G; ++h)
                        sum += exp2f(raw[h * p.rows_cta_max + i] - norm[2 * h]) * norm[2 * h + 1];
                    prow[i] = sum;   // prow aliases head 0's scores: row i is this thread's alone
                }
            named_barrier_sync(2, kConsumerWarps * 32);
            if (have_norm) {
                for (int bb = b_lo + warp * 32; bb < b_hi; bb += kConsumerWarps * 32) {
                    const int blk = bb + lane;
                    const bool in = ok && blk < b_hi;
                    float best = 0.f;
                    if (in) {
                        const int r0 = static_cast<int>(route_first_row(blk, l, s));
                        const int r1 = min(R - 1, static_cast<int>((static_cast<long long>(kBlk) * blk + kBlk - 1) / s));
                        for (int j = r0; j <= r1; ++j)
                            best = fmaxf(best, prow[j - j_lo]);
                    }
                    if (in)
                        keys0[blk] = order_key(best);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_scored, 0));
            if (rank == 0) {
                // CTA 0's consumers join its selector warp in the threshold search
                if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs)) && lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                uint32_t prefix;
                int need;
                topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + L.off_hist,
                                   base_s + L.off_ctrl + 32, tid + 32, kRouteTopkThreads, 3, prefix, need);
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
                    norm[2 * lane] = M;
                    norm[2 * lane + 1] = Z > 0.f ? 1.f / Z : 0.f;
                }
                __syncwarp();
                if (ready && lane < S && lane > 0) {
                    float *peer = static_cast<float *>(__cluster_map_shared_rank(norm, static_cast<unsigned>(lane)));
                    for (int i = 0; i < 2 * G; ++i)
                        peer[i] = norm[i];
                }
                __syncwarp();
                if (ready && lane < S)
                    mbar_arrive_cluster(dsmem_addr(bar_norm, static_cast<uint32_t>(lane)));
                if (ready)
                    ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
            }
            // the top-k threshold with CTA 0's consumers (this warp is warp 0 of the
            // group), then the list
            uint32_t prefix = 0u;
            int need = 0;
            if (score)
                topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + L.off_hist,
                                   base_s + L.off_ctrl + 32, lane, kRouteTopkThreads, 3, prefix, need);
            if (ready) {
                topk_write_warp(base_s + L.off_keys, 0u, 0, nb, p.n_init, p.n_local,
                                max(0, nb - p.n_local - p.n_init) <= p.k_sel, p.k_sel <= 0, prefix, need,
                                p.idx + static_cast<size_t>(pair) * p.k_tot, p.k_tot, p.count + pair, p.status, lane);
            } else if (lane == 0) {
                report(p.status, SPARSE_ERR_TIMEOUT);
            }
        }
        cluster_wait();
    }
}

static_assert((kRouteTopkThreads / 32) * 256 <= kCoarseBins + kTopkList, "routing radix bins");

template <int NT>
int launch_route(const RouteParams &p, const CUtensorMap &km, int S, long long pairs, size_t smem, int device,
                 cudaStream_t stream)
{
    auto kern = nsa_route_kernel<NT>;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), static_cast<int>(smem), device,
                                       configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kFThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    CUtensorMap kmap = km;
    RouteParams prm = p;
    void *args[] = {&kmap, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse_nsa_select launch");
}

}  // namespace

extern "C" SPARSE_API int sparse_nsa_select(const uint16_t *Q, const uint16_t *khat, int n_rows_cap, int cmp_len,
                                            int cmp_stride, const int *seq_len, int B, int H_q, int H_kv,
                                            float scale, int n_init, int n_local, int k, int *idx_out,
                                            int *count_out, int k_tot, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    const char *name = "sparse_nsa_select";
    if (!Q || !khat || !seq_len || !idx_out || !count_out)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(Q) || !aligned16(khat))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: Q and khat must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || n_rows_cap < 1 || n_init < 0 || n_local < 0 || k < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size", name);
    if (!(cmp_len == 0 && cmp_stride == 0) && !(cmp_stride >= 1 && cmp_stride <= cmp_len && cmp_len <= 1024))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: cmp_len=%d cmp_stride=%d", name, cmp_len, cmp_stride);
    if (!isfinite(scale) || scale < 0.f)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: scale must be finite and >= 0", name);
    if (static_cast<long long>(n_init) + n_local + k > k_tot)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: k_tot=%d < n_init+n_local+k", name, k_tot);
    const int G = H_q / H_kv;
    if (G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: G=%d > 16", name, G);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: B*H_kv=%lld > 65535", name, pairs);
    if (n_rows_cap > INT_MAX / 64)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: n_rows_cap too large", name);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    const bool block_rows = cmp_len == 0;
    const int l = block_rows ? kBlk : cmp_len, s = block_rows ? kBlk : cmp_stride;
    // the blocks a length with n_rows_cap rows can have
    const long long nbc = block_rows ? n_rows_cap
                                     : (static_cast<long long>(s) * n_rows_cap + l + kBlk - 1) / kBlk;
    const int n_blocks_cap = static_cast<int>(nbc);
    // S: CTAs per pair, one CTA per SM (a CTA keeps its rows' raw scores in shared
    // memory): the most with pairs * S <= SMs (one wave), then more if the rows do not
    // fit; stages: as many of 2..6 as fit.
    int S = 1;
    while (S < kMaxSplit && pairs * S * 2 <= dev.sm_count && n_blocks_cap / (S * 2) >= 16)
        S *= 2;
    // rows a CTA loads at most (its blocks' rows and the left halo), rounded to 4 mod 32
    auto rows_for = [&](int S_) {
        const long long bpc = (n_blocks_cap + S_ - 1) / S_;
        const long long rows = (kBlk * bpc + s - 1) / s + (l + s - 1) / s + 1;
        return static_cast<int>((rows + 27) / 32 * 32 + 4);
    };
    RouteLayout L = route_layout(2, n_blocks_cap, rows_for(S), G, S);
    while (static_cast<size_t>(L.total) + 1024 > static_cast<size_t>(dev.max_smem_optin) && S < kMaxSplit) {
        S *= 2;
        L = route_layout(2, n_blocks_cap, rows_for(S), G, S);
    }
    int stages = 2;
    while (stages < 6 &&
           static_cast<size_t>(route_layout(stages + 1, n_blocks_cap, rows_for(S), G, S).total) + 1024 <=
               static_cast<size_t>(dev.max_smem_optin))
        ++stages;
    L = route_layout(stages, n_blocks_cap, rows_for(S), G, S);
    const size_t smem = static_cast<size_t>(L.total) + 1024;
    if (smem > static_cast<size_t>(dev.max_smem_optin))
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: n_rows_cap=%d needs %zu bytes of shared memory", name, n_rows_cap,
                    smem);
    CUtensorMap km;
    if ((rc = sp_host::make_kv_tensor_map(&km, khat, n_rows_cap, pairs)) != SPARSE_OK)
        return rc;
    RouteParams p = {};
    p.Q = Q;
    p.seq_len = seq_len;
    p.idx = idx_out;
    p.count = count_out;
    p.status = status;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.n_rows_cap = n_rows_cap;
    p.cmp_len = cmp_len;
    p.cmp_stride = cmp_stride;
    p.block_rows = block_rows ? 1 : 0;
    p.n_blocks_cap = n_blocks_cap;
    p.rows_cta_max = rows_for(S);
    p.stages = stages;
    p.n_init = n_init;
    p.n_local = n_local;
    p.k_sel = k;
    p.k_tot = k_tot;
    p.scale_log2 = scale_log2_of(scale);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return G <= 8 ? launch_route<1>(p, km, S, pairs, smem, dev.device, st)
                  : launch_route<2>(p, km, S, pairs, smem, dev.device, st);
}

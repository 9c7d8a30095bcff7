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
//     that holds the k-th largest key, lists the candidates at or above it, finds the
//     remaining bits by a binary search over that list held in registers and writes the
//     list from the same registers, while (in the fused launch) the consumers attend.
//   * The dependent launch is allowed at once: a following launch starts streaming its
//     key slice as SMs free up, and waits for this one before reading what it writes.
//   * The CTAs' partial softmax states merge by push (cluster_merge_write): CTA 0 tells
//     the others when its ring is free (with the group top-k, where CTA 0 attends over
//     nothing, as soon as the scores are in), they copy their states into it and leave,
//     and CTA 0 writes O; no cluster-wide barrier at the end of the layer.
#include <string.h>

#include <mutex>

#include "attn_core.cuh"
#include "select_core.cuh"
#include "select_layout.cuh"

namespace {

// ATTN = false: the Forecast selection alone (sparse_select_topk): no block list, no
// attention, no merge; every input may be written by the kernel before this one.
// MAXS: the largest cluster the launch may use (16 for the non-portable size).  SELG:
// CTA 0's consumer warps and its selector warp take the top-k together (else the
// selector warp alone, while the consumers attend); a separate instantiation, so the
// kernels that never use the group top-k carry none of its code.
template <int NT, bool ATTN, int MAXS, bool SELG>
__global__ void __launch_bounds__(kFThreads, 2)
    decode_forecast_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const AttnParams p)
{
    // the selection alone waits for the kernel before it unless the caller promised that
    // the candidates' compressed keys and seq_len are complete (SPARSE_SELECT_KEYS_READY):
    // then the key stream starts at once and only F waits (consumers, below)
    if (!ATTN && (p.flags & SPARSE_SELECT_KEYS_READY) == 0u)
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
    if (ATTN && tid == kConsumerWarps * 32) {   // fetched while the keys stream
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    const uint32_t S = gridDim.x;       // the cluster spans gridDim.x
    const uint32_t rank = blockIdx.x;   // == %cluster_ctarank
    const int pair = blockIdx.y;
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    const int per = fused_slice_max(p.k_tot, static_cast<int>(S), SELG);   // the list words' layout
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
    // the top-k by CTA 0's consumer and selector warps together (else its selector warp
    // alone, while the consumers attend); then CTA 0 attends over nothing and the other
    // CTAs share this layer's list (the same decision in every CTA of the cluster)
    const bool group = SELG && score && p.k_sel >= 1 &&
                       topk_cta_regs_fits<kSelKPT>(nb - p.n_local - p.n_init, kSelThreads);
    const bool sel_group = group && rank == 0;
    // ... and with the pull merge CTA 0 (no state of its own) sits the merge out: it
    // arrives on the merge's first cluster barrier before its top-k, so the other CTAs
    // merge and write O while it selects
    const bool skip0 = ATTN && group && !merge_pushes<NT>(S);
    const bool cta0_out = skip0 && rank == 0;
    int i0, cap;
    fused_slice(p.k_tot, static_cast<int>(S), static_cast<int>(rank), group, &i0, &cap);
    // CTA r streams its slice of the candidates [n_init, nb - n_local) only: init and
    // local blocks are never scored (and the local ones may be the ones an append writes)
    const int n_cand = max(0, nb - p.n_local - p.n_init);
    const int chunk = (n_cand + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int r0 = score ? p.n_init + min(n_cand, static_cast<int>(rank) * chunk) : 0;
    const int n_krows = score ? p.n_init + min(n_cand, static_cast<int>(rank + 1) * chunk) - r0 : 0;
    const int n_kst = (n_krows + kKtilRowsPerStage - 1) / kKtilRowsPerStage;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_scored, S * kConsumerWarps);
        if (ATTN)
            merge_barriers_init(base_s + kOffCtrl, S, kFThreads);
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
    bool go_sent = false;   // warp 0 of CTA 0: the push merge's "go" already sent

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
        if (cta0_out)
            cluster_arrive();   // the merge's first barrier
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
                const bool cand = own;   // every streamed row is a candidate
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
        if (cta0_out)
            cluster_arrive();   // the merge's first barrier
        if (sel_group) {
            // CTA 0: once every CTA has scored its slice, the top-k with the selector warp
            const bool ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
            // every warp of this CTA is past its last key stage and it attends over
            // nothing: its ring is free, so the peers may push their states into it while
            // the top-k runs
            if (ATTN && ready && warp == 0 && merge_pushes<NT>(S)) {
                merge_send_go(base_s + kOffCtrl, S, lane);
                go_sent = true;
            }
            topk_forecast_cta<kSelKPT, kSelThreads / 32>(
                base_s + fused_off_keys(per), base_s + fused_off_hist(), base_s + fused_off_hist(), nb, p.n_init,
                p.n_local, p.k_sel, tid, kSelBar, ready, p.idx_next + static_cast<size_t>(pair) * p.k_tot_next,
                p.k_tot_next, p.count_next + pair, p.status);
        }
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
        if (cta0_out) {
            cluster_wait();
            cluster_arrive();   // the merge's first barrier
        }
        if (rank == 0 && do_sel) {
            if (len_bad && lane == 0)
                report(p.status, SPARSE_ERR_BAD_INDEX);
            bool ready = true;
            if (score)
                ready = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
            if (sel_group) {
                topk_forecast_cta<kSelKPT, kSelThreads / 32>(
                    base_s + fused_off_keys(per), base_s + fused_off_hist(), base_s + fused_off_hist(), nb, p.n_init,
                    p.n_local, p.k_sel, kConsumerWarps * 32 + lane, kSelBar, ready,
                    p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next, p.count_next + pair,
                    p.status);
            } else if (ready) {
                topk_warp(base_s + fused_off_keys(per), base_s + fused_off_hist(), base_s + fused_off_topk_list(), nb,
                          p.n_init, p.n_local, p.k_sel,
                          p.idx_next + static_cast<size_t>(pair) * p.k_tot_next, p.k_tot_next, p.count_next + pair,
                          p.status, lane);
            } else if (lane == 0) {
                report(p.status, SPARSE_ERR_TIMEOUT);
            }
        }
        if (!cta0_out)
            cluster_wait();
    }

    // ---------------------------------------------------------------- merge
    if (cta0_out) {
        // the others merge without this CTA; the second barrier: they are done with the cluster
        cluster_wait();
        cluster_sync();
    } else if (ATTN) {
        __syncthreads();
        cluster_merge_write<NT, false, MAXS>(st, base, false, p, b, g, 0, p.G, rank, S, kFThreads,
                                             base_s + kOffCtrl, false, true, false, go_sent, skip0);
    }
}

// The "scored" barrier lives in the ctrl words, 8-byte aligned.
static_assert((kOffCtrl + 4 * kCtrlScoredBar) % 8 == 0 && 4 * kCtrlScoredBar + 8 <= 64, "ctrl layout");

// Blocks per CTA up to which the fused layer's CTA 0 takes its top-k with its consumer
// warps before attending.
constexpr int kSelBlockMaxPer = 12;

template <int NT, bool ATTN, int MAXS, bool SELG>
cudaError_t fused_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute (&attr)[2], int S, long long pairs, size_t smem,
                         cudaStream_t stream)
{
    *cfg = {};
    cfg->gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg->blockDim = dim3(kFThreads, 1, 1);
    cfg->dynamicSmemBytes = smem;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 2;
    return cudaSuccess;
}

// Configure the kernel for this device once (shared memory, carveout and, for MAXS > 8,
// the non-portable cluster size).
template <int NT, bool ATTN, int MAXS, bool SELG>
int configure_fused(size_t smem, int device)
{
    auto kern = decode_forecast_kernel<NT, ATTN, MAXS, SELG>;
    static int configured[64];
    if (MAXS > kMaxSplit && device >= 0 && device < 64 && configured[device] < static_cast<int>(smem) + 1) {
        const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(kern),
                                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess)
            return sp_host::cuda_status(e, "cudaFuncSetAttribute(non-portable cluster size)");
    }
    return sp_host::configure_kernel(reinterpret_cast<const void *>(kern), static_cast<int>(smem), device,
                                     configured);
}

// Whether clusters of 16 CTAs of the wide kernel fit on this device with this shared
// memory (the occupancy query, remembered per device for the largest size that fit and
// the smallest that did not).
std::mutex g_wide_mu;
size_t g_wide_fit[64], g_wide_nofit[64];

template <int NT>
bool wide_clusters_fit(size_t smem, long long pairs, int device, cudaStream_t stream)
{
    if (device < 0 || device >= 64)
        return false;
    {
        std::lock_guard<std::mutex> lock(g_wide_mu);
        if (smem <= g_wide_fit[device])
            return true;
        if (g_wide_nofit[device] != 0 && smem >= g_wide_nofit[device])
            return false;
    }
    if (configure_fused<NT, true, 16, true>(smem, device) != SPARSE_OK)
        return false;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fused_config<NT, true, 16, true>(&cfg, attr, 16, pairs, smem, stream);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(
        &n, reinterpret_cast<const void *>(decode_forecast_kernel<NT, true, 16, true>), &cfg);
    if (e != cudaSuccess)
        (void)cudaGetLastError();   // a failed query leaves a (non-sticky) error behind: clear it
    const bool fit = e == cudaSuccess && n >= 1;
    std::lock_guard<std::mutex> lock(g_wide_mu);
    if (fit && smem > g_wide_fit[device])
        g_wide_fit[device] = smem;
    if (!fit && (g_wide_nofit[device] == 0 || smem < g_wide_nofit[device]))
        g_wide_nofit[device] = smem;
    return fit;
}

template <int NT, bool ATTN, int MAXS, bool SELG>
int launch_fused(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int S, long long pairs,
                 size_t smem, int device, cudaStream_t stream)
{
    auto kern = decode_forecast_kernel<NT, ATTN, MAXS, SELG>;
    int rc = configure_fused<NT, ATTN, MAXS, SELG>(smem, device);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fused_config<NT, ATTN, MAXS, SELG>(&cfg, attr, S, pairs, smem, stream);
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
    // up to 16 CTAs per pair (a non-portable cluster) when few pairs have to fill the GPU
    int S;
    if ((rc = choose_split(n_split, pairs, k_tot, dev.sm_count, &S, 16)) != SPARSE_OK)
        return rc;
    if (S > kMaxSplit && G <= 8 &&
        !wide_clusters_fit<1>(fused_smem_bytes(fused_slice_max(k_tot, S, true), N_cap), pairs, dev.device,
                              static_cast<cudaStream_t>(stream))) {
        if (n_split != 0)
            return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: clusters of 16 CTAs do not fit");
        S = kMaxSplit;
    }
    if (S > kMaxSplit && G > 8) {
        if (n_split != 0)
            return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_forecast: n_split = 16 needs G <= 8");
        S = kMaxSplit;
    }
    // few blocks per CTA: the layer's attention is short, so the top-k is on the path to
    // the next layer and CTA 0's consumers help with it (and leave the layer's list to the
    // other CTAs); many blocks: the selector warp alone, hidden behind the attention
    const bool sel_group = (k_tot + S - 1) / S <= kSelBlockMaxPer && G <= 8;
    const bool group_kernel = S > kMaxSplit || (G <= 8 && sel_group);   // an instantiation with SELG
    const int per = fused_slice_max(k_tot, S, group_kernel);
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
    if (S > kMaxSplit)
        return launch_fused<1, true, 16, true>(p, km, vm, S, pairs, smem, dev.device, st);
    if (G > 8)
        return launch_fused<2, true, kMaxSplit, false>(p, km, vm, S, pairs, smem, dev.device, st);
    return sel_group ? launch_fused<1, true, kMaxSplit, true>(p, km, vm, S, pairs, smem, dev.device, st)
                     : launch_fused<1, true, kMaxSplit, false>(p, km, vm, S, pairs, smem, dev.device, st);
}

namespace {

int select_impl(const uint16_t *F, const float *ktil, const int *seq_len, int B, int H_kv, int N_cap, int n_init,
                int n_local, int k, int *idx_out, int *count_out, int k_tot, unsigned flags, int *status,
                void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if ((flags & ~SPARSE_SELECT_KEYS_READY) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_select_topk_ex: unknown flags 0x%x", flags);
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
    p.flags = flags;
    CUtensorMap unused;
    memset(&unused, 0, sizeof unused);
    // nothing else to do: every warp of CTA 0 takes part in the top-k
    return launch_fused<1, false, kMaxSplit, true>(p, unused, unused, S, pairs, smem, dev.device,
                                                   static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" SPARSE_API int sparse_select_topk(const uint16_t *F, const float *ktil, const int *seq_len, int B,
                                             int H_kv, int N_cap, int n_init, int n_local, int k, int *idx_out,
                                             int *count_out, int k_tot, int *status, void *stream)
{
    return select_impl(F, ktil, seq_len, B, H_kv, N_cap, n_init, n_local, k, idx_out, count_out, k_tot, 0u, status,
                       stream);
}

extern "C" SPARSE_API int sparse_select_topk_ex(const uint16_t *F, const float *ktil, const int *seq_len, int B,
                                                int H_kv, int N_cap, int n_init, int n_local, int k, int *idx_out,
                                                int *count_out, int k_tot, unsigned flags, int *status, void *stream)
{
    return select_impl(F, ktil, seq_len, B, H_kv, N_cap, n_init, n_local, k, idx_out, count_out, k_tot, flags,
                       status, stream);
}

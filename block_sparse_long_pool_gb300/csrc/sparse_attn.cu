// sparse_attn.cu -- block-sparse GQA attention over selected 64-token KV blocks.
//
// One kernel serves two entry points:
//   * sparse_decode_attn (SparDA notes §4.1 eq.(7), Alg.1 step 4): the G query heads
//     of a (batch, KV head) pair attend over the pair's selected blocks.
//   * sparse_verify_attn_grouped (SSV notes, mechanism 1, mode A): the C x G query
//     rows of a group of verification queries attend, each over its own block set,
//     while the group's merged union of blocks is streamed from HBM once.
// Scale 1/sqrt(d) per the SSV notes' NSA selection branch (step 3); split-KV partial
// states are merged with the online-softmax recurrence (SSV notes, "online softmax
// state merging").
//
// GB300 design
//   * A thread-block cluster of S CTAs shares one work unit (pair, or pair x group);
//     CTA r takes the r-th contiguous slice of the unit's block list (split-KV).
//   * Warp 4 is the producer: one lane streams each selected block's K and V
//     (2 x 16 KB) into a 3-stage shared-memory ring with TMA tensor copies
//     (cp.async.bulk.tensor, 64 x 64 boxes, 128-byte swizzle) completing on mbarriers.
//   * Warps 0-3 consume: warp w owns tokens [16w, 16w+16) of every block.  Scores are
//     computed transposed, S^T = K Q^T, on the bf16 tensor cores (mma m16n8k16: 16
//     tokens on M, up to 8 query rows per n-tile on N, head dim on K), so G <= 8 heads
//     fill an n-tile with no padding.  Each warp keeps its own online-softmax state
//     (max, sum, O^T accumulators in fp32); P is rounded to bf16 and transposed in
//     registers with movmatrix to become the B operand of O^T += V^T P^T.
//   * The 4 x S partial states of a unit are merged through distributed shared memory
//     (mapa + ld.shared::cluster); CTA r writes output dims [r*128/S, (r+1)*128/S).
//     No global scratch memory and no second kernel.
//   * Every wait is bounded (mbar_wait, 2 s); an expired wait writes
//     SPARSE_ERR_TIMEOUT to *status and the CTA skips the rest of its work.
//
// Decode with a workspace uses a second kernel, decode_streamk_kernel: a persistent
// grid of two CTAs per SM splits the flattened (pair, selected block) list into equal
// contiguous ranges (stream-K), so every CTA streams the same number of blocks and
// all SMs finish together.  A CTA's range covers whole pairs (written directly) and
// at most two partial pairs; a partial pair's state (the four warp states merged in
// the ring stage just consumed) goes to the workspace, and the CTA that completes the
// pair's last partial merges them and resets the pair's arrival counter.
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

#include "attn_core.cuh"

namespace {

using namespace sp;

// Merged union of the group's block sets (SSV mode A): ulist ascending, umask[u] the
// queries of the group whose set contains ulist[u]; ctrl[kCtrlList] = the union size.
// Up to kUnionBitmapBlocks blocks in the sequence the union comes from a bitmap over
// the blocks (O(entries)); beyond, every entry compares itself with all others.
constexpr int kUnionBitmapBlocks = 4096;
static_assert(2 * (kUnionBitmapBlocks / 32) <= kMaxUnion, "union bitmap and prefix fit the entry scratch");
// Every thread of the CTA (NTHR of them) calls it; ulist / umask [kMaxUnion] and the
// scratch ent_v / ent_m / ent_f [kMaxUnion] are in shared memory.
template <int NTHR>
__device__ __forceinline__ void build_union(const AttnParams &p, int *ulist, uint32_t *umask, int *ent_v,
                                            uint32_t *ent_m, int *ent_f, int b, int g, int q0, int nb, int *ctrl)
{
    const int tid = threadIdx.x;
    const int nq = min(p.C, p.N_q - q0);
    const int wcount = min(p.window_blocks, nb);
    // mode B (shared layout): only the group's first query's set, marked for every query
    const bool shared = (p.flags & kVerifySharedLayout) != 0u;
    const int n_sel_ent = shared ? p.n_sel : nq * p.n_sel;
    const int n_ent = n_sel_ent + wcount;
    const uint32_t all_q = nq >= 32 ? 0xffffffffu : ((1u << nq) - 1u);
    for (int e = tid; e < n_ent; e += NTHR) {
        int v;
        uint32_t m;
        if (e < n_sel_ent) {
            const int qi = e / p.n_sel;
            v = p.idx_q[((static_cast<size_t>(b) * p.H_kv + g) * p.N_q + q0 + qi) * p.n_sel + (e - qi * p.n_sel)];
            m = shared ? all_q : 1u << qi;
            if (v < 0 || v >= nb) {
                report(p.status, SPARSE_ERR_BAD_INDEX);
                v = INT_MAX;
            }
        } else {
            v = nb - wcount + (e - n_sel_ent);
            m = all_q;
        }
        ent_v[e] = v;
        ent_m[e] = m;
    }
    for (int e = tid; e < kMaxUnion; e += NTHR)
        umask[e] = 0u;
    if (nb <= kUnionBitmapBlocks) {
        // a bitmap over the blocks: each entry sets its bit; a block's position in the
        // ascending union is the number of set bits below it
        uint32_t *bits = reinterpret_cast<uint32_t *>(ent_f);              // [kUnionBitmapBlocks / 32]
        uint32_t *pref = bits + kUnionBitmapBlocks / 32;                  // exclusive popcount prefix
        const int nw = (nb + 31) / 32;
        for (int w = tid; w < nw; w += NTHR)
            bits[w] = 0u;
        __syncthreads();
        for (int e = tid; e < n_ent; e += NTHR) {
            const int v = ent_v[e];
            if (v != INT_MAX)
                atomicOr(&bits[v >> 5], 1u << (v & 31));
        }
        __syncthreads();
        if (tid < 32) {
            constexpr int kPer = kUnionBitmapBlocks / 32 / 32;   // words per lane
            int c[kPer], sum = 0;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int w = tid * kPer + i;
                c[i] = w < nw ? __popc(bits[w]) : 0;
                sum += c[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o)
                    incl += n;
            }
            int run = incl - sum;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                pref[tid * kPer + i] = static_cast<uint32_t>(run);
                run += c[i];
            }
            if (tid == 31)
                ctrl[kCtrlList] = incl;
        }
        __syncthreads();
        for (int e = tid; e < n_ent; e += NTHR) {
            const int v = ent_v[e];
            if (v == INT_MAX)
                continue;
            const uint32_t w = bits[v >> 5];
            const int pos = static_cast<int>(pref[v >> 5]) + __popc(w & ((1u << (v & 31)) - 1u));
            ulist[pos] = v;   // equal entries write the same block
            atomicOr(&umask[pos], ent_m[e]);
        }
        return;
    }
    __syncthreads();
    for (int e = tid; e < n_ent; e += NTHR) {
        const int v = ent_v[e];
        int first = v != INT_MAX;
        for (int e2 = 0; e2 < e && first; ++e2)
            first = ent_v[e2] != v;
        ent_f[e] = first;
    }
    __syncthreads();
    for (int e = tid; e < n_ent; e += NTHR) {
        const int v = ent_v[e];
        if (v == INT_MAX)
            continue;
        int pos = 0;
        for (int e2 = 0; e2 < n_ent; ++e2)
            pos += (ent_f[e2] != 0) & (ent_v[e2] < v);
        if (ent_f[e]) {
            ulist[pos] = v;
            atomicAdd(&ctrl[kCtrlList], 1);
        }
        atomicOr(&umask[pos], ent_m[e]);
    }
}

// One CTA of a cluster: unit `unit` (a pair, or a pair x query group), slice `rank` of
// its block list; the cluster's S partial states are merged and written.
template <int NT, bool VERIFY>
__device__ __forceinline__ void attn_cluster_cta(const CUtensorMap *kmap, const CUtensorMap *vmap,
                                                 const AttnParams &p, int unit)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kOffCtrl);
    const uint32_t bar_full = base_s + kOffBars;                 // + 8 * s
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;  // + 8 * s

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t S = gridDim.x;        // the cluster spans gridDim.x
    const uint32_t rank = blockIdx.x;    // == %cluster_ctarank
    if (tid == kConsumerWarps * 32) {    // the descriptor fetches overlap the list fetch
        prefetch_tensormap(kmap);
        prefetch_tensormap(vmap);
    }

    int pair, q0 = 0, rows_valid;
    if (VERIFY) {
        pair = unit / p.n_groups;
        q0 = (unit % p.n_groups) * p.C;
        rows_valid = min(p.C, p.N_q - q0) * p.G;
    } else {
        pair = unit;
        rows_valid = p.G;
    }
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    // Programmatic dependent launch: this grid may start while the kernel before it on
    // the stream drains.  With SPARSE_ATTN_BLOCKS_READY the block list, lengths and K/V
    // are already complete (the caller's promise), so only Q and the outputs wait;
    // otherwise every input may come from that kernel and everything waits.
    const bool early = (p.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();

    if (tid == 0) {
        ctrl[kCtrlAbort] = 0;
        ctrl[kCtrlList] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // Verification: the merged union of the group's block sets (ulist / umask, whole
    // list) is built by every thread; CTA r takes a contiguous slice of it.  Decode:
    // CTA r takes entries [r * ceil(k_tot / S), ...) of the pair's table, which its
    // producer warp fetches together with the count (one round trip) into lslot / llog.
    const int *ulist = reinterpret_cast<const int *>(base + kOffList);
    const uint32_t *umask = reinterpret_cast<const uint32_t *>(base + kOffMask);
    int *lslot = reinterpret_cast<int *>(base + kOffList);
    int *llog = lslot + kMaxListCta;
    long long len = 0;
    int i0 = 0, my_n = 0, n_list = 0;
    if (VERIFY) {
        len = p.seq_len[b];
        const int nb = len <= 0 ? 0 : static_cast<int>((len + kBlk - 1) / kBlk);
        build_union<kThreads>(p, reinterpret_cast<int *>(base + kOffList), reinterpret_cast<uint32_t *>(base + kOffMask),
                              reinterpret_cast<int *>(base + kOffEntV), reinterpret_cast<uint32_t *>(base + kOffEntM),
                              reinterpret_cast<int *>(base + kOffEntF), b, g, q0, nb, ctrl);
        __syncthreads();
        n_list = ctrl[kCtrlList];
        const int per = (n_list + static_cast<int>(S) - 1) / static_cast<int>(S);
        i0 = min(n_list, static_cast<int>(rank) * per);
        my_n = min(n_list, i0 + per) - i0;
        if (rank == 0 && tid == 0 && p.blocks_loaded != nullptr)
            atomicAdd(reinterpret_cast<unsigned long long *>(p.blocks_loaded),
                      static_cast<unsigned long long>(n_list));
    }

    WarpState<NT> st;
    st.reset();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (!VERIFY) {
            const int per = (p.k_tot + static_cast<int>(S) - 1) / static_cast<int>(S);
            i0 = min(p.k_tot, static_cast<int>(rank) * per);
            my_n = producer_fetch_slice(p, pair, i0, min(p.k_tot, i0 + per) - i0, lslot, llog, ctrl, lane);
            named_barrier_arrive(1, kThreads);   // the slice and its length are in shared memory
        }
        if (lane == 0 && my_n > 0) {
            const uint64_t pol = policy_evict_first();
            for (int it = 0; it < my_n; ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const int slot = VERIFY ? ulist[i0 + it] : lslot[it];
                // an invalid slot loads an out-of-range box: zeros, never a fault
                const int row = slot >= 0 ? slot * kBlk : static_cast<int>(min(p.pair_stride, (long long)INT_MAX - kBlk));
                const uint32_t dst = base_s + s * kStageBytes;
                mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                tma_load_3d(dst, kmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kHalfBytes, kmap, bar_full + 8 * s, 64, row, pair, pol);
                tma_load_3d(dst + kTileBytes, vmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, vmap, bar_full + 8 * s, 64, row, pair, pol);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        if (early)
            griddep_wait();   // Q may be written by the kernel before this one
        QueryFrags<NT> q;
        load_query<NT, VERIFY>(q, p, b, g, q0, rows_valid, lane);
        long long tok_lo = 0;
        if (!VERIFY) {
            len = unit_len(p, b);
            if (p.range_mode == 1)
                tok_lo = len - p.win_tokens > 0 ? len - p.win_tokens : 0;
            named_barrier_sync(1, kThreads);
            my_n = ctrl[kCtrlList];
        }
        for (int it = 0; it < my_n; ++it) {
            const int s = it % kStages;
            // the verdict is made warp-uniform: the .aligned tensor-core instructions
            // below must see all 32 lanes
            const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (it / kStages) & 1, kWaitNs));
            if (!landed) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                break;
            }
            int logical;
            uint32_t qmask = 0xffffffffu;
            if (VERIFY) {
                logical = ulist[i0 + it];
                qmask = umask[i0 + it];
            } else {
                logical = llog[it];
            }
            const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
            if (logical >= 0 && tok0 < len)
                attend_block<NT, VERIFY>(st, q, base_s + s * kStageBytes, tok0, len, qmask, p.scale_log2, warp,
                                         lane, tok_lo);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        finish_row_sums<NT>(st);
    }

    // ---------------------------------------------------------------- merge
    // Every stage has been consumed; the ring memory now holds the partial states.
    // The next kernel on the stream may be scheduled from here on.
    __syncthreads();
    griddep_launch_dependents();
    cluster_merge_write<NT, VERIFY>(st, base, ctrl[kCtrlAbort] != 0, p, b, g, q0, rows_valid, rank, S, kThreads,
                                    base_s + kOffCtrl, false, false);
}

template <int NT, bool VERIFY>
__global__ void __launch_bounds__(kThreads, 2)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const __grid_constant__ AttnParams p)
{
    attn_cluster_cta<NT, VERIFY>(&kmap, &vmap, p, static_cast<int>(blockIdx.y));
}

}  // namespace

// The tensor-memory form of the same CTA (it calls build_union above).
#include "attn_tc.cuh"

namespace {

// The split-KV CTA with both contractions on the 5th-generation tensor cores: the
// verification launches and sparse_decode_attn's cluster launch.
template <int NT, bool VERIFY>
__global__ void __launch_bounds__(kTcThreads, 2)
    sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ AttnParams p)
{
    attn_tc_cta<NT, VERIFY>(&kmap, &vmap, p, static_cast<int>(blockIdx.y));
}

// ---------------------------------------------------------------- split-KV decode, workspace merge
//
// CTA (r, p) of a (S, pairs) grid attends over slice r of pair p's block list, a
// slice of ceil(k_tot / S) entries cut from the k_tot-long table (so the slice is
// known before `count` arrives).  Its producer warp fetches the slice and the count in
// one round trip and starts the TMA ring at once.  After the main loop the CTA merges
// its 4 warp states, writes the CTA state (unnormalised O, row max and sum) to the
// workspace and leaves; the CTA of the pair that arrives last merges the S states
// (the online-softmax recurrence, applied to whole partial states) and writes O.
// Early finishers free their SM for the next kernel instead of waiting on peers.

constexpr int kMaxSplitWs = 64;

template <int NT>
__host__ __device__ constexpr int split_part_floats()
{
    return 8 * NT * kD + 2 * 8 * NT + 4;   // O [ROWS][128], m [ROWS], l [ROWS], header
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const AttnParams p)
{
    constexpr int ROWS = 8 * NT;
    constexpr int PART = split_part_floats<NT>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kOffCtrl);
    const uint32_t bar_full = base_s + kOffBars;
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = static_cast<int>(gridDim.x);
    const int rank = static_cast<int>(blockIdx.x);
    const int pair = static_cast<int>(blockIdx.y);
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    if (tid == kConsumerWarps * 32) {   // the descriptor fetches overlap the list fetch
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    const bool early = (p.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();
    const int per = (p.k_tot + S - 1) / S;
    const int i0 = min(p.k_tot, rank * per);
    const int cap = min(p.k_tot, i0 + per) - i0;
    int *lslot = reinterpret_cast<int *>(base + kOffList);
    int *llog = lslot + kMaxListCta;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    WarpState<NT> st;
    st.reset();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const int n_run = producer_fetch_slice(p, pair, i0, cap, lslot, llog, ctrl, lane);
        named_barrier_arrive(1, kThreads);   // the list and its length are in shared memory
        if (lane == 0 && n_run > 0) {
            const uint64_t pol = policy_evict_first();
            for (int it = 0; it < n_run; ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const int slot = lslot[it];
                const int row = slot >= 0 ? slot * kBlk : static_cast<int>(min(p.pair_stride, (long long)INT_MAX - kBlk));
                const uint32_t dst = base_s + s * kStageBytes;
                mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                tma_load_3d(dst, &kmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * s, 64, row, pair, pol);
                tma_load_3d(dst + kTileBytes, &vmap, bar_full + 8 * s, 0, row, pair, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, bar_full + 8 * s, 64, row, pair, pol);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        if (early)
            griddep_wait();   // Q may be written by the kernel before this one
        QueryFrags<NT> q;
        load_query<NT, false>(q, p, b, g, 0, p.G, lane);
        const long long len = p.seq_len[b];
        named_barrier_sync(1, kThreads);
        const int n_run = ctrl[kCtrlList];
        for (int it = 0; it < n_run; ++it) {
            const int s = it % kStages;
            const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (it / kStages) & 1, kWaitNs));
            if (!landed) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                break;
            }
            const int logical = llog[it];
            const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
            if (logical >= 0 && tok0 < len)
                attend_block<NT, false>(st, q, base_s + s * kStageBytes, tok0, len, 0xffffffffu, p.scale_log2,
                                        warp, lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        finish_row_sums<NT>(st);
    }

    // ---------------------------------------------------------------- merge
    __syncthreads();
    griddep_launch_dependents();
    float *wo = reinterpret_cast<float *>(base);                     // [4][ROWS][kWoStride]
    float *wm = wo + kConsumerWarps * ROWS * kWoStride;              // [4][ROWS]
    float *wl = wm + kConsumerWarps * ROWS;
    float *wf = wl + kConsumerWarps * ROWS;
    float *co = wf + kConsumerWarps * ROWS;                          // [ROWS][128] CTA state
    float *cm = co + ROWS * kD;                                      // [ROWS]
    float *cl = cm + ROWS;                                           // [ROWS]
    float *sm = cl + ROWS;                                           // [kMaxSplitWs][ROWS] partial maxima
    float *sl = sm + kMaxSplitWs * ROWS;                             // [kMaxSplitWs][ROWS] partial sums -> weights
    float *rowml = sl + kMaxSplitWs * ROWS;                          // [2][ROWS]
    if (warp < kConsumerWarps)
        store_warp_state<NT>(st, wo, wm, wl, warp, lane);
    __syncthreads();
    merge_warp_states<ROWS>(wo, wm, wl, wf, co, cm, cl, tid, kThreads, [] { __syncthreads(); });
    __syncthreads();
    const float aborted_f = ctrl[kCtrlAbort] != 0 ? 1.f : 0.f;
    float *ws_pair = p.ws_part + static_cast<size_t>(pair) * S * PART;
    if (S > 1) {
        float *part = ws_pair + static_cast<size_t>(rank) * PART;
        for (int q4 = tid; q4 < ROWS * kD / 4; q4 += kThreads)
            __stcg(reinterpret_cast<float4 *>(part) + q4, reinterpret_cast<const float4 *>(co)[q4]);
        if (tid < ROWS) {
            __stcg(part + ROWS * kD + tid, cm[tid]);
            __stcg(part + ROWS * kD + ROWS + tid, cl[tid]);
        }
        if (tid == 0)
            __stcg(part + ROWS * kD + 2 * ROWS, aborted_f);
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const int prev = atomicAdd(p.ws_count + pair, 1);
            const int last = prev == S - 1;
            if (last)
                atomicExch(p.ws_count + pair, 0);   // ready for the next call
            ctrl[kCtrlLast] = last;
        }
        __syncthreads();
        if (!ctrl[kCtrlLast])
            return;
        __threadfence();
    }
    // the last CTA of the pair: row statistics of the S states, then the weighted sum
    int any_abort = 0;
    for (int t = tid; t < S * ROWS; t += kThreads) {
        const int c = t / ROWS, row = t - c * ROWS;
        if (c == rank) {
            sm[t] = cm[row];
            sl[t] = cl[row];
        } else {
            const float *part = ws_pair + static_cast<size_t>(c) * PART;
            sm[t] = __ldcg(part + ROWS * kD + row);
            sl[t] = __ldcg(part + ROWS * kD + ROWS + row);
            if (row == 0)
                any_abort |= __ldcg(part + ROWS * kD + 2 * ROWS) != 0.f;
        }
    }
    any_abort = __syncthreads_or(any_abort || aborted_f != 0.f);
    if (any_abort)
        return;   // a CTA of the pair failed its ready check: O and lse stay untouched
    if (tid < ROWS) {
        const int row = tid;
        float M = -INFINITY;
        for (int c = 0; c < S; ++c)
            M = fmaxf(M, sm[c * ROWS + row]);
        float L = 0.f;
        for (int c = 0; c < S; ++c) {
            const float mc = sm[c * ROWS + row];
            const float f = (M == -INFINITY || mc == -INFINITY) ? 0.f : exp2f(mc - M);
            L += f * sl[c * ROWS + row];
            sl[c * ROWS + row] = f;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int c = 0; c < S; ++c)
            sl[c * ROWS + row] *= inv;
        rowml[row] = M;
        rowml[ROWS + row] = L;
    }
    __syncthreads();
    for (int q4 = tid; q4 < p.G * (kD / 4); q4 += kThreads) {
        const int row = q4 / (kD / 4);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < S; c0 += 4) {
            float4 v[4];
            float f[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + j;
                f[j] = c < S ? sl[c * ROWS + row] : 0.f;
                if (c >= S)
                    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                else if (c == rank)
                    v[j] = reinterpret_cast<const float4 *>(co)[q4];
                else
                    v[j] = __ldcg(reinterpret_cast<const float4 *>(ws_pair + static_cast<size_t>(c) * PART) + q4);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o.x = fmaf(f[j], v[j].x, o.x);
                o.y = fmaf(f[j], v[j].y, o.y);
                o.z = fmaf(f[j], v[j].z, o.z);
                o.w = fmaf(f[j], v[j].w, o.w);
            }
        }
        uint2 packed;
        packed.x = pack_bf16x2(o.x, o.y);
        packed.y = pack_bf16x2(o.z, o.w);
        const size_t out = (static_cast<size_t>(b) * p.H_q + g * p.G + row) * kD + 4 * (q4 % (kD / 4));
        *reinterpret_cast<uint2 *>(p.O + out) = packed;
    }
    if (p.lse != nullptr && tid < p.G)
        p.lse[static_cast<size_t>(b) * p.H_q + g * p.G + tid] = lse_of(rowml[tid], rowml[ROWS + tid]);
}

// The split path's merge scratch must fit in the stage ring it reuses.
static_assert((kConsumerWarps * 16 * kWoStride + 3 * kConsumerWarps * 16 + 16 * kD + 2 * 16 + 2 * kMaxSplitWs * 16 +
               2 * 16) *
                      4 <=
                  kStages * kStageBytes,
              "split merge scratch exceeds the stage ring");

// ---------------------------------------------------------------- stream-K decode

// CTA whose range [N c / C, N (c+1) / C) holds `item`.
__device__ __forceinline__ int cta_of_item(long long item, long long N, long long C)
{
    long long c = item * C / N;
    while (c + 1 < C && N * (c + 1) / C <= item)
        ++c;
    while (c > 0 && N * c / C > item)
        --c;
    return static_cast<int>(c);
}

// Workspace slot holding CTA c's partial state of `pair`: 2c for the first pair of its
// range, 2c+1 for the last.
__device__ __forceinline__ long long part_slot(int c, int pair, long long N, long long C, int K)
{
    const long long first_pair = (N * c / C) / K;
    return 2LL * c + (pair == first_pair ? 0 : 1);
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_streamk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const AttnParams p)
{
    constexpr int ROWS = 8 * NT;
    constexpr int PART = ROWS * kD + 2 * ROWS + 1;   // o, max, sum, valid flag
    static_assert((kConsumerWarps * ROWS * kWoStride + 3 * kConsumerWarps * ROWS + ROWS * kD + 2 * ROWS) * 4 <=
                      kStageBytes,
                  "a segment's warp and CTA states fit the one stage it holds");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kOffCtrl);
    int *lslot = reinterpret_cast<int *>(base + kOffList);
    int *llog = lslot + kMaxListCta;
    int *seg_nv = reinterpret_cast<int *>(base + kOffSegs);
    int *seg_start = seg_nv + kMaxSegs;
    float *row_m = reinterpret_cast<float *>(base + kOffRowML);
    float *row_l = row_m + 16;
    const uint32_t bar_full = base_s + kOffBars;
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long C = gridDim.x;
    const int c = static_cast<int>(blockIdx.x);
    const long long N = p.n_items;
    const int K = p.k_tot;
    const long long lo = N * c / C, hi = N * (c + 1) / C;
    const long long p_first = lo / K;
    const int n_segs = hi > lo ? static_cast<int>((hi - 1) / K - p_first + 1) : 0;
    if (tid == kConsumerWarps * 32) {   // the descriptor fetches overlap the list fetch
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }

    const bool early = (p.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();

    if (tid == 0) {
        ctrl[kCtrlAbort] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
        if (p.ready_flag != nullptr) {
            bool ok = false;
            const uint64_t t0 = globaltimer();
            for (uint32_t it = 0; it < (1u << 26); ++it) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.ready_flag) : "memory");
                if (v >= p.ready_target) {
                    ok = true;
                    break;
                }
                if (p.timeout_ns <= 0 || globaltimer() - t0 > static_cast<uint64_t>(p.timeout_ns))
                    break;
                __nanosleep(256);
            }
            if (!ok) {
                ctrl[kCtrlAbort] = 1;
                report(p.status, p.timeout_ns > 0 ? SPARSE_ERR_TIMEOUT : SPARSE_ERR_NOT_READY);
            }
        }
    }
    // segment table: valid items of every pair the range touches, and their offsets in
    // the CTA's compact list
    if (warp == 0) {
        int carry = 0;
        for (int s0 = 0; s0 < n_segs; s0 += 32) {
            const int s = s0 + lane;
            int nv = 0;
            if (s < n_segs) {
                const long long pair = p_first + s;
                const long long ia = max(lo, pair * K) - pair * K, ib = min(hi, (pair + 1) * K) - pair * K;
                int cnt = p.count[pair];
                if (cnt < 0 || cnt > K) {
                    report(p.status, SPARSE_ERR_BAD_INDEX);
                    cnt = cnt < 0 ? 0 : K;
                }
                nv = static_cast<int>(max(0LL, min(ib, static_cast<long long>(cnt)) - ia));
            }
            int incl = nv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += n;
            }
            if (s < n_segs) {
                seg_nv[s] = nv;
                seg_start[s] = carry + incl - nv;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    const bool aborted = ctrl[kCtrlAbort] != 0;
    // the CTA's compact block list, validated (-1 = skip: an out-of-range box is loaded)
    if (!aborted) {
        for (int s = 0; s < n_segs; ++s) {
            const long long pair = p_first + s;
            const long long ia = max(lo, pair * K) - pair * K;
            for (int t = tid; t < seg_nv[s]; t += kThreads) {
                const size_t at = static_cast<size_t>(pair * K + ia + t);
                const int logical = p.blk_logical[at];
                const int slot = p.blk_slot != nullptr ? p.blk_slot[at] : logical;
                const bool ok = logical >= 0 && slot >= 0 && static_cast<long long>(slot) * kBlk < p.pair_stride;
                if (!ok)
                    report(p.status, SPARSE_ERR_BAD_INDEX);
                lslot[seg_start[s] + t] = ok ? slot : -1;
                llog[seg_start[s] + t] = ok ? logical : -1;
            }
        }
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !aborted) {
            const uint64_t pol = policy_evict_first();
            int it = 0;
            bool stop = false;
            for (int s = 0; s < n_segs && !stop; ++s) {
                const int pair = static_cast<int>(p_first + s);
                for (int t = 0; t < seg_nv[s]; ++t, ++it) {
                    const int stg = it % kStages;
                    const int use = it / kStages;
                    if (use > 0 && !mbar_wait(bar_empty + 8 * stg, (use - 1) & 1, kWaitNs)) {
                        report(p.status, SPARSE_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    const int slot = lslot[it];
                    const int row = slot >= 0 ? slot * kBlk
                                              : static_cast<int>(min(p.pair_stride, (long long)INT_MAX - kBlk));
                    const uint32_t dst = base_s + stg * kStageBytes;
                    mbar_arrive_expect_tx(bar_full + 8 * stg, kStageBytes);
                    tma_load_3d(dst, &kmap, bar_full + 8 * stg, 0, row, pair, pol);
                    tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * stg, 64, row, pair, pol);
                    tma_load_3d(dst + kTileBytes, &vmap, bar_full + 8 * stg, 0, row, pair, pol);
                    tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, bar_full + 8 * stg, 64, row, pair, pol);
                }
            }
        }
        griddep_launch_dependents();
        return;
    }

    // ---------------------------------------------------------------- consumers
    if (early)
        griddep_wait();   // Q may be written by the kernel before this one
    auto consumers_sync = [] { named_barrier_sync(1, kConsumerWarps * 32); };
    int it = 0;
    bool timed_out = false;
    for (int s = 0; s < n_segs; ++s) {
        const int pair = static_cast<int>(p_first + s);
        const int b = pair / p.H_kv, g = pair % p.H_kv;
        const long long len = p.seq_len[b];
        const long long pbase = static_cast<long long>(pair) * K;
        const long long ia = max(lo, pbase) - pbase, ib = min(hi, pbase + K) - pbase;
        const bool full = ia == 0 && ib == K;
        const int nv = aborted ? 0 : seg_nv[s];
        QueryFrags<NT> q;
        load_query<NT, false>(q, p, b, g, 0, p.G, lane);
        WarpState<NT> st;
        st.reset();
        int held = -1;   // ring stage kept for the segment's merge
        for (int t = 0; t < nv; ++t, ++it) {
            const int stg = it % kStages;
            if (!timed_out) {
                const bool landed =
                    __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * stg, (it / kStages) & 1, kWaitNs));
                if (!landed) {
                    if (lane == 0)
                        report(p.status, SPARSE_ERR_TIMEOUT);
                    timed_out = true;
                }
            }
            if (!timed_out) {
                const int logical = llog[it];
                const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
                if (logical >= 0 && tok0 < len)
                    attend_block<NT, false>(st, q, base_s + stg * kStageBytes, tok0, len, 0xffffffffu, p.scale_log2,
                                            warp, lane);
            }
            if (t + 1 < nv || timed_out) {
                __syncwarp();
                if (lane == 0 && !timed_out)
                    mbar_arrive(bar_empty + 8 * stg);
            } else {
                held = stg;
            }
        }
        finish_row_sums<NT>(st);
        const bool valid = !aborted && !timed_out;

        // ---- the segment's state: merged in the held stage, or empty
        consumers_sync();   // every consumer warp is done reading the held stage
        float *co = nullptr, *cm = nullptr, *cl = nullptr;
        if (held >= 0) {
            float *wo = reinterpret_cast<float *>(base + held * kStageBytes);
            float *wm = wo + kConsumerWarps * ROWS * kWoStride;
            float *wl = wm + kConsumerWarps * ROWS;
            float *wf = wl + kConsumerWarps * ROWS;
            co = wf + kConsumerWarps * ROWS;
            cm = co + ROWS * kD;
            cl = cm + ROWS;
            store_warp_state<NT>(st, wo, wm, wl, warp, lane);
            consumers_sync();
            merge_warp_states<ROWS>(wo, wm, wl, wf, co, cm, cl, tid, kConsumerWarps * 32, consumers_sync);
            consumers_sync();
        }
        if (full) {
            // the whole pair lies in this CTA's range: write the output directly
            if (valid) {
                for (int item = tid; item < p.G * kD; item += kConsumerWarps * 32) {
                    const int row = item / kD, d = item - row * kD;
                    const float L = co ? cl[row] : 0.f;
                    const float o = (co && L > 0.f) ? co[item] / L : 0.f;
                    store_bf16(p.O + (static_cast<size_t>(b) * p.H_q + g * p.G + row) * kD + d, o);
                }
                if (p.lse != nullptr && tid < p.G)
                    p.lse[static_cast<size_t>(b) * p.H_q + g * p.G + tid] = co ? lse_of(cm[tid], cl[tid]) : -INFINITY;
            }
        } else {
            // partial pair: state to the workspace, then the arrival count
            float *dst = p.ws_part + part_slot(c, pair, N, C, K) * PART;
            if (co != nullptr) {
                for (int i = tid; i < ROWS * kD; i += kConsumerWarps * 32)
                    dst[i] = co[i];
            }
            if (tid < ROWS) {
                dst[ROWS * kD + tid] = co ? cm[tid] : -INFINITY;
                dst[ROWS * kD + ROWS + tid] = co ? cl[tid] : 0.f;
            }
            if (tid == 0)
                dst[PART - 1] = valid ? 1.f : 0.f;
            __threadfence();
            consumers_sync();
            const int c_first = cta_of_item(pbase, N, C);
            const int c_last = cta_of_item(pbase + K - 1, N, C);
            if (tid == 0) {
                const int prev = atomicAdd(&p.ws_count[pair], 1);
                const bool last = prev == c_last - c_first;
                ctrl[kCtrlLast] = last ? 1 : 0;
                if (last) {
                    __threadfence();
                    p.ws_count[pair] = 0;   // back to zero for the next call
                }
            }
            consumers_sync();
            if (ctrl[kCtrlLast]) {
                // the pair's last partial: merge the n_seg CTA states of this pair.
                // (a) every (CTA, row) max / sum / validity into shared memory, in parallel
                const int n_seg = c_last - c_first + 1;
                float *fm = reinterpret_cast<float *>(base + kOffMergeFac);   // [n_seg][ROWS] max, then weight
                float *fl = fm + kMaxMergeSeg * ROWS;                          // [n_seg][ROWS] sum
                int *soff = reinterpret_cast<int *>(base + kOffMergeSlot);     // [n_seg] slot offsets (floats)
                if (tid < n_seg)
                    soff[tid] = static_cast<int>(part_slot(c_first + tid, pair, N, C, K) * PART);
                consumers_sync();
                for (int e = tid; e < n_seg * ROWS; e += kConsumerWarps * 32) {
                    const int row = e % ROWS;
                    const float *src = p.ws_part + soff[e / ROWS];
                    const float valid_cc = __ldcg(src + PART - 1);
                    fm[e] = __ldcg(src + ROWS * kD + row);
                    fl[e] = valid_cc != 0.f ? __ldcg(src + ROWS * kD + ROWS + row) : -1.f;   // -1 marks invalid
                }
                if (tid == 0)
                    ctrl[kCtrlMergeValid] = 1;
                consumers_sync();
                // (b) per row: max, sum, and each CTA's weight 2^(m - M) / L; a CTA whose
                // ready check failed leaves the pair's output untouched
                if (tid < ROWS) {
                    float M = -INFINITY;
                    bool all_valid = true;
                    for (int i = 0; i < n_seg; ++i) {
                        M = fmaxf(M, fm[i * ROWS + tid]);
                        all_valid = all_valid && fl[i * ROWS + tid] >= 0.f;
                    }
                    if (!all_valid)
                        atomicAnd(&ctrl[kCtrlMergeValid], 0);
                    float L = 0.f;
                    for (int i = 0; i < n_seg; ++i) {
                        const float mc = fm[i * ROWS + tid];
                        const float f = (M == -INFINITY || mc == -INFINITY) ? 0.f : exp2f(mc - M);
                        fm[i * ROWS + tid] = f;
                        L += f * fmaxf(fl[i * ROWS + tid], 0.f);
                    }
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    for (int i = 0; i < n_seg; ++i)
                        fm[i * ROWS + tid] *= inv;
                    row_m[tid] = M;
                    row_l[tid] = L;
                }
                consumers_sync();
                // (c) O: branch-free weighted sums.  Thread t owns items t + 128 j (row j,
                // dim t); the loads of 4 CTAs x 8 items are in flight together.
                if (ctrl[kCtrlMergeValid]) {
                    float o[ROWS];
#pragma unroll
                    for (int j = 0; j < ROWS; ++j)
                        o[j] = 0.f;
                    for (int i = 0; i < n_seg; i += 4) {
                        float v[4][ROWS];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < ROWS; ++j)
                                v[u][j] = (i + u < n_seg && j < p.G) ? __ldcg(p.ws_part + soff[i + u] + j * kD + tid)
                                                                     : 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < ROWS; ++j)
                                if (i + u < n_seg)
                                    o[j] = fmaf(fm[(i + u) * ROWS + j], v[u][j], o[j]);
                    }
#pragma unroll
                    for (int j = 0; j < ROWS; ++j)
                        if (j < p.G)
                            store_bf16(p.O + (static_cast<size_t>(b) * p.H_q + g * p.G + j) * kD + tid, o[j]);
                    if (p.lse != nullptr && tid < p.G)
                        p.lse[static_cast<size_t>(b) * p.H_q + g * p.G + tid] = lse_of(row_m[tid], row_l[tid]);
                }
            }
            consumers_sync();
        }
        if (held >= 0) {
            // the held stage goes back to the producer (generic writes before TMA writes)
            fence_proxy_async_smem();
            consumers_sync();
            __syncwarp();
            if (lane == 0 && !timed_out)
                mbar_arrive(bar_empty + 8 * held);
        } else {
            consumers_sync();
        }
    }
    griddep_launch_dependents();
}

template <int NT>
int launch_streamk(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int n_ctas, int device,
                   cudaStream_t stream)
{
    auto kern = decode_streamk_kernel<NT>;
    const int smem = kSmemStreamK + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CUtensorMap kmap = km, vmap = vm;
    AttnParams prm = p;
    void *args[] = {&kmap, &vmap, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse attention (stream-K) launch");
}

// Stream-K geometry: CTA count and workspace bytes (counters, then 2 partial slots per CTA).
int streamk_ctas(long long n_items, long long pairs, int n_split, int sm_count)
{
    long long c = n_split > 0 ? n_split : 2LL * sm_count;
    if (c > n_items)
        c = n_items;
    // a pair spans at most C / pairs + 2 ranges: keep that within kMaxMergeSeg
    if (c > (kMaxMergeSeg - 2) * pairs)
        c = (kMaxMergeSeg - 2) * pairs;
    const long long need = (n_items + kMaxListCta - 1) / kMaxListCta;   // at most kMaxListCta items per CTA
    if (c < need)
        c = need;
    return static_cast<int>(c < 1 ? 1 : c);
}

size_t streamk_workspace_bytes(long long pairs, int G, int n_ctas)
{
    const int rows = G <= 8 ? 8 : 16;
    const size_t part = static_cast<size_t>(rows) * kD + 2 * rows + 1;
    const size_t counters = (static_cast<size_t>(pairs) * sizeof(int) + 255) & ~static_cast<size_t>(255);
    return counters + 2ull * static_cast<size_t>(n_ctas) * part * sizeof(float);
}

template <int NT>
int launch_split(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int S, long long pairs,
                 int device, cudaStream_t stream)
{
    auto kern = decode_split_kernel<NT>;
    const int smem = kSmemDecode + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CUtensorMap kmap = km, vmap = vm;
    AttnParams prm = p;
    void *args[] = {&kmap, &vmap, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse attention (split) launch");
}

// Split path geometry: CTAs per pair.  Auto: one wave of two CTAs per SM, at least two
// blocks per CTA; a slice never exceeds the staged list (kMaxListCta).  0 = invalid.
int split_ctas_per_pair(long long pairs, int k_tot, int n_split, int sm_count)
{
    long long s;
    if (n_split > 0) {
        s = n_split;
    } else {
        s = (2LL * sm_count) / pairs;
        const long long by_list = k_tot / 2;
        if (s > by_list)
            s = by_list;
        if (s > kMaxSplitWs)
            s = kMaxSplitWs;
        if (s < 1)
            s = 1;
        while ((k_tot + s - 1) / s > kMaxListCta && s < kMaxSplitWs)
            ++s;
    }
    if (s > kMaxSplitWs || (k_tot + s - 1) / s > kMaxListCta)
        return 0;
    return static_cast<int>(s);
}

size_t split_workspace_bytes(long long pairs, int G, int S)
{
    const size_t part = G <= 8 ? split_part_floats<1>() : split_part_floats<2>();
    const size_t counters = (static_cast<size_t>(pairs) * sizeof(int) + 255) & ~static_cast<size_t>(255);
    return counters + static_cast<size_t>(pairs) * S * part * sizeof(float);
}

// TC: the tensor-memory kernel (sparse_attn_tc_kernel, SPARSE_ATTN_TENSOR_MEMORY) instead
// of the mma.sync one.
template <int NT, bool VERIFY, bool TC>
int launch(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int S, long long units,
           int device, cudaStream_t stream)
{
    auto kern = TC ? sparse_attn_tc_kernel<NT, VERIFY> : sparse_attn_kernel<NT, VERIFY>;
    const int smem = TC ? kTcSmem : (VERIFY ? kSmemVerify : kSmemDecode) + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(units), 1);
    cfg.blockDim = dim3(TC ? kTcThreads : kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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
                                "sparse attention launch");
}

// The merge scratch (warp and CTA states, weights) must fit in the ring it reuses.
static_assert((3 * kConsumerWarps * 16 + kConsumerWarps * 16 * kWoStride + 16 * kD + 2 * 16 + 4 + kMaxSplit * 16 + 2 * 16) *
                      4 <=
                  kStages * kStageBytes,
              "merge scratch exceeds the stage ring");

// The host-side checks of sparse_decode_attn's arguments that do not depend on the
// path (cluster, split or stream-K); SPARSE_OK or the error, before anything is launched.
int decode_check(const uint16_t *Q, const uint16_t *k_base, const uint16_t *v_base, long long pair_stride,
                 const int *blk_logical, const int *count, int k_tot, const int *seq_len, int B, int H_q, int H_kv,
                 float scale, const uint16_t *O, int n_split, unsigned flags, long long timeout_ns)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!Q || !k_base || !v_base || !blk_logical || !count || !seq_len || !O)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: null pointer");
    if (!aligned16(Q) || !aligned16(k_base) || !aligned16(v_base) || !aligned16(O))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: Q, K, V and O must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k_tot < 1 || pair_stride < 1)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: bad size (B=%d H_q=%d H_kv=%d k_tot=%d)", B,
                    H_q, H_kv, k_tot);
    if (pair_stride > INT_MAX - 2 * kBlk)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: pair_stride_tokens too large");
    if (!isfinite(scale))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: scale must be finite");
    if (timeout_ns < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_ex: timeout_ns < 0");
    if (H_q / H_kv > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: G=%d > 16 query heads per KV head", H_q / H_kv);
    if (static_cast<long long>(B) * H_kv > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: B*H_kv=%lld > 65535",
                    static_cast<long long>(B) * H_kv);
    if ((flags & ~(SPARSE_ATTN_BLOCKS_READY | SPARSE_ATTN_STREAM_K | SPARSE_ATTN_TENSOR_MEMORY)) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: unknown flags 0x%x", flags);
    if (n_split < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: n_split < 0");
    return SPARSE_OK;
}

int decode_impl(const uint16_t *Q, const uint16_t *k_base, const uint16_t *v_base, long long pair_stride,
                const int *blk_slot, const int *blk_logical, const int *count, int k_tot, const int *seq_len,
                int B, int H_q, int H_kv, float scale, uint16_t *O, float *lse, int n_split, unsigned flags,
                void *workspace, size_t workspace_bytes, const unsigned *ready_flag, unsigned ready_target,
                long long timeout_ns, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    int rc = decode_check(Q, k_base, v_base, pair_stride, blk_logical, count, k_tot, seq_len, B, H_q, H_kv, scale,
                          O, n_split, flags, timeout_ns);
    if (rc != SPARSE_OK)
        return rc;
    const bool tensor_memory = (flags & SPARSE_ATTN_TENSOR_MEMORY) != 0u;
    if (tensor_memory && workspace != nullptr)
        return fail(SPARSE_ERR_INVALID_ARG,
                    "sparse_decode_attn: SPARSE_ATTN_TENSOR_MEMORY runs the cluster path: pass no workspace");
    const int G = H_q / H_kv;
    const long long pairs = static_cast<long long>(B) * H_kv;
    sp_host::DeviceInfo dev;
    rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    AttnParams p = {};
    p.Q = Q;
    p.O = O;
    p.lse = lse;
    p.blk_slot = blk_slot;
    p.blk_logical = blk_logical;
    p.count = count;
    p.seq_len = seq_len;
    p.status = status;
    p.ready_flag = ready_flag;
    p.ready_target = ready_target;
    p.timeout_ns = timeout_ns > 2000000000LL ? 2000000000LL : timeout_ns;
    p.pair_stride = pair_stride;
    p.k_tot = k_tot;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.n_groups = 1;
    p.flags = flags;
    p.scale_log2 = scale_log2_of(scale);
    // With a workspace: the split path (per-pair slices, merged by the last CTA), or
    // stream-K when asked.  Without one: thread-block clusters merging through DSMEM.
    const bool stream_k = workspace != nullptr && G <= 8 && (flags & SPARSE_ATTN_STREAM_K) != 0u;
    if (workspace != nullptr && !stream_k) {
        if (!aligned16(workspace))
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: workspace must be 16-byte aligned");
        const int S = split_ctas_per_pair(pairs, k_tot, n_split, dev.sm_count);
        if (S == 0)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: n_split=%d (1..%d CTAs per pair, at most %d "
                        "blocks each)", n_split, kMaxSplitWs, kMaxListCta);
        const size_t need = split_workspace_bytes(pairs, G, S);
        if (workspace_bytes < need)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: workspace of %zu bytes, %zu needed",
                        workspace_bytes, need);
        CUtensorMap km, vm;
        if ((rc = sp_host::make_kv_tensor_map(&km, k_base, pair_stride, pairs)) != SPARSE_OK)
            return rc;
        if ((rc = sp_host::make_kv_tensor_map(&vm, v_base, pair_stride, pairs)) != SPARSE_OK)
            return rc;
        p.ws_count = static_cast<int *>(workspace);
        p.ws_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                              ((static_cast<size_t>(pairs) * sizeof(int) + 255) & ~static_cast<size_t>(255)));
        return G <= 8 ? launch_split<1>(p, km, vm, S, pairs, dev.device, st)
                      : launch_split<2>(p, km, vm, S, pairs, dev.device, st);
    }
    if (stream_k) {
        // stream-K: equal contiguous ranges of the flattened (pair, block) list
        if (!aligned16(workspace))
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: workspace must be 16-byte aligned");
        const long long n_items = pairs * k_tot;
        const int n_ctas = streamk_ctas(n_items, pairs, n_split, dev.sm_count);
        if ((n_items + n_ctas - 1) / n_ctas > kMaxListCta)
            return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: too many blocks per CTA");
        const size_t need = streamk_workspace_bytes(pairs, G, n_ctas);
        if (workspace_bytes < need)
            return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: workspace of %zu bytes, %zu needed",
                        workspace_bytes, need);
        CUtensorMap km, vm;
        if ((rc = sp_host::make_kv_tensor_map(&km, k_base, pair_stride, pairs)) != SPARSE_OK)
            return rc;
        if ((rc = sp_host::make_kv_tensor_map(&vm, v_base, pair_stride, pairs)) != SPARSE_OK)
            return rc;
        p.ws_count = static_cast<int *>(workspace);
        p.ws_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                              ((static_cast<size_t>(pairs) * sizeof(int) + 255) & ~static_cast<size_t>(255)));
        p.n_items = n_items;
        return launch_streamk<1>(p, km, vm, n_ctas, dev.device, st);
    }
    int S;
    if ((rc = choose_split(n_split, pairs, k_tot, dev.sm_count, &S)) != SPARSE_OK)
        return rc;
    while ((k_tot + S - 1) / S > kMaxListCta && S < kMaxSplit && n_split == 0)
        S *= 2;
    if ((k_tot + S - 1) / S > kMaxListCta)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: k_tot=%d needs more than %d blocks per CTA", k_tot,
                    kMaxListCta);
    CUtensorMap km, vm;
    if ((rc = sp_host::make_kv_tensor_map(&km, k_base, pair_stride, pairs)) != SPARSE_OK)
        return rc;
    if ((rc = sp_host::make_kv_tensor_map(&vm, v_base, pair_stride, pairs)) != SPARSE_OK)
        return rc;
    if (tensor_memory)
        return G <= 8 ? launch<1, false, true>(p, km, vm, S, pairs, dev.device, st)
                      : launch<2, false, true>(p, km, vm, S, pairs, dev.device, st);
    return G <= 8 ? launch<1, false, false>(p, km, vm, S, pairs, dev.device, st)
                  : launch<2, false, false>(p, km, vm, S, pairs, dev.device, st);
}

}  // namespace

extern "C" SPARSE_API int sparse_decode_attn(const uint16_t *Q, const uint16_t *k_base, const uint16_t *v_base,
                                             long long pair_stride_tokens, const int *blk_slot,
                                             const int *blk_logical, const int *count, int k_tot,
                                             const int *seq_len, int B, int H_q, int H_kv, float scale,
                                             uint16_t *O, float *lse, int n_split, unsigned flags, void *workspace,
                                             size_t workspace_bytes, int *status, void *stream)
{
    return decode_impl(Q, k_base, v_base, pair_stride_tokens, blk_slot, blk_logical, count, k_tot, seq_len, B,
                       H_q, H_kv, scale, O, lse, n_split, flags, workspace, workspace_bytes, nullptr, 0u, 0, status,
                       stream);
}

extern "C" SPARSE_API int sparse_decode_attn_ex(const uint16_t *Q, const uint16_t *k_base,
                                                const uint16_t *v_base, long long pair_stride_tokens,
                                                const int *blk_slot, const int *blk_logical, const int *count,
                                                int k_tot, const int *seq_len, int B, int H_q, int H_kv,
                                                float scale, uint16_t *O, float *lse, int n_split, unsigned flags,
                                                void *workspace, size_t workspace_bytes, const unsigned *ready_flag,
                                                unsigned ready_target, long long timeout_ns, int *status,
                                                void *stream)
{
    if (ready_flag == nullptr)
        return sp_host::fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_ex: ready_flag is null");
    return decode_impl(Q, k_base, v_base, pair_stride_tokens, blk_slot, blk_logical, count, k_tot, seq_len, B,
                       H_q, H_kv, scale, O, lse, n_split, flags, workspace, workspace_bytes, ready_flag,
                       ready_target, timeout_ns, status, stream);
}

// ---------------------------------------------------------------- allocation-free decode

// Scratch of sparse_decode_attn_noalloc: a fixed array in device memory, so the call
// allocates nothing.  Every GPU that loads the library holds these 4 MiB until the
// process exits.  All calls share it; it keeps the last call's contents.
constexpr size_t kNoallocScratchBytes = static_cast<size_t>(4) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

// The device address of g_noalloc_scratch in the current context (the host-side name of
// the array is only a stand-in, never a device address).  Looked up once per context:
// a context that is destroyed and created again (cudaDeviceReset) loads the module
// anew, so the cache is keyed on the context's unique id, not on the device ordinal.
constexpr int kNoallocCacheSlots = 64;
std::mutex g_noalloc_mu;
unsigned long long g_noalloc_ctx[kNoallocCacheSlots];   // 0 = empty (context ids are nonzero)
void *g_noalloc_ptr[kNoallocCacheSlots];
int g_noalloc_next;

int noalloc_scratch(void **ptr)
{
    unsigned long long ctx = 0;
    int rc = sp_host::current_context_id(&ctx);
    if (rc != SPARSE_OK)
        return rc;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; i < kNoallocCacheSlots; ++i)
        if (g_noalloc_ctx[i] == ctx && ctx != 0) {
            *ptr = g_noalloc_ptr[i];
            return SPARSE_OK;
        }
    void *addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || addr == nullptr)
        return sp_host::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                                    "sparse_decode_attn_noalloc: cudaGetSymbolAddress");
    const int slot = g_noalloc_next;
    g_noalloc_next = (g_noalloc_next + 1) % kNoallocCacheSlots;
    g_noalloc_ctx[slot] = ctx;
    g_noalloc_ptr[slot] = addr;
    *ptr = addr;
    return SPARSE_OK;
}

}  // namespace

extern "C" SPARSE_API int sparse_decode_attn_noalloc(const uint16_t *Q, const uint16_t *k_base,
                                                     const uint16_t *v_base, long long pair_stride_tokens,
                                                     const int *blk_slot, const int *blk_logical, const int *count,
                                                     int k_tot, const int *seq_len, int B, int H_q, int H_kv,
                                                     float scale, uint16_t *O, float *lse, int n_split,
                                                     unsigned flags, int *status, void *stream)
{
    using sp_host::fail;
    // every argument check first: a rejected call leaves the shared array untouched
    int rc = decode_check(Q, k_base, v_base, pair_stride_tokens, blk_logical, count, k_tot, seq_len, B, H_q, H_kv,
                          scale, O, n_split, flags, 0);
    if (rc != SPARSE_OK)
        return rc;
    if (H_q / H_kv > 8)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_noalloc: G=%d > 8", H_q / H_kv);
    if ((flags & SPARSE_ATTN_TENSOR_MEMORY) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG,
                    "sparse_decode_attn_noalloc: SPARSE_ATTN_TENSOR_MEMORY runs the cluster path, not this one");
    sp_host::DeviceInfo dev;
    if ((rc = sp_host::device_info(&dev)) != SPARSE_OK)
        return rc;
    const long long pairs = static_cast<long long>(B) * H_kv;
    const long long n_items = pairs * k_tot;
    const int n_ctas = streamk_ctas(n_items, pairs, n_split, dev.sm_count);
    if ((n_items + n_ctas - 1) / n_ctas > kMaxListCta)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_noalloc: too many blocks per CTA");
    const size_t need = streamk_workspace_bytes(pairs, H_q / H_kv, n_ctas);
    if (need > kNoallocScratchBytes)
        return fail(SPARSE_ERR_UNSUPPORTED,
                    "sparse_decode_attn_noalloc: these sizes need %zu bytes of scratch, more than the fixed %zu "
                    "(use sparse_decode_attn with a workspace)",
                    need, kNoallocScratchBytes);
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != SPARSE_OK)
        return rc;
    // the per-pair arrival counters must start at zero: clear them on the call's stream
    const size_t counters = (static_cast<size_t>(pairs) * sizeof(int) + 255) & ~static_cast<size_t>(255);
    rc = sp_host::cuda_status(cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)),
                              "sparse_decode_attn_noalloc: clearing the counters");
    if (rc != SPARSE_OK)
        return rc;
    return sparse_decode_attn(Q, k_base, v_base, pair_stride_tokens, blk_slot, blk_logical, count, k_tot, seq_len,
                              B, H_q, H_kv, scale, O, lse, n_split, flags | SPARSE_ATTN_STREAM_K, scratch,
                              kNoallocScratchBytes, status, stream);
}

extern "C" SPARSE_API size_t sparse_decode_attn_workspace_size(int B, int H_q, int H_kv, int k_tot, int n_split)
{
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k_tot < 1 || n_split < 0)
        return 0;
    sp_host::DeviceInfo dev;
    if (sp_host::device_info(&dev) != SPARSE_OK)
        return 0;
    const long long pairs = static_cast<long long>(B) * H_kv;
    const int G = H_q / H_kv;
    if (G > 16)
        return 0;
    const int S = split_ctas_per_pair(pairs, k_tot, n_split, dev.sm_count);
    size_t need = S > 0 ? split_workspace_bytes(pairs, G, S) : 0;
    if (G <= 8) {
        const size_t sk = streamk_workspace_bytes(pairs, G, streamk_ctas(pairs * k_tot, pairs, n_split, dev.sm_count));
        need = sk > need ? sk : need;
    }
    return need;
}

namespace {

static int verify_impl(const char *name, unsigned mode, const uint16_t *Q, const uint16_t *k_cache,
                       const uint16_t *v_cache, long long T_cap, const int *idx_q, int n_sel, int N_q, int C,
                       int window_blocks, const int *seq_len, int B, int H_q, int H_kv, float scale, uint16_t *O,
                       long long *blocks_loaded, int n_split, unsigned flags, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if ((flags & ~(SPARSE_ATTN_BLOCKS_READY | SPARSE_ATTN_TENSOR_MEMORY)) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
    if (!Q || !k_cache || !v_cache || !seq_len || !O || (n_sel > 0 && !idx_q))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(Q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(O))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: Q, K, V and O must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || N_q < 1 || C < 1 || n_sel < 0 ||
        window_blocks < 0 || T_cap < 1)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size", name);
    if (T_cap > INT_MAX - 2 * kBlk)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: T_cap too large", name);
    if (!isfinite(scale))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: scale must be finite", name);
    const int G = H_q / H_kv;
    if (C > 32 || static_cast<long long>(C) * G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: C*G=%lld rows > 16 per group", name,
                    static_cast<long long>(C) * G);
    if (static_cast<long long>(C) * n_sel + window_blocks > kMaxUnion)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: C*n_sel+window_blocks > %d", name, kMaxUnion);
    const int n_groups = (N_q + C - 1) / C;
    const long long units = static_cast<long long>(B) * H_kv * n_groups;
    if (units > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: too many groups", name);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    int S;
    const int max_list = C * n_sel + window_blocks;
    if ((rc = choose_split(n_split, units, max_list, dev.sm_count, &S)) != SPARSE_OK)
        return rc;
    CUtensorMap km, vm;
    const long long pairs = static_cast<long long>(B) * H_kv;
    if ((rc = sp_host::make_kv_tensor_map(&km, k_cache, T_cap, pairs)) != SPARSE_OK)
        return rc;
    if ((rc = sp_host::make_kv_tensor_map(&vm, v_cache, T_cap, pairs)) != SPARSE_OK)
        return rc;
    AttnParams p = {};
    p.Q = Q;
    p.O = O;
    p.seq_len = seq_len;
    p.status = status;
    p.idx_q = idx_q;
    p.blocks_loaded = blocks_loaded;
    p.pair_stride = T_cap;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.n_sel = n_sel;
    p.N_q = N_q;
    p.C = C;
    p.window_blocks = window_blocks;
    p.n_groups = n_groups;
    p.flags = mode | flags;
    p.scale_log2 = scale_log2_of(scale);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((flags & SPARSE_ATTN_TENSOR_MEMORY) != 0u)
        return C * G <= 8 ? launch<1, true, true>(p, km, vm, S, units, dev.device, st)
                          : launch<2, true, true>(p, km, vm, S, units, dev.device, st);
    return C * G <= 8 ? launch<1, true, false>(p, km, vm, S, units, dev.device, st)
                      : launch<2, true, false>(p, km, vm, S, units, dev.device, st);
}

}  // namespace

extern "C" SPARSE_API int sparse_verify_attn_grouped(const uint16_t *Q, const uint16_t *k_cache,
                                                     const uint16_t *v_cache, long long T_cap, const int *idx_q,
                                                     int n_sel, int N_q, int C, int window_blocks,
                                                     const int *seq_len, int B, int H_q, int H_kv, float scale,
                                                     uint16_t *O, long long *blocks_loaded, int n_split,
                                                     unsigned flags, int *status, void *stream)
{
    return verify_impl("sparse_verify_attn_grouped", 0u, Q, k_cache, v_cache, T_cap, idx_q, n_sel, N_q, C,
                       window_blocks, seq_len, B, H_q, H_kv, scale, O, blocks_loaded, n_split, flags, status,
                       stream);
}

extern "C" SPARSE_API int sparse_verify_attn_shared(const uint16_t *Q, const uint16_t *k_cache,
                                                    const uint16_t *v_cache, long long T_cap, const int *idx_q,
                                                    int n_sel, int N_q, int C, int window_blocks,
                                                    const int *seq_len, int B, int H_q, int H_kv, float scale,
                                                    uint16_t *O, long long *blocks_loaded, int n_split,
                                                    unsigned flags, int *status, void *stream)
{
    return verify_impl("sparse_verify_attn_shared", kVerifySharedLayout, Q, k_cache, v_cache, T_cap, idx_q, n_sel,
                       N_q, C, window_blocks, seq_len, B, H_q, H_kv, scale, O, blocks_loaded, n_split, flags,
                       status, stream);
}

// ---------------------------------------------------------------- NSA gated three-branch decode
//
// SSV notes, "NSA three-branch math" steps 3-6: the selected-block branch, the
// compressed branch and the sliding-window branch each run their own softmax, and the
// output is the gate-weighted sum g_c o^(c) + g_s o^(s) + g_w o^(w).  The notes take
// the branches to need separate kernels with intermediate results in HBM.  Here the
// three are one launch: grid (S, pairs, 3), blockIdx.z the branch, each branch a
// cluster of S CTAs per pair running the same split-KV attention as the decode path
// (the selected blocks from the table; the window as the block range of the last w
// tokens, masked token by token; the compressed rows as one more bf16 "cache" with a
// row per 64-token block).  Each cluster writes its normalised branch output o^(x) in
// fp32 to a small workspace (L2-resident: 3 x G x 512 B per pair); the last of the
// pair's 3 S CTAs to finish applies the gates and writes O.

namespace {

struct NsaParams {
    AttnParams br[3];      // 0: selected blocks, 1: sliding window, 2: compressed rows
    const float *gates;    // [B][H_q][3] = (g_c, g_s, g_w)
    const float *part;     // [3][B * H_q][128] branch outputs (br[x].O32)
    unsigned *arrivals;    // [pairs] arrival counters, zero between calls
    uint16_t *O;           // [B][H_q][128]
    unsigned target;       // 3 * S arrivals per pair
};

template <int NT>
__global__ void __launch_bounds__(kThreads, 2)
    nsa_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap khmap, const __grid_constant__ CUtensorMap vhmap,
                      const __grid_constant__ NsaParams np)
{
    __shared__ int last;
    const int branch = static_cast<int>(blockIdx.z);
    const int pair = static_cast<int>(blockIdx.y);
    const AttnParams &p = np.br[branch];
    const bool compressed = branch == 2;
    attn_cluster_cta<NT, false>(compressed ? &khmap : &kmap, compressed ? &vhmap : &vmap, p, pair);

    // this CTA's share of o^(x) is written: publish it, count the arrival
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&np.arrivals[pair], 1u);
        last = prev + 1u == np.target;
        if (last)
            np.arrivals[pair] = 0u;   // ready for the next call
    }
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    const size_t stride = static_cast<size_t>(gridDim.y / p.H_kv) * p.H_q * kD;   // one branch's outputs
    for (int item = threadIdx.x; item < p.G * (kD / 2); item += kThreads) {
        const int row = item / (kD / 2);
        const int d = 2 * (item - row * (kD / 2));
        const size_t head = static_cast<size_t>(b) * p.H_q + g * p.G + row;
        const size_t at = head * kD + d;
        const float gc = np.gates[head * 3 + 0], gs = np.gates[head * 3 + 1], gw = np.gates[head * 3 + 2];
        const float2 os = __ldcg(reinterpret_cast<const float2 *>(np.part + at));
        const float2 ow = __ldcg(reinterpret_cast<const float2 *>(np.part + stride + at));
        const float2 oc = __ldcg(reinterpret_cast<const float2 *>(np.part + 2 * stride + at));
        const float x = fmaf(gc, oc.x, fmaf(gs, os.x, gw * ow.x));
        const float y = fmaf(gc, oc.y, fmaf(gs, os.y, gw * ow.y));
        *reinterpret_cast<uint32_t *>(np.O + at) = pack_bf16x2(x, y);
    }
}

// The fused form (G <= 8): one cluster of S CTAs per pair runs all three branches.
// CTA r takes slice r of each branch's list (the selected table, the compressed-row
// tiles, the window's blocks); its producer streams the three slices back to back
// through one TMA ring and its consumer warps keep three online-softmax states in
// registers, one per branch.  One DSMEM merge then gives every CTA the three
// normalised branch outputs for its output dims, and the gated sum is formed right
// there: no intermediate reaches HBM and there is no second pass.

// Slice `rank` of a range branch (x = 1 window, 2 compressed): its first block (tile)
// and length.
__device__ __forceinline__ void nsa_range_slice(const AttnParams &p, int b, int rank, int S, int *first_out,
                                                int *n_out)
{
    const long long rows = unit_len(p, b);
    const int nb = rows <= 0 ? 0 : static_cast<int>((rows + kBlk - 1) / kBlk);
    long long w0 = p.range_mode == 1 ? rows - p.win_tokens : 0;
    w0 = w0 < 0 ? 0 : w0;
    const int first = static_cast<int>(w0 / kBlk);
    int c = nb > first ? nb - first : 0;
    if (p.range_mode == 1 && p.win_tokens <= 0)
        c = 0;
    const int per = (c + S - 1) / S;
    const int i0 = min(c, rank * per);
    *first_out = first + i0;
    *n_out = min(c, i0 + per) - i0;
}

__global__ void __launch_bounds__(kThreads, 2)
    nsa_fused_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap khmap, const __grid_constant__ CUtensorMap vhmap,
                     const __grid_constant__ NsaParams np)
{
    constexpr int NT = 1, ROWS = 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kOffCtrl);
    const uint32_t bar_full = base_s + kOffBars;
    const uint32_t bar_empty = base_s + kOffBars + 8 * kStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = static_cast<int>(gridDim.x);
    const int rank = static_cast<int>(blockIdx.x);
    const int pair = static_cast<int>(blockIdx.y);
    const AttnParams &ps = np.br[0];
    const AttnParams &pw = np.br[1];
    const AttnParams &pc = np.br[2];
    const int b = pair / ps.H_kv, g = pair % ps.H_kv;
    if (tid == kConsumerWarps * 32) {   // the descriptor fetches overlap the barrier set-up
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        prefetch_tensormap(&khmap);
        prefetch_tensormap(&vhmap);
    }
    const bool early = (ps.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();
    if (tid == 0) {
        ctrl[kCtrlAbort] = 0;
        ctrl[kCtrlList] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    int *lslot = reinterpret_cast<int *>(base + kOffList);
    int *llog = lslot + kMaxListCta;
    // the range branches' slices follow from the length alone
    int w_first, n_w, c_first, n_c;
    nsa_range_slice(pw, b, rank, S, &w_first, &n_w);
    nsa_range_slice(pc, b, rank, S, &c_first, &n_c);

    WarpState<NT> st_s, st_w, st_c;
    st_s.reset();
    st_w.reset();
    st_c.reset();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        // Ring order: the compressed tiles, the window's blocks, then the selected
        // blocks.  The range tiles need no table, so the first ring stages are issued
        // before the selected slice is fetched and that round trip is hidden.
        const int n_r = n_c + n_w;
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        auto issue = [&](int it) {
            const int s = it % kStages;
            const int use = it / kStages;
            if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kWaitNs)) {
                report(ps.status, SPARSE_ERR_TIMEOUT);
                ok = false;
                return;
            }
            const CUtensorMap *km = &kmap, *vm = &vmap;
            int row;
            if (it < n_c) {
                km = &khmap;
                vm = &vhmap;
                row = (c_first + it) * kBlk;
            } else if (it < n_r) {
                row = (w_first + it - n_c) * kBlk;
            } else {
                const int slot = lslot[it - n_r];
                row = slot >= 0 ? slot * kBlk : static_cast<int>(min(ps.pair_stride, (long long)INT_MAX - kBlk));
            }
            const uint32_t dst = base_s + s * kStageBytes;
            mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
            tma_load_3d(dst, km, bar_full + 8 * s, 0, row, pair, pol);
            tma_load_3d(dst + kHalfBytes, km, bar_full + 8 * s, 64, row, pair, pol);
            tma_load_3d(dst + kTileBytes, vm, bar_full + 8 * s, 0, row, pair, pol);
            tma_load_3d(dst + kTileBytes + kHalfBytes, vm, bar_full + 8 * s, 64, row, pair, pol);
        };
        const int pre = min(n_r, kStages);
        if (lane == 0) {
            for (int it = 0; it < pre; ++it)
                issue(it);
        }
        __syncwarp();
        const int per = (ps.k_tot + S - 1) / S;
        const int i0 = min(ps.k_tot, rank * per);
        const int n_s = producer_fetch_slice(ps, pair, i0, min(ps.k_tot, i0 + per) - i0, lslot, llog, ctrl, lane);
        named_barrier_arrive(1, kThreads);   // the selected slice and its length are in shared memory
        if (lane == 0) {
            if (compressed_rows(pc.seq_len[b], pc.cmp_len, pc.cmp_stride) > pc.pair_stride)
                report(pc.status, SPARSE_ERR_BAD_INDEX);
            for (int it = pre; it < n_r + n_s && ok; ++it)
                issue(it);
        }
    } else {
        // ------------------------------------------------------------ consumers
        if (early)
            griddep_wait();
        QueryFrags<NT> q;
        load_query<NT, false>(q, ps, b, g, 0, ps.G, lane);
        const long long len = ps.seq_len[b];
        const long long rows_c = unit_len(pc, b);
        const long long tok_lo = len - pw.win_tokens > 0 ? len - pw.win_tokens : 0;
        int it = 0;
        bool ok = true;
        // wait for ring item `it`, run `body` on its stage, release it
        auto step = [&](auto body) {
            const int s = it % kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (it / kStages) & 1, kWaitNs));
            if (!ok) {
                if (lane == 0)
                    report(ps.status, SPARSE_ERR_TIMEOUT);
                return;
            }
            body(base_s + s * kStageBytes);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
            ++it;
        };
        for (int i = 0; i < n_c && ok; ++i)
            step([&](uint32_t stage) {
                const long long r0 = static_cast<long long>(c_first + i) * kBlk + warp * 16;
                if (r0 < rows_c)
                    attend_block<NT, false>(st_c, q, stage, r0, rows_c, 0xffffffffu, ps.scale_log2, warp, lane);
            });
        for (int i = 0; i < n_w && ok; ++i)
            step([&](uint32_t stage) {
                const long long tok0 = static_cast<long long>(w_first + i) * kBlk + warp * 16;
                if (tok0 < len)
                    attend_block<NT, false>(st_w, q, stage, tok0, len, 0xffffffffu, ps.scale_log2, warp, lane,
                                            tok_lo);
            });
        named_barrier_sync(1, kThreads);
        const int n_s = ctrl[kCtrlList];
        for (int i = 0; i < n_s && ok; ++i)
            step([&](uint32_t stage) {
                const int logical = llog[i];
                const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
                if (logical >= 0 && tok0 < len)
                    attend_block<NT, false>(st_s, q, stage, tok0, len, 0xffffffffu, ps.scale_log2, warp, lane);
            });
        finish_row_sums<NT>(st_s);
        finish_row_sums<NT>(st_c);
        finish_row_sums<NT>(st_w);
    }

    // ---------------------------------------------------------------- merge + gates
    __syncthreads();
    griddep_launch_dependents();
    // The three branches' warp states side by side (branch x = s, c, w), merged into
    // three CTA states in one pass.
    constexpr int WO = kConsumerWarps * ROWS * kWoStride, WR = kConsumerWarps * ROWS;
    float *wo = reinterpret_cast<float *>(base);           // [3][4][ROWS][kWoStride]
    float *wm = wo + 3 * WO;                               // [3][4][ROWS]
    float *wl = wm + 3 * WR;
    float *wf = wl + 3 * WR;
    float *co = wf + 3 * WR;                               // [3][ROWS][128]
    float *cm = co + 3 * ROWS * kD;                        // [3][ROWS]
    float *cl = cm + 3 * ROWS;                             // [3][ROWS]
    if (warp < kConsumerWarps) {
        store_warp_state<NT>(st_s, wo, wm, wl, warp, lane);
        store_warp_state<NT>(st_c, wo + WO, wm + WR, wl + WR, warp, lane);
        store_warp_state<NT>(st_w, wo + 2 * WO, wm + 2 * WR, wl + 2 * WR, warp, lane);
    }
    __syncthreads();
    if (tid < 3 * ROWS) {
        const int x = tid / ROWS, row = tid - x * ROWS;
        const float *m4 = wm + x * WR, *l4 = wl + x * WR;
        float M = -INFINITY;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4)
            M = fmaxf(M, m4[w4 * ROWS + row]);
        float L = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4) {
            const float mw = m4[w4 * ROWS + row];
            const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
            wf[x * WR + w4 * ROWS + row] = f;
            L = fmaf(f, l4[w4 * ROWS + row], L);
        }
        cm[x * ROWS + row] = M;
        cl[x * ROWS + row] = L;
    }
    __syncthreads();
    // four adjacent dims per item (16-byte loads and stores: WO, kWoStride and the offset
    // of co are multiples of 4 floats)
    for (int item = tid; item < 3 * ROWS * (kD / 4); item += kThreads) {
        const int x = item / (ROWS * (kD / 4));
        const int r = item - x * ROWS * (kD / 4);
        const int row = r / (kD / 4), d = 4 * (r - row * (kD / 4));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4) {
            const float f = wf[x * WR + w4 * ROWS + row];
            const float4 v = *reinterpret_cast<const float4 *>(wo + x * WO + (w4 * ROWS + row) * kWoStride + d);
            o.x = fmaf(f, v.x, o.x);
            o.y = fmaf(f, v.y, o.y);
            o.z = fmaf(f, v.z, o.z);
            o.w = fmaf(f, v.w, o.w);
        }
        *reinterpret_cast<float4 *>(co + (x * ROWS + row) * kD + d) = o;
    }
    cluster_sync();

    const float *pco[kMaxSplit];
    const float *pcm[kMaxSplit];
    const float *pcl[kMaxSplit];
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) {
        const unsigned r = c < S ? static_cast<unsigned>(c) : 0u;
        pco[c] = static_cast<const float *>(__cluster_map_shared_rank(co, r));
        pcm[c] = static_cast<const float *>(__cluster_map_shared_rank(cm, r));
        pcl[c] = static_cast<const float *>(__cluster_map_shared_rank(cl, r));
    }
    // CTA `rank` writes dims [rank * 128 / S, (rank + 1) * 128 / S) of every head
    const int dims_per = kD / S;
    const int d0 = rank * dims_per;
    const int pairs_per_row = dims_per / 2;
    const int n_items = ps.G * pairs_per_row;
    for (int item = tid; item < n_items; item += kThreads) {
        const int row = item / pairs_per_row;
        const int d = d0 + 2 * (item - row * pairs_per_row);
        const size_t head = static_cast<size_t>(b) * ps.H_q + g * ps.G + row;
        float ox = 0.f, oy = 0.f;
#pragma unroll
        for (int x = 0; x < 3; ++x) {   // s, c, w
            float mc[kMaxSplit], lc[kMaxSplit];
            float2 v[kMaxSplit];
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c) {
                if (c < S) {
                    mc[c] = pcm[c][x * ROWS + row];
                    lc[c] = pcl[c][x * ROWS + row];
                    v[c] = *reinterpret_cast<const float2 *>(pco[c] + (x * ROWS + row) * kD + d);
                } else {
                    mc[c] = -INFINITY;
                    lc[c] = 0.f;
                    v[c] = make_float2(0.f, 0.f);
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c)
                M = fmaxf(M, mc[c]);
            float L = 0.f, bx = 0.f, by = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c) {
                const float f = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : exp2f(mc[c] - M);
                L = fmaf(lc[c], f, L);
                bx = fmaf(f, v[c].x, bx);
                by = fmaf(f, v[c].y, by);
            }
            // gates [head][3] = (g_c, g_s, g_w); branch x = s, c, w
            const float gate = np.gates[head * 3 + (x == 0 ? 1 : x == 1 ? 0 : 2)];
            const float scl = L > 0.f ? gate / L : 0.f;
            ox = fmaf(scl, bx, ox);
            oy = fmaf(scl, by, oy);
        }
        *reinterpret_cast<uint32_t *>(np.O + head * kD + d) = pack_bf16x2(ox, oy);
    }
    // peers may still read this CTA's states
    cluster_sync();
}

// The three-branch merge scratch must fit in the ring it reuses.
static_assert((3 * kConsumerWarps * 8 * kWoStride + 9 * kConsumerWarps * 8 + 3 * 8 * kD + 6 * 8) * 4 <=
                  kStages * kStageBytes,
              "NSA merge scratch exceeds the stage ring");
static_assert((3 * kConsumerWarps * 8 * kWoStride + 9 * kConsumerWarps * 8) % 4 == 0,
              "the NSA CTA states start 16-byte aligned");

size_t nsa_counter_bytes(long long pairs)
{
    return (static_cast<size_t>(pairs) * sizeof(unsigned) + 255) & ~static_cast<size_t>(255);
}

size_t nsa_workspace_bytes(long long pairs, int H_q_total)
{
    return nsa_counter_bytes(pairs) + static_cast<size_t>(3) * H_q_total * kD * sizeof(float);
}

template <int NT>
int launch_nsa(const NsaParams &np, const CUtensorMap *maps, int S, long long pairs, int device,
               cudaStream_t stream)
{
    auto kern = nsa_decode_kernel<NT>;
    const int smem = kSmemDecode + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 3);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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
    CUtensorMap m0 = maps[0], m1 = maps[1], m2 = maps[2], m3 = maps[3];
    NsaParams prm = np;
    void *args[] = {&m0, &m1, &m2, &m3, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse_decode_attn_nsa launch");
}

int launch_nsa_fused(const NsaParams &np, const CUtensorMap *maps, int S, long long pairs, int device,
                     cudaStream_t stream)
{
    const int smem = kSmemDecode + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(nsa_fused_kernel), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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
    CUtensorMap m0 = maps[0], m1 = maps[1], m2 = maps[2], m3 = maps[3];
    NsaParams prm = np;
    void *args[] = {&m0, &m1, &m2, &m3, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(nsa_fused_kernel), args),
                                "sparse_decode_attn_nsa launch");
}

}  // namespace

extern "C" SPARSE_API size_t sparse_decode_attn_nsa_workspace_size(int B, int H_q, int H_kv)
{
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0)
        return 0;
    return nsa_workspace_bytes(static_cast<long long>(B) * H_kv, B * H_q);
}

extern "C" SPARSE_API int sparse_decode_attn_nsa(const uint16_t *Q, const uint16_t *k_cache, const uint16_t *v_cache,
                                                 long long T_cap, const uint16_t *khat, const uint16_t *vhat,
                                                 int N_cap, int cmp_len, int cmp_stride, const int *blk_idx, const int *count, int k_tot,
                                                 const int *seq_len, int B, int H_q, int H_kv,
                                                 long long window_tokens, const float *gates, float scale,
                                                 uint16_t *O, void *workspace, size_t workspace_bytes, int n_split,
                                                 unsigned flags, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    const char *name = "sparse_decode_attn_nsa";
    if (!Q || !k_cache || !v_cache || !khat || !vhat || !blk_idx || !count || !seq_len || !gates || !O)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(Q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(khat) || !aligned16(vhat) ||
        !aligned16(O) || (workspace != nullptr && !aligned16(workspace)))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: Q, the caches, O and the workspace must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k_tot < 1 || T_cap < 1 || N_cap < 1 ||
        window_tokens < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size (B=%d H_q=%d H_kv=%d k_tot=%d N_cap=%d w=%lld)", name, B,
                    H_q, H_kv, k_tot, N_cap, window_tokens);
    if (T_cap > INT_MAX - 2 * kBlk || window_tokens > T_cap)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: T_cap or window_tokens too large", name);
    if (!isfinite(scale))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: scale must be finite", name);
    if (!(cmp_len == 0 && cmp_stride == 0) && !(cmp_stride >= 1 && cmp_stride <= cmp_len && cmp_len <= 1024))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: cmp_len=%d cmp_stride=%d (0, 0 or 1 <= stride <= len <= 1024)",
                    name, cmp_len, cmp_stride);
    if ((flags & ~(SPARSE_ATTN_BLOCKS_READY | SPARSE_NSA_BRANCH_GRID)) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
    const int G = H_q / H_kv;
    if (G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: G=%d > 16 query heads per KV head", name, G);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: B*H_kv=%lld > 65535", name, pairs);
    // the fused form holds the three branch states of G <= 8 heads in registers; the
    // branch grid (three clusters per pair, gates applied from the workspace) serves
    // the rest, or runs when asked
    const bool fused = G <= 8 && (flags & SPARSE_NSA_BRANCH_GRID) == 0u;
    const size_t need = nsa_workspace_bytes(pairs, B * H_q);
    if (!fused && (workspace == nullptr || workspace_bytes < need))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name,
                    workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes, need);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    if (n_split < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: n_split < 0", name);
    // block lists: the table, the window's blocks, the compressed rows' 64-row tiles
    const int k_win = static_cast<int>((window_tokens + kBlk - 1) / kBlk) + 1;
    const int k_cmp = (N_cap + kBlk - 1) / kBlk;
    const int k_max = fused ? k_tot + k_win + k_cmp : std::max(k_tot, std::max(k_win, k_cmp));
    int S;
    if ((rc = choose_split(n_split, pairs, k_max, dev.sm_count, &S)) != SPARSE_OK)
        return rc;
    // only the selected slice is staged in shared memory (the ranges are arithmetic)
    const int k_staged = fused ? k_tot : k_max;
    while ((k_staged + S - 1) / S > kMaxListCta && S < kMaxSplit && n_split == 0)
        S *= 2;
    if ((k_staged + S - 1) / S > kMaxListCta)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: %d blocks per CTA exceed %d", name, (k_staged + S - 1) / S,
                    kMaxListCta);
    CUtensorMap maps[4];
    if ((rc = sp_host::make_kv_tensor_map(&maps[0], k_cache, T_cap, pairs)) != SPARSE_OK ||
        (rc = sp_host::make_kv_tensor_map(&maps[1], v_cache, T_cap, pairs)) != SPARSE_OK ||
        (rc = sp_host::make_kv_tensor_map(&maps[2], khat, N_cap, pairs)) != SPARSE_OK ||
        (rc = sp_host::make_kv_tensor_map(&maps[3], vhat, N_cap, pairs)) != SPARSE_OK)
        return rc;
    float *part = fused ? nullptr
                        : reinterpret_cast<float *>(static_cast<char *>(workspace) + nsa_counter_bytes(pairs));
    const size_t branch_floats = static_cast<size_t>(B) * H_q * kD;
    NsaParams np = {};
    for (int x = 0; x < 3; ++x) {
        AttnParams &p = np.br[x];
        p.Q = Q;
        p.seq_len = seq_len;
        p.status = status;
        p.H_q = H_q;
        p.H_kv = H_kv;
        p.G = G;
        p.n_groups = 1;
        p.flags = flags & SPARSE_ATTN_BLOCKS_READY;
        p.scale_log2 = scale_log2_of(scale);
        p.O32 = fused ? nullptr : part + x * branch_floats;
    }
    np.br[0].blk_logical = blk_idx;
    np.br[0].count = count;
    np.br[0].k_tot = k_tot;
    np.br[0].pair_stride = T_cap;
    np.br[1].range_mode = 1;
    np.br[1].win_tokens = window_tokens;
    np.br[1].k_tot = k_win;
    np.br[1].pair_stride = T_cap;
    np.br[2].range_mode = 2;
    np.br[2].k_tot = k_cmp;
    np.br[2].pair_stride = N_cap;
    np.br[2].cmp_len = cmp_len;
    np.br[2].cmp_stride = cmp_stride;
    np.gates = gates;
    np.part = part;
    np.arrivals = fused ? nullptr : static_cast<unsigned *>(workspace);
    np.O = O;
    np.target = 3u * static_cast<unsigned>(S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (fused)
        return launch_nsa_fused(np, maps, S, pairs, dev.device, st);
    return G <= 8 ? launch_nsa<1>(np, maps, S, pairs, dev.device, st)
                  : launch_nsa<2>(np, maps, S, pairs, dev.device, st);
}

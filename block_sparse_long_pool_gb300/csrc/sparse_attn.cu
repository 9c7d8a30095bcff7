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
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace {

using namespace sp;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kHalfBytes = kBlk * 64 * 2;       // 64 tokens x 64 dims of bf16: one TMA box
constexpr int kTileBytes = 2 * kHalfBytes;      // one block of K (or V): 16 KB
constexpr int kStageBytes = 2 * kTileBytes;     // K + V of one block: 32 KB
constexpr int kMaxUnion = 512;
constexpr int kMaxSplit = 8;
constexpr uint64_t kWaitNs = 2000000000ull;

// Dynamic shared memory layout, offsets from a 1024-byte aligned base.
constexpr int kOffBars = kStages * kStageBytes;          // full[kStages], empty[kStages]
constexpr int kOffCtrl = kOffBars + 2 * kStages * 8;     // int ctrl[16]
constexpr int kOffList = kOffCtrl + 64;                  // verification: int ulist[kMaxUnion]
constexpr int kOffMask = kOffList + kMaxUnion * 4;       // uint32 umask[kMaxUnion]
constexpr int kOffEntV = kOffMask + kMaxUnion * 4;       // union build scratch
constexpr int kOffEntM = kOffEntV + kMaxUnion * 4;
constexpr int kOffEntF = kOffEntM + kMaxUnion * 4;
constexpr int kMaxListCta = kMaxUnion;                   // decode: staged slice of the block list
constexpr int kSmemDecode = kOffList + 2 * kMaxListCta * 4 + 1024;
constexpr int kSmemVerify = kOffEntF + kMaxUnion * 4 + 1024;

enum { kCtrlAbort = 0, kCtrlList = 1 };

struct AttnParams {
    const uint16_t *Q;
    uint16_t *O;
    float *lse;
    const int *blk_slot;
    const int *blk_logical;
    const int *count;
    const int *seq_len;
    int *status;
    const int *idx_q;
    long long *blocks_loaded;
    const unsigned *ready_flag;
    long long pair_stride;
    long long timeout_ns;
    unsigned ready_target;
    int k_tot;
    int H_q;
    int H_kv;
    int G;
    int n_sel;
    int N_q;
    int C;
    int window_blocks;
    int n_groups;
    unsigned flags;
    float scale_log2;
};

__device__ __forceinline__ uint32_t ld_b32(const uint16_t *p)
{
    return *reinterpret_cast<const uint32_t *>(p);
}

// Merged union of the group's block sets (SSV mode A): ulist ascending, umask[u] the
// queries of the group whose set contains ulist[u].  Returns the union size.
template <bool VERIFY>
__device__ __forceinline__ void build_union(const AttnParams &p, uint8_t *base, int b, int g, int q0,
                                            int nb, int *ctrl)
{
    int *ulist = reinterpret_cast<int *>(base + kOffList);
    uint32_t *umask = reinterpret_cast<uint32_t *>(base + kOffMask);
    int *ent_v = reinterpret_cast<int *>(base + kOffEntV);
    uint32_t *ent_m = reinterpret_cast<uint32_t *>(base + kOffEntM);
    int *ent_f = reinterpret_cast<int *>(base + kOffEntF);
    const int tid = threadIdx.x;
    const int nq = min(p.C, p.N_q - q0);
    const int wcount = min(p.window_blocks, nb);
    const int n_sel_ent = nq * p.n_sel;
    const int n_ent = n_sel_ent + wcount;
    const uint32_t all_q = nq >= 32 ? 0xffffffffu : ((1u << nq) - 1u);
    for (int e = tid; e < n_ent; e += kThreads) {
        int v;
        uint32_t m;
        if (e < n_sel_ent) {
            const int qi = e / p.n_sel;
            v = p.idx_q[((static_cast<size_t>(b) * p.H_kv + g) * p.N_q + q0 + qi) * p.n_sel + (e - qi * p.n_sel)];
            m = 1u << qi;
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
    for (int e = tid; e < kMaxUnion; e += kThreads)
        umask[e] = 0u;
    __syncthreads();
    for (int e = tid; e < n_ent; e += kThreads) {
        const int v = ent_v[e];
        int first = v != INT_MAX;
        for (int e2 = 0; e2 < e && first; ++e2)
            first = ent_v[e2] != v;
        ent_f[e] = first;
    }
    __syncthreads();
    for (int e = tid; e < n_ent; e += kThreads) {
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

template <int NT, bool VERIFY>
__global__ void __launch_bounds__(kThreads, 2)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const AttnParams p)
{
    constexpr int ROWS = 8 * NT;
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

    int pair, q0 = 0, rows_valid;
    if (VERIFY) {
        pair = blockIdx.y / p.n_groups;
        q0 = static_cast<int>(blockIdx.y % p.n_groups) * p.C;
        rows_valid = min(p.C, p.N_q - q0) * p.G;
    } else {
        pair = blockIdx.y;
        rows_valid = p.G;
    }
    const int b = pair / p.H_kv, g = pair % p.H_kv;
    // Programmatic dependent launch: this grid may start while the kernel before it on
    // the stream drains.  With SPARSE_ATTN_BLOCKS_READY the block list, lengths and K/V
    // are already complete (the caller's promise), so only Q and the outputs wait;
    // otherwise every input may come from that kernel and everything waits.
    const bool early = !VERIFY && (p.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();
    const long long len = p.seq_len[b];
    const int nb = len <= 0 ? 0 : static_cast<int>((len + kBlk - 1) / kBlk);

    if (tid == 0) {
        ctrl[kCtrlAbort] = 0;
        ctrl[kCtrlList] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        fence_barrier_init();
        if (p.ready_flag != nullptr) {
            // staging-ready integrity check, bounded
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
        if (!VERIFY) {
            int c = p.count[pair];
            if (c < 0 || c > p.k_tot) {
                report(p.status, SPARSE_ERR_BAD_INDEX);
                c = c < 0 ? 0 : p.k_tot;
            }
            ctrl[kCtrlList] = c;
        }
    }
    __syncthreads();
    if (VERIFY) {
        build_union<VERIFY>(p, base, b, g, q0, nb, ctrl);
        __syncthreads();
    }
    const bool aborted = ctrl[kCtrlAbort] != 0;
    const int n_list = aborted ? 0 : ctrl[kCtrlList];
    const int per = (n_list + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int i0 = min(n_list, static_cast<int>(rank) * per);
    const int i1 = min(n_list, i0 + per);
    const int my_n = i1 - i0;
    // block ids of this CTA's slice, in shared memory: verification keeps the merged
    // union (ulist/umask, whole list); decode stages its slice of the block table with
    // each entry validated (-1 = skip: an out-of-range box is loaded, never a fault)
    const int *ulist = reinterpret_cast<const int *>(base + kOffList);
    const uint32_t *umask = reinterpret_cast<const uint32_t *>(base + kOffMask);
    int *lslot = reinterpret_cast<int *>(base + kOffList);
    int *llog = lslot + kMaxListCta;
    if (!VERIFY) {
        for (int i = tid; i < my_n; i += kThreads) {
            const size_t at = static_cast<size_t>(pair) * p.k_tot + i0 + i;
            const int logical = p.blk_logical[at];
            const int slot = p.blk_slot != nullptr ? p.blk_slot[at] : logical;
            const bool ok = logical >= 0 && slot >= 0 && static_cast<long long>(slot) * kBlk < p.pair_stride;
            if (!ok)
                report(p.status, SPARSE_ERR_BAD_INDEX);
            lslot[i] = ok ? slot : -1;
            llog[i] = ok ? logical : -1;
        }
        __syncthreads();
    }

    if (VERIFY && rank == 0 && tid == 0 && p.blocks_loaded != nullptr && !aborted)
        atomicAdd(reinterpret_cast<unsigned long long *>(p.blocks_loaded),
                  static_cast<unsigned long long>(n_list));

    // per-thread softmax state (rows 2*t4 and 2*t4+1 of every n-tile) and O^T accumulators
    float m_r[NT][2], l_r[NT][2];
    float acc[8][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            m_r[nt][h] = -INFINITY;
            l_r[nt][h] = 0.f;
        }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc[mt][nt][i] = 0.f;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && my_n > 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const uint64_t pol = policy_evict_first();
            const int map_pair = pair;
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
                tma_load_3d(dst, &kmap, bar_full + 8 * s, 0, row, map_pair, pol);
                tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * s, 64, row, map_pair, pol);
                tma_load_3d(dst + kTileBytes, &vmap, bar_full + 8 * s, 0, row, map_pair, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, bar_full + 8 * s, 64, row, map_pair, pol);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int w = warp;
        const int g8 = lane >> 2, t4 = lane & 3;
        const int jm = lane >> 3, rr = lane & 7;

        if (early)
            griddep_wait();   // Q may be written by the kernel before this one
        // Q^T fragments (B operand of S^T = K Q^T): row n = g8 of each n-tile
        uint32_t qb[NT][8][2];
        bool row_ok[NT][2];
        int row_q[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = nt * 8 + g8;
            const uint16_t *qrow = nullptr;
            if (row < rows_valid) {
                if (VERIFY) {
                    const int qq = q0 + row / p.G, hh = row % p.G;
                    qrow = p.Q + ((static_cast<size_t>(b) * p.N_q + qq) * p.H_q + g * p.G + hh) * kD;
                } else {
                    qrow = p.Q + (static_cast<size_t>(b) * p.H_q + g * p.G + row) * kD;
                }
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[nt][ks][0] = qrow ? ld_b32(qrow + 16 * ks + 2 * t4) : 0u;
                qb[nt][ks][1] = qrow ? ld_b32(qrow + 16 * ks + 2 * t4 + 8) : 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = nt * 8 + 2 * t4 + h;
                row_ok[nt][h] = r < rows_valid;
                row_q[nt][h] = VERIFY ? (r < rows_valid ? r / p.G : 0) : 0;
            }
        }

        const int a_tok = w * 16 + (jm & 1) * 8 + rr;   // K rows for ldmatrix (QK A operand)
        const int v_tok = w * 16 + (jm >> 1) * 8 + rr;  // V rows for ldmatrix.trans (PV A operand)
        const uint32_t a_sw = static_cast<uint32_t>(a_tok & 7);
        const uint32_t v_sw = static_cast<uint32_t>(v_tok & 7);

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
            const int li = i0 + it;
            int logical;
            uint32_t qmask = 0xffffffffu;
            if (VERIFY) {
                logical = ulist[li];
                qmask = umask[li];
            } else {
                logical = llog[it];
            }
            const bool ok = logical >= 0;
            const long long tok0 = static_cast<long long>(logical) * kBlk + w * 16;
            if (ok && tok0 < len) {
                const uint32_t kst = base_s + s * kStageBytes;
                const uint32_t vst = kst + kTileBytes;
                float sacc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        sacc[nt][i] = 0.f;
                // S^T (16 tokens x 8*NT rows) = K (16 x 128) Q^T (128 x 8*NT)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t chunk = static_cast<uint32_t>(((ks & 3) << 1) + (jm >> 1));
                    const uint32_t addr = kst + (ks >> 2) * kHalfBytes + a_tok * 128 + ((chunk ^ a_sw) << 4);
                    uint32_t a[4];
                    ldsm_x4(addr, a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(sacc[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
                }
                // scale to log2 units, mask tokens past the length and rows not selecting the block
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int h = i & 1;
                        const long long tok = tok0 + g8 + (i >> 1) * 8;
                        bool keep = tok < len && row_ok[nt][h];
                        if (VERIFY)
                            keep = keep && ((qmask >> row_q[nt][h]) & 1u);
                        sacc[nt][i] = keep ? sacc[nt][i] * p.scale_log2 : -INFINITY;
                    }
                // online softmax per row (the 8 lanes sharing t4 hold one row's 16 tokens)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float mx = fmaxf(sacc[nt][h], sacc[nt][h + 2]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_new = fmaxf(m_r[nt][h], mx);
                        const float m_use = m_new == -INFINITY ? 0.f : m_new;
                        const float alpha = exp2f(m_r[nt][h] - m_use);
                        const float p0 = exp2f(sacc[nt][h] - m_use);
                        const float p1 = exp2f(sacc[nt][h + 2] - m_use);
                        l_r[nt][h] = l_r[nt][h] * alpha + p0 + p1;
                        m_r[nt][h] = m_new;
                        sacc[nt][h] = p0;
                        sacc[nt][h + 2] = p1;
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            acc[mt][nt][h] *= alpha;
                            acc[mt][nt][h + 2] *= alpha;
                        }
                    }
                // P^T as the B operand: transpose the bf16 (token, row) 8x8 tiles in registers
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    pb[nt][0] = movmatrix_trans(pack_bf16x2(sacc[nt][0], sacc[nt][1]));
                    pb[nt][1] = movmatrix_trans(pack_bf16x2(sacc[nt][2], sacc[nt][3]));
                }
                // O^T (128 dims x rows) += V^T (128 x 16 tokens) P^T (16 x rows)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const uint32_t chunk = static_cast<uint32_t>(((mt & 3) << 1) + (jm & 1));
                    const uint32_t addr = vst + (mt >> 2) * kHalfBytes + v_tok * 128 + ((chunk ^ v_sw) << 4);
                    uint32_t a[4];
                    ldsm_x4_trans(addr, a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(acc[mt][nt], a, pb[nt][0], pb[nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        // complete the row sums over the 8 lanes that share a row
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float l = l_r[nt][h];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_r[nt][h] = l;
            }
    }

    // ---------------------------------------------------------------- merge
    // Every stage has been consumed; the ring memory now holds the partial states.
    // The next kernel on the stream may be scheduled from here on.
    // (1) each consumer warp's state, (2) merged into this CTA's state in local shared
    // memory, (3) after one cluster barrier, CTA r merges the S CTA states for its
    // slice of output dims, reading its peers' shared memory with independent loads.
    __syncthreads();
    griddep_launch_dependents();
    float *wo = reinterpret_cast<float *>(base);                     // [4][ROWS][128]
    float *wm = wo + kConsumerWarps * ROWS * kD;                     // [4][ROWS]
    float *wl = wm + kConsumerWarps * ROWS;                          // [4][ROWS]
    float *wf = wl + kConsumerWarps * ROWS;                          // [4][ROWS] warp weights
    float *co = wf + kConsumerWarps * ROWS;                          // [ROWS][128] CTA state
    float *cm = co + ROWS * kD;                                      // [ROWS]
    float *cl = cm + ROWS;                                           // [ROWS]
    int *cabort = reinterpret_cast<int *>(cl + ROWS);                // [4]
    float *fac = reinterpret_cast<float *>(cabort + 4);              // [kMaxSplit][ROWS]
    float *row_m = fac + kMaxSplit * ROWS;
    float *row_l = row_m + ROWS;
    if (warp < kConsumerWarps) {
        const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int dim = mt * 16 + g8 + (i >> 1) * 8;
                    const int row = nt * 8 + 2 * t4 + (i & 1);
                    wo[(warp * ROWS + row) * kD + dim] = acc[mt][nt][i];
                }
        if (g8 == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = nt * 8 + 2 * t4 + h;
                    wm[warp * ROWS + row] = m_r[nt][h];
                    wl[warp * ROWS + row] = l_r[nt][h];
                }
        }
    }
    __syncthreads();
    if (tid < ROWS) {
        const int row = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4)
            M = fmaxf(M, wm[w4 * ROWS + row]);
        float L = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4) {
            const float mw = wm[w4 * ROWS + row];
            const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
            wf[w4 * ROWS + row] = f;
            L += f * wl[w4 * ROWS + row];
        }
        cm[row] = M;
        cl[row] = L;
    }
    if (tid == 0)
        cabort[0] = aborted ? 1 : 0;
    __syncthreads();
    for (int item = tid; item < ROWS * kD; item += kThreads) {
        const int row = item / kD;
        float o = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4)
            o = fmaf(wf[w4 * ROWS + row], wo[w4 * ROWS * kD + item], o);
        co[item] = o;
    }
    cluster_sync();

    // peers' CTA states (generic pointers into distributed shared memory)
    const float *peer_co[kMaxSplit];
    const float *peer_cm[kMaxSplit];
    const float *peer_cl[kMaxSplit];
    int any_abort = 0;
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) {
        const unsigned r = c < static_cast<int>(S) ? static_cast<unsigned>(c) : 0u;
        peer_co[c] = static_cast<const float *>(__cluster_map_shared_rank(co, r));
        peer_cm[c] = static_cast<const float *>(__cluster_map_shared_rank(cm, r));
        peer_cl[c] = static_cast<const float *>(__cluster_map_shared_rank(cl, r));
        const int ab = *static_cast<const int *>(__cluster_map_shared_rank(cabort, r));
        any_abort |= c < static_cast<int>(S) ? ab : 0;
    }

    // any CTA of the unit that failed its ready check leaves the output untouched
    if (!any_abort) {
        if (tid < ROWS) {
            const int row = tid;
            float mc[kMaxSplit], lc[kMaxSplit];
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c) {
                mc[c] = c < static_cast<int>(S) ? peer_cm[c][row] : -INFINITY;
                lc[c] = c < static_cast<int>(S) ? peer_cl[c][row] : 0.f;
            }
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c)
                M = fmaxf(M, mc[c]);
            float L = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c) {
                const float f = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : exp2f(mc[c] - M);
                fac[c * ROWS + row] = f;
                L += lc[c] * f;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c)
                fac[c * ROWS + row] *= inv;
            row_m[row] = M;
            row_l[row] = L;
        }
        __syncthreads();
        const int dims_per = kD / static_cast<int>(S);
        const int d0 = static_cast<int>(rank) * dims_per;
        for (int item = tid; item < rows_valid * dims_per; item += kThreads) {
            const int row = item / dims_per;
            const int d = d0 + (item - row * dims_per);
            float v[kMaxSplit];
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c)
                v[c] = c < static_cast<int>(S) ? peer_co[c][row * kD + d] : 0.f;
            float o = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxSplit; ++c)
                o = fmaf(fac[c * ROWS + row], v[c], o);
            size_t out;
            if (VERIFY) {
                const int qq = q0 + row / p.G, hh = row % p.G;
                out = ((static_cast<size_t>(b) * p.N_q + qq) * p.H_q + g * p.G + hh) * kD + d;
            } else {
                out = (static_cast<size_t>(b) * p.H_q + g * p.G + row) * kD + d;
            }
            const __nv_bfloat16 ob = __float2bfloat16_rn(o);
            p.O[out] = *reinterpret_cast<const uint16_t *>(&ob);
        }
        if (!VERIFY && rank == 0 && p.lse != nullptr) {
            for (int row = tid; row < rows_valid; row += kThreads) {
                const float L = row_l[row];
                p.lse[static_cast<size_t>(b) * p.H_q + g * p.G + row] =
                    L > 0.f ? (row_m[row] + log2f(L)) * 0.69314718055994530942f : -INFINITY;
            }
        }
    }
    // peers may still read this CTA's state
    cluster_sync();
}

template <int NT, bool VERIFY>
int launch(const AttnParams &p, const CUtensorMap &km, const CUtensorMap &vm, int S, long long units,
           int device, cudaStream_t stream)
{
    auto kern = sparse_attn_kernel<NT, VERIFY>;
    const int smem = (VERIFY ? kSmemVerify : kSmemDecode) + 1024;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(units), 1);
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
    CUtensorMap kmap = km, vmap = vm;
    AttnParams prm = p;
    void *args[] = {&kmap, &vmap, &prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse attention launch");
}

// The merge scratch (warp and CTA states, weights) must fit in the ring it reuses.
static_assert((3 * kConsumerWarps * 16 + kConsumerWarps * 16 * kD + 16 * kD + 2 * 16 + 4 + kMaxSplit * 16 + 2 * 16) *
                      4 <=
                  kStages * kStageBytes,
              "merge scratch exceeds the stage ring");

int choose_split(int n_split, long long units, int max_list, int sm_count, int *S)
{
    if (n_split == 0) {
        int s = 1;
        while (s < kMaxSplit && units * s * 2 <= 2LL * sm_count && s * 2 <= (max_list > 1 ? max_list / 2 : 1))
            s *= 2;
        *S = s;
        return SPARSE_OK;
    }
    if (n_split != 1 && n_split != 2 && n_split != 4 && n_split != 8)
        return sp_host::fail(SPARSE_ERR_INVALID_ARG, "n_split must be 0, 1, 2, 4 or 8 (got %d)", n_split);
    *S = n_split;
    return SPARSE_OK;
}

float scale_log2_of(float scale)
{
    const float s = scale == 0.f ? 1.f / sqrtf(static_cast<float>(kD)) : scale;
    return s * 1.44269504088896340736f;   // log2(e): scores are exponentiated base 2
}

int decode_impl(const uint16_t *Q, const uint16_t *k_base, const uint16_t *v_base, long long pair_stride,
                const int *blk_slot, const int *blk_logical, const int *count, int k_tot, const int *seq_len,
                int B, int H_q, int H_kv, float scale, uint16_t *O, float *lse, int n_split, unsigned flags,
                const unsigned *ready_flag, unsigned ready_target, long long timeout_ns, int *status,
                void *stream)
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
    const int G = H_q / H_kv;
    if (G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: G=%d > 16 query heads per KV head", G);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn: B*H_kv=%lld > 65535", pairs);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    if ((flags & ~SPARSE_ATTN_BLOCKS_READY) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: unknown flags 0x%x", flags);
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return G <= 8 ? launch<1, false>(p, km, vm, S, pairs, dev.device, st)
                  : launch<2, false>(p, km, vm, S, pairs, dev.device, st);
}

}  // namespace

extern "C" SPARSE_API int sparse_decode_attn(const uint16_t *Q, const uint16_t *k_base, const uint16_t *v_base,
                                             long long pair_stride_tokens, const int *blk_slot,
                                             const int *blk_logical, const int *count, int k_tot,
                                             const int *seq_len, int B, int H_q, int H_kv, float scale,
                                             uint16_t *O, float *lse, int n_split, unsigned flags, int *status,
                                             void *stream)
{
    return decode_impl(Q, k_base, v_base, pair_stride_tokens, blk_slot, blk_logical, count, k_tot, seq_len, B,
                       H_q, H_kv, scale, O, lse, n_split, flags, nullptr, 0u, 0, status, stream);
}

extern "C" SPARSE_API int sparse_decode_attn_ex(const uint16_t *Q, const uint16_t *k_base,
                                                const uint16_t *v_base, long long pair_stride_tokens,
                                                const int *blk_slot, const int *blk_logical, const int *count,
                                                int k_tot, const int *seq_len, int B, int H_q, int H_kv,
                                                float scale, uint16_t *O, float *lse, int n_split, unsigned flags,
                                                const unsigned *ready_flag, unsigned ready_target,
                                                long long timeout_ns, int *status, void *stream)
{
    if (ready_flag == nullptr)
        return sp_host::fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_ex: ready_flag is null");
    return decode_impl(Q, k_base, v_base, pair_stride_tokens, blk_slot, blk_logical, count, k_tot, seq_len, B,
                       H_q, H_kv, scale, O, lse, n_split, flags, ready_flag, ready_target, timeout_ns, status,
                       stream);
}

extern "C" SPARSE_API int sparse_verify_attn_grouped(const uint16_t *Q, const uint16_t *k_cache,
                                                     const uint16_t *v_cache, long long T_cap, const int *idx_q,
                                                     int n_sel, int N_q, int C, int window_blocks,
                                                     const int *seq_len, int B, int H_q, int H_kv, float scale,
                                                     uint16_t *O, long long *blocks_loaded, int n_split,
                                                     int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    if (!Q || !k_cache || !v_cache || !seq_len || !O || (n_sel > 0 && !idx_q))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_verify_attn_grouped: null pointer");
    if (!aligned16(Q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(O))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_verify_attn_grouped: Q, K, V and O must be 16-byte aligned");
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || N_q < 1 || C < 1 || n_sel < 0 ||
        window_blocks < 0 || T_cap < 1)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_verify_attn_grouped: bad size");
    if (T_cap > INT_MAX - 2 * kBlk)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_verify_attn_grouped: T_cap too large");
    if (!isfinite(scale))
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_verify_attn_grouped: scale must be finite");
    const int G = H_q / H_kv;
    if (C > 32 || static_cast<long long>(C) * G > 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_verify_attn_grouped: C*G=%lld rows > 16 per group",
                    static_cast<long long>(C) * G);
    if (static_cast<long long>(C) * n_sel + window_blocks > kMaxUnion)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_verify_attn_grouped: C*n_sel+window_blocks > %d", kMaxUnion);
    const int n_groups = (N_q + C - 1) / C;
    const long long units = static_cast<long long>(B) * H_kv * n_groups;
    if (units > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_verify_attn_grouped: too many groups");
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
    p.flags = 0u;
    p.scale_log2 = scale_log2_of(scale);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return C * G <= 8 ? launch<1, true>(p, km, vm, S, units, dev.device, st)
                      : launch<2, true>(p, km, vm, S, units, dev.device, st);
}

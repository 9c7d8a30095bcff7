// attn_core.cuh -- building blocks shared by the attention kernels (decode,
// grouped verification, and decode fused with the next layer's Forecast selection):
// the shared-memory ring layout, the per-warp online-softmax state, the tensor-core
// step over one 64-token block, and the merges of partial softmax states.
#pragma once

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
// The push merge's waits on the other CTAs of a cluster (see cluster_merge_write).
constexpr uint64_t kMergeWaitNs = 4 * kWaitNs;
// Row stride (floats) of the warp states in shared memory: a fragment store writes 8
// dims of 4 rows two apart, and the 4 extra floats put those rows in distinct banks.
constexpr int kWoStride = kD + 4;

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
// stream-K decode: the list of the CTA's range, its segment table and merge rows
constexpr int kMaxSegs = kMaxListCta + 2;
constexpr int kOffSegs = kOffList + 2 * kMaxListCta * 4;          // seg_nv[kMaxSegs], seg_start[kMaxSegs]
constexpr int kMaxMergeSeg = 64;                                  // CTAs sharing one pair, at most
constexpr int kOffRowML = kOffSegs + 2 * kMaxSegs * 4;            // row max / sum of a pair merge
constexpr int kOffMergeFac = kOffRowML + 2 * 16 * 4;              // [kMaxMergeSeg][8] weights (NT = 1)
constexpr int kOffMergeSlot = kOffMergeFac + 2 * kMaxMergeSeg * 8 * 4;   // [kMaxMergeSeg] slot offsets
constexpr int kSmemStreamK = kOffMergeSlot + kMaxMergeSeg * 4 + 1024;
enum { kCtrlLast = 2, kCtrlMergeValid = 3 };

enum { kCtrlAbort = 0, kCtrlList = 1 };

// Internal AttnParams::flags bit (not a public flag): grouped verification in SSV mode
// B, every query of a group on its first query's layout.
constexpr unsigned kVerifySharedLayout = 0x100u;

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
    // stream-K decode
    float *ws_part;        // [2 * n_ctas][ROWS * 128 + 2 * ROWS] partial states
    int *ws_count;         // [pairs] arrival counters, zero between calls
    long long n_items;     // pairs * k_tot
    // decode fused with the next layer's Forecast selection
    const uint16_t *F;     // [pairs][128] Forecast vectors, or null (no selection)
    const float *ktil;     // [pairs][N_cap][128] compressed keys of the next layer
    int *idx_next;         // [pairs][k_tot_next] selected blocks of the next layer
    int *count_next;       // [pairs]
    int N_cap;
    int n_init;
    int n_local;
    int k_sel;
    int k_tot_next;
    // NSA branches: fp32 output instead of bf16 O, and a block range computed from
    // seq_len instead of a block table (1: the window of the last win_tokens tokens,
    // masked token-granularly; 2: the compressed rows, one per 64-token block holding
    // a token, all of them)
    float *O32;
    long long win_tokens;
    int range_mode;
    // compressed rows of range_mode 2: one per 64-token block holding a token
    // (cmp_len = 0), or the complete windows [cmp_stride * j, cmp_stride * j + cmp_len)
    int cmp_len;
    int cmp_stride;
};

__device__ __forceinline__ uint32_t ld_b32(const uint16_t *p)
{
    return *reinterpret_cast<const uint32_t *>(p);
}

// Per-warp online-softmax state: the max and sum of rows 2*t4 and 2*t4+1 of every
// n-tile (log2 units) and the O^T accumulators of the warp's MMA fragments.
template <int NT>
struct WarpState {
    float m[NT][2], l[NT][2], acc[8][NT][4];

    __device__ __forceinline__ void reset()
    {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                m[nt][h] = -INFINITY;
                l[nt][h] = 0.f;
            }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[mt][nt][i] = 0.f;
    }
};

// Q^T fragments (the B operand of S^T = K Q^T; row n = lane/4 of each n-tile) and the
// validity / query index of the two rows this lane's softmax state covers.
template <int NT>
struct QueryFrags {
    uint32_t qb[NT][8][2];
    bool row_ok[NT][2];
    int row_q[NT][2];
};

// Query rows of a unit: decode rows are the G heads of KV head g of batch b;
// verification rows are (query q0 + r / G, head r % G).
template <int NT, bool VERIFY>
__device__ __forceinline__ void load_query(QueryFrags<NT> &q, const AttnParams &p, int b, int g, int q0,
                                           int rows_valid, int lane)
{
    const int g8 = lane >> 2, t4 = lane & 3;
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
            q.qb[nt][ks][0] = qrow ? ld_b32(qrow + 16 * ks + 2 * t4) : 0u;
            q.qb[nt][ks][1] = qrow ? ld_b32(qrow + 16 * ks + 2 * t4 + 8) : 0u;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = nt * 8 + 2 * t4 + h;
            q.row_ok[nt][h] = r < rows_valid;
            q.row_q[nt][h] = VERIFY ? (r < rows_valid ? r / p.G : 0) : 0;
        }
    }
}

// S^T (16 tokens x 8*NT rows) = K (16 x 128) Q^T (128 x 8*NT) for the tokens
// [16w, 16w+16) of the 64-row K tile at `kst` (2 x 8 KB boxes, 128-byte swizzle), on
// the bf16 tensor cores.  sacc[nt][i] holds token g8 + 8 (i >> 1) (g8 = lane / 4) and
// query row 8 nt + 2 (lane % 4) + (i & 1).
template <int NT>
__device__ __forceinline__ void score_rows(float (&sacc)[NT][4], const QueryFrags<NT> &q, uint32_t kst, int w,
                                           int lane)
{
    const int jm = lane >> 3, rr = lane & 7;
    const int a_tok = w * 16 + (jm & 1) * 8 + rr;   // K rows for ldmatrix (QK A operand)
    const uint32_t a_sw = static_cast<uint32_t>(a_tok & 7);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            sacc[nt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t chunk = static_cast<uint32_t>(((ks & 3) << 1) + (jm >> 1));
        const uint32_t addr = kst + (ks >> 2) * kHalfBytes + a_tok * 128 + ((chunk ^ a_sw) << 4);
        uint32_t a[4];
        ldsm_x4(addr, a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            mma_bf16_16816(sacc[nt], a, q.qb[nt][ks][0], q.qb[nt][ks][1]);
    }
}

// One consumer warp over tokens [16w, 16w+16) of the block held in ring stage `kst`
// (K, 2 x 8 KB swizzled boxes) and `kst + kTileBytes` (V).  tok0 is the absolute
// position of the warp's first token; qmask selects the rows' queries (verification).
template <int NT, bool VERIFY>
__device__ __forceinline__ void attend_block(WarpState<NT> &st, const QueryFrags<NT> &q, uint32_t kst, long long tok0,
                                             long long len, uint32_t qmask, float scale_log2, int w, int lane,
                                             long long tok_lo = 0)
{
    const int g8 = lane >> 2;
    const int jm = lane >> 3, rr = lane & 7;
    const int v_tok = w * 16 + (jm >> 1) * 8 + rr;  // V rows for ldmatrix.trans (PV A operand)
    const uint32_t v_sw = static_cast<uint32_t>(v_tok & 7);
    const uint32_t vst = kst + kTileBytes;
    float sacc[NT][4];
    score_rows<NT>(sacc, q, kst, w, lane);
    // scale to log2 units, mask tokens past the length and rows not selecting the block
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int h = i & 1;
            const long long tok = tok0 + g8 + (i >> 1) * 8;
            bool keep = tok < len && tok >= tok_lo && q.row_ok[nt][h];
            if (VERIFY)
                keep = keep && ((qmask >> q.row_q[nt][h]) & 1u);
            sacc[nt][i] = keep ? sacc[nt][i] * scale_log2 : -INFINITY;
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
            const float m_new = fmaxf(st.m[nt][h], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = exp2f(st.m[nt][h] - m_use);
            const float p0 = exp2f(sacc[nt][h] - m_use);
            const float p1 = exp2f(sacc[nt][h + 2] - m_use);
            st.l[nt][h] = st.l[nt][h] * alpha + p0 + p1;
            st.m[nt][h] = m_new;
            sacc[nt][h] = p0;
            sacc[nt][h + 2] = p1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                st.acc[mt][nt][h] *= alpha;
                st.acc[mt][nt][h + 2] *= alpha;
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
            mma_bf16_16816(st.acc[mt][nt], a, pb[nt][0], pb[nt][1]);
    }
}

// Complete the row sums over the 8 lanes that share a row.
template <int NT>
__device__ __forceinline__ void finish_row_sums(WarpState<NT> &st)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float l = st.l[nt][h];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            st.l[nt][h] = l;
        }
}

// Warp `warp`'s state into shared memory: wo [4][ROWS][kWoStride], wm / wl [4][ROWS].
template <int NT>
__device__ __forceinline__ void store_warp_state(const WarpState<NT> &st, float *wo, float *wm, float *wl, int warp,
                                                 int lane)
{
    constexpr int ROWS = 8 * NT;
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int dim = mt * 16 + g8 + (i >> 1) * 8;
                const int row = nt * 8 + 2 * t4 + (i & 1);
                wo[(warp * ROWS + row) * kWoStride + dim] = st.acc[mt][nt][i];
            }
    if (g8 == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = nt * 8 + 2 * t4 + h;
                wm[warp * ROWS + row] = st.m[nt][h];
                wl[warp * ROWS + row] = st.l[nt][h];
            }
    }
}

// Merge the 4 warp states (wo/wm/wl) into one CTA state: co [ROWS][128] unnormalised
// (16-byte aligned, as are the rows of wo), cm / cl [ROWS] its max and sum; wf [4][ROWS]
// scratch.  `t` / `nthreads` name the
// participating threads; the caller synchronises them between the two phases through
// `sync()`.
template <int ROWS, typename Sync>
__device__ __forceinline__ void merge_warp_states(const float *wo, const float *wm, const float *wl, float *wf,
                                                  float *co, float *cm, float *cl, int t, int nthreads, Sync sync)
{
    if (t < ROWS) {
        const int row = t;
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
    sync();
    // four adjacent dims per item (16-byte loads and stores)
    for (int item = t; item < ROWS * (kD / 4); item += nthreads) {
        const int row = item / (kD / 4);
        const int d = 4 * (item - row * (kD / 4));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4) {
            const float f = wf[w4 * ROWS + row];
            const float4 v = *reinterpret_cast<const float4 *>(wo + (w4 * ROWS + row) * kWoStride + d);
            o.x = fmaf(f, v.x, o.x);
            o.y = fmaf(f, v.y, o.y);
            o.z = fmaf(f, v.z, o.z);
            o.w = fmaf(f, v.w, o.w);
        }
        *reinterpret_cast<float4 *>(co + row * kD + d) = o;
    }
}

__device__ __forceinline__ void store_bf16(uint16_t *dst, float v)
{
    const __nv_bfloat16 ob = __float2bfloat16_rn(v);
    *dst = *reinterpret_cast<const uint16_t *>(&ob);
}

__device__ __forceinline__ float lse_of(float M, float L)
{
    return L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
}


// Producer warp of a decode CTA: the CTA's slice [i0, i0 + cap) of the pair's block
// table and the pair's count, fetched in one round trip (the slice is cut from k_tot,
// so it does not wait for the count); entries past the count are dropped and invalid
// ones become -1 (an out-of-range box is loaded for them: zeros, never a fault).  The
// ready word, if any, is checked with a bounded wait.  Writes lslot / llog[0 .. n),
// ctrl[kCtrlList] = n (0 when aborted) and ctrl[kCtrlAbort]; every lane returns n.
// Rows a unit of batch element b attends over: its tokens, or for the compressed
// branch (range_mode 2) its compressed rows, one per 64-token block holding a token.
// The compressed rows are clamped to the pair_stride rows that exist (the producer
// reports a length beyond them).
__device__ __forceinline__ long long unit_len(const AttnParams &p, int b)
{
    const long long len = p.seq_len[b];
    if (p.range_mode == 2) {
        const long long rows = compressed_rows(len, p.cmp_len, p.cmp_stride);
        return rows < p.pair_stride ? rows : p.pair_stride;
    }
    return len;
}

__device__ __forceinline__ int producer_fetch_slice(const AttnParams &p, int pair, int i0, int cap, int *lslot,
                                                    int *llog, int *ctrl, int lane)
{
    int c;
    if (p.range_mode != 0) {
        // a contiguous block range from the length: the window, or every block
        const int b = pair / p.H_kv;
        const long long len = unit_len(p, b);
        if (p.range_mode == 2 && lane == 0 && compressed_rows(p.seq_len[b], p.cmp_len, p.cmp_stride) > p.pair_stride)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        const int nb = len <= 0 ? 0 : static_cast<int>((len + kBlk - 1) / kBlk);
        long long w0 = p.range_mode == 1 ? len - p.win_tokens : 0;
        w0 = w0 < 0 ? 0 : w0;
        const int first = static_cast<int>(w0 / kBlk);
        c = nb > first ? nb - first : 0;
        if (p.range_mode == 1 && p.win_tokens <= 0)
            c = 0;
        for (int i = lane; i < cap; i += 32) {
            llog[i] = first + i0 + i;
            lslot[i] = first + i0 + i;
        }
        if (c > p.k_tot)
            c = -1;   // reported below: the range is longer than the table the host sized
    } else {
        c = lane == 0 ? p.count[pair] : 0;
        for (int i = lane; i < cap; i += 32) {
            const size_t at = static_cast<size_t>(pair) * p.k_tot + i0 + i;
            const int logical = p.blk_logical[at];
            llog[i] = logical;
            lslot[i] = p.blk_slot != nullptr ? p.blk_slot[at] : logical;
        }
        c = __shfl_sync(0xffffffffu, c, 0);
    }
    if (c < 0 || c > p.k_tot) {
        if (lane == 0)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        c = c < 0 ? 0 : p.k_tot;
    }
    const int my_n = max(0, min(cap, c - i0));
    for (int i = lane; i < my_n; i += 32) {
        const int logical = llog[i], slot = lslot[i];
        const bool ok = logical >= 0 && slot >= 0 && static_cast<long long>(slot) * kBlk < p.pair_stride;
        if (!ok) {
            report(p.status, SPARSE_ERR_BAD_INDEX);
            llog[i] = -1;
            lslot[i] = -1;
        }
    }
    int aborted = 0;
    if (lane == 0 && p.ready_flag != nullptr) {
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
            aborted = 1;
            report(p.status, p.timeout_ns > 0 ? SPARSE_ERR_TIMEOUT : SPARSE_ERR_NOT_READY);
        }
    }
    aborted = __shfl_sync(0xffffffffu, aborted, 0);
    const int n = aborted ? 0 : my_n;
    if (lane == 0) {
        ctrl[kCtrlAbort] = aborted;
        ctrl[kCtrlList] = n;
    }
    __syncwarp();
    return n;
}

// The merge of a cluster's partial states (split-KV): (1) each consumer warp's state
// into shared memory, (2) merged into this CTA's state, (3) after one cluster barrier
// The cluster merge of the S CTA states of a unit (decode pair, or verification group):
// rows [0, rows_valid) of O (and lse) written once, from every CTA's partial softmax
// state.  Every thread of every CTA of the cluster calls it (`nthreads` = blockDim.x);
// the ring at `base` is reused as scratch, so every stage must have been consumed.  A
// CTA that failed its ready check (`aborted`) makes the whole unit leave O and lse
// untouched.  `wait_cluster`: the caller arrived on the cluster barrier at its start
// and has not waited on it yet.  `allow_push`: the caller initialised the merge barriers
// (merge_barriers_init) before that arrive, and the push form may run.
//   push (when allowed and the slots fit): the leader (rank 0) tells each peer once its ring is
//     free; a peer merges its warps' states and copies its CTA state into the leader's
//     slot (16-byte distributed-shared-memory stores), arrives on the leader's barrier
//     and leaves; the leader merges the S states for every output dim.  No cluster-wide
//     barrier: the peers do not wait for one another, nor for the leader's output.
//     Lifetimes: a peer is alive until it has seen "go" (the leader's only remote access
//     to it), and the leader until it has received every state (the peers' only remote
//     accesses to it).  A CTA gives up one of these waits only after kMergeWaitNs,
//     longer than any CTA of the cluster can take to reach its merge (its pipeline
//     waits are bounded by kWaitNs and a CTA leaves its loops at the first that runs
//     out, so a stalled CTA arrives within about two such waits of starting), so a CTA
//     that gives up has outlived every remote access the others can still make --
//     unless a pipeline keeps crawling at under one stage per kWaitNs, which no bounded
//     wait can tell from progress.
//   pull: every CTA waits for all, then merges the S states for its slice of the dims
//     by reading its peers' shared memory, and all wait again before leaving.
constexpr int kCtrlGoBar = 10;            // ctrl[10..11]: "the leader's slots are free" (every CTA)
constexpr int kCtrlRecvBar = 12;          // ctrl[12..13]: the peers' states have landed (leader)

// The leader's slots: in its ring past the merge scratch (the 4 warp states, the warp
// weights and the CTA state, with the abort words), on a 1 KB boundary.
template <int NT>
__host__ __device__ constexpr int push_recv_off()
{
    return ((kConsumerWarps * 8 * NT * kWoStride + 3 * kConsumerWarps * 8 * NT + 8 * NT * kD + 2 * 8 * NT + 4) * 4 +
            1023) / 1024 * 1024;
}

template <int NT>
__host__ __device__ constexpr int push_slot_floats()
{
    return 8 * NT * kD + 2 * 8 * NT + 4;   // CTA state: O [ROWS][128], m [ROWS], l [ROWS], abort flag
}
static_assert(push_slot_floats<1>() % 4 == 0 && push_slot_floats<2>() % 4 == 0,
              "each slot starts 16-byte aligned, so its rows take 16-byte loads");

// Whether the push form runs: at most kMaxSplit CTAs (beyond, one leader merging every
// state for all 128 dims takes longer than the pull form, where each CTA merges its own
// 128 / S dims: measured at 16 CTAs) and the S - 1 slots fit in the leader's ring.
template <int NT>
__host__ __device__ constexpr bool merge_pushes(uint32_t S)
{
    return S > 1 && S <= static_cast<uint32_t>(kMaxSplit) &&
           push_recv_off<NT>() + static_cast<int>(S - 1) * push_slot_floats<NT>() * 4 <= kStages * kStageBytes;
}
static_assert(merge_pushes<1>(8) && merge_pushes<2>(4), "the push merge serves the fused layer's clusters");

// Thread 0 at kernel start, before fence_barrier_init and the cluster arrive.
__device__ __forceinline__ void merge_barriers_init(uint32_t ctrl_s, uint32_t S, int nthreads)
{
    mbar_init(ctrl_s + 4 * kCtrlGoBar, 1);
    mbar_init(ctrl_s + 4 * kCtrlRecvBar, (S > 1 ? S - 1 : 1) * static_cast<uint32_t>(nthreads / 32));
}

__device__ __forceinline__ void dsmem_st_v4(uint32_t addr, float4 v)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// Four adjacent output dims [d, d + 4) of one row (16-byte aligned: d % 4 == 0).
template <int NT, bool VERIFY>
__device__ __forceinline__ void merge_write_item4(const AttnParams &p, int b, int g, int q0, int row, int d, float M,
                                                  float L, float4 o, bool write_lse)
{
    const float inv = L > 0.f ? 1.f / L : 0.f;
    size_t out;
    if (VERIFY) {
        const int qq = q0 + row / p.G, hh = row % p.G;
        out = ((static_cast<size_t>(b) * p.N_q + qq) * p.H_q + g * p.G + hh) * kD + d;
    } else {
        out = (static_cast<size_t>(b) * p.H_q + g * p.G + row) * kD + d;
    }
    if (p.O32 != nullptr)
        *reinterpret_cast<float4 *>(p.O32 + out) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    else
        *reinterpret_cast<uint2 *>(p.O + out) = make_uint2(pack_bf16x2(o.x * inv, o.y * inv),
                                                           pack_bf16x2(o.z * inv, o.w * inv));
    if (!VERIFY && write_lse && d == 0 && p.lse != nullptr)
        p.lse[static_cast<size_t>(b) * p.H_q + g * p.G + row] = lse_of(M, L);
}

// The CTA state's place in the ring (merge scratch): co [ROWS][128] unnormalised O,
// cm / cl [ROWS] its row max and sum, past the 4 warp states.
template <int NT>
__device__ __forceinline__ float *merge_cta_state(uint8_t *base)
{
    constexpr int ROWS = 8 * NT;
    return reinterpret_cast<float *>(base) + kConsumerWarps * ROWS * kWoStride + 3 * kConsumerWarps * ROWS;
}

// The leader (warp 0 of CTA 0) tells each peer that its ring is consumed: the peers may
// fill its slots.  Once per launch.  Lane r arrives on peer r: remote arrives issued one
// after another by one thread each wait for the previous one's release (~0.7 us each on
// GB300), while one per lane go out together.
__device__ __forceinline__ void merge_send_go(uint32_t ctrl_s, uint32_t S, int lane)
{
    if (lane >= 1 && static_cast<uint32_t>(lane) < S)
        mbar_arrive_cluster(dsmem_addr(ctrl_s + 4 * kCtrlGoBar, static_cast<uint32_t>(lane)));
}

// `cta_state_ready`: the caller has written the CTA state (merge_cta_state) itself, and
// `st` is not read.  `go_sent`: the leader's warp 0 already called merge_send_go (its
// ring was free early).
template <int NT, bool VERIFY, int MAXS = kMaxSplit>
__device__ __forceinline__ void cluster_merge_write(const WarpState<NT> &st, uint8_t *base, bool aborted,
                                                    const AttnParams &p, int b, int g, int q0, int rows_valid,
                                                    uint32_t rank, uint32_t S, int nthreads, uint32_t ctrl_s,
                                                    bool wait_cluster, bool allow_push, bool cta_state_ready = false,
                                                    bool go_sent = false, bool skip0 = false)
{
    constexpr int ROWS = 8 * NT;
    constexpr int SLOT = push_slot_floats<NT>();
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    float *wo = reinterpret_cast<float *>(base);                     // [4][ROWS][kWoStride]
    float *wm = wo + kConsumerWarps * ROWS * kWoStride;              // [4][ROWS]
    float *wl = wm + kConsumerWarps * ROWS;                          // [4][ROWS]
    float *wf = wl + kConsumerWarps * ROWS;                          // [4][ROWS] warp weights
    float *co = wf + kConsumerWarps * ROWS;                          // [ROWS][128] CTA state
    float *cm = co + ROWS * kD;                                      // [ROWS]
    float *cl = cm + ROWS;                                           // [ROWS]
    int *cabort = reinterpret_cast<int *>(cl + ROWS);                // [4]
    const bool push = allow_push && merge_pushes<NT>(S);
    const uint32_t bar_go = ctrl_s + 4 * kCtrlGoBar, bar_recv = ctrl_s + 4 * kCtrlRecvBar;
    if (wait_cluster)
        cluster_wait();   // every CTA's merge barriers are initialised
    if (push && rank == 0 && warp == 0 && !go_sent)
        merge_send_go(ctrl_s, S, lane);
    if (!cta_state_ready && warp < kConsumerWarps)
        store_warp_state<NT>(st, wo, wm, wl, warp, lane);
    if (tid == 0)
        cabort[0] = aborted ? 1 : 0;
    __syncthreads();
    if (!cta_state_ready) {
        merge_warp_states<ROWS>(wo, wm, wl, wf, co, cm, cl, tid, nthreads, [] { __syncthreads(); });
        __syncthreads();   // the CTA state (co, cm, cl, cabort) is complete
    }
    if (push) {
        const float *slots = reinterpret_cast<const float *>(base + push_recv_off<NT>());   // [S - 1][SLOT]
        if (rank != 0) {
            // a peer: copy the CTA state, contiguous from co, into slot rank - 1 of the leader
            const bool go = __all_sync(0xffffffffu, mbar_wait_cluster(bar_go, 0, kMergeWaitNs));
            if (!go) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                return;
            }
            const uint32_t dst = dsmem_addr(smem_u32(base + push_recv_off<NT>()) + (rank - 1) * SLOT * 4, 0);
            const float4 *src = reinterpret_cast<const float4 *>(co);
            for (int q4 = tid; q4 < SLOT / 4; q4 += nthreads)
                dsmem_st_v4(dst + 16 * q4, src[q4]);
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_recv, 0));
            return;
        }
        // the leader: the S states, own first, then the slots in rank order
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar_recv, 0, kMergeWaitNs))) {
            if (lane == 0)
                report(p.status, SPARSE_ERR_TIMEOUT);
            return;
        }
        int any_abort = cabort[0];
        for (uint32_t c = 1; c < S; ++c)
            any_abort |= reinterpret_cast<const int *>(slots + (c - 1) * SLOT + ROWS * kD + 2 * ROWS)[0];
        if (any_abort)
            return;
        // four adjacent dims per item (the slots are 16-byte aligned: SLOT % 4 == 0)
        const int n_items = rows_valid * (kD / 4);
        for (int item = tid; item < n_items; item += nthreads) {
            const int row = item / (kD / 4);
            const int d = 4 * (item - row * (kD / 4));
            float mc[MAXS], lc[MAXS];
            float4 v[MAXS];
#pragma unroll
            for (int c = 0; c < MAXS; ++c) {
                if (c < static_cast<int>(S)) {
                    const float *src = c == 0 ? co : slots + (c - 1) * SLOT;
                    mc[c] = src[ROWS * kD + row];
                    lc[c] = src[ROWS * kD + ROWS + row];
                    v[c] = *reinterpret_cast<const float4 *>(src + row * kD + d);
                } else {
                    mc[c] = -INFINITY;
                    lc[c] = 0.f;
                    v[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < MAXS; ++c)
                M = fmaxf(M, mc[c]);
            float L = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < MAXS; ++c) {
                const float f = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : exp2f(mc[c] - M);
                L = fmaf(lc[c], f, L);
                o.x = fmaf(f, v[c].x, o.x);
                o.y = fmaf(f, v[c].y, o.y);
                o.z = fmaf(f, v[c].z, o.z);
                o.w = fmaf(f, v[c].w, o.w);
            }
            merge_write_item4<NT, VERIFY>(p, b, g, q0, row, d, M, L, o, true);
        }
        return;
    }
    cluster_sync();

    // Peers' CTA states (generic pointers into distributed shared memory).  Every value
    // a thread needs for an output pair is loaded before any is used, so the remote
    // loads of an item overlap (one round trip).  With `skip0` CTA 0 holds no state and
    // takes no part: the states and the dims are those of CTAs 1 .. S-1.
    const int c0 = skip0 ? 1 : 0;
    const int Si = static_cast<int>(S) - c0;
    // each peer's CTA state as a shared::cluster address (co; cm and cl follow it)
    uint32_t pst[MAXS];
    int any_abort = 0;
#pragma unroll
    for (int c = 0; c < MAXS; ++c) {
        const uint32_t r = c < Si ? static_cast<uint32_t>(c + c0) : static_cast<uint32_t>(c0);
        pst[c] = dsmem_addr(smem_u32(co), r);
        if (c < Si)
            any_abort |= static_cast<int>(dsmem_ld_u32(pst[c] + 4u * static_cast<uint32_t>(ROWS * kD + 2 * ROWS)));
    }
    // CTA `rank` writes quads [qa, qb) (four adjacent dims each) of every row: with
    // every CTA taking part, dims [rank * 128 / S, (rank + 1) * 128 / S); with up to 16
    // rows and S >= 4, one item per thread, so the remote loads of the whole slice are
    // one round trip
    const int me = static_cast<int>(rank) - c0;
    const int qa = me * (kD / 4) / Si, qb = (me + 1) * (kD / 4) / Si;
    const int quads_per_row = qb - qa;
    const int n_items = rows_valid * quads_per_row;
    for (int item = tid; item < n_items; item += nthreads) {
        const int row = item / quads_per_row;
        const int d = 4 * (qa + item - row * quads_per_row);
        float mc[MAXS], lc[MAXS];
        float4 v[MAXS];
#pragma unroll
        for (int c = 0; c < MAXS; ++c) {
            if (c < Si) {
                mc[c] = dsmem_ld_f32(pst[c] + 4u * static_cast<uint32_t>(ROWS * kD + row));
                lc[c] = dsmem_ld_f32(pst[c] + 4u * static_cast<uint32_t>(ROWS * kD + ROWS + row));
                v[c] = dsmem_ld_v4(pst[c] + 4u * static_cast<uint32_t>(row * kD + d));
            } else {
                mc[c] = -INFINITY;
                lc[c] = 0.f;
                v[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        // any CTA of the unit that failed its ready check leaves the output untouched
        if (any_abort)
            break;
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < MAXS; ++c)
            M = fmaxf(M, mc[c]);
        float L = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < MAXS; ++c) {
            const float f = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : exp2f(mc[c] - M);
            L = fmaf(lc[c], f, L);
            o.x = fmaf(f, v[c].x, o.x);
            o.y = fmaf(f, v[c].y, o.y);
            o.z = fmaf(f, v[c].z, o.z);
            o.w = fmaf(f, v[c].w, o.w);
        }
        merge_write_item4<NT, VERIFY>(p, b, g, q0, row, d, M, L, o, true);   // lse with dim 0
    }
    // peers may still read this CTA's state
    cluster_sync();
}

// ---------------------------------------------------------------- host helpers

// Cluster size S (CTAs sharing one unit's list) for the cluster kernels: auto = enough
// units x S to cover the SMs twice, at least two blocks per CTA; at most max_s (8, the
// portable cluster size, or 16 for a kernel that allows the non-portable size).
inline int choose_split(int n_split, long long units, int max_list, int sm_count, int *S, int max_s = kMaxSplit)
{
    if (n_split == 0) {
        int s = 1;
        while (s < max_s && units * s * 2 <= 2LL * sm_count && s * 2 <= (max_list > 1 ? max_list / 2 : 1))
            s *= 2;
        *S = s;
        return SPARSE_OK;
    }
    if (n_split != 1 && n_split != 2 && n_split != 4 && n_split != 8 && !(n_split == 16 && max_s >= 16))
        return sp_host::fail(SPARSE_ERR_INVALID_ARG, "n_split must be 0, 1, 2, 4 or 8%s (got %d)",
                             max_s >= 16 ? " or 16" : "", n_split);
    *S = n_split;
    return SPARSE_OK;
}

inline float scale_log2_of(float scale)
{
    const float s = scale == 0.f ? 1.f / sqrtf(static_cast<float>(kD)) : scale;
    return s * 1.44269504088896340736f;   // log2(e): scores are exponentiated base 2
}

}  // namespace

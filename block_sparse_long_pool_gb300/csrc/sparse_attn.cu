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

#include <mutex>

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

// One consumer warp over tokens [16w, 16w+16) of the block held in ring stage `kst`
// (K, 2 x 8 KB swizzled boxes) and `kst + kTileBytes` (V).  tok0 is the absolute
// position of the warp's first token; qmask selects the rows' queries (verification).
template <int NT, bool VERIFY>
__device__ __forceinline__ void attend_block(WarpState<NT> &st, const QueryFrags<NT> &q, uint32_t kst, long long tok0,
                                             long long len, uint32_t qmask, float scale_log2, int w, int lane)
{
    const int g8 = lane >> 2;
    const int jm = lane >> 3, rr = lane & 7;
    const int a_tok = w * 16 + (jm & 1) * 8 + rr;   // K rows for ldmatrix (QK A operand)
    const int v_tok = w * 16 + (jm >> 1) * 8 + rr;  // V rows for ldmatrix.trans (PV A operand)
    const uint32_t a_sw = static_cast<uint32_t>(a_tok & 7);
    const uint32_t v_sw = static_cast<uint32_t>(v_tok & 7);
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
            mma_bf16_16816(sacc[nt], a, q.qb[nt][ks][0], q.qb[nt][ks][1]);
    }
    // scale to log2 units, mask tokens past the length and rows not selecting the block
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int h = i & 1;
            const long long tok = tok0 + g8 + (i >> 1) * 8;
            bool keep = tok < len && q.row_ok[nt][h];
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

// Warp `warp`'s state into shared memory: wo [4][ROWS][128], wm / wl [4][ROWS].
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
                wo[(warp * ROWS + row) * kD + dim] = st.acc[mt][nt][i];
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

// Merge the 4 warp states (wo/wm/wl) into one CTA state: co [ROWS][128] unnormalised,
// cm / cl [ROWS] its max and sum; wf [4][ROWS] scratch.  `t` / `nthreads` name the
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
    for (int item = t; item < ROWS * kD; item += nthreads) {
        const int row = item / kD;
        float o = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < kConsumerWarps; ++w4)
            o = fmaf(wf[w4 * ROWS + row], wo[w4 * ROWS * kD + item], o);
        co[item] = o;
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

    WarpState<NT> st;
    st.reset();

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
        if (early)
            griddep_wait();   // Q may be written by the kernel before this one
        QueryFrags<NT> q;
        load_query<NT, VERIFY>(q, p, b, g, q0, rows_valid, lane);
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
            const long long tok0 = static_cast<long long>(logical) * kBlk + warp * 16;
            if (logical >= 0 && tok0 < len)
                attend_block<NT, VERIFY>(st, q, base_s + s * kStageBytes, tok0, len, qmask, p.scale_log2, warp,
                                         lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        finish_row_sums<NT>(st);
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
    if (warp < kConsumerWarps)
        store_warp_state<NT>(st, wo, wm, wl, warp, lane);
    if (tid == 0)
        cabort[0] = aborted ? 1 : 0;
    __syncthreads();
    merge_warp_states<ROWS>(wo, wm, wl, wf, co, cm, cl, tid, kThreads, [] { __syncthreads(); });
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
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
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
            float *wm = wo + kConsumerWarps * ROWS * kD;
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
                void *workspace, size_t workspace_bytes, const unsigned *ready_flag, unsigned ready_target,
                long long timeout_ns, int *status, void *stream)
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
    if ((flags & ~(SPARSE_ATTN_BLOCKS_READY | SPARSE_ATTN_STREAM_K)) != 0u)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: unknown flags 0x%x", flags);
    if (n_split < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn: n_split < 0");
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
    // Stream-K when asked, or when the pairs are too few for clusters of CTAs to cover
    // the SMs; otherwise the cluster path (the faster one once every SM is busy).
    const bool stream_k = workspace != nullptr && G <= 8 &&
                          ((flags & SPARSE_ATTN_STREAM_K) != 0u || pairs * 4 < dev.sm_count);
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
    return G <= 8 ? launch<1, false>(p, km, vm, S, pairs, dev.device, st)
                  : launch<2, false>(p, km, vm, S, pairs, dev.device, st);
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

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];   // device address of the array, per device

// The device address of g_noalloc_scratch on the current device (the host-side name of
// the array is only a stand-in, never a device address).  Looked up once per device.
int noalloc_scratch(int device, void **ptr)
{
    if (device < 0 || device >= 64)
        return sp_host::fail(SPARSE_ERR_UNSUPPORTED, "device ordinal %d out of range", device);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[device] == nullptr) {
        void *addr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess || addr == nullptr)
            return sp_host::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                                        "sparse_decode_attn_noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[device] = addr;
    }
    *ptr = g_noalloc_ptr[device];
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
    if (B < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || k_tot < 1 || n_split < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "sparse_decode_attn_noalloc: bad size");
    if (H_q / H_kv > 8)
        return fail(SPARSE_ERR_UNSUPPORTED, "sparse_decode_attn_noalloc: G=%d > 8", H_q / H_kv);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    const long long pairs = static_cast<long long>(B) * H_kv;
    const int n_ctas = streamk_ctas(pairs * k_tot, pairs, n_split, dev.sm_count);
    const size_t need = streamk_workspace_bytes(pairs, H_q / H_kv, n_ctas);
    if (need > kNoallocScratchBytes)
        return fail(SPARSE_ERR_UNSUPPORTED,
                    "sparse_decode_attn_noalloc: these sizes need %zu bytes of scratch, more than the fixed %zu "
                    "(use sparse_decode_attn with a workspace)",
                    need, kNoallocScratchBytes);
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(dev.device, &scratch)) != SPARSE_OK)
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
    if (G > 8)
        return 0;   // the cluster path (no workspace) serves G > 8
    return streamk_workspace_bytes(pairs, G, streamk_ctas(pairs * k_tot, pairs, n_split, dev.sm_count));
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

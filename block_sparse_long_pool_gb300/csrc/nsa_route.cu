// nsa_route.cu -- NSA's routing over its compressed keys (per-head softmax summed over
// the GQA group, max-pooled onto the 64-token selection blocks, top-k).
#include <limits.h>
#include <math.h>

#include "attn_core.cuh"
#include "select_core.cuh"
#include "select_layout.cuh"

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
//   3. p_j for the CTA's rows (four rows per thread at a time) and the block maxima as
//      order keys -> CTA 0, whose consumers and selector warp take the top-k together
//      (topk_cta_regs: the summed probabilities share an exponent, so the bits every
//      key shares are decided at once and a binary search with block-wide counts finds
//      the rest; past 2720 candidates a block-wide radix threshold and a one-warp
//      write).

namespace {

constexpr int kRouteStageBytes = kTileBytes;   // 64 rows x 128 dims, bf16: two 64 x 64 boxes
constexpr int kRouteTopkThreads = (kConsumerWarps + 1) * 32;   // CTA 0's consumers + selector
constexpr int kRouteKpt = 17;   // candidate keys per thread in the register top-k (2720 blocks)

struct RouteParams {
    const uint16_t *Q;
    const int *seq_len;
    int *idx;
    int *count;
    int *status;
    int H_q, H_kv, G;
    int N_q;              // queries per batch element (each routed on its own)
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
    if (threadIdx.x == kConsumerWarps * 32)   // the descriptor is a parameter: fetched while waiting
        prefetch_tensormap(&kmap);
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
    const int unit = static_cast<int>(blockIdx.y);   // (pair, query)
    const int pair = unit / p.N_q, qi = unit - pair * p.N_q;
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
    const bool regs_topk = topk_cta_regs_fits<kRouteKpt>(nb - p.n_local - p.n_init, kRouteTopkThreads);
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
            ap.Q = p.Q + static_cast<size_t>(b) * (p.N_q - 1) * p.H_q * kD +
                   static_cast<size_t>(qi) * p.H_q * kD;   // query qi of batch element b
            ap.H_q = p.H_q;
            ap.G = G;
            load_query<NT, false>(q, ap, b, g, 0, G, lane);
        }
        cluster_wait();
        uint32_t *keys0 = static_cast<uint32_t *>(__cluster_map_shared_rank(keys, 0));
        float *stats0 = static_cast<float *>(__cluster_map_shared_rank(stats, 0));
        const int g8 = lane >> 2, t4 = lane & 3;
        bool ok = true;
        // owned rows in local indices; each lane keeps the running max of its heads
        // (nt * 8 + 2 * t4 + hb) over the owned rows it scores (two fmaxf per score)
        const int own0 = o_lo - j_lo, own1 = b_hi > b_lo ? o_hi - j_lo : own0;
        float mrun[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            mrun[nt][0] = mrun[nt][1] = -INFINITY;
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
                    if (lr >= own0 && lr < own1)
                        mrun[nt][i & 1] = fmaxf(mrun[nt][i & 1], sacc[nt][i] * p.scale_log2);
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * st);
        }
        // the warp's max per head (the 8 lanes that share t4) -> wmax [warp][16 heads],
        // past CTA 0's top-k scratch in its radix-bin region
        float *wmax = reinterpret_cast<float *>(base + L.off_hist) + 64;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float m = mrun[nt][hb];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const int h = nt * 8 + 2 * t4 + hb;
                if (g8 == 0 && h < G)
                    wmax[warp * 16 + h] = m;
            }
        named_barrier_sync(2, kConsumerWarps * 32);   // every raw score and warp max is written
        if (score) {
            // (2) per head: max and sum of exp2 over the owned rows, merged by CTA 0 (one
            // warp per scheduler: four independent accumulators per lane)
            for (int h = warp; h < G; h += kConsumerWarps) {
                const float *rh = raw + h * p.rows_cta_max;
                float m = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    m = fmaxf(m, wmax[w * 16 + h]);
                float z4[4] = {0.f, 0.f, 0.f, 0.f};
                if (m != -INFINITY)
                    for (int i = own0 + lane; i < own1; i += 128)
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float e = ex2_approx(rh[min(i + 32 * q4, own1 - 1)] - m);
                            z4[q4] += i + 32 * q4 < own1 ? e : 0.f;
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
            const bool have_norm = __all_sync(0xffffffffu, mbar_wait_cluster(bar_norm, 0, kWaitNs));
            if (!have_norm && lane == 0)
                report(p.status, SPARSE_ERR_TIMEOUT);
            // (3) p_j of the loaded rows, then the block maxima -> keys of CTA 0 (every
            // consumer warp reaches the barrier, whatever its wait gave)
            if (have_norm) {
                // four rows per pass, every load of a pass before its stores (one warp per
                // scheduler: the rows' exp2 chains overlap within the thread); heads past G
                // read head G-1's row and add an exact 0, so the body has no branch
                constexpr int HM = 8 * NT;
                float nm[HM], ni[HM];
                const float *rowh[HM];
#pragma unroll
                for (int h = 0; h < HM; ++h) {
                    nm[h] = h < G ? norm[2 * h] : INFINITY;
                    ni[h] = h < G ? norm[2 * h + 1] : 0.f;
                    rowh[h] = raw + min(h, G - 1) * p.rows_cta_max;
                }
                constexpr int kPass = 4, kStride = kConsumerWarps * 32;
                for (int i0 = tid; i0 < n_loc; i0 += kPass * kStride) {
                    float sum[kPass];
#pragma unroll
                    for (int q4 = 0; q4 < kPass; ++q4) {
                        const int i = min(i0 + q4 * kStride, n_loc - 1);
                        float acc = 0.f;
#pragma unroll
                        for (int h = 0; h < HM; ++h)
                            acc += ex2_approx(rowh[h][i] - nm[h]) * ni[h];
                        sum[q4] = acc;
                    }
#pragma unroll
                    for (int q4 = 0; q4 < kPass; ++q4) {
                        const int i = i0 + q4 * kStride;
                        if (i < n_loc)
                            prow[i] = sum[q4];   // prow aliases head 0's scores: row i is this thread's alone
                    }
                }
            }
            named_barrier_sync(2, kConsumerWarps * 32);
            if (have_norm) {
                // rows meeting block blk: [(64 blk - l) / s + 1, (64 blk + 63) / s] (32-bit; a
                // shift for a power-of-two stride)
                const bool pow2 = (s & (s - 1)) == 0;
                const int sh = __ffs(s) - 1;
                auto div_s = [&](int x) { return pow2 ? x >> sh : x / s; };
                for (int bb = b_lo + warp * 32; bb < b_hi; bb += kConsumerWarps * 32) {
                    const int blk = bb + lane;
                    const bool in = ok && blk < b_hi;
                    float best = 0.f;
                    if (in) {
                        const int x = kBlk * blk - l;
                        const int r0 = x < 0 ? 0 : div_s(x) + 1;
                        const int r1 = min(R - 1, div_s(kBlk * blk + kBlk - 1));
                        for (int j = r0; j <= r1; j += 4)   // four rows a step, clamped and masked
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float v = prow[min(j + c, r1) - j_lo];
                                best = fmaxf(best, j + c <= r1 ? v : 0.f);
                            }
                    }
                    if (in)
                        keys0[blk] = order_key(best);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(dsmem_addr(bar_scored, 0));
            if (rank == 0) {
                // CTA 0's consumers join its selector warp in the top-k
                const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(bar_scored, 0, kWaitNs));
                if (!got && lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                if (regs_topk) {
                    topk_cta_regs<kRouteKpt>(base_s + L.off_keys, nb, p.n_init, p.n_local, p.k_sel,
                                             base_s + L.off_hist, tid + 32, kRouteTopkThreads, 3, got,
                                             p.idx + static_cast<size_t>(unit) * p.k_tot, p.k_tot, p.count + unit,
                                             p.status);
                } else {
                    uint32_t prefix;
                    int need;
                    topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + L.off_hist,
                                       base_s + L.off_ctrl + 32, tid + 32, kRouteTopkThreads, 3, prefix, need);
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
            // the top-k with CTA 0's consumers (this warp is warp 0 of the group): keys in
            // registers and the list written by the group, or the radix threshold and the
            // list written by this warp
            uint32_t prefix = 0u;
            int need = 0;
            if (score && regs_topk) {
                topk_cta_regs<kRouteKpt>(base_s + L.off_keys, nb, p.n_init, p.n_local, p.k_sel, base_s + L.off_hist,
                                         lane, kRouteTopkThreads, 3, ready, p.idx + static_cast<size_t>(unit) * p.k_tot,
                                         p.k_tot, p.count + unit, p.status);
            } else {
                if (score)
                    topk_threshold_cta(base_s + L.off_keys, p.n_init, nb - p.n_local, p.k_sel, base_s + L.off_hist,
                                       base_s + L.off_ctrl + 32, lane, kRouteTopkThreads, 3, prefix, need);
                if (ready) {
                    topk_write_warp(base_s + L.off_keys, 0u, 0, nb, p.n_init, p.n_local,
                                    max(0, nb - p.n_local - p.n_init) <= p.k_sel, p.k_sel <= 0, prefix, need,
                                    p.idx + static_cast<size_t>(unit) * p.k_tot, p.k_tot, p.count + unit, p.status,
                                    lane);
                } else if (lane == 0) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                }
            }
        }
        cluster_wait();
    }
}

static_assert((kRouteTopkThreads / 32) * 256 <= kCoarseBins + kTopkList, "routing radix bins");

template <int NT>
int launch_route(const RouteParams &p, const CUtensorMap &km, int S, long long units, size_t smem, int device,
                 cudaStream_t stream)
{
    auto kern = nsa_route_kernel<NT>;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), static_cast<int>(smem), device,
                                       configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(units), 1);
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
                                            int cmp_stride, const int *seq_len, int B, int N_q, int H_q, int H_kv,
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
    if (B < 1 || N_q < 1 || H_kv < 1 || H_q < H_kv || H_q % H_kv != 0 || n_rows_cap < 1 || n_init < 0 ||
        n_local < 0 || k < 0)
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
    const long long units = pairs * N_q;
    if (units > 65535)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: B*H_kv*N_q=%lld > 65535", name, units);
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
    while (S < kMaxSplit && units * S * 2 <= dev.sm_count && n_blocks_cap / (S * 2) >= 16)
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
    p.N_q = N_q;
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
    return G <= 8 ? launch_route<1>(p, km, S, units, smem, dev.device, st)
                  : launch_route<2>(p, km, S, units, smem, dev.device, st);
}

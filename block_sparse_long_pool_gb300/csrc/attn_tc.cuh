// attn_tc.cuh -- split-KV attention of one unit (a decode pair, or a verification group
// of C queries x G heads) with both contractions on the 5th-generation tensor cores.
//
// Per 64-token block of the CTA's slice, with K and V in a stage of the TMA ring (two
// 64-dim boxes each, 128-byte swizzle):
//   S^T = K Q^T      tcgen05.mma M = 64 tokens, N = 16 rows (the G x C tile, zero rows
//                    past it), K = 128 dims; K-major A (the K tile) and B (the Q tile);
//                    f32 into one of two tensor-memory buffers
//   softmax          the 4 softmax warps read S^T (warp w: tokens 16w .. 16w+15, one per
//                    lane), mask, take the block's row maxima across the warps, and
//                    write P = exp2(s - m) in bf16 to shared memory (K-major, swizzled)
//   O^T += V^T P^T   M = 128 dims, N = 16 rows, K = 64 tokens; MN-major A (the V tile
//                    as stored), K-major B (P); f32 accumulator in tensor memory
// One thread of the MMA warp issues both products; the row max is updated lazily (O is
// rescaled in tensor memory only when a row's max grows by more than 2^8), so P <= 2^8.
// The CTA state is read from tensor memory once at the end and merged with the
// cluster's other CTAs as in the mma.sync kernels (pull merge).
#pragma once

#include "attn_core.cuh"

namespace {

constexpr int kTcWarps = kConsumerWarps + 2;   // 0-3 softmax, 4 TMA producer, 5 MMA issuer
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcN = 16;                       // MMA N: query rows of the tile
constexpr int kTcCols = 64;                    // tensor-memory columns: S [0, 32) (two buffers), O [32, 48)
constexpr int kTcColO = 32;
constexpr float kTcRescaleLog2 = 8.f;          // lazy rescale threshold (log2 units)
constexpr int kTcTileBytes = kTcN * 128;       // one 64-dim box of Q, or one P buffer: 16 rows x 128 B

// Shared memory (offsets from the 1024-byte aligned base): the ring, then the Q tile
// (two boxes), two P buffers, the barriers, control words, the cross-warp row
// reductions and the block list.  The union build's scratch uses the last ring stage:
// the ring is idle until the union exists.
constexpr int kTcOffQ = kStages * kStageBytes;
constexpr int kTcOffP = kTcOffQ + 2 * kTcTileBytes;
constexpr int kTcOffBars = kTcOffP + 2 * kTcTileBytes;
enum {
    kTcFull = 0,     // [kStages] K and V of a stage landed (TMA)
    kTcEmpty = 3,    // [kStages] the stage's products are done (tcgen05.commit)
    kTcSFull = 6,    // [2] S buffer written (commit)
    kTcSFree = 8,    // [2] S buffer read by the 4 softmax warps
    kTcPFull = 10,   // [2] P buffer written (and O rescaled) by the 4 softmax warps
    kTcPv = 12,      // [2] O += V^T P^T of a block done (commit); block k on barrier k & 1
    kTcQFull = 14,   // the Q tile is in shared memory
    kTcDrain = 15,   // every product the MMA warp issued is done
    kTcNumBars = 16
};
constexpr int kTcOffCtrl = kTcOffBars + 8 * kTcNumBars;   // int ctrl[16]; ctrl[15] = tensor-memory base
constexpr int kTcCtrlTmem = 15;
constexpr int kTcOffRed = kTcOffCtrl + 64;                 // f32 [2][4 warps][16 rows]
constexpr int kTcOffList = kTcOffRed + 2 * kConsumerWarps * kTcN * 4;
constexpr int kTcSmem = kTcOffList + 2 * kMaxUnion * 4 + 1024;
constexpr int kTcOffEnt = 2 * kStageBytes;
static_assert(kTcOffQ % 1024 == 0 && kTcOffP % 1024 == 0 && kTcTileBytes % 1024 == 0,
              "swizzled tiles start on 1024-byte atoms");
static_assert(kTcOffEnt + 3 * kMaxUnion * 4 <= kStages * kStageBytes, "the union scratch fits in the last stage");
static_assert(kMaxListCta <= kMaxUnion, "the decode slice fits the list words");
static_assert(2 * (kTcSmem + 1024) <= 233472, "two CTAs per SM");

// Maximum (or sum) over the warp of 16 values per lane, one row each: a transposed
// butterfly (8 + 4 + 2 + 1 + 1 shuffles); lane l returns row l >> 1's result.
template <bool MAX>
__device__ __forceinline__ float tc_row_reduce(const float (&x)[16], int lane)
{
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
    float t8[8], t4[4], t2[2];
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0, h4 = (lane & 4) != 0, h2 = (lane & 2) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float keep = h16 ? x[i + 8] : x[i], send = h16 ? x[i] : x[i + 8];
        t8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = h8 ? t8[i + 4] : t8[i], send = h8 ? t8[i] : t8[i + 4];
        t4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = h4 ? t4[i + 2] : t4[i], send = h4 ? t4[i] : t4[i + 2];
        t2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    const float keep = h2 ? t2[1] : t2[0], send = h2 ? t2[0] : t2[1];
    const float t1 = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    return op(t1, __shfl_xor_sync(0xffffffffu, t1, 1));
}

template <int NT, bool VERIFY>
__device__ __forceinline__ void attn_tc_cta(const CUtensorMap *kmap, const CUtensorMap *vmap, const AttnParams &p,
                                            int unit)
{
    constexpr int ROWS = 8 * NT;
    static_assert(ROWS <= kTcN, "the output rows fit the MMA tile");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    int *ctrl = reinterpret_cast<int *>(base + kTcOffCtrl);
    const uint32_t bars = base_s + kTcOffBars;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t S = gridDim.x;       // the cluster spans gridDim.x
    const uint32_t rank = blockIdx.x;   // == %cluster_ctarank
    if (tid == kConsumerWarps * 32) {
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
    // Programmatic dependent launch, as in attn_cluster_cta: with SPARSE_ATTN_BLOCKS_READY
    // only Q and the outputs wait for the kernel before this one.
    const bool early = (p.flags & SPARSE_ATTN_BLOCKS_READY) != 0u;
    if (!early)
        griddep_wait();

    if (tid == 0) {
        ctrl[kCtrlAbort] = 0;
        ctrl[kCtrlList] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars + 8 * (kTcFull + s), 1);
            mbar_init(bars + 8 * (kTcEmpty + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars + 8 * (kTcSFull + i), 1);
            mbar_init(bars + 8 * (kTcSFree + i), kConsumerWarps);
            mbar_init(bars + 8 * (kTcPFull + i), kConsumerWarps);
            mbar_init(bars + 8 * (kTcPv + i), 1);
        }
        mbar_init(bars + 8 * kTcQFull, kConsumerWarps);
        mbar_init(bars + 8 * kTcDrain, 1);
        fence_barrier_init();
    }
    if (warp == kConsumerWarps + 1)
        tc_alloc(base_s + kTcOffCtrl + 4 * kTcCtrlTmem, kTcCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(ctrl[kTcCtrlTmem]);

    // The slice: verification, a contiguous slice of the group's merged union (built
    // here by every thread); decode, entries [r * ceil(k_tot / S), ...) of the pair's
    // table, fetched with the count by the producer warp.
    int *ulist = reinterpret_cast<int *>(base + kTcOffList);
    uint32_t *umask = reinterpret_cast<uint32_t *>(ulist + kMaxUnion);
    int *lslot = ulist;
    int *llog = ulist + kMaxListCta;
    long long len = 0;
    int i0 = 0, my_n = 0;
    if (VERIFY) {
        len = p.seq_len[b];
        const int nb = len <= 0 ? 0 : static_cast<int>((len + kBlk - 1) / kBlk);
        int *ent = reinterpret_cast<int *>(base + kTcOffEnt);
        build_union<kTcThreads>(p, ulist, umask, ent, reinterpret_cast<uint32_t *>(ent + kMaxUnion),
                                ent + 2 * kMaxUnion, b, g, q0, nb, ctrl);
        __syncthreads();
        const int n_list = ctrl[kCtrlList];
        const int per = (n_list + static_cast<int>(S) - 1) / static_cast<int>(S);
        i0 = min(n_list, static_cast<int>(rank) * per);
        my_n = min(n_list, i0 + per) - i0;
        if (rank == 0 && tid == 0 && p.blocks_loaded != nullptr)
            atomicAdd(reinterpret_cast<unsigned long long *>(p.blocks_loaded),
                      static_cast<unsigned long long>(n_list));
    } else {
        len = p.seq_len[b];
    }
    // the running row maxima (log2 units), the same in every softmax thread
    float m[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        m[r] = -INFINITY;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ TMA producer
        if (!VERIFY) {
            const int per = (p.k_tot + static_cast<int>(S) - 1) / static_cast<int>(S);
            i0 = min(p.k_tot, static_cast<int>(rank) * per);
            my_n = producer_fetch_slice(p, pair, i0, min(p.k_tot, i0 + per) - i0, lslot, llog, ctrl, lane);
            named_barrier_arrive(1, kTcThreads);   // the slice and its length are in shared memory
        }
        if (lane == 0 && my_n > 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int it = 0; it < my_n; ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                if (use > 0 && !mbar_wait(bars + 8 * (kTcEmpty + s), (use - 1) & 1, kWaitNs)) {
                    report(p.status, SPARSE_ERR_TIMEOUT);
                    break;
                }
                const int slot = VERIFY ? ulist[i0 + it] : lslot[it];
                // an invalid slot loads an out-of-range box: zeros, never a fault
                const int row = slot >= 0 ? slot * kBlk : static_cast<int>(min(p.pair_stride, (long long)INT_MAX - kBlk));
                const uint32_t dst = base_s + s * kStageBytes;
                const uint32_t full = bars + 8 * (kTcFull + s);
                mbar_arrive_expect_tx(full, kStageBytes);
                tma_load_3d(dst, kmap, full, 0, row, pair, pol);
                tma_load_3d(dst + kHalfBytes, kmap, full, 64, row, pair, pol);
                tma_load_3d(dst + kTileBytes, vmap, full, 0, row, pair, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, vmap, full, 64, row, pair, pol);
                issued = it + 1;
            }
            // no copy is still in flight when the CTA leaves
            for (int it = max(0, issued - kStages); it < issued; ++it)
                mbar_wait(bars + 8 * (kTcFull + it % kStages), (it / kStages) & 1, kWaitNs);
        }
    } else if (warp == kConsumerWarps + 1) {
        // ------------------------------------------------------------ MMA issuer
        if (!VERIFY) {
            named_barrier_sync(1, kTcThreads);
            my_n = ctrl[kCtrlList];
        }
        if (lane == 0 && my_n > 0) {
            // Issue whichever product is ready, the pending O^T += V^T P^T first (it frees
            // a ring stage): S^T of block ns once its stage has landed and its S buffer
            // has been read back (block ns - 2); O of block npv once its P is written.
            constexpr uint32_t idS = tc_idesc_bf16(64, kTcN, 0, 0);    // K-major K tile, K-major Q
            constexpr uint32_t idO = tc_idesc_bf16(128, kTcN, 1, 0);   // MN-major V tile, K-major P
            const uint32_t q_s = base_s + kTcOffQ, p_s = base_s + kTcOffP;
            bool ok = mbar_wait(bars + 8 * kTcQFull, 0, kWaitNs);
            int ns = 0, npv = 0;
            uint64_t t_idle = 0;
            for (uint32_t spin = 0; ok && npv < my_n; ++spin) {
                if (npv < ns && mbar_test(bars + 8 * (kTcPFull + (npv & 1)), (npv >> 1) & 1)) {
                    const int s = npv % kStages, pb = npv & 1;
                    tc_fence_after();
                    const uint32_t v_s = base_s + s * kStageBytes + kTileBytes;
#pragma unroll
                    for (int j = 0; j < 4; ++j)   // 16 tokens a step: two 8-token atoms of the V tile
                        tc_mma(tmem + kTcColO, tc_sdesc(v_s + j * 2048, kHalfBytes, 1024),
                               tc_sdesc(p_s + pb * kTcTileBytes + j * 32, 16, 1024), idO, npv > 0 || j > 0);
                    tc_commit(bars + 8 * (kTcEmpty + s));
                    tc_commit(bars + 8 * (kTcPv + pb));
                    ++npv;
                    t_idle = 0;
                } else if (ns < my_n && mbar_test(bars + 8 * (kTcFull + ns % kStages), (ns / kStages) & 1) &&
                           (ns < 2 || mbar_test(bars + 8 * (kTcSFree + (ns & 1)), ((ns - 2) >> 1) & 1))) {
                    const int s = ns % kStages, sb = ns & 1;
                    tc_fence_after();
                    const uint32_t k_s = base_s + s * kStageBytes;
#pragma unroll
                    for (int j = 0; j < 8; ++j)   // 16 dims a step; steps 4-7 in the second box
                        tc_mma(tmem + sb * kTcN, tc_sdesc(k_s + (j >> 2) * kHalfBytes + (j & 3) * 32, 16, 1024),
                               tc_sdesc(q_s + (j >> 2) * kTcTileBytes + (j & 3) * 32, 16, 1024), idS, j > 0);
                    tc_commit(bars + 8 * (kTcSFull + sb));
                    ++ns;
                    t_idle = 0;
                } else if ((spin & 63u) == 63u) {
                    const uint64_t now = globaltimer();
                    if (t_idle == 0)
                        t_idle = now;
                    else if (now - t_idle > kWaitNs)
                        ok = false;   // nothing became ready for kWaitNs
                }
            }
            if (!ok)
                report(p.status, SPARSE_ERR_TIMEOUT);
            // every product issued is complete before the tensor memory is read or freed
            tc_commit(bars + 8 * kTcDrain);
            mbar_wait(bars + 8 * kTcDrain, 0, kWaitNs);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        if (early)
            griddep_wait();   // Q may be written by the kernel before this one
        // the Q tile, 128-byte swizzled in two 64-dim boxes; rows past the tile are zero
        for (int i = tid; i < kTcN * 16; i += kConsumerWarps * 32) {
            const int r = i >> 4, c = i & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows_valid) {
                const uint16_t *qrow;
                if (VERIFY) {
                    const int qq = q0 + r / p.G, hh = r % p.G;
                    qrow = p.Q + ((static_cast<size_t>(b) * p.N_q + qq) * p.H_q + g * p.G + hh) * kD;
                } else {
                    qrow = p.Q + (static_cast<size_t>(b) * p.H_q + g * p.G + r) * kD;
                }
                v = *reinterpret_cast<const uint4 *>(qrow + c * 8);
            }
            *reinterpret_cast<uint4 *>(base + kTcOffQ + (c >> 3) * kTcTileBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bars + 8 * kTcQFull);
        if (!VERIFY) {
            named_barrier_sync(1, kTcThreads);
            my_n = ctrl[kCtrlList];
        }
        // the query of each tile row (verification masks rows by their query's set)
        int rq[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            rq[r] = VERIFY && r < rows_valid ? r / p.G : 0;
        const uint32_t row_all = rows_valid >= 16 ? 0xffffu : ((1u << rows_valid) - 1u);
        float l[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            l[r] = 0.f;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float *red = reinterpret_cast<float *>(base + kTcOffRed);
        bool ok = true, warp_ok = true;
        for (int it = 0; it < my_n; ++it) {
            const int sb = it & 1;
            // S^T of this block, and O done for block it - 2 (whose P buffer this block
            // reuses); a failed wait of this warp's earlier rescale counts too
            const bool w_ok = __all_sync(
                0xffffffffu, warp_ok && mbar_wait(bars + 8 * (kTcSFull + sb), (it >> 1) & 1, kWaitNs) &&
                                 (it < 2 || mbar_wait(bars + 8 * (kTcPv + (it & 1)), ((it - 2) >> 1) & 1, kWaitNs)));
            float v[16];
            if (w_ok) {
                tc_fence_after();
                tc_ld16(tmem + lane_base + sb * kTcN, v);
            } else {
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    v[r] = 0.f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bars + 8 * (kTcSFree + sb));
            int logical;
            uint32_t rowmask = row_all;
            if (VERIFY) {
                logical = ulist[i0 + it];
                const uint32_t qmask = umask[i0 + it];
                rowmask = 0u;
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    rowmask |= ((qmask >> rq[r]) & 1u) << r;
                rowmask &= row_all;
            } else {
                logical = llog[it];
            }
            const long long tok = static_cast<long long>(logical) * kBlk + warp * 16 + lane;
            const bool tok_ok = w_ok && lane < 16 && logical >= 0 && tok < len;
            float s[16];
#pragma unroll
            for (int r = 0; r < 16; ++r)
                s[r] = tok_ok && ((rowmask >> r) & 1u) ? v[r] * p.scale_log2 : -INFINITY;
            // the block's row maxima over the 4 warps (and every warp's verdict on its waits)
            float *rb = red + (it & 1) * (kConsumerWarps * kTcN);
            const float wmax = tc_row_reduce<true>(s, lane);
            if ((lane & 1) == 0)
                rb[warp * kTcN + (lane >> 1)] = wmax;
            if (!named_barrier_and(3, kConsumerWarps * 32, w_ok)) {
                ok = false;
                break;
            }
            float bm[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float4 x = *reinterpret_cast<const float4 *>(rb + 4 * q4);
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) {
                    const float4 y = *reinterpret_cast<const float4 *>(rb + w * kTcN + 4 * q4);
                    x = make_float4(fmaxf(x.x, y.x), fmaxf(x.y, y.y), fmaxf(x.z, y.z), fmaxf(x.w, y.w));
                }
                bm[4 * q4 + 0] = x.x;
                bm[4 * q4 + 1] = x.y;
                bm[4 * q4 + 2] = x.z;
                bm[4 * q4 + 3] = x.w;
            }
            // lazy max update (the same values, hence the same decision, in every thread)
            float alpha[16];
            bool rescale = false;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float nm = m[r];
                if (bm[r] != -INFINITY) {
                    if (m[r] == -INFINITY) {
                        nm = bm[r];
                    } else if (bm[r] > m[r] + kTcRescaleLog2) {
                        nm = bm[r];
                        rescale = true;
                    }
                }
                alpha[r] = (m[r] == -INFINITY || nm == m[r]) ? 1.f : exp2f(m[r] - nm);
                m[r] = nm;
            }
            if (rescale && it > 0) {
                // O complete up to block it - 1, then scaled in place (this warp's 32 dims);
                // a failed wait stops the loop at the next block's vote
                warp_ok = __all_sync(0xffffffffu, mbar_wait(bars + 8 * (kTcPv + ((it - 1) & 1)),
                                                            ((it - 1) >> 1) & 1, kWaitNs));
                if (warp_ok) {
                    float o[16];
                    tc_fence_after();
                    tc_ld16(tmem + lane_base + kTcColO, o);
#pragma unroll
                    for (int r = 0; r < 16; ++r)
                        o[r] *= alpha[r];
                    tc_st16(tmem + lane_base + kTcColO, o);
                }
            }
            // P of this block into buffer it & 1 (free: block it - 2's product is done)
            uint8_t *pbuf = base + kTcOffP + (it & 1) * kTcTileBytes;
            const int t = warp * 16 + lane;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float pr = s[r] == -INFINITY ? 0.f : exp2f(s[r] - m[r]);
                l[r] = l[r] * alpha[r] + pr;
                if (lane < 16) {
                    const __nv_bfloat16 pb = __float2bfloat16_rn(pr);
                    *reinterpret_cast<__nv_bfloat16 *>(pbuf + r * 128 + ((((t >> 3) ^ (r & 7))) << 4) + (t & 7) * 2) = pb;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bars + 8 * (kTcPFull + (it & 1)));
        }
        if (!ok && lane == 0)
            report(p.status, SPARSE_ERR_TIMEOUT);
        // the CTA's row sums: over the warp's lanes, then (below) over the 4 warps, in
        // the reduction buffer the last block did not use (others may still read that one)
        const float wsum = tc_row_reduce<false>(l, lane);
        if ((lane & 1) == 0)
            red[(my_n & 1) * (kConsumerWarps * kTcN) + warp * kTcN + (lane >> 1)] = wsum;
    }

    // Every product is done (the MMA warp drained them) and every copy has landed: the
    // ring is free for the merge scratch and O can be read from tensor memory.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float *co = merge_cta_state<NT>(base);
    if (warp < kConsumerWarps) {
        float o[16];
        if (my_n > 0) {
            tc_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kTcColO, o);
        } else {
#pragma unroll
            for (int r = 0; r < 16; ++r)
                o[r] = 0.f;
        }
        const int d = warp * 32 + lane;
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
            co[r * kD + d] = o[r];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kConsumerWarps + 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTcCols);
    }
    if (tid < ROWS) {
        const float *rs = reinterpret_cast<const float *>(base + kTcOffRed) + (my_n & 1) * (kConsumerWarps * kTcN);
        float *cl = co + ROWS * kD + ROWS;
        cl[tid] = rs[tid] + rs[kTcN + tid] + rs[2 * kTcN + tid] + rs[3 * kTcN + tid];
    }
    if (tid == 0) {   // a softmax thread: its m is the CTA's
        float *cm = co + ROWS * kD;
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
            cm[r] = m[r];
    }
    // ---------------------------------------------------------------- merge
    // The next kernel on the stream may be scheduled from here on.
    griddep_launch_dependents();
    WarpState<NT> unused;
    cluster_merge_write<NT, VERIFY>(unused, base, ctrl[kCtrlAbort] != 0, p, b, g, q0, rows_valid, rank, S,
                                    kTcThreads, base_s + kTcOffCtrl, false, false, true);
}

}  // namespace

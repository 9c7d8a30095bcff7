// prefill.cu -- the Forecast selection of every prefill position.
//
// SparDA notes §4.3 eq.(16): at prefill the Forecast indexer scores every position's
// Forecast vector (one per GQA group) against the compressed keys, H_kv * T * N_b * d
// multiply-adds per layer, then each position takes its own top-k (eq.(6), Alg.1 step 2)
// among the blocks it can see: position t sees the blocks holding tokens 0..t, and its
// local blocks end at the block holding t.
//
// GB300 design.  The scores of a tile of RQ positions against 64 compressed keys are a
// dense contraction (RQ x 64 x 128), so they run on the tensor cores: S = F Khat^T with
// F (bf16, exact) as the A operand and the fp32 compressed keys split into three bf16
// terms (hi + mid + lo carries all 24 bits of an fp32 mantissa), three mma per
// fragment, fp32 accumulation: the products are exact and the sums are those of an fp32
// dot product up to the order of addition.
//   * One CTA per (pair, RQ positions), RQ = 64, 32 or 16 positions as the pair's
//     compressed keys grow (their order keys for all RQ rows stay in shared memory).
//     All RQ positions lie in one 64-token block, so they share their candidate blocks.
//   * Warp 4 streams the candidate keys in tiles of 64 rows (one 1-D bulk copy per
//     row into rows padded to 528 bytes, so the fragment loads hit distinct banks),
//     two ring stages.
//   * Warps 0-7: warp w takes positions [16 (w % PG), +16) and a share of each tile's
//     64 keys (PG = RQ / 16 position groups); the scores become order keys in shared
//     memory.  Then each warp selects rows: the row's keys in registers, a binary
//     search over their bits for the k-th largest (stopping once every remaining key is
//     needed), and the list written in block order.
#include <limits.h>

#include "common.cuh"
#include "select_core.cuh"

namespace {

using namespace sp;

constexpr int kPfConsumerWarps = 8;
constexpr int kPfThreads = (kPfConsumerWarps + 1) * 32;
constexpr int kPfStages = 2;
constexpr int kPfRowBytes = kD * 4 + 16;                 // a padded fp32 key row
constexpr int kPfFRowBytes = kD * 2 + 16;                // a padded bf16 Forecast row
constexpr uint64_t kPfWaitNs = 2000000000ull;

struct PrefillParams {
    const uint16_t *F;       // [pairs][T_cap][128]
    const float *ktil;       // [pairs][N_cap][128]
    const int *seq_len;      // [B]
    int *idx;                // [pairs][T_cap][k_tot]
    int *count;              // [pairs][T_cap]
    int *status;
    long long T_cap;
    int H_kv;
    int N_cap;
    int key_stride;          // order keys per row in shared memory (= 8 mod 32)
    int n_init, n_local, k, k_tot;
};

struct PfLayout {
    int off_bars, off_f, off_keys, total;
};

__host__ __device__ inline PfLayout pf_layout(int RQ, int TK, int key_stride)
{
    PfLayout l;
    l.off_bars = kPfStages * TK * kPfRowBytes;                  // ring; then full[2], empty[2]
    l.off_f = l.off_bars + 64;                                  // [RQ][kPfFRowBytes]
    l.off_keys = l.off_f + RQ * kPfFRowBytes;                   // [RQ][key_stride] u32
    l.total = l.off_keys + RQ * key_stride * 4;
    return l;
}

// x = hi + mid + lo with each term a bf16 (together all 24 mantissa bits of x).
__device__ __forceinline__ void split3(float x, float &hi, float &mid, float &lo)
{
    hi = __bfloat162float(__float2bfloat16_rn(x));
    const float r = x - hi;
    mid = __bfloat162float(__float2bfloat16_rn(r));
    lo = r - mid;
}

__device__ __forceinline__ void split3_pack(float2 v, uint32_t &hi, uint32_t &mid, uint32_t &lo)
{
    float h0, m0, l0, h1, m1, l1;
    split3(v.x, h0, m0, l0);
    split3(v.y, h1, m1, l1);
    hi = pack_bf16x2(h0, h1);
    mid = pack_bf16x2(m0, m1);
    lo = pack_bf16x2(l0, l1);
}

// RQ positions per CTA; TK compressed keys per ring stage; KPL: candidate keys per
// lane in the top-k (32 * KPL >= N_cap).
template <int RQ, int TK, int KPL>
__global__ void __launch_bounds__(kPfThreads, KPL <= 32 ? 2 : 1) prefill_select_kernel(const __grid_constant__ PrefillParams p)
{
    constexpr int PG = RQ / 16;                       // position groups of 16
    constexpr int BQ = kPfConsumerWarps / PG;         // key groups of a tile
    constexpr int NTT = TK / 8;                       // n-tiles (8 keys) of a tile
    constexpr int NTW = NTT >= BQ ? NTT / BQ : 1;     // n-tiles per warp (warps with bq >= NTT idle)
    constexpr int kStageBytes = TK * kPfRowBytes;
    griddep_wait();   // every input may be written by the kernel before this one
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 127u) & ~127u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    const PfLayout L = pf_layout(RQ, TK, p.key_stride);
    const uint32_t bar_full = base_s + L.off_bars;
    const uint32_t bar_empty = bar_full + 8 * kPfStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int pair = static_cast<int>(blockIdx.y);
    const int b = pair / p.H_kv;
    const long long t0 = static_cast<long long>(blockIdx.x) * RQ;
    long long len = p.seq_len[b];
    if (len > p.T_cap) {   // positions past the buffers are not read (reported by the first tile)
        if (blockIdx.x == 0 && threadIdx.x == 0)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        len = p.T_cap;
    }
    if (t0 >= len)
        return;   // no position of this tile is present
    const int rows_valid = static_cast<int>(len - t0 < RQ ? len - t0 : RQ);
    long long nb_ll = t0 / kBlk + 1;   // every position of the tile lies in block t0 / 64
    const bool len_bad = nb_ll > p.N_cap;
    nb_ll = nb_ll < p.N_cap ? nb_ll : p.N_cap;
    const int nb = static_cast<int>(nb_ll);
    const int c_lo = p.n_init, c_hi = nb - p.n_local;
    const int n_cand = max(0, c_hi - c_lo);
    const bool take_all = n_cand <= p.k, take_none = p.k <= 0;
    const bool score = !take_all && !take_none;
    const int n_tiles = score ? (n_cand + TK - 1) / TK : 0;

    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kPfConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == kPfConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && len_bad)
            report(p.status, SPARSE_ERR_BAD_INDEX);
        const float *kt = p.ktil + (static_cast<size_t>(pair) * p.N_cap + c_lo) * kD;
        const uint64_t pol = policy_evict_last();   // re-read by every tile of the pair
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % kPfStages;
            const int use = t / kPfStages;
            bool ok = true;
            if (lane == 0 && use > 0)
                ok = mbar_wait(bar_empty + 8 * s, (use - 1) & 1, kPfWaitNs);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                break;
            }
            const int rows = min(TK, n_cand - t * TK);
            if (lane == 0)
                mbar_arrive_expect_tx(bar_full + 8 * s, static_cast<uint32_t>(rows * kD * 4));
            __syncwarp();
            for (int r = lane; r < rows; r += 32)
                bulk_load(base_s + s * kStageBytes + r * kPfRowBytes, kt + static_cast<size_t>(t * TK + r) * kD,
                          kD * 4, bar_full + 8 * s, pol);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int pg = warp % PG, bq = warp / PG;
        const int g8 = lane >> 2, t4 = lane & 3;
        // the tile's Forecast rows (zeros past the length) into padded shared rows
        for (int i = tid; i < RQ * 16; i += kPfConsumerWarps * 32) {
            const int r = i >> 4, c = i & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows_valid)
                v = *reinterpret_cast<const uint4 *>(p.F + (static_cast<size_t>(pair) * p.T_cap + t0 + r) * kD + c * 8);
            *reinterpret_cast<uint4 *>(base + L.off_f + r * kPfFRowBytes + c * 16) = v;
        }
        named_barrier_sync(2, kPfConsumerWarps * 32);
        uint32_t afr[8][4];
        {
            const int row = pg * 16 + (lane & 15);
            const uint32_t a0 = base_s + L.off_f + row * kPfFRowBytes + (lane >> 4) * 16;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                ldsm_x4(a0 + ks * 32, afr[ks]);
        }
        const uint32_t keys_s = base_s + L.off_keys;
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % kPfStages;
            const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (t / kPfStages) & 1, kPfWaitNs));
            if (!landed) {
                if (lane == 0)
                    report(p.status, SPARSE_ERR_TIMEOUT);
                break;
            }
            const uint8_t *stage = base + s * kStageBytes;
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                if (bq >= NTT)
                    break;
                const int kr = bq * (8 * NTW) + nt * 8 + g8;   // key row within the tile
                const float *krow = reinterpret_cast<const float *>(stage + kr * kPfRowBytes);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const float2 lo2 = *reinterpret_cast<const float2 *>(krow + ks * 16 + 2 * t4);
                    const float2 hi2 = *reinterpret_cast<const float2 *>(krow + ks * 16 + 2 * t4 + 8);
                    uint32_t b0h, b0m, b0l, b1h, b1m, b1l;
                    split3_pack(lo2, b0h, b0m, b0l);
                    split3_pack(hi2, b1h, b1m, b1l);
                    mma_bf16_16816(acc, afr[ks], b0l, b1l);
                    mma_bf16_16816(acc, afr[ks], b0m, b1m);
                    mma_bf16_16816(acc, afr[ks], b0h, b1h);
                }
                // acc[i]: position pg*16 + g8 + 8 (i >> 1), key 8 nt + 2 t4 + (i & 1) of the share
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = pg * 16 + g8 + (i >> 1) * 8;
                    const int j = c_lo + t * TK + bq * (8 * NTW) + nt * 8 + 2 * t4 + (i & 1);
                    if (row < rows_valid && j < c_hi)
                        sts_u32(keys_s + 4 * (row * p.key_stride + j), order_key(acc[i]));
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }
        named_barrier_sync(2, kPfConsumerWarps * 32);   // every order key is in place
        for (int r = warp; r < rows_valid; r += kPfConsumerWarps) {
            const uint32_t row_keys = keys_s + 4 * r * p.key_stride;
            const size_t at = static_cast<size_t>(pair) * p.T_cap + t0 + r;
            int *row_out = p.idx + at * p.k_tot;
            if (score) {
                // registers for the candidates this tile has (they grow with the position)
                if (KPL >= 16 && n_cand <= 8 * KPL)
                    topk_range_regs<(KPL >= 16 ? KPL / 4 : KPL)>(row_keys, nb, p.n_init, p.n_local, p.k, row_out,
                                                                 p.k_tot, p.count + at, p.status, lane);
                else if (KPL >= 8 && n_cand <= 16 * KPL)
                    topk_range_regs<(KPL >= 8 ? KPL / 2 : KPL)>(row_keys, nb, p.n_init, p.n_local, p.k, row_out,
                                                                p.k_tot, p.count + at, p.status, lane);
                else
                    topk_range_regs<KPL>(row_keys, nb, p.n_init, p.n_local, p.k, row_out, p.k_tot, p.count + at,
                                         p.status, lane);
            } else {
                topk_write_warp(row_keys, 0u, 0, nb, p.n_init, p.n_local, take_all, take_none, 0u, 0, row_out,
                                p.k_tot, p.count + at, p.status, lane);
            }
        }
    }
}

template <int RQ, int TK, int KPL>
int launch_prefill(const PrefillParams &p, long long pairs, int device, cudaStream_t stream)
{
    auto kern = prefill_select_kernel<RQ, TK, KPL>;
    const PfLayout L = pf_layout(RQ, TK, p.key_stride);
    const int smem = L.total + 128;
    static int configured[64];
    int rc = sp_host::configure_kernel(reinterpret_cast<const void *>(kern), smem, device, configured);
    if (rc != SPARSE_OK)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((p.T_cap + RQ - 1) / RQ), static_cast<unsigned>(pairs), 1);
    cfg.blockDim = dim3(kPfThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PrefillParams prm = p;
    void *args[] = {&prm};
    return sp_host::cuda_status(cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args),
                                "sparse_prefill_select launch");
}

}  // namespace

extern "C" SPARSE_API int sparse_prefill_select(const uint16_t *F, long long T_cap, const float *ktil, int N_cap,
                                                const int *seq_len, int B, int H_kv, int n_init, int n_local, int k,
                                                int *idx_out, int *count_out, int k_tot, int *status, void *stream)
{
    using sp_host::aligned16;
    using sp_host::fail;
    const char *name = "sparse_prefill_select";
    if (!F || !ktil || !seq_len || !idx_out || !count_out)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(F) || !aligned16(ktil))
        return fail(SPARSE_ERR_INVALID_ARG, "%s: F and ktil must be 16-byte aligned", name);
    if (B < 1 || H_kv < 1 || T_cap < 1 || N_cap < 1 || n_init < 0 || n_local < 1 || k < 0)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: bad size (n_local must be >= 1: the block of a position is local)",
                    name);
    if (static_cast<long long>(n_init) + n_local + k > k_tot)
        return fail(SPARSE_ERR_INVALID_ARG, "%s: k_tot=%d < n_init+n_local+k", name, k_tot);
    if (N_cap > 2048)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: N_cap=%d > 2048 compressed keys (131072 tokens)", name, N_cap);
    const long long pairs = static_cast<long long>(B) * H_kv;
    if (pairs > 65535 || T_cap > (1LL << 31) * 16)
        return fail(SPARSE_ERR_UNSUPPORTED, "%s: too many pairs or positions", name);
    sp_host::DeviceInfo dev;
    int rc = sp_host::device_info(&dev);
    if (rc != SPARSE_OK)
        return rc;
    PrefillParams p = {};
    p.F = F;
    p.ktil = ktil;
    p.seq_len = seq_len;
    p.idx = idx_out;
    p.count = count_out;
    p.status = status;
    p.T_cap = T_cap;
    p.H_kv = H_kv;
    p.N_cap = N_cap;
    p.key_stride = (N_cap + 23) / 32 * 32 + 8;   // >= N_cap, = 8 mod 32
    p.n_init = n_init;
    p.n_local = n_local;
    p.k = k;
    p.k_tot = k_tot;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // two CTAs per SM up to 1024 keys (the order keys of a CTA's rows: <= 66 KB)
    if (N_cap <= 512)
        return launch_prefill<32, 32, 16>(p, pairs, dev.device, st);
    if (N_cap <= 1024)
        return launch_prefill<16, 32, 32>(p, pairs, dev.device, st);
    return launch_prefill<16, 32, 64>(p, pairs, dev.device, st);
}

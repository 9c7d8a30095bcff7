// select_layout.cuh -- the thread counts and shared-memory layout that the Forecast
// selection kernel and the multi-head selector share (both stream compressed-key
// slices through the attention ring and gather order keys in CTA 0).
#pragma once

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
static_assert(kOffList % 16 == 0, "the coarse histogram takes 16-byte reads");
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

// The slice [i0, i0 + cap) of the k_tot-long block list that CTA `rank` of a fused layer
// attends over.  With the group top-k (`cta0_free`: CTA 0's consumer warps take the next
// layer's top-k first) CTA 0 attends over nothing and the other S - 1 CTAs share the
// list, the first k_tot % (S - 1) of them one block more; otherwise CTA 0 takes what is
// left of k_tot after the other S - 1 take ceil(k_tot / S) each.
__host__ __device__ inline void fused_slice(int k_tot, int S, int rank, bool cta0_free, int *i0, int *cap)
{
    if (cta0_free && S > 1) {
        if (rank == 0) {
            *i0 = 0;
            *cap = 0;
            return;
        }
        const int n = S - 1, r = rank - 1, base = k_tot / n, rem = k_tot % n;
        *i0 = r * base + (r < rem ? r : rem);
        *cap = base + (r < rem ? 1 : 0);
        return;
    }
    // CTA 0 (the merge leader, whose selector warp shares its SM time) takes the short
    // slice: entries [0, k_tot - (S - 1) * per), then the others ceil(k_tot / S) each
    const int per = (k_tot + S - 1) / S;
    const int cap0 = k_tot - (S - 1) * per > 0 ? k_tot - (S - 1) * per : 0;
    if (rank == 0) {
        *i0 = 0;
        *cap = cap0;
        return;
    }
    const int a = cap0 + (rank - 1) * per;
    *i0 = a < k_tot ? a : k_tot;
    *cap = (*i0 + per < k_tot ? *i0 + per : k_tot) - *i0;
}

// The longest slice either way, for a kernel that may free CTA 0 (`group`); the shared
// memory layout is sized for it.
__host__ __device__ inline int fused_slice_max(int k_tot, int S, bool group)
{
    const int per = (k_tot + S - 1) / S;
    if (!group || S < 2)
        return per;
    const int per1 = (k_tot + S - 2) / (S - 1);
    return per1 > per ? per1 : per;
}

// The group top-k of CTA 0 (topk_forecast_cta): its 4 consumer warps and the selector
// warp, on named barrier 2, with up to kSelKPT candidates per thread (2720 in all), its
// scratch over the coarse histogram and the threshold list.
constexpr int kSelThreads = (kConsumerWarps + 1) * 32;
constexpr int kSelKPT = 17;
constexpr int kSelBar = 2;
static_assert(topk_forecast_scratch_words(kSelThreads / 32) * 4 <= fused_off_slice() - fused_off_hist(),
              "the group top-k's scratch fits over the histogram and the list");

}  // namespace

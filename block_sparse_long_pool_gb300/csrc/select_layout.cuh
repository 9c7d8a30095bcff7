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

// The group top-k of CTA 0 (topk_forecast_cta): its 4 consumer warps and the selector
// warp, on named barrier 2, with up to kSelKPT candidates per thread (2720 in all), its
// scratch over the coarse histogram and the threshold list.
constexpr int kSelThreads = (kConsumerWarps + 1) * 32;
constexpr int kSelKPT = 17;
constexpr int kSelBar = 2;
static_assert(topk_forecast_scratch_words(kSelThreads / 32) * 4 <= fused_off_slice() - fused_off_hist(),
              "the group top-k's scratch fits over the histogram and the list");

}  // namespace

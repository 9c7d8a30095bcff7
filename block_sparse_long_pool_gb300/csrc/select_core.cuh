// select_core.cuh -- exact top-k of order keys in shared memory, shared by the Forecast
// selection (decode), the multi-head selector, the NSA routing and the prefill selection.
//
// Keys are order_key(score): larger score -> larger key, equal scores -> equal keys.
// The top-k takes the k largest keys of the candidates [n_init, nb - n_local), equal
// keys in block order (the lower block first), and writes B_init, the selected
// candidates and B_local in ascending block order (SparDA notes eq.(6), Alg.1 step 2).
#pragma once

#include "common.cuh"

namespace {

using namespace sp;

constexpr int kTopkList = 512;                                    // keys gathered in the threshold bin
constexpr int kCoarseShift = 22;                                  // coarse bin = key >> 22
constexpr int kCoarseBins = 1 << (32 - kCoarseShift);             // 1024

// Histogram of byte digit (key >> shift) & 255 over the keys whose bits above the digit
// equal `prefix` (under `pmask`), by one warp: keys[i] for i in [lo, hi), or
// keys[list[i]] when list_s is non-zero.  Lanes holding the same digit add once
// (warp-aggregated shared-memory atomics).  All arrays are shared-space addresses.
__device__ __forceinline__ void warp_digit_hist(uint32_t keys_s, uint32_t list_s, int lo, int hi, uint32_t pmask,
                                                uint32_t prefix, int shift, uint32_t hist_s, int lane)
{
    for (int d = lane; d < 256; d += 32)
        sts_u32(hist_s + 4 * d, 0u);
    __syncwarp();
    for (int ib = lo; ib < hi; ib += 32) {
        const int i = ib + lane;
        uint32_t digit = 0xFFFFFFFFu;
        if (i < hi) {
            const uint32_t j = list_s != 0u ? lds_u32(list_s + 4 * i) : static_cast<uint32_t>(i);
            const uint32_t key = lds_u32(keys_s + 4 * j);
            if ((key & pmask) == prefix)
                digit = (key >> shift) & 255u;
        }
        const uint32_t same = __match_any_sync(0xffffffffu, digit);
        if (digit != 0xFFFFFFFFu && lane == __ffs(same) - 1)
            asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(hist_s + 4 * digit), "r"(__popc(same)) : "memory");
    }
    __syncwarp();
}

// From a digit histogram, the digit that holds the need-th largest key (counting from
// the top digit) and the number of keys still needed within it.
__device__ __forceinline__ void warp_pick_digit(uint32_t hist_s, int &need, uint32_t &digit, int lane)
{
    // lane l holds digits 255 - 8l - i (i = 0..7): lanes run from the top digit down
    int c[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c[i] = static_cast<int>(lds_u32(hist_s + 4 * (255 - 8 * lane - i)));
        sum += c[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    const int excl = incl - sum;
    int dsel = -1, need_new = 0;
    if (excl < need && need <= incl) {
        int acc = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (dsel < 0 && acc + c[i] >= need) {
                dsel = 255 - 8 * lane - i;
                need_new = need - acc;
            }
            acc += c[i];
        }
    }
    const unsigned m = __ballot_sync(0xffffffffu, dsel >= 0);
    const int src = m != 0u ? __ffs(m) - 1 : 0;
    dsel = __shfl_sync(0xffffffffu, dsel, src);
    need_new = __shfl_sync(0xffffffffu, need_new, src);
    if (m == 0u) {   // cannot happen with 1 <= need <= keys counted; keep the state sane
        dsel = 0;
        need_new = need;
    }
    digit = static_cast<uint32_t>(dsel);
    need = need_new;
}

// B_init (blocks [0, min(n_init, nb))) at the head of a row; returns how many.  One warp.
__device__ __forceinline__ int write_init_blocks(int nb, int n_init, int *out, int k_tot, bool &overflow, int lane)
{
    const int n_i = min(n_init, nb);
    for (int j = lane; j < n_i; j += 32) {
        if (j < k_tot)
            out[j] = j;
        else
            overflow = true;
    }
    return n_i;
}

// B_local (the last n_local blocks, after B_init) from position pos0, -1 in the rest of
// the row, and the count.  One warp.
__device__ __forceinline__ void write_local_and_close(int nb, int n_init, int n_local, int pos0, int *out, int k_tot,
                                                      int *count_out, int *status, bool overflow, int lane)
{
    const int l0 = max(nb - n_local, min(n_init, nb));
    for (int j = l0 + lane; j < nb; j += 32) {
        const int pos = pos0 + (j - l0);
        if (pos < k_tot)
            out[pos] = j;
        else
            overflow = true;
    }
    pos0 += max(0, nb - l0);
    if (__any_sync(0xffffffffu, overflow) && lane == 0)
        report(status, SPARSE_ERR_BAD_INDEX);
    for (int i = pos0 + lane; i < k_tot; i += 32)
        out[i] = -1;
    if (lane == 0)
        *count_out = min(pos0, k_tot);
}

// The selection in ascending block order: B_init, the candidates above the threshold
// key `prefix` plus the first `need` of those equal to it (lower index first; from the
// list of candidate ids when list_s is non-zero, else from all candidates), B_local;
// the rest of the row is -1.  One warp.
__device__ void topk_write_warp(uint32_t keys_s, uint32_t list_s, int n_list, int nb, int n_init, int n_local,
                                bool take_all, bool take_none, uint32_t prefix, int need, int *out, int k_tot,
                                int *count_out, int *status, int lane)
{
    const int cand_lo = n_init, cand_hi = nb - n_local;
    const int n_cand = max(0, cand_hi - cand_lo);
    const unsigned lt = (1u << lane) - 1u;
    int eq_seen = 0;
    bool overflow = false;
    int pos0 = write_init_blocks(nb, n_init, out, k_tot, overflow, lane);
    if (take_all) {
        for (int j = cand_lo + lane; j < cand_hi; j += 32) {
            const int pos = pos0 + (j - cand_lo);
            if (pos < k_tot)
                out[pos] = j;
            else
                overflow = true;
        }
        pos0 += n_cand;
    } else if (!take_none) {
        const bool from_list = list_s != 0u;
        const int hi = from_list ? n_list : cand_hi;
        for (int ib = from_list ? 0 : cand_lo; ib < hi; ib += 32) {
            const int i = ib + lane;
            int j = -1;
            uint32_t key = 0u;
            if (i < hi) {
                j = from_list ? static_cast<int>(lds_u32(list_s + 4 * i)) : i;
                key = lds_u32(keys_s + 4 * j);
            }
            bool sel = i < hi && key > prefix;
            const bool eq = i < hi && key == prefix;
            const unsigned em = __ballot_sync(0xffffffffu, eq);
            if (eq)
                sel = eq_seen + __popc(em & lt) < need;
            eq_seen += __popc(em);
            const unsigned sm = __ballot_sync(0xffffffffu, sel);
            if (sel) {
                const int pos = pos0 + __popc(sm & lt);
                if (pos < k_tot)
                    out[pos] = j;
                else
                    overflow = true;
            }
            pos0 += __popc(sm);
        }
    }
    write_local_and_close(nb, n_init, n_local, pos0, out, k_tot, count_out, status, overflow, lane);
}

// Steps 3 and 4 of topk_warp when the keys at or above the coarse bin are listed
// (n_list <= 32 * KPL, ascending block ids at list_s): lane l holds entries l + 32 m in
// registers.  The bits below the decided ones (`pmask`, value `prefix`) are found by a
// binary search from bit low_bits - 1 down, carrying how many listed keys share the
// decided bits; once all of them are needed their smallest key is the threshold.  The
// row is then written from the registers: B_init, the listed keys above the threshold
// and the first `need` equal to it (block order), B_local.
template <int KPL>
__device__ __forceinline__ void topk_list_regs(uint32_t keys_s, uint32_t list_s, int n_list, int low_bits,
                                               uint32_t prefix, uint32_t pmask, int need, int nb, int n_init,
                                               int n_local, int *out, int k_tot, int *count_out, int *status, int lane)
{
    uint32_t key[KPL];
    int id[KPL];
    const int nv = max(0, (n_list - lane + 31) / 32);   // this lane's valid entries
#pragma unroll
    for (int m = 0; m < KPL; ++m)
        id[m] = m < nv ? static_cast<int>(lds_u32(list_s + 4 * (lane + 32 * m))) : -1;
#pragma unroll
    for (int m = 0; m < KPL; ++m)
        key[m] = m < nv ? lds_u32(keys_s + 4 * id[m]) : 0u;
    int mt = 0;   // listed keys sharing the decided bits
#pragma unroll
    for (int m = 0; m < KPL; ++m)
        mt += (m < nv && (key[m] & pmask) == prefix) ? 1 : 0;
    mt = __reduce_add_sync(0xffffffffu, mt);
    uint32_t P = prefix, hmask = pmask;
    for (int b = low_bits - 1; b >= 0; --b) {
        if (mt == need) {
            uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
            for (int m = 0; m < KPL; ++m)
                if (m < nv && (key[m] & hmask) == P)
                    mn = min(mn, key[m]);
            mn = __reduce_min_sync(0xffffffffu, mn);
            int eq = 0;
#pragma unroll
            for (int m = 0; m < KPL; ++m)
                eq += (m < nv && key[m] == mn) ? 1 : 0;
            P = mn;
            need = __reduce_add_sync(0xffffffffu, eq);
            break;
        }
        const uint32_t bit = 1u << b;
        const uint32_t m2 = hmask | bit, want = P | bit;
        int c = 0;
#pragma unroll
        for (int m = 0; m < KPL; ++m)
            c += (m < nv && (key[m] & m2) == want) ? 1 : 0;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= need) {
            P = want;
            mt = c;
        } else {
            need -= c;
            mt -= c;
        }
        hmask = m2;
    }
    // the row: masks over this lane's entries, then a short loop over the list's rows of
    // 32 (this once-run code stays small; block ids are read back from the list)
    uint32_t gt_mask = 0u, eq_mask = 0u;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        gt_mask |= (m < nv && key[m] > P) ? (1u << m) : 0u;
        eq_mask |= (m < nv && key[m] == P) ? (1u << m) : 0u;
    }
    const unsigned lt = (1u << lane) - 1u;
    bool overflow = false;
    int pos0 = write_init_blocks(nb, n_init, out, k_tot, overflow, lane);
    int eq_seen = 0;
#pragma unroll 1
    for (int m = 0; 32 * m < n_list; ++m) {
        const bool eq = (eq_mask >> m) & 1u;
        bool sel = (gt_mask >> m) & 1u;
        const unsigned em = __ballot_sync(0xffffffffu, eq);
        if (eq)
            sel = eq_seen + __popc(em & lt) < need;
        eq_seen += __popc(em);
        const unsigned sm = __ballot_sync(0xffffffffu, sel);
        if (sel) {
            const int pos = pos0 + __popc(sm & lt);
            if (pos < k_tot)
                out[pos] = static_cast<int>(lds_u32(list_s + 4 * (lane + 32 * m)));
            else
                overflow = true;
        }
        pos0 += __popc(sm);
    }
    write_local_and_close(nb, n_init, n_local, pos0, out, k_tot, count_out, status, overflow, lane);
}

// The exact top-k of one row by one warp with its candidates [n_init, nb - n_local)
// (at most 32 * KPL of them) in registers, lane l holding candidates l + 32 m, written
// like topk_write_warp.  The k-th largest key value is the largest T with at least k
// keys >= T: the leading bits every key shares (a warp AND and OR) are decided at once,
// then one bit at a time, each step one compare and one add per key (an empty slot
// holds 0 and is never counted, every probe being nonzero).  A probe that exactly k
// keys reach ends the search: those k keys are the selection.  The row is written from
// the registers (bit masks, a short loop over rows of 32).  Requires
// nb - n_local - n_init > k >= 1.
template <int KPL>
__device__ __forceinline__ void topk_range_regs(uint32_t keys_s, int nb, int n_init, int n_local, int k, int *out,
                                                int k_tot, int *count_out, int *status, int lane)
{
    static_assert(KPL <= 64, "a lane's keys are bits of one 64-bit mask");
    const int cand_lo = n_init, cand_hi = nb - n_local;
    const int n_cand = cand_hi - cand_lo;
    const int nv = max(0, (n_cand - lane + 31) / 32);   // this lane's valid slots
    uint32_t key[KPL];
    uint32_t kand = 0xFFFFFFFFu, kor = 0u;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        key[m] = m < nv ? lds_u32(keys_s + 4 * (cand_lo + lane + 32 * m)) : 0u;
        if (m < nv) {
            kand &= key[m];
            kor |= key[m];
        }
    }
    kand = __reduce_and_sync(0xffffffffu, kand);
    kor = __reduce_or_sync(0xffffffffu, kor);
    const int lead = __clz(kand ^ kor);   // 32: every key equal
    uint32_t T = lead >= 32 ? kand : kand & ~(0xFFFFFFFFu >> lead);
    bool exact = false;
    for (int b = 31 - lead; b >= 0; --b) {
        const uint32_t probe = T | (1u << b);
        int c = 0;
#pragma unroll
        for (int m = 0; m < KPL; ++m)
            c += key[m] >= probe ? 1 : 0;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= k) {
            T = probe;
            if (c == k) {
                exact = true;
                break;
            }
        }
    }
    // threshold P and how many keys equal to it are taken
    uint32_t P = T;
    int need;
    if (exact) {
        uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
        for (int m = 0; m < KPL; ++m)
            if (m < nv && key[m] >= T)
                mn = min(mn, key[m]);
        P = __reduce_min_sync(0xffffffffu, mn);
    }
    uint64_t gt_mask = 0ull, eq_mask = 0ull;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        gt_mask |= (m < nv && key[m] > P) ? (1ull << m) : 0ull;
        eq_mask |= (m < nv && key[m] == P) ? (1ull << m) : 0ull;
    }
    need = exact ? __reduce_add_sync(0xffffffffu, __popcll(eq_mask))
                 : k - __reduce_add_sync(0xffffffffu, __popcll(gt_mask));
    const unsigned lt = (1u << lane) - 1u;
    bool overflow = false;
    int pos0 = write_init_blocks(nb, n_init, out, k_tot, overflow, lane);
    int eq_seen = 0;
#pragma unroll 1
    for (int m = 0; 32 * m < n_cand; ++m) {
        const bool eq = (eq_mask >> m) & 1ull;
        bool sel = (gt_mask >> m) & 1ull;
        const unsigned em = __ballot_sync(0xffffffffu, eq);
        if (eq)
            sel = eq_seen + __popc(em & lt) < need;
        eq_seen += __popc(em);
        const unsigned sm = __ballot_sync(0xffffffffu, sel);
        if (sel) {
            const int pos = pos0 + __popc(sm & lt);
            if (pos < k_tot)
                out[pos] = cand_lo + lane + 32 * m;
            else
                overflow = true;
        }
        pos0 += __popc(sm);
    }
    write_local_and_close(nb, n_init, n_local, pos0, out, k_tot, count_out, status, overflow, lane);
}

// The coarse bin that holds the k-th largest key, from the histogram of key >> 22 at
// coarse_s (kCoarseBins counts), by one warp: every lane sums its 32 bins [1024 - 32(l+1),
// 1024 - 32l) with eight 16-byte reads in a rotated order (lane l starts at its chunk
// l mod 8, so each quarter-warp's reads cover 8 distinct 16-byte bank groups), a prefix
// sum from the top bin finds the lane that holds the k-th key, and the warp then reads
// that lane's 32 bins, one a lane, for a second prefix sum that finds the bin.  Gives
// the bin (-1 if the histogram counts fewer than k keys), the keys still needed within
// it and its count, on every lane.
__device__ __forceinline__ void coarse_pick_warp(uint32_t coarse_s, int k, int lane, int &bsel, int &need_new,
                                                 int &cnt)
{
    constexpr int kPer = kCoarseBins / 32;
    static_assert(kPer == 32, "one warp, 32 bins a lane");
    const int bin0 = kCoarseBins - kPer * (lane + 1);
    int c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = lds_v4(coarse_s + 4u * static_cast<uint32_t>(bin0 + 4 * ((j + lane) & 7)));
        c += static_cast<int>(v.x + v.y + v.z + v.w);
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    const int excl = incl - c;
    const unsigned hit = __ballot_sync(0xffffffffu, excl < k && k <= incl);
    bsel = -1;
    need_new = 0;
    cnt = 0;
    if (hit == 0u)
        return;   // fewer than k keys counted
    const int src = __ffs(hit) - 1;
    const int above = __shfl_sync(0xffffffffu, excl, src);   // keys in the bins above src's
    // src's bins, the top one on lane 0: a prefix sum from the top finds the bin
    const int bin = kCoarseBins - kPer * src - 1 - lane;
    const int cb = static_cast<int>(lds_u32(coarse_s + 4u * static_cast<uint32_t>(bin)));
    int in2 = cb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, in2, o);
        if (lane >= o)
            in2 += n;
    }
    const unsigned hit2 = __ballot_sync(0xffffffffu, above + in2 - cb < k && k <= above + in2);
    const int src2 = __ffs(hit2) - 1;   // always found: the bins of src hold the k-th key
    bsel = kCoarseBins - kPer * src - 1 - src2;
    need_new = k - __shfl_sync(0xffffffffu, above + in2 - cb, src2);
    cnt = __shfl_sync(0xffffffffu, cb, src2);
}

// The exact top-k of one pair by one warp over the order keys of blocks [0, nb) (shared
// array at keys_s): the k largest keys among candidates [n_init, nb - n_local) (equal
// keys: lower block first), united with B_init and B_local, written ascending to
// out[0 .. count) and -1 after.  coarse_s holds the histogram of key >> 22 over the
// candidates (built while the keys were scored).
//   1. The coarse bin where the count from the top reaches k.
//   2. One pass: each lane tests a contiguous run of candidates against the bin's lower
//      bound (rotated so the lanes hit distinct banks) and writes the block ids of the
//      keys at or above it, ascending, into list_s (kTopkList entries at most).
//   3. The remaining 22 bits of the k-th key by a binary search over the listed keys,
//      held in registers (topk_list_regs).
//   4. B_init, then the listed keys above the k-th key and the first `need` equal to it
//      (block order), then B_local, written from the same registers.
// More than 2048 candidates, or more than kTopkList keys at or above the bin, take a
// slower path: an MSB-first radix select over byte digits that scans every candidate
// for each digit (coarse_s is reused for the digits).
__device__ void topk_warp(uint32_t keys_s, uint32_t coarse_s, uint32_t list_s, int nb, int n_init, int n_local, int k,
                          int *out, int k_tot, int *count_out, int *status, int lane)
{
    const int cand_lo = n_init, cand_hi = nb - n_local;
    const int n_cand = max(0, cand_hi - cand_lo);
    const bool take_all = n_cand <= k;
    const bool take_none = k <= 0;
    uint32_t prefix = 0, pmask = 0;
    int need = k;
    bool listed = false;
    int n_list = 0;
    if (!take_all && !take_none) {
        // 1. the coarse bin
        int bsel, need_new, m;
        coarse_pick_warp(coarse_s, need, lane, bsel, need_new, m);
        if (bsel >= 0) {   // always, when the histogram counts every candidate
            prefix = static_cast<uint32_t>(bsel) << kCoarseShift;
            pmask = ~((1u << kCoarseShift) - 1u);
            // keys strictly above the bin: k - need_new; the list holds them and the bin
            const int expect = k - need_new + m;
            need = need_new;
            if (n_cand <= 32 * 64 && expect <= kTopkList) {
                // 2. one pass over the candidates
                const int per = ((n_cand + 31) / 32 + 31) & ~31;   // 32 or 64 (a multiple of 32)
                const int jb = cand_lo + lane * per;
                uint64_t hits = 0ull;
#pragma unroll 8
                for (int i = 0; i < per; ++i) {
                    const int ii = (i + lane) & (per - 1);
                    const int j = jb + ii;
                    const uint32_t key = j < cand_hi ? lds_u32(keys_s + 4 * j) : 0u;
                    if (j < cand_hi && key >= prefix)
                        hits |= 1ull << ii;
                }
                const int cnt = __popcll(hits);
                int off = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, off, o);
                    if (lane >= o)
                        off += n;
                }
                n_list = __shfl_sync(0xffffffffu, off, 31);
                off -= cnt;
                while (hits != 0ull) {
                    const int bpos = __ffsll(static_cast<long long>(hits)) - 1;
                    if (off < kTopkList)
                        sts_u32(list_s + 4 * off, static_cast<uint32_t>(jb + bpos));
                    ++off;
                    hits &= hits - 1ull;
                }
                __syncwarp();
                listed = n_list <= kTopkList;   // equal to `expect` unless the histogram was off
            }
        } else {
            need = k;
        }
        if (listed) {   // 3 and 4 with the listed keys in registers
            topk_list_regs<kTopkList / 32>(keys_s, list_s, n_list, kCoarseShift, prefix, pmask, need, nb, n_init,
                                           n_local, out, k_tot, count_out, status, lane);
            return;
        }
        // otherwise 3. the digits below the coarse bin over every candidate (bits 23..16,
        // 15..8, 7..0; 23 and 22 are fixed), or all four digits without a coarse bin
        const uint32_t src_list = 0u;
        const int lo = cand_lo, hi = cand_hi;
        uint32_t d;
        if (pmask == 0u) {
            warp_digit_hist(keys_s, src_list, lo, hi, 0u, 0u, 24, coarse_s, lane);
            warp_pick_digit(coarse_s, need, d, lane);
            prefix = d << 24;
            pmask = 0xFF000000u;
        }
        warp_digit_hist(keys_s, src_list, lo, hi, pmask, prefix, 16, coarse_s, lane);
        warp_pick_digit(coarse_s, need, d, lane);
        prefix |= d << 16;
        pmask = 0xFFFF0000u;
        warp_digit_hist(keys_s, src_list, lo, hi, pmask, prefix, 8, coarse_s, lane);
        warp_pick_digit(coarse_s, need, d, lane);
        prefix |= d << 8;
        pmask = 0xFFFFFF00u;
        warp_digit_hist(keys_s, src_list, lo, hi, pmask, prefix, 0, coarse_s, lane);
        warp_pick_digit(coarse_s, need, d, lane);
        prefix |= d;
    }
    // 4. ascending output
    topk_write_warp(keys_s, 0u, 0, nb, n_init, n_local, take_all, take_none, prefix, need, out, k_tot, count_out,
                    status, lane);
}

// The threshold of the top-k among keys[cand_lo, cand_hi) by `nthreads` threads (whole
// warps, synchronised on named barrier `bar`; the thread with tid 0 is in warp 0): four
// passes of 8-bit digits from the top, each a histogram in per-warp shared-memory bins
// (hist_s: [nthreads / 32][256] u32, plain shared atomics, so keys packed into a few
// values cost no more than spread ones), the digit holding the need-th largest key
// picked by warp 0.  Gives the k-th largest key and how many keys equal to it are
// taken.  ctrl_s: two words that broadcast the running prefix and need.  Every
// participant must call it.
__device__ __forceinline__ void topk_threshold_cta(uint32_t keys_s, int cand_lo, int cand_hi, int k, uint32_t hist_s,
                                                   uint32_t ctrl_s, int tid, int nthreads, int bar, uint32_t &prefix_out,
                                                   int &need_out)
{
    const int warp = tid >> 5, lane = tid & 31;
    const int n_warps = nthreads >> 5;
    uint32_t prefix = 0u, pmask = 0u;
    int need = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const uint32_t my_hist = hist_s + 4u * 256u * static_cast<uint32_t>(warp);
        for (int d = lane; d < 256; d += 32)
            sts_u32(my_hist + 4 * d, 0u);
        named_barrier_sync(bar, nthreads);
        for (int ib = cand_lo + (tid & ~31); ib < cand_hi; ib += nthreads) {
            const int i = ib + lane;
            uint32_t digit = 0xFFFFFFFFu;
            if (i < cand_hi) {
                const uint32_t key = lds_u32(keys_s + 4 * i);
                if ((key & pmask) == prefix)
                    digit = (key >> shift) & 255u;
            }
            // keys close in value share their upper digits: one add for a warp that agrees
            const uint32_t d0 = __shfl_sync(0xffffffffu, digit, 0);
            const unsigned agree = __ballot_sync(0xffffffffu, digit == d0);
            if (agree == 0xffffffffu) {
                if (lane == 0 && d0 != 0xFFFFFFFFu)
                    asm volatile("red.shared.add.u32 [%0], 32;" ::"r"(my_hist + 4 * d0) : "memory");
            } else if (digit != 0xFFFFFFFFu) {
                asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(my_hist + 4 * digit) : "memory");
            }
        }
        named_barrier_sync(bar, nthreads);
        if (warp == 0) {
            for (int d = lane; d < 256; d += 32) {
                uint32_t sum = 0u;
                for (int w = 0; w < n_warps; ++w)
                    sum += lds_u32(hist_s + 4u * (256u * w + d));
                sts_u32(hist_s + 4 * d, sum);
            }
            __syncwarp();
            uint32_t d;
            warp_pick_digit(hist_s, need, d, lane);
            if (lane == 0) {
                sts_u32(ctrl_s, prefix | (d << shift));
                sts_u32(ctrl_s + 4, static_cast<uint32_t>(need));
            }
        }
        named_barrier_sync(bar, nthreads);
        prefix = lds_u32(ctrl_s);
        need = static_cast<int>(lds_u32(ctrl_s + 4));
        pmask |= 255u << shift;
    }
    prefix_out = prefix;
    need_out = need;
}

// Whether topk_cta_regs<KPT> holds n_cand candidates with nthreads threads.
template <int KPT>
__host__ __device__ constexpr bool topk_cta_regs_fits(int n_cand, int nthreads)
{
    return (((n_cand + nthreads - 1) / nthreads) | 1) <= KPT;
}

// Block-wide reductions for a group of threads (whole warps, t in [0, n_warps * 32),
// synchronised on named barrier `bar`).  buf_s: 16 words of shared memory; calls must
// alternate between two such buffers (one barrier per call: a thread may write the next
// call's buffer while another still reads this one).
__device__ __forceinline__ int group_sum(int v, uint32_t buf_s, int t, int n_warps, int bar)
{
    v = __reduce_add_sync(0xffffffffu, v);
    if ((t & 31) == 0)
        sts_u32(buf_s + 4 * (t >> 5), static_cast<uint32_t>(v));
    named_barrier_sync(bar, n_warps * 32);
    int sum = 0;
#pragma unroll
    for (int w = 0; w < 16; ++w)   // a fixed trip count: the loads issue together
        sum += w < n_warps ? static_cast<int>(lds_u32(buf_s + 4 * w)) : 0;
    return sum;
}

__device__ __forceinline__ uint32_t group_min(uint32_t v, uint32_t buf_s, int t, int n_warps, int bar)
{
    v = __reduce_min_sync(0xffffffffu, v);
    if ((t & 31) == 0)
        sts_u32(buf_s + 4 * (t >> 5), v);
    named_barrier_sync(bar, n_warps * 32);
    uint32_t m = 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < 16; ++w)
        m = w < n_warps ? min(m, lds_u32(buf_s + 4 * w)) : m;
    return m;
}

// Exclusive prefix sum of v over the group in thread order, and the total.
__device__ __forceinline__ int group_exclusive_scan(int v, uint32_t buf_s, int t, int n_warps, int bar, int &total)
{
    const int lane = t & 31;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane == 31)
        sts_u32(buf_s + 4 * (t >> 5), static_cast<uint32_t>(incl));
    named_barrier_sync(bar, n_warps * 32);
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < 16; ++w) {
        const int c = w < n_warps ? static_cast<int>(lds_u32(buf_s + 4 * w)) : 0;
        if (w < (t >> 5))
            before += c;
        total += c;
    }
    return before + incl - v;
}

// Step 3 of the group top-k selections: thread t holds keys key[0 .. nv) of the
// consecutive candidates lo, lo + 1, ...; a key is above the threshold when its bits
// under hmask exceed P, equal to it when they match P, and of the keys equal to it the
// first `need` in block order are taken.  Each thread counts its keys above and equal;
// one group prefix sum of the two counts (packed in one word) gives each thread its
// share of the `need` equal keys and its output offset; B_init, the selection and
// B_local are written ascending, -1 after, and the count.  buf_s: a 16-word reduction
// buffer.  (Bit m of a mask stands for the thread's key m; the loops run over set bits,
// so this once-run code stays short.)
template <int KPT>
__device__ __forceinline__ void cta_write_list(const uint32_t (&key)[KPT], int nv, int lo, uint32_t P, uint32_t hmask,
                                               int need, int nb, int n_init, int n_local, uint32_t buf_s, int t,
                                               int nthreads, int bar, int *out, int k_tot, int *count_out, int *status)
{
    const int n_warps = nthreads >> 5;
    uint32_t gt_mask = 0u, eq_mask = 0u;
#pragma unroll
    for (int m = 0; m < KPT; ++m) {
        const uint32_t km = key[m] & hmask;
        gt_mask |= (m < nv && km > P) ? (1u << m) : 0u;
        eq_mask |= (m < nv && km == P) ? (1u << m) : 0u;
    }
    const int n_eq = __popc(eq_mask);
    // (equal << 16) | above: both counts stay below 2^16 (at most 16 warps x 32 keys each)
    int total;
    const int before = group_exclusive_scan((n_eq << 16) | __popc(gt_mask), buf_s, t, n_warps, bar, total);
    const int eq_before = before >> 16, gt_before = before & 0xFFFF;
    const int take_eq = max(0, min(n_eq, need - eq_before));
    uint32_t sel = gt_mask, rest = eq_mask;
    for (int c = 0; c < take_eq; ++c) {   // the first take_eq equal keys, in block order
        sel |= rest & (0u - rest);
        rest &= rest - 1u;
    }
    const int sel_before = gt_before + min(eq_before, need);
    const int total_sel = (total & 0xFFFF) + min(total >> 16, need);
    const int n_i = min(n_init, nb);
    bool overflow = false;
    int pos = n_i + sel_before;
    for (; sel != 0u; sel &= sel - 1u, ++pos) {
        if (pos < k_tot)
            out[pos] = lo + __ffs(sel) - 1;
        else
            overflow = true;
    }
    for (int j = t; j < n_i; j += nthreads) {
        if (j < k_tot)
            out[j] = j;
        else
            overflow = true;
    }
    const int l0 = max(nb - n_local, n_i);
    const int pos_l = n_i + total_sel;
    for (int j = l0 + t; j < nb; j += nthreads) {
        const int q = pos_l + (j - l0);
        if (q < k_tot)
            out[q] = j;
        else
            overflow = true;
    }
    const int end = pos_l + max(0, nb - l0);
    for (int i = end + t; i < k_tot; i += nthreads)
        out[i] = -1;
    if (overflow)
        report(status, SPARSE_ERR_BAD_INDEX);
    if (t == 0)
        *count_out = min(end, k_tot);
}

// The exact top-k of one pair by a group of threads (whole warps, t in [0, nthreads),
// nthreads <= 256, synchronised on named barrier `bar`) with the candidate keys in
// registers: thread t holds the run of `per` consecutive candidates starting at
// n_init + t * per (per odd, so a warp's loads hit distinct banks; per <= KPT).  The k
// largest keys among candidates [n_init, nb - n_local) (equal keys: the lower block
// first), united with B_init and B_local, are written ascending to out[0 .. count) and
// -1 after.  Requires n_init + n_local + k < nb and k >= 1 (else topk_write_warp's
// take-all / take-none forms apply) and topk_cta_regs_fits<KPT>(n_cand, nthreads).
//   1. The leading bits that every candidate shares (the AND and the OR of the keys
//      agree there) are decided at once.
//   2. The rest by a binary search from the top, each step a group count of the keys
//      that share the decided bits and have the next bit set; the count of keys sharing
//      the decided bits is carried, and once all of them are needed their smallest key
//      is the threshold.
//   3. Each thread counts its keys above the threshold and equal to it; a group prefix
//      sum of the equal ones gives each thread its share of the `need` equal keys taken
//      (block order), a second one its output offset.
// ok: this thread's view of its inputs is complete; false on any thread: nothing is
// written and a timeout is reported.  scratch_s: 64 words of shared memory.
template <int KPT>
__device__ void topk_cta_regs(uint32_t keys_s, int nb, int n_init, int n_local, int k, uint32_t scratch_s, int t,
                              int nthreads, int bar, bool ok, int *out, int k_tot, int *count_out, int *status)
{
    static_assert(KPT % 2 == 1, "an odd run length keeps a warp's loads on distinct banks");
    static_assert(KPT <= 32, "a thread's keys are bits of one mask");
    const int n_warps = nthreads >> 5;
    const int cand_lo = n_init, cand_hi = nb - n_local;
    const int n_cand = cand_hi - cand_lo;
    const int per = ((n_cand + nthreads - 1) / nthreads) | 1;
    const int lo = cand_lo + t * per;
    const int nv = max(0, min(per, cand_hi - lo));
    uint32_t key[KPT];
    uint32_t kand = 0xFFFFFFFFu, kor = 0u;
#pragma unroll
    for (int m = 0; m < KPT; ++m) {
        key[m] = m < nv ? lds_u32(keys_s + 4 * (lo + m)) : 0u;
        if (m < nv) {
            kand &= key[m];
            kor |= key[m];
        }
    }
    // 1. shared leading bits, and whether every thread is ready (three reductions in one
    //    round: buffers 0 and 1 hold the AND and the OR, buffer 2 the not-ready count)
    {
        const uint32_t wa = __reduce_and_sync(0xffffffffu, kand);
        const uint32_t wo = __reduce_or_sync(0xffffffffu, kor);
        const int wn = __reduce_add_sync(0xffffffffu, ok ? 0 : 1);
        if ((t & 31) == 0) {
            sts_u32(scratch_s + 4 * (t >> 5), wa);
            sts_u32(scratch_s + 4 * (16 + (t >> 5)), wo);
            sts_u32(scratch_s + 4 * (32 + (t >> 5)), static_cast<uint32_t>(wn));
        }
        named_barrier_sync(bar, nthreads);
        kand = 0xFFFFFFFFu;
        kor = 0u;
        int not_ready = 0;
        for (int w = 0; w < n_warps; ++w) {
            kand &= lds_u32(scratch_s + 4 * w);
            kor |= lds_u32(scratch_s + 4 * (16 + w));
            not_ready += static_cast<int>(lds_u32(scratch_s + 4 * (32 + w)));
        }
        if (not_ready != 0) {
            if (t == 0)
                report(status, SPARSE_ERR_TIMEOUT);
            return;
        }
    }
    const int lead = __clz(kand ^ kor);   // 32 when every key is equal
    uint32_t hmask = lead >= 32 ? 0xFFFFFFFFu : ~(0xFFFFFFFFu >> lead);
    uint32_t P = kand & hmask;
    int need = k, mt = n_cand;
    int ph = 0;   // alternates the reduction buffers (words 48.. and 56..)
    auto buf = [&]() { return scratch_s + 4 * (48 + 8 * (ph++ & 1)); };
    // 2. the remaining bits
    for (int b = 31 - lead; b >= 0; --b) {
        if (mt == need)
            break;
        const uint32_t bit = 1u << b;
        const uint32_t m2 = hmask | bit, want = P | bit;
        int c = 0;
#pragma unroll
        for (int m = 0; m < KPT; ++m)
            c += (m < nv && (key[m] & m2) == want) ? 1 : 0;
        c = group_sum(c, buf(), t, n_warps, bar);
        if (c >= need) {
            P = want;
            mt = c;
        } else {
            need -= c;
            mt -= c;
        }
        hmask = m2;
    }
    if (mt == need && hmask != 0xFFFFFFFFu) {
        // every key sharing the decided bits is taken: the smallest is the threshold
        uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
        for (int m = 0; m < KPT; ++m)
            if (m < nv && (key[m] & hmask) == P)
                mn = min(mn, key[m]);
        mn = group_min(mn, buf(), t, n_warps, bar);
        int eq = 0;
#pragma unroll
        for (int m = 0; m < KPT; ++m)
            eq += (m < nv && key[m] == mn) ? 1 : 0;
        P = mn;
        need = group_sum(eq, buf(), t, n_warps, bar);
    }
    // 3. the ascending list
    cta_write_list<KPT>(key, nv, lo, P, 0xFFFFFFFFu, need, nb, n_init, n_local, buf(), t, nthreads, bar, out, k_tot,
                        count_out, status);
}

// Shared-memory words that topk_forecast_cta uses at scratch_s for n_warps warps: the
// warps' digit histograms, then its control words (placed past the coarse histogram, so
// scratch_s may be the histogram's own address).
__host__ __device__ constexpr int topk_forecast_scratch_words(int n_warps)
{
    return (n_warps * 256 > kCoarseBins ? n_warps * 256 : kCoarseBins) + 56;
}

// The exact top-k of one pair's Forecast scores by a group of NW warps (t in [0, 32 NW),
// at most 16 warps, synchronised on named barrier `bar`; t = 0 is in warp 0), with the candidate keys in registers as topk_cta_regs holds them and the coarse
// histogram of key >> 22 over the candidates at coarse_s (built while the keys were
// scored).  The k largest keys among candidates [n_init, nb - n_local) (equal keys: the
// lower block first), united with B_init and B_local, are written ascending to
// out[0 .. count) and -1 after.
//   1. Warp 0 finds the coarse bin that holds the k-th largest key: 10 bits decided.
//   2. The other 22 in passes of 8, 8 and 6 bits: each warp histograms the digit of its
//      keys that share the decided bits in 256 bins of its own (scratch, over the coarse
//      histogram once warp 0 has read it), warp 0 adds the warps' bins and picks the
//      digit that holds the need-th largest.  A bucket that holds exactly the keys still
//      needed ends the search: every key in it is taken.
//   3. The list, as topk_cta_regs writes it, above / equal meaning the decided bits.
// Requires n_init + n_local + k < nb, k >= 1 and topk_cta_regs_fits<KPT>(n_cand,
// nthreads).  ok: this thread's view of its inputs is complete; false on any thread:
// nothing is written and a timeout is reported.
template <int KPT, int NW>
__device__ void topk_forecast_cta(uint32_t keys_s, uint32_t coarse_s, uint32_t scratch_s, int nb, int n_init,
                                  int n_local, int k, int t, int bar, bool ok, int *out, int k_tot, int *count_out,
                                  int *status)
{
    static_assert(KPT % 2 == 1, "an odd run length keeps a warp's loads on distinct banks");
    static_assert(KPT <= 32, "a thread's keys are bits of one mask");
    static_assert(NW >= 1 && NW <= 16, "at most 16 warps");
    constexpr int n_warps = NW;
    constexpr int nthreads = 32 * NW;
    const int warp = t >> 5, lane = t & 31;
    const int cand_lo = n_init, cand_hi = nb - n_local;
    const int n_cand = cand_hi - cand_lo;
    const int per = ((n_cand + nthreads - 1) / nthreads) | 1;
    const int lo = cand_lo + t * per;
    const int nv = max(0, min(per, cand_hi - lo));
    // control words: [0..2] and [4..6] broadcast slots (prefix, need, bucket count),
    // [8..23] and [24..39] reduction buffers, [40..55] the warps' not-ready counts
    const uint32_t ctrl_s = scratch_s + 4u * static_cast<uint32_t>(topk_forecast_scratch_words(n_warps) - 56);
    uint32_t key[KPT];
#pragma unroll
    for (int m = 0; m < KPT; ++m)
        key[m] = m < nv ? lds_u32(keys_s + 4 * (lo + m)) : 0u;
    const int wn = __reduce_add_sync(0xffffffffu, ok ? 0 : 1);
    if (lane == 0)
        sts_u32(ctrl_s + 4 * (40 + warp), static_cast<uint32_t>(wn));
    // 1. the coarse bin: lane l holds bins [1024 - 32(l+1), 1024 - 32l)
    if (warp == 0) {
        int bsel, need_new, cnt;
        coarse_pick_warp(coarse_s, k, lane, bsel, need_new, cnt);
        const unsigned hit = __ballot_sync(0xffffffffu, bsel >= 0);
        if (hit != 0u && lane == __ffs(hit) - 1) {
            sts_u32(ctrl_s, static_cast<uint32_t>(bsel) << kCoarseShift);
            sts_u32(ctrl_s + 4, static_cast<uint32_t>(need_new));
            sts_u32(ctrl_s + 8, static_cast<uint32_t>(cnt));
            sts_u32(ctrl_s + 12, 1u);
        } else if (hit == 0u && lane == 0) {   // cannot happen when the histogram counts every candidate
            sts_u32(ctrl_s, 0u);
            sts_u32(ctrl_s + 4, static_cast<uint32_t>(k));
            sts_u32(ctrl_s + 8, static_cast<uint32_t>(n_cand));
            sts_u32(ctrl_s + 12, 0u);
        }
    }
    named_barrier_sync(bar, nthreads);
    int not_ready = 0;
#pragma unroll
    for (int w = 0; w < n_warps; ++w)
        not_ready += static_cast<int>(lds_u32(ctrl_s + 4 * (40 + w)));
    if (not_ready != 0) {
        if (t == 0)
            report(status, SPARSE_ERR_TIMEOUT);
        return;
    }
    uint32_t P = lds_u32(ctrl_s);
    int need = static_cast<int>(lds_u32(ctrl_s + 4));
    int cnt = static_cast<int>(lds_u32(ctrl_s + 8));
    int top = lds_u32(ctrl_s + 12) != 0u ? kCoarseShift : 32;
    uint32_t hmask = top == 32 ? 0u : ~((1u << kCoarseShift) - 1u);
    // 2. the digits below the decided bits
    int slot = 1;
    while (top > 0 && cnt != need) {
        const int w = top < 8 ? top : 8;
        const int shift = top - w;
        const uint32_t dmask = (1u << w) - 1u;
        const uint32_t my_hist = scratch_s + 4u * 256u * static_cast<uint32_t>(warp);
        for (int d = lane; d < 256; d += 32)
            sts_u32(my_hist + 4 * d, 0u);
        __syncwarp();
#pragma unroll
        for (int m = 0; m < KPT; ++m)
            if (m < nv && (key[m] & hmask) == P)
                asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(my_hist + 4 * ((key[m] >> shift) & dmask)) : "memory");
        named_barrier_sync(bar, nthreads);
        if (warp == 0) {
            // lane l holds digits 255 - 8l - i (i = 0..7), summed over the warps' bins
            // (two 16-byte reads per warp's bins: digits [248 - 8l, 256 - 8l))
            int c[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sum = 0;
#pragma unroll
            for (int ww = 0; ww < n_warps; ++ww) {
                const uint32_t wb = scratch_s + 4u * (256u * ww + 248u - 8u * static_cast<uint32_t>(lane));
                const uint4 d0 = lds_v4(wb), d1 = lds_v4(wb + 16);
                c[0] += static_cast<int>(d1.w);
                c[1] += static_cast<int>(d1.z);
                c[2] += static_cast<int>(d1.y);
                c[3] += static_cast<int>(d1.x);
                c[4] += static_cast<int>(d0.w);
                c[5] += static_cast<int>(d0.z);
                c[6] += static_cast<int>(d0.y);
                c[7] += static_cast<int>(d0.x);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                sum += c[i];
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += n;
            }
            const int excl = incl - sum;
            int dsel = -1, need_new = 0, cdig = 0;
            if (excl < need && need <= incl) {
                int acc = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (dsel < 0 && acc + c[i] >= need) {
                        dsel = 255 - 8 * lane - i;
                        need_new = need - acc;
                        cdig = c[i];
                    }
                    acc += c[i];
                }
            }
            const unsigned hit = __ballot_sync(0xffffffffu, dsel >= 0);
            // (always found: the bins count exactly the cnt >= need keys sharing the decided bits)
            const int src = hit != 0u ? __ffs(hit) - 1 : 0;
            if (lane == src) {
                const uint32_t so = ctrl_s + 16u * static_cast<uint32_t>(slot);
                sts_u32(so, P | (static_cast<uint32_t>(dsel < 0 ? 0 : dsel) << shift));
                sts_u32(so + 4, static_cast<uint32_t>(hit != 0u ? need_new : need));
                sts_u32(so + 8, static_cast<uint32_t>(hit != 0u ? cdig : need));
            }
        }
        named_barrier_sync(bar, nthreads);
        const uint32_t so = ctrl_s + 16u * static_cast<uint32_t>(slot);
        P = lds_u32(so);
        need = static_cast<int>(lds_u32(so + 4));
        cnt = static_cast<int>(lds_u32(so + 8));
        hmask |= dmask << shift;
        top = shift;
        slot ^= 1;
    }
    // 3. the ascending list
    cta_write_list<KPT>(key, nv, lo, P, hmask, need, nb, n_init, n_local, ctrl_s + 4 * 8, t, nthreads, bar, out,
                        k_tot, count_out, status);
}

}  // namespace

/*
 * sparse_pool.h -- C ABI of libsparsepool, block-sparse GQA decode attention with
 * learned block selection, for one GB300 GPU (sm_103a).
 *
 * The method (two reading-note pages on the web):
 *   [SparDA] "SparDA: sparse decoupled attention" notes, zhongzhuzhou.org/blog/2026-06-24
 *   [SSV]    "SSV: sparse speculative verification" notes, zhongzhuzhou.org/blog/2026-07-01
 *
 * Conventions shared by every entry point
 *   - Head dimension d = 128 and block size 64 tokens are fixed.
 *   - bf16 tensors are passed as uint16_t* holding the bf16 bit patterns.
 *   - "pair" = (batch b, KV head g), flattened as p = b * H_kv + g.  Query head h of a
 *     batch belongs to KV head floor(h / G), G = H_q / H_kv (contiguous groups).
 *   - All pointers are device-accessible addresses (device memory, or host memory
 *     mapped into the device address space where stated), at least 16-byte aligned.
 *     The caller owns every buffer; the library allocates no device memory.
 *   - Every call is asynchronous on the given CUDA stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Arguments are validated on the host
 *     before any launch; a rejected call launches nothing and returns a negative
 *     status.  Errors found on the device (bad block ids, a wait that timed out) are
 *     written to the optional int32 `status` word in device memory (first error wins,
 *     0 = OK) and never trap.
 *   - Calls return SPARSE_OK or a negative SPARSE_ERR_* code; sparse_last_error()
 *     gives a message for the last failing call on the calling host thread.
 */
#ifndef SPARSE_POOL_H
#define SPARSE_POOL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPARSE_API __attribute__((visibility("default")))
#else
#define SPARSE_API
#endif

enum {
    SPARSE_OK = 0,
    SPARSE_ERR_INVALID_ARG = -1,   /* a null pointer, a bad size or misaligned buffer  */
    SPARSE_ERR_UNSUPPORTED = -2,   /* a size outside what the kernels handle           */
    SPARSE_ERR_CUDA = -3,          /* a CUDA runtime call failed                       */
    SPARSE_ERR_TIMEOUT = -4,       /* device: a bounded wait gave up                   */
    SPARSE_ERR_NOT_READY = -5,     /* device: a staging slot was not marked ready      */
    SPARSE_ERR_BAD_INDEX = -6      /* device: a block id outside the cache was skipped */
};

/* Message for a status code (static storage). */
SPARSE_API const char *sparse_status_string(int status);

/* Message of the last failing call on this host thread ("" if none). */
SPARSE_API const char *sparse_last_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
SPARSE_API int sparse_version(void);

/*
 * sparse_pool_append -- [SparDA] §4.2 Alg.1 step 1 and background eq.(4).
 * Appends n_new tokens to every pair's K and V cache at positions
 * [len_before, len_before + n_new) and updates the compressed key of every block
 * those tokens touch, at O(d) cost per block:
 *     ktil[p][j] = (n_old * ktil[p][j] + sum of the new keys in block j) / n_total,
 * n_old / n_total the tokens of block j before / after the append.  After the call
 * ktil[p][j] is the mean of the keys present in block j (the last block may be
 * partial).  Blocks that were empty before are overwritten, not read.
 *   k_cache, v_cache  [B][H_kv][T_cap][128] bf16, written.
 *   ktil              [B][H_kv][N_cap][128] fp32, read-modify-written, N_cap >= ceil((len_before+n_new)/64).
 *   k_new, v_new      [B][H_kv][n_new][128] bf16, read.
 * Requires len_before >= 0, n_new >= 1, len_before + n_new <= T_cap.  The caches may
 * be device memory or mapped pinned host memory.
 * Launch order: programmatic stream serialization.  The kernel waits for the kernel
 * before it on the stream before reading anything, and lets the kernel after it be
 * scheduled at once; that kernel must wait (as every call of this library does,
 * unless a flag promises otherwise) before reading what this one writes.
 */
SPARSE_API int sparse_pool_append(uint16_t *k_cache, uint16_t *v_cache, float *ktil,
                                  const uint16_t *k_new, const uint16_t *v_new,
                                  int B, int H_kv, long long T_cap, int N_cap,
                                  long long len_before, int n_new, void *stream);

/*
 * sparse_pool_append_kv -- sparse_pool_append that also keeps the compressed values,
 * the rows of NSA's compressed branch ([SSV] "NSA three-branch math", step 4, read
 * as mean pooling like the keys, [SparDA] eq.(4)):
 *     vtil[p][j] = (n_old * vtil[p][j] + sum of the new values in block j) / n_total,
 * and, when khat / vhat are given, bf16 copies (round to nearest even) of every ktil
 * and vtil row it writes: the compressed cache that sparse_decode_attn_nsa reads.
 *   vtil         [B][H_kv][N_cap][128] fp32, read-modify-written (required).
 *   khat, vhat   [B][H_kv][N_cap][128] bf16, written for the touched rows; either may
 *                be NULL.
 * Every other argument and requirement is that of sparse_pool_append.
 */
SPARSE_API int sparse_pool_append_kv(uint16_t *k_cache, uint16_t *v_cache, float *ktil,
                                     float *vtil, uint16_t *khat, uint16_t *vhat,
                                     const uint16_t *k_new, const uint16_t *v_new,
                                     int B, int H_kv, long long T_cap, int N_cap,
                                     long long len_before, int n_new, void *stream);

/*
 * sparse_select_topk -- [SparDA] §4.1 eq.(6), §4.2 Alg.1 step 2, §4.3 eq.(9).
 * For every pair: N_b = ceil(seq_len[b] / 64); B_init = blocks [0, n_init);
 * B_local = the last n_local blocks [N_b - n_local, N_b); every other block j is a
 * candidate with score s_j = sum_d F[p][d] * ktil[p][j][d] (fp32).  The k candidates
 * of largest score are taken (equal scores: the lower block index wins; the softmax
 * and temperature of eq.(9) are monotone and do not change the top-k), and
 * idx_out[p][0 .. count_out[p]) = B_init ∪ B_local ∪ top-k in ascending order, the
 * rest of the row filled with -1.  count = min(N_b, n_init + n_local + k).
 *   F          [B][H_kv][128] bf16: one Forecast vector per GQA group.
 *   ktil       [B][H_kv][N_cap][128] fp32 compressed keys of the layer selected for.
 *   seq_len    [B] int32 (device): tokens present per batch element.
 *   idx_out    [B][H_kv][k_tot] int32, k_tot >= n_init + n_local + k.
 *   count_out  [B][H_kv] int32.
 *   status     optional int32 device word (a length beyond N_cap*64 is reported).
 */
SPARSE_API int sparse_select_topk(const uint16_t *F, const float *ktil, const int *seq_len,
                                  int B, int H_kv, int N_cap, int n_init, int n_local, int k,
                                  int *idx_out, int *count_out, int k_tot, int *status,
                                  void *stream);

/*
 * sparse_select_topk_ex -- sparse_select_topk with launch-order flags (the same
 * arguments, results and launch order otherwise; flags = 0 is sparse_select_topk).
 *   flags  0 or SPARSE_SELECT_KEYS_READY: the caller promises that seq_len and the
 *          compressed keys of the candidate blocks [n_init, N_b - n_local) are not
 *          written by the kernel before this one on the stream (e.g. a decode step's
 *          sparse_pool_append, which only touches the block holding the new token: a
 *          local block).  The selection then streams those keys at once, overlapping
 *          that kernel, and waits for it only before reading F.  Only candidate keys
 *          are read in any case.
 */
#define SPARSE_SELECT_KEYS_READY 8u

SPARSE_API int sparse_select_topk_ex(const uint16_t *F, const float *ktil, const int *seq_len,
                                     int B, int H_kv, int N_cap, int n_init, int n_local, int k,
                                     int *idx_out, int *count_out, int k_tot, unsigned flags,
                                     int *status, void *stream);

/*
 * sparse_prefill_select -- the Forecast selection of every prefill position, [SparDA]
 * §4.3 eq.(16) (the indexer scores all T positions against the compressed keys,
 * H_kv * T * N_b * d multiply-adds) with the per-position selection of sparse_select_topk:
 * position t < seq_len[b] of pair p sees the blocks holding tokens 0..t,
 * N_t = floor(t / 64) + 1; s_j = F[p][t] . ktil[p][j]; B_init = [0, n_init),
 * B_local = [N_t - n_local, N_t), and the k candidates of largest score (ties to the
 * lower block), written ascending, padded with -1.  The scores run on the tensor cores
 * with the fp32 keys split into three bf16 terms (exact products, fp32 sums).
 *   F          [B][H_kv][T_cap][128] bf16: the Forecast vector of every position.
 *   ktil       [B][H_kv][N_cap][128] fp32 compressed keys of the prefill (the block
 *              holding t may include later tokens: it is local, so n_local >= 1).
 *   idx_out    [B][H_kv][T_cap][k_tot] int32, count_out [B][H_kv][T_cap] int32; rows at
 *              or past seq_len[b] are not written.
 * N_cap <= 2048 (131072 tokens).
 */
SPARSE_API int sparse_prefill_select(const uint16_t *F, long long T_cap, const float *ktil, int N_cap,
                                     const int *seq_len, int B, int H_kv, int n_init, int n_local,
                                     int k, int *idx_out, int *count_out, int k_tot, int *status,
                                     void *stream);

/*
 * sparse_select_topk_heads -- the multi-head block selector of InfLLM-V2, the baseline
 * that [SparDA] §4.3 (eq.(8) and its Figure 3) compares the Forecast selector with:
 * every one of the G = H_q / H_kv query heads of pair p scores every compressed key,
 *     a^h_j = scale * q_h . ktil_j,   j < N_b = ceil(seq_len[b] / 64),
 * each head's scores pass through a softmax over the pair's N_b blocks, and
 *     s_j = sum_h softmax_j(a^h)
 * replaces the Forecast score; the k largest s_j outside B_init and B_local are taken
 * (equal keys: lower block index) and idx_out / count_out are written as by
 * sparse_select_topk.  (The notes' max-pooling onto selection blocks is the identity
 * for non-overlapping 64-token blocks.)  Scores and sums are fp32.
 *   Q          [B][H_q][128] bf16: the query heads of the layer selected for.
 *   ktil, seq_len, N_cap, n_init, n_local, k, idx_out, count_out, k_tot, status
 *              as for sparse_select_topk.
 *   scale      0 selects 1/sqrt(128).  G <= 16.
 * Launch order as for sparse_select_topk (every input may come from the kernel before).
 */
SPARSE_API int sparse_select_topk_heads(const uint16_t *Q, const float *ktil, const int *seq_len,
                                        int B, int H_q, int H_kv, int N_cap, float scale,
                                        int n_init, int n_local, int k, int *idx_out,
                                        int *count_out, int k_tot, int *status, void *stream);

/*
 * sparse_decode_attn -- [SparDA] §4.1 eq.(7), §4.2 Alg.1 step 4; scale 1/sqrt(d) per
 * the [SSV] NSA selection branch (step 3); split-KV merge by the online-softmax
 * recurrence of [SSV] "online softmax state merging".
 * For every query head h of pair p = (b, floor(h/G)):
 *     O[b][h] = sum_t softmax_t(scale * q_h . k_t) v_t
 * over the tokens t = 64 * blk_logical[p][i] + r (i < count[p], r < 64) with
 * t < seq_len[b].  Token rows are read from the pair's region of k_base / v_base at
 * row 64 * slot + r, slot = blk_slot[p][i]; with blk_slot NULL the slot is the
 * logical id itself (a resident cache).  A staging ring that holds the selected
 * blocks in list order passes the slot table slot[p][i] = i.  The listed blocks are
 * expected to be distinct (a repeated id contributes its tokens once per listing).
 *   Q            [B][H_q][128] bf16.
 *   k_base,v_base [B*H_kv][pair_stride_tokens][128] bf16 (a resident cache with
 *                pair_stride_tokens = T_cap, or a staging ring with k_tot * 64).
 *   blk_slot     [B*H_kv][k_tot] int32, or NULL for slot = logical id.
 *   blk_logical  [B*H_kv][k_tot] int32 logical block ids (as sparse_select_topk writes).
 *   count        [B*H_kv] int32 (device), 0 <= count <= k_tot.
 *   seq_len      [B] int32 (device).
 *   scale        0 selects 1/sqrt(128).
 *   O            [B][H_q][128] bf16;  lse [B][H_q] fp32 natural-log LSE, or NULL.
 *   n_split      CTAs sharing one pair's list.  Without a workspace 1, 2, 4 or 8 (one
 *                thread-block cluster per pair); with a workspace 1 .. 64; with a
 *                workspace and SPARSE_ATTN_STREAM_K the total CTA count.  0 = chosen
 *                from the SM count.  The result does not depend on it beyond fp32
 *                rounding.
 *   flags        SPARSE_ATTN_BLOCKS_READY and / or SPARSE_ATTN_STREAM_K (below), or 0.
 *   workspace    NULL, or device memory of sparse_decode_attn_workspace_size() bytes
 *                (workspace_bytes gives its size).
 *                Without a workspace the CTAs of a pair form a thread-block cluster and
 *                merge their partial softmax states through distributed shared memory
 *                (no scratch; the cluster waits for its slowest CTA).
 *                With a workspace (the split path) CTA r of a pair attends over entries
 *                [r * ceil(k_tot / S), (r + 1) * ceil(k_tot / S)) of its list, writes its
 *                partial state to the workspace and exits; the CTA of the pair that
 *                arrives last merges the S states and writes O and lse.
 *                With a workspace, SPARSE_ATTN_STREAM_K and G <= 8, the stream-K path
 *                runs instead: a persistent grid of two CTAs per SM splits the
 *                flattened (pair, block) list into equal ranges, merged the same way.
 *                The workspace must be all zero before the first call that uses it;
 *                every call returns its arrival counters to zero.  Calls that share a
 *                workspace must not run at the same time.
 * A row with no valid token gets O = 0 and lse = -inf.  G = H_q / H_kv <= 16,
 * k_tot <= 4096.
 *
 * Launch order.  The kernel is launched with programmatic stream serialization: it
 * may be scheduled while the kernel before it on the stream is still running, and it
 * waits for that kernel (griddepcontrol.wait) before reading any input -- unless the
 * caller passes SPARSE_ATTN_BLOCKS_READY, which promises that the block table,
 * count, seq_len and the K/V rows are already complete while that preceding kernel
 * runs: none of them is written by it (they come from an earlier kernel on the stream,
 * or from another stream ordered by an event).  Then the kernel stages its block list
 * and starts streaming K/V at once and waits only before reading Q and writing O and
 * lse.  This is SparDA's decoupling (§4.1): the blocks of layer l+1 are chosen one
 * layer ahead, so their loads need not wait for Q_{l+1}.
 * Every kernel of this library lets its successor start only after its own wait,
 * except sparse_decode_attn_forecast, which lets it start at once: an input written
 * two launches back is complete, unless the launch in between is
 * sparse_decode_attn_forecast.
 */
#define SPARSE_ATTN_BLOCKS_READY 1u
/* Use the stream-K path whenever a workspace is given (see `workspace`). */
#define SPARSE_ATTN_STREAM_K 2u
/*
 * Run both contractions of the cluster path on the 5th-generation tensor cores:
 * S^T = K Q^T and O^T += V^T P^T as tcgen05.mma (bf16 operands in the 128-byte
 * swizzled shared-memory tiles the TMA ring holds, f32 accumulators in tensor memory,
 * one issuing thread), the softmax in 4 warps that read S^T from tensor memory and
 * write P to shared memory, the row max updated lazily (O rescaled in tensor memory
 * only when a row's max grows by more than 2^8).  Without it the contractions are
 * warp-level mma.sync with the accumulators in registers.  Same results up to
 * rounding; it runs the cluster path only, so it may not be combined with a workspace
 * (SPARSE_ERR_INVALID_ARG).  On these memory-bound shapes (at most 16 query rows a
 * pair) it is measured slower: every ring stage stays held while its product goes
 * through the issuing thread, tensor memory, the softmax warps and back, and with
 * three stages per CTA that hold time bounds the bandwidth.  The verification calls
 * take the same flag.
 */
#define SPARSE_ATTN_TENSOR_MEMORY 16u

SPARSE_API int sparse_decode_attn(const uint16_t *Q, const uint16_t *k_base,
                                  const uint16_t *v_base, long long pair_stride_tokens,
                                  const int *blk_slot, const int *blk_logical, const int *count,
                                  int k_tot, const int *seq_len, int B, int H_q, int H_kv,
                                  float scale, uint16_t *O, float *lse, int n_split,
                                  unsigned flags, void *workspace, size_t workspace_bytes,
                                  int *status, void *stream);

/*
 * Bytes of the sparse_decode_attn workspace for these sizes on the current device
 * (n_split as for sparse_decode_attn): enough for the split path and, for G <= 8, the
 * stream-K path; 0 when the sizes are invalid.  The SparDA notes have no counterpart:
 * this is the size of the per-pair arrival counters and the partial softmax states.
 */
SPARSE_API size_t sparse_decode_attn_workspace_size(int B, int H_q, int H_kv, int k_tot, int n_split);

/*
 * sparse_decode_attn_noalloc -- sparse_decode_attn for callers that cannot allocate
 * device memory.  The SparDA and SSV notes have no counterpart to this call.
 * Some callers have no device allocator to hand or may not use one here: a plain C
 * host without a caching allocator (a cudaMalloc per call would synchronise the
 * device), a serving engine whose device memory is planned up front and forbids
 * ad-hoc allocation, or a runtime that hands this library only the tensors of the
 * layer.  This call takes the same arguments as sparse_decode_attn without the
 * workspace and runs the stream-K path (G <= 8) on scratch held in a fixed 4 MiB
 * array of device memory inside the library; every GPU that loads the library keeps
 * that array until the process exits.  Sizes whose scratch would exceed 4 MiB are
 * rejected with SPARSE_ERR_UNSUPPORTED before any launch (B*H_kv = 64 pairs at
 * k_tot = 67 need about 2.6 MB).  The call allocates nothing: no cudaMalloc or
 * cudaFree, no allocating library routine.
 * The first call in a CUDA context looks up the array's device address (once per
 * context, with the context's device current; a context created again after
 * cudaDeviceReset holds a new copy of the array and is looked up anew); make that
 * first call before any stream capture.  Every argument is checked before anything
 * is queued: a rejected call leaves the array untouched.  Each accepted call first
 * clears the array's per-pair counters on its stream.  All calls share the one array,
 * so calls that overlap on the GPU (other streams, other threads) race: order them on
 * one stream.
 */
SPARSE_API int sparse_decode_attn_noalloc(const uint16_t *Q, const uint16_t *k_base,
                                          const uint16_t *v_base, long long pair_stride_tokens,
                                          const int *blk_slot, const int *blk_logical,
                                          const int *count, int k_tot, const int *seq_len, int B,
                                          int H_q, int H_kv, float scale, uint16_t *O, float *lse,
                                          int n_split, unsigned flags, int *status, void *stream);

/*
 * sparse_decode_attn_ex -- sparse_decode_attn that first checks a staging-ready word.
 * Before reading, every CTA polls *ready_flag (device memory, acquire) until it is
 * >= ready_target, for at most timeout_ns nanoseconds (0 = check once, capped at
 * 2 s).  If the word does not reach the target, the call reads no K/V, leaves the
 * O and lse rows it could not complete untouched and reports SPARSE_ERR_TIMEOUT (timeout_ns > 0) or
 * SPARSE_ERR_NOT_READY (timeout_ns == 0) in *status.  Ordering the producer before
 * this call (same stream, or an event) is the caller's job; the word is an integrity
 * check, not a substitute for stream order.
 */
SPARSE_API int sparse_decode_attn_ex(const uint16_t *Q, const uint16_t *k_base,
                                     const uint16_t *v_base, long long pair_stride_tokens,
                                     const int *blk_slot, const int *blk_logical,
                                     const int *count, int k_tot, const int *seq_len, int B,
                                     int H_q, int H_kv, float scale, uint16_t *O, float *lse,
                                     int n_split, unsigned flags, void *workspace,
                                     size_t workspace_bytes, const unsigned *ready_flag,
                                     unsigned ready_target, long long timeout_ns, int *status,
                                     void *stream);

/*
 * sparse_decode_attn_forecast -- one decode layer: the attention of layer l fused with
 * the Forecast selection for layer l+1.  [SparDA] §4.1 (the Forecast vector F_l of
 * layer l selects the blocks of layer l+1 from its compressed keys, eq.(6), so that
 * selection runs while layer l attends, eq.(7)) and §4.2 Alg.1 steps 2 and 4.
 * It computes exactly what these two calls compute, in one kernel:
 *     sparse_decode_attn(Q, k_cache, v_cache, T_cap, NULL, blk_idx, count, k_tot,
 *                        seq_len, B, H_q, H_kv, scale, O, lse, n_split, flags, ...)
 *     sparse_select_topk(F, ktil_next, seq_len, B, H_kv, N_cap, n_init, n_local, k,
 *                        idx_next, count_next, k_tot_next, ...)
 * (the selection scores with the same fp32 arithmetic, so its lists are identical to
 * sparse_select_topk's).  The attention reads a resident cache (slot = logical id).
 *   Q, k_cache, v_cache, T_cap, blk_idx, count, k_tot, seq_len, B, H_q, H_kv, scale,
 *   O, lse       as for sparse_decode_attn (k_cache / v_cache [B][H_kv][T_cap][128]).
 *   F            [B][H_kv][128] bf16 Forecast vectors of layer l, or NULL: attention
 *                only (ktil_next .. k_tot_next are then ignored).
 *   ktil_next    [B][H_kv][N_cap][128] fp32 compressed keys of layer l+1.
 *   N_cap, n_init, n_local, k, idx_next [B][H_kv][k_tot_next], count_next [B][H_kv]
 *                as for sparse_select_topk; idx_next / count_next must not alias
 *                blk_idx / count.
 *   n_split      CTAs per pair (1, 2, 4, 8 or, for G <= 8, 16; 0 = chosen from the SM
 *                count): each takes a slice of the pair's block list and of its
 *                compressed keys.  16 is a non-portable cluster size: it is used (and
 *                chosen automatically, when few pairs have to fill the GPU) only where
 *                the device can schedule such clusters; an explicit 16 that cannot be
 *                scheduled is rejected with SPARSE_ERR_UNSUPPORTED.
 *   flags        0 or SPARSE_ATTN_BLOCKS_READY (as for sparse_decode_attn).
 * Shared memory holds the pair's N_cap keys: N_cap up to about 28000.
 *
 * Launch order.  seq_len and ktil_next must not be written by the kernel preceding
 * this one on the stream (compressed keys are updated by the append of the previous
 * decode step): each CTA streams its slice of ktil_next at once.  Q and F may
 * be written by that preceding kernel; so may blk_idx and count unless
 * SPARSE_ATTN_BLOCKS_READY is passed.  The kernel lets the next kernel on the stream be
 * scheduled as soon as it has started, so a chain of these calls, layer after layer
 * (idx_next of one call is blk_idx of the next), overlaps each layer's compressed-key
 * stream with the end of the layer before.
 */
SPARSE_API int sparse_decode_attn_forecast(const uint16_t *Q, const uint16_t *k_cache,
                                           const uint16_t *v_cache, long long T_cap,
                                           const int *blk_idx, const int *count, int k_tot,
                                           const int *seq_len, int B, int H_q, int H_kv,
                                           float scale, uint16_t *O, float *lse,
                                           const uint16_t *F, const float *ktil_next, int N_cap,
                                           int n_init, int n_local, int k, int *idx_next,
                                           int *count_next, int k_tot_next, int n_split,
                                           unsigned flags, int *status, void *stream);

/*
 * sparse_verify_attn_grouped -- [SSV] mechanism 1, mode A (exact merged schedule).
 * N_q verification queries per sequence (already flattened in BFS order) are split
 * into groups of C consecutive queries.  For group [q0, q0 + C) of pair (b, g) the
 * merged set U = ∪_q (I_q ∪ W) is loaded once, W = the last window_blocks blocks
 * [N_b - window_blocks, N_b) of the committed sequence, and every query head h of
 * every query q of the group attends over its own set I_q ∪ W only:
 *     O[b][q][h] = sum_t softmax_t(scale * q_{q,h} . k_t) v_t,  t in I_q ∪ W, t < seq_len[b].
 *   Q        [B][N_q][H_q][128] bf16.
 *   k_cache, v_cache [B][H_kv][T_cap][128] bf16 (committed tokens).
 *   idx_q    [B][H_kv][N_q][n_sel] int32 per-query block ids (any order; repeats and
 *            blocks of W count once; ids outside [0, N_b) are skipped and reported).
 *   O        [B][N_q][H_q][128] bf16.
 *   blocks_loaded  optional int64 device counter: += |U| for every group (the blocks
 *            this call streams from HBM).  Without grouping the count would be
 *            sum_q |I_q ∪ W|.
 *   flags    SPARSE_ATTN_TENSOR_MEMORY: the contractions on tcgen05 (as for
 *            sparse_decode_attn).  SPARSE_ATTN_BLOCKS_READY: the caller promises that
 *            idx_q, seq_len and the K/V rows are not written by the kernel preceding this one on the
 *            stream (e.g. the lists of a reuse layer, routed layers earlier; the
 *            launch-order rule of sparse_decode_attn), so the union is built and the
 *            blocks stream while that kernel drains; only Q and the outputs wait for
 *            it.  Without the flag every input may be that kernel's output and
 *            everything waits.
 * Limits: C * G <= 16 rows per group tile; C * n_sel + window_blocks <= 512.
 */
SPARSE_API int sparse_verify_attn_grouped(const uint16_t *Q, const uint16_t *k_cache,
                                          const uint16_t *v_cache, long long T_cap,
                                          const int *idx_q, int n_sel, int N_q, int C,
                                          int window_blocks, const int *seq_len, int B,
                                          int H_q, int H_kv, float scale, uint16_t *O,
                                          long long *blocks_loaded, int n_split, unsigned flags,
                                          int *status, void *stream);

/*
 * sparse_verify_attn_shared -- [SSV] mechanism 1, mode B (approximate shared index
 * layout).  Same arguments and layouts as sparse_verify_attn_grouped, but every query
 * of a group attends over the layout of the group's representative, its first query:
 *     O[b][q][h] = attention over I_{q_rep} ∪ W,   q_rep = the first query of q's group,
 * so the group loads that one layout (|I_{q_rep} ∪ W| blocks, added to *blocks_loaded)
 * instead of the merged union.  An approximation of the per-query sets, which the SSV
 * notes recommend when the overlap is high.
 */
SPARSE_API int sparse_verify_attn_shared(const uint16_t *Q, const uint16_t *k_cache,
                                         const uint16_t *v_cache, long long T_cap,
                                         const int *idx_q, int n_sel, int N_q, int C,
                                         int window_blocks, const int *seq_len, int B,
                                         int H_q, int H_kv, float scale, uint16_t *O,
                                         long long *blocks_loaded, int n_split, unsigned flags,
                                         int *status, void *stream);

/*
 * sparse_decode_attn_nsa -- NSA's gated three-branch decode output, [SSV] "NSA
 * three-branch math" steps 3-6 (the three-branch sum of its background section):
 *     o = g_c o^(c) + g_s o^(s) + g_w o^(w)
 * for every query head of every pair, each branch its own softmax with scale 1/sqrt(d)
 * (or `scale`):
 *   o^(s)  over the tokens of the selected blocks blk_idx[p][0 .. count[p])
 *          (sparse_decode_attn's table, logical block ids, no slot indirection);
 *   o^(w)  over the last window_tokens tokens [len - w, len), token-granular;
 *   o^(c)  over the compressed rows khat / vhat [p][0 .. R): with cmp_len = cmp_stride
 *          = 0 one row per 64-token block holding a token, R = ceil(len / 64)
 *          (sparse_pool_append_kv keeps them); otherwise NSA's overlapping windows
 *          [cmp_stride * j, cmp_stride * j + cmp_len), complete ones only,
 *          R = floor((len - cmp_len) / cmp_stride) + 1 (sparse_nsa_compress keeps them);
 * a branch with no rows contributes zero.  The gates are inputs: NSA learns them.
 *   Q                 [B][H_q][128] bf16.
 *   k_cache, v_cache  [B][H_kv][T_cap][128] bf16.
 *   khat, vhat        [B][H_kv][N_cap][128] bf16 compressed rows, N_cap >= R (a longer
 *                     length is reported and its rows clipped).
 *   cmp_len, cmp_stride  0, 0 or 1 <= cmp_stride <= cmp_len <= 1024 (above).
 *   blk_idx, count    [B*H_kv][k_tot] int32 and [B*H_kv] int32, as sparse_select_topk
 *                     writes them; ids outside [0, T_cap / 64) are skipped and reported.
 *   seq_len           [B] int32 tokens present.
 *   window_tokens     w, 0 <= w <= T_cap.
 *   gates             [B][H_q][3] fp32 = (g_c, g_s, g_w) per query head.
 *   O                 [B][H_q][128] bf16, written.
 *   workspace         needed by the branch grid only (NULL is fine otherwise): device
 *                     memory of sparse_decode_attn_nsa_workspace_size() bytes, per-pair
 *                     arrival counters, then the three branch outputs (fp32).  It must
 *                     be all zero before the first call; every call returns the
 *                     counters to zero.  Calls that share it must not overlap.
 *   n_split           CTAs per pair (per branch in the branch grid): 1, 2, 4 or 8;
 *                     0 = chosen from the SM count.
 *   flags             SPARSE_ATTN_BLOCKS_READY (as for sparse_decode_attn) and / or
 *                     SPARSE_NSA_BRANCH_GRID, or 0.
 * One launch runs the three branches (the notes run three kernels).  For G <= 8 the
 * launch is fully fused: one cluster of CTAs per pair streams the slices of all three
 * branches, keeps one softmax state per branch and forms the gated sum after one
 * merge through distributed shared memory; no intermediate reaches HBM.  For G > 8,
 * or with SPARSE_NSA_BRANCH_GRID, each branch is its own cluster (grid z = branch),
 * the branch outputs go to the workspace and the last CTA of the pair applies the
 * gates.  G = H_q / H_kv <= 16.
 */
SPARSE_API int sparse_decode_attn_nsa(const uint16_t *Q, const uint16_t *k_cache,
                                      const uint16_t *v_cache, long long T_cap,
                                      const uint16_t *khat, const uint16_t *vhat, int N_cap,
                                      int cmp_len, int cmp_stride, const int *blk_idx, const int *count, int k_tot,
                                      const int *seq_len, int B, int H_q, int H_kv,
                                      long long window_tokens, const float *gates, float scale,
                                      uint16_t *O, void *workspace, size_t workspace_bytes,
                                      int n_split, unsigned flags, int *status, void *stream);

/*
 * sparse_nsa_compress -- NSA's overlapping compression ([SparDA] background eq.(4) with
 * the inference kernel 32 and stride 16 of its §4.4; [SSV] "NSA" branch 1): after
 * tokens [len_before, len_before + n_new) are in the caches, writes the rows of every
 * window they complete,
 *     khat[p][j] = bf16(mean of k_cache[p][s*j .. s*j + l)),  vhat likewise,
 * for W(len_before) <= j < W(len_before + n_new), W(len) = floor((len - l) / s) + 1
 * (0 below l).  Call it after the append of those tokens; n_new = 0 writes nothing.
 *   k_cache, v_cache  [B][H_kv][T_cap][128] bf16, read.
 *   khat, vhat        [B][H_kv][n_rows_cap][128] bf16, written (rows j only).
 *   cmp_len l, cmp_stride s   1 <= s <= l <= 1024.
 */
SPARSE_API int sparse_nsa_compress(const uint16_t *k_cache, const uint16_t *v_cache, long long T_cap,
                                   int B, int H_kv, long long len_before, int n_new, int cmp_len,
                                   int cmp_stride, uint16_t *khat, uint16_t *vhat, int n_rows_cap,
                                   void *stream);

/*
 * sparse_nsa_select -- NSA's routing over its compressed keys ([SSV] "NSA three-branch
 * math" steps 1-2; the per-head softmax summed over the GQA group and the max-pooling
 * onto the selection grid of [SparDA] §4.3-§4.4 / InfLLM-V2):
 *     a^h_j = scale * q_h . khat_j   (j < R compressed rows, as sparse_decode_attn_nsa),
 *     p_j   = sum_h softmax_j(a^h),
 *     s_b   = max { p_j : row j's tokens meet block b's [64b, 64b + 64) }, 0 if none,
 * then B_init ∪ B_local ∪ top-k of the 64-token blocks b < N_b = ceil(len / 64) as
 * sparse_select_topk writes them (ties to the lower block).  The scores are computed on
 * the bf16 tensor cores from the bf16 rows, exactly as the compressed branch scores
 * them; with cmp_len = cmp_stride = 0 the rows are the blocks themselves.
 *   Q           [B][N_q][H_q][128] bf16: N_q queries per batch element, each routed on
 *               its own (N_q = 1 at decode; the verification queries of [SSV]'s refresh
 *               layers, whose lists the reuse layers then take as they are).
 *   khat        [B][H_kv][n_rows_cap][128] bf16.
 *   idx_out     [B][H_kv][N_q][k_tot] int32;  count_out [B][H_kv][N_q] int32.
 * G = H_q / H_kv <= 16; B * H_kv * N_q <= 65535.
 */
SPARSE_API int sparse_nsa_select(const uint16_t *Q, const uint16_t *khat, int n_rows_cap, int cmp_len,
                                 int cmp_stride, const int *seq_len, int B, int N_q, int H_q, int H_kv,
                                 float scale, int n_init, int n_local, int k, int *idx_out,
                                 int *count_out, int k_tot, int *status, void *stream);

/* sparse_decode_attn_nsa: run the branch grid (see `flags`) even when G <= 8. */
#define SPARSE_NSA_BRANCH_GRID 4u

/* Bytes of the sparse_decode_attn_nsa workspace for these sizes; 0 if they are invalid. */
SPARSE_API size_t sparse_decode_attn_nsa_workspace_size(int B, int H_q, int H_kv);

/*
 * sparse_gather_offloaded -- [SparDA] §4.5 (persistent prefetch of selected blocks,
 * re-designed as a gather kernel on the copy stream).  Copies the K and V rows of
 * block idx[p][i] (i < count[p]) of every pair from the host cache into slot i of the
 * staging ring: ring[p][i][r][:] = cache[p][64 * idx[p][i] + r][:], rows at or past
 * T_host written as zero.  After its copies every CTA adds 1 to *ready_flag (release,
 * device scope), so the word grows by n_ctas per call.
 *   k_host, v_host  [B][H_kv][T_host][128] bf16 in pinned host memory mapped into the
 *                   device address space (or any device-accessible memory).
 *   idx, count      as written by sparse_select_topk ([B*H_kv][k_tot], [B*H_kv]).
 *   k_ring, v_ring  [B*H_kv][k_tot][64][128] bf16 device memory (one ring slot).
 *   ready_flag      optional uint32 device word.
 *   n_ctas          gather CTAs (1..1024); 0 = chosen from the SM count.
 */
SPARSE_API int sparse_gather_offloaded(const uint16_t *k_host, const uint16_t *v_host,
                                       long long T_host, const int *idx, const int *count,
                                       int k_tot, int B, int H_kv, uint16_t *k_ring,
                                       uint16_t *v_ring, unsigned *ready_flag, int n_ctas,
                                       int *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_POOL_H */

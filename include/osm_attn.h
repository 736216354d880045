/*
 * osm_attn.h -- C ABI of libosmattn.so: exact attention forward with the online softmax, and
 * the standalone single-pass row softmax, on NVIDIA GB300 (sm_103a).
 *
 * All pointers are DEVICE pointers (CUDA global memory) unless a comment says otherwise.
 * The caller owns every buffer; the library allocates no device memory in any call listed
 * here.  It caches host-side kernel attributes and the CUDA driver entry point it needs for
 * TMA descriptors.  Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 * NULL is the legacy default stream) and returns an fa_status code.  Argument errors are
 * found on the host before anything is launched.
 *
 * One process drives one GPU: the cached kernel attributes and the address of the device
 * status word are taken for the device current at the first call that needs them, so every
 * call must be made with that same device current (run one process per GPU).
 */
#ifndef OSM_ATTN_H
#define OSM_ATTN_H

#include <stdint.h>

/* Only the functions declared here are exported from the shared library. */
#if defined(__GNUC__)
#define OSM_ATTN_API __attribute__((visibility("default")))
#else
#define OSM_ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null, negative or inconsistent sizes, misaligned pointer,
                               non-finite or non-positive scale, O aliasing an input */
    FA_ERR_UNSUPPORTED = 2, /* a valid request this build does not serve (d not 64/128) */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch error, no device) */
    FA_ERR_TIMEOUT = 4,     /* a kernel gave up a bounded wait (reported by
                               osm_attn_device_status) */
    FA_ERR_SCRATCH_LIMIT = 5 /* fa_fwd_splitkv_noalloc: the partial states of this shape do not
                                fit in the library's fixed scratch array */
} fa_status;

/*
 * fa_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V and LSE, for every (b, h, i).
 *
 * Defines the operation of "How FlashAttention avoids storing the giant score table"
 * (spicyshark.co, Online softmax lesson), section "From softmax to attention": the score of
 * key j for query i is s_ij = scale * (q_i . k_j); the output is the softmax-weighted sum of
 * the value rows, O_i = sum_j exp(s_ij - m_i) v_j / l_i with m_i = max_j s_ij and
 * l_i = sum_j exp(s_ij - m_i).  It is computed tile by tile with the running max / running
 * sum / rescaled accumulator of that section's block recipe (and of "kbwen.com
 * FlashAttention", sections "Two blocks" and "More than two blocks"), with the divide by l
 * deferred to the end, so the N x N score matrix never reaches device memory.
 *
 *   Q, K, V  bf16, [B, H, N, d] contiguous (d innermost), 16-byte aligned, read only.
 *   O        bf16, [B, H, N, d] contiguous, 16-byte aligned, written; must not be Q, K or V.
 *   LSE      fp32, [B, H, N], 4-byte aligned, written; may be NULL (not written).
 *            LSE_i = m_i + ln l_i, the natural-log log-sum-exp of the SCALED scores.
 *   B, H, N  batch, heads, sequence length (queries = keys = N); any N >= 0.
 *            B*H*N == 0 is a no-op returning FA_OK.
 *   d        head dimension: 64 or 128 (other values: FA_ERR_UNSUPPORTED).
 *   scale    finite and > 0 (typically 1/sqrt(d)).
 *   causal   0: every key; non-zero: key j is allowed for query i only when j <= i.
 *   stream   cudaStream_t, or NULL.
 * Precision: bf16 inputs, fp32 accumulation of both products, probabilities rounded to bf16
 * for the second product, fp32 running max/sum, bf16 output, fp32 LSE.
 */
OSM_ATTN_API int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                        void* stream);

/*
 * fa_fwd_host -- fa_fwd with its inputs and outputs in host memory, the host <-> device
 * copies overlapped with the attention.
 *
 * Same computation as fa_fwd (the lesson's "From softmax to attention"; each (b, h) is its own
 * problem, "The implementation").  The B*H heads are cut into n_chunks groups of consecutive
 * heads, and each group is pipelined:
 *   1. its Q, K, V are copied from host to the device staging buffers, on an internal stream;
 *   2. fa_fwd runs on those heads once they have landed, on `stream`;
 *   3. its O and LSE are copied back once the group is done, on a second internal stream.
 * So the next group's inputs and the previous group's outputs move while a group computes.
 *
 *   Q_host, K_host, V_host  bf16 [B, H, N, d] in host memory, read.  Page-locked memory
 *            (cudaHostAlloc, cudaHostRegister) lets the copies overlap; pageable memory is
 *            correct but serialises them.
 *   O_host   bf16 [B, H, N, d] in host memory, written.
 *   LSE_host fp32 [B, H, N] in host memory, written; NULL exactly when LSE_dev is NULL.
 *   Q_dev, K_dev, V_dev, O_dev  device buffers of the same shape (16-byte aligned, none
 *            overlapping another), LSE_dev fp32 [B, H, N] device (4-byte aligned) or NULL:
 *            staging owned by the caller, overwritten (O_dev and LSE_dev end holding O, LSE).
 *   B, H, N, d, scale, causal  as fa_fwd.
 *   n_chunks 0: chosen here (one group per 12 MB of Q, K, V, 1 to 16 groups); 1 .. 64
 *            groups otherwise (more groups than heads means one head per group; above 64 is
 *            FA_ERR_INVALID_ARG).
 *   stream   cudaStream_t or NULL.  The work is ordered after everything issued to `stream`
 *            before the call, and everything issued to `stream` after the call waits for all
 *            of it, the copies back to the host included: synchronise `stream` before reading
 *            O_host or reusing any buffer.  Calls from several host threads are serialised
 *            while they enqueue.
 * Returns as soon as the work is enqueued.  B*H*N == 0 is a no-op.  Errors: as fa_fwd, plus
 * FA_ERR_INVALID_ARG for a NULL host pointer, LSE_host without LSE_dev or the reverse, or
 * overlapping device buffers; FA_ERR_CUDA when a copy, an internal stream or an event fails.
 */
OSM_ATTN_API int fa_fwd_host(const void* Q_host, const void* K_host, const void* V_host,
                             void* O_host, float* LSE_host, void* Q_dev, void* K_dev,
                             void* V_dev, void* O_dev, float* LSE_dev, int64_t B, int64_t H,
                             int64_t N, int64_t d, float scale, int causal, int64_t n_chunks,
                             void* stream);

/*
 * fa_fwd_splitkv -- attention of Nq queries against Nk keys with the keys cut into n_splits
 * contiguous ranges that are processed in parallel (Flash-Decoding), then combined.
 *
 * The same lesson, section "Where this is used in practice" (Flash-Decoding splits the keys
 * across several workers when there are few queries and combines the partial results) and
 * the two-worker merge at the end of "From softmax to attention": each range yields its
 * normalised partial output O_s and log-sum-exp LSE_s; the combine takes M = max_s LSE_s,
 * w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s and LSE = M + ln sum_s w_s.
 *
 *   Q        bf16 [B, H, Nq, d]; K, V bf16 [B, H, Nk, d]; all contiguous, 16-byte aligned.
 *   O, LSE   as fa_fwd, shaped [B, H, Nq, d] and [B, H, Nq]; LSE may be NULL.
 *   causal   non-zero: the Nq queries are the last Nq of the Nk positions, so query i sees keys
 *            j <= i + (Nk - Nq) (Nq == Nk: the usual mask; a query with no allowed key gets
 *            O = 0 and LSE = -inf).
 *   n_splits 1 .. 256, normally the value fa_fwd_splitkv_plan returns.  1 runs the one-pass
 *            kernel directly (no workspace needed).
 *   ws_O     fp32 workspace of n_splits * B*H*Nq * d floats, 16-byte aligned (n_splits > 1);
 *   ws_LSE   fp32 workspace of n_splits * B*H*Nq floats (n_splits > 1).  Both owned by the
 *            caller, overwritten, and must not overlap any input or output.
 * Nk == 0 writes O = 0 and LSE = -inf; B*H*Nq == 0 is a no-op.  Errors as fa_fwd.
 */
OSM_ATTN_API int fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O,
                                float* LSE, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                                int64_t d, float scale, int causal, int64_t n_splits,
                                float* ws_O, float* ws_LSE, void* stream);

/*
 * fa_fwd_gqa -- fa_fwd_splitkv with grouped key/value heads and per-sequence key lengths.
 *
 * Grouped heads: "FlashAttention" (paweldubiel.com notes), section "Averaging block results is
 * not enough" (grouped-query attention keeps fewer key/value heads and combines with the tiled
 * computation): H_kv key/value heads serve the H query heads, query head h of a sequence
 * reading key/value head h / (H / H_kv) of it.  Key lengths: the masking of "How FlashAttention
 * avoids storing the giant score table" (spicyshark.co, Online softmax lesson), section "The
 * implementation" (a position a query may not look at gets score -inf, and a block whose scores
 * are all -inf adds nothing): keys j >= kv_lens[b] of sequence b are masked, on top of the
 * causal mask when causal is set.  A query left with no key gets O = 0 and LSE = -inf.
 *
 *   Q, O     bf16 [B, H, Nq, d]; K, V bf16 [B, H_kv, Nk, d]; LSE fp32 [B, H, Nq] or NULL.
 *   H_kv     >= 1 and divides H (H_kv == H: every query head has its own key/value head).
 *   kv_lens  DEVICE pointer to B int32 key counts, 4-byte aligned, read only; NULL means Nk for
 *            every sequence.  Values are read by the kernel: below 0 counts as 0, above Nk as Nk.
 *   causal   as fa_fwd_splitkv: query i sees keys j <= i + (Nk - Nq), and j < kv_lens[b].
 *   n_splits, ws_O, ws_LSE  as fa_fwd_splitkv (fa_fwd_gqa_plan gives them; 1 runs one pass
 *            and needs no workspace).
 * Errors as fa_fwd_splitkv, plus FA_ERR_INVALID_ARG when H_kv does not divide H or kv_lens is
 * misaligned or overlaps an output.
 */
OSM_ATTN_API int fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk,
                            int64_t d, float scale, int causal, const int32_t* kv_lens,
                            int64_t n_splits, float* ws_O, float* ws_LSE, void* stream);

/*
 * fa_fwd_gqa_plan -- fa_fwd_splitkv_plan for fa_fwd_gqa: the number of key ranges and the
 * workspace for Q [B, H, Nq, d] against K, V [B, H_kv, Nk, d].  The kernel runs the H / H_kv
 * query heads that share a key/value head as one block of (H / H_kv) * Nq rows, so the choice
 * counts blocks, not heads.  n_splits = 0 lets the library choose.  Host pointers; errors as
 * fa_fwd_splitkv_plan, plus FA_ERR_INVALID_ARG when H_kv does not divide H.
 */
OSM_ATTN_API int fa_fwd_gqa_plan(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk,
                                 int64_t d, int64_t n_splits, int64_t* splits_out,
                                 int64_t* ws_o_floats, int64_t* ws_lse_floats);

/*
 * fa_fwd_splitkv_plan -- the number of key ranges fa_fwd_splitkv should use for this shape and
 * the workspace it then needs.  n_splits = 0 asks the library to choose (enough CTAs for about
 * eight waves on this GPU, at most 64 ranges and one key tile per range); 1 .. 256 is clamped to
 * the number of 128-key tiles.  Writes *splits_out (0 when Nk == 0), *ws_o_floats and
 * *ws_lse_floats (both 0 when one range suffices).  All three are HOST pointers.  Queries the
 * current CUDA device for its SM count when choosing.
 */
OSM_ATTN_API int fa_fwd_splitkv_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                                     int64_t d, int64_t n_splits, int64_t* splits_out,
                                     int64_t* ws_o_floats, int64_t* ws_lse_floats);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without any workspace argument and without any
 * device allocation (the pages have no counterpart: it serves callers that cannot allocate
 * device memory during a call, such as a plugin or custom-operator hook whose host framework
 * forbids allocation there, or a latency-critical decode loop).
 *
 * Same arguments and results as fa_fwd_splitkv, minus ws_O / ws_LSE; n_splits = 0 lets the
 * library choose as fa_fwd_splitkv_plan does.  The per-range partial states live in a fixed
 * array of 4 Mi floats (16 MiB) that every GPU loading the library holds until the process
 * exits: a shape needs splits * B*H*Nq * (d + 1) floats of it, where splits is the count
 * fa_fwd_splitkv_plan returns for the same B, H, Nq, Nk, d and n_splits (the library's choice
 * when n_splits = 0, and never more than the key tiles, ceil(Nk / 128)); a caller can check a
 * shape in advance with that call.  A shape that needs more returns FA_ERR_SCRATCH_LIMIT
 * without launching anything.  The first call made with a device current resolves that
 * device's array address (cudaGetSymbolAddress) and caches it for the life of the process;
 * make that first call before any stream capture.  The cached address belongs to the device's
 * context as it was then: after cudaDeviceReset of that device the process must not call this
 * entry point again.  All calls on a device share the one array: calls that can overlap on the
 * GPU (different streams, or streams not ordered with each other) race on it and must be
 * serialised by the caller.  The array keeps the last call's contents; every entry a call
 * reads is written earlier in the same call, so nothing needs clearing between calls -- unless
 * a kernel of the call gave up a bounded wait: then the combine may read entries an earlier
 * call left behind, and O and LSE of that call are undefined.  osm_attn_device_status reports
 * that case (FA_ERR_TIMEOUT); a caller that needs to know must read it after the call.
 */
OSM_ATTN_API int fa_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O,
                                        float* LSE, int64_t B, int64_t H, int64_t Nq,
                                        int64_t Nk, int64_t d, float scale, int causal,
                                        int64_t n_splits, void* stream);

/*
 * fa_fwd_mask -- fa_fwd with an explicit mask: an arbitrary set of (query, key) pairs excluded.
 *
 * "How FlashAttention avoids storing the giant score table" (spicyshark.co, Online softmax
 * lesson), section "The implementation": a position a query may not look at gets score -inf,
 * a block whose scores are all -inf adds nothing, and a row with no allowed key keeps the
 * empty state (here O = 0, LSE = -inf).  Key j is allowed for query i of head (b, h) when bit
 * j % 32 of word j / 32 of the row at
 *     mask + b * mask_b_stride + h * mask_h_stride + i * W,   W = 4 * ceil(Nk / 128)
 * is set, and, when causal is set, j <= i + (Nk - Nq).
 *
 *   Q, O     bf16 [B, H, Nq, d]; K, V bf16 [B, H, Nk, d]; LSE fp32 [B, H, Nq] or NULL.
 *   mask     DEVICE pointer to uint32 words, 16-byte aligned, read only; each row holds W words
 *            (the bits past Nk are ignored).
 *   mask_b_stride, mask_h_stride   words between the masks of consecutive sequences and heads,
 *            >= 0 and multiples of 4; 0 repeats one mask over all sequences or heads (e.g.
 *            a [Nq, W] mask shared by every head of every sequence).
 *   tile_map optional DEVICE workspace of tile_map_words uint32 words (at least what
 *            fa_fwd_mask_plan returns), 4-byte aligned, owned by the caller, apart from every
 *            input and output; NULL skips nothing.  When given, a pre-pass on the same stream
 *            writes into it, for every 128-row query tile and mask instance, which 128-key
 *            tiles hold an allowed key, and the attention then skips the tiles that hold none
 *            (a block of -inf scores adds nothing, so the results are those without skipping
 *            up to the order of the floating-point sums).  Its contents are rewritten by every
 *            call; calls that overlap on the GPU need their own.
 * Errors as fa_fwd_gqa, plus FA_ERR_INVALID_ARG for a NULL or misaligned mask, bad strides, a
 * mask reaching O or LSE, or a tile map that is misaligned, too small or overlaps an input or
 * output.
 */
OSM_ATTN_API int fa_fwd_mask(const void* Q, const void* K, const void* V, void* O, float* LSE,
                             int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                             float scale, int causal, const uint32_t* mask,
                             int64_t mask_b_stride, int64_t mask_h_stride, uint32_t* tile_map,
                             int64_t tile_map_words, void* stream);

/*
 * fa_fwd_mask_plan -- the size of fa_fwd_mask's tile map for a shape and mask strides: one row
 * of ceil(ceil(Nk / 128) / 32) words per 128-row query tile and mask instance (B instances
 * when mask_b_stride != 0, times H when mask_h_stride != 0).  Host pointer; writes
 * *tile_map_words.  FA_ERR_INVALID_ARG for negative or oversized arguments or a NULL output.
 */
OSM_ATTN_API int fa_fwd_mask_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                                  int64_t mask_b_stride, int64_t mask_h_stride,
                                  int64_t* tile_map_words);

/*
 * fa_fwd_gqa_mask -- the attention with every option at once: grouped key/value heads and
 * per-sequence key lengths (as fa_fwd_gqa), an explicit mask with its optional tile map (as
 * fa_fwd_mask), and one pass or split keys (as fa_fwd_splitkv).
 *
 * "How FlashAttention avoids storing the giant score table" (spicyshark.co, Online softmax
 * lesson): a key that a query may not look at -- masked, past its sequence's length, or after
 * it when causal -- gets score -inf ("The implementation"), and partial states over disjoint
 * key ranges combine with the two-worker merge ("From softmax to attention"; "Where this is
 * used in practice"); "FlashAttention" (paweldubiel.com notes), "Averaging block results is not
 * enough": grouped-query attention combines with the tiled computation.  Key j is allowed for
 * query i of head (b, h) when its mask bit is set (the mask layout of fa_fwd_mask), when
 * j < kv_lens[b] (if kv_lens is given), and, when causal is set, j <= i + (Nk - Nq).  Query head
 * h reads key/value head h / (H / H_kv).  A row with no allowed key gets O = 0, LSE = -inf.
 *
 *   Q, O     bf16 [B, H, Nq, d]; K, V bf16 [B, H_kv, Nk, d]; LSE fp32 [B, H, Nq] or NULL.
 *   kv_lens  optional DEVICE int32 [B] (clamped to [0, Nk]); NULL: every key is valid.
 *   mask, mask_b_stride, mask_h_stride, tile_map, tile_map_words   as fa_fwd_mask (strides
 *            over query heads: the mask of (b, h) starts at mask + b * mask_b_stride +
 *            h * mask_h_stride); the tile map's size comes from fa_fwd_gqa_mask_plan.
 *   n_splits 1: one pass, no workspace; > 1: that many key ranges, the partial states in the
 *            caller's ws_O (fp32 [n_splits, B*H*Nq, d], 16-byte aligned) and ws_LSE (fp32
 *            [n_splits, B*H*Nq]), as fa_fwd_splitkv.  fa_fwd_gqa_mask_plan chooses a count.
 * The call is asynchronous on `stream`; the mask, tile map and workspaces are the caller's.
 * Errors: the union of fa_fwd_gqa's and fa_fwd_mask's.
 */
OSM_ATTN_API int fa_fwd_gqa_mask(const void* Q, const void* K, const void* V, void* O,
                                 float* LSE, int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                 int64_t Nk, int64_t d, float scale, int causal,
                                 const int32_t* kv_lens, const uint32_t* mask,
                                 int64_t mask_b_stride, int64_t mask_h_stride, uint32_t* tile_map,
                                 int64_t tile_map_words, int64_t n_splits, float* ws_O,
                                 float* ws_LSE, void* stream);

/*
 * fa_fwd_gqa_mask_plan -- for fa_fwd_gqa_mask: the key ranges to use (n_splits = 0: chosen for
 * about eight waves of work items, as fa_fwd_splitkv_plan; > 0: that request, capped at the key
 * tiles), the workspace sizes in floats for that count (0 for one pass), and the tile map's
 * size in words (as fa_fwd_mask_plan).  Host pointers; FA_ERR_INVALID_ARG for negative or
 * oversized arguments, H not a multiple of H_kv, or a NULL output; FA_ERR_UNSUPPORTED for
 * d not in {64, 128}.
 */
OSM_ATTN_API int fa_fwd_gqa_mask_plan(int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                      int64_t Nk, int64_t d, int64_t mask_b_stride,
                                      int64_t mask_h_stride, int64_t n_splits,
                                      int64_t* splits_out, int64_t* ws_o_floats,
                                      int64_t* ws_lse_floats, int64_t* tile_map_words);

/*
 * fa_bwd -- the gradients dQ, dK, dV of fa_fwd's attention for an output gradient dO.
 *
 * "FlashAttention" (paweldubiel.com notes), "Mechanism and details", and "How FlashAttention
 * avoids storing the giant score table" (spicyshark.co, Online softmax lesson), "Where this is
 * used in practice": training recomputes the scores in the backward pass instead of storing
 * them.  With the forward's LSE the shares are P_ij = exp(scale q_i . k_j - LSE_i); the
 * gradients are the derivative of the definition: D_i = dO_i . O_i, dP_ij = dO_i . v_j,
 * dS_ij = P_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i,
 * dV_j = sum_i P_ij dO_i (causal: only the pairs j <= i).
 *
 *   Q, K, V, O, dO  bf16 [B, H, N, d] contiguous, 16-byte aligned, read only (O and LSE as
 *            fa_fwd wrote them for the same Q, K, V, scale and causal).
 *   LSE      fp32 [B, H, N], read only.
 *   dQ, dK, dV  bf16 [B, H, N, d], 16-byte aligned, written.
 *   ws_D     fp32 workspace of B*H*N floats (D_i), 4-byte aligned, owned by the caller and
 *            overwritten.  No output or the workspace may overlap an input or another output.
 *   d        64 or 128; scale finite and > 0.  B*H*N == 0 is a no-op.
 * Precision: P and dS are rounded to bf16 for the tensor-core products, which accumulate in
 * fp32 in a fixed order (the results repeat bit for bit).  Errors as fa_fwd.
 */
OSM_ATTN_API int fa_bwd(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                        float* ws_D, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                        int causal, void* stream);

/*
 * fa_bwd_gqa -- fa_bwd for the forward of fa_fwd_gqa: grouped key/value heads and per-sequence
 * key lengths (square attention, Nq = Nk = N).
 *
 * The same passages as fa_bwd; grouped-query attention ("FlashAttention" (paweldubiel.com
 * notes), "Averaging block results is not enough") shares one key/value head among the H / H_kv
 * query heads of a group, so its key and value gradients are the sums over those query heads;
 * a key at or past its sequence's length takes no part ("How FlashAttention avoids storing the
 * giant score table" (spicyshark.co), "The implementation"): its gradients are exactly 0, and a
 * query with no allowed key (a sequence of length 0) has dQ = 0.
 *
 *   Q, O, dO  bf16 [B, H, N, d]; K, V bf16 [B, H_kv, N, d], H_kv dividing H (query head h reads
 *            key/value head h / (H / H_kv)); all contiguous, 16-byte aligned, read only; O and
 *            LSE as fa_fwd_gqa wrote them for the same inputs, key lengths, scale and causal.
 *   LSE      fp32 [B, H, N], read only.
 *   dQ       bf16 [B, H, N, d]; dK, dV bf16 [B, H_kv, N, d]; 16-byte aligned, written.
 *   ws_D     fp32 workspace of B*H*N floats, as fa_bwd.
 *   kv_lens  optional DEVICE int32 [B], 4-byte aligned, read only (clamped to [0, N]); NULL:
 *            every key is valid.
 * Errors as fa_bwd, plus FA_ERR_INVALID_ARG when H_kv does not divide H or kv_lens is
 * misaligned or overlaps an output.
 */
OSM_ATTN_API int fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            float* ws_D, int64_t B, int64_t H, int64_t H_kv, int64_t N, int64_t d,
                            float scale, int causal, const int32_t* kv_lens, void* stream);

/*
 * osm_softmax_topk -- the k largest entries of every row with their softmax shares, in one
 * read of the row.
 *
 * "How FlashAttention avoids storing the giant score table" (spicyshark.co, Online softmax
 * lesson), section "Where this is used in practice": the online normaliser also serves softmax
 * fused with top-k selection, keeping only the k largest scores.  For row r:
 * indices[r, 0..k) are the columns of the k largest x[r, :] in descending order (ties: the
 * smaller column first), values[r, t] = exp(x[r, c] - m_r) / l_r for c = indices[r, t] (m_r
 * the row max, l_r = sum_j exp(x[r, j] - m_r)), and lse[r] = m_r + ln l_r.
 *
 *   x        fp32 [rows, cols] contiguous, 4-byte aligned, read only; no NaN (NaN rows give
 *            unspecified results).  A row of -inf gives values 0 and lse -inf.
 *   k        1 .. min(cols, 1024) (k > 1024: FA_ERR_UNSUPPORTED; k > cols: FA_ERR_INVALID_ARG).
 *            k <= 32 reads each row once (a warp-wide list of the best k).  Larger k also
 *            reads each row once (its first 64 T columns twice, T = 256 threads up to
 *            k = 256, 512 above): a floor under the k-th largest value rises as the row
 *            streams by, and every entry at or above it goes into a buffer that is sorted at
 *            the end.  A row whose entries overflow the buffer (16 T of them; rows in
 *            ascending order, for one) is read once more against the final floor; rows where
 *            more than 16 T entries reach the final floor fall back to radix selection, five
 *            more passes.
 *   values   fp32 [rows, k], indices int32 [rows, k], lse fp32 [rows] or NULL; written; none
 *            may overlap x or each other.
 * rows == 0 is a no-op.  All pointers are device pointers; asynchronous on `stream`.
 */
OSM_ATTN_API int osm_softmax_topk(const float* x, int64_t rows, int64_t cols, int64_t k,
                                  float* values, int32_t* indices, float* lse, void* stream);

/*
 * osm_softmax -- y = softmax(x) of every row, single pass over HBM, and its log-sum-exp.
 *
 * Defines the operation of the same lesson, sections "The idea" and "The implementation":
 * the running maximum m and running sum l = sum exp(x - m), rescaled by exp(m_old - m_new)
 * whenever the maximum grows, give both statistics in one read; partial states of disjoint
 * parts of a row combine by the lesson's two-worker merge; y_j = exp(x_j - m) / l.  Rows up
 * to 16384 columns are read from HBM once and kept on chip for the write (one read, one
 * write per element); longer rows are read twice (statistics, then output), the lesson's
 * "online softmax with the output written".
 *
 *   x     fp32 [rows, cols] contiguous, 4-byte aligned, read only.
 *   y     fp32 [rows, cols] contiguous, written; may equal x (in place).
 *   lse   fp32 [rows] (m + ln l), written; may be NULL.
 *   rows, cols >= 0; rows*cols == 0 is a no-op (lse is not written).
 *   A row with no finite entry (all -inf) gives y = 0 and lse = -inf.
 */
OSM_ATTN_API int osm_softmax(const float* x, float* y, int64_t rows, int64_t cols,
                             float* lse, void* stream);

/* A static, human-readable name for a status code (never NULL). */
OSM_ATTN_API const char* fa_status_string(int status);

/*
 * osm_attn_device_status -- synchronises `stream`, then reads and clears the device status
 * word the kernels set when a bounded wait gives up (FA_OK when none did).  *status
 * (HOST pointer) receives the code; the return value is FA_OK or FA_ERR_CUDA.
 */
OSM_ATTN_API int osm_attn_device_status(void* stream, int* status);

/*
 * osm_attn_selftest_wait -- diagnostic for the bounded-wait error path (the pages have no
 * counterpart).  Launches one warp that waits, with the same bounded mbarrier wait the
 * attention kernel uses, on a barrier that nothing ever completes; after `timeout_us`
 * microseconds (1 .. 10 000 000) the wait gives up and records FA_ERR_TIMEOUT in the device
 * status word, which osm_attn_device_status then returns (and clears).  No GPU fault is
 * involved: the kernel exits normally and the context stays usable.  Returns FA_OK when the
 * launch succeeded, FA_ERR_INVALID_ARG for a timeout out of range, FA_ERR_CUDA otherwise.
 */
OSM_ATTN_API int osm_attn_selftest_wait(int64_t timeout_us, void* stream);

/* ABI version of this header (incremented on any incompatible change). */
OSM_ATTN_API int osm_attn_abi_version(void);

#define OSM_ATTN_ABI_VERSION 10

#ifdef __cplusplus
}
#endif

#endif /* OSM_ATTN_H */

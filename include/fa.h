/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused attention forward library
 * (libfa_gb300.so).
 *
 * The library computes, for every batch entry b, query head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j  over visible j) * v_j
 *     LSE[b,h,i] = ln sum_{visible j} exp(scale * q_i . k_j)
 *
 * ("b200-flash-attention4-planner", section E step 1 fixes these semantics:
 * shapes, layout, head_dim, causal, GQA ratio, scale, output and LSE; its
 * section A1 "Streaming online softmax" is the tile-by-tile method the
 * kernels use: running row_max / row_sum, O rebased when the max grows,
 * divided by row_sum only at the end).
 *
 * Conventions shared by every entry point below:
 *   Layout    q, o : [batch, hq,  sq, head_dim]  bf16, contiguous (row-major)
 *             k, v : [batch, hkv, sk, head_dim]  bf16, contiguous
 *             lse  : [batch, hq,  sq]            fp32, contiguous
 *             bf16 is passed as raw 16-bit patterns.
 *   Pointers  q, k, v, o, lse and seqlens_k are DEVICE pointers of the
 *             current CUDA device.  All buffers are owned by the caller; the
 *             library neither frees nor retains them after the call returns.
 *             q, k, v and o must be 16-byte aligned (TMA requirement).
 *   GQA       hq must be a multiple of hkv; query head h reads key/value head
 *             h / (hq / hkv) (consecutive query heads share a key/value head).
 *   Lengths   seqlens_k: device int32[batch] of valid key counts L_b, or NULL
 *             (then L_b = sk).  Values are clamped to [0, sk] on the device.
 *             Key/value rows j >= L_b are never read (their contents may be
 *             anything, including NaN).
 *   Causal    bottom-right aligned: key j is visible to query row i iff
 *             j <= i + (L_b - sq); for sq == sk == L_b this is the usual
 *             lower-triangular mask.  A row with no visible key gets O = 0
 *             and LSE = -infinity.
 *   Scale     must be finite and > 0 (typically 1/sqrt(head_dim)).
 *   LSE units natural log of the sum of exp(scaled score).
 *   Streams   work is enqueued on `stream` (NULL = legacy default stream);
 *             the calls are asynchronous and never synchronise the device.
 *   Errors    argument checks run on the host before anything is enqueued;
 *             on any error nothing is launched.  No C++ exception crosses
 *             this interface.  A kernel wait that exceeds its time limit
 *             makes the kernel finish early and records FA_ERR_TIMEOUT in a
 *             device error word, read by fa_get_device_error() (the word,
 *             from fa_get_device_error_word(), holds the wait site in bits
 *             0-15 and the CTA index in bits 16-31).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                    /* same type as cudaStream_t */
typedef struct CUstream_st *fa_stream_t;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, hq % hkv != 0,
                                 bad scale, decode with sq > FA_DECODE_MAX_SQ */
    FA_ERR_UNSUPPORTED = 2,   /* head_dim not 64/96/128/256/512 (prefill) or
                                 not 64/128/256 (decode); device not sm_103 */
    FA_ERR_MISALIGNED = 3,    /* q, k, v or o not 16-byte aligned */
    FA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = 5        /* a kernel wait ran out of time (device word) */
} fa_status;

/* Largest query count per sequence accepted by the decode entry points. */
#define FA_DECODE_MAX_SQ 16

/*
 * Prefill forward.  Runs the warp-specialised tcgen05/TMEM kernel for
 * head_dim in {64, 96, 128, 256, 512}: a TMA producer warp streams K/V tiles
 * through an mbarrier ring, one warp issues the score MMA (S = Q K^T) and the
 * value MMA (O += P V) into tensor memory, softmax warpgroups turn S into P
 * with exp2, and a correction/epilogue warpgroup rebases O and writes O and
 * LSE ("b200-flash-attention4-planner", section A1 "Role example" and
 * section E steps 3-8).  One CTA per query block (two at head_dim 512, each
 * computing the scores over all 512 dimensions -- the head dimension's
 * sub-tiles summed before the softmax, "STAGE_D.md" hd=512 -- and one
 * 256-column half of O; LSE is stored by the first).  At head_dim 256, when
 * no query block is split and the sequences are not packed, one persistent
 * CTA per SM processes the query blocks in turn instead (heaviest first over
 * the SMs, keeping its pipeline state from one block to the next and
 * storing each block's O while the next one starts).  At head_dim 96 and 128
 * without a window, paged caches or packed sequences (causal or not), a
 * persistent kernel with 256-key score blocks and query blocks
 * of 128 rows runs instead: one N = 256 score MMA per K-step, P in tensor
 * memory columns of its own, the next block's score MMA issued while the
 * softmax of this one runs, each row's softmax split over two warpgroups
 * (128 keys each) that exchange their block maxima; with GQA and short
 * queries (sq <= 64) that kernel packs the query heads of a kv group into
 * one 128-row tile (P heads x 128 / P positions, P a power of two dividing
 * hq / hkv: see fa_debug_prefill_plan_gqa), so that they share each K/V tile
 * ("b200-flash-attention4-planner" E.7, head-packed GQA); when its
 * non-causal units fill at most half the SMs, it cuts each into 2-8 pieces
 * along the key axis, one per CTA, merged on the device.  For the other
 * non-causal problems the query blocks of the last, partial wave are split
 * along the key axis over several CTAs and merged on the device (see
 * fa_debug_prefill_plan_ex).  A split launch
 * takes a stream-ordered scratch allocation (cudaMallocAsync, freed
 * with cudaFreeAsync on the same stream) of at most SMs * 130 KB (head_dim
 * 128; in proportion for other head dims).
 * Sizes: batch, hq, hkv, sq, sk >= 0 (any zero size is a no-op returning
 * FA_OK, except sk == 0 with non-empty outputs, which writes O = 0 and
 * LSE = -inf); batch <= 65535, hq <= 65535.
 */
fa_status fa_fwd_prefill(const void *q, const void *k, const void *v, void *o,
                         float *lse, int batch, int hq, int hkv, int sq, int sk,
                         const int *seqlens_k, int head_dim, float scale,
                         int causal, fa_stream_t stream);

/*
 * Prefill with a sliding window and/or attention sinks ("2026-05-28_STATUS.md":
 * D3 "SWA length mask", D4 "causal mask on SWA", D5c "sink merge").
 *   window  > 0: key j is visible to query row i only if j > i + (L_b - sq) -
 *           window (with causal: the row's own key and the window - 1 keys
 *           before it); <= 0: no window.  Query blocks with a window are not
 *           split across CTAs.
 *   sinks   NULL, or a device float[hq] (4-byte aligned) of per-query-head
 *           sink logits in the units of the scaled score: each row's softmax
 *           becomes e^{s_j} / (e^{sinks[h]} + sum_j e^{s_j}); the sink
 *           carries no value, and LSE includes it (a row with no visible key
 *           gets O = 0 and LSE = sinks[h]).
 * Everything else as fa_fwd_prefill (which is this call with window 0 and
 * no sinks).
 */
fa_status fa_fwd_prefill_ex(const void *q, const void *k, const void *v, void *o,
                            float *lse, int batch, int hq, int hkv, int sq, int sk,
                            const int *seqlens_k, int head_dim, float scale, int causal,
                            int window, const float *sinks, fa_stream_t stream);

/*
 * Decode forward (few queries per sequence against a long key/value cache).
 * Split-KV ("fa4-sm120-research" lists SplitKV among the features its kernels
 * lack; "STAGE_D.md" gives the merge of attention over disjoint key sets by
 * their LSE): each CTA handles one (batch entry, key/value head, key split),
 * streams its keys with coalesced 16-byte loads, packs all query heads of the
 * group onto the tensor-core M dimension and writes a partial (O_s, LSE_s);
 * a second kernel combines the splits, weighting each by exp(LSE_s).  The
 * merge is exact because the splits cover disjoint key sets.
 * Same arguments as fa_fwd_prefill; sq must be 1..FA_DECODE_MAX_SQ and
 * head_dim one of 64, 128, 256.  The partials live in a workspace that the
 * call allocates and frees stream-ordered (cudaMallocAsync/cudaFreeAsync on
 * `stream`).  At head_dim 128 with (hq / hkv) * sq >= 32 query rows per
 * key/value head (several queries of a GQA group), this call and
 * fa_fwd_decode_ex without a window run the prefill kernel with the group's
 * query heads packed into one tile instead (the same result as
 * fa_fwd_prefill / fa_fwd_prefill_ex, bit for bit; it allocates a workspace
 * only when it splits its units along the keys): past 16 rows per
 * key/value head the split kernel is bound by its tensor-core work, the
 * packed kernel by HBM.  fa_fwd_decode_splits, the paged and the
 * no-allocation entry points always run the split kernel.
 */
fa_status fa_fwd_decode(const void *q, const void *k, const void *v, void *o,
                        float *lse, int batch, int hq, int hkv, int sq, int sk,
                        const int *seqlens_k, int head_dim, float scale,
                        int causal, fa_stream_t stream);

/*
 * Prefill / decode over paged K/V caches ("fa4-sm120-research" names paged
 * KV among the features its kernels lack; "2026-05-28_STATUS.md" lists a
 * paged cache in its KV-cache infrastructure).  The caches are
 *     k_cache, v_cache : [num_pages, hkv, page_size, head_dim] bf16, 16-byte
 *                        aligned, caller-owned;
 *     block_table      : device int32[batch, max_pages]: key j of sequence b
 *                        is row j % page_size of page
 *                        block_table[b * max_pages + j / page_size];
 *     seqlens_k        : device int32[batch], required: L_b keys of sequence
 *                        b (clamped to [0, max_pages * page_size]).
 * Only the pages that hold keys j < L_b are read (page indices outside
 * [0, num_pages) read as zeros in prefill and are clamped in decode).  The
 * prefill kernel loads 128-key tiles with TMA, so page_size must be a
 * multiple of 128 (else FA_ERR_UNSUPPORTED); decode takes any page_size >= 1.
 * Everything else as fa_fwd_prefill / fa_fwd_decode with sk = max_pages *
 * page_size.  Returns FA_ERR_INVALID_ARG for a NULL block table or seqlens_k,
 * or non-positive max_pages / page_size / num_pages.
 */
fa_status fa_fwd_prefill_paged(const void *q, const void *k_cache, const void *v_cache, void *o,
                               float *lse, int batch, int hq, int hkv, int sq,
                               const int *seqlens_k, const int *block_table, int max_pages,
                               int page_size, int num_pages, int head_dim, float scale,
                               int causal, fa_stream_t stream);
fa_status fa_fwd_decode_paged(const void *q, const void *k_cache, const void *v_cache, void *o,
                              float *lse, int batch, int hq, int hkv, int sq,
                              const int *seqlens_k, const int *block_table, int max_pages,
                              int page_size, int num_pages, int head_dim, float scale,
                              int causal, fa_stream_t stream);

/*
 * Prefill over packed variable-length sequences ("b200-flash-attention4-
 * planner", section B, lists variable-length packed sequences among the
 * extensions its forward design leaves open).  Sequence b owns query tokens
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key tokens
 * [cu_seqlens_k[b], cu_seqlens_k[b+1]); each sequence is attended on its own,
 * exactly as fa_fwd_prefill_ex with batch 1, sq = its query length and
 * sk = its key length (causal alignment bottom-right, the same window and
 * sink semantics).  Layouts (bf16, 16-byte aligned, caller-owned):
 *     q, o         : [total_q, hq, head_dim]   (token-major, heads adjacent)
 *     k, v         : [total_k, hkv, head_dim]
 *     lse          : [hq, total_q] fp32
 *     cu_seqlens_q : device int32[batch + 1], nondecreasing, [0] = 0,
 *                    [batch] = total_q; cu_seqlens_k likewise with total_k.
 * max_seqlen_q / max_seqlen_k must be at least every sequence's query / key
 * length (the launch covers max_seqlen_q query rows per sequence; rows of a
 * longer sequence beyond that are not written).  Offsets are clamped to
 * [0, total] on the device, so malformed offsets never address memory outside
 * the tensors.  Sequences without keys give O = 0 and LSE = -inf (or the
 * sink).  head_dim 64, 96, 128, 256 or 512.  Returns FA_ERR_INVALID_ARG for
 * negative sizes, NULL offsets, or max_seqlen_q = 0 with total_q > 0;
 * FA_ERR_MISALIGNED for offsets not 4-byte aligned.
 */
fa_status fa_fwd_prefill_varlen(const void *q, const void *k, const void *v, void *o,
                                float *lse, const int *cu_seqlens_q, const int *cu_seqlens_k,
                                int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                                int total_k, int hq, int hkv, int head_dim, float scale,
                                int causal, int window, const float *sinks,
                                fa_stream_t stream);

/*
 * Packed queries over paged K/V caches: the queries, O and LSE of
 * fa_fwd_prefill_varlen (q, o [total_q, hq, head_dim], lse [hq, total_q],
 * cu_seqlens_q [batch + 1]) with the keys of fa_fwd_prefill_paged (k_cache,
 * v_cache [num_pages, hkv, page_size, head_dim], block_table
 * [batch, max_pages], seqlens_k [batch] required, page_size a multiple of
 * 128).  Sequence b's query token t (0-based within the sequence) is row
 * t + seqlens_k[b] - Lq_b of the causal alignment, as everywhere: the typical
 * use is a chunk of new tokens whose keys, together with the earlier ones,
 * are already in the caches.  Same window, sink and error rules as the two
 * calls it combines.
 */
fa_status fa_fwd_prefill_varlen_paged(const void *q, const void *k_cache, const void *v_cache,
                                      void *o, float *lse, const int *cu_seqlens_q,
                                      const int *seqlens_k, const int *block_table,
                                      int max_pages, int page_size, int num_pages, int batch,
                                      int max_seqlen_q, int total_q, int hq, int hkv,
                                      int head_dim, float scale, int causal, int window,
                                      const float *sinks, fa_stream_t stream);

/*
 * Decode with a sliding window and/or attention sinks: the same window and
 * sink semantics as fa_fwd_prefill_ex (for sq = 1 the window keeps the last
 * `window` keys of each sequence).  Splits wholly below a row's window are
 * not read.  Everything else as fa_fwd_decode.
 */
fa_status fa_fwd_decode_ex(const void *q, const void *k, const void *v, void *o,
                           float *lse, int batch, int hq, int hkv, int sq, int sk,
                           const int *seqlens_k, int head_dim, float scale, int causal,
                           int window, const float *sinks, fa_stream_t stream);

/*
 * fa_fwd_decode with an explicit number of key splits (num_splits <= 0 picks
 * it automatically, exactly like fa_fwd_decode).  The splits partition
 * [0, sk) into equal chunks of a multiple of 64 keys; any split count gives
 * the same result up to rounding.
 */
fa_status fa_fwd_decode_splits(const void *q, const void *k, const void *v,
                               void *o, float *lse, int batch, int hq, int hkv,
                               int sq, int sk, const int *seqlens_k,
                               int head_dim, float scale, int causal,
                               int num_splits, fa_stream_t stream);

/*
 * Decode forward that allocates nothing (no counterpart in the source pages;
 * it exists for users of this library).
 *
 * Who needs it: callers that cannot allocate device memory while they run --
 * a serving loop that must not allocate once it is up (an allocation can
 * stall or fail at an unpredictable moment), a process whose device memory
 * is already held by another allocator so a new allocation would fail, or a
 * deployment that must declare all of its device memory up front.
 *
 * Same arguments, layout and results as fa_fwd_decode.  Instead of a
 * per-call workspace, the split partials live in one fixed device array of
 * FA_DECODE_NOALLOC_SCRATCH_BYTES inside this library; every GPU that loads
 * the library holds that array until the process exits.  A call needs
 * n_splits * batch * hq * sq * (head_dim + 1) * 4 bytes of it; the call
 * uses fewer key splits when needed to fit, and returns FA_ERR_INVALID_ARG
 * when even one split does not fit (batch * hq * sq * (head_dim + 1) * 4 >
 * FA_DECODE_NOALLOC_SCRATCH_BYTES).  The call itself makes no cudaMalloc,
 * cudaFree or other allocating call.
 *
 * The first call on each device does a one-time set-up with that device
 * current (it resolves the array's device address); make that first call
 * before any stream capture.  Under the CUDA runtime's default lazy module
 * loading, that first call is also what loads this array's module on the
 * device and so commits its 16 MiB there: make it at start-up, before
 * another allocator reserves the device's memory (or run with
 * CUDA_MODULE_LOADING=EAGER, which commits the array when the library's
 * device code is loaded).  If the array cannot be committed, that call
 * returns FA_ERR_CUDA.  All calls on a device share the one array and
 * it keeps the last call's contents: nothing in it needs clearing (each call
 * writes every partial it reads), but calls that overlap on the GPU -- on
 * different streams, or from different host threads -- race on it and give
 * wrong results.  Serialise them.
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

fa_status fa_fwd_decode_noalloc(const void *q, const void *k, const void *v,
                                void *o, float *lse, int batch, int hq, int hkv,
                                int sq, int sk, const int *seqlens_k,
                                int head_dim, float scale, int causal,
                                fa_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *fa_status_string(fa_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns FA_ERR_TIMEOUT if any kernel recorded a wait time-out since
 * the last call, FA_ERR_CUDA if synchronising failed, else FA_OK.
 */
fa_status fa_get_device_error(fa_stream_t stream);

/*
 * Like fa_get_device_error, and also stores the raw error word in *word_out
 * (0 if none; FA time-outs are 0x1000 | site, where site numbers the wait
 * that gave up).  word_out may be NULL.
 */
fa_status fa_get_device_error_word(fa_stream_t stream, unsigned int *word_out);

/*
 * Self-test of the time-out path: launches one block that waits on an
 * mbarrier nobody arrives at, with a limit of `limit_ns` nanoseconds
 * (clamped to [1e3, 1e9]).  The kernel gives up, records FA_ERR_TIMEOUT in
 * the device error word and exits normally, so the context stays usable.
 */
fa_status fa_selftest_wait_timeout(long long limit_ns, fa_stream_t stream);

/*
 * Self-test of tensor memory: `in` and `out` are device fp32 [128 x 64].
 * Row r is stored to tensor-memory lane r, loaded, multiplied by 1, stored,
 * loaded again and written to `out`; the result must equal `in` bit for bit.
 * (This is the "no-op round trip" that "STAGE_D.md" reports as corrupting
 * data in its kernel; the prefill kernel's rebase and epilogue rely on it.)
 */
fa_status fa_selftest_tmem_roundtrip(const float *in, float *out, fa_stream_t stream);

/*
 * Self-test of one 128 x 128 output tile through the prefill kernel's
 * shared-memory layout, descriptors and tcgen05.mma forms.  d: device fp32
 * [128 x 128].
 *   mode 0 (score MMA): a, b device bf16 [128 x kdim], kdim in {64, 128, 256};
 *           d = a * b^T.
 *   mode 1 (value MMA): a = P, b = V, both device bf16 [128 x 128]; P is placed
 *           in tensor memory, V in shared memory (MN-major); d = a * b.
 * Returns FA_ERR_INVALID_ARG for other modes or sizes.
 */
fa_status fa_selftest_mma_tile(const void *a, const void *b, float *d, int mode,
                               int kdim, fa_stream_t stream);

/*
 * Self-test of the polynomial exp2 that the prefill softmax uses for part of
 * its exponentials (x, y: device fp32 [n]); y[i] approximates 2^x[i] with a
 * relative error below 1e-4 for x in [-125, 126]; inputs below -125 are
 * clamped, giving about 2^-125.  Tested against the exact 2^x.
 */
fa_status fa_selftest_exp2_poly(const float *x, float *y, int n, fa_stream_t stream);

/*
 * Debug tracing of the prefill kernel (not for production use; not
 * thread-safe).  With `buf` a device buffer of at least 5 * 4096 uint64
 * values, the following prefill launches make one thread of each role of the
 * CTA with linear index `block` (x + gridDim.x * (y + gridDim.y * z)) record
 * SM clock stamps at its pipeline events: role r (0 MMA issue, 1 and 2
 * softmax of query tile 0 and 1 -- of key half 0 and 1 in the 256-key
 * kernel --, 3 correction/epilogue, 4 TMA producer), event e of key/value
 * iteration j at buf[r * 4096 + j * 16 + e], for the CTA's first work item
 * (the persistent kernels: j counts the key blocks of all its work items in
 * turn).  Unused slots are left
 * untouched.  buf = NULL
 * switches tracing off.  The stamps are compiled in only when the library is
 * built with FA_PREFILL_TRACE=1 (the Python build reads it from the
 * environment); otherwise a non-NULL buf returns FA_ERR_UNSUPPORTED.
 */
fa_status fa_debug_prefill_trace(unsigned long long *buf, int block);

/*
 * The work split a prefill launch would use on a device with `num_sms` SMs,
 * computed on the host (no device needed).  window: as fa_fwd_prefill_ex;
 * paged: nonzero for fa_fwd_prefill_paged; packed: nonzero for the packed
 * sequences of fa_fwd_prefill_varlen (sq is then the largest query length).
 * A unit is one (batch entry, query head, query block of out[3] rows); it
 * visits nk = ceil(sk / out[4]) key blocks; at head_dim 512 it runs as two
 * CTAs and is never split.  out[5] == 1: min(out[0] + out[1] * out[2],
 * num_sms) persistent CTAs process the work in turn (the 256-key kernel of
 * head_dim 96 / 128, and head_dim 256 when nothing is split); the 256-key
 * kernel splits only when its non-causal units fill at most half the SMs
 * (out[0] = 0: every unit in out[2] pieces of >= 4 key blocks, one piece per
 * CTA).  Otherwise the grid's first out[0] CTAs each process a whole unit,
 * and the remaining out[1] units (the last partial wave) are each processed
 * by out[2] CTAs.  Piece i of a unit takes key blocks [i nk / out[2],
 * (i + 1) nk / out[2]); the last piece to finish merges the pieces' partial
 * results.  out: int[6]
 *   out[0] n_full, out[1] n_tail, out[2] split, out[3] query rows of a unit
 *   (128 or 256), out[4] keys of a score block (128 or 256), out[5]
 *   persistent.
 * Returns FA_ERR_INVALID_ARG for sizes that fa_fwd_prefill rejects or
 * num_sms < 1.
 */
fa_status fa_debug_prefill_plan_ex(int batch, int hq, int sq, int sk, int head_dim, int causal,
                                   int window, int paged, int packed, int num_sms, int *out);

/*
 * fa_debug_prefill_plan_ex with the kv head count: the same plan, with the
 * 256-key kernel's GQA head packing ("b200-flash-attention4-planner" E.7).
 * With hq / hkv = G, rows per head R = the next power of two >= sq, at least
 * 16, at most 128, and P = 128 / R reduced to a power of two dividing G; a
 * unit is then (batch entry, P consecutive query heads of one kv group,
 * query block of R positions), its tile row r being head h0 + r / R at
 * position row0 + r % R.  out: int[7], out[0..5] as fa_debug_prefill_plan_ex
 * (out[3] = R, the query positions of a unit per head) and out[6] = P, the
 * query heads per unit (1: no packing).  FA_ERR_INVALID_ARG also when
 * hkv < 1 or hq is not a multiple of hkv.
 */
fa_status fa_debug_prefill_plan_gqa(int batch, int hq, int hkv, int sq, int sk, int head_dim,
                                    int causal, int window, int paged, int packed, int num_sms,
                                    int *out);

/* fa_debug_prefill_plan_ex of a dense launch without a window (window = 0,
 * paged = packed = 0), out[0..2] only (out: int[3]). */
fa_status fa_debug_prefill_plan(int batch, int hq, int sq, int sk, int head_dim, int causal,
                                int num_sms, int *out);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */

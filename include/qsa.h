/*
 * qsa.h -- exact QSA block selection on one GB300 (sm_103a): block scoring
 * and an exact per-query top-k, as a C ABI over caller-owned device memory.
 *
 * What is computed (the "QSA select" step of query-aware sparse attention):
 * each query is 4 query heads of D = 128 fp32 values that share one KV head.
 * The KV cache is cut into 4-cell blocks, each summarised by one key of 128
 * values. A query's score for a block is the sum over its 4 heads of the
 * head's dot product with the block key; only the first `active_blocks`
 * blocks exist for this batch, whatever the cache capacity. The top-k then
 * keeps, per query, the k highest-scoring block ids exactly.
 * Passages: "#3108 optimize exact QSA block scoring and top-k selection on
 * gfx12", Summary items 1, 2 and 4 (4-head block score, radix top-k,
 * bitwise parity of scores and ids); "#337 gfx12 QSA select", What items 1-2
 * (select over the active blocks, not the capacity `max_context/4 + 2`;
 * split-bf16 tensor-core scorer with the hi*hi products in their own
 * accumulator; FP64 gate at 1e-6 of the score scale).
 *
 * Conventions for every call below:
 *  - All pointers are DEVICE pointers owned by the caller; the library keeps
 *    no state between calls beyond a per-device error word (see
 *    qsa_get_device_error), the fixed device arrays of the two
 *    allocation-free calls (qsa_block_select_static, qsa_block_select_small)
 *    and the process-wide wait settings of qsa_debug_inject; it allocates
 *    nothing, never synchronises (except qsa_get_device_error), and enqueues
 *    its kernels on `stream` (0 = the legacy default stream).
 *  - Every pointer that is dereferenced must be 16-byte aligned.
 *  - Arguments are checked before anything is launched; a bad argument
 *    returns QSA_ERR_INVALID and launches nothing. A launch failure returns
 *    QSA_ERR_CUDA. Errors of already-enqueued work surface as CUDA errors of
 *    the stream, as for any kernel.
 *  - Calls with no work (nq == 0, or active_blocks == 0 for the scorers)
 *    return QSA_OK without touching memory; pointers may then be NULL.
 *  - Inputs are expected to be finite. In the top-k a NaN score counts as
 *    -infinity (it ties with -inf, below every finite score); -0.0 and +0.0
 *    are equal (and therefore tie).
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID = 1,      /* bad argument; nothing was launched            */
    QSA_ERR_UNSUPPORTED = 2,  /* valid, but beyond this library's size limits  */
    QSA_ERR_CUDA = 3          /* a CUDA runtime call or launch failed          */
} qsa_status;

/* Head dimension and query heads per KV head (fixed). */
#define QSA_D 128
#define QSA_HEADS 4

/* Largest active_blocks the top-k accepts (its per-row bitmaps live in shared memory). */
#define QSA_TOPK_MAX_ACTIVE 393216

/*
 * Block scores, fp32 summary keys.
 *   scores[i][b] = sum_{h<4} sum_{d<128} q[i][h][d] * kblk[b][d],  b < active_blocks
 * q       fp32 [nq][4][128], contiguous.
 * kblk    fp32 [max_blocks][128], block-major; only rows < active_blocks are read.
 * scores  fp32 [nq][active_blocks], written; row stride = active_blocks.
 * max_blocks is the key buffer's capacity (validation only: active_blocks <=
 * max_blocks); the launch is sized from active_blocks alone.
 * Accuracy: |scores - exact| <= 1e-6 * max_b |exact[i][b]| per row for
 * finite inputs; scores are exact when every product and partial sum is an
 * integer below 2^24 in magnitude.
 * Kernels: nq >= 5 runs on the tensor cores (3-way exact bf16 split, hi*hi in
 * its own accumulator); nq <= 4 (decode) on CUDA cores with one fp32 FMA
 * chain per query and key row. Both meet the accuracy bound above.
 * ("#3108 ...", Summary item 4; "#337 ...", What items 1-2.)
 */
qsa_status qsa_block_scores(const float *q, const float *kblk, int nq, int max_blocks,
                            int active_blocks, float *scores, cudaStream_t stream);

/*
 * Block scores, int8 summary keys with one IEEE binary16 scale per block
 * (the engine's `--kv int8` cache form; key element = kblk_q8[b][d] *
 * kscale_f16[b], exact in fp32).
 * kblk_q8    int8   [max_blocks][128]
 * kscale_f16 uint16 [max_blocks] (binary16 bit patterns; 2-byte aligned suffices)
 * Other arguments, layouts and accuracy as qsa_block_scores.
 * ("#3108 ...", End-to-End `--kv int8`; "#337 ...", What: `--kv int8`.)
 */
qsa_status qsa_block_scores_q8(const float *q, const int8_t *kblk_q8, const uint16_t *kscale_f16,
                               int nq, int max_blocks, int active_blocks, float *scores,
                               cudaStream_t stream);

/*
 * Block scores on the CUDA cores (FP32 FMA, head-summed query, natural d
 * order) -- the same contract as qsa_block_scores; kept as the measured
 * alternative to the tensor-core scorer. kblk_q8/kscale_f16 may be given
 * instead of kblk (then kblk must be NULL) for the int8 key form.
 */
qsa_status qsa_block_scores_ffma(const float *q, const float *kblk, const int8_t *kblk_q8,
                                 const uint16_t *kscale_f16, int nq, int max_blocks,
                                 int active_blocks, float *scores, cudaStream_t stream);

/*
 * Exact per-query top-k of packed scores.
 * scores  fp32  [nq][active_blocks] (row stride = active_blocks).
 * ids     int32 [nq][k], written: for each row, the ids of the k highest
 *         scores in ascending id order; among equal scores the lower block
 *         id is taken first. If k > active_blocks the row holds all
 *         active_blocks ids ascending followed by -1 (active_blocks == 0
 *         gives a row of -1).
 * k >= 1 and active_blocks <= QSA_TOPK_MAX_ACTIVE (else QSA_ERR_UNSUPPORTED).
 * ("#3108 ...", Summary item 2: radix-bin top-k; "#337 ...", What item 1:
 * the active block count, not the capacity, bounds the selection.)
 */
qsa_status qsa_block_topk(const float *scores, int nq, int active_blocks, int k, int32_t *ids,
                          cudaStream_t stream);

/* Blocks per group of the group-maximum side output (below). */
#define QSA_GROUP_BLOCKS 32

/*
 * Block scores plus their group maxima, for qsa_block_topk_gmax.
 * group_max  uint32 [nq][ceil(active_blocks / 32)], written: element [i][g]
 *            is key(max of scores[i][32 g .. 32 g + 31]) over the blocks
 *            < active_blocks, where key(x) is the order-preserving radix key
 *            of the top-k (-0 counted as +0 and NaN as -inf, then the bits
 *            of a negative x inverted and the sign bit of a positive x set),
 *            so a larger score has a larger unsigned key.
 * 16-byte aligned. Other arguments, layouts and accuracy as qsa_block_scores
 * (the scores are the same bits); the maxima add 1/32 of the score bytes.
 */
qsa_status qsa_block_scores_gmax(const float *q, const float *kblk, int nq, int max_blocks,
                                 int active_blocks, float *scores, uint32_t *group_max,
                                 cudaStream_t stream);

/* The int8-key form of qsa_block_scores_gmax (arguments as qsa_block_scores_q8). */
qsa_status qsa_block_scores_q8_gmax(const float *q, const int8_t *kblk_q8, const uint16_t *kscale_f16,
                                    int nq, int max_blocks, int active_blocks, float *scores,
                                    uint32_t *group_max, cudaStream_t stream);

/*
 * Group maxima of given packed scores (the group_max of
 * qsa_block_scores_gmax, for scores that come from elsewhere).
 * scores     fp32   [nq][active_blocks]
 * group_max  uint32 [nq][ceil(active_blocks / 32)], written (16-byte aligned).
 */
qsa_status qsa_block_group_max(const float *scores, int nq, int active_blocks, uint32_t *group_max,
                               cudaStream_t stream);

/*
 * qsa_block_topk with the group maxima of the same scores (as written by
 * qsa_block_scores_gmax or qsa_block_scores_q8_gmax; 16-byte aligned). The
 * result is identical to qsa_block_topk's. The maxima fix a threshold that
 * at least k groups, hence at least k scores, reach, so a row reads only the
 * groups at or above it; rows where that does not pay (k above half the
 * group count, a threshold list past capacity) take qsa_block_topk's path.
 * group_max that does not match `scores` gives undefined ids (never an
 * out-of-bounds access).
 */
qsa_status qsa_block_topk_gmax(const float *scores, const uint32_t *group_max, int nq, int active_blocks,
                               int k, int32_t *ids, cudaStream_t stream);

/* Largest nq * ceil(active_blocks / 32) qsa_block_select_static accepts:
 * its scratch is a fixed 1 MiB device array of that many uint32. */
#define QSA_SELECT_STATIC_GROUPS_MAX 262144

/*
 * Scores and exact top-k in one call that allocates nothing: exactly
 * qsa_block_scores_gmax followed by qsa_block_topk_gmax, with the group
 * maxima kept in a file-scope device array of QSA_SELECT_STATIC_GROUPS_MAX
 * uint32 (1 MiB, part of the library image) instead of caller memory.
 * scores  fp32  [nq][active_blocks], written (as qsa_block_scores).
 * ids     int32 [nq][k], written (as qsa_block_topk).
 * nq * ceil(active_blocks / 32) > QSA_SELECT_STATIC_GROUPS_MAX returns
 * QSA_ERR_UNSUPPORTED before anything is launched (e.g. 256 queries up to
 * 32,768 active blocks, 128 up to 65,536). The scratch is one per device:
 * calls on one device must be ordered (one stream, or streams joined by
 * events); overlapping calls on unordered streams give undefined ids.
 * Other arguments, errors and accuracy as the two calls it stands for.
 */
qsa_status qsa_block_select_static(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks,
                                   int k, float *scores, int32_t *ids, cudaStream_t stream);

/*
 * Scores and exact top-k for a few queries (decode: 1 <= nq <= 4) in one
 * cooperative kernel launch: the whole grid scores every active block (and
 * its 32-block group maxima, kept in a fixed device array of the library),
 * then nq of its CTAs each select one query's top k from those maxima. The
 * scores and ids equal qsa_block_scores(_q8) followed by qsa_block_topk.
 * Give kblk (fp32 keys) or kblk_q8 + kscale_f16 (int8 keys), not both; the
 * layouts are those of qsa_block_scores / qsa_block_scores_q8.
 * scores  fp32  [nq][active_blocks], written.
 * ids     int32 [nq][k], written (as qsa_block_topk).
 * nq > 4 or active_blocks > QSA_TOPK_MAX_ACTIVE returns QSA_ERR_UNSUPPORTED.
 * Nothing is allocated. The grid meets at a device-wide counter and a
 * generation word of library state, so calls on one device must be ordered
 * (one stream, or streams joined by events). When k >= active_blocks the call
 * runs the scorer and a fill.
 * Passage: "#3108 optimize exact QSA block scoring and top-k selection on
 * gfx12", Summary item 4 (a row kernel for a handful of queries) and the
 * Microbenchmark & Parity Evidence table (decode scores + top-k per layer).
 */
qsa_status qsa_block_select_small(const float *q, const float *kblk, const int8_t *kblk_q8,
                                  const uint16_t *kscale_f16, int nq, int max_blocks, int active_blocks, int k,
                                  float *scores, int32_t *ids, cudaStream_t stream);

/*
 * Attention over the selected blocks: each query's 4 heads attend the KV
 * cells of the blocks listed in its row of ids (block b holds cells
 * 4b .. 4b+3; cells at or past ncells, negative ids and ids at or past the
 * last block are skipped; a block listed twice counts twice):
 *   logit[h][c] = (sum_d q[i][h][d] * k_cells[c][d]) * k_scale[c] / sqrt(128)
 *   out[i][h][d] = sum_c softmax_c(logit[h][.]) * v_cells[c][d] * v_scale[c]
 * and out = 0 for a query with no attended cell. Accumulation is fp32 in a
 * fixed order (the result does not depend on scheduling). With at most half
 * as many queries as the device has SMs the products are fp32 on CUDA cores;
 * with more, they run on the tensor cores (mma.sync): q (per head) and the softmax
 * weights times v_scale, each scaled by a power of two chosen from the data,
 * enter as binary16 high parts plus remainders (about 22 significant bits),
 * the int8 cells exactly, with fp32 accumulation.
 * q        fp32 [nq][4][128], 16-byte aligned.
 * k_cells, v_cells  int8 [ncells][128], 16-byte aligned; k_scale_f16,
 *          v_scale_f16  IEEE binary16 bit patterns [ncells], 2-byte aligned
 *          (may be NULL when ncells == 0).
 * ids      int32 [nq][k] (e.g. qsa_block_topk's output), 16-byte aligned.
 * out      fp32 [nq][4][128], written, 16-byte aligned.
 * nq < 0, k < 1 or ncells < 0 returns QSA_ERR_INVALID; nq == 0 is a no-op;
 * ncells > INT_MAX - 4 returns QSA_ERR_UNSUPPORTED. Allocates nothing and
 * keeps no state.
 * Passages: "#3224 [Engine] perf(hip): tune RDNA4 QSA prompt WMMA path
 * (STRATA_HIP_WMMA stays opt-in)", Summary and Evidence section 2 (int8-KV
 * QSA attention with binary16 k/v scales, gated against FP64); "#3102
 * perf(hip): enable wave32 QSA decode attention and MMVQ row reuse on
 * gfx12", item D5 (decode attention in chunks merged in sequential order).
 * The softmax temperature 1/sqrt(128), the per-cell scales and the 4 heads
 * sharing the cells are readings: the pages print no formula.
 */
qsa_status qsa_sparse_attn(const float *q, const int8_t *k_cells, const uint16_t *k_scale_f16,
                           const int8_t *v_cells, const uint16_t *v_scale_f16, int ncells, const int32_t *ids,
                           int nq, int k, float *out, cudaStream_t stream);

/*
 * Block summary keys from int8 KV cells, for blocks block_begin ..
 * block_end-1 (after an append: block_begin = old ncells / 4, block_end =
 * ceil(new ncells / 4)):
 *   kblk[b][d]    = (sum over the present cells c = 4b .. 4b+3 (< ncells) of
 *                    k_cells[c][d] * k_scale[c]) / (number of present cells)
 *   kblk_scale[b] = binary16(max_d |kblk[b][d]| / 127), round to nearest even
 *   kblk_q8[b][d] = rint(kblk[b][d] / kblk_scale[b])  (0 when the scale is 0)
 * computed in fp32 in that order (IEEE single operations), so the int8 form
 * is reproducible bit for bit; a block with no present cell gets zeros.
 * k_cells  int8 [ncells][128], 16-byte aligned; k_scale_f16 binary16 [ncells],
 *          2-byte aligned (both may be NULL when ncells == 0).
 * kblk     fp32 [>= block_end][128] (row b written), 16-byte aligned, or NULL.
 * kblk_q8  int8 [>= block_end][128] and kblk_scale_f16 binary16 [>= block_end]
 *          (the qsa_block_scores_q8 key layout), both or neither.
 * ncells < 0, block_begin < 0, block_end < block_begin, or no output returns
 * QSA_ERR_INVALID; an empty range is a no-op; 4 * block_end + 4 > INT_MAX
 * returns QSA_ERR_UNSUPPORTED. Allocates nothing.
 * Passage: "#3108 optimize exact QSA block scoring and top-k selection on
 * gfx12", the Microbenchmark & Parity Evidence table (the decode layer's
 * "append" step). The pages do not define the summary function: the mean of
 * the present cells and the int8 form are readings.
 */
qsa_status qsa_block_summary(const int8_t *k_cells, const uint16_t *k_scale_f16, int ncells, int block_begin,
                             int block_end, float *kblk, int8_t *kblk_q8, uint16_t *kblk_scale_f16,
                             cudaStream_t stream);

/*
 * qsa_block_select: the ids of qsa_block_topk(qsa_block_scores(...)) --
 * exactly the same ids -- without writing the scores in the common case
 * (fp32 keys; q, kblk, ids as qsa_block_scores / qsa_block_topk).
 * Method: per query row, a threshold from a strided sample of 1,024 blocks
 * (CUDA cores), chosen so that about 1.8 k scores reach it; the tensor-core
 * scorer then appends every score at or above its row's threshold, with its
 * block id, to the row's list (at most QSA_SELECT_LIST_CAP entries) instead
 * of storing the scores; a row whose list holds at least k entries (and did
 * not overflow) holds its whole top-k and is selected from the list exactly.
 * The other rows' query groups (128 rows each) are scored into `scores` and
 * their rows selected by qsa_block_topk's kernel. When nq <= 4, active_blocks
 * <= QSA_SELECT_LIST_MIN_ACTIVE or k > QSA_SELECT_LIST_K_MAX, it runs the two
 * plain calls (scores written). k >= active_blocks: ids as qsa_block_topk.
 * scores: [nq][active_blocks] fp32, caller-owned; its contents afterwards are
 * unspecified (written only where the fallback ran).
 * scratch: device memory of at least qsa_block_select_scratch_bytes(nq)
 * bytes, 16-byte aligned, caller-owned (thresholds, list counts, failure
 * flags, lists; no contents need survive between calls). Five launches on
 * `stream`; allocates nothing.
 * Errors: as qsa_block_scores and qsa_block_topk, plus QSA_ERR_INVALID for a
 * missing, misaligned or too small scratch.
 * Passages: "#3108 optimize exact QSA block scoring and top-k selection on
 * gfx12", Microbenchmark & Parity Evidence section 2 (selection inside the
 * decode layer, where the scores are only an intermediate); "#337 gfx12 QSA
 * select", What item 1 (scores, then top-k over the active blocks).
 */
#define QSA_SELECT_LIST_CAP 4096
#define QSA_SELECT_LIST_MIN_ACTIVE 8192
#define QSA_SELECT_LIST_K_MAX 1024
size_t qsa_block_select_scratch_bytes(int nq);
qsa_status qsa_block_select(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks, int k,
                            float *scores, int32_t *ids, void *scratch, size_t scratch_bytes, cudaStream_t stream);

/*
 * Reads and clears the current device's error word: nonzero when a kernel
 * of this library gave up a bounded wait (its outputs are then invalid).
 * Bit 0x100: a wait of the tensor-core scorer's pipeline ran out (the CTA
 * then abandons its remaining waits at once, lets its own copies and MMAs
 * in flight finish, and exits); bit 0x2: the fused decode select's grid
 * barrier ran out. Synchronises `stream`. *code receives the word.
 */
qsa_status qsa_get_device_error(uint32_t *code, cudaStream_t stream);

/*
 * Diagnostics for the bounded waits (not for production use; the pages have
 * no counterpart). For the kernels launched after the call: every spin-wait
 * gives up after wait_limit_ns (default 2,000,000,000), and `faults` plants
 * a wait that cannot complete so that the time-out path runs:
 *   bit 0: the tensor-core scorer's CTA 0 never loads its first key piece
 *          (qsa_block_scores, _q8, _gmax and _select_static with nq > 4);
 *   bit 1: the fused decode select's grid barrier waits for one arrival
 *          more than its grid has (qsa_block_select_small).
 * The outputs of such calls are invalid and qsa_get_device_error reports
 * them; the device stays usable. Call qsa_debug_inject(0, 2000000000) to
 * restore normal operation. Process-wide; not thread-safe against
 * concurrent launches. faults with other bits, or wait_limit_ns == 0 or
 * above 60 s, returns QSA_ERR_INVALID.
 */
qsa_status qsa_debug_inject(uint32_t faults, uint64_t wait_limit_ns);

/* Static description of a status code. */
const char *qsa_status_string(qsa_status status);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */

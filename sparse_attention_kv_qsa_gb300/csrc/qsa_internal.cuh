// Internal launch interface between the C ABI (qsa_api.cu) and the kernels.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace qsa {

constexpr int D = 128;
constexpr int HEADS = 4;
// Consecutive blocks per group of the group-maximum side output.
constexpr int GROUP_BLOCKS = 32;

// Order-preserving radix key of a score: -0 becomes +0 (x + 0) and NaN
// becomes -inf (max(., -inf)), then negatives are bit-inverted and positives
// get the sign bit set, so a larger score has a larger unsigned key.
__device__ __forceinline__ uint32_t score_key(float x) {
    const float f = fmaxf(__fadd_rn(x, 0.0f), -INFINITY);
    const uint32_t u = __float_as_uint(f);
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Streaming multiprocessor count of the current device (cached per device).
int device_sm_count();

// Scores on CUDA cores. Exactly one of kblk / (kq8, kscale) is non-null.
cudaError_t launch_scores_ffma(const float *q, const float *kblk, const int8_t *kq8,
                               const uint16_t *kscale, int nq, int active, float *scores,
                               cudaStream_t stream);

// The fused select's per-row candidate lists: LIST_CAP (fp32 score bits, block id) pairs.
constexpr int LIST_CAP = 4096;

// Extra modes of the tensor-core scorer for the fused select (fp32 keys):
// list mode (thr set): no scores are stored; every score >= thr[row] is
// appended to the row's list cand[row][0 .. LIST_CAP) as (fp32 bits, id), counted
// in cnt[row]; the scorer waits for the previous grid (which writes thr and
// clears cnt) only before its first append. Gated mode (gate set): only the
// CTAs of query groups g with gate[g] != 0 run (after waiting for the
// previous grid), the others exit at once.
struct TcSelect {
    const float *thr = nullptr;
    uint32_t *cnt = nullptr;
    uint2 *cand = nullptr;
    const uint32_t *gate = nullptr;
};

// Scores on the tensor cores (3-way bf16 split; int8 keys: one slice).
// Exactly one of kblk / (kq8, kscale) is non-null. gmax (may be null):
// [nq][ceil(active / GROUP_BLOCKS)] keys of each group's largest score.
cudaError_t launch_scores_tc(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                             int nq, int active, float *scores, uint32_t *gmax, cudaStream_t stream,
                             const TcSelect &sel = TcSelect());

// gmax from packed scores (the decode scorer's companion).
cudaError_t launch_group_max(const float *scores, int nq, int active, uint32_t *gmax, cudaStream_t stream);

// Scores for nq <= 4 (decode) on CUDA cores, the grid spanning key rows.
// Exactly one of kblk / (kq8, kscale) is non-null; gmax as launch_scores_tc.
constexpr int SMALL_NQ_MAX = 4;
cudaError_t launch_scores_rows(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                               int nq, int active, float *scores, uint32_t *gmax, cudaStream_t stream);

// Exact top-k (k < active); one CTA per row. gmax (may be null): the
// group maxima of these scores, which let a row read only the groups that
// can hold its top k.
cudaError_t launch_topk(const float *scores, const uint32_t *gmax, int nq, int active, int k, int32_t *ids,
                        cudaStream_t stream, const uint32_t *gate = nullptr);

// Fused select (see topk.cu): the per-row thresholds (and the cleared list
// counts and failure flags), and the exact selection from the lists.
cudaError_t launch_select_threshold(const float *q, const float *kblk, int nq, int active, int k, float *thr,
                                    uint32_t *cnt, uint32_t *fail, uint32_t *gfail, cudaStream_t stream);
cudaError_t launch_select_list(const uint2 *cand, const uint32_t *cnt, int nq, int active, int k, int32_t *ids,
                               uint32_t *fail, uint32_t *gfail, cudaStream_t stream);

// Scores and top-k for nq <= 4 in one cooperative launch (k < active):
// scores written, group maxima in a fixed device array; calls on one device
// must be ordered (the launch shares that array and two sync words).
cudaError_t launch_select_decode(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                                 int nq, int active, int k, float *scores, int32_t *ids, cudaStream_t stream);

// Summary keys of blocks b0 .. b1-1 from int8 cells (csrc/summary.cu); key
// (fp32 rows) and kq8 + kscale (int8 rows, binary16 scales) may each be null.
cudaError_t launch_block_summary(const int8_t *kc, const uint16_t *ks, int ncells, int b0, int b1, float *key,
                                 int8_t *kq8, uint16_t *kscale, cudaStream_t stream);

// Attention of each query's 4 heads over the int8 KV cells of its listed
// blocks (csrc/attn.cu: CUDA cores for nq below the SM count, else the
// tensor-core kernel of csrc/attn_tc.cu, which launch_sparse_attn_tc runs
// for any nq >= 1).
cudaError_t launch_sparse_attn(const float *q, const int8_t *kc, const uint16_t *ks, const int8_t *vc,
                               const uint16_t *vs, int ncells, const int32_t *ids, int nq, int k, float *out,
                               cudaStream_t stream);
cudaError_t launch_sparse_attn_tc(const float *q, const int8_t *kc, const uint16_t *ks, const int8_t *vc,
                                  const uint16_t *vs, int ncells, const int32_t *ids, int nq, int k, float *out,
                                  cudaStream_t stream);

// ids[i][j] = j < active ? j : -1 (the k >= active case).
cudaError_t launch_topk_all(int nq, int active, int k, int32_t *ids, cudaStream_t stream);

// Error words of the kernels (bounded waits that gave up); read and clear.
cudaError_t topk_error_read_clear(uint32_t *word, cudaStream_t stream);
// Upper bound (ns) of every spin-wait in the kernels launched from now on:
// 2 s, unless qsa_debug_inject changed it.
uint64_t wait_limit_ns();
// qsa_debug_inject's fault bits for the kernels launched from now on (0 in use).
uint32_t debug_inject();
cudaError_t tc_error_read_clear(uint32_t *word, cudaStream_t stream);

}  // namespace qsa

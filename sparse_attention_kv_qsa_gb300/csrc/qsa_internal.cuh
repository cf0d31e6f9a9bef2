// Internal launch interface between the C ABI (qsa_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qsa {

constexpr int D = 128;
constexpr int HEADS = 4;

// Streaming multiprocessor count of the current device (cached per device).
int device_sm_count();

// Scores on CUDA cores. Exactly one of kblk / (kq8, kscale) is non-null.
cudaError_t launch_scores_ffma(const float *q, const float *kblk, const int8_t *kq8,
                               const uint16_t *kscale, int nq, int active, float *scores,
                               cudaStream_t stream);

// Scores on the tensor cores (3-way bf16 split; int8 keys: one slice).
// Exactly one of kblk / (kq8, kscale) is non-null.
cudaError_t launch_scores_tc(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                             int nq, int active, float *scores, cudaStream_t stream);

// Scores for nq <= 4 (decode) on CUDA cores, the grid spanning key rows.
// Exactly one of kblk / (kq8, kscale) is non-null.
constexpr int SMALL_NQ_MAX = 4;
cudaError_t launch_scores_rows(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                               int nq, int active, float *scores, cudaStream_t stream);

// Exact top-k (k < active); one CTA per row.
cudaError_t launch_topk(const float *scores, int nq, int active, int k, int32_t *ids,
                        cudaStream_t stream);

// ids[i][j] = j < active ? j : -1 (the k >= active case).
cudaError_t launch_topk_all(int nq, int active, int k, int32_t *ids, cudaStream_t stream);

// Error words of the kernels (bounded waits that gave up); read and clear.
cudaError_t topk_error_read_clear(uint32_t *word, cudaStream_t stream);
cudaError_t tc_error_read_clear(uint32_t *word, cudaStream_t stream);

}  // namespace qsa

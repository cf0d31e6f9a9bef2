// Decode scorer (nq <= 4) on CUDA cores: one chunk of key rows per CTA; the
// scoring itself is decode_rows.cuh's.
#include "decode_rows.cuh"

namespace qsa {
namespace {

constexpr int ROWS_THREADS = 256;

template <int NQ, bool kInt8>
__global__ void __launch_bounds__(ROWS_THREADS)
    scores_rows_kernel(const float *__restrict__ q, const float *__restrict__ kblk,
                       const int8_t *__restrict__ kq8, const __half *__restrict__ kscale, int nq, int active,
                       float *__restrict__ scores, uint32_t *__restrict__ gmax) {
    __shared__ __align__(16) float qs[NQ][DEC_QROW];   // head-summed queries, zero past nq
    __shared__ uint32_t gk[NQ][ROWS_THREADS / dec_tpr<kInt8>()];
    grid_dependency_wait();   // q and the keys may come from the previous grid
    grid_launch_dependents();
    DecKeys<kInt8> kv;
    dec_load_keys<kInt8, ROWS_THREADS>(blockIdx.x, kblk, kq8, active, kv);   // in flight during the build
    dec_build_queries<NQ, ROWS_THREADS>(q, nq, qs);
    __syncthreads();
    dec_score_chunk<NQ, kInt8, ROWS_THREADS>(qs, blockIdx.x, kv, kscale, nq, active, scores, gmax, gk);
}

template <int NQ>
cudaError_t launch_rows(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale, int nq,
                        int active, float *scores, uint32_t *gmax, cudaStream_t stream) {
    const int tpr = kq8 != nullptr ? 2 : 4;
    const long long threads = static_cast<long long>(active) * tpr;
    const long long grid = (threads + ROWS_THREADS - 1) / ROWS_THREADS;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(ROWS_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kq8 != nullptr)
        return cudaLaunchKernelEx(&cfg, scores_rows_kernel<NQ, true>, q, static_cast<const float *>(nullptr), kq8,
                                  reinterpret_cast<const __half *>(kscale), nq, active, scores, gmax);
    return cudaLaunchKernelEx(&cfg, scores_rows_kernel<NQ, false>, q, kblk, static_cast<const int8_t *>(nullptr),
                              static_cast<const __half *>(nullptr), nq, active, scores, gmax);
}

// Group maxima of packed scores: one warp per 32-block group, lane j taking
// block 32 g + j; the group's largest key is a warp max.
__global__ void __launch_bounds__(ROWS_THREADS)
    group_max_kernel(const float *__restrict__ scores, int nq, int active, int ngr, uint32_t *__restrict__ gmax) {
    grid_dependency_wait();   // the scores come from the previous grid
    grid_launch_dependents();
    const long long w = (static_cast<long long>(blockIdx.x) * ROWS_THREADS + threadIdx.x) >> 5;   // warp-uniform
    if (w >= static_cast<long long>(nq) * ngr) return;
    const int lane = threadIdx.x & 31;
    const int r = static_cast<int>(w / ngr), g = static_cast<int>(w % ngr);
    const int b = g * GROUP_BLOCKS + lane;
    uint32_t key = 0u;
    if (b < active) key = score_key(ld_in(scores + static_cast<size_t>(r) * active + b));
    key = __reduce_max_sync(FULL_MASK, key);
    if (lane == 0) gmax[w] = key;
}

}  // namespace

cudaError_t launch_group_max(const float *scores, int nq, int active, uint32_t *gmax, cudaStream_t stream) {
    static_assert(GROUP_BLOCKS == 32, "one warp per group");
    const int ngr = (active + GROUP_BLOCKS - 1) / GROUP_BLOCKS;
    const long long threads = static_cast<long long>(nq) * ngr * 32;
    const long long grid = (threads + ROWS_THREADS - 1) / ROWS_THREADS;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(ROWS_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, group_max_kernel, scores, nq, active, ngr, gmax);
}

cudaError_t launch_scores_rows(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                               int nq, int active, float *scores, uint32_t *gmax, cudaStream_t stream) {
    switch (nq) {
        case 1: return launch_rows<1>(q, kblk, kq8, kscale, nq, active, scores, gmax, stream);
        case 2: return launch_rows<2>(q, kblk, kq8, kscale, nq, active, scores, gmax, stream);
        case 3:
        case 4: return launch_rows<4>(q, kblk, kq8, kscale, nq, active, scores, gmax, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qsa

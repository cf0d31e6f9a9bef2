// Block scoring for a handful of queries (decode: nq <= 4), on CUDA cores.
//
//   score[i][b] = sum_{d<128} s[i][d] * key[b][d],   s[i][d] = ((q0 + q1) + q2) + q3
//
// Passages: "#3108 optimize exact QSA block scoring and top-k selection on
// gfx12", Summary items 1 and 4 (the 4-head block score); "#337 gfx12 QSA
// select", What (decode with `--kv int8`: int8 keys, one binary16 scale per
// block).
//
// With one to four query rows the scoring is a matrix-vector product: every
// key byte is used nq times, so the tensor-core tile (128 query rows) would be
// almost all padding. Here the grid spans the key rows instead: a key row is
// split over TPR threads (fp32: 4 threads x 32 values; int8: 2 threads x 64
// values), each thread streams its part with 16-byte read-only loads and
// accumulates one fp32 FMA chain per query against the head-summed queries
// in shared memory (read as broadcasts), and the TPR partial sums meet by
// warp shuffles. Rows at or beyond `active` are never read.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int ROWS_THREADS = 256;
// Shared query rows get 4 floats of padding after every 32, so the TPR parts
// of a row (32 or 64 values apart) read different banks.
constexpr int QROW = D + D / 8;
__device__ __forceinline__ int qidx(int d) { return d + (d >> 5) * 4; }

template <int NQ, bool kInt8>
__global__ void __launch_bounds__(ROWS_THREADS)
    scores_rows_kernel(const float *__restrict__ q, const float *__restrict__ kblk,
                       const int8_t *__restrict__ kq8, const __half *__restrict__ kscale, int nq, int active,
                       float *__restrict__ scores, uint32_t *__restrict__ gmax) {
    constexpr int TPR = kInt8 ? 2 : 4;          // threads per key row
    constexpr int PER = D / TPR;                // values per thread: 64 (int8) or 32 (fp32)
    __shared__ __align__(16) float qs[NQ][QROW];   // head-summed queries, zero past nq

    grid_dependency_wait();   // q and the keys may come from the previous grid
    grid_launch_dependents();
    for (int e = threadIdx.x; e < NQ * D; e += ROWS_THREADS) {
        const int r = e / D, d = e % D;
        float v = 0.0f;
        if (r < nq) {
            const float *p = q + static_cast<size_t>(r) * (HEADS * D) + d;
            v = __fadd_rn(__fadd_rn(__fadd_rn(__ldg(p), __ldg(p + D)), __ldg(p + 2 * D)), __ldg(p + 3 * D));
        }
        qs[r][qidx(d)] = v;
    }
    __syncthreads();

    const long long t = static_cast<long long>(blockIdx.x) * ROWS_THREADS + threadIdx.x;
    const long long b = t / TPR;               // key row
    const int part = static_cast<int>(t % TPR);
    const bool live = b < active;
    float acc[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) acc[r] = 0.0f;
    if (live) {
        if constexpr (!kInt8) {
            const float4 *row = reinterpret_cast<const float4 *>(kblk + b * D + part * PER);
            float4 kv[PER / 4];
#pragma unroll
            for (int c = 0; c < PER / 4; ++c) kv[c] = __ldg(row + c);
#pragma unroll
            for (int c = 0; c < PER / 4; ++c) {
#pragma unroll
                for (int r = 0; r < NQ; ++r) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&qs[r][qidx(part * PER + 4 * c)]);
                    acc[r] = fmaf(qv.x, kv[c].x, acc[r]);
                    acc[r] = fmaf(qv.y, kv[c].y, acc[r]);
                    acc[r] = fmaf(qv.z, kv[c].z, acc[r]);
                    acc[r] = fmaf(qv.w, kv[c].w, acc[r]);
                }
            }
        } else {
            const uint4 *row = reinterpret_cast<const uint4 *>(kq8 + b * D + part * PER);
            uint4 kv[PER / 16];
#pragma unroll
            for (int c = 0; c < PER / 16; ++c) kv[c] = __ldg(row + c);
#pragma unroll
            for (int c = 0; c < PER / 16; ++c) {
                const uint32_t w4[4] = {kv[c].x, kv[c].y, kv[c].z, kv[c].w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    float kf[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        kf[e] = static_cast<float>(static_cast<int8_t>((w4[wi] >> (8 * e)) & 0xFFu));
#pragma unroll
                    for (int r = 0; r < NQ; ++r) {
                        const float4 qv =
                            *reinterpret_cast<const float4 *>(&qs[r][qidx(part * PER + 16 * c + 4 * wi)]);
                        acc[r] = fmaf(qv.x, kf[0], acc[r]);
                        acc[r] = fmaf(qv.y, kf[1], acc[r]);
                        acc[r] = fmaf(qv.z, kf[2], acc[r]);
                        acc[r] = fmaf(qv.w, kf[3], acc[r]);
                    }
                }
            }
        }
    }
    // The TPR threads of a row are adjacent lanes: add their partial sums.
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) acc[r] = __fadd_rn(acc[r], __shfl_xor_sync(FULL_MASK, acc[r], o));
    }
    if (live && part == 0) {
        const float scale = kInt8 ? __half2float(kscale[b]) : 1.0f;
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
            if (kInt8) acc[r] = __fmul_rn(acc[r], scale);
            if (r < nq) scores[static_cast<size_t>(r) * active + b] = acc[r];
        }
    }
    // Group maxima (when asked): this CTA's rows are whole 32-block groups;
    // their keys meet in shared memory and one warp per (query, group) takes
    // the maximum.
    if (gmax != nullptr) {   // uniform
        constexpr int ROWS = ROWS_THREADS / TPR;      // rows of this CTA: 64 (fp32) or 128 (int8)
        constexpr int GROUPS = ROWS / GROUP_BLOCKS;
        __shared__ uint32_t gk[NQ][ROWS];
        const int rl = threadIdx.x / TPR;
        if (part == 0) {
#pragma unroll
            for (int r = 0; r < NQ; ++r) gk[r][rl] = live ? score_key(acc[r]) : 0u;
        }
        __syncthreads();
        const int ngr = (active + GROUP_BLOCKS - 1) / GROUP_BLOCKS;
        const int lane = threadIdx.x & 31;
        for (int w = threadIdx.x >> 5; w < NQ * GROUPS; w += ROWS_THREADS / 32) {   // warp-uniform
            const int r = w / GROUPS, gl = w % GROUPS;
            const uint32_t key = __reduce_max_sync(FULL_MASK, gk[r][gl * GROUP_BLOCKS + lane]);
            const long long g = static_cast<long long>(blockIdx.x) * GROUPS + gl;
            if (lane == 0 && r < nq && g < ngr) gmax[static_cast<size_t>(r) * ngr + g] = key;
        }
    }
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
    if (b < active) key = score_key(__ldg(scores + static_cast<size_t>(r) * active + b));
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

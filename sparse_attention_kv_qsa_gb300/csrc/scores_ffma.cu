// Block scoring on the CUDA cores (FP32 FMA).
//
//   score[i][b] = sum_{h<4} sum_{d<128} q[i][h][d] * key[b][d]
//               = sum_{d<128} s[i][d] * key[b][d],   s[i][d] = ((q0 + q1) + q2) + q3
//
// ("#3108 optimize exact QSA block scoring and top-k selection on gfx12",
// Summary items 1 and 4: the 4-head block score.) Summing the heads first is
// an algebraic identity that cuts the contraction four-fold; it changes the
// rounding only at the level of fp32 dot-product error, far inside the gate
// of 1e-6 of the row's largest score ("#337 gfx12 QSA select", What item 2).
// Integer-valued inputs whose partial sums stay below 2^24 score exactly.
//
// Tiling: a CTA keeps the head-summed, d-major tile of 128 queries in shared
// memory and walks 128-block key tiles; each thread accumulates an 8 x 8
// (query x block) outer product per d step. Key rows at or beyond `active`
// are never read. int8 keys are converted exactly to fp32 and their binary16
// scale is applied once per score in the epilogue.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int FQ = 128;        // queries per CTA
constexpr int FB = 128;        // blocks per key tile
constexpr int FDC = 32;        // d per staged key chunk
constexpr int SPAD = FQ + 4;   // row stride of the query tile (floats)
constexpr int KPAD = FB + 4;   // row stride of the key chunk (floats)
constexpr int FTHREADS = 256;
constexpr size_t FFMA_SMEM = static_cast<size_t>(D * SPAD + FDC * KPAD) * sizeof(float);

template <bool kInt8>
__global__ void __launch_bounds__(FTHREADS, 2)
    scores_ffma_kernel(const float *__restrict__ q, const float *__restrict__ kblk,
                       const int8_t *__restrict__ kq8, const __half *__restrict__ kscale, int nq,
                       int active, int ntiles, float *__restrict__ scores) {
    extern __shared__ __align__(16) float smem[];
    float *s_t = smem;               // [D][SPAD]:  s_t[d][j] = s[q0 + j][d]
    float *k_t = smem + D * SPAD;    // [FDC][KPAD]: k_t[d][c] = key[b0 + c][dc + d]
    const int tid = threadIdx.x;
    const int q0 = blockIdx.y * FQ;

    // Head-summed query tile. A warp covers 8 consecutive d of 4 queries per
    // step: 32-byte global segments, and distinct banks on the transposed store.
    {
        const int lane = tid & 31, warp = tid >> 5;
        const int doff = lane & 7, qoff = lane >> 3;
        for (int it = warp; it < (FQ / 4) * (D / 8); it += FTHREADS / 32) {
            const int j = (it / (D / 8)) * 4 + qoff;
            const int d = (it % (D / 8)) * 8 + doff;
            float v = 0.f;
            if (q0 + j < nq) {
                const float *qp = q + static_cast<size_t>(q0 + j) * (HEADS * D) + d;
                v = ((ld_in(qp) + ld_in(qp + D)) + ld_in(qp + 2 * D)) + ld_in(qp + 3 * D);
            }
            s_t[d * SPAD + j] = v;
        }
    }

    const int tb = tid & 15, tq = tid >> 4;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int b0 = tile * FB;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

#pragma unroll 1
        for (int dc = 0; dc < D; dc += FDC) {
            __syncthreads();  // previous chunk consumed (and the query tile written)
            {
                // thread -> (block c, half h): 16 consecutive d of one key row
                const int c = tid & (FB - 1), h = tid >> 7;
                const int b = b0 + c;
                float v[16];
                if (b < active) {
                    if constexpr (!kInt8) {
                        const float4 *src =
                            reinterpret_cast<const float4 *>(kblk + static_cast<size_t>(b) * D + dc + h * 16);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float4 f = ld_in(src + u);
                            v[4 * u] = f.x;
                            v[4 * u + 1] = f.y;
                            v[4 * u + 2] = f.z;
                            v[4 * u + 3] = f.w;
                        }
                    } else {
                        const uint4 raw =
                            ld_in(reinterpret_cast<const uint4 *>(kq8 + static_cast<size_t>(b) * D + dc + h * 16));
                        const int w[4] = {static_cast<int>(raw.x), static_cast<int>(raw.y), static_cast<int>(raw.z),
                                          static_cast<int>(raw.w)};
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                v[4 * u + e] = static_cast<float>(static_cast<int8_t>((w[u] >> (8 * e)) & 0xFF));
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u) v[u] = 0.f;
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) k_t[(h * 16 + u) * KPAD + c] = v[u];
            }
            __syncthreads();
#pragma unroll 4
            for (int d = 0; d < FDC; ++d) {
                const float *sr = s_t + (dc + d) * SPAD;
                const float *kr = k_t + d * KPAD;
                const float4 a0 = *reinterpret_cast<const float4 *>(sr + tq * 4);
                const float4 a1 = *reinterpret_cast<const float4 *>(sr + 64 + tq * 4);
                const float4 c0 = *reinterpret_cast<const float4 *>(kr + tb * 4);
                const float4 c1 = *reinterpret_cast<const float4 *>(kr + 64 + tb * 4);
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], c[j], acc[i][j]);
            }
        }

        // Epilogue: rows q0 + {tq*4 .. +3, 64 + tq*4 .. +3}, columns
        // b0 + {tb*4 .. +3, 64 + tb*4 .. +3}.
        const bool vec_ok = (active & 3) == 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int bb = b0 + half * 64 + tb * 4;
            float sc[4] = {1.f, 1.f, 1.f, 1.f};
            if constexpr (kInt8) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (bb + e < active) sc[e] = __half2float(__ushort_as_half(ld_in_u16(kscale + bb + e)));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int qi = q0 + (i < 4 ? tq * 4 + i : 64 + tq * 4 + (i - 4));
                if (qi >= nq) continue;
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = kInt8 ? acc[i][half * 4 + e] * sc[e] : acc[i][half * 4 + e];
                float *dst = scores + static_cast<size_t>(qi) * active + bb;
                if (vec_ok && bb + 3 < active) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (bb + e < active) dst[e] = o[e];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_scores_ffma(const float *q, const float *kblk, const int8_t *kq8,
                               const uint16_t *kscale, int nq, int active, float *scores,
                               cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(scores_ffma_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, FFMA_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(scores_ffma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     FFMA_SMEM);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int ntiles = (active + FB - 1) / FB;
    const int nqt = (nq + FQ - 1) / FQ;
    // Two CTAs per SM; even out the key tiles per CTA.
    int gmax = (2 * device_sm_count()) / nqt;
    if (gmax < 1) gmax = 1;
    const int per = (ntiles + gmax - 1) / gmax;
    const int gx = (ntiles + per - 1) / per;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(nqt));
    if (kq8 != nullptr) {
        scores_ffma_kernel<true><<<grid, FTHREADS, FFMA_SMEM, stream>>>(
            q, nullptr, kq8, reinterpret_cast<const __half *>(kscale), nq, active, ntiles, scores);
    } else {
        scores_ffma_kernel<false><<<grid, FTHREADS, FFMA_SMEM, stream>>>(q, kblk, nullptr, nullptr, nq, active,
                                                                           ntiles, scores);
    }
    return cudaGetLastError();
}

}  // namespace qsa

// Block summary keys, brought up to date when cells are appended.
//
//   key[b][d] = (sum over the present cells c = 4b .. 4b+3 (< ncells) of
//                kq[c][d] * ks[c]) / n          (n = number of present cells)
//   s[b]      = binary16(max_d |key[b][d]| / 127)   (round to nearest even)
//   kq8[b][d] = rint(key[b][d] / s[b])              (0 when s[b] is 0)
//
// Passage: "#3108 optimize exact QSA block scoring and top-k selection on
// gfx12", the Microbenchmark & Parity Evidence table (the decode layer times
// "append + scores + topk + attn"). The pages do not define the summary
// function; the mean of the block's present cells is the reading taken, and
// the int8 form (one binary16 scale per block) is the decode scorer's key
// format. The integer codes are decided by float arithmetic, so every value
// equals that of single IEEE operations in one fixed order: the sum adds the
// cells in turn (each int8 x binary16 product is exact, so a fused
// multiply-add rounds the same), the mean divides by n (a multiply by 1/4,
// 1/2 or 1 rounds the same), and each code is rint of the rounded quotient
// (computed from one reciprocal and an exact residual, which lands on the
// same integer).
//
// GB300 mapping: an elementwise pass over the cells (bound by instruction
// issue more than by HBM on this GPU). One warp per block; lane l
// owns d = 4l .. 4l+3, reads one 4-byte word of each present cell's row (a
// 128-byte line per row and warp) and writes one 16-byte key word and one
// 4-byte code word; the block's max |key| is a warp max over the float bit
// patterns (non-negative floats order like their bits).
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int SUM_WARPS = 8;

__global__ void __launch_bounds__(SUM_WARPS * 32)
    summary_kernel(const int8_t *__restrict__ kc, const __half *__restrict__ ks, int ncells, int b0, int nblk,
                   float *__restrict__ key, int8_t *__restrict__ kq8, __half *__restrict__ kscale) {
    grid_dependency_wait();   // the cells may come from the previous grid (the append itself)
    const int lane = threadIdx.x & 31;
    const int j = static_cast<int>(blockIdx.x) * SUM_WARPS + (threadIdx.x >> 5);
    if (j >= nblk) return;   // the whole warp
    const int b = b0 + j;
    int n = ncells - 4 * b;   // present cells (ncells and 4b + 4 fit in int: checked by the host)
    n = n > 4 ? 4 : (n < 0 ? 0 : n);

    // One 64-bit base per block; the 4 rows and scales sit at fixed offsets.
    const uint32_t *rows = reinterpret_cast<const uint32_t *>(kc + static_cast<size_t>(b) * (4 * D)) + lane;
    const __half *scl = ks + static_cast<size_t>(b) * 4;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (t < n) {
            w[t] = ld_in(rows + t * (D / 4));
            sc[t] = __half2float(__ushort_as_half(ld_in_u16(scl + t)));
        }
    }
    float m[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        // Each int8 x binary16 product is exact in fp32, so one fused
        // multiply-add rounds exactly like the multiply and the add in turn.
        float sum = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (t < n)
                sum = __fmaf_rn(static_cast<float>(static_cast<int8_t>((w[t] >> (8 * e)) & 0xFFu)), sc[t], sum);
        m[e] = sum;
    }
    // The mean: dividing by 4, 2 or 1 is multiplying by 0.25, 0.5 or 1 (one
    // rounding either way); only a block of 3 present cells divides (n is
    // the same across the warp, so this branch does not diverge).
    if (n == 3) {
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = __fdiv_rn(m[e], 3.0f);
    } else {
        const float inv = n == 4 ? 0.25f : (n == 2 ? 0.5f : 1.0f);   // n == 0 leaves the zero sums
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = __fmul_rn(m[e], inv);
    }
    const size_t out = static_cast<size_t>(b) * D + 4 * lane;
    if (key != nullptr) *reinterpret_cast<float4 *>(key + out) = make_float4(m[0], m[1], m[2], m[3]);
    if (kq8 != nullptr) {
        float top = fmaxf(fmaxf(fabsf(m[0]), fabsf(m[1])), fmaxf(fabsf(m[2]), fabsf(m[3])));
        top = __uint_as_float(__reduce_max_sync(FULL_MASK, __float_as_uint(top)));
        const __half sh = __float2half_rn(__fdiv_rn(top, 127.0f));
        const float s = __half2float(sh);
        // rint(m / s) without a division per code: q0 = rint(m * (1/s)) is
        // within one of it, and the residual r = m - q0 * s is exact in fp32
        // (q0 * s has at most 19 significant bits and |r| is about s / 2 or
        // less), so comparing |r| with s / 2 (exact) settles the nearest
        // integer, ties to even.
        uint32_t codes = 0u;
        if (s > 0.0f) {
            const float rs = __frcp_rn(s), hs = 0.5f * s;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q = rintf(__fmul_rn(m[e], rs));
                const float r = __fmaf_rn(-q, s, m[e]);
                const float ar = fabsf(r);
                const float step = r > 0.0f ? 1.0f : -1.0f;
                if (ar > hs || (ar == hs && fmodf(q, 2.0f) != 0.0f)) q += step;
                int c = static_cast<int>(q);
                c = c > 127 ? 127 : (c < -127 ? -127 : c);
                codes |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * e);
            }
        }
        *reinterpret_cast<uint32_t *>(kq8 + out) = codes;
        if (lane == 0) kscale[b] = sh;
    }
}

}  // namespace

cudaError_t launch_block_summary(const int8_t *kc, const uint16_t *ks, int ncells, int b0, int b1, float *key,
                                 int8_t *kq8, uint16_t *kscale, cudaStream_t stream) {
    const long long nblk = static_cast<long long>(b1) - b0;
    if (nblk <= 0) return cudaSuccess;
    if (4LL * b1 + 4 > 0x7FFFFFFFLL) return cudaErrorInvalidValue;   // cell indices stay in int
    const long long grid = (nblk + SUM_WARPS - 1) / SUM_WARPS;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(SUM_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, summary_kernel, kc, reinterpret_cast<const __half *>(ks),
                              ncells, b0, static_cast<int>(nblk), key, kq8,
                              reinterpret_cast<__half *>(kscale));
}

}  // namespace qsa

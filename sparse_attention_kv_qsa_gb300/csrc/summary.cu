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
// GB300 mapping: an elementwise pass over the cells. Eight lanes per block,
// four blocks per warp: lane l of a block's group owns d = 16 l .. 16 l + 15,
// reads 16 bytes of each present cell's row (a block's group reads whole
// 128-byte rows) and writes four 16-byte key words and one 16-byte code word;
// the block's max |key| is a maximum of float bit patterns over the group's
// 8 lanes (non-negative floats order like their bits). The per-block work
// that does not scale with d (the scale, its reciprocal, the block's cell
// count) is thus shared by 8 lanes instead of 32, which roughly halves the
// instructions per block.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int SUM_WARPS = 8;
constexpr int LANES_PER_BLOCK = 8;
constexpr int BLOCKS_PER_WARP = 32 / LANES_PER_BLOCK;

// Byte e of a word whose bytes were biased by 128 (xored with 0x80), as the
// signed int8 value it came from, exactly: the biased byte becomes the low
// mantissa bits of 2^23 (one byte permute), and subtracting 2^23 + 128
// leaves the value (one add; no integer-to-float conversion).
__device__ __forceinline__ float byte_f(uint32_t wx, int e) {
    return __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | static_cast<uint32_t>(e))) - 8388736.0f;
}

__global__ void __launch_bounds__(SUM_WARPS * 32)
    summary_kernel(const int8_t *__restrict__ kc, const __half *__restrict__ ks, int ncells, int b0, int nblk,
                   float *__restrict__ key, int8_t *__restrict__ kq8, __half *__restrict__ kscale) {
    grid_dependency_wait();   // the cells may come from the previous grid (the append itself)
    const int lane = threadIdx.x & 31, sub = lane & (LANES_PER_BLOCK - 1);
    const int j = (static_cast<int>(blockIdx.x) * SUM_WARPS + (threadIdx.x >> 5)) * BLOCKS_PER_WARP +
                  lane / LANES_PER_BLOCK;
    // A warp's four blocks may straddle the range's end: lanes past it run
    // with no present cell (the group shuffles need every lane) and store
    // nothing.
    const bool mine = j < nblk;
    const int b = b0 + j;
    int n = mine ? ncells - 4 * b : 0;   // present cells (ncells and 4b + 4 fit in int: checked by the host)
    n = n > 4 ? 4 : (n < 0 ? 0 : n);

    // One 64-bit base per block; the 4 rows and scales sit at fixed offsets.
    const uint4 *rows = reinterpret_cast<const uint4 *>(kc + static_cast<size_t>(mine ? b : 0) * (4 * D)) + sub;
    const __half *scl = ks + static_cast<size_t>(mine ? b : 0) * 4;
    uint4 w[4];
    float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        w[t] = make_uint4(0u, 0u, 0u, 0u);
        if (t < n) {
            w[t] = ld_in(rows + t * (D / 16));
            sc[t] = __half2float(__ushort_as_half(ld_in_u16(scl + t)));
        }
    }
    float m[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // Each int8 x binary16 product is exact in fp32, so one fused
            // multiply-add rounds exactly like the multiply and the add in turn.
            float sum = 0.0f;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (t < n) sum = __fmaf_rn(byte_f((&w[t].x)[q] ^ 0x80808080u, e), sc[t], sum);
            m[4 * q + e] = sum;
        }
    }
    // The mean: dividing by 4, 2 or 1 is multiplying by 0.25, 0.5 or 1 (one
    // rounding either way); only a block of 3 present cells divides.
    if (n == 3) {
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = __fdiv_rn(m[e], 3.0f);
    } else {
        const float inv = n == 4 ? 0.25f : (n == 2 ? 0.5f : 1.0f);   // n == 0 leaves the zero sums
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = __fmul_rn(m[e], inv);
    }
    const size_t out = static_cast<size_t>(b) * D + 16 * sub;
    if (key != nullptr && mine) {
        float4 *kp = reinterpret_cast<float4 *>(key + out);
#pragma unroll
        for (int q = 0; q < 4; ++q) kp[q] = make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
    }
    if (kq8 != nullptr) {
        // Per 4 consecutive d a float maximum, then the maximum of the bit
        // patterns over the block's 16 quads (NaN handled as before: a quad
        // of 4 NaN keeps NaN, whose bits are above every finite value).
        uint32_t tb = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tb = max(tb, __float_as_uint(fmaxf(fmaxf(fabsf(m[4 * q]), fabsf(m[4 * q + 1])),
                                               fmaxf(fabsf(m[4 * q + 2]), fabsf(m[4 * q + 3])))));
#pragma unroll
        for (int o = 1; o < LANES_PER_BLOCK; o <<= 1) tb = max(tb, __shfl_xor_sync(FULL_MASK, tb, o));
        const float top = __uint_as_float(tb);
        const __half sh = __float2half_rn(__fdiv_rn(top, 127.0f));
        const float s = __half2float(sh);
        // rint(m / s) without a division per code: q0 = rint(m * (1/s)) is
        // within one of it, and the residual r = m - q0 * s is exact in fp32
        // (q0 * s has at most 19 significant bits and |r| is about s / 2 or
        // less), so comparing |r| with s / 2 (exact) settles the nearest
        // integer, ties to even. m * (1/s) is below 2^22 in magnitude (about
        // 127 at most), so adding 1.5 * 2^23 rounds it to an integer (nearest,
        // ties to even: the sum's unit in the last place is 1), whose value is
        // the sum's low mantissa bits, and subtracting it back is exact.
        uint32_t codes[4] = {0u, 0u, 0u, 0u};
        if (s > 0.0f) {
            const float rs = __frcp_rn(s), hs = 0.5f * s;
            constexpr float RND = 12582912.0f;   // 1.5 * 2^23
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float t = __fadd_rn(__fmul_rn(m[e], rs), RND);
                const float q = __fsub_rn(t, RND);
                int c = __float_as_int(t) - __float_as_int(RND);
                const float r = __fmaf_rn(-q, s, m[e]);
                const float ar = fabsf(r);
                if (ar > hs || (ar == hs && (c & 1) != 0)) c += r > 0.0f ? 1 : -1;
                c = c > 127 ? 127 : (c < -127 ? -127 : c);
                codes[e >> 2] |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * (e & 3));
            }
        }
        if (mine) {
            *reinterpret_cast<uint4 *>(kq8 + out) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            if (sub == 0) kscale[b] = sh;
        }
    }
}

}  // namespace

cudaError_t launch_block_summary(const int8_t *kc, const uint16_t *ks, int ncells, int b0, int b1, float *key,
                                 int8_t *kq8, uint16_t *kscale, cudaStream_t stream) {
    const long long nblk = static_cast<long long>(b1) - b0;
    if (nblk <= 0) return cudaSuccess;
    if (4LL * b1 + 4 > 0x7FFFFFFFLL) return cudaErrorInvalidValue;   // cell indices stay in int
    constexpr long long per_cta = SUM_WARPS * BLOCKS_PER_WARP;
    const long long grid = (nblk + per_cta - 1) / per_cta;
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

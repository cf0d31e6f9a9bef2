// Block scoring for a handful of queries (decode: nq <= 4) on CUDA cores,
// one chunk of key rows at a time: shared by the decode scorer and the fused
// decode select.
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
// almost all padding. A key row is split over TPR threads (fp32: 4 threads x
// 32 values; int8: 2 threads x 64 values); each thread streams its part with
// 16-byte L2-only loads and accumulates one fp32 FMA chain per query
// against the head-summed queries in shared memory (read as broadcasts), and
// the TPR partial sums meet by warp shuffles. Rows at or beyond `active` are
// never read.
#pragma once

#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {

// Shared query rows get 4 floats of padding after every 32, so the TPR parts
// of a row (32 or 64 values apart) read different banks.
constexpr int DEC_QROW = D + D / 8;
__device__ __forceinline__ int dec_qidx(int d) { return d + (d >> 5) * 4; }

template <bool kInt8>
__host__ __device__ constexpr int dec_tpr() { return kInt8 ? 2 : 4; }   // threads per key row

// Head-summed queries into shared memory, zero past nq (the caller syncs).
template <int NQ, int THREADS>
__device__ __forceinline__ void dec_build_queries(const float *__restrict__ q, int nq, float (*qs)[DEC_QROW]) {
    for (int e = threadIdx.x; e < NQ * D; e += THREADS) {
        const int r = e / D, d = e % D;
        float v = 0.0f;
        if (r < nq) {
            const float *p = q + static_cast<size_t>(r) * (HEADS * D) + d;
            v = __fadd_rn(__fadd_rn(__fadd_rn(ld_in(p), ld_in(p + D)), ld_in(p + 2 * D)), ld_in(p + 3 * D));
        }
        qs[r][dec_qidx(d)] = v;
    }
}

// This thread's part of its key row in a chunk (16-byte words: 8 of fp32
// keys, 4 of int8 keys), loaded by dec_load_keys before the queries are built
// so that the two loads' round trips overlap.
template <bool kInt8>
struct DecKeys {
    uint4 w[kInt8 ? D / 2 / 16 : D / 4 / 4];
};

template <bool kInt8, int THREADS>
__device__ __forceinline__ void dec_load_keys(long long chunk, const float *__restrict__ kblk,
                                              const int8_t *__restrict__ kq8, int active, DecKeys<kInt8> &kv) {
    constexpr int TPR = dec_tpr<kInt8>();
    constexpr int PER = D / TPR;
    constexpr int ROWS = THREADS / TPR;
    const long long b = chunk * ROWS + threadIdx.x / TPR;   // key row
    const int part = static_cast<int>(threadIdx.x % TPR);
    constexpr int NW = sizeof(kv.w) / sizeof(uint4);
    if (b < active) {
        const uint4 *row = kInt8 ? reinterpret_cast<const uint4 *>(kq8 + b * D + part * PER)
                                 : reinterpret_cast<const uint4 *>(kblk + b * D + part * PER);
#pragma unroll
        for (int c = 0; c < NW; ++c) kv.w[c] = ld_in(row + c);
    } else {
#pragma unroll
        for (int c = 0; c < NW; ++c) kv.w[c] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Scores of key rows chunk * ROWS .. + ROWS - 1 (ROWS = THREADS / TPR) for
// all queries, from the keys dec_load_keys loaded for the same chunk, and,
// when gmax is given, the key of each of the chunk's 32-block groups'
// largest score (the chunk's rows are whole groups; their keys meet in gk and
// one warp per (query, group) takes the maximum). Every thread of the CTA
// calls this; it ends with the CTA synchronised.
template <int NQ, bool kInt8, int THREADS>
__device__ __forceinline__ void dec_score_chunk(const float (*qs)[DEC_QROW], long long chunk,
                                                const DecKeys<kInt8> &keys, const __half *__restrict__ kscale,
                                                int nq, int active, float *__restrict__ scores,
                                                uint32_t *__restrict__ gmax,
                                                uint32_t (*gk)[THREADS / dec_tpr<kInt8>()]) {
    constexpr int TPR = dec_tpr<kInt8>();
    constexpr int PER = D / TPR;                // values per thread: 64 (int8) or 32 (fp32)
    constexpr int ROWS = THREADS / TPR;
    static_assert(ROWS % GROUP_BLOCKS == 0, "a chunk holds whole groups");
    const long long b = chunk * ROWS + threadIdx.x / TPR;   // key row
    const int part = static_cast<int>(threadIdx.x % TPR);
    const bool live = b < active;
    float acc[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) acc[r] = 0.0f;
    if (live) {
        if constexpr (!kInt8) {
            float4 kv[PER / 4];
#pragma unroll
            for (int c = 0; c < PER / 4; ++c)
                kv[c] = make_float4(__uint_as_float(keys.w[c].x), __uint_as_float(keys.w[c].y),
                                    __uint_as_float(keys.w[c].z), __uint_as_float(keys.w[c].w));
#pragma unroll
            for (int c = 0; c < PER / 4; ++c) {
#pragma unroll
                for (int r = 0; r < NQ; ++r) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&qs[r][dec_qidx(part * PER + 4 * c)]);
                    acc[r] = fmaf(qv.x, kv[c].x, acc[r]);
                    acc[r] = fmaf(qv.y, kv[c].y, acc[r]);
                    acc[r] = fmaf(qv.z, kv[c].z, acc[r]);
                    acc[r] = fmaf(qv.w, kv[c].w, acc[r]);
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < PER / 16; ++c) {
                const uint32_t w4[4] = {keys.w[c].x, keys.w[c].y, keys.w[c].z, keys.w[c].w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    // int8 -> fp32 exactly, without a conversion instruction:
                    // the byte + 128 becomes the low mantissa bits of 2^23,
                    // and subtracting 2^23 + 128 leaves the value.
                    const uint32_t wx = w4[wi] ^ 0x80808080u;
                    float kf[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        kf[e] = __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | static_cast<uint32_t>(e))) -
                                8388736.0f;
#pragma unroll
                    for (int r = 0; r < NQ; ++r) {
                        const float4 qv =
                            *reinterpret_cast<const float4 *>(&qs[r][dec_qidx(part * PER + 16 * c + 4 * wi)]);
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
        const float scale = kInt8 ? __half2float(__ushort_as_half(ld_in_u16(kscale + b))) : 1.0f;
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
            if (kInt8) acc[r] = __fmul_rn(acc[r], scale);
            if (r < nq) scores[static_cast<size_t>(r) * active + b] = acc[r];
        }
    }
    if (gmax != nullptr) {   // uniform
        constexpr int GROUPS = ROWS / GROUP_BLOCKS;
        if (part == 0) {
            const int rl = threadIdx.x / TPR;
#pragma unroll
            for (int r = 0; r < NQ; ++r) gk[r][rl] = live ? score_key(acc[r]) : 0u;
        }
        __syncthreads();
        const int ngr = (active + GROUP_BLOCKS - 1) / GROUP_BLOCKS;
        const int lane = threadIdx.x & 31;
        for (int w = threadIdx.x >> 5; w < NQ * GROUPS; w += THREADS / 32) {   // warp-uniform
            const int r = w / GROUPS, gl = w % GROUPS;
            const uint32_t key = __reduce_max_sync(FULL_MASK, gk[r][gl * GROUP_BLOCKS + lane]);
            const long long g = chunk * GROUPS + gl;
            if (lane == 0 && r < nq && g < ngr) gmax[static_cast<size_t>(r) * ngr + g] = key;
        }
    }
    __syncthreads();   // gk may be rewritten by the next chunk
}

}  // namespace qsa

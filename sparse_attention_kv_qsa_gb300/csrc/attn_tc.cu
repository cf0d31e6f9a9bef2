// Attention of each query's 4 heads over the KV cells of its selected blocks
// on the tensor cores (mma.sync, fp16 operands, fp32 accumulation): the
// many-query path of qsa_sparse_attn, the same definition as csrc/attn.cu:
//
//   logit[h][c] = (sum_d q[i][h][d] * kq[c][d]) * ks[c] / sqrt(128)
//   out[i][h][d] = sum_c softmax_c(logit[h][.]) * vq[c][d] * vs[c]
//
// over the cells c = 4b .. 4b+3 (< ncells) of every listed block b of query i
// (negative or past-the-end ids are padding).
//
// Passage: "#3224 [Engine] perf(hip): tune RDNA4 QSA prompt WMMA path
// (STRATA_HIP_WMMA stays opt-in)", Summary items 1-3 and Evidence section 2:
// prompt attention runs on the matrix cores with q and p split into FP16
// high and low parts and is gated against an FP64 reference.
//
// GB300 mapping. One CTA per query (this path is taken when the queries alone
// fill the GPU): 16 warps up to the SM count, 8 warps (two CTAs per SM) up to
// twice it, 4 warps (four per SM) beyond, so every query of a call of up to
// 4x the SM count is resident at once and each SM runs 16 warps. A warp step
// covers two listed blocks (8 cells). The int8 K and V bytes are exact in fp16; q (per head) and the
// weights p * vs are split into a binary16 high part and a remainder scaled
// by 2^11, so two fp16 rows per head carry about 22 significant bits and the
// products accumulate in fp32:
//   q . k: A = the 4 heads' high rows (rows 0-3) and remainder rows (4-7),
//          B = 16 d x 8 cells, eight m16n8k16 MMAs over d = 0..127;
//   p . v: A = the weights of the 8 cells in the same row order, B = 8 cells
//          x 8 d, sixteen m16n8k8 MMAs over d = 0..127.
// High + remainder / 2^11 combine across the lanes 16 apart. Each warp keeps
// an online softmax per head (running maximum, normaliser, the head's 128
// outputs), in base 2, rescaling only in steps where a maximum moved. The K
// and V rows of a warp's next 3 steps are in flight at once: asynchronous
// 16-byte copies (through L2) into a 4-step ring in shared memory, so no
// registers wait for them; the cell scales load one step ahead. The warps'
// partials merge in warp order, so the output does not depend on
// scheduling.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

// A CTA of kWarps warps per query, 16 / kWarps CTAs per SM (the registers of
// 16 warps at most 128 each): 16 warps while the queries fit one CTA per SM,
// then 8 and 4, so that every query of a call up to 4 times the SM count is
// resident at once (one wave) and each SM holds 16 warps.
constexpr int STEP_IDS = 2;                              // listed blocks per warp step
constexpr int STAGES = 4;                                // steps in each warp's ring (a power of two)
// Dynamic shared memory: the warps' rings (16-byte slots [warp][stage][4][32])
// and each slot's first V cell per lane ([warp][stage][32]).
__host__ __device__ constexpr int ring_bytes(int warps) { return warps * STAGES * 4 * 32 * 16; }
__host__ __device__ constexpr int dyn_bytes(int warps) { return ring_bytes(warps) + warps * STAGES * 32 * 4; }
// Logits are kept in base-2 units: (q . k) * ks / sqrt(128) * log2(e), so the
// softmax weights are 2^(logit - max) (the same weights as e^ of the natural
// logits); log2(e) / sqrt(128), rounded to fp32.
constexpr float LOGIT2_SCALE = 0.12751743082459868f;

constexpr int ACC_HSTRIDE = 132, ACC_TSTRIDE = 33;    // per head, per 32 d
constexpr int ACC_WORDS = HEADS * ACC_HSTRIDE;
__host__ __device__ constexpr int acc_off(int h, int d) {
    return h * ACC_HSTRIDE + (d >> 5) * ACC_TSTRIDE + (d & 31);
}
static_assert(ACC_WORDS >= 16 * 32, "the q fragments fit a warp's accumulator rows");

template <int kWarps>
struct AttnShared {
    float m[kWarps][HEADS];                     // warp partials: running maximum,
    float l[kWarps][HEADS];                     // normaliser,
    // and unnormalised outputs, head h, d = 32 t + 16 e + u at acc_off(h, d):
    // rows padded so that the 16 lanes holding a (e, u) pair write distinct
    // banks (during the loop: the warp's q fragments).
    alignas(16) float acc[kWarps][ACC_WORDS];
};

// Two signed bytes of wx (bytes 0,1: sel 0x4140; bytes 2,3: sel 0x4342; wx
// the word with every byte's sign bit flipped, i.e. byte + 128) as an exact
// half2: 0x64 above each byte reads 1024 + byte + 128, minus 1152 leaves the
// byte.
__device__ __forceinline__ uint32_t i8x2_h2(uint32_t wx, uint32_t sel) {
    const uint32_t h = __byte_perm(wx, 0x64u, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), __halves2half2(__ushort_as_half(0x6480u),
                                                                                      __ushort_as_half(0x6480u)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// 2^e for -126 <= e <= 127 (a normal float).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// eq such that mx * 2^-eq lies in [2^14, 2^15) for a normal mx, clamped so
// that 2^eq and 2^-eq are normal floats (0 -> -126, inf or NaN -> 113).
__device__ __forceinline__ int q_exponent(float mx) {
    const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 14;
    return min(max(e, -126), 113);
}

// Exponent field of a binary16 pattern, read as 1 for zero and subnormals
// and as 30 for inf and NaN: |h| < 2^(result - 14) for finite h.
__device__ __forceinline__ uint32_t half_exponent(uint32_t h) { return min(max((h >> 10) & 31u, 1u), 30u); }

// (x, y) as a half2 of their high parts (binary16 rounding), or of their
// remainders times `scale` (rounded again), for the remainder rows.
__device__ __forceinline__ uint32_t split_pack(float x, float y, bool remainder, float scale) {
    const __half hx = __float2half_rn(x), hy = __float2half_rn(y);
    const __half2 r = remainder ? __floats2half2_rn((x - __half2float(hx)) * scale, (y - __half2float(hy)) * scale)
                                : __halves2half2(hx, hy);
    return *reinterpret_cast<const uint32_t *>(&r);
}

// D (rows g, g+8; columns 2t, 2t+1) += A (16 x 16, rows g+8 zero: a1 = a3 = 0)
// x B (16 x 8), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float &c0, float &c1, float &c2, float &c3, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Row g of D (columns 2t, 2t+1) += A (16 x 8, rows g+8 zero) x B (8 x 8); the
// zero rows' results are dropped.
// (d2 and d3 are asm outputs that nothing reads: the diagnostic for that is off here.)
#pragma nv_diag_suppress 550
__device__ __forceinline__ void mma_1688(float &c0, float &c1, uint32_t a0, uint32_t b0) {
    float d2, d3;   // rows g + 8 (zero): dropped
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %7, %7};"
        : "+f"(c0), "+f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(0u), "r"(b0), "f"(0.0f));
}
#pragma nv_diag_default 550

template <int kWarps>
__global__ void __launch_bounds__(kWarps * 32, 16 / kWarps)
    attn_tc_kernel(const float *__restrict__ q, const int8_t *__restrict__ kc, const __half *__restrict__ ks,
                const int8_t *__restrict__ vc, const __half *__restrict__ vs, int ncells,
                const int32_t *__restrict__ ids, int k, float *__restrict__ out) {
    constexpr int AT_THREADS = kWarps * 32;
    __shared__ AttnShared<kWarps> sh;
    extern __shared__ __align__(16) uint8_t attn_dyn[];   // dyn_bytes(kWarps)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = static_cast<int>(blockIdx.x);   // query
    const int32_t *ids_i = ids + static_cast<size_t>(i) * k;
    const int nblocks = (ncells + 3) / 4;

    grid_dependency_wait();   // q, the cells and the ids may come from the previous grid

    // Lane roles in the mma fragments: g = lane / 4 (a row of A, a column of
    // B), t = lane % 4. Rows 0-3 of A are the 4 heads' high parts, rows 4-7
    // their scaled remainders (rows 8-15 are zero), so a lane's rows belong to
    // head g % 4.
    const int g = lane >> 2, t = lane & 3;
    const int hd = g & 3;
    const bool lo_row = g >= 4;

    // q . k: K-step s covers d = 32 t + 4 s + {0, 1} (A columns 2t, 2t+1) and
    // d = 32 t + 4 s + {2, 3} (columns 2t+8, 2t+9); every lane of a column
    // group uses the same map, so A and B agree (a permutation of d).
    // The fragments (16 words per lane) live in the warp's part of sh.acc
    // until the warp partials are written: word 2 st + j of lane l at
    // [(2 st + j) * 32 + l] (lane-contiguous, conflict-free).
    uint32_t *aq = reinterpret_cast<uint32_t *>(&sh.acc[warp][0]);
    // Head hd's q enters the fragments times 2^-eq, which puts its largest
    // magnitude in [2^14, 2^15) (no binary16 overflow, no subnormal high
    // parts); the logits take the 2^eq back (qs).
    float qs;
    {
        const float4 *qh = reinterpret_cast<const float4 *>(q + (static_cast<size_t>(i) * HEADS + hd) * D + 32 * t);
        float4 x[8];
        float mx = 0.0f;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            x[st] = ld_in(qh + st);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x[st].x), fabsf(x[st].y)), fmaxf(fabsf(x[st].z), fabsf(x[st].w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 2));
        const int eq = q_exponent(mx);
        const float down = pow2f(-eq);
        qs = LOGIT2_SCALE * pow2f(eq);
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            aq[(2 * st) * 32 + lane] = split_pack(x[st].x * down, x[st].y * down, lo_row, 2048.0f);
            aq[(2 * st + 1) * 32 + lane] = split_pack(x[st].z * down, x[st].w * down, lo_row, 2048.0f);
        }
        __syncwarp();
    }

    const int nsteps = (k - 1) / STEP_IDS + 1;   // k >= 1
    // This warp's steps are wg, wg + nw, ...: the j-th is wg + j * nw.
    const int wg = warp, nw = kWarps;
    const int nj = wg < nsteps ? (nsteps - 1 - wg) / nw + 1 : 0;

    // Block ids 16 steps at a time: lane l holds block l % 2 of the warp's
    // step 16 c + l / 2 of chunk c (raw; -1 past k); the next chunk's ids
    // load while this one's are used. Blocks are checked when taken.
    auto chunk_ids = [&](int c) -> int {
        const int st = wg + (16 * c + (lane >> 1)) * nw, slot = STEP_IDS * st + (lane & 1);
        return st < nsteps && slot < k ? ld_in(ids_i + slot) : -1;
    };
    int id_chunk = 0, id_cur = chunk_ids(0), id_next = chunk_ids(1);
    auto step_block = [&](int j, int which) {   // warp-uniform j, nondecreasing over calls
        if ((j >> 4) != id_chunk) {
            id_chunk = j >> 4;
            id_cur = id_next;
            id_next = chunk_ids(id_chunk + 1);
        }
        const int b = __shfl_sync(FULL_MASK, id_cur, 2 * (j & 15) + which);
        return b >= 0 && b < nblocks ? b : -1;
    };

    // The warp's ring of STAGES steps: each lane copies its own rows into its
    // own slots, 16 bytes at a time, asynchronously through L2 (so only the
    // lane's own copies need waiting for): slot c of lane l at [c][l], c = 0, 1
    // its K bytes (cell g, d = 32 t .. +31), c = 2, 3 its V bytes (cells 2t,
    // 2t+1, d = 16 g .. +15); dead cells are not copied (their logits are
    // masked and their weights are 0, so stale bytes never count). cellv: the
    // lane's first V cell of the step, or -1.
    uint4 *ring = reinterpret_cast<uint4 *>(attn_dyn) + static_cast<size_t>(warp) * STAGES * 4 * 32;
    int *cellv = reinterpret_cast<int *>(attn_dyn + ring_bytes(kWarps)) + warp * STAGES * 32;
    auto issue = [&](int j) {
        const int b0 = step_block(j, 0), b1 = step_block(j, 1);
        const int sl = j & (STAGES - 1);
        uint4 *slot = ring + sl * 128;
        const int bk = (g >> 2) ? b1 : b0, ck = 4 * bk + (g & 3);
        if (bk >= 0 && ck < ncells) {
            const int8_t *src = kc + static_cast<size_t>(ck) * D + 32 * t;
            cp_async_16(slot + lane, src);
            cp_async_16(slot + 32 + lane, src + 16);
        }
        const int bv = (t >> 1) ? b1 : b0, cv = 4 * bv + 2 * (t & 1);
        if (bv >= 0 && cv < ncells) cp_async_16(slot + 64 + lane, vc + static_cast<size_t>(cv) * D + 16 * g);
        if (bv >= 0 && cv + 1 < ncells) cp_async_16(slot + 96 + lane, vc + static_cast<size_t>(cv + 1) * D + 16 * g);
        cp_async_commit();
        cellv[sl * 32 + lane] = bv >= 0 ? cv : -1;
    };
    // The binary16 scales of the lane's two V cells (K scales low, V scales
    // high half each): loaded one step before they are used.
    auto load_scales = [&](int j, uint32_t &kk, uint32_t &vv) {
        const int c0 = j < nj ? cellv[(j & (STAGES - 1)) * 32 + lane] : -1;
        const bool l0 = c0 >= 0 && c0 < ncells, l1 = c0 >= 0 && c0 + 1 < ncells;
        kk = (l0 ? ld_in_u16(ks + c0) : 0u) | (l1 ? static_cast<uint32_t>(ld_in_u16(ks + c0 + 1)) << 16 : 0u);
        vv = (l0 ? ld_in_u16(vs + c0) : 0u) | (l1 ? static_cast<uint32_t>(ld_in_u16(vs + c0 + 1)) << 16 : 0u);
    };

    float m = -INFINITY, lsum = 0.0f;   // head hd: running maximum; this lane's normaliser part
    // The weights enter the p . v MMAs as p * vs * 2^(29 - vf), vf the largest
    // binary16 exponent field of the value scales seen so far (warp-uniform),
    // so that they stay below 2^15; the outputs carry the same factor.
    uint32_t vf = 1;
    float sw = pow2f(28);
    // p . v accumulators: n-tile u, column n: head hd (high or remainder row),
    // d = 16 n + u with n = 2t, 2t+1 (a permutation of d for the B loads).
    float acc[16][2];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u][0] = acc[u][1] = 0.0f;

    auto run_step = [&](int j, uint32_t ksc, uint32_t vsc) {
        const int sl = j & (STAGES - 1);
        const uint4 *slot = ring + sl * 128;
        // Logits of cells 2t, 2t+1 for head hd: eight m16n8k16 MMAs.
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
        {
            const uint4 ka = slot[lane], kb = slot[32 + lane];
            const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint32_t wx = kw[st] ^ 0x80808080u;
                mma_16816(c0, c1, c2, c3, aq[(2 * st) * 32 + lane], aq[(2 * st + 1) * 32 + lane],
                          i8x2_h2(wx, 0x4140u), i8x2_h2(wx, 0x4342u));
            }
        }
        // High part + remainder (from the lane 16 apart), in the same order in both lanes.
        const float o0 = __shfl_xor_sync(FULL_MASK, c0, 16), o1 = __shfl_xor_sync(FULL_MASK, c1, 16);
        const float dot0 = (lo_row ? o0 : c0) + (lo_row ? c0 : o0) * (1.0f / 2048.0f);
        const float dot1 = (lo_row ? o1 : c1) + (lo_row ? c1 : o1) * (1.0f / 2048.0f);
        const int cell0 = cellv[sl * 32 + lane];
        const bool live0 = cell0 >= 0 && cell0 < ncells, live1 = cell0 >= 0 && cell0 + 1 < ncells;
        const float lg0 = live0 ? dot0 * __half2float(__ushort_as_half(static_cast<unsigned short>(ksc))) * qs : -INFINITY;
        const float lg1 = live1 ? dot1 * __half2float(__ushort_as_half(static_cast<unsigned short>(ksc >> 16))) * qs
                                : -INFINITY;
        // Online softmax of head hd over the step's 8 cells (lanes 4g .. 4g+3).
        float bm = fmaxf(lg0, lg1);
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 2));
        const float mn = fmaxf(m, bm);
        const float alpha = mn == -INFINITY ? 1.0f : exp2f(m - mn);
        const float p0 = live0 ? exp2f(lg0 - mn) : 0.0f;
        const float p1 = live1 ? exp2f(lg1 - mn) : 0.0f;
        m = mn;
        lsum = fmaf(lsum, alpha, p0 + p1);
        const uint32_t v0 = vsc & 0xFFFFu, v1 = vsc >> 16;   // 0 for dead cells
        const uint32_t f = __reduce_max_sync(FULL_MASK, max(half_exponent(v0), half_exponent(v1)));
        float shrink = 1.0f;
        if (f > vf) {   // warp-uniform: a larger value scale than any before
            shrink = pow2f(static_cast<int>(vf) - static_cast<int>(f));
            vf = f;
            sw = pow2f(29 - static_cast<int>(vf));
        }
        // Rescale only when some head's running maximum moved (alpha is
        // exactly 1 otherwise) or the weight factor shrank (powers of two).
        const float fac = alpha * shrink;
        if (__any_sync(FULL_MASK, fac != 1.0f)) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                acc[u][0] *= fac;
                acc[u][1] *= fac;
            }
        }
        // p * vs * 2^(29 - vf) as high part / scaled remainder.
        const float w0 = p0 * __half2float(__ushort_as_half(static_cast<unsigned short>(v0))) * sw;
        const float w1 = p1 * __half2float(__ushort_as_half(static_cast<unsigned short>(v1))) * sw;
        const uint32_t ap = split_pack(w0, w1, lo_row, 2048.0f);
        // p . v: sixteen m16n8k8 MMAs, n-tile u takes byte u of cells 2t and 2t+1.
        const uint4 sa = slot[64 + lane], sb = slot[96 + lane];
        const uint32_t va[4] = {sa.x ^ 0x80808080u, sa.y ^ 0x80808080u, sa.z ^ 0x80808080u, sa.w ^ 0x80808080u};
        const uint32_t vb[4] = {sb.x ^ 0x80808080u, sb.y ^ 0x80808080u, sb.z ^ 0x80808080u, sb.w ^ 0x80808080u};
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            const uint32_t lo2 = __byte_perm(va[wd], vb[wd], 0x5140u);   // a0 b0 a1 b1
            const uint32_t hi2 = __byte_perm(va[wd], vb[wd], 0x7362u);   // a2 b2 a3 b3
            mma_1688(acc[4 * wd + 0][0], acc[4 * wd + 0][1], ap, i8x2_h2(lo2, 0x4140u));
            mma_1688(acc[4 * wd + 1][0], acc[4 * wd + 1][1], ap, i8x2_h2(lo2, 0x4342u));
            mma_1688(acc[4 * wd + 2][0], acc[4 * wd + 2][1], ap, i8x2_h2(hi2, 0x4140u));
            mma_1688(acc[4 * wd + 3][0], acc[4 * wd + 3][1], ap, i8x2_h2(hi2, 0x4342u));
        }
    };

    // STAGES - 1 steps in flight ahead of the one being computed; every issue
    // commits one group (empty past the warp's last step), so waiting for all
    // but the STAGES - 1 newest groups leaves step j's rows in place. A stale
    // V byte of a dead cell stays a finite int8 value times a zero weight.
    for (int a = 0; a < STAGES - 1; ++a) issue(a);
    uint32_t ksc, vsc;
    load_scales(0, ksc, vsc);
    for (int j = 0; j < nj; ++j) {   // warp-uniform
        issue(j + STAGES - 1);
        cp_async_wait<STAGES - 1>();
        uint32_t nks, nvs;
        load_scales(j + 1, nks, nvs);
        run_step(j, ksc, vsc);
        ksc = nks;
        vsc = nvs;
    }
    cp_async_wait<0>();

    // Warp partials: head hd's normaliser sums over its 4 lanes; its outputs
    // are high part + remainder / 2^11 (from the lane 16 apart), / 2^(29 - vf).
    const float unscale = pow2f(static_cast<int>(vf) - 29);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 1);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 2);
    __syncwarp();   // the q fragments in sh.acc[warp] are no longer read
    if (g < HEADS && t == 0) {
        sh.m[warp][hd] = m;
        sh.l[warp][hd] = lsum;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float other = __shfl_xor_sync(FULL_MASK, acc[u][e], 16);
            if (!lo_row)
                sh.acc[warp][acc_off(hd, 16 * (2 * t + e) + u)] = (acc[u][e] + other * (1.0f / 2048.0f)) * unscale;
        }
    }
    __syncthreads();

    // The CTA's warps merged in warp order: thread = (head, d), HEADS * D / AT_THREADS each.
#pragma unroll 1
    for (int hd_i = threadIdx.x; hd_i < HEADS * D; hd_i += AT_THREADS) {
        const int h = hd_i >> 7, d = hd_i & (D - 1);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sh.m[w][h]);
        float A = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = sh.m[w][h];
                if (mw != -INFINITY) {
                    const float f = exp2f(mw - M);
                    A = fmaf(sh.acc[w][acc_off(h, d)], f, A);
                    L = fmaf(sh.l[w][h], f, L);
                }
            }
        }
        float *o = out + (static_cast<size_t>(i) * HEADS + h) * D + d;
        *o = L > 0.0f ? A / L : 0.0f;
    }
}

template <int kWarps>
cudaError_t launch_attn_tc(const float *q, const int8_t *kc, const uint16_t *ks, const int8_t *vc,
                           const uint16_t *vs, int ncells, const int32_t *ids, int nq, int k, float *out,
                           cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        const cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<kWarps>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_bytes(kWarps));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = dyn_bytes(kWarps);
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<kWarps>, q, kc, reinterpret_cast<const __half *>(ks), vc,
                              reinterpret_cast<const __half *>(vs), ncells, ids, k, out);
}

}  // namespace

cudaError_t launch_sparse_attn_tc(const float *q, const int8_t *kc, const uint16_t *ks, const int8_t *vc,
                                  const uint16_t *vs, int ncells, const int32_t *ids, int nq, int k, float *out,
                                  cudaStream_t stream) {
    if (ncells > 0x7FFFFFFF - 4) return cudaErrorInvalidValue;
    const int sms = device_sm_count();
    if (nq <= sms) return launch_attn_tc<16>(q, kc, ks, vc, vs, ncells, ids, nq, k, out, stream);
    if (nq <= 2 * sms) return launch_attn_tc<8>(q, kc, ks, vc, vs, ncells, ids, nq, k, out, stream);
    return launch_attn_tc<4>(q, kc, ks, vc, vs, ncells, ids, nq, k, out, stream);
}

}  // namespace qsa

// Attention of each query's 4 heads over the KV cells of its selected blocks
// (int8 K and V cells, one binary16 scale per cell for each).
//
//   logit[h][c] = (sum_d q[i][h][d] * kq[c][d]) * ks[c] / sqrt(128)
//   out[i][h][d] = sum_c softmax_c(logit[h][.]) * vq[c][d] * vs[c]
//
// over the cells c = 4b .. 4b+3 (< ncells) of every listed block b of query i
// (negative or past-the-end ids are padding).
//
// Passages: "#3224 [Engine] perf(hip): tune RDNA4 QSA prompt WMMA path
// (STRATA_HIP_WMMA stays opt-in)", Summary and Evidence section 2 (the QSA
// attention reads int8 K and V cells with binary16 k/v scales and is gated
// against an FP64 reference); "#3102 perf(hip): enable wave32 QSA decode
// attention and MMVQ row reuse on gfx12", item D5 (decode attention in
// chunks of cells whose partial results merge in sequential order).
//
// This file is the CUDA-core path, taken when there are fewer queries than
// SMs; csrc/attn_tc.cu holds the tensor-core path for more.
//
// GB300 mapping. A cluster of 2 or 4 CTAs of 16 warps per query (this kernel
// runs for at most half as many queries as SMs, decode included), so that
// the cells of one query stream through several SMs; a single CTA per query
// (no cluster) is kept for generality. A warp step covers two listed blocks
// (8 cells): every lane loads its 4 bytes (d = 4 lane .. +3) of each cell's
// K and V row (one 128-byte line per row and warp), forms the 8 x 4 partial
// dot products against its slice of the 4 head queries, and a butterfly
// reduce-scatter (31 shuffles) leaves lane l with the full logit of cell
// l / 4 for head l % 4. Each warp keeps an online softmax per head (running
// maximum, normaliser, and the head's 128 output values, 4 per lane), in
// base 2, rescaling the outputs only in steps where a maximum moved; the
// next step's rows are loaded before the current step is used. Partial
// results merge in a fixed order: the CTA's warps in warp order, then the
// cluster's CTAs in rank order through distributed shared memory, so the
// output does not depend on scheduling.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int AT_WARPS = 16;
constexpr int AT_THREADS = AT_WARPS * 32;
constexpr int STEP_IDS = 2;                              // listed blocks per warp step
constexpr int STEP_CELLS = STEP_IDS * 4;                 // 8 cells
// Logits are kept in base-2 units: (q . k) * ks / sqrt(128) * log2(e), so the
// softmax weights are 2^(logit - max) (the same weights as e^ of the natural
// logits); log2(e) / sqrt(128), rounded to fp32.
constexpr float LOGIT2_SCALE = 0.12751743082459868f;
constexpr int MAX_CLUSTER = 4;

struct AttnShared {
    alignas(16) float p[AT_WARPS][32];          // a step's weights times the value scales, per warp
    float m[AT_WARPS][HEADS];                   // warp partials: running maximum,
    float l[AT_WARPS][HEADS];                   // normaliser,
    alignas(16) float acc[AT_WARPS][HEADS][D];  // and unnormalised outputs
    float cm[HEADS], cl[HEADS];                 // the CTA's merged partial (read by rank 0)
    alignas(16) float cacc[HEADS][D];
};

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Lane l returns the warp-wide sum of v[l]: five halving steps, each lane
// keeping the half of its values selected by one bit of its lane index and
// adding the partner's copy of that half.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int n = 16; n >= 1; n >>= 1) {
        const bool up = (lane & n) != 0;
#pragma unroll
        for (int j = 0; j < n; ++j) {
            const float keep = up ? v[j + n] : v[j];
            const float send = up ? v[j] : v[j + n];
            v[j] = keep + __shfl_xor_sync(FULL_MASK, send, n);
        }
    }
    return v[0];
}

// The signed byte e of w as a float, exactly, without an integer-to-float
// conversion: with the sign bit flipped the byte is b + 128 in [0, 255];
// placed as the low mantissa byte of 2^23 it reads 2^23 + b + 128, and
// subtracting 2^23 + 128 leaves b.
__device__ __forceinline__ float byte_f(uint32_t w, int e) {
    const uint32_t bits = __byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540u + static_cast<uint32_t>(e));
    return __uint_as_float(bits) - 8388736.0f;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_kernel(const float *__restrict__ q, const int8_t *__restrict__ kc, const __half *__restrict__ ks,
                const int8_t *__restrict__ vc, const __half *__restrict__ vs, int ncells,
                const int32_t *__restrict__ ids, int k, float *__restrict__ out, int csize) {
    __shared__ AttnShared sh;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = csize > 1 ? cluster_ctarank() : 0u;
    const int i = static_cast<int>(blockIdx.x) / csize;   // query
    const int32_t *ids_i = ids + static_cast<size_t>(i) * k;
    const int nblocks = (ncells + 3) / 4;

    grid_dependency_wait();   // q, the cells and the ids may come from the previous grid

    float qv[HEADS][4];       // this lane's slice d = 4 lane .. +3 of each head's query
#pragma unroll
    for (int h = 0; h < HEADS; ++h) {
        const float4 t = ld_in(reinterpret_cast<const float4 *>(q + (static_cast<size_t>(i) * HEADS + h) * D) + lane);
        qv[h][0] = t.x, qv[h][1] = t.y, qv[h][2] = t.z, qv[h][3] = t.w;
    }

    const int nsteps = (k - 1) / STEP_IDS + 1;   // k >= 1
    const int wg = static_cast<int>(rank) * AT_WARPS + warp;
    const int nw = csize * AT_WARPS;

    // A step's data: its two listed blocks (-1 when past k, padding or past
    // the last block) and word `lane` of each of their cells' K and V rows
    // (0 for dead cells). Block and cell indices are 32-bit (the host keeps
    // ncells + 4 within int); each block's rows are addressed from one base.
    struct Step {
        int b[STEP_IDS];
        uint32_t kw[STEP_CELLS], vw[STEP_CELLS];
    };
    auto load_step = [&](int st, Step &s) {
#pragma unroll
        for (int j = 0; j < STEP_IDS; ++j) {
            const int slot = STEP_IDS * st + j;
            const int b = st < nsteps && slot < k ? ld_in(ids_i + slot) : -1;
            s.b[j] = b >= 0 && b < nblocks ? b : -1;
        }
#pragma unroll
        for (int j = 0; j < STEP_IDS; ++j) {
            const int b = s.b[j];
            const size_t base = static_cast<size_t>(b < 0 ? 0 : b) * (4 * D);
            const uint32_t *krow = reinterpret_cast<const uint32_t *>(kc + base) + lane;
            const uint32_t *vrow = reinterpret_cast<const uint32_t *>(vc + base) + lane;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const bool live = b >= 0 && 4 * b + t < ncells;
                s.kw[4 * j + t] = live ? ld_in(krow + t * (D / 4)) : 0u;
                s.vw[4 * j + t] = live ? ld_in(vrow + t * (D / 4)) : 0u;
            }
        }
    };

    const int mc = lane >> 2;                  // this lane holds the logit of cell mc for head lane % 4
    float m = -INFINITY, lsum = 0.0f;          // that head: running maximum, this lane's normaliser part
    float acc[HEADS][4];
#pragma unroll
    for (int h = 0; h < HEADS; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = 0.0f;

    auto run_step = [&](const Step &s) {
        float v[32];   // v[4 c + h]: this lane's part of cell c's dot product with head h
#pragma unroll
        for (int c = 0; c < STEP_CELLS; ++c) {
            const float k0 = byte_f(s.kw[c], 0), k1 = byte_f(s.kw[c], 1);
            const float k2 = byte_f(s.kw[c], 2), k3 = byte_f(s.kw[c], 3);
#pragma unroll
            for (int h = 0; h < HEADS; ++h)
                v[4 * c + h] = fmaf(qv[h][3], k3, fmaf(qv[h][2], k2, fmaf(qv[h][1], k1, qv[h][0] * k0)));
        }
        const float dot = reduce_scatter32(v, lane);
        const int b = (mc >> 2) != 0 ? s.b[1] : s.b[0];
        const int cell = 4 * b + (mc & 3);
        const bool live = b >= 0 && cell < ncells;
        const float logit = live ? dot * __half2float(__ushort_as_half(ld_in_u16(ks + cell))) * LOGIT2_SCALE : -INFINITY;

        // Online softmax of head lane % 4 over this step's cells (the lanes with that head).
        float bm = logit;
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 16));
        const float mn = fmaxf(m, bm);
        const float alpha = mn == -INFINITY ? 1.0f : exp2f(m - mn);
        const float p = live ? exp2f(logit - mn) : 0.0f;
        m = mn;
        lsum = fmaf(lsum, alpha, p);
        sh.p[warp][lane] = live ? p * __half2float(__ushort_as_half(ld_in_u16(vs + cell))) : 0.0f;
        __syncwarp();
        // Rescale the outputs only when some head's running maximum moved
        // (alpha is exactly 1 otherwise; the test is warp-uniform).
        if (__any_sync(FULL_MASK, alpha != 1.0f)) {
            float al[HEADS];
#pragma unroll
            for (int h = 0; h < HEADS; ++h) al[h] = __shfl_sync(FULL_MASK, alpha, h);
#pragma unroll
            for (int h = 0; h < HEADS; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[h][e] *= al[h];
        }
#pragma unroll
        for (int c = 0; c < STEP_CELLS; ++c) {
            const float4 pc = *reinterpret_cast<const float4 *>(&sh.p[warp][4 * c]);   // heads 0..3
            const float pw[HEADS] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float ve = byte_f(s.vw[c], e);
#pragma unroll
                for (int h = 0; h < HEADS; ++h) acc[h][e] = fmaf(pw[h], ve, acc[h][e]);
            }
        }
        __syncwarp();   // sh.p is rewritten by the next step
    };

    // Two step buffers in turn: the next step's rows load while this one runs.
    Step s0, s1;
    int st = wg;
    load_step(st, s0);
    while (st < nsteps) {   // warp-uniform
        load_step(st + nw, s1);
        run_step(s0);
        st += nw;
        if (st >= nsteps) break;
        load_step(st + nw, s0);
        run_step(s1);
        st += nw;
    }

    // Warp partials: the normaliser of head lane % 4 sums over the lanes holding it.
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 4);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 8);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 16);
    if (lane < HEADS) {
        sh.m[warp][lane] = m;
        sh.l[warp][lane] = lsum;
    }
#pragma unroll
    for (int h = 0; h < HEADS; ++h)
        *reinterpret_cast<float4 *>(&sh.acc[warp][h][4 * lane]) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    __syncthreads();

    // The CTA's warps merged in warp order: thread = (head, d).
    const int h = threadIdx.x >> 7, d = threadIdx.x & (D - 1);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < AT_WARPS; ++w) M = fmaxf(M, sh.m[w][h]);
    float A = 0.0f, L = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < AT_WARPS; ++w) {
            const float mw = sh.m[w][h];
            if (mw != -INFINITY) {
                const float f = exp2f(mw - M);
                A = fmaf(sh.acc[w][h][d], f, A);
                L = fmaf(sh.l[w][h], f, L);
            }
        }
    }
    float *o = out + (static_cast<size_t>(i) * HEADS + h) * D + d;
    if (csize == 1) {
        *o = L > 0.0f ? A / L : 0.0f;
        return;
    }
    // The cluster's CTAs merged by rank 0, in rank order.
    sh.cacc[h][d] = A;
    if (d == 0) {
        sh.cm[h] = M;
        sh.cl[h] = L;
    }
    cluster_sync_all();
    if (rank == 0) {
        float Mc = -INFINITY, mr[MAX_CLUSTER];
#pragma unroll
        for (int r = 0; r < MAX_CLUSTER; ++r) {
            mr[r] = -INFINITY;
            if (r < csize) mr[r] = ld_shared_cluster_f32(map_shared_rank(smem_u32(&sh.cm[h]), r));
            Mc = fmaxf(Mc, mr[r]);
        }
        float Ac = 0.0f, Lc = 0.0f;
        if (Mc != -INFINITY) {
#pragma unroll
            for (int r = 0; r < MAX_CLUSTER; ++r) {
                if (r < csize && mr[r] != -INFINITY) {
                    const float f = exp2f(mr[r] - Mc);
                    Ac = fmaf(ld_shared_cluster_f32(map_shared_rank(smem_u32(&sh.cacc[h][d]), r)), f, Ac);
                    Lc = fmaf(ld_shared_cluster_f32(map_shared_rank(smem_u32(&sh.cl[h]), r)), f, Lc);
                }
            }
        }
        *o = Lc > 0.0f ? Ac / Lc : 0.0f;
    }
    cluster_sync_all();   // no CTA leaves while rank 0 may still read it
}

}  // namespace

cudaError_t launch_sparse_attn(const float *q, const int8_t *kc, const uint16_t *ks, const int8_t *vc,
                               const uint16_t *vs, int ncells, const int32_t *ids, int nq, int k, float *out,
                               cudaStream_t stream) {
    // More queries than half the SMs (where this kernel would run one CTA per
    // query, without a cluster): the tensor-core kernel (csrc/attn_tc.cu),
    // measured faster there (100 queries: 35.5 against 41.6 us); fewer: this
    // one, whose clusters spread each query over 2 or 4 SMs (64 queries: 27.3
    // against 35.5 us).
    const int sms = device_sm_count();
    if (2 * nq > sms) return launch_sparse_attn_tc(q, kc, ks, vc, vs, ncells, ids, nq, k, out, stream);
    // Few queries: a cluster per query spreads its cells over several SMs.
    int csize = 1;
    for (int c = MAX_CLUSTER; c > 1; c >>= 1) {
        if (static_cast<long long>(nq) * c <= sms) {
            csize = c;
            break;
        }
    }
    const long long grid = static_cast<long long>(nq) * csize;
    if (grid > 0x7FFFFFFFLL || ncells > 0x7FFFFFFF - 4) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(AT_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = static_cast<unsigned>(csize);
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, attn_kernel, q, kc, reinterpret_cast<const __half *>(ks), vc,
                              reinterpret_cast<const __half *>(vs), ncells, ids, k, out, csize);
}

}  // namespace qsa

// Exact per-query top-k over block scores: MSD radix select with 8-bit
// digits, one thread-block cluster per query row.
//
// Method ("#3108 optimize exact QSA block scoring and top-k selection on
// gfx12", Summary item 2: radix-bin search with parallel prefix scans;
// "#337 gfx12 QSA select", What item 1: the selection is bounded by the
// batch's active blocks, never the capacity):
//  1. Each fp32 score maps to an order-preserving uint32 key (-0 -> +0,
//     negatives bit-inverted, positives with the sign bit set; NaN -> 0, the
//     lowest key).
//  2. Up to four passes, most significant byte first. A pass builds a 256-bin
//     histogram of the current digit over the keys that match the prefix
//     fixed so far, sums the histograms of the cluster's CTAs through
//     distributed shared memory, and scans the bins from the top to find the
//     bin where the running count reaches the number still to select. That
//     bin's digit extends the prefix; the count above it is taken.
//  3. Ordered gather: keys above the prefix are selected; keys equal to it
//     are selected in ascending id order until k ids are taken (ties to the
//     lower block id). Ids are written in ascending order.
//
// GB300 layout: a row of `active` scores is split into C <= 8 contiguous
// chunks, one per CTA of a cluster. Each chunk is copied once from global
// memory into shared memory with a 1-D bulk async copy (the misaligned head
// and tail with plain loads); all passes then run from shared memory, so
// each score crosses HBM once. Cluster barriers order the passes.
#include <cooperative_groups.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int TOPK_THREADS = 256;
constexpr int TOPK_WARPS = TOPK_THREADS / 32;
constexpr int BINS = 256;
constexpr int CLUSTER_MAX = 8;
constexpr int CHUNK_MAX = 49152;     // keys per CTA: 192 KiB of shared memory
constexpr int CHUNK_TARGET = 16384;  // preferred keys per CTA (64 KiB)
constexpr int CHUNK_MIN_SPLIT = 2048;

__device__ uint32_t g_topk_error;

struct TopkShared {
    uint32_t hist[2][BINS];  // per-pass digit histograms (double-buffered: read remotely)
    uint32_t warp_tot[TOPK_WARPS];
    uint32_t warp_gt[TOPK_WARPS];
    uint32_t warp_eq[TOPK_WARPS];
    uint32_t sel_bin, sel_excl, sel_cnt;
    uint32_t cnt_gt, cnt_eq;  // this CTA's gather counts (read remotely)
    uint32_t pad_;
    uint64_t mbar;
};

constexpr int KEYS_OFFSET = (sizeof(TopkShared) + 15) / 16 * 16;

__device__ __forceinline__ uint32_t float_bits_to_key(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN ranks lowest
    if (u == 0x80000000u) u = 0u;                     // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(TOPK_THREADS)
    topk_cluster_kernel(const float *__restrict__ scores, int active, int k, int chunk,
                        int32_t *__restrict__ ids) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int r = static_cast<int>(cluster.block_rank());
    const size_t row = blockIdx.x / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    TopkShared &sh = *reinterpret_cast<TopkShared *>(smem_raw);
    uint32_t *kbuf = reinterpret_cast<uint32_t *>(smem_raw + KEYS_OFFSET);

    const int c0 = min(active, r * chunk);
    const int c1 = min(active, c0 + chunk);
    const int n = c1 - c0;
    const float *g = scores + row * static_cast<size_t>(active) + c0;

    // Element i of the chunk lives at kb[i]; kb + head is 16-byte aligned so
    // the aligned body can be bulk-copied.
    const uintptr_t addr = reinterpret_cast<uintptr_t>(g);
    int head = static_cast<int>(((16u - (addr & 15u)) & 15u) >> 2);
    if (head > n) head = n;
    const int body = (n - head) & ~3;
    const int tail0 = head + body;
    uint32_t *kb = kbuf + ((4 - head) & 3);

    if (tid == 0) {
        mbar_init(&sh.mbar, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0 && body > 0) {
        mbar_arrive_expect_tx(&sh.mbar, static_cast<uint32_t>(body) * 4u);
        bulk_g2s(kb + head, g + head, static_cast<uint32_t>(body) * 4u, &sh.mbar);
    }
    const uint32_t *gu = reinterpret_cast<const uint32_t *>(g);
    for (int i = tid; i < head; i += TOPK_THREADS) kb[i] = gu[i];
    for (int i = tail0 + tid; i < n; i += TOPK_THREADS) kb[i] = gu[i];
    for (int i = tid; i < BINS; i += TOPK_THREADS) sh.hist[0][i] = 0u;
    if (body > 0 && !mbar_wait(&sh.mbar, 0)) atomicOr(&g_topk_error, 1u);
    __syncthreads();

    uint32_t prefix = 0u, mask = 0u;
    uint32_t kk = static_cast<uint32_t>(k);  // still to select among keys matching prefix

#pragma unroll 1
    for (int p = 0; p < 4; ++p) {
        const int shift = 24 - 8 * p;
        uint32_t *hist = sh.hist[p & 1];
        if (p > 0) {
            for (int i = tid; i < BINS; i += TOPK_THREADS) hist[i] = 0u;
            __syncthreads();
        }
        // Digit histogram of the matching keys (warp-aggregated increments:
        // the leading digit is heavily skewed, as exponents cluster).
#pragma unroll 1
        for (int i0 = 0; i0 < n; i0 += TOPK_THREADS) {
            const int i = i0 + tid;
            const bool valid = i < n;
            uint32_t key = 0u;
            if (valid) {
                key = kb[i];
                if (p == 0) {
                    key = float_bits_to_key(key);
                    kb[i] = key;
                }
            }
            const bool match = valid && ((key & mask) == prefix);
            const uint32_t bin = (key >> shift) & 0xFFu;
            const uint32_t who = __ballot_sync(FULL_MASK, match);
            if (match) {
                const uint32_t peers = __match_any_sync(who, bin);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
            }
        }
        cluster.sync();

        // Thread t owns bin 255 - t; an inclusive scan over t counts the keys
        // whose digit is >= that bin, across the whole cluster.
        const uint32_t bin = static_cast<uint32_t>(BINS - 1 - tid);
        uint32_t cnt = 0u;
        for (int rr = 0; rr < C; ++rr) cnt += cluster.map_shared_rank(hist, rr)[bin];
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sh.warp_tot[warp] = incl;
        __syncthreads();
        for (int w = 0; w < warp; ++w) incl += sh.warp_tot[w];
        const uint32_t excl = incl - cnt;
        if (excl < kk && incl >= kk) {
            sh.sel_bin = bin;
            sh.sel_excl = excl;
            sh.sel_cnt = cnt;
        }
        __syncthreads();
        kk -= sh.sel_excl;
        prefix |= sh.sel_bin << shift;
        mask |= 0xFFu << shift;
        if (sh.sel_cnt == kk) break;  // every key with this prefix is taken
    }

    // Ordered gather. Warp w owns the contiguous range [w*L, w*L + L) of the
    // chunk; ids leave in ascending order.
    const int L = ((n + TOPK_WARPS - 1) / TOPK_WARPS + 31) & ~31;
    const int w0 = min(n, warp * L), w1 = min(n, w0 + L);
    uint32_t gt = 0u, eq = 0u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool v = i < w1;
        const uint32_t km = v ? (kb[i] & mask) : 0u;
        gt += __popc(__ballot_sync(FULL_MASK, v && km > prefix));
        eq += __popc(__ballot_sync(FULL_MASK, v && km == prefix));
    }
    if (lane == 0) {
        sh.warp_gt[warp] = gt;
        sh.warp_eq[warp] = eq;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t a = 0u, b = 0u;
        for (int w = 0; w < TOPK_WARPS; ++w) {
            a += sh.warp_gt[w];
            b += sh.warp_eq[w];
        }
        sh.cnt_gt = a;
        sh.cnt_eq = b;
    }
    cluster.sync();

    // Offsets of this CTA, then of this warp, in selected and in tied keys.
    uint32_t eq_run = 0u, sel_run = 0u;
    for (int rr = 0; rr < r; ++rr) {
        const uint32_t rgt = *cluster.map_shared_rank(&sh.cnt_gt, rr);
        const uint32_t req = *cluster.map_shared_rank(&sh.cnt_eq, rr);
        const uint32_t take = kk > eq_run ? min(kk - eq_run, req) : 0u;
        sel_run += rgt + take;
        eq_run += req;
    }
    for (int w = 0; w < warp; ++w) {
        const uint32_t take = kk > eq_run ? min(kk - eq_run, sh.warp_eq[w]) : 0u;
        sel_run += sh.warp_gt[w] + take;
        eq_run += sh.warp_eq[w];
    }
    int32_t *out = ids + row * static_cast<size_t>(k);
    const uint32_t lt = lanemask_lt();
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool v = i < w1;
        const uint32_t km = v ? (kb[i] & mask) : 0u;
        const bool is_gt = v && km > prefix;
        const bool is_eq = v && km == prefix;
        const uint32_t eqm = __ballot_sync(FULL_MASK, is_eq);
        const bool sel = is_gt || (is_eq && eq_run + __popc(eqm & lt) < kk);
        const uint32_t selm = __ballot_sync(FULL_MASK, sel);
        if (sel) out[sel_run + __popc(selm & lt)] = c0 + i;
        eq_run += __popc(eqm);
        sel_run += __popc(selm);
    }
    cluster.sync();  // keep this CTA's shared memory alive for remote readers
}

__global__ void topk_all_kernel(int active, int k, size_t total, int32_t *__restrict__ ids) {
    for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(t % static_cast<size_t>(k));
        ids[t] = j < active ? j : -1;
    }
}

}  // namespace

cudaError_t launch_topk(const float *scores, int nq, int active, int k, int32_t *ids,
                        cudaStream_t stream) {
    // Cluster size: enough CTAs that no chunk exceeds CHUNK_TARGET keys (or
    // CHUNK_MAX at 8 CTAs); for few rows, more CTAs per row to occupy the SMs.
    const int sms = device_sm_count();
    int C = (active + CHUNK_TARGET - 1) / CHUNK_TARGET;
    while (C < CLUSTER_MAX && static_cast<long long>(nq) * C < sms &&
           active / (2 * C) >= CHUNK_MIN_SPLIT)
        C *= 2;
    if (C > CLUSTER_MAX) C = CLUSTER_MAX;
    if (C < 1) C = 1;
    const int chunk = (active + C - 1) / C;
    if (chunk > CHUNK_MAX) return cudaErrorInvalidValue;
    const size_t smem = KEYS_OFFSET + (static_cast<size_t>(chunk) + 4) * sizeof(uint32_t);

    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             KEYS_OFFSET + (CHUNK_MAX + 4) * 4);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(nq) * C), 1, 1);
    cfg.blockDim = dim3(TOPK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, active, k, chunk, ids);
}

cudaError_t launch_topk_all(int nq, int active, int k, int32_t *ids, cudaStream_t stream) {
    const size_t total = static_cast<size_t>(nq) * static_cast<size_t>(k);
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    topk_all_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(active, k, total, ids);
    return cudaGetLastError();
}

cudaError_t topk_error_read_clear(uint32_t *word, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_topk_error, sizeof(uint32_t), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_topk_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace qsa

// Exact per-query top-k over block scores: MSD radix select, one CTA per
// query row.
//
// Method ("#3108 optimize exact QSA block scoring and top-k selection on
// gfx12", Summary item 2: radix-bin search with parallel prefix scans;
// "#337 gfx12 QSA select", What item 1: the selection is bounded by the
// batch's active blocks, never the capacity):
//  1. Each fp32 score maps to an order-preserving uint32 key: -0 becomes +0
//     and NaN becomes -inf (x + 0 then max(., -inf)), negatives are
//     bit-inverted and positives get the sign bit set.
//  2. The digits are bits 31..21 (11 bits), then 20..13, 12..5 and 4..0. For
//     each digit, a histogram of the keys that match the prefix fixed so far
//     is scanned from the top bin to find the bin where the running count
//     reaches the number still to select; that digit extends the prefix and
//     the count above it is taken. A bin taken whole ends the search early.
//  3. Keys above the final prefix are selected; keys equal to it are ties,
//     taken in ascending id order until k ids are selected (ties go to the
//     lower block id). Ids leave in ascending order.
//
// GB300 layout. One 512-thread CTA owns one row and streams it with
// vectorised read-only loads (16 B per thread, four in flight):
//  Pass A reads the row from HBM and builds the 11-bit histogram in shared
//  memory.
//  Pass B streams the row again -- from L2, where pass A just left it -- and
//  marks keys above the leading bin in a shared-memory selection bitmap while
//  listing the keys inside it (~1% of a row for smooth data) as candidates.
//  The later digits visit only that candidate list (if it would overflow its
//  capacity, they re-stream the row and filter by prefix instead).
// No CTA ever waits on another: no cluster, no grid-wide synchronisation, no
// global scratch.
#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int ROW_THREADS = 512;
constexpr int ROW_WARPS = ROW_THREADS / 32;
constexpr int HIST_A = 2048;             // leading digit: bits 31..21
constexpr int GROUP = 8;                 // leading-digit bins per group
constexpr int NGROUPS = HIST_A / GROUP;  // 256: one group per thread
constexpr int BINS_R = 256;              // refinement digits: 20..13, 12..5, 4..0
constexpr int UNROLL = 4;                // 16-byte loads in flight per thread
constexpr int CAND_MAX = 2048;           // candidate-list capacity
constexpr int MAX_ACTIVE = 393216;

__device__ uint32_t g_topk_error;

struct RowShared {
    uint32_t histA[HIST_A];
    uint32_t groupA[NGROUPS];
    uint32_t histR[BINS_R];
    uint32_t cand_key[CAND_MAX];
    uint32_t cand_idx[CAND_MAX];
    uint32_t scan_tot[ROW_WARPS];
    uint32_t sel_bin, sel_excl, sel_cnt;
    uint32_t t1_bin, t1_above, t1_cnt;
    uint32_t cand_n, n_tie;
};

constexpr size_t SHARED_BYTES = (sizeof(RowShared) + 15) / 16 * 16;

__host__ __device__ constexpr size_t row_smem_bytes(int active) {
    return SHARED_BYTES + 2 * static_cast<size_t>((active + 31) / 32) * 4;
}

__device__ __forceinline__ uint32_t float_bits_to_key(uint32_t bits) {
    // -0 + 0 = +0 and max(NaN, -inf) = -inf; the compiler may not drop either
    // step (no fast-math), so ties and NaN follow the documented order.
    const float f = fmaxf(__fadd_rn(__uint_as_float(bits), 0.0f), -INFINITY);
    const uint32_t u = __float_as_uint(f);
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Block-wide exclusive prefix sum over threads (every thread must call).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *tot, int lane, int warp) {
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0u;
    for (int w = 0; w < warp; ++w) before += tot[w];
    __syncthreads();
    return before + incl - v;
}

// Thread t holds the count of item 255 - t (items in descending order).
// Finds the item at which the running count from the top reaches kk; leaves
// it, the count above it and its own count in sh.sel_*.
__device__ __forceinline__ void select_desc(uint32_t cnt, uint32_t kk, RowShared &sh, int tid, int lane,
                                            int warp) {
    const uint32_t excl = block_excl_scan(cnt, sh.scan_tot, lane, warp);
    if (excl < kk && excl + cnt >= kk) {
        sh.sel_bin = static_cast<uint32_t>(BINS_R - 1 - tid);
        sh.sel_excl = excl;
        sh.sel_cnt = cnt;
    }
    __syncthreads();
}

// Calls fn(i, bits) once for every element of the row (row index i, raw
// fp32 bits), each from some thread; every thread must call it. The aligned
// body moves as 16-byte read-only loads, UNROLL in flight per thread; the
// <= 3 ragged scores at either end as single words.
template <typename Fn>
__device__ __forceinline__ void stream_row(const uint32_t *g, int n, int head, int nvec, int tid, Fn &&fn) {
    for (int i = tid; i < head; i += ROW_THREADS) fn(i, __ldg(g + i));
    for (int i = head + 4 * nvec + tid; i < n; i += ROW_THREADS) fn(i, __ldg(g + i));
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g + head);
#pragma unroll 1
    for (int v0 = 0; v0 < nvec; v0 += ROW_THREADS * UNROLL) {
        uint4 x[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int v = v0 + u * ROW_THREADS + tid;
            x[u] = v < nvec ? __ldg(g4 + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int v = v0 + u * ROW_THREADS + tid;
            if (v < nvec) {
                const int i = head + 4 * v;
                fn(i, x[u].x);
                fn(i + 1, x[u].y);
                fn(i + 2, x[u].z);
                fn(i + 3, x[u].w);
            }
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(ROW_THREADS)
    topk_row_kernel(const float *__restrict__ scores, int active, int k, int32_t *__restrict__ ids) {
    const size_t row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = active;
    const int nwords = (n + 31) >> 5;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem_raw);
    uint32_t *selbits = reinterpret_cast<uint32_t *>(smem_raw + SHARED_BYTES);
    uint32_t *tiebits = selbits + nwords;

    const uint32_t *g = reinterpret_cast<const uint32_t *>(scores + row * static_cast<size_t>(n));
    const uintptr_t addr = reinterpret_cast<uintptr_t>(g);
    int head = static_cast<int>(((16u - (addr & 15u)) & 15u) >> 2);
    if (head > n) head = n;
    const int nvec = (n - head) >> 2;

    if (tid == 0) {
        sh.cand_n = 0u;
        sh.n_tie = 0u;
    }
    for (int i = tid; i < HIST_A; i += ROW_THREADS) sh.histA[i] = 0u;
    for (int i = tid; i < nwords; i += ROW_THREADS) {
        selbits[i] = 0u;
        tiebits[i] = 0u;
    }
    __syncthreads();

    // Pass A: the 11-bit leading-digit histogram.
    stream_row(g, n, head, nvec, tid, [&](int, uint32_t bits) {
        atomicAdd(&sh.histA[float_bits_to_key(bits) >> 21], 1u);
    });
    if (tid < NGROUPS) {
        const uint4 a = *reinterpret_cast<const uint4 *>(&sh.histA[tid * GROUP]);
        const uint4 b = *reinterpret_cast<const uint4 *>(&sh.histA[tid * GROUP + 4]);
        sh.groupA[tid] = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
    }
    __syncthreads();
    uint32_t kk = static_cast<uint32_t>(k);
    select_desc(tid < NGROUPS ? sh.groupA[NGROUPS - 1 - tid] : 0u, kk, sh, tid, lane, warp);
    if (warp == 0) {
        const uint32_t grp = sh.sel_bin, above = sh.sel_excl;
        const uint32_t b = grp * GROUP + (GROUP - 1) - static_cast<uint32_t>(lane);
        const uint32_t c = lane < GROUP ? sh.histA[b] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane < GROUP && above + incl - c < kk && above + incl >= kk) {
            sh.t1_bin = b;
            sh.t1_above = above + incl - c;
            sh.t1_cnt = c;
        }
    }
    __syncthreads();
    const uint32_t T1 = sh.t1_bin;
    kk -= sh.t1_above;
    const bool doneA = sh.t1_cnt == kk;  // the whole leading bin is taken
    const bool compact = !doneA && sh.t1_cnt <= static_cast<uint32_t>(CAND_MAX);

    // Pass B: keys above the leading bin are selected; keys inside it are
    // listed as candidates (or all selected, when the bin is taken whole).
    stream_row(g, n, head, nvec, tid, [&](int i, uint32_t bits) {
        const uint32_t key = float_bits_to_key(bits);
        const uint32_t d = key >> 21;
        if (d < T1) return;
        if (d > T1 || doneA) {
            atomicOr(&selbits[i >> 5], 1u << (i & 31));
        } else if (compact) {
            const uint32_t slot = atomicAdd(&sh.cand_n, 1u);
            if (slot < static_cast<uint32_t>(CAND_MAX)) {
                sh.cand_key[slot] = key;
                sh.cand_idx[slot] = static_cast<uint32_t>(i);
            }
        }
    });

    // Refinement digits over the candidates.
    uint32_t prefix = T1 << 21, mask = 0xFFE00000u;
    bool done = doneA;
    int shift = 21;
    const int m = min(static_cast<int>(sh.cand_n), CAND_MAX);
#pragma unroll 1
    for (int p = 0; p < 3 && !done; ++p) {
        const int width = p < 2 ? 8 : 5;
        shift -= width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int i = tid; i < BINS_R; i += ROW_THREADS) sh.histR[i] = 0u;
        __syncthreads();
        if (compact) {
            for (int j = tid; j < m; j += ROW_THREADS) {
                const uint32_t key = sh.cand_key[j];
                if ((key & mask) == prefix) atomicAdd(&sh.histR[(key >> shift) & dmask], 1u);
            }
            __syncthreads();
        } else {
            stream_row(g, n, head, nvec, tid, [&](int, uint32_t bits) {
                const uint32_t key = float_bits_to_key(bits);
                if ((key & mask) == prefix) atomicAdd(&sh.histR[(key >> shift) & dmask], 1u);
            });
        }
        select_desc(tid < BINS_R ? sh.histR[BINS_R - 1 - tid] : 0u, kk, sh, tid, lane, warp);
        kk -= sh.sel_excl;
        prefix |= sh.sel_bin << shift;
        mask |= dmask << shift;
        done = sh.sel_cnt == kk;
    }

    // Marking: keys of the leading bin above the final prefix are selected;
    // keys equal to it are ties.
    if (!doneA) {
        if (compact) {
            for (int j = tid; j < m; j += ROW_THREADS) {
                const uint32_t km = sh.cand_key[j] & mask;
                const uint32_t i = sh.cand_idx[j];
                if (km > prefix) {
                    atomicOr(&selbits[i >> 5], 1u << (i & 31u));
                } else if (km == prefix) {
                    atomicOr(&tiebits[i >> 5], 1u << (i & 31u));
                    atomicAdd(&sh.n_tie, 1u);
                }
            }
            __syncthreads();
        } else {
            stream_row(g, n, head, nvec, tid, [&](int i, uint32_t bits) {
                const uint32_t key = float_bits_to_key(bits);
                if ((key >> 21) != T1) return;
                const uint32_t km = key & mask;
                if (km > prefix) {
                    atomicOr(&selbits[i >> 5], 1u << (i & 31));
                } else if (km == prefix) {
                    atomicOr(&tiebits[i >> 5], 1u << (i & 31));
                    atomicAdd(&sh.n_tie, 1u);
                }
            });
        }
    }

    // Each thread owns a contiguous run of bitmap words, so ids stay ordered.
    const int wpt = (nwords + ROW_THREADS - 1) / ROW_THREADS;
    const int wb = min(nwords, tid * wpt), we = min(nwords, wb + wpt);
    const uint32_t take = doneA ? 0u : min(kk, sh.n_tie);
    if (take > 0u) {  // uniform in the CTA
        uint32_t c = 0u;
        for (int wd = wb; wd < we; ++wd) c += __popc(tiebits[wd]);
        uint32_t run = block_excl_scan(c, sh.scan_tot, lane, warp);
        for (int wd = wb; wd < we && run < take; ++wd) {
            uint32_t bits = tiebits[wd], add = 0u;
            while (bits != 0u && run < take) {
                add |= bits & (~bits + 1u);
                bits &= bits - 1u;
                ++run;
            }
            selbits[wd] |= add;
        }
        __syncthreads();
    }
    {
        uint32_t c = 0u;
        for (int wd = wb; wd < we; ++wd) c += __popc(selbits[wd]);
        uint32_t pos = block_excl_scan(c, sh.scan_tot, lane, warp);
        int32_t *out = ids + row * static_cast<size_t>(k);
        for (int wd = wb; wd < we; ++wd) {
            uint32_t bits = selbits[wd];
            while (bits != 0u) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (pos < static_cast<uint32_t>(k)) out[pos] = wd * 32 + b;  // always, for consistent counts
                ++pos;
            }
        }
    }
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
    if (active > MAX_ACTIVE) return cudaErrorInvalidValue;
    static_assert(ROW_THREADS >= NGROUPS && ROW_THREADS >= BINS_R, "one scan item per thread");
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(row_smem_bytes(MAX_ACTIVE)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    topk_row_kernel<<<static_cast<unsigned>(nq), ROW_THREADS, row_smem_bytes(active), stream>>>(scores, active,
                                                                                               k, ids);
    return cudaGetLastError();
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

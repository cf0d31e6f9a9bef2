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
//  3. Keys above the final prefix are selected. A bin taken whole is selected
//     with them; otherwise keys equal to the full 32-bit prefix are ties,
//     taken in ascending id order until k ids are selected (ties go to the
//     lower block id). Ids leave in ascending order.
//
// GB300 layout. One 512-thread CTA owns one row (two CTAs per SM, so every row
// of a 256-query call is in flight at once):
//  With the scorer's group maxima (the key of each 32-block group's largest
//  score), a threshold that at least k groups reach is at most the k-th
//  score, so every score of the top k lies in a group at or above it: the row
//  lists only those groups (about k of them, one 128-byte line each) and the
//  digits below run on that list.
//  Without them, rows of at least 8,192 scores first try a listing path. A strided 1/32
//  sample of the row fixes a threshold expected to pass about 1.8k scores;
//  one pass of 16-byte L2-only loads then lists every score at or above
//  the threshold, and the digits below run on that list alone. A list shorter than k or longer
//  than its capacity sends the row to the exact passes, so the result is
//  exact either way.
//  Rows of at most 8,192 scores are read once into registers (up to 16 per
//  thread) and the whole digit search runs on them (topk_reg_row).
//  Exact passes: pass A reads the row and builds the 11-bit histogram in
//  shared memory; pass B streams the row again -- from L2, where pass A just
//  left it -- and marks keys above the leading bin in a shared-memory
//  selection bitmap while listing the keys inside it as candidates. The later
//  digits visit only that candidate list (if it would overflow its capacity,
//  they re-stream the row and filter by prefix instead).
//  Each digit's histogram is built by all warps with shared-memory atomics and
//  scanned by warp 0 alone (two block barriers per digit).
// In topk_row_kernel no CTA ever waits on another: no cluster, no grid-wide
// synchronisation, no global scratch. The fused decode select at the end of
// this file is the exception: a cooperative launch whose CTAs meet at a
// bounded grid-wide barrier, with its group maxima and arrival counters in
// fixed device arrays (so its calls must be ordered on a device).
#include "decode_rows.cuh"
#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int ROW_THREADS = 512;
constexpr int ROW_WARPS = ROW_THREADS / 32;
constexpr int HIST_A = 2048;             // leading digit: bits 31..21
constexpr int GROUP = 8;                 // leading-digit bins per group sum
constexpr int BINS_R = 256;              // refinement digits: 20..13, 12..5, 4..0
constexpr int UNROLL = 4;                // 16-byte loads in flight per thread (exact passes)
constexpr int LIST_VEC = 8;              // 16-byte loads per thread per listing step: 32 scores
constexpr int CAND_MAX = 4096;           // candidate-list capacity
constexpr int SAMPLE_STRIDE = 32;        // one 16-byte group of scores sampled per 512 bytes
constexpr int SAMPLE_SHIFT = 18;         // sample bins: 2^18 keys = 1/32 octave; 256 bins span 8
constexpr int GMAX_SHIFT = 15;           // group-maximum bins: 2^15 keys = 1/256 octave; 2,048 bins span 8
constexpr int FAST_MIN_ACTIVE = 8192;    // shorter rows take the exact passes directly
constexpr int MAX_ACTIVE = 393216;
constexpr int SAMPLE_REGS = (MAX_ACTIVE / 4 / SAMPLE_STRIDE + ROW_THREADS - 1) / ROW_THREADS;
constexpr uint32_t NEG_INF_KEY = 0x007FFFFFu;  // key of -inf (and of NaN)
constexpr uint32_t QNAN_BITS = 0x7FC00000u;

__device__ uint32_t g_topk_error;

struct RowShared {
    uint32_t histA[HIST_A];
    uint32_t groupA[HIST_A / GROUP];
    uint32_t histR[BINS_R];
    uint32_t cand_key[CAND_MAX];
    uint32_t cand_idx[CAND_MAX];
    alignas(16) uint32_t scan_tot[ROW_WARPS];
    uint32_t sel_bin, sel_above, sel_cnt;
    uint32_t cand_n;
    uint32_t glist_n;  // groups listed from the group maxima (their ids in histA)
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

// Score and group-maximum loads. The top-k kernels read data that the
// previous grid on the stream wrote, cached in L2 only (ld_in: the grid may
// have started before that grid finished); the fused decode kernel reads
// scores its own grid wrote before a grid-wide release, through coherent
// GPU-scope loads (kCoherent true).
template <bool kCoherent>
__device__ __forceinline__ uint32_t ld_word(const uint32_t *p) {
    if constexpr (kCoherent) {
        uint32_t v;
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        return v;
    } else {
        return ld_in(p);
    }
}
template <bool kCoherent>
__device__ __forceinline__ uint4 ld_quad(const uint4 *p) {
    if constexpr (kCoherent) {
        uint4 v;
        asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p)
                     : "memory");
        return v;
    } else {
        return ld_in(p);
    }
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL_MASK, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Block-wide exclusive prefix sum over threads (every thread must call).
// With trailing_sync false the warp totals are left as they are for good (the
// caller's last use of tot before the CTA ends).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *tot, int lane, int warp,
                                                    bool trailing_sync = true) {
    static_assert(ROW_WARPS == 16, "warp totals are read as four 16-byte words");
    const uint32_t incl = warp_incl_scan(v, lane);
    if (lane == 31) tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0u;
#pragma unroll
    for (int q = 0; q < ROW_WARPS / 4; ++q) {
        const uint4 t = *reinterpret_cast<const uint4 *>(tot + 4 * q);
        before += (4 * q + 0 < warp ? t.x : 0u) + (4 * q + 1 < warp ? t.y : 0u) + (4 * q + 2 < warp ? t.z : 0u) +
                  (4 * q + 3 < warp ? t.w : 0u);
    }
    if (trailing_sync) __syncthreads();
    return before + incl - v;
}

// Warp 0 alone. Walking the 256 bins of `hist` from the top, finds the bin
// where the running count reaches `target` (1 <= target <= total); every lane
// receives the bin, the count above it and its own count. Lane l owns bins
// 255 - 8l down to 248 - 8l. Clears the histogram when `clear` is set.
__device__ __forceinline__ void warp_find_256(uint32_t *hist, uint32_t target, bool clear, int lane,
                                              uint32_t &bin, uint32_t &above, uint32_t &cnt) {
    uint4 *p = reinterpret_cast<uint4 *>(hist + 8 * (31 - lane));
    const uint4 lo = p[0], hi = p[1];
    const uint32_t c[8] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};
    uint32_t s = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += c[i];
    const uint32_t incl = warp_incl_scan(s, lane);
    const uint32_t owner = __ballot_sync(FULL_MASK, incl - s < target && incl >= target);
    const int src = owner != 0u ? __ffs(owner) - 1 : 0;
    uint32_t b = 0u, a = 0u, n = 0u;
    if (lane == src) {
        uint32_t run = incl - s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (run < target && run + c[i] >= target) {
                b = static_cast<uint32_t>(255 - 8 * lane - i);
                a = run;
                n = c[i];
            }
            run += c[i];
        }
    }
    bin = __shfl_sync(FULL_MASK, b, src);
    above = __shfl_sync(FULL_MASK, a, src);
    cnt = __shfl_sync(FULL_MASK, n, src);
    if (clear) {
        p[0] = make_uint4(0u, 0u, 0u, 0u);
        p[1] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Warp 0 alone: the digit of a 256-bin histogram, left in sh.sel_*; clears it.
__device__ __forceinline__ void warp_select_256(uint32_t *hist, uint32_t target, RowShared &sh, int lane) {
    uint32_t bin, above, cnt;
    warp_find_256(hist, target, true, lane, bin, above, cnt);
    if (lane == 0) {
        sh.sel_bin = bin;
        sh.sel_above = above;
        sh.sel_cnt = cnt;
    }
}

// Warp 0 alone: the leading digit, from the 256 group sums (8 bins each) in
// sh.groupA and then the 8 bins of the group found; left in sh.sel_*.
__device__ __forceinline__ void warp_select_2048(uint32_t target, RowShared &sh, int lane) {
    uint32_t gb, ga, gc;
    warp_find_256(sh.groupA, target, false, lane, gb, ga, gc);
    const uint32_t c = lane < GROUP ? sh.histA[GROUP * gb + (GROUP - 1) - lane] : 0u;
    const uint32_t incl = ga + warp_incl_scan(c, lane);
    const uint32_t owner = __ballot_sync(FULL_MASK, lane < GROUP && incl - c < target && incl >= target);
    if (owner != 0u && lane == __ffs(owner) - 1) {
        sh.sel_bin = GROUP * gb + (GROUP - 1) - static_cast<uint32_t>(lane);
        sh.sel_above = incl - c;
        sh.sel_cnt = c;
    }
}

// Calls fn(i, bits) once for every element of the row (row index i, raw
// fp32 bits), each from some thread; every thread must call it. The aligned
// body moves as 16-byte L2-only loads, UNROLL in flight per thread; the
// <= 3 ragged scores at either end as single words.
template <bool kCoherent, typename Fn>
__device__ __forceinline__ void stream_row(const uint32_t *g, int n, int head, int nvec, int tid, Fn &&fn) {
    for (int i = tid; i < head; i += ROW_THREADS) fn(i, ld_word<kCoherent>(g + i));
    for (int i = head + 4 * nvec + tid; i < n; i += ROW_THREADS) fn(i, ld_word<kCoherent>(g + i));
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g + head);
#pragma unroll 1
    for (int v0 = 0; v0 < nvec; v0 += ROW_THREADS * UNROLL) {
        uint4 x[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int v = v0 + u * ROW_THREADS + tid;
            x[u] = v < nvec ? ld_quad<kCoherent>(g4 + v) : make_uint4(0u, 0u, 0u, 0u);
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

// The end of one row's selection, shared by every path: selbits marks the
// selected ids; when `ties` is set, the first kk ids marked in tiebits (in id
// order) join them. Writes the row's k ids in ascending order to out. It is
// the CTA's last step (one row per CTA), so its final block scan leaves the
// warp totals without a closing barrier.
__device__ __forceinline__ void finish_row(uint32_t *selbits, const uint32_t *tiebits, int nwords, bool ties,
                                           uint32_t kk, int k, int32_t *__restrict__ out, RowShared &sh, int tid,
                                           int lane, int warp) {
    // Each thread owns a contiguous run of bitmap words, so ids stay ordered.
    const int wpt = (nwords + ROW_THREADS - 1) / ROW_THREADS;
    const int wb = min(nwords, tid * wpt), we = min(nwords, wb + wpt);
    if (ties) {  // uniform: the first kk ties in id order join the selection
        uint32_t c = 0u;
        for (int wd = wb; wd < we; ++wd) c += __popc(tiebits[wd]);
        uint32_t run = block_excl_scan(c, sh.scan_tot, lane, warp);
        for (int wd = wb; wd < we && run < kk; ++wd) {
            uint32_t bits = tiebits[wd], add = 0u;
            while (bits != 0u && run < kk) {
                add |= bits & (~bits + 1u);
                bits &= bits - 1u;
                ++run;
            }
            selbits[wd] |= add;
        }
        __syncthreads();
    }
    if (wpt == 4) {
        // Up to 65,536 scores (nwords <= 2,048): a thread's four words as one
        // conflict-free 16-byte load, kept in registers for both passes.
        uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
        if (wb < nwords) w4 = *reinterpret_cast<const uint4 *>(selbits + wb);
        // Words past nwords (the last thread, when nwords % 4 != 0) belong to
        // the tie bitmap that follows: drop them.
        const uint32_t wv[4] = {w4.x, wb + 1 < nwords ? w4.y : 0u, wb + 2 < nwords ? w4.z : 0u,
                                wb + 3 < nwords ? w4.w : 0u};
        uint32_t pos = block_excl_scan(__popc(wv[0]) + __popc(wv[1]) + __popc(wv[2]) + __popc(wv[3]), sh.scan_tot,
                                       lane, warp, false);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t bits = wv[e];
            while (bits != 0u) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (pos < static_cast<uint32_t>(k)) out[pos] = (wb + e) * 32 + b;  // always, for consistent counts
                ++pos;
            }
        }
    } else {
        uint32_t c = 0u;
        for (int wd = wb; wd < we; ++wd) c += __popc(selbits[wd]);
        uint32_t pos = block_excl_scan(c, sh.scan_tot, lane, warp, false);
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

// One row's exact top-k by one 512-thread CTA (the whole of topk_row_kernel;
// also the second phase of the fused decode kernel). Dynamic shared memory:
// row_smem_bytes(active).
template <bool kCoherent>
__device__ __forceinline__ void topk_row(const float *__restrict__ scores, const uint32_t *__restrict__ gmax,
                                         int active, int k, int32_t *__restrict__ ids, size_t row) {
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
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g + head);

    // Listing path (rows of at least FAST_MIN_ACTIVE scores). A strided sample
    // (one 16-byte group of scores per 512 bytes) gives a threshold that about
    // 1.8k + 8 n / samples scores of the row are expected to reach: the
    // sample's r-th largest key with r = ceil(1.8 k * samples / n) + 8, found to
    // 1/32 of an octave. The sample keys above the true k-th key number
    // Binomial(samples, k / n) (mean 16 at k = 512 of 65,536), so a list
    // shorter than k needs that count to reach r (37 there): about 5 standard
    // deviations. One pass then lists every score at or above it. A list of
    // at least k entries holds the whole top-k, ties included, so when it also
    // fits its capacity the exact selection runs on the list alone; otherwise
    // the row takes the exact two-pass path.
    const int nsv = nvec / SAMPLE_STRIDE;
    const uint32_t nsamp = 4u * static_cast<uint32_t>(nsv);
    const uint32_t r_target =
        static_cast<uint32_t>((9ull * static_cast<uint64_t>(k) * nsamp + 5ull * n - 1) / (5ull * n)) + 8u;
    // Group-maximum mode: with the maxima of the row's 32-block groups, the
    // threshold comes from them instead of a sample, and the listing reads
    // only the groups whose maximum reaches it (rows of at most 2,048 groups,
    // k at most half of them).
    const int ngr = (n + GROUP_BLOCKS - 1) / GROUP_BLOCKS;
    const bool use_gmax = gmax != nullptr && 2 * k <= ngr && ngr <= 4 * ROW_THREADS;
    const bool try_list = use_gmax || (n >= FAST_MIN_ACTIVE && r_target <= nsamp / 2);

    // Shared memory is cleared before the wait below (it does not depend on
    // the previous grid).
    if (tid == 0) {
        sh.cand_n = 0u;
        sh.glist_n = 0u;
    }
    if (!try_list || use_gmax) {   // the exact path's histogram, or the group-maximum bins
        static_assert(HIST_A == 4 * ROW_THREADS, "one 16-byte store per thread clears histA");
        reinterpret_cast<uint4 *>(sh.histA)[tid] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (use_gmax && tid < HIST_A / GROUP) sh.groupA[tid] = 0u;   // counted with histA below
    for (int i = tid; i < BINS_R; i += ROW_THREADS) sh.histR[i] = 0u;
    for (int i = tid; i < nwords; i += ROW_THREADS) {
        selbits[i] = 0u;
        tiebits[i] = 0u;
    }

    // The scores may come from the previous grid on the stream (launched as
    // its programmatic dependent); nothing global is read before this.
    grid_dependency_wait();

    // The sample (or this thread's 4 group maxima) is requested before anything else.
    uint4 sx[SAMPLE_REGS];
    if (use_gmax) {
        const uint32_t *gm = gmax + row * static_cast<size_t>(ngr);
        sx[0] = make_uint4(0u, 0u, 0u, 0u);
        if ((ngr & 3) == 0) {
            if (4 * tid < ngr) sx[0] = ld_quad<kCoherent>(reinterpret_cast<const uint4 *>(gm) + tid);
        } else {
            if (4 * tid + 0 < ngr) sx[0].x = ld_word<kCoherent>(gm + 4 * tid + 0);
            if (4 * tid + 1 < ngr) sx[0].y = ld_word<kCoherent>(gm + 4 * tid + 1);
            if (4 * tid + 2 < ngr) sx[0].z = ld_word<kCoherent>(gm + 4 * tid + 2);
            if (4 * tid + 3 < ngr) sx[0].w = ld_word<kCoherent>(gm + 4 * tid + 3);
        }
#pragma unroll
        for (int u = 1; u < SAMPLE_REGS; ++u) sx[u] = make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
        for (int u = 0; u < SAMPLE_REGS; ++u) {
            const int s = tid + u * ROW_THREADS;
            sx[u] = try_list && s < nsv ? ld_quad<kCoherent>(g4 + s * SAMPLE_STRIDE + SAMPLE_STRIDE / 2)
                                        : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    if (use_gmax) {   // the group maxima's warp maxima ride on the same barrier
        uint32_t m = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (4 * tid + e < ngr) m = max(m, (&sx[0].x)[e]);
        m = __reduce_max_sync(FULL_MASK, m);
        if (lane == 0) sh.scan_tot[warp] = m;
        if (tid == 0) sh.sel_cnt = 0u;   // stays 0 when no threshold bin is found
    }
    __syncthreads();

    uint32_t kk = static_cast<uint32_t>(k);
    bool listed = false;
    bool first_hist = false;   // the first refinement digit was counted while gathering the list
    uint32_t tg = 0u, kmax = 0u;
    if (try_list) {
        const uint32_t gk[4] = {sx[0].x, sx[0].y, sx[0].z, sx[0].w};   // group-maximum mode's keys
        if (use_gmax) {
            // Group-maximum threshold: the group maxima are counted by their
            // distance below the largest, smax, in 2,048 bins of 2^15 keys
            // (1/256 of an octave for normal floats) spanning 8 octaves. tg is
            // the lowest key of the bin where the count of groups from the top
            // reaches k: at least k groups, hence at least k scores, are >= tg,
            // and few groups beyond k are. A k-th group maximum below the
            // window leaves tg = 0: the exact path.
            uint32_t smax = 0u;
#pragma unroll
            for (int q = 0; q < ROW_WARPS / 4; ++q) {
                const uint4 t = *reinterpret_cast<const uint4 *>(sh.scan_tot + 4 * q);
                smax = max(max(smax, t.x), max(t.y, max(t.z, t.w)));
            }
            kmax = smax;   // the row maximum: every listed key lies in [tg, smax]
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t d = smax - gk[e];
                if (4 * tid + e < ngr && d < (static_cast<uint32_t>(HIST_A) << GMAX_SHIFT)) {
                    const uint32_t bin = HIST_A - 1 - (d >> GMAX_SHIFT);
                    atomicAdd(&sh.histA[bin], 1u);
                    atomicAdd(&sh.groupA[bin / GROUP], 1u);   // the group sums, without a pass of their own
                }
            }
            __syncthreads();
            if (warp == 0) warp_select_2048(kk, sh, lane);
            __syncthreads();
            const uint32_t below = (static_cast<uint32_t>(HIST_A) - sh.sel_bin) << GMAX_SHIFT;   // (b + 1) bins
            tg = sh.sel_cnt != 0u && smax >= below ? smax - below + 1u : 0u;
        } else {
            // Sample threshold. The largest sample key smax tops a window of 256
            // bins, each 2^18 keys wide (1/32 of an octave for normal floats),
            // reaching 8 octaves below it. Counting the sample keys by their
            // distance below smax spreads them over the bins (bins of fixed key
            // digits crowd them into a few, which serialises the shared-memory
            // atomics). tg is the lowest key of the bin where the count from the
            // top reaches r, so at least r sample keys are >= tg. A sample whose
            // r-th key lies below the window leaves tg = 0: the exact path.
            uint32_t ks[SAMPLE_REGS][4];
            uint32_t m = 0u;
#pragma unroll
            for (int u = 0; u < SAMPLE_REGS; ++u) {
                ks[u][0] = float_bits_to_key(sx[u].x);
                ks[u][1] = float_bits_to_key(sx[u].y);
                ks[u][2] = float_bits_to_key(sx[u].z);
                ks[u][3] = float_bits_to_key(sx[u].w);
                if (tid + u * ROW_THREADS < nsv) m = max(m, max(max(ks[u][0], ks[u][1]), max(ks[u][2], ks[u][3])));
            }
            m = __reduce_max_sync(FULL_MASK, m);
            if (lane == 0) sh.scan_tot[warp] = m;
            __syncthreads();
            uint32_t smax = 0u;
#pragma unroll
            for (int q = 0; q < ROW_WARPS / 4; ++q) {
                const uint4 t = *reinterpret_cast<const uint4 *>(sh.scan_tot + 4 * q);
                smax = max(max(smax, t.x), max(t.y, max(t.z, t.w)));
            }
#pragma unroll
            for (int u = 0; u < SAMPLE_REGS; ++u) {
                if (tid + u * ROW_THREADS < nsv) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t d = smax - ks[u][e];
                        if (d < (static_cast<uint32_t>(BINS_R) << SAMPLE_SHIFT))
                            atomicAdd(&sh.histR[BINS_R - 1 - (d >> SAMPLE_SHIFT)], 1u);
                    }
                }
            }
            __syncthreads();
            // A target past the window's count finds no bin (count 0).
            if (warp == 0) warp_select_256(sh.histR, r_target, sh, lane);
            __syncthreads();
            const uint32_t below = (static_cast<uint32_t>(BINS_R) - sh.sel_bin) << SAMPLE_SHIFT;  // (b + 1) bins
            tg = sh.sel_cnt != 0u && smax >= below ? smax - below + 1u : 0u;
        }

        // Listing pass. key(x) >= tg is tested as the fp32 comparison x >= ft,
        // ft being the value whose key is tg: both orders agree on every x (NaN
        // fails the comparison and has the key of -inf, which is below any tg
        // past the -inf key). A tg at or below the -inf key would list the
        // whole row, so such a row takes the exact path at once. Each thread
        // gathers one hit bit per score of a 32-score step; a warp scan of the
        // hit counts and one shared-memory atomic per warp and step give every
        // hit its list slot, which records the score's index; the score itself
        // is copied into the slot by an asynchronous 4-byte copy (re-reading it
        // into a register, or gathering the listed scores after the pass,
        // each stalled on an L2 round trip).
        if (tg > NEG_INF_KEY) {
            const float ft = __uint_as_float(tg >= 0x80000000u ? (tg ^ 0x80000000u) : ~tg);
            // Slots for one 32-score step's hits: bit j of `hits` is the score
            // at index idx(j); the slot records the index, and the listed
            // scores are gathered after the pass (the registers that held
            // them are reused by then).
            auto book = [&](uint32_t hits, auto idx) {
                const uint32_t c = __popc(hits);
                const uint32_t incl = warp_incl_scan(c, lane);
                const uint32_t total = __shfl_sync(FULL_MASK, incl, 31);
                if (total != 0u) {  // warp-uniform
                    uint32_t base = 0u;
                    if (lane == 31) base = atomicAdd(&sh.cand_n, total);
                    uint32_t slot = __shfl_sync(FULL_MASK, base, 31) + incl - c;
                    while (hits != 0u) {
                        const int j = __ffs(hits) - 1;
                        hits &= hits - 1u;
                        if (slot < static_cast<uint32_t>(CAND_MAX)) sh.cand_idx[slot] = static_cast<uint32_t>(idx(j));
                        ++slot;
                    }
                }
            };
            auto hit_bits = [&](const uint4 &y, int u) {
                return static_cast<uint32_t>(__uint_as_float(y.x) >= ft) << (4 * u) |
                       static_cast<uint32_t>(__uint_as_float(y.y) >= ft) << (4 * u + 1) |
                       static_cast<uint32_t>(__uint_as_float(y.z) >= ft) << (4 * u + 2) |
                       static_cast<uint32_t>(__uint_as_float(y.w) >= ft) << (4 * u + 3);
            };
            if (use_gmax) {
                // The groups whose maximum reaches tg (every score >= tg lies in
                // one) are compacted into histA, then each thread lists one
                // group (32 scores, one 128-byte line) per round.
                uint32_t mine = 0u;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * tid + e < ngr && gk[e] >= tg) mine |= 1u << e;
                {
                    const uint32_t c = __popc(mine);
                    const uint32_t incl = warp_incl_scan(c, lane);
                    const uint32_t total = __shfl_sync(FULL_MASK, incl, 31);
                    uint32_t base = 0u;
                    if (lane == 31 && total != 0u) base = atomicAdd(&sh.glist_n, total);
                    uint32_t slot = __shfl_sync(FULL_MASK, base, 31) + incl - c;
                    while (mine != 0u) {   // slot < ngr <= HIST_A
                        const int e = __ffs(mine) - 1;
                        mine &= mine - 1u;
                        sh.histA[slot++] = static_cast<uint32_t>(4 * tid + e);
                    }
                }
                __syncthreads();
                // A warp lists 4 groups per load instruction: lane l reads the
                // 16-byte piece l % 8 of group l / 8, so each instruction
                // touches 4 whole 128-byte lines; GU instructions per round.
                constexpr int GU = 8;
                const int ngl = static_cast<int>(sh.glist_n);
                const bool vec = (n & 3) == 0;   // every group starts 16-byte aligned
                const int piece = lane & 7;
#pragma unroll 1
                for (int r0 = 4 * GU * warp; r0 < ngl; r0 += 4 * GU * ROW_WARPS) {   // warp-uniform
                    int base[GU];                  // index of this lane's first score in each group
                    uint32_t hits = 0u;
#pragma unroll
                    for (int u = 0; u < GU; ++u) {
                        const int j = r0 + 4 * u + (lane >> 3);
                        base[u] = j < ngl ? static_cast<int>(sh.histA[j]) * GROUP_BLOCKS + 4 * piece : n;
                    }
                    if (vec) {
                        uint4 y[GU];
#pragma unroll
                        for (int u = 0; u < GU; ++u)
                            y[u] = base[u] + 4 <= n ? ld_quad<kCoherent>(reinterpret_cast<const uint4 *>(g + base[u]))
                                                    : make_uint4(QNAN_BITS, QNAN_BITS, QNAN_BITS, QNAN_BITS);
#pragma unroll
                        for (int u = 0; u < GU; ++u) hits |= hit_bits(y[u], u);
                    } else {
#pragma unroll
                        for (int u = 0; u < GU; ++u) {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (base[u] + c < n && __uint_as_float(ld_word<kCoherent>(g + base[u] + c)) >= ft)
                                    hits |= 1u << (4 * u + c);
                        }
                    }
                    // A hit's group is read again from the list (hits are few).
                    book(hits, [&](int jj) {
                        return static_cast<int>(sh.histA[r0 + 4 * (jj >> 2) + (lane >> 3)]) * GROUP_BLOCKS +
                               4 * piece + (jj & 3);
                    });
                }
            } else {
                auto list_scalar = [&](int i) {
                    if (__uint_as_float(ld_word<kCoherent>(g + i)) >= ft) {
                        const uint32_t slot = atomicAdd(&sh.cand_n, 1u);
                        if (slot < static_cast<uint32_t>(CAND_MAX)) sh.cand_idx[slot] = static_cast<uint32_t>(i);
                    }
                };
                for (int i = tid; i < head; i += ROW_THREADS) list_scalar(i);
                for (int i = head + 4 * nvec + tid; i < n; i += ROW_THREADS) list_scalar(i);
                // The next step's loads are issued as soon as this step's hit bits
                // are taken, ahead of the slot bookkeeping.
                uint4 x[LIST_VEC];
                auto load_step = [&](int v0) {
#pragma unroll
                    for (int u = 0; u < LIST_VEC; ++u) {
                        const int v = v0 + u * ROW_THREADS + tid;
                        // Past the end: NaN, which no comparison lists.
                        x[u] = v < nvec ? ld_quad<kCoherent>(g4 + v)
                                        : make_uint4(QNAN_BITS, QNAN_BITS, QNAN_BITS, QNAN_BITS);
                    }
                };
                load_step(0);
#pragma unroll 1
                for (int v0 = 0; v0 < nvec; v0 += ROW_THREADS * LIST_VEC) {
                    // A list already past its capacity is abandoned (warp-uniform test).
                    if (__shfl_sync(FULL_MASK, *reinterpret_cast<volatile uint32_t *>(&sh.cand_n), 0) >
                        static_cast<uint32_t>(CAND_MAX))
                        break;
                    uint32_t hits = 0u;
#pragma unroll
                    for (int u = 0; u < LIST_VEC; ++u) hits |= hit_bits(x[u], u);
                    if (v0 + ROW_THREADS * LIST_VEC < nvec) load_step(v0 + ROW_THREADS * LIST_VEC);
                    const int i0 = head + 4 * (v0 + tid);
                    book(hits, [&](int jj) { return i0 + 4 * ROW_THREADS * (jj >> 2) + (jj & 3); });
                }
            }
        } else if (tid == 0) {
            sh.cand_n = static_cast<uint32_t>(CAND_MAX) + 1u;  // would list the whole row
        }
        __syncthreads();
        const uint32_t nc = sh.cand_n;
        listed = nc >= kk && nc <= static_cast<uint32_t>(CAND_MAX);
        if (listed && use_gmax) {
            // The listed scores are gathered (one L2 round trip for the whole
            // list) as keys (their maximum, the row's, is known from the group
            // maxima). Every listed key lies in [tg, kmax], so all of them
            // match the digit search's starting prefix and the first
            // refinement digit's histogram is counted in the same loop (when
            // that search will run).
            const uint32_t diff = tg ^ kmax;
            const int s0 = diff == 0u ? 0 : 32 - __clz(static_cast<int>(diff));
            const int w0 = min(8, s0);
            const uint32_t dm0 = (1u << w0) - 1u;
            first_hist = s0 > 0 && nc != kk;
#pragma unroll 4
            for (int j = tid; j < static_cast<int>(nc); j += ROW_THREADS) {
                const uint32_t key = float_bits_to_key(ld_word<kCoherent>(g + sh.cand_idx[j]));
                sh.cand_key[j] = key;
                if (first_hist) atomicAdd(&sh.histR[(key >> (s0 - w0)) & dm0], 1u);
            }
            __syncthreads();
        } else if (listed) {
            // The listed scores are gathered as keys; the largest is kept.
#pragma unroll 4
            for (int j = tid; j < static_cast<int>(nc); j += ROW_THREADS) {
                const uint32_t key = float_bits_to_key(ld_word<kCoherent>(g + sh.cand_idx[j]));
                sh.cand_key[j] = key;
                kmax = max(kmax, key);
            }
            kmax = __reduce_max_sync(FULL_MASK, kmax);
            if (lane == 0) sh.scan_tot[warp] = kmax;
            __syncthreads();
#pragma unroll
            for (int q = 0; q < ROW_WARPS / 4; ++q) {
                const uint4 t = *reinterpret_cast<const uint4 *>(sh.scan_tot + 4 * q);
                kmax = max(max(kmax, t.x), max(t.y, max(t.z, t.w)));
            }
        } else {  // uniform: the list is abandoned; the exact path follows
            __syncthreads();
            if (tid == 0) sh.cand_n = 0u;
            for (int i = tid; i < HIST_A; i += ROW_THREADS) sh.histA[i] = 0u;
            __syncthreads();
        }
    }

    // Digit search. On the list, every key lies in [tg, kmax], so the search
    // starts below the bits those two share. On the exact path, the leading
    // 11 bits come from pass A over the whole row.
    uint32_t prefix, mask, T1 = 0u;
    int shift;
    bool done, doneA = false, compact = true;
    if (listed) {
        const uint32_t diff = tg ^ kmax;
        shift = diff == 0u ? 0 : 32 - __clz(static_cast<int>(diff));
        mask = shift == 32 ? 0u : 0xFFFFFFFFu << shift;
        prefix = tg & mask;
        done = sh.cand_n == kk;  // the whole list is the top-k
    } else {
        // Pass A: the 11-bit leading-digit histogram of the whole row.
        stream_row<kCoherent>(g, n, head, nvec, tid, [&](int, uint32_t bits) {
            atomicAdd(&sh.histA[float_bits_to_key(bits) >> 21], 1u);
        });
        if (tid < HIST_A / GROUP) {
            const uint4 a = *reinterpret_cast<const uint4 *>(&sh.histA[GROUP * tid]);
            const uint4 b = *reinterpret_cast<const uint4 *>(&sh.histA[GROUP * tid + 4]);
            sh.groupA[tid] = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
        }
        __syncthreads();
        if (warp == 0) warp_select_2048(kk, sh, lane);
        __syncthreads();
        T1 = sh.sel_bin;
        const uint32_t t1_cnt = sh.sel_cnt;
        kk -= sh.sel_above;
        // A leading bin taken whole is marked by pass B directly.
        doneA = t1_cnt == kk;
        done = doneA;
        compact = !doneA && t1_cnt <= static_cast<uint32_t>(CAND_MAX);
        prefix = T1 << 21;
        mask = 0xFFE00000u;
        shift = 21;

        // Pass B: keys above the leading bin are selected; keys inside it are
        // listed as candidates (or all selected, when the bin is taken whole).
        stream_row<kCoherent>(g, n, head, nvec, tid, [&](int i, uint32_t bits) {
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
    }

    // Refinement digits (at most 8 bits each) over the candidates; histR is
    // clear here.
    const int m = min(static_cast<int>(sh.cand_n), CAND_MAX);
#pragma unroll 1
    while (!done && shift > 0) {
        const int width = min(8, shift);
        shift -= width;
        const uint32_t dmask = (1u << width) - 1u;
        if (first_hist) {
            first_hist = false;   // this digit's histogram is complete already
        } else if (compact) {
            for (int j = tid; j < m; j += ROW_THREADS) {
                const uint32_t key = sh.cand_key[j];
                if ((key & mask) == prefix) atomicAdd(&sh.histR[(key >> shift) & dmask], 1u);
            }
            __syncthreads();
        } else {
            stream_row<kCoherent>(g, n, head, nvec, tid, [&](int, uint32_t bits) {
                const uint32_t key = float_bits_to_key(bits);
                if ((key & mask) == prefix) atomicAdd(&sh.histR[(key >> shift) & dmask], 1u);
            });
        }
        if (warp == 0) warp_select_256(sh.histR, kk, sh, lane);
        __syncthreads();
        kk -= sh.sel_above;
        prefix |= sh.sel_bin << shift;
        mask |= dmask << shift;
        done = sh.sel_cnt == kk;
    }

    // Marking. Keys above the final prefix are selected. When the search ended
    // on a bin taken whole (done), keys equal to the prefix are selected too;
    // otherwise they are ties of the full key, of which kk are taken below.
    if (!doneA) {
        if (compact) {
            for (int j = tid; j < m; j += ROW_THREADS) {
                const uint32_t km = sh.cand_key[j] & mask;
                const uint32_t i = sh.cand_idx[j];
                if (km > prefix || (done && km == prefix)) {
                    atomicOr(&selbits[i >> 5], 1u << (i & 31u));
                } else if (km == prefix) {
                    atomicOr(&tiebits[i >> 5], 1u << (i & 31u));
                }
            }
            __syncthreads();
        } else {
            stream_row<kCoherent>(g, n, head, nvec, tid, [&](int i, uint32_t bits) {
                const uint32_t key = float_bits_to_key(bits);
                if ((key >> 21) != T1) return;
                const uint32_t km = key & mask;
                if (km > prefix || (done && km == prefix)) {
                    atomicOr(&selbits[i >> 5], 1u << (i & 31));
                } else if (km == prefix) {
                    atomicOr(&tiebits[i >> 5], 1u << (i & 31));
                }
            });
        }
    }

    finish_row(selbits, tiebits, nwords, !doneA && !done, kk, k, ids + row * static_cast<size_t>(k), sh, tid,
               lane, warp);
}

// Register-resident exact top-k of a short row (n <= PER * 512 scores,
// k < n): every score is read once, into registers (thread t holds scores
// t, t + 512, ...), and the digit search runs on those registers: the 11-bit
// leading digit, then 8, 8 and 5 bits over the keys that match the prefix,
// each a shared-memory histogram scanned from the top (the same digits and
// tie rule as topk_row). The selection and tie bitmaps are built by warp
// ballots: with this layout one warp's 32 scores of step j are exactly one
// bitmap word.
// The digit search of a register-resident selection: key[j] for valid j
// (bit j of `valid`) are this thread's keys; every thread of the CTA calls it.
// Returns the final prefix and mask, the number kk still to take among keys
// equal to the prefix, and whether the search ended on a bin taken whole
// (done: every key matching the prefix is selected). histA and histR must be
// clear, and a CTA barrier must separate their clearing from the call.
struct DigitResult {
    uint32_t prefix, mask, kk;
    bool done;
};
template <int PER>
__device__ __forceinline__ DigitResult reg_digit_search(const uint32_t (&key)[PER], uint32_t valid, int k,
                                                        RowShared &sh, int tid, int lane, int warp) {
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (valid >> j & 1u) atomicAdd(&sh.histA[key[j] >> 21], 1u);
    __syncthreads();
    if (tid < HIST_A / GROUP) {
        const uint4 a = *reinterpret_cast<const uint4 *>(&sh.histA[GROUP * tid]);
        const uint4 b = *reinterpret_cast<const uint4 *>(&sh.histA[GROUP * tid + 4]);
        sh.groupA[tid] = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
    }
    __syncthreads();
    DigitResult r;
    r.kk = static_cast<uint32_t>(k);
    if (warp == 0) warp_select_2048(r.kk, sh, lane);
    __syncthreads();
    r.kk -= sh.sel_above;
    r.done = sh.sel_cnt == r.kk;
    r.prefix = sh.sel_bin << 21;
    r.mask = 0xFFE00000u;
    int shift = 21;
#pragma unroll 1
    while (!r.done && shift > 0) {
        const int width = min(8, shift);
        shift -= width;
        const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if ((valid >> j & 1u) && (key[j] & r.mask) == r.prefix) atomicAdd(&sh.histR[(key[j] >> shift) & dmask], 1u);
        __syncthreads();
        if (warp == 0) warp_select_256(sh.histR, r.kk, sh, lane);   // also clears histR
        __syncthreads();
        r.kk -= sh.sel_above;
        r.prefix |= sh.sel_bin << shift;
        r.mask |= dmask << shift;
        r.done = sh.sel_cnt == r.kk;
    }
    return r;
}

// Register-resident exact top-k of a short row (n <= PER * 512 scores,
// k < n): every score is read once, into registers (thread t holds scores
// t, t + 512, ...), and the digit search runs on those registers: the 11-bit
// leading digit, then 8, 8 and 5 bits over the keys that match the prefix,
// each a shared-memory histogram scanned from the top (the same digits and
// tie rule as topk_row). The selection and tie bitmaps are built by warp
// ballots: with this layout one warp's 32 scores of step j are exactly one
// bitmap word.
template <int PER, bool kCoherent>
__device__ __forceinline__ void topk_reg_row(const float *__restrict__ scores, int n, int k,
                                             int32_t *__restrict__ ids, size_t row) {
    static_assert(PER >= 1 && PER <= 32, "one validity bit per register");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwords = (n + 31) >> 5;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem_raw);
    uint32_t *selbits = reinterpret_cast<uint32_t *>(smem_raw + SHARED_BYTES);
    uint32_t *tiebits = selbits + nwords;
    const uint32_t *g = reinterpret_cast<const uint32_t *>(scores + row * static_cast<size_t>(n));

    static_assert(HIST_A == 4 * ROW_THREADS && BINS_R <= ROW_THREADS, "one clearing store per thread");
    reinterpret_cast<uint4 *>(sh.histA)[tid] = make_uint4(0u, 0u, 0u, 0u);   // before the wait: no global data
    if (tid < BINS_R) sh.histR[tid] = 0u;
    grid_dependency_wait();   // the scores may come from the previous grid
    uint32_t key[PER];
    uint32_t valid = 0u;      // bit j: score j * 512 + tid exists
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = j * ROW_THREADS + tid;
        key[j] = 0u;
        if (i < n) {
            key[j] = ld_word<kCoherent>(g + i);
            valid |= 1u << j;
        }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) key[j] = float_bits_to_key(key[j]);
    __syncthreads();
    const DigitResult r = reg_digit_search<PER>(key, valid, k, sh, tid, lane, warp);
    // Keys above the prefix are selected; keys equal to it are selected too
    // when the search ended on a bin taken whole, else they are ties.
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const uint32_t km = key[j] & r.mask;
        const bool ok = (valid >> j & 1u) != 0u;
        const uint32_t sel = __ballot_sync(FULL_MASK, ok && (km > r.prefix || (r.done && km == r.prefix)));
        const uint32_t tie = __ballot_sync(FULL_MASK, ok && !r.done && km == r.prefix);
        const int wd = j * ROW_WARPS + warp;
        if (lane == 0 && wd < nwords) {
            selbits[wd] = sel;
            tiebits[wd] = tie;
        }
    }
    __syncthreads();
    finish_row(selbits, tiebits, nwords, !r.done, r.kk, k, ids + row * static_cast<size_t>(k), sh, tid, lane, warp);
}

__global__ void __launch_bounds__(ROW_THREADS, 2)
    topk_row_kernel(const float *__restrict__ scores, const uint32_t *__restrict__ gmax, int active, int k,
                    int32_t *__restrict__ ids, const uint32_t *__restrict__ gate) {
    if (gate != nullptr) {   // the fused select's fallback: only rows whose list failed
        grid_dependency_wait();
        if (ld_in(gate + blockIdx.x) == 0u) return;
    }
    topk_row<false>(scores, gmax, active, k, ids, blockIdx.x);
}

// Rows of at most REG_MAX_ACTIVE scores take the register-resident path; PER
// is the smallest of 4, 8, 16 that holds the row. (At 16,384 scores, 32 per
// thread, the full-row histogram's shared-memory atomics crowd into a few
// exponent bins and the sampled listing path is faster.)
constexpr int REG_MAX_ACTIVE = 16 * ROW_THREADS;   // 8,192

template <int PER>
__global__ void __launch_bounds__(ROW_THREADS, 2)
    topk_reg_kernel(const float *__restrict__ scores, int active, int k, int32_t *__restrict__ ids,
                    const uint32_t *__restrict__ gate) {
    if (gate != nullptr) {
        grid_dependency_wait();
        if (ld_in(gate + blockIdx.x) == 0u) return;
    }
    topk_reg_row<PER, false>(scores, active, k, ids, blockIdx.x);
}

// Fused decode select (nq <= 4): one cooperative launch scores every key row
// (and the group maxima) across the whole grid, then its first nq CTAs each
// take one row's top-k. Each CTA releases its scores with an acquire-release
// atomic increment of an arrival counter, and the top-k CTAs wait (bounded; a
// cooperative launch keeps every CTA resident, so all of them arrive) until
// they read the full count with an acquire load. Two counters alternate by
// the parity of a generation word: each CTA reads the generation before it
// arrives, and only the last arrival advances it, so all of them use the
// same counter; the last arrival also clears the other counter, the one the
// next launch uses (this launch's counter keeps its count until then). The
// group maxima live in a fixed device array, so the call allocates nothing.
// Launches of this kernel on one device therefore run one at a time.
__device__ uint32_t g_decode_sync[3];   // arrivals (two, by generation parity), generation
static __device__ __align__(256) uint32_t g_decode_gmax[SMALL_NQ_MAX * (MAX_ACTIVE / GROUP_BLOCKS)];

template <int NQ, bool kInt8>
__global__ void __launch_bounds__(ROW_THREADS, 2)
    select_decode_kernel(const float *__restrict__ q, const float *__restrict__ kblk,
                         const int8_t *__restrict__ kq8, const __half *__restrict__ kscale, int nq, int active,
                         int k, float *__restrict__ scores, int32_t *__restrict__ ids, uint64_t wait_ns,
                         uint32_t inject) {
    constexpr int ROWS = ROW_THREADS / dec_tpr<kInt8>();
    __shared__ __align__(16) float qs[NQ][DEC_QROW];   // head-summed queries, zero past nq
    __shared__ uint32_t gk[NQ][ROWS];
    grid_dependency_wait();   // q and the keys may come from the previous grid
    grid_launch_dependents();
    uint32_t gen = 0u;
    if (threadIdx.x == 0) gen = ld_acquire_gpu(&g_decode_sync[2]);
    const long long nchunks = (static_cast<long long>(active) + ROWS - 1) / ROWS;
    DecKeys<kInt8> kv;
    long long c = blockIdx.x;
    if (c < nchunks) dec_load_keys<kInt8, ROW_THREADS>(c, kblk, kq8, active, kv);   // in flight during the build
    dec_build_queries<NQ, ROW_THREADS>(q, nq, qs);
    __syncthreads();
    for (; c < nchunks; c += gridDim.x) {
        if (c != blockIdx.x) dec_load_keys<kInt8, ROW_THREADS>(c, kblk, kq8, active, kv);
        dec_score_chunk<NQ, kInt8, ROW_THREADS>(qs, c, kv, kscale, nq, active, scores, g_decode_gmax, gk);
    }
    if (threadIdx.x == 0) {
        // The arrival releases this CTA's scores and group maxima (ordered
        // before it by the CTA barrier that ends the scoring); a top-k CTA's
        // acquire load that reads the full count synchronises with every
        // arrival.
        if (atom_add_acq_rel_gpu(&g_decode_sync[gen & 1u], 1u) == gridDim.x - 1) {
            g_decode_sync[(gen + 1u) & 1u] = 0u;   // read by the next launch only, after this grid completes
            g_decode_sync[2] = gen + 1u;
        }
    }
    if (blockIdx.x >= static_cast<unsigned>(nq)) return;   // the whole CTA
    // (Diagnostics only, qsa_debug_inject: wait for one arrival more than the
    // grid has, so the wait runs out.)
    const uint32_t target = gridDim.x + ((inject & 2u) != 0u ? 1u : 0u);
    if (threadIdx.x == 0 && !wait_word_reaches(&g_decode_sync[gen & 1u], target, wait_ns))
        atomicOr(&g_topk_error, 2u);
    __syncthreads();
    // Short rows take the register-resident path.
    if (active <= 4 * ROW_THREADS)
        topk_reg_row<4, true>(scores, active, k, ids, blockIdx.x);
    else if (active <= 8 * ROW_THREADS)
        topk_reg_row<8, true>(scores, active, k, ids, blockIdx.x);
    else if (active <= REG_MAX_ACTIVE)
        topk_reg_row<16, true>(scores, active, k, ids, blockIdx.x);
    else
        topk_row<true>(scores, g_decode_gmax, active, k, ids, blockIdx.x);
}

// ---- fused select: scores and top-k without the scores ----------------------
// Step 1 (select_threshold_kernel, one CTA per SEL_ROWS query rows): a threshold that
// about 1.8 k + 8 n / S of the row's n scores are expected to reach: the
// r-th largest key, r = ceil(1.8 k S / n) + 8, of a strided sample of S =
// LIST_SAMPLE blocks scored on CUDA cores (the same head-summed query and
// fp32 FMA; its rounding only moves the threshold). Step 2 (the tensor-core
// scorer in list mode) appends every score at or above its row's threshold,
// as (fp32 bits, block id), to the row's list instead of storing scores. Step 3
// (select_list_kernel): when a row's list holds at least k entries and did
// not overflow, it holds every score at or above the threshold and therefore
// the whole top-k, ties included, and the exact digit search runs on it;
// otherwise the row is flagged and its query group goes through the plain
// scorer and top-k (steps 4 and 5). The result is exact either way.
constexpr int LIST_SAMPLE = 1024;
constexpr int LIST_PER = LIST_CAP / ROW_THREADS;   // list entries per thread in step 3
static_assert(LIST_CAP % ROW_THREADS == 0 && LIST_PER <= 32, "list entries in registers");

// SEL_ROWS query rows per CTA share each sample key row (read once from L2 for
// all of them); a warp scores one sample block per step, SEL_BATCH blocks'
// loads in flight.
constexpr int SEL_ROWS = 2;
constexpr int SEL_BATCH = 16;
static_assert(LIST_SAMPLE % (ROW_WARPS * SEL_BATCH) == 0, "whole sample batches");
static_assert(SEL_ROWS * D <= ROW_THREADS, "one thread per query value");

__global__ void __launch_bounds__(ROW_THREADS, 1)
    select_threshold_kernel(const float *__restrict__ q, const float *__restrict__ kblk, int nq, int active, int k,
                            float *__restrict__ thr, uint32_t *__restrict__ cnt, uint32_t *__restrict__ fail,
                            uint32_t *__restrict__ gfail) {
    __shared__ __align__(16) float qs[SEL_ROWS][D];
    __shared__ uint32_t keys[SEL_ROWS][LIST_SAMPLE];
    __shared__ __align__(16) uint32_t hist[BINS_R];
    __shared__ uint32_t sel[3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row0 = blockIdx.x * SEL_ROWS;
    const int nr = min(SEL_ROWS, nq - row0);
    if (tid < BINS_R) hist[tid] = 0u;
    // q and the keys may come from the previous grid; the scorer that follows
    // may start once every CTA is past this wait (it reads q and the keys,
    // not these thresholds, before waiting for this grid).
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid < SEL_ROWS * D) {
        const int r = tid / D, d = tid % D;
        float v = 0.0f;
        if (r < nr) {
            const float *p = q + static_cast<size_t>(row0 + r) * (HEADS * D) + d;
            v = __fadd_rn(__fadd_rn(__fadd_rn(ld_in(p), ld_in(p + D)), ld_in(p + 2 * D)), ld_in(p + 3 * D));
        }
        qs[r][d] = v;
    }
    if (tid < nr) {
        const int row = row0 + tid;
        cnt[row] = 0u;
        fail[row] = 0u;
        if (row % 128 == 0) gfail[row / 128] = 0u;
    }
    __syncthreads();
    // Sample block j: j * n / S (a warp per block: 16 bytes of the key row per lane).
    float4 qv[SEL_ROWS];
#pragma unroll
    for (int r = 0; r < SEL_ROWS; ++r) qv[r] = *reinterpret_cast<const float4 *>(&qs[r][4 * lane]);
#pragma unroll 1
    for (int j0 = warp; j0 < LIST_SAMPLE; j0 += ROW_WARPS * SEL_BATCH) {
        float4 kv[SEL_BATCH];
#pragma unroll
        for (int u = 0; u < SEL_BATCH; ++u) {
            const long long b = static_cast<long long>(j0 + u * ROW_WARPS) * active / LIST_SAMPLE;
            kv[u] = ld_in(reinterpret_cast<const float4 *>(kblk + b * D) + lane);
        }
#pragma unroll
        for (int u = 0; u < SEL_BATCH; ++u) {
#pragma unroll
            for (int r = 0; r < SEL_ROWS; ++r) {
                float acc = fmaf(qv[r].w, kv[u].w, fmaf(qv[r].z, kv[u].z, fmaf(qv[r].y, kv[u].y, qv[r].x * kv[u].x)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
                if (lane == 0) keys[r][j0 + u * ROW_WARPS] = score_key(acc);
            }
        }
    }
    __syncthreads();
    // Per row, the r-th largest sample key, 8 bits at a time (two keys per
    // thread); each digit's find clears the histogram for the next.
    static_assert(LIST_SAMPLE == 2 * ROW_THREADS, "two sample keys per thread");
#pragma unroll 1
    for (int rr = 0; rr < nr; ++rr) {   // uniform
        const uint32_t k0 = keys[rr][tid], k1 = keys[rr][tid + ROW_THREADS];
        uint32_t r = static_cast<uint32_t>((9ull * static_cast<uint64_t>(k) * LIST_SAMPLE + 5ull * active - 1) /
                                           (5ull * active)) + 8u;
        if (r > LIST_SAMPLE) r = LIST_SAMPLE;
        uint32_t prefix = 0u, mask = 0u;
#pragma unroll 1
        for (int shift = 24; shift >= 0; shift -= 8) {
            if ((k0 & mask) == prefix) atomicAdd(&hist[(k0 >> shift) & 255u], 1u);
            if ((k1 & mask) == prefix) atomicAdd(&hist[(k1 >> shift) & 255u], 1u);
            __syncthreads();
            if (warp == 0) {
                uint32_t bin, above, c;
                warp_find_256(hist, r, true, lane, bin, above, c);
                if (lane == 0) {
                    sel[0] = bin;
                    sel[1] = above;
                    sel[2] = c;
                }
            }
            __syncthreads();
            r -= sel[1];
            prefix |= sel[0] << shift;
            mask |= 255u << shift;
            const bool whole = sel[2] == r;   // every key of the bin is among the r largest
            __syncthreads();                   // sel read by all before the next digit rewrites it
            if (whole) break;                  // (uniform) prefix is a key at least r sample keys reach
        }
        if (tid == 0) {
            // x >= ft exactly when key(x) >= prefix (NaN, key of -inf, fails it).
            thr[row0 + rr] = __uint_as_float(prefix >= 0x80000000u ? (prefix ^ 0x80000000u) : ~prefix);
        }
    }
}

// Step 3: one CTA per row; the row's list (at most LIST_CAP (score bits, id) pairs,
// LIST_PER per thread) is read into registers and selected exactly, the ids
// marked in bitmaps over [0, active) and written ascending. A row whose list
// is short or overflowed is flagged (and its query group), and left to the
// fallback steps.
__global__ void __launch_bounds__(ROW_THREADS, 2)
    select_list_kernel(const uint2 *__restrict__ cand, const uint32_t *__restrict__ cnt, int active, int k,
                       int32_t *__restrict__ ids, uint32_t *__restrict__ fail, uint32_t *__restrict__ gfail) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int nwords = (active + 31) >> 5;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem_raw);
    uint32_t *selbits = reinterpret_cast<uint32_t *>(smem_raw + SHARED_BYTES);
    uint32_t *tiebits = selbits + nwords;
    reinterpret_cast<uint4 *>(sh.histA)[tid] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < BINS_R) sh.histR[tid] = 0u;
    for (int i = tid; i < 2 * nwords; i += ROW_THREADS) selbits[i] = 0u;   // both bitmaps
    grid_dependency_wait();   // the lists of the scorer before this grid
    const uint32_t n = ld_in(cnt + row);
    if (n < static_cast<uint32_t>(k) || n > static_cast<uint32_t>(LIST_CAP)) {   // uniform: the whole CTA
        if (tid == 0) {
            fail[row] = 1u;
            atomicOr(&gfail[row / 128], 1u);
        }
        return;
    }
    const uint2 *c = cand + static_cast<size_t>(row) * LIST_CAP;
    uint32_t key[LIST_PER], id[LIST_PER];
    uint32_t valid = 0u;
#pragma unroll
    for (int j = 0; j < LIST_PER; ++j) {
        const uint32_t e = static_cast<uint32_t>(j * ROW_THREADS + tid);
        key[j] = 0u;
        id[j] = 0u;
        if (e < n) {
            const uint2 v = __ldcg(c + e);
            key[j] = score_key(__uint_as_float(v.x));
            id[j] = v.y;
            valid |= 1u << j;
        }
    }
    __syncthreads();
    const DigitResult r = reg_digit_search<LIST_PER>(key, valid, k, sh, tid, lane, warp);
#pragma unroll
    for (int j = 0; j < LIST_PER; ++j) {
        if (!(valid >> j & 1u)) continue;
        const uint32_t km = key[j] & r.mask;
        const uint32_t b = id[j];
        if (km > r.prefix || (r.done && km == r.prefix))
            atomicOr(&selbits[b >> 5], 1u << (b & 31u));
        else if (km == r.prefix)
            atomicOr(&tiebits[b >> 5], 1u << (b & 31u));
    }
    __syncthreads();
    finish_row(selbits, tiebits, nwords, !r.done, r.kk, k, ids + static_cast<size_t>(row) * k, sh, tid, lane, warp);
}

__global__ void topk_all_kernel(int active, int k, size_t total, int32_t *__restrict__ ids) {
    for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(t % static_cast<size_t>(k));
        ids[t] = j < active ? j : -1;
    }
}

}  // namespace

cudaError_t launch_topk(const float *scores, const uint32_t *gmax, int nq, int active, int k, int32_t *ids,
                        cudaStream_t stream, const uint32_t *gate) {
    if (active > MAX_ACTIVE) return cudaErrorInvalidValue;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(row_smem_bytes(MAX_ACTIVE)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq));
    cfg.blockDim = dim3(ROW_THREADS);
    cfg.dynamicSmemBytes = row_smem_bytes(active);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (active <= REG_MAX_ACTIVE) {
        if (active <= 4 * ROW_THREADS)
            return cudaLaunchKernelEx(&cfg, topk_reg_kernel<4>, scores, active, k, ids, gate);
        if (active <= 8 * ROW_THREADS)
            return cudaLaunchKernelEx(&cfg, topk_reg_kernel<8>, scores, active, k, ids, gate);
        return cudaLaunchKernelEx(&cfg, topk_reg_kernel<16>, scores, active, k, ids, gate);
    }
    return cudaLaunchKernelEx(&cfg, topk_row_kernel, scores, gmax, active, k, ids, gate);
}

template <int NQ, bool kInt8>
cudaError_t launch_decode_nq(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale, int nq,
                             int active, int k, float *scores, int32_t *ids, cudaStream_t stream) {
    auto kernel = select_decode_kernel<NQ, kInt8>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(row_smem_bytes(MAX_ACTIVE)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const size_t smem = row_smem_bytes(active);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, ROW_THREADS, smem);
    if (e != cudaSuccess) return e;
    constexpr int ROWS = ROW_THREADS / dec_tpr<kInt8>();
    const long long nchunks = (static_cast<long long>(active) + ROWS - 1) / ROWS;
    long long grid = static_cast<long long>(per_sm) * device_sm_count();   // all resident at once
    if (grid > nchunks) grid = nchunks;
    if (grid < nq) grid = nq;
    if (per_sm < 1 || grid > static_cast<long long>(per_sm) * device_sm_count()) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(ROW_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, q, kblk, kq8, reinterpret_cast<const __half *>(kscale), nq, active, k,
                              scores, ids, wait_limit_ns(), debug_inject());
}

cudaError_t launch_select_decode(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale,
                                 int nq, int active, int k, float *scores, int32_t *ids, cudaStream_t stream) {
    if (active > MAX_ACTIVE || k >= active || nq < 1 || nq > SMALL_NQ_MAX) return cudaErrorInvalidValue;
    const bool i8 = kq8 != nullptr;
    switch (nq) {
        case 1:
            return i8 ? launch_decode_nq<1, true>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream)
                      : launch_decode_nq<1, false>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream);
        case 2:
            return i8 ? launch_decode_nq<2, true>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream)
                      : launch_decode_nq<2, false>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream);
        default:
            return i8 ? launch_decode_nq<4, true>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream)
                      : launch_decode_nq<4, false>(q, kblk, kq8, kscale, nq, active, k, scores, ids, stream);
    }
}

cudaError_t launch_select_threshold(const float *q, const float *kblk, int nq, int active, int k, float *thr,
                                    uint32_t *cnt, uint32_t *fail, uint32_t *gfail, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((nq + SEL_ROWS - 1) / SEL_ROWS));
    cfg.blockDim = dim3(ROW_THREADS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_threshold_kernel, q, kblk, nq, active, k, thr, cnt, fail, gfail);
}

cudaError_t launch_select_list(const uint2 *cand, const uint32_t *cnt, int nq, int active, int k, int32_t *ids,
                               uint32_t *fail, uint32_t *gfail, cudaStream_t stream) {
    if (active > MAX_ACTIVE) return cudaErrorInvalidValue;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(select_list_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(row_smem_bytes(MAX_ACTIVE)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq));
    cfg.blockDim = dim3(ROW_THREADS);
    cfg.dynamicSmemBytes = row_smem_bytes(active);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_list_kernel, cand, cnt, active, k, ids, fail, gfail);
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

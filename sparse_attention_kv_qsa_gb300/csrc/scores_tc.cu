// Block scoring on the 5th-generation tensor cores (tcgen05, TMEM), with
// fp32 operands split exactly into three bf16 slices.
//
//   score[i][b] = sum_{h<4} sum_{d<128} q[i][h][d] * key[b][d]
//               = sum_{d<128} s[i][d] * key[b][d],   s[i][d] = ((q0 + q1) + q2) + q3
//
// Passages: "#3108 optimize exact QSA block scoring and top-k selection on
// gfx12", Summary items 1 and 4 (the 4-head block score); "#337 gfx12 QSA
// select", What item 2 (a tensor-core scorer splits each fp32 operand into
// three exact 8-bit-mantissa bf16 slices hi/mid/lo, sums the six products of
// order <= 2, keeps hi*hi in its own accumulator and the five corrections in
// another, and adds the two once at the end).
//
// Split: hi = x with the low 16 bits cleared, r = x - hi (exact), mid = r
// with the low 16 bits cleared, lo = r - mid (exact, at most 8 significant
// bits), so x = hi + mid + lo exactly for normal x. The dropped products
// (mid*lo, lo*mid, lo*lo) are of relative order 2^-24.
//
// int8 keys (times one binary16 scale per block) are exact in one bf16 slice,
// so that form needs three products; the scale multiplies the sum.
//
// GB300 mapping, one persistent CTA per SM, CTAs grouped by 128 queries:
//  - MMA D[query][block] = A[query][d] . B[block][d], M = 128 queries,
//    N = 128 blocks per tile, K = 16 per instruction (an N = 128 MMA does
//    twice the work of an N = 64 one in about 1.45 times the cycles).
//  - A: the group's head-summed queries, three slices resident in TMEM
//    (192 of the 512 columns), written once by the epilogue warps.
//  - B: key tiles in K-halves. A producer warp loads raw key pieces of
//    64 rows x 64 d with 2-D tensor copies (16 KiB fp32) into a 6-slot
//    ring; 6 converter warps split them into three 128-byte-swizzled
//    K-major bf16 slices of a K-half stage (3 x 16 KiB), 2 stages in flight.
//  - One thread issues tcgen05.mma into two accumulators (hi*hi;
//    corrections), 128 columns each, and frees each K-half stage and hands
//    the finished tile to the epilogue with tcgen05.commit. Its SM
//    sub-partition also holds two epilogue warps and one converter.
//  - 8 epilogue warps (two per TMEM lane quarter, one per column half;
//    thread = query row) read both accumulators out at once, so the next
//    tile's MMAs can start, add them, and store the scores by 2-D tensor
//    stores (or coalesced direct stores when rows are not 16-byte aligned);
//    on request they also store the key of each 32-block group's largest
//    score (the group maxima the top-k can use).
//  - Key rows at or beyond `active` are never read; the grid comes from
//    `active` and nq alone.
// Every mbarrier wait is bounded; a timeout sets the error word.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int TILE_N = 128;                    // key blocks per tile (MMA N)
constexpr int QGROUP = 128;                    // queries per CTA group (MMA M)
constexpr int KHALF = D / 2;                   // d per K-half: one 128-byte row of bf16
constexpr int PIECE_ROWS = 64;                 // key rows per raw piece (one K-half)
constexpr int RAW_SLOTS = 6;
constexpr int RAW_SLOT_BYTES = PIECE_ROWS * KHALF * 4;   // 16 KiB (fp32)
constexpr int KS_STAGES = 2;                   // K-half key stages in flight
constexpr int KS_SUB_BYTES = TILE_N * 128;     // one slice of one K-half: 128 rows x 128 B
constexpr int KS_STAGE_BYTES = 3 * KS_SUB_BYTES;    // 48 KiB
constexpr int OUT_BOX_COLS = 32;                   // tensor-store box: 32 scores (128 B) x 128 rows
constexpr int OUT_BOX_BYTES = QGROUP * OUT_BOX_COLS * 4;   // 16 KiB, 128-byte swizzled
constexpr int OUT_BYTES = 2 * OUT_BOX_BYTES;               // one column half of a tile: 32 KiB
constexpr int OUT_ROWS = 8;                                // direct stores: rows per warp transpose
constexpr int OUT_ROW_BYTES = (TILE_N / 2) * 4 + 16;       // padded: conflict-free 16-byte stores
// Warp roles. Warp w runs on SM sub-partition w % 4 and reads TMEM lanes
// 32 (w % 4) .. +31. The MMA issuer (warp 1) shares its sub-partition with two
// epilogue warps (5, 9) and one converter (13): at one MMA per ~70 cycles the
// issuer needs few issue slots.
constexpr int PRODUCER_WARP = 0, MMA_WARP = 1;
constexpr int EPI_WARP0 = 2, EPI_WARPS = 8;       // warps 2..9: lane quarters 2, 3, 0, 1 twice
constexpr int CONV_WARPS = 6;                     // warps 10..15
constexpr int TC_THREADS = 16 * 32;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COLS_PER_SLICE = D / 2;   // 64 columns: 128 bf16 packed in pairs
constexpr uint32_t ACC0_COL = 3 * A_COLS_PER_SLICE;   // 192: hi*hi, 128 columns
constexpr uint32_t ACC1_COL = ACC0_COL + TILE_N;      // 320: corrections, 128 columns
static_assert(ACC1_COL + TILE_N <= TMEM_COLS, "accumulators fit TMEM");

// Shared memory, from a 1,024-byte-aligned base.
constexpr int KS_OFF = 0;                                   // 2 x 48 KiB
constexpr int RAW_OFF = KS_OFF + KS_STAGES * KS_STAGE_BYTES;  // 6 x 16 KiB
constexpr int OUT_OFF = RAW_OFF + RAW_SLOTS * RAW_SLOT_BYTES;   // 32 KiB, 1,024-byte aligned
constexpr int BAR_OFF = OUT_OFF + OUT_BYTES;
static_assert(OUT_OFF % 1024 == 0, "128-byte swizzled staging needs 1,024-byte alignment");
static_assert(EPI_WARPS * OUT_ROWS * OUT_ROW_BYTES <= OUT_BYTES, "direct-store staging fits");

struct TcBarriers {
    uint64_t raw_full[RAW_SLOTS];   // producer -> converters (tensor copy landed)
    uint64_t raw_empty[RAW_SLOTS];  // converters -> producer
    uint64_t ks_full[KS_STAGES];    // converters -> MMA: key slices written
    uint64_t ks_empty[KS_STAGES];   // MMA -> converters: key slices consumed
    uint64_t acc_full[2];           // MMA -> epilogue: accumulator 0 (hi*hi) / 1 final for the tile
    uint64_t acc_empty[2];          // epilogue -> MMA: accumulator 0 / 1 read out
    uint64_t a_ready;               // query slices in TMEM
    uint64_t q_peer;                // CTA pairs: the peer's half of the query slices landed
    uint64_t mma_drain;             // MMA thread: every MMA it issued has completed
    uint32_t tmem_base;
    uint32_t abort;                 // set by the first timed-out wait: later waits return at once
};

static_assert(sizeof(TcBarriers) <= 256, "barriers fit their slot");
// Group-maximum exchange: the second column team's two keys per query row,
// read by the first team, which stores the tile's four with one 16-byte store.
constexpr int GX_OFF = BAR_OFF + 256;
constexpr size_t TC_SMEM = GX_OFF + QGROUP * 8 + 1024;

__device__ uint32_t g_tc_error;

// Barrier 1 over every warp but the producer (which is already streaming).
__device__ __forceinline__ void sync_non_producer() {
    asm volatile("bar.sync 1, %0;" ::"r"(TC_THREADS - 32) : "memory");
}

// Query slices are staged once through the (still unused) key-slice stages:
// slice s, row r, 16-byte chunk c at QS_OFF + s * 32 KiB + r * 256 + (c ^ (r & 15)) * 16.
constexpr int QS_OFF = KS_OFF;
constexpr int QS_SLICE_BYTES = QGROUP * (D / 8) * 16;   // 32 KiB
static_assert(3 * QS_SLICE_BYTES <= KS_STAGES * KS_STAGE_BYTES, "query staging fits the key stages");
static_assert(TC_SMEM <= 232448, "shared memory per CTA");
constexpr uint32_t QS_PEER_BYTES = 3u * (QGROUP / 2) * (D / 8) * 16u;   // the peer's 64 rows, 3 slices

// Converter index of a warp, or -1.
__device__ __forceinline__ int converter_index(int warp) { return warp < 10 ? -1 : warp - 10; }

__device__ __forceinline__ uint32_t qs_off(int s, int r, int c) {
    return QS_OFF + s * QS_SLICE_BYTES + r * 256 + ((c ^ (r & 15)) << 4);
}

// A bounded wait of the pipeline. The first one that runs out sets the
// error word and the CTA's abort word; from then on every wait of the CTA
// returns false at once, so the roles leave their loops (each first waits,
// bounded, for its own asynchronous operations in flight) instead of each
// running out in turn.
__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, uint32_t *abort, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;   // the common case reads no abort word
    volatile uint32_t *ab = abort;
    if (*ab != 0u) return false;
    if (mbar_wait(bar, parity, limit_ns, ab)) return true;
    *ab = 1u;
    atomicOr(&g_tc_error, 1u);
    return false;
}

// x = hi + mid + lo, each an fp32 bit pattern whose low 16 bits are zero
// (a bf16 in the upper half).
__device__ __forceinline__ void split3(float x, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    hi = __float_as_uint(x) & 0xFFFF0000u;
    const float r = __fsub_rn(x, __uint_as_float(hi));
    mid = __float_as_uint(r) & 0xFFFF0000u;
    lo = __float_as_uint(__fsub_rn(r, __uint_as_float(mid)));
}

// bf16x2 word from the upper halves of two fp32 patterns (a in the low half).
__device__ __forceinline__ uint32_t pack2(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

// Byte offset of 16-byte chunk c (8 bf16) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(c ^ (r & 7)) << 4);
}

// kSelect: the fused select's list and gated modes (sel), compiled apart so
// that the plain scorer carries none of their code.
template <bool kInt8, bool kSelect>
__global__ void __launch_bounds__(TC_THREADS, 1)
    scores_tc_kernel(const float *__restrict__ q, const __half *__restrict__ kscale, int nq, int active,
                     int ntiles, int ctas_per_group, float *__restrict__ scores, uint32_t *__restrict__ gmax,
                     const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap out_map,
                     int use_tma, int pair, uint64_t wait_ns, uint32_t inject, const TcSelect sel) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t base = raw + pad;
    TcBarriers *bars = reinterpret_cast<TcBarriers *>(smem_raw + pad + BAR_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = blockIdx.x / ctas_per_group;
    const int j0 = blockIdx.x % ctas_per_group;
    const int q0 = group * QGROUP;
    const int qn = min(QGROUP, nq - q0);
    const int nlocal = j0 < ntiles ? (ntiles - 1 - j0) / ctas_per_group + 1 : 0;
    if (kSelect && sel.gate != nullptr) {
        // Gated (the fused select's fallback): only query groups with a
        // flagged row; both CTAs of a pair belong to the same group.
        grid_dependency_wait();
        if (ld_in(sel.gate + group) == 0u) return;
    }
    const bool list_mode = kSelect && !kInt8 && sel.thr != nullptr;
    constexpr uint32_t PIECE_BYTES = PIECE_ROWS * KHALF * (kInt8 ? 1 : 4);
    auto tile_b0 = [&](int li) { return (j0 + li * ctas_per_group) * TILE_N; };

    if (tid == 0) {
        for (int s = 0; s < RAW_SLOTS; ++s) {
            mbar_init(&bars->raw_full[s], 1);
            mbar_init(&bars->raw_empty[s], CONV_THREADS);
        }
        for (int s = 0; s < KS_STAGES; ++s) {
            mbar_init(&bars->ks_full[s], CONV_THREADS);
            mbar_init(&bars->ks_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->acc_full[s], 1);
            mbar_init(&bars->acc_empty[s], EPI_THREADS);
        }
        mbar_init(&bars->a_ready, EPI_THREADS);
        mbar_init(&bars->q_peer, 1);
        mbar_init(&bars->mma_drain, 1);
        bars->abort = 0u;
        if (pair) mbar_arrive_expect_tx(&bars->q_peer, QS_PEER_BYTES);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();  // barriers initialised, TMEM allocated
    if (pair) cluster_sync_all();  // ... in both CTAs of the pair
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    uint32_t *abort = &bars->abort;
    // The pipeline's waits: bounded by wait_ns, abandoned once the CTA aborts.
    auto wait = [&](uint64_t *bar, uint32_t parity) { return wait_or_flag(bar, parity, abort, wait_ns); };
    // Inputs may come from the previous grid on the stream; the next grid (the
    // top-k) may launch now and waits for this one's scores itself. In list
    // mode the previous grid (the thresholds) let this one start only after
    // it had waited for its own predecessor, so q and the keys are final;
    // the epilogue waits for the thresholds themselves.
    if (!list_mode) grid_dependency_wait();
    grid_launch_dependents();

    const int npieces = 4 * nlocal;
    // Diagnostics only (qsa_debug_inject): CTA 0 never loads its first piece,
    // so a wait of the pipeline runs out.
    const bool skip_first = (inject & 1u) != 0u && blockIdx.x == 0;
    auto issue_piece = [&](int p) {   // piece p: tile p / 4, K-half (p / 2) % 2, rows 64 * (p % 2) .. +63
        const int slot = p % RAW_SLOTS;
        const int row0 = tile_b0(p >> 2) + (p & 1) * PIECE_ROWS;
        if (p == 0 && skip_first) return;
        if (row0 < active) {
            mbar_arrive_expect_tx(&bars->raw_full[slot], PIECE_BYTES);
            tma_load_2d(base + RAW_OFF + slot * RAW_SLOT_BYTES, &key_map, ((p >> 1) & 1) * KHALF, row0,
                        &bars->raw_full[slot]);
        } else {
            mbar_arrive(&bars->raw_full[slot]);
        }
    };

    // Head-summed query slices: every warp but the producer (which is already
    // streaming keys) builds them into shared memory, one task per 4 d of one
    // query: a warp's 32 tasks read 512 contiguous bytes of one head row per
    // load, so every L2 sector is fetched once; each thread has the loads of
    // four tasks in flight at a time.
    // CTA pairs (a cluster of two in the same query group) split the rows:
    // each builds 64 and also writes them into its peer's staging with
    // asynchronous cluster stores that count on the peer's q_peer barrier, so
    // every query is read from L2 by half as many CTAs. Each CTA also starts at
    // its own rotation of the task order, so that the CTAs of a group do not
    // all hit the same L2 lines at once.
    if (warp != PRODUCER_WARP) {
        const uint32_t rank = pair ? cluster_ctarank() : 0u;
        const int rows0 = pair ? static_cast<int>(rank) * (QGROUP / 2) : 0;
        const int ntask = (pair ? QGROUP / 2 : QGROUP) * (D / 4);   // a power of two
        const uint32_t peer_bar = pair ? map_shared_rank(smem_u32(&bars->q_peer), rank ^ 1u) : 0u;
        const uint32_t peer_base = pair ? map_shared_rank(base, rank ^ 1u) : 0u;
        const int rot = (j0 * 37 * 32) & (ntask - 1);   // a multiple of 32: warps keep whole rows
        constexpr int BUILDERS = TC_THREADS - 32, TPT = 4;   // tasks per thread in flight
#pragma unroll 1
        for (int t0 = tid - 32; t0 < ntask; t0 += TPT * BUILDERS) {
            // All loads of TPT tasks first (the stores below are volatile asm,
            // which the compiler does not move loads across).
            float4 a[TPT][4];
#pragma unroll
            for (int u = 0; u < TPT; ++u) {
                const int tu = t0 + u * BUILDERS;
                const int t = (tu + rot) & (ntask - 1);
                const int r = rows0 + (t >> 5), c4 = t & 31;
                if (tu < ntask && r < qn) {
                    const float4 *p =
                        reinterpret_cast<const float4 *>(q + static_cast<size_t>(q0 + r) * (HEADS * D)) + c4;
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) a[u][hh] = ld_in(p + hh * (D / 4));
                } else {
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) a[u][hh] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < TPT; ++u) {
                const int tu = t0 + u * BUILDERS;
                if (tu >= ntask) break;
                const int t = (tu + rot) & (ntask - 1);
                const int r = rows0 + (t >> 5), c4 = t & 31;
                const float x[4] = {
                    __fadd_rn(__fadd_rn(__fadd_rn(a[u][0].x, a[u][1].x), a[u][2].x), a[u][3].x),
                    __fadd_rn(__fadd_rn(__fadd_rn(a[u][0].y, a[u][1].y), a[u][2].y), a[u][3].y),
                    __fadd_rn(__fadd_rn(__fadd_rn(a[u][0].z, a[u][1].z), a[u][2].z), a[u][3].z),
                    __fadd_rn(__fadd_rn(__fadd_rn(a[u][0].w, a[u][1].w), a[u][2].w), a[u][3].w)};
                uint32_t h[4], m[4], l[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split3(x[e], h[e], m[e], l[e]);
                const uint32_t w[3][2] = {{pack2(h[0], h[1]), pack2(h[2], h[3])},
                                          {pack2(m[0], m[1]), pack2(m[2], m[3])},
                                          {pack2(l[0], l[1]), pack2(l[2], l[3])}};
                // 8 bytes: half (c4 % 2) of the 16-byte chunk c4 / 2 of row r.
#pragma unroll
                for (int sl = 0; sl < 3; ++sl) {
                    const uint32_t off = qs_off(sl, r, c4 >> 1) + 8u * (c4 & 1);
                    st_shared_v2(base + off, w[sl][0], w[sl][1]);
                    if (pair) st_async_v2(peer_base + off, peer_bar, w[sl][0], w[sl][1]);
                }
            }
        }
        sync_non_producer();
    }

    if (warp == PRODUCER_WARP) {
        // ---- raw key pieces -> ring (2-D tensor copies) ------------------------
        // Piece p: tile p / 4, K-half (p / 2) % 2, rows 64 * (p % 2) .. +63.
        if (lane == 0) {
            int p = 0;
            for (; p < npieces; ++p) {
                if (!wait(&bars->raw_empty[p % RAW_SLOTS], ((p / RAW_SLOTS) & 1) ^ 1)) break;
                issue_piece(p);
            }
            // The copies started here must have landed before the CTA leaves:
            // the last RAW_SLOTS pieces (earlier ones were consumed). Without an
            // abort these waits return at once.
            for (int d = p > RAW_SLOTS ? p - RAW_SLOTS : 0; d < p; ++d)
                if (!(d == 0 && skip_first)) mbar_wait(&bars->raw_full[d % RAW_SLOTS], (d / RAW_SLOTS) & 1, wait_ns);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ---- MMA issuer ------------------------------------------------------------
        // Per K-half: the 4 hi*hi MMAs, then the 20 corrections. In the second
        // K-half the hi*hi MMAs come first and are committed on their own, so
        // that accumulator is final (and drained) ~20 MMAs before the tile
        // ends, and the next tile's hi*hi MMAs queue behind this tile's last
        // ones while the corrections accumulator is read out.
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(QGROUP, TILE_N);
            const uint32_t d0 = tmem + ACC0_COL, d1 = tmem + ACC1_COL;
            bool ok = wait(&bars->a_ready, 0);
            tc_fence_after_sync();
            for (int li = 0; ok && li < nlocal; ++li) {
                for (int kh = 0; kh < 2; ++kh) {
                    const int t = 2 * li + kh, ks = t % KS_STAGES;
                    ok = wait(&bars->ks_full[ks], (t / KS_STAGES) & 1);
                    if (ok && kh == 0) ok = wait(&bars->acc_empty[0], (li & 1) ^ 1);
                    if (!ok) break;
                    tc_fence_after_sync();
                    // Slice s of this K-half at stage + s * KS_SUB_BYTES; +32 B per K-step.
                    const uint64_t kdesc = sw128_kmajor_desc(base + KS_OFF + ks * KS_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < KHALF / 16; ++kk)   // hi . hi
                        tc_mma_bf16_ta(d0, tmem + (4 * kh + kk) * 8, kdesc + static_cast<uint64_t>((kk * 32) >> 4),
                                       idesc, (kh | kk) != 0 ? 1u : 0u);
                    if (kh == 1) tc_commit(&bars->acc_full[0]);
                    if (kh == 0) {
                        ok = wait(&bars->acc_empty[1], (li & 1) ^ 1);
                        if (!ok) break;
                        tc_fence_after_sync();
                    }
#pragma unroll
                    for (int kk = 0; kk < KHALF / 16; ++kk) {
                        const uint64_t B0 = kdesc + static_cast<uint64_t>((kk * 32) >> 4);
                        const uint32_t A0 = tmem + (4 * kh + kk) * 8;
                        tc_mma_bf16_ta(d1, A0 + A_COLS_PER_SLICE, B0, idesc, (kh | kk) != 0 ? 1u : 0u);  // mid . hi
                        tc_mma_bf16_ta(d1, A0 + 2 * A_COLS_PER_SLICE, B0, idesc, 1u);                 // lo . hi
                        if constexpr (!kInt8) {
                            const uint64_t B1 = B0 + (KS_SUB_BYTES >> 4), B2 = B0 + ((2 * KS_SUB_BYTES) >> 4);
                            tc_mma_bf16_ta(d1, A0, B1, idesc, 1u);                                     // hi . mid
                            tc_mma_bf16_ta(d1, A0 + A_COLS_PER_SLICE, B1, idesc, 1u);                // mid . mid
                            tc_mma_bf16_ta(d1, A0, B2, idesc, 1u);                                     // hi . lo
                        }
                    }
                    tc_commit(&bars->ks_empty[ks]);
                }
                if (ok) tc_commit(&bars->acc_full[1]);
            }
            // Every MMA issued here has completed before TMEM is freed (at
            // once without an abort: the epilogue has read the last tile).
            tc_commit(&bars->mma_drain);
            mbar_wait(&bars->mma_drain, 0, wait_ns);
        }
        __syncwarp();
    } else if (warp < EPI_WARP0 + EPI_WARPS) {
        // ---- epilogue warps: query slices into TMEM, then scores out -------------
        const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31
        const int team = (warp - EPI_WARP0) >> 2;           // column half of a tile: 0 or 1
        const int row = 32 * quarter + lane;                // query row within the group
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        // The epilogue's waits are not acted on: after an abort they return at
        // once, and the remaining tiles read (garbage) TMEM and store garbage
        // scores -- invalid outputs, reported by the error word -- with the
        // same barrier pattern, so no warp is left waiting at a barrier.
        if (pair) wait(&bars->q_peer, 0);   // the peer's 64 rows have landed
        // This warp's 32 query rows, half of the 16-byte chunks: staged slices -> TMEM.
        for (int c = 8 * team; c < 8 * team + 8; ++c) {
#pragma unroll
            for (int sl = 0; sl < 3; ++sl) {
                const uint4 v = ld_shared_v4(base + qs_off(sl, row, c));
                tmem_st4(lane_addr + sl * A_COLS_PER_SLICE + 4 * c, v.x, v.y, v.z, v.w);
            }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&bars->a_ready);   // the key stages may now be overwritten

        // Scores leave by tensor store (use_tma: rows 16-byte aligned): each
        // team writes its 128 x 64 half of the tile into two 128-byte-swizzled
        // boxes of 32 columns, one team after the other through the same
        // staging, and one thread stores the boxes asynchronously. Otherwise,
        // through a per-warp shared-memory transpose, 8 rows at a time.
        const int epi_tid = tid - EPI_WARP0 * 32;
        const int col0 = 64 * team;                         // first column of this thread's half
        const bool vec_ok = (active & 3) == 0;              // 16-byte aligned row segments
        const uint32_t stage0 = base + OUT_OFF + (warp - EPI_WARP0) * OUT_ROWS * OUT_ROW_BYTES;
        float ft = 0.f;   // list mode: this row's threshold
        if (list_mode) {
            grid_dependency_wait();
            if (row < qn) ft = ld_in(sel.thr + q0 + row);
        }
        for (int li = 0; li < nlocal; ++li) {
            const int b0 = tile_b0(li);
            const int nb = min(TILE_N, active - b0);
            // hi*hi first (final early), then the corrections.
            float v[TILE_N / 2];
            wait(&bars->acc_full[0], li & 1);
            tc_fence_after_sync();
            {
                uint32_t x0[32], x1[32];
                tmem_ld32(lane_addr + ACC0_COL + col0, x0);
                tmem_ld32(lane_addr + ACC0_COL + col0 + 32, x1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = __uint_as_float(x0[j]);
                    v[32 + j] = __uint_as_float(x1[j]);
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&bars->acc_empty[0]);
            wait(&bars->acc_full[1], li & 1);
            tc_fence_after_sync();
            {
                uint32_t x0[32], x1[32];
                tmem_ld32(lane_addr + ACC1_COL + col0, x0);
                tmem_ld32(lane_addr + ACC1_COL + col0 + 32, x1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = __fadd_rn(v[j], __uint_as_float(x0[j]));
                    v[32 + j] = __fadd_rn(v[32 + j], __uint_as_float(x1[j]));
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&bars->acc_empty[1]);               // TMEM free for the next tile
            if constexpr (kInt8) {
#pragma unroll
                for (int j = 0; j < TILE_N / 2; ++j)
                    if (col0 + j < nb)
                        v[j] = __fmul_rn(v[j], __half2float(__ushort_as_half(ld_in_u16(kscale + b0 + col0 + j))));
            }
            if (list_mode) {
                // Append the scores at or above the threshold (x >= ft: NaN
                // fails) to the row's list, as (fp32 bits, block id: the list
                // select takes the keys); one atomic per thread and tile
                // reserves the slots.
                uint32_t h0 = 0u, h1 = 0u;
                if (nb == TILE_N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        h0 |= v[j] >= ft ? 1u << j : 0u;
                        h1 |= v[32 + j] >= ft ? 1u << j : 0u;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        h0 |= static_cast<uint32_t>(col0 + j < nb && v[j] >= ft) << j;
                        h1 |= static_cast<uint32_t>(col0 + 32 + j < nb && v[32 + j] >= ft) << j;
                    }
                }
                const uint32_t c = __popc(h0) + __popc(h1);
                if (c != 0u && row < qn) {
                    uint32_t slot = atomicAdd(sel.cnt + q0 + row, c);
                    uint2 *dst = sel.cand + static_cast<size_t>(q0 + row) * LIST_CAP;
#pragma unroll
                    for (int j = 0; j < TILE_N / 2; ++j) {
                        if (((j < 32 ? h0 : h1) >> (j & 31)) & 1u) {
                            if (slot < static_cast<uint32_t>(LIST_CAP))
                                dst[slot] = make_uint2(__float_as_uint(v[j]), static_cast<uint32_t>(b0 + col0 + j));
                            ++slot;
                        }
                    }
                }
                continue;
            }
            // Group maxima: this thread's 64 columns are two 32-block groups.
            // fmaxf skips NaN (an all-NaN group stays NaN, whose key is that of
            // -inf) and the key maps -0 and +0 together, so the key of the
            // float maximum is the maximum key.
            const int ngr = (active + GROUP_BLOCKS - 1) / GROUP_BLOCKS;
            uint32_t gk[2] = {0u, 0u};
            if (gmax != nullptr) {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int c0 = col0 + GROUP_BLOCKS * g;
                    float m = v[GROUP_BLOCKS * g];
                    if (c0 + GROUP_BLOCKS <= nb) {
#pragma unroll
                        for (int j = 1; j < GROUP_BLOCKS; ++j) m = fmaxf(m, v[GROUP_BLOCKS * g + j]);
                    } else {
#pragma unroll
                        for (int j = 1; j < GROUP_BLOCKS; ++j)
                            if (c0 + j < nb) m = fmaxf(m, v[GROUP_BLOCKS * g + j]);
                    }
                    gk[g] = score_key(m);
                }
            }
            // Whole tiles with 16-byte aligned maxima rows go out as one store
            // of four keys per row (the teams meet at the store barriers);
            // otherwise each thread stores its own.
            const bool gvec = gmax != nullptr && use_tma && (ngr & 3) == 0 && nb == TILE_N;
            if (gmax != nullptr && !gvec && row < qn) {
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    if (col0 + GROUP_BLOCKS * g < nb)
                        gmax[static_cast<size_t>(q0 + row) * ngr + (b0 + col0) / GROUP_BLOCKS + g] = gk[g];
            }
            if (gvec && team == 1) st_shared_v2(base + GX_OFF + row * 8, gk[0], gk[1]);
            if (use_tma && li == nlocal - 1) {
                // The CTA's last tile: its MMAs have completed (acc_full[1]),
                // so the key stages are idle. Each team stages its half in one
                // of them and both halves leave at once: no wait for earlier
                // stores to finish reading a shared staging.
                const uint32_t stg = base + KS_OFF + team * KS_STAGE_BYTES;
#pragma unroll
                for (int j = 0; j < TILE_N / 8; ++j) {
                    const int box = j >> 3, chunk = j & 7;
                    st_shared_v4(stg + box * OUT_BOX_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4),
                                 __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                 __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                }
                fence_proxy_async_smem();
                named_bar_sync(2, EPI_THREADS);
                if (gvec && team == 0 && row < qn) {
                    const uint2 o = ld_shared_v2(base + GX_OFF + row * 8);
                    *reinterpret_cast<uint4 *>(gmax + static_cast<size_t>(q0 + row) * ngr + b0 / GROUP_BLOCKS) =
                        make_uint4(gk[0], gk[1], o.x, o.y);
                }
                if (epi_tid == 0) {
#pragma unroll
                    for (int tm = 0; tm < 2; ++tm) {
                        const uint32_t src = base + KS_OFF + tm * KS_STAGE_BYTES;
                        const int x0 = b0 + 64 * tm;
                        if (x0 < active) tma_store_2d(&out_map, src, x0, q0);
                        if (x0 + OUT_BOX_COLS < active)
                            tma_store_2d(&out_map, src + OUT_BOX_BYTES, x0 + OUT_BOX_COLS, q0);
                    }
                    bulk_commit();
                }
                continue;
            }
            if (use_tma) {
#pragma unroll 1
                for (int tm = 0; tm < 2; ++tm) {
                    if (epi_tid == 0) bulk_wait_read0();    // earlier stores have read the staging
                    named_bar_sync(2, EPI_THREADS);
                    if (tm == 0 && gvec && team == 0 && row < qn) {
                        const uint2 o = ld_shared_v2(base + GX_OFF + row * 8);
                        *reinterpret_cast<uint4 *>(gmax + static_cast<size_t>(q0 + row) * ngr + b0 / GROUP_BLOCKS) =
                            make_uint4(gk[0], gk[1], o.x, o.y);
                    }
                    if (team == tm) {
#pragma unroll
                        for (int j = 0; j < TILE_N / 8; ++j) {
                            const int box = j >> 3, chunk = j & 7;
                            st_shared_v4(base + OUT_OFF + box * OUT_BOX_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4),
                                         __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                         __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                        }
                        fence_proxy_async_smem();
                    }
                    named_bar_sync(2, EPI_THREADS);
                    if (epi_tid == 0) {
                        const int x0 = b0 + 64 * tm;
                        if (x0 < active) tma_store_2d(&out_map, base + OUT_OFF, x0, q0);
                        if (x0 + OUT_BOX_COLS < active)
                            tma_store_2d(&out_map, base + OUT_OFF + OUT_BOX_BYTES, x0 + OUT_BOX_COLS, q0);
                        bulk_commit();
                    }
                }
                continue;
            }
#pragma unroll 1
            for (int h = 0; h < 4; ++h) {
                if ((lane >> 3) == h) {
#pragma unroll
                    for (int j = 0; j < TILE_N / 2; j += 4)
                        st_shared_v4(stage0 + (lane & 7) * OUT_ROW_BYTES + 4 * j, __float_as_uint(v[j]),
                                     __float_as_uint(v[j + 1]), __float_as_uint(v[j + 2]), __float_as_uint(v[j + 3]));
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int id = 32 * i + lane;
                    const int sr = id >> 4, pc = 4 * (id & 15);   // staging row, first column
                    const int r = 32 * quarter + 8 * h + sr;      // query row within the group
                    const int col = col0 + pc;
                    if (r < qn && col < nb) {
                        const uint4 w4 = ld_shared_v4(stage0 + sr * OUT_ROW_BYTES + 4 * pc);
                        float *dst = scores + static_cast<size_t>(q0 + r) * active + b0 + col;
                        if (vec_ok && col + 4 <= nb) {
                            *reinterpret_cast<uint4 *>(dst) = w4;
                        } else {
                            const uint32_t e[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (col + c < nb) dst[c] = __uint_as_float(e[c]);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (epi_tid == 0) bulk_wait0();                     // stores complete before the CTA leaves
    } else if (converter_index(warp) >= 0) {
        // ---- converters: raw pieces -> swizzled bf16 key slices ----------------
        // Half a warp converts one row of a piece (64 d of one key): lane l
        // takes d = 4 (l % 16) .. +3 (one conflict-free 16-byte read) and
        // stores 8 bytes per slice into half of a swizzled 16-byte chunk.
        const int cw = converter_index(warp);
        const int sub = lane & 15, rsel = lane >> 4;
        const int c = sub >> 1, part = sub & 1;
        const int nstage = wait(&bars->a_ready, 0) ? 2 * nlocal : 0;   // query staging has left the key stages
        for (int t = 0; t < nstage; ++t) {             // K-half stage t: tile t / 2, K-half t % 2
            const int ks = t % KS_STAGES;
            const uint32_t kbase = base + KS_OFF + ks * KS_STAGE_BYTES;
            if (!wait(&bars->ks_empty[ks], ((t / KS_STAGES) & 1) ^ 1)) break;
            bool ok = true;
            for (int rh = 0; rh < 2; ++rh) {
                const int p = 2 * t + rh;
                const int slot = p % RAW_SLOTS;
                if (!wait(&bars->raw_full[slot], (p / RAW_SLOTS) & 1)) {
                    ok = false;
                    break;
                }
                const int row0 = tile_b0(t >> 1) + rh * PIECE_ROWS;
                const uint32_t src = base + RAW_OFF + slot * RAW_SLOT_BYTES;
                // A warp's row pairs are i = cw + CONV_WARPS j; all of its reads
                // are issued before any conversion.
                constexpr int NPAIR = PIECE_ROWS / 2;
                constexpr int PER_WARP = (NPAIR + CONV_WARPS - 1) / CONV_WARPS;
                if constexpr (!kInt8) {
                    uint4 a[PER_WARP];
#pragma unroll
                    for (int j = 0; j < PER_WARP; ++j) {
                        const int r = 2 * (cw + CONV_WARPS * j) + rsel;     // row in the piece
                        a[j] = make_uint4(0u, 0u, 0u, 0u);
                        if (r < PIECE_ROWS && row0 + r < active) a[j] = ld_shared_v4(src + r * (KHALF * 4) + 16 * sub);
                    }
#pragma unroll
                    for (int j = 0; j < PER_WARP; ++j) {
                        const int r = 2 * (cw + CONV_WARPS * j) + rsel;
                        if (r < PIECE_ROWS) {
                            const uint32_t dst = kbase + swz(rh * PIECE_ROWS + r, c) + 8 * part;
                            const float x[4] = {__uint_as_float(a[j].x), __uint_as_float(a[j].y),
                                                __uint_as_float(a[j].z), __uint_as_float(a[j].w)};
                            uint32_t h[4], m[4], l[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) split3(x[e], h[e], m[e], l[e]);
                            st_shared_v2(dst, pack2(h[0], h[1]), pack2(h[2], h[3]));
                            st_shared_v2(dst + KS_SUB_BYTES, pack2(m[0], m[1]), pack2(m[2], m[3]));
                            st_shared_v2(dst + 2 * KS_SUB_BYTES, pack2(l[0], l[1]), pack2(l[2], l[3]));
                        }
                    }
                } else {
                    // 4 int8 keys per lane: exact in bf16 (at most 7 significant bits).
                    uint32_t a[PER_WARP];
#pragma unroll
                    for (int j = 0; j < PER_WARP; ++j) {
                        const int r = 2 * (cw + CONV_WARPS * j) + rsel;
                        a[j] = 0u;
                        if (r < PIECE_ROWS && row0 + r < active) a[j] = ld_shared_u32(src + r * KHALF + 4 * sub);
                    }
#pragma unroll
                    for (int j = 0; j < PER_WARP; ++j) {
                        const int r = 2 * (cw + CONV_WARPS * j) + rsel;
                        if (r < PIECE_ROWS) {
                            const uint32_t dst = kbase + swz(rh * PIECE_ROWS + r, c) + 8 * part;
                            uint32_t f[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                f[e] = __float_as_uint(static_cast<float>(static_cast<int8_t>((a[j] >> (8 * e)) & 0xFFu)));
                            st_shared_v2(dst, pack2(f[0], f[1]), pack2(f[2], f[3]));
                        }
                    }
                }
                mbar_arrive(&bars->raw_empty[slot]);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            mbar_arrive(&bars->ks_full[ks]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (pair) cluster_sync_all();  // no CTA leaves while its pair may still touch it
    if (warp == MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time
// dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Tensor map of the scores [nq][active] fp32 for 32 x 128 boxes, 128-byte
// swizzle; false when rows are not 16-byte aligned (active % 4 != 0).
bool encode_out_map(CUtensorMap *map, float *scores, int nq, int active) {
    if ((active & 3) != 0 || (reinterpret_cast<uintptr_t>(scores) & 15u) != 0) return false;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(active), static_cast<cuuint64_t>(nq)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(active) * 4u};
    const cuuint32_t box[2] = {OUT_BOX_COLS, QGROUP};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, scores, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the first `active` key rows ([active][128], fp32 or int8) for
// raw pieces of 64 rows x 64 d, unswizzled; rows past `active` read as zeros.
// The rows are 16-byte aligned (the boundary checks the pointer).
bool encode_key_map(CUtensorMap *map, const void *keys, int active, bool int8) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(active)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * (int8 ? 1u : 4u)};
    const cuuint32_t box[2] = {KHALF, PIECE_ROWS};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(keys), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_scores_tc(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale, int nq,
                             int active, float *scores, uint32_t *gmax, cudaStream_t stream, const TcSelect &sel) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(scores_tc_kernel<false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(TC_SMEM));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(scores_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(TC_SMEM));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(scores_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(TC_SMEM));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int ntiles = (active + TILE_N - 1) / TILE_N;
    const int ngroups = (nq + QGROUP - 1) / QGROUP;
    int per = device_sm_count() / ngroups;
    if (per < 1) per = 1;
    if (per > ntiles) per = ntiles;
    const long long grid = static_cast<long long>(per) * ngroups;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = TC_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // CTA pairs when every group's CTA count is even (always at full size).
    const int pair = (per % 2 == 0) ? 1 : 0;
    cudaLaunchAttribute attrs[2];
    attrs[0] = attr[0];
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = pair ? 2 : 1;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    CUtensorMap out_map, key_map;
    memset(&out_map, 0, sizeof(out_map));
    memset(&key_map, 0, sizeof(key_map));
    const int use_tma = scores != nullptr && encode_out_map(&out_map, scores, nq, active) ? 1 : 0;
    const bool int8 = kq8 != nullptr;
    if (!encode_key_map(&key_map, int8 ? static_cast<const void *>(kq8) : static_cast<const void *>(kblk), active,
                        int8))
        return cudaErrorNotSupported;
    if (int8)
        return cudaLaunchKernelEx(&cfg, scores_tc_kernel<true, false>, q, reinterpret_cast<const __half *>(kscale), nq,
                                  active, ntiles, per, scores, gmax, key_map, out_map, use_tma, pair,
                                  wait_limit_ns(), debug_inject(), TcSelect());
    if (sel.thr != nullptr || sel.gate != nullptr)
        return cudaLaunchKernelEx(&cfg, scores_tc_kernel<false, true>, q, static_cast<const __half *>(nullptr), nq,
                                  active, ntiles, per, scores, gmax, key_map, out_map, use_tma, pair,
                                  wait_limit_ns(), debug_inject(), sel);
    return cudaLaunchKernelEx(&cfg, scores_tc_kernel<false, false>, q, static_cast<const __half *>(nullptr), nq,
                              active, ntiles, per, scores, gmax, key_map, out_map, use_tma, pair, wait_limit_ns(),
                              debug_inject(), sel);
}

cudaError_t tc_error_read_clear(uint32_t *word, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_tc_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace qsa

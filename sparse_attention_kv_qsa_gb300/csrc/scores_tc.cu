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
//    N = 64 blocks per tile, K = 16 per instruction.
//  - A: the group's head-summed queries, three slices resident in TMEM
//    (192 of the 512 columns), written once by the epilogue warps.
//  - B: key tiles. A producer warp streams raw key rows (contiguous, 16 KiB
//    = 32 fp32 rows per copy) into a 4-slot shared-memory ring with bulk
//    async copies; 8 converter warps split them into three 128-byte-swizzled
//    K-major bf16 slices in a 3-stage ring (3 x 48 KiB).
//  - One thread issues tcgen05.mma into two accumulators (hi*hi;
//    corrections) per tile, double-buffered (4 x 64 TMEM columns), and
//    signals stages with tcgen05.commit. Its SM sub-partition holds no
//    converter warp, so the 48 issues of a tile are not slowed by them.
//  - 4 epilogue warps (thread = query row) read the accumulators, add them,
//    and store the scores through a per-warp shared-memory transpose as
//    coalesced 16-byte stores (two 256-byte row segments per instruction).
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

constexpr int TILE_N = 64;                     // key blocks per tile (MMA N)
constexpr int QGROUP = 128;                    // queries per CTA group (MMA M)
constexpr int RAW_ROWS = 32;                   // key rows per raw copy
constexpr int RAW_SLOTS = 3;
constexpr int KS_STAGES = 3;                   // converted key tiles in flight
constexpr int RAW_SLOT_BYTES = RAW_ROWS * D * 4;    // 16 KiB (fp32 rows)
constexpr int KS_SUB_BYTES = TILE_N * 128;          // one slice, one K-half: 64 rows x 128 B
constexpr int KS_STAGE_BYTES = 6 * KS_SUB_BYTES;    // 3 slices x 2 K-halves = 48 KiB
constexpr int OUT_ROW_BYTES = TILE_N * 4 + 16;      // padded: conflict-free 16-byte stores
constexpr int OUT_BOX_COLS = 32;                   // tensor-store box: 32 scores (128 B) x 128 rows
constexpr int OUT_BOX_BYTES = QGROUP * OUT_BOX_COLS * 4;   // 16 KiB, 128-byte swizzled
constexpr int OUT_BYTES = (TILE_N / OUT_BOX_COLS) * OUT_BOX_BYTES;   // 32 KiB
// Warp roles. Warp w runs on SM sub-partition w % 4. The MMA issuers (warps 1
// and 13) share their sub-partition only with one epilogue warp (5) and one
// warp that has no role (9), so nothing competes with the issue of
// tcgen05.mma.
constexpr int PRODUCER_WARP = 0, MMA_WARP = 1, MMA_WARP2 = 13;
constexpr int EPI_WARP0 = 2, EPI_WARPS = 4;       // warps 2..5: TMEM lane quarters 2, 3, 0, 1
constexpr int CONV_WARPS = 8;                     // warps 6, 7, 8, 10, 11, 12, 14, 15
constexpr int TC_THREADS = 16 * 32;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COLS_PER_SLICE = D / 2;   // 64 columns: 128 bf16 packed in pairs
constexpr uint32_t ACC_COL0 = 3 * A_COLS_PER_SLICE;   // 192: accumulators after the query slices
constexpr uint32_t ACC_STAGE_COLS = 2 * TILE_N;       // hi*hi and corrections, 64 columns each

// Shared memory, from a 1,024-byte-aligned base.
constexpr int KS_OFF = 0;                                   // 3 x 48 KiB
constexpr int RAW_OFF = KS_OFF + KS_STAGES * KS_STAGE_BYTES;  // 3 x 16 KiB
constexpr int OUT_OFF = RAW_OFF + RAW_SLOTS * RAW_SLOT_BYTES;   // 32 KiB, 1,024-byte aligned
constexpr int BAR_OFF = OUT_OFF + OUT_BYTES;
static_assert(OUT_OFF % 1024 == 0, "128-byte swizzled staging needs 1,024-byte alignment");
static_assert(EPI_WARPS * 16 * OUT_ROW_BYTES <= OUT_BYTES, "direct-store staging fits");

struct TcBarriers {
    uint64_t raw_full[RAW_SLOTS];   // producer -> converters (bulk copy landed)
    uint64_t raw_empty[RAW_SLOTS];  // converters -> producer
    uint64_t ks_full[KS_STAGES];    // converters -> MMA: key slices written
    uint64_t ks_empty[KS_STAGES];   // MMA -> converters: key slices consumed
    uint64_t acc_full[2];           // MMA -> epilogue
    uint64_t acc_empty[2];          // epilogue -> MMA
    uint64_t a_ready;               // query slices in TMEM
    uint64_t q_peer;                // CTA pairs: the peer's half of the query slices landed
    uint32_t tmem_base;
};

constexpr size_t TC_SMEM = BAR_OFF + sizeof(TcBarriers) + 1024;

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

// Converter index of a warp (warps 9 and 13 have no role), or -1.
__device__ __forceinline__ int converter_index(int warp) {
    return (warp < 6 || warp == 9 || warp == 13) ? -1 : warp - 6 - (warp > 9) - (warp > 13);
}

__device__ __forceinline__ uint32_t qs_off(int s, int r, int c) {
    return QS_OFF + s * QS_SLICE_BYTES + r * 256 + ((c ^ (r & 15)) << 4);
}

__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity) {
    if (!mbar_wait(bar, parity)) atomicOr(&g_tc_error, 1u);
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

template <bool kInt8>
__global__ void __launch_bounds__(TC_THREADS, 1)
    scores_tc_kernel(const float *__restrict__ q, const float *__restrict__ kblk,
                     const int8_t *__restrict__ kq8, const __half *__restrict__ kscale, int nq, int active,
                     int ntiles, int ctas_per_group, float *__restrict__ scores,
                     const __grid_constant__ CUtensorMap out_map, int use_tma, int pair) {
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
    constexpr int ROW_BYTES = kInt8 ? D : D * 4;
    const char *keys = kInt8 ? reinterpret_cast<const char *>(kq8) : reinterpret_cast<const char *>(kblk);
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
    // Inputs may come from the previous grid on the stream; the next grid (the
    // top-k) may launch now and waits for this one's scores itself.
    grid_dependency_wait();
    grid_launch_dependents();

    // Head-summed query slices: every warp but the producer builds them (one
    // 8-d chunk of one query per task, coalesced loads) into shared memory.
    // CTA pairs (a cluster of two in the same query group) split the rows:
    // each builds 64 and also writes them into its peer's staging with
    // asynchronous cluster stores that count on the peer's q_peer barrier, so
    // every query is read from L2 by half as many CTAs. Each CTA also starts at
    // its own rotation of the task order, so that the CTAs of a group do not
    // all hit the same L2 lines at once.
    if (warp != PRODUCER_WARP) {
        const uint32_t rank = pair ? cluster_ctarank() : 0u;
        const int rows0 = pair ? static_cast<int>(rank) * (QGROUP / 2) : 0;
        const int ntask = (pair ? QGROUP / 2 : QGROUP) * (D / 8);   // a power of two
        const uint32_t peer_bar = pair ? map_shared_rank(smem_u32(&bars->q_peer), rank ^ 1u) : 0u;
        const uint32_t peer_base = pair ? map_shared_rank(base, rank ^ 1u) : 0u;
        const int rot = (j0 * 37 * 16) & (ntask - 1);
#pragma unroll 2
        for (int t0 = tid - 32; t0 < ntask; t0 += TC_THREADS - 32) {
            const int t = (t0 + rot) & (ntask - 1);
            const int r = rows0 + (t >> 4), c = t & 15;
            float x[8];
            if (r < qn) {
                const float4 *p =
                    reinterpret_cast<const float4 *>(q + static_cast<size_t>(q0 + r) * (HEADS * D) + 8 * c);
                float4 a[4][2];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    a[h][0] = __ldg(p + h * (D / 4));
                    a[h][1] = __ldg(p + h * (D / 4) + 1);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v0 = e < 4 ? (&a[0][0].x)[e] : (&a[0][1].x)[e - 4];
                    const float v1 = e < 4 ? (&a[1][0].x)[e] : (&a[1][1].x)[e - 4];
                    const float v2 = e < 4 ? (&a[2][0].x)[e] : (&a[2][1].x)[e - 4];
                    const float v3 = e < 4 ? (&a[3][0].x)[e] : (&a[3][1].x)[e - 4];
                    x[e] = __fadd_rn(__fadd_rn(__fadd_rn(v0, v1), v2), v3);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
            uint32_t h[8], m[8], l[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) split3(x[e], h[e], m[e], l[e]);
            const uint32_t w[3][4] = {{pack2(h[0], h[1]), pack2(h[2], h[3]), pack2(h[4], h[5]), pack2(h[6], h[7])},
                                      {pack2(m[0], m[1]), pack2(m[2], m[3]), pack2(m[4], m[5]), pack2(m[6], m[7])},
                                      {pack2(l[0], l[1]), pack2(l[2], l[3]), pack2(l[4], l[5]), pack2(l[6], l[7])}};
#pragma unroll
            for (int sl = 0; sl < 3; ++sl) {
                st_shared_v4(base + qs_off(sl, r, c), w[sl][0], w[sl][1], w[sl][2], w[sl][3]);
                if (pair) st_async_v4(peer_base + qs_off(sl, r, c), peer_bar, w[sl][0], w[sl][1], w[sl][2], w[sl][3]);
            }
        }
        sync_non_producer();
    }

    if (warp == PRODUCER_WARP) {
        // ---- raw key rows -> ring (bulk async copies) --------------------------
        if (lane == 0) {
            const int npieces = 2 * nlocal;
            for (int p = 0; p < npieces; ++p) {
                const int slot = p % RAW_SLOTS;
                wait_or_flag(&bars->raw_empty[slot], ((p / RAW_SLOTS) & 1) ^ 1);
                const int row0 = tile_b0(p >> 1) + (p & 1) * RAW_ROWS;
                const int rows = min(RAW_ROWS, active - row0);
                if (rows > 0) {
                    const uint32_t bytes = static_cast<uint32_t>(rows * ROW_BYTES);
                    mbar_arrive_expect_tx(&bars->raw_full[slot], bytes);
                    bulk_g2s(smem_raw + pad + RAW_OFF + slot * RAW_SLOT_BYTES,
                             keys + static_cast<size_t>(row0) * ROW_BYTES, bytes, &bars->raw_full[slot]);
                } else {
                    mbar_arrive(&bars->raw_full[slot]);
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP || warp == MMA_WARP2) {
        // ---- MMA issuers ---------------------------------------------------------
        // Two threads take alternate tiles (each then owns one accumulator
        // stage), so one issues while the other waits for its next tile's
        // barriers and the tensor pipe never drains between tiles.
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(QGROUP, TILE_N);
            wait_or_flag(&bars->a_ready, 0);
            tc_fence_after_sync();
            for (int li = (warp == MMA_WARP ? 0 : 1); li < nlocal; li += 2) {
                const int st = li & 1, use = li >> 1;
                const int ks = li % KS_STAGES, ks_use = li / KS_STAGES;
                wait_or_flag(&bars->acc_empty[st], (use & 1) ^ 1);
                wait_or_flag(&bars->ks_full[ks], ks_use & 1);
                tc_fence_after_sync();
                const uint32_t d0 = tmem + ACC_COL0 + st * ACC_STAGE_COLS, d1 = d0 + TILE_N;
                const uint32_t kbase = base + KS_OFF + ks * KS_STAGE_BYTES;
                // Fully unrolled: the 48 descriptors differ from the first by constants.
                const uint64_t kdesc = sw128_kmajor_desc(kbase);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // key slice s, K-half h at kbase + (2*s + h) * KS_SUB_BYTES; +32 B per K-step
                    const uint64_t B0 = kdesc + static_cast<uint64_t>(((kk >> 2) * KS_SUB_BYTES + (kk & 3) * 32) >> 4);
                    const uint32_t A0 = tmem + kk * 8;
                    const uint32_t acc = kk == 0 ? 0u : 1u;
                    tc_mma_bf16_ta(d0, A0, B0, idesc, acc);                                   // hi . hi
                    tc_mma_bf16_ta(d1, A0 + A_COLS_PER_SLICE, B0, idesc, acc);               // mid . hi
                    tc_mma_bf16_ta(d1, A0 + 2 * A_COLS_PER_SLICE, B0, idesc, 1u);            // lo . hi
                    if constexpr (!kInt8) {
                        const uint64_t B1 = B0 + ((2 * KS_SUB_BYTES) >> 4), B2 = B0 + ((4 * KS_SUB_BYTES) >> 4);
                        tc_mma_bf16_ta(d1, A0, B1, idesc, 1u);                                // hi . mid
                        tc_mma_bf16_ta(d1, A0 + A_COLS_PER_SLICE, B1, idesc, 1u);           // mid . mid
                        tc_mma_bf16_ta(d1, A0, B2, idesc, 1u);                                // hi . lo
                    }
                }
                tc_commit(&bars->ks_empty[ks]);
                tc_commit(&bars->acc_full[st]);
            }
        }
        __syncwarp();
    } else if (warp < EPI_WARP0 + EPI_WARPS) {
        // ---- epilogue warps: query slices into TMEM, then scores out -------------
        const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31
        const int row = 32 * quarter + lane;                // query row within the group
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        if (pair) wait_or_flag(&bars->q_peer, 0);   // the peer's 64 rows have landed
        // This warp's 32 query rows: staged slices -> TMEM (A operand).
        for (int c = 0; c < D / 8; ++c) {
#pragma unroll
            for (int sl = 0; sl < 3; ++sl) {
                const uint4 v = ld_shared_v4(base + qs_off(sl, row, c));
                tmem_st4(lane_addr + sl * A_COLS_PER_SLICE + 4 * c, v.x, v.y, v.z, v.w);
            }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&bars->a_ready);   // the key stages may now be overwritten

        // Scores leave by tensor store (use_tma: rows 16-byte aligned): the 128
        // threads write the tile's 128 x 64 scores into two 128-byte-swizzled
        // boxes of 32 columns, and one thread stores both asynchronously.
        // Otherwise, through a per-warp shared-memory transpose, half a warp at
        // a time: 16 threads write their query rows' 64 scores to padded staging
        // rows, then the warp stores two rows per instruction.
        const int epi_tid = tid - EPI_WARP0 * 32;
        const bool vec_ok = (active & 3) == 0;              // 16-byte aligned row segments
        const uint32_t stage0 = base + OUT_OFF + quarter * 16 * OUT_ROW_BYTES;
        const uint32_t my_stage = stage0 + (lane & 15) * OUT_ROW_BYTES;
        const int pr = lane >> 4, pc = 4 * (lane & 15);    // row of a pair, first column
        for (int li = 0; li < nlocal; ++li) {
            const int st = li & 1, use = li >> 1;
            const int b0 = tile_b0(li);
            const int nb = min(TILE_N, active - b0);
            wait_or_flag(&bars->acc_full[st], use & 1);
            tc_fence_after_sync();
            const uint32_t t0 = lane_addr + ACC_COL0 + st * ACC_STAGE_COLS;
            uint32_t x0[32], x1[32];
            float v[TILE_N];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(t0 + 32 * half, x0);
                tmem_ld32(t0 + TILE_N + 32 * half, x1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[32 * half + j] = __fadd_rn(__uint_as_float(x0[j]), __uint_as_float(x1[j]));
            }
            tc_fence_before_sync();
            mbar_arrive(&bars->acc_empty[st]);              // TMEM free for the tile after next
            if constexpr (kInt8) {
#pragma unroll
                for (int j = 0; j < TILE_N; ++j)
                    if (j < nb) v[j] = __fmul_rn(v[j], __half2float(kscale[b0 + j]));
            }
            if (use_tma) {
                if (epi_tid == 0) bulk_wait_read0();        // the previous tile's stores have read the boxes
                named_bar_sync(2, EPI_THREADS);
#pragma unroll
                for (int j = 0; j < TILE_N / 4; ++j) {
                    const int box = j >> 3, chunk = j & 7;
                    st_shared_v4(base + OUT_OFF + box * OUT_BOX_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4),
                                 __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                 __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                }
                fence_proxy_async_smem();
                named_bar_sync(2, EPI_THREADS);
                if (epi_tid == 0) {
                    tma_store_2d(&out_map, base + OUT_OFF, b0, q0);
                    if (b0 + OUT_BOX_COLS < active) tma_store_2d(&out_map, base + OUT_OFF + OUT_BOX_BYTES, b0 + OUT_BOX_COLS, q0);
                    bulk_commit();
                }
                continue;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if ((lane >> 4) == h) {
#pragma unroll
                    for (int j = 0; j < TILE_N; j += 4)
                        st_shared_v4(my_stage + 4 * j, __float_as_uint(v[j]), __float_as_uint(v[j + 1]),
                                     __float_as_uint(v[j + 2]), __float_as_uint(v[j + 3]));
                }
                __syncwarp();
#pragma unroll 4
                for (int i = 0; i < 8; ++i) {
                    const int sr = 2 * i + pr;                   // staging row
                    const int r = 32 * quarter + 16 * h + sr;    // query row within the group
                    if (r < qn) {
                        const uint4 w4 = ld_shared_v4(stage0 + sr * OUT_ROW_BYTES + 4 * pc);
                        float *dst = scores + static_cast<size_t>(q0 + r) * active + b0 + pc;
                        if (vec_ok && pc + 4 <= nb) {
                            *reinterpret_cast<uint4 *>(dst) = w4;
                        } else {
                            const uint32_t e[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (pc + c < nb) dst[c] = __uint_as_float(e[c]);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (epi_tid == 0) bulk_wait0();                     // stores complete before the CTA leaves
    } else if (converter_index(warp) >= 0) {
        // ---- converters: raw rows -> swizzled bf16 key slices ------------------
        // A warp converts whole rows: lane l takes d = 4l .. 4l+3 (one conflict-free
        // 16-byte read per lane) and stores 8 bytes per slice into half of a
        // swizzled 16-byte chunk (the two lanes of a chunk share a bank group).
        const int cw = converter_index(warp);
        const int khalf = lane >> 4, c = (lane >> 1) & 7, part = lane & 1;
        wait_or_flag(&bars->a_ready, 0);   // query staging has left the key stages
        int ks = 0, ks_use = 0;
        for (int li = 0; li < nlocal; ++li) {
            const uint32_t kbase = base + KS_OFF + ks * KS_STAGE_BYTES;
            wait_or_flag(&bars->ks_empty[ks], (ks_use & 1) ^ 1);
            for (int half = 0; half < 2; ++half) {
                const int p = 2 * li + half;
                const int slot = p % RAW_SLOTS;
                wait_or_flag(&bars->raw_full[slot], (p / RAW_SLOTS) & 1);
                const int row0 = tile_b0(li) + half * RAW_ROWS;
                const uint32_t src = base + RAW_OFF + slot * RAW_SLOT_BYTES;
#pragma unroll
                for (int i = 0; i < RAW_ROWS / CONV_WARPS; ++i) {
                    const int r = cw + CONV_WARPS * i;               // row in the piece
                    const bool live = row0 + r < active;
                    const uint32_t dst = kbase + khalf * KS_SUB_BYTES + swz(half * RAW_ROWS + r, c) + 8 * part;
                    if constexpr (!kInt8) {
                        uint4 a = make_uint4(0u, 0u, 0u, 0u);
                        if (live) a = ld_shared_v4(src + r * (D * 4) + 16 * lane);
                        const float x[4] = {__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                                            __uint_as_float(a.w)};
                        uint32_t h[4], m[4], l[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) split3(x[e], h[e], m[e], l[e]);
                        st_shared_v2(dst, pack2(h[0], h[1]), pack2(h[2], h[3]));
                        st_shared_v2(dst + 2 * KS_SUB_BYTES, pack2(m[0], m[1]), pack2(m[2], m[3]));
                        st_shared_v2(dst + 4 * KS_SUB_BYTES, pack2(l[0], l[1]), pack2(l[2], l[3]));
                    } else {
                        // 4 int8 keys: exact in bf16 (at most 7 significant bits).
                        uint32_t w = 0u;
                        if (live) w = ld_shared_u32(src + r * D + 4 * lane);
                        uint32_t f[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            f[e] = __float_as_uint(static_cast<float>(static_cast<int8_t>((w >> (8 * e)) & 0xFFu)));
                        st_shared_v2(dst, pack2(f[0], f[1]), pack2(f[2], f[3]));
                    }
                }
                mbar_arrive(&bars->raw_empty[slot]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->ks_full[ks]);
            if (++ks == KS_STAGES) {
                ks = 0;
                ++ks_use;
            }
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

}  // namespace

cudaError_t launch_scores_tc(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale, int nq,
                             int active, float *scores, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(scores_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(TC_SMEM));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(scores_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    CUtensorMap out_map;
    memset(&out_map, 0, sizeof(out_map));
    const int use_tma = encode_out_map(&out_map, scores, nq, active) ? 1 : 0;
    if (kq8 != nullptr)
        return cudaLaunchKernelEx(&cfg, scores_tc_kernel<true>, q, static_cast<const float *>(nullptr), kq8,
                                  reinterpret_cast<const __half *>(kscale), nq, active, ntiles, per, scores,
                                  out_map, use_tma, pair);
    return cudaLaunchKernelEx(&cfg, scores_tc_kernel<false>, q, kblk, static_cast<const int8_t *>(nullptr),
                              static_cast<const __half *>(nullptr), nq, active, ntiles, per, scores, out_map,
                              use_tma, pair);
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

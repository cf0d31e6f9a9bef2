// C ABI of the QSA selection library: argument checks, then launches on the
// caller's stream. Declarations and the contract: include/qsa.h.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/qsa.h"
#include "qsa_internal.cuh"

namespace qsa {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<uint32_t> g_inject{0u};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
uint32_t debug_inject() { return g_inject.load(std::memory_order_relaxed); }

int device_sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace qsa

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

// Largest nq the scorer grid accepts (grid.y = ceil(nq / 128) <= 65535).
constexpr long long MAX_NQ = 65535LL * 128;

qsa_status check_score_args(const float *q, int nq, int max_blocks, int active_blocks,
                            const float *scores) {
    if (nq < 0 || max_blocks < 0 || active_blocks < 0 || active_blocks > max_blocks) return QSA_ERR_INVALID;
    if (nq == 0 || active_blocks == 0) return QSA_OK;
    if (q == nullptr || scores == nullptr) return QSA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(scores)) return QSA_ERR_INVALID;
    if (nq > MAX_NQ) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

// Scores (and, when gmax is given, group maxima) through the kernel for nq.
qsa_status run_scores(const float *q, const float *kblk, const int8_t *kq8, const uint16_t *kscale, int nq,
                      int active, float *scores, uint32_t *gmax, cudaStream_t stream) {
    if (nq <= qsa::SMALL_NQ_MAX)
        return from_cuda(qsa::launch_scores_rows(q, kblk, kq8, kscale, nq, active, scores, gmax, stream));
    return from_cuda(qsa::launch_scores_tc(q, kblk, kq8, kscale, nq, active, scores, gmax, stream));
}

qsa_status scores_f32(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks, float *scores,
                      uint32_t *gmax, bool want_gmax, cudaStream_t stream) {
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK || nq == 0 || active_blocks == 0) return s;
    if (kblk == nullptr || !aligned16(kblk)) return QSA_ERR_INVALID;
    if (want_gmax && (gmax == nullptr || !aligned16(gmax))) return QSA_ERR_INVALID;
    return run_scores(q, kblk, nullptr, nullptr, nq, active_blocks, scores, gmax, stream);
}

qsa_status scores_q8(const float *q, const int8_t *kblk_q8, const uint16_t *kscale_f16, int nq, int max_blocks,
                     int active_blocks, float *scores, uint32_t *gmax, bool want_gmax, cudaStream_t stream) {
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK || nq == 0 || active_blocks == 0) return s;
    if (kblk_q8 == nullptr || kscale_f16 == nullptr || !aligned16(kblk_q8)) return QSA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(kscale_f16) & 1u) != 0) return QSA_ERR_INVALID;
    if (want_gmax && (gmax == nullptr || !aligned16(gmax))) return QSA_ERR_INVALID;
    return run_scores(q, nullptr, kblk_q8, kscale_f16, nq, active_blocks, scores, gmax, stream);
}

qsa_status topk(const float *scores, const uint32_t *gmax, bool want_gmax, int nq, int active_blocks, int k,
                int32_t *ids, cudaStream_t stream) {
    if (nq < 0 || active_blocks < 0 || k < 1) return QSA_ERR_INVALID;
    if (nq == 0) return QSA_OK;
    if (ids == nullptr || !aligned16(ids)) return QSA_ERR_INVALID;
    if (active_blocks > QSA_TOPK_MAX_ACTIVE) return QSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(nq) * k > (1LL << 40)) return QSA_ERR_UNSUPPORTED;
    if (k >= active_blocks) return from_cuda(qsa::launch_topk_all(nq, active_blocks, k, ids, stream));
    if (scores == nullptr || !aligned16(scores)) return QSA_ERR_INVALID;
    if (want_gmax && (gmax == nullptr || !aligned16(gmax))) return QSA_ERR_INVALID;
    if (static_cast<long long>(nq) * 8 > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED;
    return from_cuda(qsa::launch_topk(scores, gmax, nq, active_blocks, k, ids, stream));
}

// Scratch of qsa_block_select_static: the group maxima between its two
// kernels, in the library image (no allocation at call time).
static __device__ __align__(256) uint32_t g_select_gmax[QSA_SELECT_STATIC_GROUPS_MAX];

// Device address of g_select_gmax in the current device's context (looked up
// once per device).
uint32_t *select_scratch() {
    static std::mutex mu;
    static std::vector<uint32_t *> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, nullptr);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_select_gmax) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<uint32_t *>(p);
    }
    return cache[dev];
}

// The fused select's scratch: per row a threshold, a list count, a failure
// flag and a list of LIST_CAP (fp32 score bits, block id) pairs; per query group a flag.
struct SelectScratch {
    float *thr;
    uint32_t *cnt, *fail, *gfail;
    uint2 *cand;
    size_t bytes;
};
size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }
SelectScratch select_layout(void *base, int nq) {
    char *b = static_cast<char *>(base);
    const size_t n = static_cast<size_t>(nq), ngroups = (n + 127) / 128;
    SelectScratch s;
    size_t off = 0;
    s.thr = reinterpret_cast<float *>(b + off);
    off = round16(off + 4 * n);
    s.cnt = reinterpret_cast<uint32_t *>(b + off);
    off = round16(off + 4 * n);
    s.fail = reinterpret_cast<uint32_t *>(b + off);
    off = round16(off + 4 * n);
    s.gfail = reinterpret_cast<uint32_t *>(b + off);
    off = round16(off + 4 * ngroups);
    s.cand = reinterpret_cast<uint2 *>(b + off);
    off += sizeof(uint2) * static_cast<size_t>(qsa::LIST_CAP) * n;
    s.bytes = off;
    return s;
}

}  // namespace

extern "C" {

qsa_status qsa_block_scores(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks,
                            float *scores, cudaStream_t stream) {
    return scores_f32(q, kblk, nq, max_blocks, active_blocks, scores, nullptr, false, stream);
}

qsa_status qsa_block_scores_gmax(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks,
                                 float *scores, uint32_t *group_max, cudaStream_t stream) {
    return scores_f32(q, kblk, nq, max_blocks, active_blocks, scores, group_max, true, stream);
}

qsa_status qsa_block_scores_q8(const float *q, const int8_t *kblk_q8, const uint16_t *kscale_f16, int nq,
                               int max_blocks, int active_blocks, float *scores, cudaStream_t stream) {
    return scores_q8(q, kblk_q8, kscale_f16, nq, max_blocks, active_blocks, scores, nullptr, false, stream);
}

qsa_status qsa_block_scores_q8_gmax(const float *q, const int8_t *kblk_q8, const uint16_t *kscale_f16, int nq,
                                    int max_blocks, int active_blocks, float *scores, uint32_t *group_max,
                                    cudaStream_t stream) {
    return scores_q8(q, kblk_q8, kscale_f16, nq, max_blocks, active_blocks, scores, group_max, true, stream);
}

qsa_status qsa_block_scores_ffma(const float *q, const float *kblk, const int8_t *kblk_q8,
                                 const uint16_t *kscale_f16, int nq, int max_blocks, int active_blocks,
                                 float *scores, cudaStream_t stream) {
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK || nq == 0 || active_blocks == 0) return s;
    const bool f32 = kblk != nullptr;
    const bool i8 = kblk_q8 != nullptr || kscale_f16 != nullptr;
    if (f32 == i8) return QSA_ERR_INVALID;
    if (f32 && !aligned16(kblk)) return QSA_ERR_INVALID;
    if (i8 && (kblk_q8 == nullptr || kscale_f16 == nullptr || !aligned16(kblk_q8) ||
               (reinterpret_cast<uintptr_t>(kscale_f16) & 1u) != 0))
        return QSA_ERR_INVALID;
    return from_cuda(
        qsa::launch_scores_ffma(q, kblk, kblk_q8, kscale_f16, nq, active_blocks, scores, stream));
}

qsa_status qsa_block_topk(const float *scores, int nq, int active_blocks, int k, int32_t *ids,
                          cudaStream_t stream) {
    return topk(scores, nullptr, false, nq, active_blocks, k, ids, stream);
}

qsa_status qsa_block_group_max(const float *scores, int nq, int active_blocks, uint32_t *group_max,
                               cudaStream_t stream) {
    if (nq < 0 || active_blocks < 0) return QSA_ERR_INVALID;
    if (nq == 0 || active_blocks == 0) return QSA_OK;
    if (scores == nullptr || group_max == nullptr || !aligned16(scores) || !aligned16(group_max))
        return QSA_ERR_INVALID;
    return from_cuda(qsa::launch_group_max(scores, nq, active_blocks, group_max, stream));
}

qsa_status qsa_block_topk_gmax(const float *scores, const uint32_t *group_max, int nq, int active_blocks, int k,
                               int32_t *ids, cudaStream_t stream) {
    return topk(scores, group_max, true, nq, active_blocks, k, ids, stream);
}

qsa_status qsa_block_select_static(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks,
                                   int k, float *scores, int32_t *ids, cudaStream_t stream) {
    // Arguments first (the scratch bound included), then both calls.
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK) return s;
    if (k < 1) return QSA_ERR_INVALID;
    if (nq == 0) return QSA_OK;
    if (ids == nullptr || !aligned16(ids)) return QSA_ERR_INVALID;
    if (active_blocks > 0 && (kblk == nullptr || !aligned16(kblk))) return QSA_ERR_INVALID;
    const long long groups = static_cast<long long>(nq) * ((active_blocks + qsa::GROUP_BLOCKS - 1) / qsa::GROUP_BLOCKS);
    if (groups > QSA_SELECT_STATIC_GROUPS_MAX) return QSA_ERR_UNSUPPORTED;
    // The top-k's own size limits, before the scorer launches.
    if (active_blocks > QSA_TOPK_MAX_ACTIVE) return QSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(nq) * k > (1LL << 40)) return QSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(nq) * 8 > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED;
    uint32_t *gm = select_scratch();
    if (gm == nullptr) return QSA_ERR_CUDA;
    if (active_blocks > 0) {
        s = scores_f32(q, kblk, nq, max_blocks, active_blocks, scores, gm, true, stream);
        if (s != QSA_OK) return s;
    }
    return topk(scores, gm, true, nq, active_blocks, k, ids, stream);
}

static_assert(QSA_SELECT_LIST_CAP == qsa::LIST_CAP, "one list capacity");

size_t qsa_block_select_scratch_bytes(int nq) { return nq > 0 ? select_layout(nullptr, nq).bytes : 0; }

qsa_status qsa_block_select(const float *q, const float *kblk, int nq, int max_blocks, int active_blocks, int k,
                            float *scores, int32_t *ids, void *scratch, size_t scratch_bytes, cudaStream_t stream) {
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK) return s;
    if (k < 1) return QSA_ERR_INVALID;
    if (nq == 0) return QSA_OK;
    if (ids == nullptr || !aligned16(ids)) return QSA_ERR_INVALID;
    if (active_blocks > 0 && (kblk == nullptr || !aligned16(kblk) || scores == nullptr)) return QSA_ERR_INVALID;
    if (scratch == nullptr || !aligned16(scratch) || scratch_bytes < select_layout(nullptr, nq).bytes)
        return QSA_ERR_INVALID;
    if (active_blocks > QSA_TOPK_MAX_ACTIVE) return QSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(nq) * k > (1LL << 40)) return QSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(nq) * 8 > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED;
    if (k >= active_blocks) return from_cuda(qsa::launch_topk_all(nq, active_blocks, k, ids, stream));
    // The list path needs the tensor-core scorer (nq > 4), rows past the
    // register-resident top-k's reach and k well inside a list's capacity;
    // otherwise the two plain calls give the same ids.
    if (nq <= qsa::SMALL_NQ_MAX || active_blocks <= QSA_SELECT_LIST_MIN_ACTIVE || k > QSA_SELECT_LIST_K_MAX) {
        s = scores_f32(q, kblk, nq, max_blocks, active_blocks, scores, nullptr, false, stream);
        if (s != QSA_OK) return s;
        return topk(scores, nullptr, false, nq, active_blocks, k, ids, stream);
    }
    const SelectScratch x = select_layout(scratch, nq);
    qsa::TcSelect list;
    list.thr = x.thr;
    list.cnt = x.cnt;
    list.cand = x.cand;
    qsa::TcSelect gated;
    gated.gate = x.gfail;
    cudaError_t e = qsa::launch_select_threshold(q, kblk, nq, active_blocks, k, x.thr, x.cnt, x.fail, x.gfail, stream);
    if (e == cudaSuccess)
        e = qsa::launch_scores_tc(q, kblk, nullptr, nullptr, nq, active_blocks, nullptr, nullptr, stream, list);
    if (e == cudaSuccess) e = qsa::launch_select_list(x.cand, x.cnt, nq, active_blocks, k, ids, x.fail, x.gfail, stream);
    // Rows whose list failed: their query groups' scores, then their top-k
    // (both launches exit at once when no row failed).
    if (e == cudaSuccess)
        e = qsa::launch_scores_tc(q, kblk, nullptr, nullptr, nq, active_blocks, scores, nullptr, stream, gated);
    if (e == cudaSuccess) e = qsa::launch_topk(scores, nullptr, nq, active_blocks, k, ids, stream, x.fail);
    return from_cuda(e);
}

qsa_status qsa_block_select_small(const float *q, const float *kblk, const int8_t *kblk_q8,
                                  const uint16_t *kscale_f16, int nq, int max_blocks, int active_blocks, int k,
                                  float *scores, int32_t *ids, cudaStream_t stream) {
    qsa_status s = check_score_args(q, nq, max_blocks, active_blocks, scores);
    if (s != QSA_OK) return s;
    if (k < 1) return QSA_ERR_INVALID;
    if (nq == 0) return QSA_OK;
    if (nq > qsa::SMALL_NQ_MAX) return QSA_ERR_UNSUPPORTED;
    if (ids == nullptr || !aligned16(ids)) return QSA_ERR_INVALID;
    const bool f32 = kblk != nullptr;
    const bool i8 = kblk_q8 != nullptr || kscale_f16 != nullptr;
    if (f32 == i8) return QSA_ERR_INVALID;
    if (f32 && !aligned16(kblk)) return QSA_ERR_INVALID;
    if (i8 && (kblk_q8 == nullptr || kscale_f16 == nullptr || !aligned16(kblk_q8) ||
               (reinterpret_cast<uintptr_t>(kscale_f16) & 1u) != 0))
        return QSA_ERR_INVALID;
    if (active_blocks > QSA_TOPK_MAX_ACTIVE) return QSA_ERR_UNSUPPORTED;
    if (active_blocks == 0) return from_cuda(qsa::launch_topk_all(nq, 0, k, ids, stream));
    if (k >= active_blocks) {
        cudaError_t e = qsa::launch_scores_rows(q, kblk, kblk_q8, kscale_f16, nq, active_blocks, scores, nullptr,
                                                stream);
        if (e == cudaSuccess) e = qsa::launch_topk_all(nq, active_blocks, k, ids, stream);
        return from_cuda(e);
    }
    return from_cuda(qsa::launch_select_decode(q, kblk, kblk_q8, kscale_f16, nq, active_blocks, k, scores, ids,
                                               stream));
}

qsa_status qsa_sparse_attn(const float *q, const int8_t *k_cells, const uint16_t *k_scale_f16,
                           const int8_t *v_cells, const uint16_t *v_scale_f16, int ncells, const int32_t *ids,
                           int nq, int k, float *out, cudaStream_t stream) {
    if (nq < 0 || k < 1 || ncells < 0) return QSA_ERR_INVALID;
    if (nq == 0) return QSA_OK;
    if (ncells > 0x7FFFFFFF - 4) return QSA_ERR_UNSUPPORTED;   // cell indices stay in int
    if (q == nullptr || ids == nullptr || out == nullptr || !aligned16(q) || !aligned16(ids) || !aligned16(out))
        return QSA_ERR_INVALID;
    if (ncells > 0 && (k_cells == nullptr || v_cells == nullptr || k_scale_f16 == nullptr ||
                       v_scale_f16 == nullptr || !aligned16(k_cells) || !aligned16(v_cells) ||
                       (reinterpret_cast<uintptr_t>(k_scale_f16) & 1u) != 0 ||
                       (reinterpret_cast<uintptr_t>(v_scale_f16) & 1u) != 0))
        return QSA_ERR_INVALID;
    return from_cuda(qsa::launch_sparse_attn(q, k_cells, k_scale_f16, v_cells, v_scale_f16, ncells, ids, nq, k, out,
                                             stream));
}

qsa_status qsa_block_summary(const int8_t *k_cells, const uint16_t *k_scale_f16, int ncells, int block_begin,
                             int block_end, float *kblk, int8_t *kblk_q8, uint16_t *kblk_scale_f16,
                             cudaStream_t stream) {
    if (ncells < 0 || block_begin < 0 || block_end < block_begin) return QSA_ERR_INVALID;
    if (kblk == nullptr && kblk_q8 == nullptr) return QSA_ERR_INVALID;
    if ((kblk_q8 == nullptr) != (kblk_scale_f16 == nullptr)) return QSA_ERR_INVALID;
    if (block_end == block_begin) return QSA_OK;
    if (static_cast<long long>(block_end) * 4 + 4 > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED;   // cell indices in int
    if (ncells > 0 && (k_cells == nullptr || k_scale_f16 == nullptr || !aligned16(k_cells) ||
                       (reinterpret_cast<uintptr_t>(k_scale_f16) & 1u) != 0))
        return QSA_ERR_INVALID;
    if ((kblk != nullptr && !aligned16(kblk)) || (kblk_q8 != nullptr && !aligned16(kblk_q8)) ||
        (kblk_scale_f16 != nullptr && (reinterpret_cast<uintptr_t>(kblk_scale_f16) & 1u) != 0))
        return QSA_ERR_INVALID;
    return from_cuda(qsa::launch_block_summary(k_cells, k_scale_f16, ncells, block_begin, block_end, kblk, kblk_q8,
                                               kblk_scale_f16, stream));
}

qsa_status qsa_get_device_error(uint32_t *code, cudaStream_t stream) {
    if (code == nullptr) return QSA_ERR_INVALID;
    *code = 0;
    uint32_t a = 0, b = 0;
    cudaError_t e = qsa::topk_error_read_clear(&a, stream);
    if (e == cudaSuccess) e = qsa::tc_error_read_clear(&b, stream);
    *code = a | (b << 8);
    return from_cuda(e);
}

qsa_status qsa_debug_inject(uint32_t faults, uint64_t wait_limit_ns) {
    if ((faults & ~3u) != 0u || wait_limit_ns == 0 || wait_limit_ns > 60000000000ull) return QSA_ERR_INVALID;
    qsa::g_inject.store(faults, std::memory_order_relaxed);
    qsa::g_wait_limit_ns.store(wait_limit_ns, std::memory_order_relaxed);
    return QSA_OK;
}

const char *qsa_status_string(qsa_status status) {
    switch (status) {
        case QSA_OK: return "QSA_OK";
        case QSA_ERR_INVALID: return "QSA_ERR_INVALID: invalid argument (nothing launched)";
        case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED: size beyond this library's limits";
        case QSA_ERR_CUDA: return "QSA_ERR_CUDA: a CUDA call or launch failed";
    }
    return "QSA_ERR_UNKNOWN";
}

}  // extern "C"

// host.cpp -- host-only parts of the C ABI: status strings, the block-mask builders of the
// TileLang block-sparse Flash-Attention guide (sections 3.1 / 3.2), its split-count rule
// (section 6.3), the device status word and the wait budget.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "bsattn.h"
#include "host_internal.h"

namespace {
std::atomic<unsigned long long> g_wait_budget_ns{2000000000ull};
thread_local std::string g_status_text;
}  // namespace

namespace bsattn {
unsigned long long wait_budget_ns() { return g_wait_budget_ns.load(); }
}  // namespace bsattn

extern "C" {

const char* bsattn_version(void) { return "bsattn 0.1 (sm_103a)"; }

const char* bsattn_status_string(int status) {
    if (status == BSATTN_OK) return "BSATTN_OK";
    std::string s;
    const struct { int bit; const char* name; } names[] = {
        {BSATTN_ERR_INVALID_ARG, "BSATTN_ERR_INVALID_ARG"},
        {BSATTN_ERR_UNSUPPORTED, "BSATTN_ERR_UNSUPPORTED"},
        {BSATTN_ERR_CUDA, "BSATTN_ERR_CUDA"},
        {BSATTN_ERR_TIMEOUT, "BSATTN_ERR_TIMEOUT"},
        {BSATTN_ERR_BAD_INDEX, "BSATTN_ERR_BAD_INDEX"},
    };
    int rest = status;
    for (const auto& n : names) {
        if (status & n.bit) {
            if (!s.empty()) s += "|";
            s += n.name;
            rest &= ~n.bit;
        }
    }
    if (rest) {
        if (!s.empty()) s += "|";
        s += "BSATTN_UNKNOWN(" + std::to_string(rest) + ")";
    }
    g_status_text = s;
    return g_status_text.c_str();
}

void bsattn_set_wait_budget_ns(unsigned long long ns) { g_wait_budget_ns.store(ns); }

int bsattn_get_device_status(void* workspace, void* stream) {
    if (!workspace) return BSATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return BSATTN_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return BSATTN_ERR_CUDA;
    }
    return word;
}

// ---------------------------------------------------------------- split-count rule

int bsattn_num_splits_heuristic(int total_mblocks, int num_SMs, int num_n_blocks,
                                int num_m_blocks, long long size_one_kv_head,
                                int is_causal_or_local, int max_splits) {
    if (num_SMs <= 0 || max_splits <= 0) return 1;
    if (static_cast<double>(total_mblocks) >= 0.8 * num_SMs) {
        const long long size_l2 = 50LL * 1024 * 1024;
        if (size_one_kv_head > size_l2 && num_m_blocks > 2 * num_SMs && !is_causal_or_local) {
            long long s = (size_one_kv_head + size_l2 - 1) / size_l2;
            return static_cast<int>(std::min<long long>(s, max_splits));
        }
        return 1;
    }
    if (num_n_blocks <= 4) return 1;
    const int limit = std::min(max_splits, std::min(num_SMs, num_n_blocks));
    std::vector<double> eff(static_cast<size_t>(std::max(limit, 0)));
    double best = 0.0;
    for (int s = 1; s <= limit; ++s) {
        double waves = static_cast<double>(total_mblocks) * s / num_SMs;
        eff[s - 1] = waves / std::ceil(waves);
        best = std::max(best, eff[s - 1]);
    }
    for (int s = 1; s <= limit; ++s)
        if (eff[s - 1] >= 0.85 * best) return s;
    return 1;
}

// ---------------------------------------------------------------- mask builders

static int check_scores(const float* scores, int B, int H, int nq, int nk, const uint8_t* out) {
    if (!scores || !out || B < 0 || H < 0 || nq < 0 || nk < 0) return BSATTN_ERR_INVALID_ARG;
    const size_t n = static_cast<size_t>(B) * H * nq * nk;
    for (size_t i = 0; i < n; ++i)
        if (std::isnan(scores[i])) return BSATTN_ERR_INVALID_ARG;
    return BSATTN_OK;
}

// Section 3.1 / 3.2 tail: last two query-block rows forced on, then the block lower triangle.
static void dense_last_and_tril(uint8_t* m, int nq, int nk, int dense_last, int tril) {
    if (dense_last)
        for (int r = std::max(0, nq - 2); r < nq; ++r) std::memset(m + size_t(r) * nk, 1, nk);
    if (tril)
        for (int r = 0; r < nq; ++r)
            for (int c = r + 1; c < nk; ++c) m[size_t(r) * nk + c] = 0;
}

int bsattn_mask_from_topk(const float* scores, int B, int H, int nq, int nk, int topk,
                          int use_dense_for_last_block, int apply_tril, uint8_t* mask_out) {
    int rc = check_scores(scores, B, H, nq, nk, mask_out);
    if (rc) return rc;
    if (topk < 0) return BSATTN_ERR_INVALID_ARG;
    const int keep = std::min(topk, nk);
    std::vector<int> order(static_cast<size_t>(nk));
    for (long long bh = 0; bh < static_cast<long long>(B) * H; ++bh) {
        uint8_t* m = mask_out + static_cast<size_t>(bh) * nq * nk;
        const float* x = scores + static_cast<size_t>(bh) * nq * nk;
        for (int r = 0; r < nq; ++r) {
            const float* row = x + size_t(r) * nk;
            uint8_t* mrow = m + size_t(r) * nk;
            std::memset(mrow, 0, nk);
            std::iota(order.begin(), order.end(), 0);
            // highest score first; equal scores: lower column first
            auto better = [row](int a, int b) {
                return row[a] > row[b] || (row[a] == row[b] && a < b);
            };
            std::partial_sort(order.begin(), order.begin() + keep, order.end(), better);
            for (int i = 0; i < keep; ++i) mrow[order[i]] = 1;
        }
        dense_last_and_tril(m, nq, nk, use_dense_for_last_block, apply_tril);
    }
    return BSATTN_OK;
}

int bsattn_mask_from_threshold(const float* scores, int B, int H, int nq, int nk,
                               float threshold, int use_dense_for_last_block, int apply_tril,
                               uint8_t* mask_out) {
    int rc = check_scores(scores, B, H, nq, nk, mask_out);
    if (rc) return rc;
    for (long long bh = 0; bh < static_cast<long long>(B) * H; ++bh) {
        uint8_t* m = mask_out + static_cast<size_t>(bh) * nq * nk;
        const float* x = scores + static_cast<size_t>(bh) * nq * nk;
        for (size_t i = 0; i < size_t(nq) * nk; ++i) m[i] = x[i] > threshold ? 1 : 0;
        dense_last_and_tril(m, nq, nk, use_dense_for_last_block, apply_tril);
    }
    return BSATTN_OK;
}

int bsattn_mask_from_cumulative_threshold(const float* attn_sum, int B, int H, int nq, int nk,
                                          double threshold, int causal, uint8_t* mask_out) {
    int rc = check_scores(attn_sum, B, H, nq, nk, mask_out);
    if (rc) return rc;
    std::vector<int> order;
    order.reserve(static_cast<size_t>(nk));
    for (long long r = 0; r < static_cast<long long>(B) * H * nq; ++r) {
        const int i = static_cast<int>(r % nq);
        const float* row = attn_sum + static_cast<size_t>(r) * nk;
        uint8_t* m = mask_out + static_cast<size_t>(r) * nk;
        std::memset(m, 0, nk);
        if (nk == 0) continue;
        double total = 0.0;
        for (int j = 0; j < nk; ++j) total += static_cast<double>(row[j]);
        m[0] = 1;                                   // the sink block
        if (causal && i < nk) m[i] = 1;             // the diagonal block
        order.clear();
        for (int j = 0; j < nk; ++j)
            if (!m[j]) order.push_back(j);
        std::stable_sort(order.begin(), order.end(), [row](int a, int b) { return row[a] > row[b]; });
        const double required = total * threshold;
        double acc = 0.0;
        for (int j : order) {
            if (acc >= required) break;
            m[j] = 1;
            acc += static_cast<double>(row[j]);
        }
    }
    return BSATTN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- TMA descriptor encoding

namespace bsattn {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

int encode_3d(CUtensorMap* map, const void* base, int elem_bytes_is_2_dtype_bf16,
              uint64_t dim0, uint64_t dim1, uint64_t dim2, uint64_t stride1_bytes,
              uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return BSATTN_ERR_CUDA;
    cuuint64_t dims[3] = {dim0, dim1, dim2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t es[3] = {1, 1, 1};
    CUtensorMapDataType dt = elem_bytes_is_2_dtype_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BSATTN_OK : BSATTN_ERR_INVALID_ARG;
}

int num_sms_of_current_device() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace bsattn

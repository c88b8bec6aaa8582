// prefill.cu -- block-sparse attention forward (prefill) for sm_103a.
//
// Method: TileLang block-sparse Flash-Attention guide, sections 4.1-4.7.  One CTA owns one
// (batch, head, 64-row query block).  It compacts its row of the block mask into a list of
// key blocks to visit (section 4.4: only set blocks are loaded and multiplied; causal rows
// stop at the diagonal), then streams those K/V tiles through shared memory with TMA and
// runs, per visited block,
//     S = Q K^T                      (tcgen05.mma, M=64 N=64 K=d, fp32 in TMEM)
//     token mask on the diagonal / sequence tail (section 4.5)
//     exp2 online softmax            (section 4.6, scale log2(e)/sqrt(d) folded in)
//     O += P V                       (tcgen05.mma, M=64 N=d K=64, P rounded to the input type)
// and finally O / l (section 4.7; a row with no visible key stores exactly 0).
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (warp w owns TMEM lanes 32w..32w+15,
// i.e. query rows 16w..16w+15 of the M=64 accumulator layout), warp 4 allocates TMEM and
// issues the MMAs, warp 5 issues the TMA loads.
//
// Differences from the page's kernel (made for this hardware):
//  * the mask row is compacted once per CTA, so masked K/V tiles are never addressed;
//  * S and P are double-buffered so Q K^T of block i+1 and P V of block i-1 overlap the
//    softmax of block i;
//  * O lives in TMEM and is rescaled only when a row maximum grows by more than 2^8
//    (exact: the final normaliser l is accumulated against the same reference maximum).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "host_internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr int kStages = 2;              // K/V ring depth
constexpr uint32_t kTmemCols = 256;     // S[0] cols 0-63, S[1] 64-127, O 128-(128+d)
constexpr uint32_t kOCol = 128;
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by > 2^8

struct PrefillParams {
    const uint8_t* mask;
    int* status;
    void* out;
    int B, H, Sq, Sk, nq, nk;
    int causal;
    float scale_log2;                   // log2(e) / sqrt(d)
    unsigned long long budget_ns;
};

template <int D>
struct Layout {
    static constexpr uint32_t kTile = (D / 64) * 8192;   // one [64 x D] 16-bit tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kTile;
    static constexpr uint32_t kV = kK + kStages * kTile;
    static constexpr uint32_t kP = kV + kStages * kTile;   // two [64 x 64] P tiles
    static constexpr uint32_t kBars = kP + 2 * 8192;
    static constexpr uint32_t kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 1;
    static constexpr uint32_t kMisc = kBars + 8 * kNumBars;
    static constexpr uint32_t kList = kMisc + 32;
    static uint32_t bytes(int nk) { return 1024 + kList + ((2 * nk + 15) & ~15); }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillParams p) {
    using L = Layout<D>;
    constexpr uint32_t kTile = L::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* sq = sm + L::kQ;
    uint8_t* sk = sm + L::kK;
    uint8_t* sv = sm + L::kV;
    uint8_t* sp = sm + L::kP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    uint64_t* q_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = kv_full + kStages;
    uint64_t* s_full = kv_empty + kStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_done = p_full + 2;
    uint64_t* fin = o_done + 2;
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L::kMisc);  // tmem, count, abort, epi
    uint16_t* list = reinterpret_cast<uint16_t*>(sm + L::kList);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[2]);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BH = p.B * p.H;
    const int qb = p.nq - 1 - static_cast<int>(blockIdx.x) / BH;   // heaviest rows first
    const int bh = static_cast<int>(blockIdx.x) % BH;
    const int past = p.Sk - p.Sq;                                   // bottom-right causal
    const uint64_t deadline = global_timer_ns() + p.budget_ns;

    int kb_end = p.nk;
    if (p.causal) {
        const long long last_key = static_cast<long long>(min(qb * 64 + 63, p.Sq - 1)) + past;
        const long long lim = last_key / 64 + 1;
        kb_end = last_key < 0 ? 0 : (lim < p.nk ? static_cast<int>(lim) : p.nk);
    }

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&s_full[j], 1);
            mbar_init(&p_full[j], 128);
            mbar_init(&o_done[j], 1);
        }
        mbar_init(fin, 1);
        misc[2] = 0;
        misc[3] = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // active-list compaction: key blocks kb < kb_end with mask != 0, ascending
        const uint8_t* mrow = p.mask + (static_cast<size_t>(bh) * p.nq + qb) * p.nk;
        int count = 0;
        for (int base = 0; base < kb_end; base += 32) {
            const int kb = base + lane;
            const bool on = kb < kb_end && mrow[kb] != 0;
            const uint32_t ballot = __ballot_sync(0xffffffffu, on);
            if (on) list[count + __popc(ballot & ((1u << lane) - 1u))] = static_cast<uint16_t>(kb);
            count += __popc(ballot);
        }
        if (lane == 0) misc[1] = count;
    }
    __syncthreads();
    const int n = static_cast<int>(misc[1]);

    using T = std::conditional_t<BF16, __nv_bfloat16, __half>;
    if (n == 0) {
        // no visible key anywhere in this query block: the rows are exactly zero
        const int rows = min(64, p.Sq - qb * 64);
        uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                              (static_cast<size_t>(bh) * p.Sq + qb * 64) * D);
        const int n16 = rows * D * 2 / 16;
        for (int i = tid; i < n16; i += kThreads) out[i] = make_uint4(0, 0, 0, 0);
        return;
    }

    if (warp == kMmaWarp) {
        tmem_alloc(&misc[0], kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = misc[0];

    if (warp == kTmaWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(q_full, kTile);
            for (int h = 0; h < D / 64; ++h) tma_load_3d(sq + h * 8192, &tm_q, q_full, h * 64, qb * 64, bh);
            int issued = 0;
            for (int j = 0; j < n; ++j) {
                const int st = j % kStages;
                if (j >= kStages &&
                    !wait_parity(&kv_empty[st], ((j / kStages) - 1) & 1, deadline, abort_flag, p.status))
                    break;
                const int kb = list[j];
                mbar_arrive_expect_tx(&kv_full[st], 2 * kTile);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(sk + st * kTile + h * 8192, &tm_k, &kv_full[st], h * 64, kb * 64, bh);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(sv + st * kTile + h * 8192, &tm_v, &kv_full[st], h * 64, kb * 64, bh);
                issued = j + 1;
            }
            if (*abort_flag) {
                // let copies already in flight land before this CTA's shared memory is released
                const uint64_t dl = global_timer_ns() + 200000000ull;
                wait_parity_drain(q_full, 0, dl);
                for (int j = max(0, issued - kStages); j < issued; ++j)
                    wait_parity_drain(&kv_full[j % kStages], (j / kStages) & 1, dl);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(64, 64, BF16, false);
            constexpr uint32_t idO = idesc_f16(64, D, BF16, true);
            auto issue_pv = [&](int j) -> bool {
                const int pb = j & 1;
                if (!wait_parity(&p_full[pb], (j >> 1) & 1, deadline, abort_flag, p.status)) return false;
                tc_fence_after();
                const int st = j % kStages;
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sdesc_sw128(smem_u32(sp + pb * 8192) + kk * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(smem_u32(sv + st * kTile) + kk * 2048, 8192, 1024);
                    mma_f16_ss(tbase + kOCol, a, b, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&o_done[pb]);
                mma_commit(&kv_empty[st]);
                return true;
            };
            bool ok = wait_parity(q_full, 0, deadline, abort_flag, p.status);
            for (int i = 0; ok && i < n; ++i) {
                const int st = i % kStages;
                if (!wait_parity(&kv_full[st], (i / kStages) & 1, deadline, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int sb = i & 1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    const uint64_t a = sdesc_sw128(smem_u32(sq) + off, 16, 1024);
                    const uint64_t b = sdesc_sw128(smem_u32(sk + st * kTile) + off, 16, 1024);
                    mma_f16_ss(tbase + sb * 64, a, b, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[sb]);
                if (i >= 1 && !issue_pv(i - 1)) ok = false;
            }
            if (ok) issue_pv(n - 1);
            // every MMA issued above must finish before TMEM is released
            mma_commit(fin);
            wait_parity_drain(fin, 0, global_timer_ns() + 200000000ull);
        }
    } else {
        // ---------------------------------------------------------------- softmax warps 0-3
        const int quad = lane >> 2, qi = lane & 3;
        const int lrowA = 16 * warp + quad;           // local rows of this thread
        const int lrowB = lrowA + 8;
        const int rowA = qb * 64 + lrowA, rowB = qb * 64 + lrowB;
        const uint32_t tl = tbase + (static_cast<uint32_t>(32 * warp) << 16);
        const float c = p.scale_log2;
        float m_used[2] = {-INFINITY, -INFINITY};
        float l[2] = {0.f, 0.f};
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int sb = i & 1;
            if (!warp_wait_parity(&s_full[sb], (i >> 1) & 1, deadline, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r[32];
            tmem_ld_16x256b_x8(tl + sb * 64, r);
            tmem_wait_ld();
            float s[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) s[e] = __uint_as_float(r[e]);

            const int key0 = static_cast<int>(list[i]) * 64;
            if (key0 + 63 >= p.Sk || (p.causal && key0 + 63 > qb * 64 + past)) {
#pragma unroll
                for (int rep = 0; rep < 8; ++rep)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = key0 + 8 * rep + 2 * qi + e;
                        const bool inA = key < p.Sk && (!p.causal || key <= rowA + past);
                        const bool inB = key < p.Sk && (!p.causal || key <= rowB + past);
                        if (!inA) s[4 * rep + e] = -INFINITY;
                        if (!inB) s[4 * rep + 2 + e] = -INFINITY;
                    }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int rep = 0; rep < 8; ++rep) {
                mx[0] = fmaxf(mx[0], fmaxf(s[4 * rep], s[4 * rep + 1]));
                mx[1] = fmaxf(mx[1], fmaxf(s[4 * rep + 2], s[4 * rep + 3]));
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            }
            float alpha[2], mc[2];
            bool rescale_o = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool grow = mx[h] * c > m_used[h] * c + kRescaleLog2;
                const float m_new = grow ? mx[h] : m_used[h];
                alpha[h] = grow ? ex2_approx((m_used[h] - m_new) * c) : 1.f;
                if (grow && m_used[h] != -INFINITY) rescale_o = true;
                m_used[h] = m_new;
                mc[h] = m_new == -INFINITY ? 0.f : m_new * c;
            }
            float sum[2] = {0.f, 0.f};
#pragma unroll
            for (int rep = 0; rep < 8; ++rep) {
                s[4 * rep + 0] = ex2_approx(fmaf(s[4 * rep + 0], c, -mc[0]));
                s[4 * rep + 1] = ex2_approx(fmaf(s[4 * rep + 1], c, -mc[0]));
                s[4 * rep + 2] = ex2_approx(fmaf(s[4 * rep + 2], c, -mc[1]));
                s[4 * rep + 3] = ex2_approx(fmaf(s[4 * rep + 3], c, -mc[1]));
                sum[0] += s[4 * rep + 0] + s[4 * rep + 1];
                sum[1] += s[4 * rep + 2] + s[4 * rep + 3];
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
                sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
                l[h] = l[h] * alpha[h] + sum[h];
            }
            if (__any_sync(0xffffffffu, rescale_o)) {
                // O must hold every product issued so far (P V of block i-1) before scaling
                if (!warp_wait_parity(&o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, deadline, abort_flag,
                                      p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[16];
                    tmem_ld_16x256b_x4(tl + kOCol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int rep = 0; rep < 4; ++rep) {
                        o[4 * rep + 0] = __float_as_uint(__uint_as_float(o[4 * rep + 0]) * alpha[0]);
                        o[4 * rep + 1] = __float_as_uint(__uint_as_float(o[4 * rep + 1]) * alpha[0]);
                        o[4 * rep + 2] = __float_as_uint(__uint_as_float(o[4 * rep + 2]) * alpha[1]);
                        o[4 * rep + 3] = __float_as_uint(__uint_as_float(o[4 * rep + 3]) * alpha[1]);
                    }
                    tmem_st_16x256b_x4(tl + kOCol + c0, o);
                }
                tmem_wait_st();
            }
            // P buffer (i & 1) is free once P V of block i-2 has completed
            if (i >= 2 && !warp_wait_parity(&o_done[i & 1], ((i - 2) >> 1) & 1, deadline, abort_flag,
                                            p.status)) {
                ok = false;
                break;
            }
            uint8_t* pbuf = sp + (i & 1) * 8192;
#pragma unroll
            for (int rep = 0; rep < 8; ++rep) {
                const int col = 8 * rep + 2 * qi;
                *reinterpret_cast<uint32_t*>(pbuf + sw128_offset(lrowA, col)) =
                    pack2<BF16>(s[4 * rep + 0], s[4 * rep + 1]);
                *reinterpret_cast<uint32_t*>(pbuf + sw128_offset(lrowB, col)) =
                    pack2<BF16>(s[4 * rep + 2], s[4 * rep + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[i & 1]);
        }
        if (ok && warp_wait_parity(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, deadline, abort_flag,
                                   p.status)) {
            tc_fence_after();
            const float inv[2] = {l[0] > 0.f ? 1.f / l[0] : 0.f, l[1] > 0.f ? 1.f / l[1] : 0.f};
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[16];
                tmem_ld_16x256b_x4(tl + kOCol + c0, o);
                tmem_wait_ld();
#pragma unroll
                for (int rep = 0; rep < 4; ++rep) {
                    const int col = c0 + 8 * rep + 2 * qi;
                    uint8_t* half = sq + (col >> 6) * 8192;   // Q tile reused as output staging
                    *reinterpret_cast<uint32_t*>(half + sw128_offset(lrowA, col & 63)) =
                        pack2<BF16>(__uint_as_float(o[4 * rep + 0]) * inv[0],
                                    __uint_as_float(o[4 * rep + 1]) * inv[0]);
                    *reinterpret_cast<uint32_t*>(half + sw128_offset(lrowB, col & 63)) =
                        pack2<BF16>(__uint_as_float(o[4 * rep + 2]) * inv[1],
                                    __uint_as_float(o[4 * rep + 3]) * inv[1]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) atomicAdd(&misc[3], 1u);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0 && misc[3] == 4 && !*abort_flag) {
        // rows >= Sq of the last query block fall outside the tensor map and are clipped
        for (int h = 0; h < D / 64; ++h) tma_store_3d(&tm_o, sq + h * 8192, h * 64, qb * 64, bh);
        tma_store_commit();
        tma_store_wait_read0();
    }
}

template <int D, bool BF16>
int launch(const void* q, const void* k, const void* v, void* out, const PrefillParams& prm,
           cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const uint64_t BH = static_cast<uint64_t>(prm.B) * prm.H;
    int rc = 0;
    rc |= encode_3d(&tq, q, BF16, D, prm.Sq, BH, D * 2ull, uint64_t(prm.Sq) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&tk, k, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&tv, v, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&to, out, BF16, D, prm.Sq, BH, D * 2ull, uint64_t(prm.Sq) * D * 2, 64, 64, 1, true);
    if (rc) return rc;
    // at most two CTAs per SM: each holds 256 of the SM's 512 TMEM columns
    uint32_t smem = Layout<D>::bytes(prm.nk);
    if (smem < 78u * 1024u) smem = 78u * 1024u;
    if (smem > 227u * 1024u) return BSATTN_ERR_UNSUPPORTED;
    auto kern = prefill_kernel<D, BF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    const uint64_t grid = BH * static_cast<uint64_t>(prm.nq);
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tq, tk, tv, to, prm);
    return cudaGetLastError() == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // namespace
}  // namespace bsattn

extern "C" size_t bsattn_prefill_workspace_size(int, int, int, int) { return 256; }

extern "C" int bsattn_prefill(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                              int is_causal, void* out, int B, int H, int Sq, int Sk, int d,
                              bsattn_dtype dtype, void* workspace, size_t workspace_bytes,
                              void* stream) {
    using namespace bsattn;
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return BSATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return BSATTN_ERR_UNSUPPORTED;
    if (dtype != BSATTN_F16 && dtype != BSATTN_BF16) return BSATTN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < bsattn_prefill_workspace_size(B, H, Sq, Sk))
        return BSATTN_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    if (BH == 0 || Sq == 0) return BSATTN_OK;
    if (!q || !k || !v || !out || !block_mask) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return BSATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Sk == 0) {
        // no keys at all: every row is exactly zero
        return cudaMemsetAsync(out, 0, static_cast<size_t>(BH) * Sq * d * 2, st) == cudaSuccess
                   ? BSATTN_OK
                   : BSATTN_ERR_CUDA;
    }
    const int nq = (Sq + 63) / 64, nk = (Sk + 63) / 64;
    if (nk > 65535 || BH * nq > 0x7fffffffLL || BH > 0x7fffffffLL) return BSATTN_ERR_UNSUPPORTED;
    PrefillParams prm{};
    prm.mask = block_mask;
    prm.status = static_cast<int*>(workspace);
    prm.out = out;
    prm.B = B;
    prm.H = H;
    prm.Sq = Sq;
    prm.Sk = Sk;
    prm.nq = nq;
    prm.nk = nk;
    prm.causal = is_causal ? 1 : 0;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    prm.budget_ns = wait_budget_ns();
    const bool bf16 = dtype == BSATTN_BF16;
    if (d == 64) return bf16 ? launch<64, true>(q, k, v, out, prm, st) : launch<64, false>(q, k, v, out, prm, st);
    return bf16 ? launch<128, true>(q, k, v, out, prm, st) : launch<128, false>(q, k, v, out, prm, st);
}

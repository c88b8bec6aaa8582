// decode.cu -- GQA variable-length sparse decode for sm_103a.
//
// Method: TileLang block-sparse Flash-Attention guide, sections 6.1-6.3.  One query token per
// sequence; the G = Hq/Hkv query heads of kv head g share that head's selected 64-token
// blocks.  The block_indices slots of each (b, g) are cut into num_splits contiguous slices
// (section 6.2: the first len % num_splits slices get one extra slot); each slice is one CTA,
// which writes a partial output and its log-sum-exp, and the partials are merged with
// weights exp2(lse - max lse) (section 6.1's merge stage).
//
// This path is bound by HBM bandwidth (each K/V byte is used once, by G heads), so it is
// built around bytes in flight: a producer warp streams the K and V tiles of the slice with
// TMA (128-byte swizzle) into three stages of half a block (K and V of 32 tokens), four CTAs
// per SM.  Each stage is read by a pair of consumer warps, 16 tokens each.  The [G x 64 x d]
// products are small, so they run on warp-level mma.sync, transposed so that the G <= 8 query
// heads are the n = 8 side of the m16n8k16 shape, straight out of the swizzled tiles.  The
// merge is fused: the last CTA of a (b, g) group to finish (atomic ticket) combines the
// partials and resets the ticket, so a call is a single kernel launch.
//
// Differences from the page's kernel: every block that crosses cache_seqlens is masked token
// by token (the page masks only the first slot and relies on descending order), so the
// result does not depend on the order of the indices; indices at or past the sequence end
// are skipped and reported instead of read.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "host_internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);   // + one producer warp
constexpr int kStages = 3;              // half-block (32-token) K+V stages
constexpr size_t kHeaderBytes = 256;                   // status word + padding

// Where a CTA's key blocks come from (all give the same token set semantics):
//   kIndices  block_indices [B, Hkv, max_sel] int32, contiguous cache [B, Smax, Hkv, d]
//   kMask     block_mask [B, Hkv, max_sel] uint8 (slot j <-> block j), contiguous cache
//   kPaged    block_indices as kIndices; K/V in pages [num_pages, page_size, Hkv, d] reached
//             through block_table [B, max_pages] (guide section 7)
enum DecodeMode { kIndices = 0, kMask = 1, kPaged = 2 };

struct DecodeParams {
    const void* q;
    const int32_t* seqlens;
    const int32_t* indices;
    const uint8_t* mask;
    const int32_t* block_table;
    int mode;
    int page_size, max_pages, num_pages;
    void* out;
    int* status;
    int* tickets;       // [B * Hkv]
    float* lse_part;    // [B, Hq, ns]
    float* o_part;      // [B, Hq, ns, d]
    int B, Hq, Hkv, Smax, max_sel, num_splits;
    float scale_log2;   // log2(e) / sqrt(d)
    unsigned long long budget_ns;
};

template <int D>
struct DLayout {
    // a stage holds 32 tokens (half a block) of K and of V: per 64-column d-half one TMA box
    // of [32 x 64] 16-bit values, 128-byte swizzled
    static constexpr uint32_t kBox = 32 * 128;                // one [32 x 64] box
    static constexpr uint32_t kHalfK = (D / 64) * kBox;       // K (or V) of one stage
    static constexpr uint32_t kStage = 2 * kHalfK;            // K then V
    // per-warp partials (m[8], l[8], O[8 x D]) reuse the stages once they are drained
    static constexpr uint32_t kMerge = 0;
    static constexpr int kMergeRow = D + 8;                  // padded: 2-way bank spread
    static constexpr uint32_t kMergeWarp = (16 + 8 * kMergeRow) * 4;
    static constexpr uint32_t kBars = kStages * kStage;
    // full[stage][warp pair], empty[stage], listed
    static constexpr uint32_t kMisc = kBars + 8 * (3 * kStages + 1);
    static constexpr uint32_t kList = kMisc + 16;
    // two int lists per slot: logical block (sequence-end masking) and TMA row of its tile
    static uint32_t bytes(int max_slots) { return 1024 + kList + 2 * ((4 * max_slots + 15) & ~15); }
    static_assert(kConsumerWarps * kMergeWarp <= kStages * kStage, "merge scratch must fit");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit values held one 32-bit pair per lane (lane t: row
// t/4, columns 2 (t%4), 2 (t%4) + 1), returned in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

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

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t raw) {
    if constexpr (BF16) {
        return __bfloat162float(__ushort_as_bfloat16(raw));
    } else {
        return __half2float(__ushort_as_half(raw));
    }
}

// Four consecutive outputs rounded to the 16-bit type in one 8-byte store.
template <bool BF16>
__device__ __forceinline__ void store4(void* dst, const float4 v) {
    uint2 w;
    w.x = pack2<BF16>(v.x, v.y);
    w.y = pack2<BF16>(v.z, v.w);
    *reinterpret_cast<uint2*>(dst) = w;
}

// Address (shared-space) of element (row, col) of a swizzled [rows x D] tile stored as D/64
// column halves of [rows x 64].
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int half_stride, int row, int col) {
    return base + (col >> 6) * half_stride + sw128_offset(row, col & 63);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 4)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p) {
    using L = DLayout<D>;
    using T = std::conditional_t<BF16, __nv_bfloat16, __half>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::kBars);
    // Half-block hs goes to stage hs % 3 and is read by warp pair hs % 2.  Each pair waits on a
    // full barrier of its own per stage (used every 6th half-block, always by that pair, in
    // order): with one barrier per stage, pair 0 could wait for half-block 6 while half-block 3
    // (pair 1) was still landing in the same stage, and parity cannot tell those phases apart.
    uint64_t* empty = full + 2 * kStages;
    uint64_t* listed = empty + kStages;          // the producer has compacted the slice
    int* misc = reinterpret_cast<int*>(sm + L::kMisc);   // [0] count, [1] abort, [2] last
    int* list = reinterpret_cast<int*>(sm + L::kList);
    const int slot_cap = (p.max_sel + p.num_splits - 1) / p.num_splits;
    int* rows = list + ((4 * slot_cap + 15) & ~15) / 4;
    float* merge = reinterpret_cast<float*>(sm + L::kMerge);
    volatile int* abort_flag = &misc[1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = p.Hq / p.Hkv;
    const int seqlen = p.seqlens[b];
    const int nb_valid = (seqlen + 63) / 64;
    const uint64_t deadline = global_timer_ns() + p.budget_ns;

    // this split's slots (section 6.2 of the guide)
    const int bps = p.max_sel / p.num_splits, rem = p.max_sel % p.num_splits;
    const int slot0 = bps * split + min(split, rem);
    const int nslot = bps + (split < rem ? 1 : 0);

    if (tid == 0) {
        for (int s = 0; s < 2 * kStages; ++s) mbar_init(&full[s], 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&empty[s], kConsumerWarps / 2);   // the two warps on this half-block
        }
        mbar_init(listed, 1);
        misc[1] = 0;
        misc[2] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // consumer state: O^T tile fragments (row = d, column = query head) and, for the two heads
    // 2(lane%4) and 2(lane%4)+1 of this lane, the running maximum and sum
    float o[D / 16][4];
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool ok = true;
    if (warp == kConsumerWarps) {
        // producer: compact the slice, keeping blocks 0 <= t < nb_valid with the TMA row of
        // each, and start streaming at once (the consumers load q meanwhile)
        const size_t sel_off = (static_cast<size_t>(b) * p.Hkv + g) * p.max_sel + slot0;
        int count = 0;
        bool bad = false;
        for (int base = 0; base < nslot; base += 32) {
            const int j = base + lane;
            int t = -1;
            if (j < nslot) {
                if (p.mode == kMask) {
                    t = p.mask[sel_off + j] ? slot0 + j : -1;   // mask slots past the end: ignored
                    if (t >= nb_valid) t = -1;
                } else {
                    t = p.indices[sel_off + j];
                }
            }
            bool on = t >= 0 && t < nb_valid;
            bad |= t >= nb_valid;                               // an index past the sequence end
            int row = 0;
            if (on) {
                if (p.mode == kPaged) {
                    const long long pos = static_cast<long long>(t) * 64;
                    const long long lp = pos / p.page_size;
                    const int page = lp < p.max_pages ? p.block_table[static_cast<size_t>(b) * p.max_pages + lp] : -1;
                    if (page < 0 || page >= p.num_pages) {
                        on = false;                             // unmapped page: skip, flag
                        bad = true;
                    } else {
                        row = page * p.page_size + static_cast<int>(pos - lp * p.page_size);
                    }
                } else {
                    row = b * p.Smax + t * 64;
                }
            }
            const uint32_t ballot = __ballot_sync(0xffffffffu, on);
            if (on) {
                const int pos = count + __popc(ballot & ((1u << lane) - 1u));
                list[pos] = t;
                rows[pos] = row;
            }
            count += __popc(ballot);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, BSATTN_ERR_BAD_INDEX);
        __syncwarp();
        if (lane == 0) {
            misc[0] = count;
            mbar_arrive(listed);                 // release: list, rows and count are visible
        }
        const int n = count;
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int issued = 0;
            for (int hs = 0; hs < 2 * n; ++hs) {
                // half-stage hs: tokens [32 (hs % 2), +32) of listed block hs / 2
                const int st = hs % kStages;
                if (hs >= kStages &&
                    !wait_parity(&empty[st], ((hs / kStages) - 1) & 1, deadline, abort_flag, p.status))
                    break;
                const int row = rows[hs >> 1] + 32 * (hs & 1);
                uint8_t* stage = sm + st * L::kStage;
                uint64_t* fb = &full[2 * st + (hs & 1)];
                mbar_arrive_expect_tx(fb, L::kStage);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(stage + h * L::kBox, &tm_k, fb, h * 64, g, row);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d(stage + L::kHalfK + h * L::kBox, &tm_v, fb, h * 64, g, row);
                issued = hs + 1;
            }
            if (*abort_flag) {
                const uint64_t dl = global_timer_ns() + 200000000ull;
                for (int j = max(0, issued - kStages); j < issued; ++j)
                    wait_parity_drain(&full[2 * (j % kStages) + (j & 1)], (j / (2 * kStages)) & 1, dl);
            }
        }
    } else {
        // ------------------------------------------------------------ consumer warps 0-3
        // Transposed products, so that the G <= 8 query heads are the n = 8 side of each
        // m16n8k16 MMA and no accumulator row is padding:
        //   S^T [16 tokens x 8 heads] = K [16 tokens x d] . Q^T [d x 8 heads]
        //   O^T [d x 8 heads]        += V^T [d x 16 tokens] . P^T [16 tokens x 8 heads]
        // Each warp takes 16 tokens of every block.  P^T reaches the B-operand layout of the
        // second product through an in-register 8x8 transpose (movmatrix).
        if (!warp_wait_parity(listed, 0, deadline, abort_flag, p.status)) ok = false;
        const int n = ok ? misc[0] : 0;
        const float c = p.scale_log2;
        // warps 0-1 take the first 32 tokens of every block, warps 2-3 the last 32; a warp's
        // 16 tokens start at row tok0 of its half-block stage
        const int half = warp >> 1;
        const int tok0 = 16 * (warp & 1);
        // Q^T fragments (B operand): lane holds Q[head lane/4][d = 16 kk + 2 (lane%4) + {0,1}]
        // and the same 8 columns further; heads >= G are zero
        uint32_t qb[D / 16][2];
        {
            const T* qg = reinterpret_cast<const T*>(p.q) + (static_cast<size_t>(b) * p.Hq + g * G) * D;
            const int hq = lane >> 2;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int col = kk * 16 + 2 * (lane & 3);
                qb[kk][0] = hq < G ? *reinterpret_cast<const uint32_t*>(qg + hq * D + col) : 0u;
                qb[kk][1] = hq < G ? *reinterpret_cast<const uint32_t*>(qg + hq * D + col + 8) : 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        for (int j = 0; j < n; ++j) {
            const int hs = 2 * j + half;
            const int st = hs % kStages;
            if (!warp_wait_parity(&full[2 * st + half], (hs / (2 * kStages)) & 1, deadline, abort_flag,
                                  p.status)) {
                ok = false;
                break;
            }
            const uint32_t kbase = smem_u32(sm + st * L::kStage);
            const uint32_t vbase = kbase + L::kHalfK;
            const int key0 = list[j] * 64 + 32 * half + tok0;
            if (key0 + 16 > seqlen) {
                // tokens at or past the sequence end may hold anything: zero their V rows so
                // that P = 0 cannot meet a NaN
                for (int e = lane; e < 16 * (D / 8); e += 32) {
                    const int r = e / (D / 8), col = (e % (D / 8)) * 8;
                    if (key0 + r >= seqlen)
                        *reinterpret_cast<uint4*>(sm + st * L::kStage + L::kHalfK + (col >> 6) * L::kBox +
                                                  sw128_offset(tok0 + r, col & 63)) =
                            make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // S^T: A = this warp's 16 K rows (x4: rows 0-7 | 8-15 of d 0-7, then of d 8-15)
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int mat = lane >> 3;
                const int tok = tok0 + (mat & 1) * 8 + (lane & 7);
                const int col = kk * 16 + (mat >> 1) * 8;
                uint32_t a[4];
                ldsm_x4(tile_addr<D>(kbase, L::kBox, tok, col), a[0], a[1], a[2], a[3]);
                mma16816<BF16>(sc, a, qb[kk][0], qb[kk][1]);
            }
            // lane holds tokens t = lane/4 (sc[0..1]) and t + 8 (sc[2..3]), heads 2 (lane%4) + {0,1}
            const int ta = key0 + (lane >> 2), tb = ta + 8;
            float x[4];
            x[0] = ta < seqlen ? sc[0] * c : -INFINITY;
            x[1] = ta < seqlen ? sc[1] * c : -INFINITY;
            x[2] = tb < seqlen ? sc[2] * c : -INFINITY;
            x[3] = tb < seqlen ? sc[3] * c : -INFINITY;
            float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
            }
            float alpha[2], mref[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float m_new = fmaxf(m[h], mx[h]);
                mref[h] = m_new == -INFINITY ? 0.f : m_new;
                alpha[h] = ex2_approx(m[h] - mref[h]);
                m[h] = m_new;
            }
            const float p0 = ex2_approx(x[0] - mref[0]), p1 = ex2_approx(x[1] - mref[1]);
            const float p2 = ex2_approx(x[2] - mref[0]), p3 = ex2_approx(x[3] - mref[1]);
            float sum[2] = {p0 + p2, p1 + p3};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 4);
                sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 8);
                sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 16);
                l[h] = l[h] * alpha[h] + sum[h];
            }
            // P^T as the B operand: the two 8x8 (token x head) halves, transposed in registers
            const uint32_t pb0 = movmatrix_trans(pack2<BF16>(p0, p1));
            const uint32_t pb1 = movmatrix_trans(pack2<BF16>(p2, p3));
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][0] *= alpha[0];
                o[mt][1] *= alpha[1];
                o[mt][2] *= alpha[0];
                o[mt][3] *= alpha[1];
            }
            // O^T += V^T P^T: A = V^T from the V tile (token rows) through transposing loads
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int mat = lane >> 3;
                const int tok = tok0 + (mat >> 1) * 8 + (lane & 7);
                const int col = mt * 16 + (mat & 1) * 8;
                uint32_t a[4];
                ldsm_x4_t(tile_addr<D>(vbase, L::kBox, tok, col), a[0], a[1], a[2], a[3]);
                mma16816<BF16>(o[mt], a, pb0, pb1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
    }
    // every warp is done with the K/V stages (and the producer has drained) before they
    // become merge scratch
    __syncthreads();
    if (warp < kConsumerWarps) {
        // per-warp partial -> shared memory: [m of 8 heads | l of 8 heads | O rows of 8 heads]
        float* mw = merge + warp * (L::kMergeWarp / 4);
        const int h0 = 2 * (lane & 3);
        if (lane < 4) {
            mw[h0] = ok ? m[0] : -INFINITY;
            mw[h0 + 1] = ok ? m[1] : -INFINITY;
            mw[8 + h0] = ok ? l[0] : 0.f;
            mw[8 + h0 + 1] = ok ? l[1] : 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = mt * 16 + (lane >> 2);
            mw[16 + h0 * L::kMergeRow + d0] = o[mt][0];
            mw[16 + (h0 + 1) * L::kMergeRow + d0] = o[mt][1];
            mw[16 + h0 * L::kMergeRow + d0 + 8] = o[mt][2];
            mw[16 + (h0 + 1) * L::kMergeRow + d0 + 8] = o[mt][3];
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- combine warps, emit
    // G rows x D columns in groups of four columns, spread over all threads
    const bool aborted = *abort_flag != 0;
    const size_t row_base = static_cast<size_t>(b) * p.Hq + g * G;   // first query head row
    constexpr int kW = L::kMergeWarp / 4;                             // floats per warp record
    for (int e = tid; e < G * (D / 4); e += kThreads) {
        const int row = e / (D / 4), c4 = e % (D / 4);
        float mk[kConsumerWarps];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            mk[w] = merge[w * kW + row];
            M = fmaxf(M, mk[w]);
        }
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float wt = ex2_approx(mk[w] - M);
                const float4 ov = *reinterpret_cast<const float4*>(merge + w * kW + 16 + row * L::kMergeRow + 4 * c4);
                num.x += wt * ov.x;
                num.y += wt * ov.y;
                num.z += wt * ov.z;
                num.w += wt * ov.w;
                den += wt * merge[w * kW + 8 + row];
            }
        }
        const float4 val = den > 0.f ? make_float4(num.x / den, num.y / den, num.z / den, num.w / den)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.num_splits == 1) {
            if (!aborted) store4<BF16>(reinterpret_cast<T*>(p.out) + (row_base + row) * D + 4 * c4, val);
        } else {
            const size_t pr = (row_base + row) * p.num_splits + split;
            *reinterpret_cast<float4*>(p.o_part + pr * D + 4 * c4) = val;
            if (c4 == 0) p.lse_part[pr] = den > 0.f ? M + log2f(den) : -INFINITY;
        }
    }
    if (p.num_splits == 1) return;

    // the last CTA of this (b, g) to finish merges the num_splits partials; one fence by the
    // ticket holder after the barrier publishes every thread's partial writes
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int ticket = atomicAdd(&p.tickets[b * p.Hkv + g], 1);
        misc[2] = ticket == p.num_splits - 1;
        if (misc[2]) __threadfence();
    }
    __syncthreads();
    if (!misc[2]) return;
    // partials are read through L2 only (ld.global.cg): an SM's L1 may hold stale copies from
    // an earlier call.  Up to eight splits at a time, every LSE value and partial row is loaded
    // before any is used, so one L2 round trip serves them all; an online rescale joins chunks.
    for (int e = tid; e < G * (D / 4); e += kThreads) {
        const int row = e / (D / 4), c4 = e % (D / 4);
        const size_t r0 = (row_base + row) * p.num_splits;
        const float* lse = p.lse_part + r0;
        const float4* op = reinterpret_cast<const float4*>(p.o_part + r0 * D) + c4;
        float M = -INFINITY, den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < p.num_splits; s0 += 8) {
            float lv[8];
            float4 ov[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const bool in = s0 + k < p.num_splits;
                lv[k] = in ? __ldcg(lse + s0 + k) : -INFINITY;
                ov[k] = in ? __ldcg(op + static_cast<size_t>(s0 + k) * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float Mc = M;
#pragma unroll
            for (int k = 0; k < 8; ++k) Mc = fmaxf(Mc, lv[k]);
            if (Mc == -INFINITY) continue;
            const float r = ex2_approx(M - Mc);          // 0 while M is still -inf
            num.x *= r;
            num.y *= r;
            num.z *= r;
            num.w *= r;
            den *= r;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float wt = ex2_approx(lv[k] - Mc);
                num.x += wt * ov[k].x;
                num.y += wt * ov[k].y;
                num.z += wt * ov[k].z;
                num.w += wt * ov[k].w;
                den += wt;
            }
            M = Mc;
        }
        const float4 val = den > 0.f ? make_float4(num.x / den, num.y / den, num.z / den, num.w / den)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        store4<BF16>(reinterpret_cast<T*>(p.out) + (row_base + row) * D + 4 * c4, val);
    }
    if (tid == 0) p.tickets[b * p.Hkv + g] = 0;   // ready for the next call
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t tickets, lse, opart, total;
};

WsLayout ws_layout(int B, int Hq, int Hkv, int d, int ns) {
    WsLayout w{};
    w.tickets = kHeaderBytes;
    w.lse = w.tickets + align256(sizeof(int) * static_cast<size_t>(B) * Hkv);
    w.opart = w.lse + align256(sizeof(float) * static_cast<size_t>(B) * Hq * ns);
    w.total = w.opart + align256(sizeof(float) * static_cast<size_t>(B) * Hq * ns * d);
    return w;
}

template <int D, bool BF16>
int launch(const void* k, const void* v, const DecodeParams& prm, cudaStream_t stream) {
    CUtensorMap tk, tv;
    // rows of the K/V tensors as TMA sees them: B * Smax tokens, or num_pages * page_size
    const uint64_t nrows = prm.mode == kPaged ? static_cast<uint64_t>(prm.num_pages) * prm.page_size
                                              : static_cast<uint64_t>(prm.B) * prm.Smax;
    int rc = 0;
    rc |= encode_3d(&tk, k, BF16, D, prm.Hkv, nrows, D * 2ull, uint64_t(prm.Hkv) * D * 2, 64, 1, 32, true);
    rc |= encode_3d(&tv, v, BF16, D, prm.Hkv, nrows, D * 2ull, uint64_t(prm.Hkv) * D * 2, 64, 1, 32, true);
    if (rc) return rc;
    const int slots_per_split = (prm.max_sel + prm.num_splits - 1) / prm.num_splits;
    const uint32_t smem = DLayout<D>::bytes(slots_per_split);
    if (smem > 227u * 1024u) return BSATTN_ERR_UNSUPPORTED;
    auto kern = decode_kernel<D, BF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    dim3 grid(prm.num_splits, prm.Hkv, prm.B);
    kern<<<grid, kThreads, smem, stream>>>(tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // namespace
}  // namespace bsattn

namespace bsattn {
namespace {

// Resident decode CTAs per SM for head dim d (smem sized for a slice of max_sel slots).
int decode_ctas_per_sm(int d, int max_sel) {
    int occ = 0;
    cudaError_t e;
    if (d == 64) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<64, true>, kThreads,
                                                          DLayout<64>::bytes(max_sel));
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<128, true>, kThreads,
                                                          DLayout<128>::bytes(max_sel));
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return occ;
}

}  // namespace
}  // namespace bsattn

extern "C" int bsattn_decode_default_splits(int B, int Hkv, int max_sel, int d, int num_sms) {
    if (num_sms <= 0) num_sms = bsattn::num_sms_of_current_device();
    if (num_sms <= 0) num_sms = 148;
    const long long groups = static_cast<long long>(B) * Hkv;
    if (groups <= 0 || max_sel <= 0) return 1;
    int per_sm = (d == 64 || d == 128) ? bsattn::decode_ctas_per_sm(d, max_sel) : 0;
    if (per_sm <= 0) per_sm = 4;
    // at most as many splits as fill one wave of resident CTAs (every CTA streams its slice
    // from the start, and no second, mostly empty wave follows); then the fewest splits whose
    // largest slice is as short: 64 slots over 9 splits leave slices of 8 and 7, over 8 all 8
    long long s = static_cast<long long>(per_sm) * num_sms / groups;
    if (s > max_sel) s = max_sel;
    if (s > 64) s = 64;
    if (s < 1) s = 1;
    const long long longest = (max_sel + s - 1) / s;
    s = (max_sel + longest - 1) / longest;
    return static_cast<int>(s);
}

extern "C" size_t bsattn_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_sel,
                                               int num_splits) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return bsattn::kHeaderBytes;
    int ns = num_splits > 0 ? num_splits : bsattn_decode_default_splits(B, Hkv, max_sel, d, 0);
    return bsattn::ws_layout(B, Hq, Hkv, d, ns).total;
}

namespace bsattn {
namespace {

// Shared body of the decode entry points: argument checks, split count, workspace carving.
int decode_impl(DecodeParams prm, const void* k, const void* v, int num_splits, int d,
                bsattn_dtype dtype, void* workspace, size_t workspace_bytes, cudaStream_t st) {
    const int B = prm.B, Hq = prm.Hq, Hkv = prm.Hkv, max_sel = prm.max_sel;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_sel < 0 || num_splits < 0) return BSATTN_ERR_INVALID_ARG;
    if (Hq % Hkv) return BSATTN_ERR_INVALID_ARG;
    if (Hq / Hkv > 8) return BSATTN_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return BSATTN_ERR_UNSUPPORTED;
    if (dtype != BSATTN_F16 && dtype != BSATTN_BF16) return BSATTN_ERR_UNSUPPORTED;
    if (!workspace) return BSATTN_ERR_INVALID_ARG;
    if (B == 0) return BSATTN_OK;
    const bool sel_ok = prm.mode == kMask ? prm.mask != nullptr : prm.indices != nullptr;
    if (!prm.q || !k || !v || !prm.out || !prm.seqlens || (!sel_ok && max_sel > 0) ||
        (prm.mode == kPaged && !prm.block_table))
        return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(prm.q) || !aligned16(k) || !aligned16(v) || !aligned16(prm.out)) return BSATTN_ERR_INVALID_ARG;
    if (B > 65535 || Hkv > 65535) return BSATTN_ERR_UNSUPPORTED;
    if (prm.mode == kPaged) {
        if (prm.page_size <= 0 || prm.page_size % 64 || prm.num_pages <= 0 || prm.max_pages <= 0)
            return prm.page_size > 0 && prm.page_size % 64 ? BSATTN_ERR_UNSUPPORTED : BSATTN_ERR_INVALID_ARG;
        if (static_cast<long long>(prm.num_pages) * prm.page_size > 0x7fffffffLL) return BSATTN_ERR_UNSUPPORTED;
    } else {
        if (prm.Smax < 0) return BSATTN_ERR_INVALID_ARG;
        if (static_cast<long long>(B) * prm.Smax > 0x7fffffffLL) return BSATTN_ERR_UNSUPPORTED;
    }
    int ns = num_splits > 0 ? num_splits : bsattn_decode_default_splits(B, Hkv, max_sel, d, 0);
    if (max_sel == 0) ns = 1;
    if (ns > max_sel && max_sel > 0) ns = max_sel;
    const WsLayout w = ws_layout(B, Hq, Hkv, d, ns);
    if (workspace_bytes < w.total) return BSATTN_ERR_INVALID_ARG;
    if (max_sel == 0 || (prm.mode != kPaged && prm.Smax == 0)) {
        return cudaMemsetAsync(prm.out, 0, static_cast<size_t>(B) * Hq * d * 2, st) == cudaSuccess
                   ? BSATTN_OK
                   : BSATTN_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    prm.status = reinterpret_cast<int*>(ws);
    prm.tickets = reinterpret_cast<int*>(ws + w.tickets);
    prm.lse_part = reinterpret_cast<float*>(ws + w.lse);
    prm.o_part = reinterpret_cast<float*>(ws + w.opart);
    prm.num_splits = ns;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    prm.budget_ns = wait_budget_ns();
    const bool bf16 = dtype == BSATTN_BF16;
    if (d == 64) return bf16 ? launch<64, true>(k, v, prm, st) : launch<64, false>(k, v, prm, st);
    return bf16 ? launch<128, true>(k, v, prm, st) : launch<128, false>(k, v, prm, st);
}

}  // namespace
}  // namespace bsattn

extern "C" int bsattn_decode_varlen(const void* q, const void* k, const void* v,
                                    const int32_t* cache_seqlens, const int32_t* block_indices,
                                    int num_splits, void* out, int B, int Hq, int Hkv, int Smax,
                                    int d, int max_sel, bsattn_dtype dtype, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    bsattn::DecodeParams prm{};
    prm.q = q;
    prm.seqlens = cache_seqlens;
    prm.indices = block_indices;
    prm.mode = bsattn::kIndices;
    prm.out = out;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Smax = Smax;
    prm.max_sel = max_sel;
    return bsattn::decode_impl(prm, k, v, num_splits, d, dtype, workspace, workspace_bytes,
                               static_cast<cudaStream_t>(stream));
}

extern "C" int bsattn_decode_varlen_mask(const void* q, const void* k, const void* v,
                                         const int32_t* cache_seqlens, const uint8_t* block_mask,
                                         int num_splits, void* out, int B, int Hq, int Hkv,
                                         int Smax, int d, int num_blocks, bsattn_dtype dtype,
                                         void* workspace, size_t workspace_bytes, void* stream) {
    bsattn::DecodeParams prm{};
    prm.q = q;
    prm.seqlens = cache_seqlens;
    prm.mask = block_mask;
    prm.mode = bsattn::kMask;
    prm.out = out;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Smax = Smax;
    prm.max_sel = num_blocks;
    return bsattn::decode_impl(prm, k, v, num_splits, d, dtype, workspace, workspace_bytes,
                               static_cast<cudaStream_t>(stream));
}

extern "C" int bsattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* cache_seqlens, const int32_t* block_indices,
                                   const int32_t* block_table, int num_splits, void* out, int B,
                                   int Hq, int Hkv, int num_pages, int page_size,
                                   int max_pages_per_seq, int d, int max_sel, bsattn_dtype dtype,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    bsattn::DecodeParams prm{};
    prm.q = q;
    prm.seqlens = cache_seqlens;
    prm.indices = block_indices;
    prm.block_table = block_table;
    prm.mode = bsattn::kPaged;
    prm.page_size = page_size;
    prm.max_pages = max_pages_per_seq;
    prm.num_pages = num_pages;
    prm.out = out;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Smax = 0;
    prm.max_sel = max_sel;
    return bsattn::decode_impl(prm, k_pages, v_pages, num_splits, d, dtype, workspace,
                               workspace_bytes, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- allocation-free variant
//
// Some callers cannot allocate device memory at the point where they attend: code running
// inside a custom allocator or memory pool (which must not re-enter it), a runtime that
// pre-plans every buffer and forbids allocation after start-up, or a host integration
// that only ever hands over pointers to buffers it already owns.  For them the scratch the
// decode needs (split partials, LSE values, merge tickets) lives in the fixed array below,
// part of the library's own image: every GPU that loads the library holds it until exit.

namespace bsattn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side symbol is only
// a stand-in, so the address is looked up once per device with that device current.
int noalloc_scratch(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BSATTN_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return BSATTN_OK;
}

}  // namespace
}  // namespace bsattn

extern "C" int bsattn_decode_varlen_noalloc(const void* q, const void* k, const void* v,
                                            const int32_t* cache_seqlens,
                                            const int32_t* block_indices, int num_splits,
                                            void* out, int B, int Hq, int Hkv, int Smax, int d,
                                            int max_sel, bsattn_dtype dtype, void* stream) {
    using namespace bsattn;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_sel < 0 || num_splits < 0) return BSATTN_ERR_INVALID_ARG;
    int ns = num_splits > 0 ? num_splits : bsattn_decode_default_splits(B, Hkv, max_sel, d, 0);
    if (max_sel == 0) ns = 1;
    if (ns > max_sel && max_sel > 0) ns = max_sel;
    const size_t need = bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, ns);
    if (need > kNoAllocScratchBytes) return BSATTN_ERR_UNSUPPORTED;   // shape beyond the array
    // the array's address is per device: the stream must run on the device it was looked up on
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (sdev != cur) return BSATTN_ERR_INVALID_ARG;
    void* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    // the array keeps the previous call's contents: the status word and the merge tickets
    // must start at zero
    const WsLayout w = ws_layout(B > 0 ? B : 1, Hq, Hkv, d, ns);
    if (cudaMemsetAsync(scratch, 0, w.lse, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    return bsattn_decode_varlen(q, k, v, cache_seqlens, block_indices, ns, out, B, Hq, Hkv, Smax,
                                d, max_sel, dtype, scratch, kNoAllocScratchBytes, stream);
}

// The status word of the allocation-free decode sits at the start of the scratch array, where
// the workspace of the other decode entry points keeps its own: read and cleared the same way,
// after synchronising the stream (a 4-byte copy to a host word; nothing is allocated).
extern "C" int bsattn_decode_noalloc_status(void* stream) {
    using namespace bsattn;
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (sdev != cur) return BSATTN_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return bsattn_get_device_status(scratch, stream);
}

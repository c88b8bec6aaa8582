// prefill128.cu -- block-sparse attention forward (prefill) with 128-token mask blocks, sm_103a.
//
// Method: TileLang block-sparse Flash-Attention guide, sections 4.1-4.7, at the block size of the
// XAttention algorithm guide, "BSA (Block Sparse Attention)", block size requirement (the
// block-sparse library that consumes XAttention's selection takes 128-token blocks).  Under a
// 128-token mask the two 64-row halves of a query block visit the same keys, so the unit of work
// is one (batch, head, 128-row query block) and every product is a full-rate M = 128 MMA:
//     S = Q K^T     tcgen05.mma M=128 N=64 K=d per 64-key tile (a 128-token key block is two
//                   tiles), fp32 in TMEM
//     token mask on the diagonal / sequence tail
//     exp2 online softmax, one thread per query row (TMEM lane = row: no partner-lane shuffles)
//     O += P V      tcgen05.mma M=128 N=d K=64 with A = P in TMEM (rounded to the input type and
//                   written over its own S buffer, as the scores are already in registers)
// and finally O / l (a row with no visible key stores exactly 0).
//
// Persistent kernel, 256 threads, the warp roles of the 64-row kernel:
//   warp 7      scheduler: claims items from an atomic counter (the last two 128-row blocks of
//               every head first, then windows of heads whose K and V fit in 32 MB), compacts the
//               item's mask row into a list of 64-key tiles, publishes it;
//   warp 5      producers: lane 0 loads Q (128 rows) and streams K tiles, lane 1 streams V tiles,
//               every stage released by the MMA commit that last reads it;
//   warp 4      allocates TMEM and issues Q K^T into S[g % 2] once P V of block g - 2 (whose P
//               sat in that buffer) is done;
//   warp 6      issues P V with A = P from TMEM (S buffer g % 2) into O;
//   warps 0-3   softmax: thread t of warp w owns query row 32 w + t.  A tile's 64 scores are read
//               from TMEM in two passes of 32 so that 32 are live at a time (the second half for
//               its maximum, then the first half, then the second half again).
// TMEM: S / P buffers at columns 0-63 and 64-127, O at 128-(128+d).  Shared memory holds only Q
// and the K and V rings (see Cfg): P never leaves TMEM, so the softmax neither waits for a P tile
// to free nor fences shared-memory writes before P V.  Every wait is bounded: on expiry the CTA
// records BSATTN_ERR_TIMEOUT, drains the copies and MMAs in flight, frees its TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "host_internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kThreads = 256;
constexpr int kSWarp = 4;               // issues Q K^T, owns TMEM
constexpr int kProdWarp = 5;            // TMA producer
constexpr int kPVWarp = 6;              // issues P V
constexpr int kSchedWarp = 7;           // fetches items, compacts their mask rows
constexpr uint32_t kTmemCols = 256;     // S[0] 0-63, S[1] 64-127, O 128-(128+d)
constexpr uint32_t kOCol = 128;
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by > 2^8
// workspace words (int) shared with the 64-row kernel: status, work counter, finished CTAs
constexpr int kWsStatus = 0;
constexpr int kWsNext = 16;
constexpr int kWsDone = 32;

// Shared-memory configurations (P lives in TMEM, so only Q and the K / V rings are here).
// d = 64: Q, four K and four V stages, three item slots with 16-bit tile lists: 80 KB, two CTAs
// per SM.  d = 128, masks up to 256 key tiles (narrow): Q, three K and two V stages, two item
// slots with 8-bit tile lists, laid out from the dynamic shared memory base itself (which the
// kernel checks is 1024-byte aligned): 112.8 KB, so that two CTAs share an SM.  d = 128, wider
// masks: Q, three K and three V stages, three slots, 16-bit lists: 129 KB, one CTA per SM.
template <int D, bool NARROW = false>
struct Cfg {
    static_assert(!NARROW || D == 128, "the narrow configuration is for d = 128");
    static constexpr int kKS = D == 64 ? 4 : 3;         // K stages
    static constexpr int kVS = D == 64 ? 4 : (NARROW ? 2 : 3);   // V stages
    static constexpr int kPT = 2;                       // S / P buffers in TMEM
    static constexpr int kSlots = NARROW ? 2 : 3;       // items published ahead of the consumers
    using ListT = std::conditional_t<NARROW, uint8_t, uint16_t>;
    static constexpr int kMaxNk = NARROW ? 256 : 65535;
    static constexpr uint32_t kSlack = NARROW ? 0 : 1024;   // room to align the base up
    static constexpr int kCtasPerSm = (D == 64 || NARROW) ? 2 : 1;
    static constexpr uint32_t kKTile = (D / 64) * 8192;     // [64 keys x D] 16-bit
    static constexpr uint32_t kQTile = (D / 64) * 16384;    // [128 rows x D]
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kQTile;
    static constexpr uint32_t kV = kK + kKS * kKTile;
    static constexpr uint32_t kBars = kV + kVS * kKTile;
    // q_full q_free k_full[KS] k_empty[KS] v_full[VS] v_empty[VS] s_full[2] s_free[2]
    // p_full[PT] o_free item_full[slots] item_empty[slots] loaded fin_s fin_pv
    static constexpr uint32_t kNumBars = 2 + 2 * kKS + 2 * kVS + 4 + kPT + 1 + 2 * kSlots + 3;
    static constexpr uint32_t kMisc = kBars + 8 * kNumBars;   // tmem, abort, then 4 ints per slot
    static constexpr uint32_t kList = kMisc + 16 + 16 * kSlots;
    static constexpr uint32_t kSmemMax = kCtasPerSm == 2 ? 113u * 1024u : 227u * 1024u;
    __host__ __device__ static uint32_t list_stride(int nk) {
        return (static_cast<uint32_t>(sizeof(ListT)) * nk + 15) & ~15u;
    }
    static uint32_t bytes(int nk) { return kSlack + kList + kSlots * list_stride(nk); }
};

struct Params128 {
    const uint8_t* mask;                // [B, H, nq, mk], one entry per 128 x 128 tokens
    int* ws;                            // status word + scheduler counters
    void* out;
    int B, H, Sq, Sk;
    int nq, nk;                         // 128-row query blocks, 64-key tiles
    int mk;                             // 128-token key blocks per mask row
    int causal;
    int total_items;
    float scale_log2;                   // log2(e) / sqrt(d)
    unsigned long long budget_ns;
};

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float2 fma2f(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float2 add2f(float2 a, float2 b) {
    unsigned long long ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
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

// 32 TMEM lanes x 32 columns: thread t of the warp reads lane (warp's lane quarter + t),
// register j holding column col + j -- one row of an M = 128 accumulator per thread.
__device__ __forceinline__ void tmem_ld_row32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// The matching store (same lane / column mapping).
__device__ __forceinline__ void tmem_st_row32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 TMEM lanes x 16 columns store: thread t writes lane (quarter base + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_st_row16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16, issued by one lane of a converged warp under a guard
// predicate.  A (M = 128 rows x K = 16) sits in 128 TMEM lanes x 8 columns, two 16-bit values
// per column, lower K index in the low half.
__device__ __forceinline__ void mma_f16_ts_if(bool lead, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(lead ? 1u : 0u)
        : "memory");
}

// Item t -> (bh, qb): the first min(2, nq) * BH items are the last two query blocks of every head
// (under a causal mask they visit the most keys), then window by window, `win` heads at a time,
// from the last query block to the first across the window's heads.
__device__ __forceinline__ void decode_item(int t, int BH, int nq, int win, int& bh, int& qb) {
    const int lead = nq < 2 ? nq : 2;
    if (t < lead * BH) {
        qb = nq - 1 - t / BH;
        bh = t - (t / BH) * BH;
        return;
    }
    t -= lead * BH;
    const int rows = nq - lead;
    const int per_win = win * rows;
    const int w = t / per_win;
    const int r = t - w * per_win;
    const int h0 = w * win;
    const int wh = min(win, BH - h0);
    qb = rows - 1 - r / wh;
    bh = h0 + (r - (r / wh) * wh);
}

template <int D, bool BF16, bool NARROW>
__global__ void __launch_bounds__(kThreads, Cfg<D, NARROW>::kCtasPerSm)
    prefill128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Params128 p) {
    using C = Cfg<D, NARROW>;
    using T = std::conditional_t<BF16, __nv_bfloat16, __half>;
    using ListT = typename C::ListT;
    constexpr int kKS = C::kKS, kVS = C::kVS, kPT = C::kPT, kSlots = C::kSlots;
    // TMEM columns: S buffers 0-63 and 64-127 (narrow: P of block g written over the first 32
    // columns of its own S buffer once the scores are in registers), O from 128
    extern __shared__ uint8_t smem_raw[];
    if constexpr (NARROW) {
        // this layout has no slack to align the base up: every CTA leaves (counted as finished)
        // with an error if the base is not 1024-byte aligned
        if (smem_u32(smem_raw) & 1023u) {
            if (threadIdx.x == 0) {
                atomicOr(p.ws + kWsStatus, BSATTN_ERR_CUDA);
                __threadfence();
                if (atomicAdd(p.ws + kWsDone, 1) == static_cast<int>(gridDim.x) - 1) {
                    atomicExch(p.ws + kWsNext, 0);
                    atomicExch(p.ws + kWsDone, 0);
                }
            }
            return;
        }
    }
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* sq = sm + C::kQ;
    uint8_t* sk = sm + C::kK;
    uint8_t* sv = sm + C::kV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
    uint64_t* q_full = bars;
    uint64_t* q_free = q_full + 1;
    uint64_t* k_full = q_free + 1;        // [KS]
    uint64_t* k_empty = k_full + kKS;     // [KS]
    uint64_t* v_full = k_empty + kKS;     // [VS]
    uint64_t* v_empty = v_full + kVS;     // [VS]
    uint64_t* s_full = v_empty + kVS;     // [2] (one used when narrow)
    uint64_t* s_free = s_full + 2;        // [2]
    uint64_t* p_full = s_free + 2;        // [PT]
    uint64_t* o_free = p_full + kPT;
    uint64_t* item_full = o_free + 1;     // [slots]
    uint64_t* item_empty = item_full + kSlots;
    uint64_t* loaded = item_empty + kSlots;
    uint64_t* fin_s = loaded + 1;
    uint64_t* fin_pv = fin_s + 1;
    int* misc = reinterpret_cast<int*>(sm + C::kMisc);   // [0] tmem [1] abort
    int* item_of = misc + 4;                             // [slots]
    int* count_of = item_of + kSlots;                    // [slots] key tiles of the item
    int* bh_of = count_of + kSlots;                      // [slots]
    int* qb_of = bh_of + kSlots;                         // [slots]
    const uint32_t lstride = C::list_stride(p.nk);
    ListT* lists = reinterpret_cast<ListT*>(sm + C::kList);
    volatile int* abort_flag = &misc[1];
    int* status = p.ws + kWsStatus;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int past = p.Sk - p.Sq;                                   // bottom-right causal
    const int BH = p.B * p.H;
    const uint64_t deadline = global_timer_ns() + p.budget_ns;

    if (tid == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int s = 0; s < kKS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&s_full[j], 1);
            mbar_init(&s_free[j], 1);                  // P V of the block (P sits in the buffer)
        }
        for (int j = 0; j < kPT; ++j) {
            mbar_init(&p_full[j], 4);
        }
        mbar_init(o_free, 4);
        for (int j = 0; j < kSlots; ++j) {
            mbar_init(&item_full[j], 1);
            mbar_init(&item_empty[j], 4 + 4);          // 2 producer lanes, 2 issuers, 4 softmax warps
        }
        mbar_init(loaded, 1);
        mbar_init(fin_s, 1);
        mbar_init(fin_pv, 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == kSWarp) {
        tmem_alloc(reinterpret_cast<uint32_t*>(&misc[0]), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = static_cast<uint32_t>(misc[0]);

    if (warp == kSchedWarp) {
        // ------------------------------------------------------------ scheduler warp
        const long long head_kv = 4LL * p.Sk * D;
        const long long wq = (32LL << 20) / (head_kv > 0 ? head_kv : 1);
        const int win = static_cast<int>(wq < 1 ? 1 : (wq > BH ? BH : wq));
        const int long_row = p.nk / 2 > 32 ? p.nk / 2 : 32;
        auto fresh = [&]() -> int {
            int v = 0;
            if (lane == 0) v = atomicAdd(p.ws + kWsNext, 1);
            v = __shfl_sync(0xffffffffu, v, 0);
            if (v < p.total_items) {
                int pbh, pqb;
                decode_item(v, BH, p.nq, win, pbh, pqb);
                const uint8_t* row = p.mask + (static_cast<size_t>(pbh) * p.nq + pqb) * p.mk;
                for (int off = lane * 128; off < p.mk; off += 32 * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
            }
            return v;
        };
        int next_t = fresh();
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            // publish item n only once the producer has issued every K load of item n - 1
            if (n >= 1 && !warp_wait_parity(loaded, (n - 1) & 1, deadline, abort_flag, status)) break;
            if (n >= kSlots && !warp_wait_parity(&item_empty[slot], ((n / kSlots) - 1) & 1, deadline,
                                                 abort_flag, status))
                break;
            if (next_t < 0) next_t = fresh();
            const int t = next_t;
            if (t >= p.total_items) {
                if (lane == 0) {
                    item_of[slot] = -1;
                    mbar_arrive(&item_full[slot]);
                }
                break;
            }
            int bh, qb;
            decode_item(t, BH, p.nq, win, bh, qb);
            int kb_end = p.nk;
            if (p.causal) {
                const long long last_key = static_cast<long long>(min(qb * 128 + 127, p.Sq - 1)) + past;
                const long long lim = last_key / 64 + 1;
                kb_end = last_key < 0 ? 0 : (lim < p.nk ? static_cast<int>(lim) : p.nk);
            }
            // compact the mask row into the visited 64-key tiles, ascending: tile kb reads
            // entry kb / 2 of the row
            const uint8_t* mrow = p.mask + (static_cast<size_t>(bh) * p.nq + qb) * p.mk;
            ListT* list = lists + slot * (lstride / sizeof(ListT));
            int count = 0;
            for (int base = 0; base < kb_end; base += 256) {
                uint32_t bits = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int kb = base + 32 * u + lane;
                    if (kb < kb_end && mrow[kb >> 1] != 0) bits |= 1u << u;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int kb = base + 32 * u + lane;
                    const bool on = (bits >> u) & 1u;
                    const uint32_t ballot = __ballot_sync(0xffffffffu, on);
                    if (on) list[count + __popc(ballot & ((1u << lane) - 1u))] = static_cast<ListT>(kb);
                    count += __popc(ballot);
                }
            }
            __syncwarp();
            if (lane == 0) {
                item_of[slot] = t;
                count_of[slot] = count;
                bh_of[slot] = bh;
                qb_of[slot] = qb;
                mbar_arrive(&item_full[slot]);   // release: the list is visible to the waiters
            }
            // a long row keeps this CTA busy: claiming ahead would hold an item back from CTAs
            // that become free sooner
            next_t = count <= long_row ? fresh() : -1;
        }
    } else if (warp == kProdWarp) {
        // ------------------------------------------------------------ TMA producers
        if (lane < 2) {
            const bool kside = lane == 0;
            if (kside) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
            } else {
                tma_prefetch_desc(&tm_v);
            }
            int kblk = 0, vblk = 0, qloads = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n % kSlots;
                if (!wait_parity(&item_full[slot], (n / kSlots) & 1, deadline, abort_flag, status)) break;
                const int t = item_of[slot];
                const int count = count_of[slot];
                if (t < 0) break;
                if (count > 0) {
                    const int bh = bh_of[slot], qb = qb_of[slot];
                    const ListT* list = lists + slot * (lstride / sizeof(ListT));
                    if (kside) {
                        // the previous item's Q K^T must be done before its Q is overwritten
                        if (qloads >= 1 && !wait_parity(q_free, (qloads - 1) & 1, deadline, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(q_full, C::kQTile);
                        for (int h = 0; h < D / 64; ++h) tma_load_3d(sq + h * 16384, &tm_q, q_full, h * 64, qb * 128, bh);
                        ++qloads;
                        for (int j = 0; ok && j < count; ++j) {
                            const int ks = kblk % kKS;
                            if (kblk >= kKS &&
                                !wait_parity(&k_empty[ks], ((kblk / kKS) - 1) & 1, deadline, abort_flag, status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&k_full[ks], C::kKTile);
                            for (int h = 0; h < D / 64; ++h)
                                tma_load_3d(sk + ks * C::kKTile + h * 8192, &tm_k, &k_full[ks], h * 64, list[j] * 64, bh);
                            ++kblk;
                        }
                    } else {
                        for (int j = 0; ok && j < count; ++j) {
                            const int vs = vblk % kVS;
                            if (vblk >= kVS &&
                                !wait_parity(kVS == 2 ? &s_free[vs] : &v_empty[vs], ((vblk / kVS) - 1) & 1, deadline,
                                             abort_flag, status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&v_full[vs], C::kKTile);
                            for (int h = 0; h < D / 64; ++h)
                                tma_load_3d(sv + vs * C::kKTile + h * 8192, &tm_v, &v_full[vs], h * 64, list[j] * 64, bh);
                            ++vblk;
                        }
                    }
                }
                if (ok) {
                    if (kside) mbar_arrive(loaded);
                    mbar_arrive(&item_empty[slot]);
                }
            }
            if (*abort_flag) {
                // let copies already in flight land before the shared memory is released
                const uint64_t dl = global_timer_ns() + 200000000ull;
                if (kside) {
                    if (qloads > 0) wait_parity_drain(q_full, (qloads - 1) & 1, dl);
                    for (int j = max(0, kblk - kKS); j < kblk; ++j)
                        wait_parity_drain(&k_full[j % kKS], (j / kKS) & 1, dl);
                } else {
                    for (int j = max(0, vblk - kVS); j < vblk; ++j)
                        wait_parity_drain(&v_full[j % kVS], (j / kVS) & 1, dl);
                }
            }
        }
    } else if (warp == kSWarp) {
        // ------------------------------------------------------------ Q K^T issuer
        // converged: the whole warp waits, lane 0 issues under a guard predicate
        const bool lead = lane == 0;
        constexpr uint32_t idS = idesc_f16(128, 64, BF16, false);
        const uint64_t a_base = sdesc_sw128(smem_u32(sq), 16, 1024);
        const uint64_t b_base = sdesc_sw128(smem_u32(sk), 16, 1024);
        int blk = 0, qloads = 0;
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            if (!warp_wait_parity(&item_full[slot], (n / kSlots) & 1, deadline, abort_flag, status)) break;
            const int item = item_of[slot];
            const int cnt = count_of[slot];
            if (item < 0) break;
            bool ok = true;
            if (cnt > 0) {
                if (!warp_wait_parity(q_full, qloads & 1, deadline, abort_flag, status)) break;
                for (int i = 0; i < cnt; ++i) {
                    const int g = blk + i;
                    const int ks = g % kKS;
                    const int sb = g & 1;
                    if (!warp_wait_parity(&k_full[ks], (g / kKS) & 1, deadline, abort_flag, status) ||
                        (g >= 2 && !warp_wait_parity(&s_free[sb], ((g - 2) >> 1) & 1, deadline, abort_flag,
                                                     status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptor start addresses advance by (byte offset >> 4); a 64-column half
                    // of Q is 16 KB (128 rows), of K 8 KB (64 rows)
                    const uint64_t b_stage = b_base + ((ks * C::kKTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t a_off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        const uint32_t b_off = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                        mma_f16_ss_if(lead, tbase + sb * 64, a_base + a_off, b_stage + b_off, idS,
                                      kk > 0 ? 1u : 0u);
                    }
                    mma_commit_if(lead, &s_full[sb]);
                    mma_commit_if(lead, &k_empty[ks]);                 // K stage free
                    if (i == cnt - 1) mma_commit_if(lead, q_free);     // Q no longer read
                }
                blk += cnt;
                ++qloads;
            }
            if (!ok) break;
            mbar_arrive_if(lead, &item_empty[slot]);
        }
        mma_commit_if(lead, fin_s);
        wait_parity_drain(fin_s, 0, global_timer_ns() + 200000000ull);
        __syncwarp();
    } else if (warp == kPVWarp) {
        // ------------------------------------------------------------ P V issuer
        const bool lead = lane == 0;
        constexpr uint32_t idO = idesc_f16(128, D, BF16, true);
        const uint64_t v_desc = sdesc_sw128(smem_u32(sv), 8192, 1024);
        int blk = 0, items = 0;
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            if (!warp_wait_parity(&item_full[slot], (n / kSlots) & 1, deadline, abort_flag, status)) break;
            const int item = item_of[slot];
            const int cnt = count_of[slot];
            if (item < 0) break;
            bool ok = true;
            for (int i = 0; i < cnt; ++i) {
                const int g = blk + i;
                const int vs = g % kVS;
                // V has usually landed long before P is written: polling v_full first leaves
                // p_full the last wait before the issue
                if (!warp_wait_parity(&v_full[vs], (g / kVS) & 1, deadline, abort_flag, status) ||
                    (i == 0 && items >= 1 &&
                     !warp_wait_parity(o_free, (items - 1) & 1, deadline, abort_flag, status)) ||
                    !warp_wait_parity(&p_full[g % kPT], (g / kPT) & 1, deadline, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // 16 keys of P are 32 bytes along its rows; 16 tokens of V are 16 rows of 128 bytes
                const uint64_t b0 = v_desc + static_cast<uint32_t>(vs) * (C::kKTile >> 4);
                // A = P of block g in TMEM, over the first 32 columns of S buffer g % 2: 16 keys
                // are 8 columns
                const uint32_t a0 = tbase + 64 * (g & 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16_ts_if(lead, tbase + kOCol, a0 + 8 * kk, b0 + ((kk * 2048) >> 4), idO,
                                  (i > 0 || kk > 0) ? 1u : 0u);
                // P V of g done: S / P buffer g % 2 is free for Q K^T of g + 2, O holds block g (the
                // epilogue and the O rescale wait on this commit too) and, with two V stages, V stage
                // g % 2 is free; a deeper V ring has its own release barrier.  Fewer commits per tile
                // leave more of the tensor core's issue pipe to the MMAs.
                mma_commit_if(lead, &s_free[g & 1]);
                if constexpr (kVS != 2) mma_commit_if(lead, &v_empty[vs]);
            }
            if (!ok) break;
            if (cnt > 0) {
                blk += cnt;
                ++items;
            }
            mbar_arrive_if(lead, &item_empty[slot]);
        }
        mma_commit_if(lead, fin_pv);
        wait_parity_drain(fin_pv, 0, global_timer_ns() + 200000000ull);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps 0-3
        // Thread t of warp w owns query row 32 w + t of the item, TMEM lane 32 w + t.
        const int lrow = 32 * warp + lane;
        const uint32_t tl = tbase + (static_cast<uint32_t>(32 * warp) << 16);
        const float c = p.scale_log2;
        int blk = 0;
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            if (!warp_wait_parity(&item_full[slot], (n / kSlots) & 1, deadline, abort_flag, status)) break;
            const int item = item_of[slot];
            const int cnt = count_of[slot];
            if (item < 0) break;
            const int bh = bh_of[slot], qb = qb_of[slot];
            const ListT* list = lists + slot * (lstride / sizeof(ListT));
            if (cnt == 0) {
                // no visible key anywhere in this query block: its rows are exactly zero
                const int rows = min(128, p.Sq - qb * 128);
                uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                      (static_cast<size_t>(bh) * p.Sq + qb * 128) * D);
                const int n16 = rows * D * 2 / 16;
                for (int e = tid; e < n16; e += 128) out[e] = make_uint4(0, 0, 0, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(&item_empty[slot]);
                continue;
            }
            const int row = qb * 128 + lrow;
            // keys at or past `lim` are not visible to this row (sequence end; causal diagonal)
            const int lim = p.causal ? min(p.Sk, row + past + 1) : p.Sk;
            float m_used = -INFINITY;
            float l = 0.f;
            bool ok = true;
            for (int i = 0; i < cnt; ++i) {
                const int g = blk + i;
                const int sb = g & 1;
                if (!warp_wait_parity(&s_full[sb], (g >> 1) & 1, deadline, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int key0 = static_cast<int>(list[i]) * 64;
                const bool edge = key0 + 63 >= lim;
                // 32 scores of half h of the tile, masked on the diagonal / sequence tail
                auto load_half = [&](int h, float (&sc)[32]) {
                    uint32_t r[32];
                    tmem_ld_row32(tl + sb * 64 + 32 * h, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) sc[e] = __uint_as_float(r[e]);
                    if (edge) {
                        const int n = lim - (key0 + 32 * h);          // visible scores of this half
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e >= n) sc[e] = -INFINITY;
                    }
                };
                auto max32 = [&](const float (&sc)[32]) -> float {
                    float m4[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float x = max3f(sc[j], sc[j + 4], sc[j + 8]);
                        x = max3f(x, sc[j + 12], sc[j + 16]);
                        x = max3f(x, sc[j + 20], sc[j + 24]);
                        m4[j] = fmaxf(x, sc[j + 28]);
                    }
                    return fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
                };
                float sc[32];
                load_half(1, sc);
                const float m1 = max32(sc);
                load_half(0, sc);
                const float mx = fmaxf(max32(sc), m1);
                const bool grow = mx * c > m_used * c + kRescaleLog2;
                const float m_new = grow ? mx : m_used;
                const float alpha = grow ? ex2_approx((m_used - m_new) * c) : 1.f;
                const bool rescale_o = grow && m_used != -INFINITY;
                m_used = m_new;
                const float mc = m_new == -INFINITY ? 0.f : m_new * c;
                // exp2, the row sum (four packed f32x2 accumulators), the rounding to the input type
                // and the store of P in one pass: P of block g goes over the first 32 columns of its
                // own S buffer (half h of the row: 16 columns of two values), whose scores are in
                // registers by then; Q K^T refills the buffer only after P V of g has read it
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                auto exp_store = [&](int h, const float (&x)[32]) {
                    uint32_t pv[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 y = fma2f(make_float2(x[8 * k + e], x[8 * k + e + 1]), make_float2(c, c),
                                                   make_float2(-mc, -mc));
                            const float2 ev = make_float2(ex2_approx(y.x), ex2_approx(y.y));
                            acc[e >> 1] = add2f(acc[e >> 1], ev);
                            pv[4 * k + (e >> 1)] = pack2<BF16>(ev.x, ev.y);
                        }
                    }
                    tmem_st_row16(tl + sb * 64 + 16 * h, pv);
                };
                exp_store(0, sc);
                load_half(1, sc);
                exp_store(1, sc);
                const float2 a2 = add2f(add2f(acc[0], acc[1]), add2f(acc[2], acc[3]));
                l = l * alpha + (a2.x + a2.y);
                if (__any_sync(0xffffffffu, rescale_o)) {
                    // O is scaled once it holds every block before g: P V of g - 1 must be done
                    if (g >= 1 && !warp_wait_parity(&s_free[(g - 1) & 1], ((g - 1) >> 1) & 1, deadline,
                                                    abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld_row32(tl + kOCol + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st_row32(tl + kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
                tmem_wait_st();                         // P is in TMEM before P V reads it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[g % kPT]);
            }
            if (!ok) break;
            // ---- epilogue: O / l, written from registers straight to global memory
            const int glast = blk + cnt - 1;
            if (!warp_wait_parity(&s_free[glast & 1], (glast >> 1) & 1, deadline, abort_flag, status)) break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) + (static_cast<size_t>(bh) * p.Sq + row) * D);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_row32(tl + kOCol + c0, o);
                tmem_wait_ld();
                if (c0 + 32 == D) {
                    // O is in registers: the next item's first P V may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_free);
                }
                uint32_t ob[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    ob[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                if (row < p.Sq) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[c0 / 8 + k] = make_uint4(ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            blk += cnt;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kSWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0) {
        // the last CTA to finish resets the scheduler for the next call on this workspace
        __threadfence();
        const int done = atomicAdd(p.ws + kWsDone, 1);
        if (done == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.ws + kWsNext, 0);
            atomicExch(p.ws + kWsDone, 0);
        }
    }
}

template <int D, bool BF16, bool NARROW = false>
int launch128(const void* q, const void* k, const void* v, const Params128& prm, cudaStream_t stream) {
    using C = Cfg<D, NARROW>;
    const uint32_t smem = C::bytes(prm.nk);
    if (smem > C::kSmemMax || prm.nk > C::kMaxNk) return BSATTN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    const uint64_t BH = static_cast<uint64_t>(prm.B) * prm.H;
    int rc = 0;
    rc |= encode_3d(&tq, q, BF16, D, prm.Sq, BH, D * 2ull, uint64_t(prm.Sq) * D * 2, 64, 128, 1, true);
    rc |= encode_3d(&tk, k, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&tv, v, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    if (rc) return rc;
    auto kern = prefill128_kernel<D, BF16, NARROW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    int sms = num_sms_of_current_device();
    if (sms <= 0) sms = 148;
    long long grid = static_cast<long long>(C::kCtasPerSm) * sms;
    if (grid > prm.total_items) grid = prm.total_items;
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // namespace

// The 128-row kernel for a 128-token mask; BSATTN_ERR_UNSUPPORTED when the mask rows do not fit
// its shared memory (the caller then runs the 64-row kernels).  Arguments are checked by the caller.
int prefill128_launch(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                      int is_causal, void* out, int B, int H, int Sq, int Sk, int d, bool bf16,
                      void* workspace, cudaStream_t stream) {
    Params128 prm{};
    prm.mask = block_mask;
    prm.ws = static_cast<int*>(workspace);
    prm.out = out;
    prm.B = B;
    prm.H = H;
    prm.Sq = Sq;
    prm.Sk = Sk;
    prm.nq = (Sq + 127) / 128;
    prm.nk = (Sk + 63) / 64;
    prm.mk = (Sk + 127) / 128;
    prm.causal = is_causal ? 1 : 0;
    const long long items = static_cast<long long>(B) * H * prm.nq;
    if (items > 0x7fffffffLL) return BSATTN_ERR_UNSUPPORTED;
    prm.total_items = static_cast<int>(items);
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    prm.budget_ns = wait_budget_ns();
    if (d == 64) return bf16 ? launch128<64, true>(q, k, v, prm, stream) : launch128<64, false>(q, k, v, prm, stream);
    if (d == 128) {
        // two CTAs per SM (the narrow layout) whenever the mask rows allow it
        if (prm.nk <= Cfg<128, true>::kMaxNk && Cfg<128, true>::bytes(prm.nk) <= Cfg<128, true>::kSmemMax)
            return bf16 ? launch128<128, true, true>(q, k, v, prm, stream)
                        : launch128<128, false, true>(q, k, v, prm, stream);
        return bf16 ? launch128<128, true>(q, k, v, prm, stream) : launch128<128, false>(q, k, v, prm, stream);
    }
    return BSATTN_ERR_UNSUPPORTED;
}

}  // namespace bsattn

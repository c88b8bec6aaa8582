// prefill.cu -- block-sparse attention forward (prefill) for sm_103a.
//
// Method: TileLang block-sparse Flash-Attention guide, sections 4.1-4.7.  The unit of work is
// one (batch, head, 64-row query block).  Its row of the block mask is compacted into the list
// of key blocks to visit (section 4.4: only set blocks are loaded and multiplied; causal rows
// stop at the diagonal), those K/V tiles are streamed through shared memory with TMA, and per
// visited block
//     S = Q K^T                      (tcgen05.mma, M=64 N=64 K=d, fp32 in TMEM)
//     token mask on the diagonal / sequence tail (section 4.5)
//     exp2 online softmax            (section 4.6, scale log2(e)/sqrt(d) folded in)
//     O += P V                       (tcgen05.mma, M=64 N=d K=64, P rounded to the input type)
// and finally O / l (section 4.7; a row with no visible key stores exactly 0).
//
// Persistent kernel: two CTAs per SM (each holds half of the SM's 512 TMEM columns) pull work
// items from an atomic counter in the workspace.  Items are ordered from the last query block
// to the first across all heads (under a causal mask the late blocks visit the most keys), so
// the longest items start first and the tail is short.  Warp roles (288 threads):
//   warp 7      scheduler: claims the next item from the counter one ahead (not while the CTA
//               is on a long row) and pulls its mask row and its Q tile into L2; publishes it
//               once the producer has issued the previous item's K loads, after compacting its
//               mask row;
//   warps 5, 8  producers: warp 5 loads each item's Q and streams its K tiles, warp 8 streams
//               its V tiles, into K and V rings -- running ahead across items (one lane each: in
//               separate warps neither stream's waits hold up the other's issue).  Two stages
//               each at d = 128 (three K stages and one P tile in the deeper variant, used
//               whenever its shared memory fits), three each at d = 64;
//   warp 4      allocates TMEM and issues Q K^T as soon as a K tile and an S buffer are free;
//   warp 6      issues P V as soon as the softmax has written P (two issuing threads keep the
//               M=64 tensor pipe fed: one thread issues at most about one MMA per 67 cycles);
//               warps 4 and 6 run converged, lane 0 issuing under a guard predicate;
//   warps 0-3   softmax (lanes t and t+16 of warp w own query row 16w + t%16, TMEM lane
//               32w + t%16 of the M=64 accumulator, and read its two 32-column halves through
//               the 16x32bx2 shape; three-input max, packed f32x2 FMA and adds) and the
//               epilogue, which writes O / l from registers with 16-byte stores.
// In the deeper variants P stays in TMEM: the softmax writes it (16x32bx2 stores, in the M = 64
// accumulator layout) over the first 32 columns of its block's S buffer, P V reads it as the A
// operand from tensor memory, and the commit of P V(g) frees that S buffer for the Q K^T of the
// block that reuses it (g + 2; g + 3 at d = 64, which has three S buffers) and marks P V(g) done --
// no P tile to wait for and no shared-memory fence before P V.
// Every mbarrier wait is polled by the whole warp (one non-blocking probe, then a bounded loop):
// a wait by one lane behind a branch costs several times more on this hardware.
// Rows that can span 1024+ key blocks and visit more than 96 are split into 64-block parts: the
// CTA that compacts such a row keeps part 0 and queues the rest for free CTAs; the last part to
// finish merges the partial outputs by log-sum-exp.
//
// Differences from the page's kernel (made for this hardware):
//  * the mask row is compacted once per item, so masked K/V tiles are never addressed;
//  * S and P are double- or triple-buffered and a K stage is released as soon as its Q K^T is
//    done (where a ring is as deep as the S buffers, the commits that complete S and free the S
//    buffer also free its K and V stages; the third K stage at d = 128 has its own barrier), so
//    Q K^T of the next blocks runs while the softmax works, and the softmax of block g+1 runs
//    while P V of block g is in the tensor pipe; the next item's loads overlap the current
//    item's work;
//  * O lives in TMEM and is rescaled only when a row maximum grows by more than 2^8
//    (exact: the final normaliser l is accumulated against the same reference maximum).
// Every wait is bounded: on expiry the CTA records BSATTN_ERR_TIMEOUT, drains the copies and
// MMAs it has in flight, frees its TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "host_internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kThreads = 288;
constexpr int kSWarp = 4;               // issues Q K^T, owns TMEM
constexpr int kProdWarp = 5;            // TMA producer
constexpr int kPVWarp = 6;              // issues P V
constexpr int kSchedWarp = 7;           // fetches items, compacts their mask rows
constexpr int kVProdWarp = 8;           // TMA producer of the V tiles
// K and V rings: a K stage frees when the Q K^T reading it is done, a V stage when its P V is
// done.  Where a ring is as deep as the S buffers, its stage g % SB coincides with S buffer g % SB
// of block g, and the commits that complete S (Q K^T) or free the S buffer (P V) also free the
// stage: fewer tcgen05.commit per block, each of which occupies the tensor core's issue pipe.
// At d = 128 two stages of each are what shared memory allows beside Q and P at two CTAs per SM;
// the deeper d = 128 variant has a third K stage with its own k_empty barrier.  At d = 64 the
// deeper variant has three K and three V stages, as deep as its three S buffers (four stages
// with their own release barriers measured 3 % slower on the C4 workload).  The deeper variants
// keep P in TMEM (the shared-memory P tiles then go unused) and are used whenever their shared
// memory (which grows with the mask-row lists) fits: always at d = 64, up to 1304 key blocks at
// d = 128.
constexpr int kRingD64 = 3;
template <int D, bool DEEP>
struct Rings {
    static constexpr int kK = D == 64 ? (DEEP ? kRingD64 : 2) : (DEEP ? 3 : 2);
    static constexpr int kV = D == 64 ? (DEEP ? kRingD64 : 2) : 2;
    // P tiles in shared memory: two (double-buffered), one in the deeper d = 128 variant.  p_full
    // and o_done are rings of parity barriers indexed by block: two at d = 128; four in the deeper
    // d = 64 variant, whose three S buffers let the softmax run three blocks ahead of P V (a ring
    // of two would then let a parity wait on block g pass on the phase of block g - 2).  Kernels
    // that keep P in TMEM use neither the P tiles nor o_done (s_free marks P V done).
    static constexpr int kPTiles = (D == 128 && DEEP) ? 1 : 2;
    static constexpr int kPF = (D == 64 && DEEP) ? 4 : 2;
    static constexpr int kOD = (D == 64 && DEEP) ? 4 : 2;
    static_assert(kV != 2 || kOD == 2, "two V stages are released through o_done[g % 2]");
};
constexpr uint32_t kTmemCols = 256;     // S buffers of 64 columns from 0, then O (d columns)
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by > 2^8
constexpr int kCtasPerSm = 2;
constexpr int kSlots = 3;               // items published ahead of the consumers
constexpr uint32_t kSmemPerCtaMax = 113u * 1024u;   // dynamic shared memory at two CTAs per SM

// workspace words (int): status, work counter, finished-CTA counter, continuation queue head,
// partial-slot counter, call epoch; then the continuation entries, the per-row merge tickets,
// the partial LSE values and the partial outputs of rows split across CTAs
constexpr int kWsStatus = 0;
constexpr int kWsNext = 16;
constexpr int kWsDone = 32;
constexpr int kWsContHead = 48;
constexpr int kWsPoolNext = 49;
constexpr int kWsEpoch = 50;
constexpr int kWsQTail = 51;
constexpr size_t kWsHeaderBytes = 1024;
constexpr int kMaxSlots = 2048;         // partial outputs that can be in use at once
constexpr int kSplitMinNk = 1024;       // rows are split only when they can be this long
constexpr int kEntryInts = 8;           // t, start, len, part, nparts, slot base, ready, -

struct PrefillParams {
    const uint8_t* mask;
    int* ws;                            // status word + scheduler counters
    int* entries;                       // [kMaxSlots][kEntryInts]; nullptr: no splitting
    int split_min;                      // rows visiting more key blocks than this are split
    int split_len;                      // ... into parts of this many blocks
    int long_row;                       // a CTA on a row longer than this claims no item ahead
    int* tickets;                       // [kMaxSlots]
    float* lse;                         // [kMaxSlots][64]
    float* opart;                       // [kMaxSlots][64][d]
    void* out;
    int B, H, Sq, Sk, nq, nk;           // nq, nk: 64-row query / 64-key blocks
    int bshift;                         // mask block = 64 << bshift tokens (64 or 128)
    int mq, mk;                         // block_mask row count and row length per (b, h)
    int causal;
    int total_items;
    float scale_log2;                   // log2(e) / sqrt(d)
    unsigned long long budget_ns;
};

template <int D, bool DEEP>
struct Layout {
    using R = Rings<D, DEEP>;
    static constexpr uint32_t kTile = (D / 64) * 8192;   // one [64 x D] 16-bit tile
    static constexpr uint32_t kQ = 0;                     // Q of the current item
    static constexpr uint32_t kK = kTile;
    static constexpr uint32_t kV = kK + R::kK * kTile;
    static constexpr uint32_t kP = kV + R::kV * kTile;   // [64 x 64] P tiles
    static constexpr uint32_t kBars = kP + R::kPTiles * 8192;
    // q_full q_free k_full[KS] v_full[VS] s_full[2] s_free[2]
    // p_full[PF] o_done[OD] o_free item_full[slots] item_empty[slots] fin_s fin_pv loaded pdone mdec
    // k_empty[KS] v_empty[VS]
    static constexpr uint32_t kNumBars = 2 + 2 * (R::kK + R::kV) + 6 + R::kPF + R::kOD + 1 + 2 * kSlots + 5;
    static constexpr uint32_t kMisc = kBars + 8 * kNumBars;   // tmem, abort, per-slot item info
    static constexpr uint32_t kList = kMisc + 16 + 28 * kSlots + 16;
    __host__ __device__ static constexpr uint32_t list_stride(int nk) { return (2 * nk + 15) & ~15; }
    static constexpr uint32_t bytes(int nk) { return 1024 + kList + kSlots * list_stride(nk); }
};

// max(a, b, c) in one instruction (three-input max.f32)
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed f32x2 arithmetic (one instruction for two fp32 lanes of a register pair).
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

// 16 TMEM lanes x 32 bits in two halves, 16 columns each: lane t < 16 of the warp writes lane
// (quarter base + t), columns [col, col + 16); lane t >= 16 writes lane (quarter base + t - 16),
// columns [col + 16, col + 32).  For an M = 64 operand (rows 16w..16w+15 in lanes 32w..32w+15)
// lanes t and t + 16 thus write the two 16-column halves of the same row.
__device__ __forceinline__ void tmem_st_16x32bx2_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 16, "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16, issued by one lane of a converged warp under a guard
// predicate; A in tensor memory in the accumulator layout of its M, two 16-bit values per column.
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

// Item t -> (bh, qb).  The first min(2, nq) * BH items are the last two query blocks of every
// head: under a causal mask they visit the most keys (dense last rows visit all of them), so
// the longest items start first.  The rest run window by window, `win` heads at a time (heads
// whose K and V fit in a share of L2), and inside a window from the last query block to the
// first across its heads: the K/V tiles that a window's rows share stay in L2 while it runs.
__device__ __forceinline__ void decode_item(int t, int BH, int nq, int win, int& bh, int& qb) {
    const int lead = nq < 2 ? nq : 2;
    if (t < lead * BH) {
        qb = nq - 1 - t / BH;
        bh = t - (t / BH) * BH;
        return;
    }
    t -= lead * BH;
    const int rows = nq - lead;                 // > 0 here
    const int per_win = win * rows;
    const int w = t / per_win;
    const int r = t - w * per_win;
    const int h0 = w * win;
    const int wh = min(win, BH - h0);           // the last window may hold fewer heads
    qb = rows - 1 - r / wh;
    bh = h0 + (r - (r / wh) * wh);
}

template <int D, bool BF16, bool DEEP, bool SPLIT, bool TPV>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using L = Layout<D, DEEP>;
    using R = Rings<D, DEEP>;
    using T = std::conditional_t<BF16, __nv_bfloat16, __half>;
    constexpr uint32_t kTile = L::kTile;
    constexpr int kKStages = R::kK;
    constexpr int kVStages = R::kV;
    constexpr int kPT = R::kPTiles;
    constexpr int kPF = R::kPF;
    constexpr int kOD = R::kOD;
    // S buffers in TMEM (64 columns each): three at d = 64 with P in TMEM (P over its S buffer ties
    // the buffer up until P V is done, and 3 x 64 + 64 columns fit), else two; O follows them
    constexpr int kSB = (TPV && D == 64) ? 3 : 2;
    constexpr uint32_t kOCol = kSB * 64;
    // Barriers that do double duty keep the tcgen05.commit count per block down (each commit
    // occupies the tensor core's issue pipe, which limits the d = 64 kernels): with P in TMEM the
    // commit that frees an S buffer after P V also marks that P V done (the epilogue and the O
    // rescale wait on it) and frees V stage g % SB when the V ring is as deep as the S buffers;
    // the commit that completes S frees K stage g % SB when the K ring is.  Without P in TMEM,
    // o_done marks P V done and frees V stage g % 2.
    constexpr bool kKbyS = kKStages == kSB;
    constexpr bool kVbyS = TPV && kVStages == kSB;
    constexpr bool kVbyO = !TPV && kVStages == 2;
    static_assert(kPF >= kSB && kOD >= kSB, "p_full / o_done rings at least as deep as the S buffers");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* sq = sm + L::kQ;
    uint8_t* sk = sm + L::kK;
    uint8_t* sv = sm + L::kV;
    uint8_t* sp = sm + L::kP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    uint64_t* q_full = bars;
    uint64_t* q_free = q_full + 1;
    uint64_t* k_full = q_free + 1;                 // [KS]
    uint64_t* v_full = k_full + kKStages;          // [VS]
    uint64_t* s_full = v_full + kVStages;          // [SB] (at d = 128 without TMEM P it also frees K stage g % 2)
    uint64_t* s_free = s_full + 3;                 // [SB]
    uint64_t* p_full = s_free + 3;                 // [PF] P of block g written (index g % PF)
    uint64_t* o_done = p_full + kPF;               // [OD] P V of block g done (index g % OD)
    uint64_t* o_free = o_done + kOD;
    uint64_t* item_full = o_free + 1;              // [slots]
    uint64_t* item_empty = item_full + kSlots;     // [slots]
    uint64_t* fin_s = item_empty + kSlots;
    uint64_t* fin_pv = fin_s + 1;
    uint64_t* loaded = fin_pv + 1;                 // the K lane issued an item's Q and K loads
    uint64_t* pdone = loaded + 1;                  // softmax warps wrote a split part's partial
    uint64_t* mdec = pdone + 1;                    // merge decision of a split row is known
    uint64_t* k_empty = mdec + 1;                  // [KS] Q K^T reading the stage is done
    uint64_t* v_empty = k_empty + kKStages;        // [VS] P V reading the stage is done
    int* misc = reinterpret_cast<int*>(sm + L::kMisc);   // [0] tmem [1] abort [2..] item, count
    int* item_of = misc + 4;                             // [slots]
    int* count_of = item_of + kSlots;                    // [slots] blocks of this (part of a) row
    int* part_of = count_of + kSlots;                    // [slots]
    int* nparts_of = part_of + kSlots;                   // [slots] 1 = row not split
    int* sbase_of = nparts_of + kSlots;                  // [slots] first partial slot of the row
    int* bh_of = sbase_of + kSlots;                      // [slots] (batch, head) of the item
    int* qb_of = bh_of + kSlots;                         // [slots] query block of the item
    int* merge_flag = qb_of + kSlots;                    // [1]
    const uint32_t lstride = L::list_stride(p.nk);
    uint16_t* lists = reinterpret_cast<uint16_t*>(sm + L::kList);
    volatile int* abort_flag = &misc[1];
    int* status = p.ws + kWsStatus;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int past = p.Sk - p.Sq;                                   // bottom-right causal
    const int BH = p.B * p.H;
    const uint64_t deadline = global_timer_ns() + p.budget_ns;

    if (tid == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int j = 0; j < kSB; ++j) {
            mbar_init(&s_full[j], 1);
            // one arrival per softmax warp; with P in TMEM over S, the commit of P V of the block
            mbar_init(&s_free[j], TPV ? 1 : 4);
        }
        for (int j = 0; j < kSlots; ++j) {
            mbar_init(&item_full[j], 1);
            mbar_init(&item_empty[j], 4 + 4);          // 2 producers, S and PV issuers, 4 softmax warps
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int j = 0; j < kPF; ++j) mbar_init(&p_full[j], 4);   // one arrival per softmax warp
        for (int j = 0; j < kOD; ++j) mbar_init(&o_done[j], 1);
        mbar_init(o_free, 4);
        mbar_init(fin_s, 1);
        mbar_init(fin_pv, 1);
        mbar_init(loaded, 1);                          // the K producer lane
        mbar_init(pdone, 4);
        mbar_init(mdec, 1);
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
        const int epoch = p.ws[kWsEpoch];
        volatile int* vws = p.ws;
        // heads per window of the work order: as many as keep the window's K and V within 32 MB,
        // a quarter of L2, so that the tiles its rows revisit are still there
        const long long head_kv = 4LL * p.Sk * D;
        const long long wq = (32LL << 20) / (head_kv > 0 ? head_kv : 1);
        const int win = static_cast<int>(wq < 1 ? 1 : (wq > BH ? BH : wq));
        // the next fresh item is claimed one ahead, and its mask row and Q tile pulled into L2,
        // so that neither the counter's round trip nor the row's first read delays publishing
        // it, and its Q load (issued once the previous item's Q K^T is done) hits L2
        auto fresh = [&]() -> int {
            int v = 0;
            if (lane == 0) v = atomicAdd(p.ws + kWsNext, 1);
            v = __shfl_sync(0xffffffffu, v, 0);
            if (v < p.total_items) {
                int pbh, pqb;
                decode_item(v, BH, p.nq, win, pbh, pqb);
                const uint8_t* row = p.mask + (static_cast<size_t>(pbh) * p.mq + (pqb >> p.bshift)) * p.mk;
                for (int off = lane * 128; off < p.mk; off += 32 * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
                if (lane == 0)
                    for (int h = 0; h < D / 64; ++h)
                        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                                         reinterpret_cast<uint64_t>(&tm_q)),
                                     "r"(h * 64), "r"(pqb * 64), "r"(pbh)
                                     : "memory");
            }
            return v;
        };
        int next_t = fresh();
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            // publish item n only once the producer has issued every K load of item n-1: a CTA
            // then holds at most one item besides the one it computes (and one claimed ahead),
            // so a CTA busy with a long item does not keep short ones from idle CTAs
            if (n >= 1 && !warp_wait_parity(loaded, (n - 1) & 1, deadline, abort_flag, status)) break;
            if (n >= kSlots && !warp_wait_parity(&item_empty[slot], ((n / kSlots) - 1) & 1, deadline,
                                                 abort_flag, status))
                break;
            // 1. a continuation part of a long row split by another CTA, if one is queued; once
            //    the work counter is exhausted the queue is drained before this CTA stops
            auto claim = [&]() -> int {
                int e = -1;
                if (SPLIT && lane == 0 && p.entries) {
                    for (;;) {
                        const int h = vws[kWsContHead];
                        const int tl = vws[kWsQTail];
                        if (h >= tl) break;
                        if (atomicCAS(p.ws + kWsContHead, h, h + 1) != h) continue;
                        volatile int* ent = p.entries + h * kEntryInts;
                        // the entry is written right after its slot is reserved
                        uint32_t spins = 0;
                        bool ready;
                        while (!(ready = ent[6] == epoch + 1)) {
                            if ((spins++ & 63u) == 0 && global_timer_ns() > deadline) {
                                atomicOr(status, BSATTN_ERR_TIMEOUT);
                                *abort_flag = 1;
                                break;
                            }
                        }
                        if (!ready) break;
                        __threadfence();
                        e = h;
                        break;
                    }
                }
                return __shfl_sync(0xffffffffu, e, 0);
            };
            int e = claim();
            if (*abort_flag) break;
            int t, start = 0, len = 0x7fffffff, part = 0, nparts = 1, sbase = -1;
            bool took_fresh = false;
            if (e < 0) {
                if (next_t < 0) next_t = fresh();   // not claimed ahead (after a long row)
                t = next_t;
                took_fresh = t < p.total_items;
                if (t >= p.total_items) {
                    // no fresh rows left: parts other CTAs queued may still arrive until every
                    // CTA has taken its last row, and queued parts are always run by someone
                    e = claim();
                    if (*abort_flag) break;
                }
            }
            if (e >= 0) {
                volatile int* ent = p.entries + e * kEntryInts;
                t = ent[0];
                start = ent[1];
                len = ent[2];
                part = ent[3];
                nparts = ent[4];
                sbase = ent[5];
            }
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
                const long long last_key = static_cast<long long>(min(qb * 64 + 63, p.Sq - 1)) + past;
                const long long lim = last_key / 64 + 1;
                kb_end = last_key < 0 ? 0 : (lim < p.nk ? static_cast<int>(lim) : p.nk);
            }
            // 2. compact the mask row (visited key blocks in ascending order) into the slot's
            //    list, keeping entries [start, start + len) of it
            // a mask entry covers (64 << bshift)^2 tokens: the 64-row item reads row qb >> bshift,
            // and key block kb (64 keys) reads entry kb >> bshift of it
            const uint8_t* mrow = p.mask + (static_cast<size_t>(bh) * p.mq + (qb >> p.bshift)) * p.mk;
            uint16_t* list = lists + slot * (lstride / 2);
            int count = 0;
            for (int base = 0; base < kb_end; base += 256) {
                // eight independent loads per lane first, then the ordered ballots
                uint32_t bits = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int kb = base + 32 * u + lane;
                    if (kb < kb_end && mrow[kb >> p.bshift] != 0) bits |= 1u << u;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int kb = base + 32 * u + lane;
                    const bool on = (bits >> u) & 1u;
                    const uint32_t ballot = __ballot_sync(0xffffffffu, on);
                    const int pos = count + __popc(ballot & ((1u << lane) - 1u)) - start;
                    if (on && pos >= 0 && pos < len) list[pos] = static_cast<uint16_t>(kb);
                    count += __popc(ballot);
                }
            }
            // 3. a fresh row that visits many key blocks is split: this CTA keeps the first
            //    part, the others are queued for any CTA to take
            if (SPLIT && e < 0 && p.entries && count > p.split_min) {
                const int np = (count + p.split_len - 1) / p.split_len;
                int base_slot = 0, q0 = 0;
                if (lane == 0) {
                    base_slot = atomicAdd(p.ws + kWsPoolNext, np);
                    // queue entries only for parts 1..np-1: part 0 stays with this CTA
                    if (base_slot + np <= kMaxSlots) q0 = atomicAdd(p.ws + kWsQTail, np - 1);
                }
                base_slot = __shfl_sync(0xffffffffu, base_slot, 0);
                q0 = __shfl_sync(0xffffffffu, q0, 0);
                if (base_slot + np <= kMaxSlots) {               // else: the pool is full, no split
                    for (int i = 1 + lane; i < np; i += 32) {
                        int* ent = p.entries + (q0 + i - 1) * kEntryInts;
                        const int st = i * p.split_len;
                        ent[0] = t;
                        ent[1] = st;
                        ent[2] = min(p.split_len, count - st);
                        ent[3] = i;
                        ent[4] = np;
                        ent[5] = base_slot;
                        __threadfence();
                        reinterpret_cast<volatile int*>(ent)[6] = epoch + 1;
                    }
                    nparts = np;
                    sbase = base_slot;
                    len = p.split_len;
                }
            }
            __syncwarp();
            if (lane == 0) {
                item_of[slot] = t;
                count_of[slot] = min(count - start, len);
                part_of[slot] = part;
                nparts_of[slot] = nparts;
                sbase_of[slot] = sbase;
                bh_of[slot] = bh;
                qb_of[slot] = qb;
                mbar_arrive(&item_full[slot]);   // release: the list is visible to the waiters
            }
            // a long row keeps this CTA busy: claiming ahead would hold an item back from CTAs
            // that become free sooner
            if (took_fresh && (e >= 0 || count <= p.long_row)) next_t = fresh();
            else if (took_fresh) next_t = -1;
        }
    } else if (warp == kProdWarp || warp == kVProdWarp) {
        // ------------------------------------------------------------ TMA producers
        // lane 0 of warp 5 streams each item's Q and K tiles, lane 0 of warp 8 its V tiles: the
        // two rings drain at different points (a K stage after Q K^T, a V stage after P V), so
        // neither stream waits for the other's slower ring
        if (lane == 0) {
            const bool kside = warp == kProdWarp;
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
                    const uint16_t* list = lists + slot * (lstride / 2);
                    if (kside) {
                        // the previous item's Q K^T must be done before its Q is overwritten
                        if (qloads >= 1 && !wait_parity(q_free, (qloads - 1) & 1, deadline, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(q_full, kTile);
                        for (int h = 0; h < D / 64; ++h) tma_load_3d(sq + h * 8192, &tm_q, q_full, h * 64, qb * 64, bh);
                        ++qloads;
                        for (int j = 0; ok && j < count; ++j) {
                            const int ks = kblk % kKStages;
                            if (kblk >= kKStages &&
                                !wait_parity(kKbyS ? &s_full[ks] : &k_empty[ks], ((kblk / kKStages) - 1) & 1,
                                             deadline, abort_flag,
                                             status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&k_full[ks], kTile);
                            for (int h = 0; h < D / 64; ++h)
                                tma_load_3d(sk + ks * kTile + h * 8192, &tm_k, &k_full[ks], h * 64, list[j] * 64, bh);
                            ++kblk;
                        }
                    } else {
                        for (int j = 0; ok && j < count; ++j) {
                            const int vs = vblk % kVStages;
                            if (vblk >= kVStages &&
                                !wait_parity(kVbyS ? &s_free[vs] : (kVbyO ? &o_done[vs] : &v_empty[vs]), ((vblk / kVStages) - 1) & 1,
                                             deadline, abort_flag,
                                             status)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&v_full[vs], kTile);
                            for (int h = 0; h < D / 64; ++h)
                                tma_load_3d(sv + vs * kTile + h * 8192, &tm_v, &v_full[vs], h * 64, list[j] * 64, bh);
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
                    for (int j = max(0, kblk - kKStages); j < kblk; ++j)
                        wait_parity_drain(&k_full[j % kKStages], (j / kKStages) & 1, dl);
                } else {
                    for (int j = max(0, vblk - kVStages); j < vblk; ++j)
                        wait_parity_drain(&v_full[j % kVStages], (j / kVStages) & 1, dl);
                }
            }
        }
    } else if (warp == kSWarp) {
        // ------------------------------------------------------------ Q K^T issuer
        // the whole warp runs the loop and waits (converged polls are cheap); lane 0 alone
        // issues the MMAs, commits and arrivals, under a guard predicate
        const bool lead = lane == 0;
        constexpr uint32_t idS = idesc_f16(64, 64, BF16, false);
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
                    const int ks = g % kKStages;
                    const int sb = kSB == 2 ? (g & 1) : g % kSB;
                    if (!warp_wait_parity(&k_full[ks], (g / kKStages) & 1, deadline, abort_flag, status) ||
                        (g >= kSB && !warp_wait_parity(&s_free[sb], ((g / kSB) - 1) & 1, deadline, abort_flag,
                                                       status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptor start addresses advance by (byte offset >> 4)
                    const uint64_t b_stage = b_base + ((ks * kTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                        mma_f16_ss_if(lead, tbase + sb * 64, a_base + off, b_stage + off, idS,
                                      kk > 0 ? 1u : 0u);
                    }
                    mma_commit_if(lead, &s_full[sb]);
                    if constexpr (!kKbyS) mma_commit_if(lead, &k_empty[ks]);   // K stage free
                    if (i == cnt - 1) mma_commit_if(lead, q_free);   // Q no longer read
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
        // converged like the Q K^T issuer: lane 0 issues under a guard predicate
        const bool lead = lane == 0;
        constexpr uint32_t idO = idesc_f16(64, D, BF16, true);
        const uint64_t p_desc = sdesc_sw128(smem_u32(sp), 16, 1024);
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
                const int vs = g % kVStages;
                // V has usually landed long before P is written: polling v_full first leaves
                // p_full the last wait before the issue
                if (!warp_wait_parity(&v_full[vs], (g / kVStages) & 1, deadline, abort_flag, status) ||
                    (i == 0 && items >= 1 &&
                     !warp_wait_parity(o_free, (items - 1) & 1, deadline, abort_flag, status)) ||
                    !warp_wait_parity(&p_full[g % kPF], (g / kPF) & 1, deadline, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // descriptor start addresses advance by (byte offset >> 4): 16 keys of P are 32 bytes
                // along its rows, 16 tokens of V are 16 rows of 128 bytes
                const uint64_t b0 = v_desc + static_cast<uint32_t>(vs) * (kTile >> 4);
                if constexpr (TPV) {
                    // A = P of block g in TMEM over the first 32 columns of S buffer g % 2: 16 keys
                    // are 8 columns
                    const uint32_t a0 = tbase + 64 * (kSB == 2 ? (g & 1) : g % kSB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_ts_if(lead, tbase + kOCol, a0 + 8 * kk, b0 + ((kk * 2048) >> 4), idO,
                                      (i > 0 || kk > 0) ? 1u : 0u);
                } else {
                    const uint64_t a0 = p_desc + static_cast<uint32_t>(g % kPT) * (8192u >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_ss_if(lead, tbase + kOCol, a0 + ((kk * 32) >> 4), b0 + ((kk * 2048) >> 4), idO,
                                      (i > 0 || kk > 0) ? 1u : 0u);
                }
                if constexpr (!TPV) mma_commit_if(lead, &o_done[g % kOD]);  // P V of g done: its P tile is free
                if constexpr (TPV) mma_commit_if(lead, &s_free[kSB == 2 ? (g & 1) : g % kSB]);   // S / P buffer free
                if constexpr (!kVbyS && !kVbyO) mma_commit_if(lead, &v_empty[vs]);   // V stage free
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
        // Lanes t and t + 16 of warp w own local query row 16w + t%16 (TMEM lane 32w + t%16 of
        // the M = 64 accumulator); lane t takes columns [32 (t/16), +32) of every S tile and
        // columns [(d/2) (t/16), +d/2) of O, through the 16x32bx2 access shape.
        const int hf = lane >> 4;
        const int lrow = 16 * warp + (lane & 15);
        const uint32_t tl = tbase + (static_cast<uint32_t>(32 * warp) << 16);
        const float c = p.scale_log2;
        int blk = 0, qloads = 0, nsplit = 0;
        for (int n = 0;; ++n) {
            const int slot = n % kSlots;
            if (!warp_wait_parity(&item_full[slot], (n / kSlots) & 1, deadline, abort_flag, status)) break;
            const int item = item_of[slot];
            const int cnt = count_of[slot];
            if (item < 0) break;
            const int part = part_of[slot], nparts = nparts_of[slot], sbase = sbase_of[slot];
            const int bh = bh_of[slot], qb = qb_of[slot];
            const uint16_t* list = lists + slot * (lstride / 2);
            if (cnt == 0) {
                // no visible key anywhere in this query block: its rows are exactly zero
                const int rows = min(64, p.Sq - qb * 64);
                uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                      (static_cast<size_t>(bh) * p.Sq + qb * 64) * D);
                const int n16 = rows * D * 2 / 16;
                for (int e = tid; e < n16; e += 128) out[e] = make_uint4(0, 0, 0, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(&item_empty[slot]);
                continue;
            }
            const int row = qb * 64 + lrow;
            float m_used = -INFINITY;
            float l = 0.f;
            bool ok = true;
            for (int i = 0; i < cnt; ++i) {
                const int g = blk + i;
                const int sb = kSB == 2 ? (g & 1) : g % kSB;
                if (!warp_wait_parity(&s_full[sb], (g / kSB) & 1, deadline, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r[32];
                tmem_ld_16x32bx2_x32<32>(tl + sb * 64, r);
                tmem_wait_ld();
                if constexpr (!TPV) {
                    // this warp's lanes of S[sb] are in registers: Q K^T of block g+2 may reuse it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_free[sb]);
                }
                float s[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) s[e] = __uint_as_float(r[e]);

                const int key0 = static_cast<int>(list[i]) * 64 + 32 * hf;
                if (key0 + 31 >= p.Sk || (p.causal && key0 + 31 > row + past)) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = key0 + e;
                        if (key >= p.Sk || (p.causal && key > row + past)) s[e] = -INFINITY;
                    }
                }
                // row maximum: four chains of three-input maxima over this lane's 32 columns, then
                // the partner lane's half
                float m4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x = max3f(s[j], s[j + 4], s[j + 8]);
                    x = max3f(x, s[j + 12], s[j + 16]);
                    x = max3f(x, s[j + 20], s[j + 24]);
                    m4[j] = fmaxf(x, s[j + 28]);
                }
                const float m0 = fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
                const float mx = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 16));
                const bool grow = mx * c > m_used * c + kRescaleLog2;
                const float m_new = grow ? mx : m_used;
                const float alpha = grow ? ex2_approx((m_used - m_new) * c) : 1.f;
                const bool rescale_o = grow && m_used != -INFINITY;
                m_used = m_new;
                const float mc = m_new == -INFINITY ? 0.f : m_new * c;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    // S c - m c for two columns in one packed f32x2 FMA, then exp2 of each
                    const float2 x = fma2f(make_float2(s[e], s[e + 1]), make_float2(c, c), make_float2(-mc, -mc));
                    s[e] = ex2_approx(x.x);
                    s[e + 1] = ex2_approx(x.y);
                }
                // row sum: a tree of packed f32x2 adds over column pairs, then the partner lane's half
                float2 p2[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    p2[e] = add2f(make_float2(s[2 * e], s[2 * e + 1]), make_float2(s[2 * e + 16], s[2 * e + 17]));
#pragma unroll
                for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
                    for (int e = 0; e < w2; ++e) p2[e] = add2f(p2[e], p2[e + w2]);
                const float sum0 = p2[0].x + p2[0].y;
                const float sum = sum0 + __shfl_xor_sync(0xffffffffu, sum0, 16);
                l = l * alpha + sum;
                uint32_t pk[16];                  // P in the input type, ready for the P tile
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(s[2 * e], s[2 * e + 1]);
                // P tile g % PT is free once P V of block g - PT is done (P in TMEM: it goes over
                // this block's own S buffer, which Q K^T could only refill after that P V)
                if (!TPV && g >= kPT && !warp_wait_parity(&o_done[(g - kPT) % kOD], ((g - kPT) / kOD) & 1, deadline,
                                                          abort_flag, status)) {
                    ok = false;
                    break;
                }
                if (__any_sync(0xffffffffu, rescale_o)) {
                    // O is scaled once it holds every block before g: P V of g-1 must be done
                    if (g >= 1 && !warp_wait_parity(TPV ? &s_free[(g - 1) % kSB] : &o_done[(g - 1) % kOD],
                                                    TPV ? ((g - 1) / kSB) & 1 : ((g - 1) / kOD) & 1, deadline,
                                                    abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D / 2; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld_16x32bx2_x32<D / 2>(tl + kOCol + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st_16x32bx2_x32<D / 2>(tl + kOCol + c0, o);
                    }
                    tmem_wait_st();
                }
                if constexpr (TPV) {
                    // P -> TMEM over the first 32 columns of S buffer sb (this lane's 32 keys are
                    // 16 columns: the first or the second half of its row)
                    tmem_st_16x32bx2_x16(tl + sb * 64, pk);
                    tmem_wait_st();
                } else {
                    // P -> the swizzled P tile: this lane's 32 columns are 16-byte chunks
                    // 4 hf .. 4 hf + 3 of its row; a chunk c of row r sits at r * 128 + (c ^ (r % 8)) * 16
                    uint8_t* prow = sp + (g % kPT) * 8192 + lrow * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int chunk = (4 * hf + k) ^ (lrow & 7);
                        *reinterpret_cast<uint4*>(prow + chunk * 16) =
                            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[g % kPF]);
            }
            if (!ok) break;
            // ---- epilogue: O / l, written from registers straight to global memory
            const int glast = blk + cnt - 1;
            if (!warp_wait_parity(TPV ? &s_free[glast % kSB] : &o_done[glast % kOD],
                                  TPV ? (glast / kSB) & 1 : (glast / kOD) & 1, deadline, abort_flag, status))
                break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (SPLIT && nparts > 1) {
                // one part of a row split across CTAs: its O / l (fp32) and log2-sum-exp go to the
                // row's partial slots; the last part to finish merges them with LSE weights
                float* op = p.opart + static_cast<size_t>(sbase + part) * 64 * D + lrow * D + hf * (D / 2);
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_16x32bx2_x32<D / 2>(tl + kOCol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(op + c0 + e) =
                            make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                        __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
                if (hf == 0)
                    p.lse[static_cast<size_t>(sbase + part) * 64 + lrow] =
                        l > 0.f ? m_used * c + log2f(l) : -INFINITY;
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(pdone);
                if (tid == 0) {
                    int last = 0;
                    if (wait_parity(pdone, nsplit & 1, deadline, abort_flag, status)) {
                        last = atomicAdd(p.tickets + sbase, 1) == nparts - 1;
                        if (last) p.tickets[sbase] = 0;   // ready for the next call
                    }
                    *merge_flag = last;
                    mbar_arrive(mdec);
                }
                if (!warp_wait_parity(mdec, nsplit & 1, deadline, abort_flag, status)) break;
                ++nsplit;
                if (*reinterpret_cast<volatile int*>(merge_flag)) {
                    __threadfence();
                    // lanes t and t + 16 of warp w merge local row 16w + t%16, d/2 columns each,
                    // 32 at a time: per part one weight and eight independent 16-byte loads
                    // from L2 (where the parts' writes landed)
                    const float* lsr = p.lse + static_cast<size_t>(sbase) * 64 + lrow;
                    const float* opr = p.opart + (static_cast<size_t>(sbase) * 64 + lrow) * D + hf * (D / 2);
                    float M = -INFINITY;
#pragma unroll 4
                    for (int pp = 0; pp < nparts; ++pp) M = fmaxf(M, __ldcg(lsr + pp * 64));
                    float den = 0.f;
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                          (static_cast<size_t>(bh) * p.Sq + row) * D + hf * (D / 2));
#pragma unroll 1
                    for (int c0 = 0; c0 < D / 2; c0 += 32) {
                        float acc[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                        if (M != -INFINITY) {
#pragma unroll 2
                            for (int pp = 0; pp < nparts; ++pp) {
                                const float w = ex2_approx(__ldcg(lsr + pp * 64) - M);
                                if (c0 == 0) den += w;
                                const float4* src = reinterpret_cast<const float4*>(opr + static_cast<size_t>(pp) * 64 * D + c0);
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    const float4 v4 = __ldcg(src + k);
                                    acc[4 * k + 0] += w * v4.x;
                                    acc[4 * k + 1] += w * v4.y;
                                    acc[4 * k + 2] += w * v4.z;
                                    acc[4 * k + 3] += w * v4.w;
                                }
                            }
                        }
                        const float invd = den > 0.f ? 1.f / den : 0.f;
                        if (row < p.Sq) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                dst[c0 / 8 + k] = make_uint4(pack2<BF16>(acc[8 * k + 0] * invd, acc[8 * k + 1] * invd),
                                                             pack2<BF16>(acc[8 * k + 2] * invd, acc[8 * k + 3] * invd),
                                                             pack2<BF16>(acc[8 * k + 4] * invd, acc[8 * k + 5] * invd),
                                                             pack2<BF16>(acc[8 * k + 6] * invd, acc[8 * k + 7] * invd));
                        }
                    }
                }
            } else {
                // this lane's d/2 columns of its row, 32 at a time: packed, stored as 16-byte vectors
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                      (static_cast<size_t>(bh) * p.Sq + row) * D + hf * (D / 2));
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_16x32bx2_x32<D / 2>(tl + kOCol + c0, o);
                    tmem_wait_ld();
                    if (c0 + 32 == D / 2) {
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            blk += cnt;
            ++qloads;
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
            atomicExch(p.ws + kWsContHead, 0);
            atomicExch(p.ws + kWsPoolNext, 0);
            atomicExch(p.ws + kWsQTail, 0);
            atomicAdd(p.ws + kWsEpoch, 1);       // queue entries of this call are now stale
            atomicExch(p.ws + kWsDone, 0);
        }
    }
}

template <int D, bool BF16, bool DEEP, bool TPV = false>
int launch(const void* q, const void* k, const void* v, const PrefillParams& prm,
           cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    const uint64_t BH = static_cast<uint64_t>(prm.B) * prm.H;
    int rc = 0;
    rc |= encode_3d(&tq, q, BF16, D, prm.Sq, BH, D * 2ull, uint64_t(prm.Sq) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&tk, k, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    rc |= encode_3d(&tv, v, BF16, D, prm.Sk, BH, D * 2ull, uint64_t(prm.Sk) * D * 2, 64, 64, 1, true);
    if (rc) return rc;
    // at most two CTAs per SM: each holds 256 of the SM's 512 TMEM columns
    uint32_t smem = Layout<D, DEEP>::bytes(prm.nk);
    if (smem < 78u * 1024u) smem = 78u * 1024u;
    if (smem > kSmemPerCtaMax) return BSATTN_ERR_UNSUPPORTED;
    // rows are split across CTAs only when the continuation queue is set up (rows that can span
    // 1024+ key blocks): the kernel without that code is smaller, which keeps its hot loops in the
    // instruction cache
    auto kern = prm.entries ? prefill_kernel<D, BF16, DEEP, true, TPV> : prefill_kernel<D, BF16, DEEP, false, TPV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    int sms = num_sms_of_current_device();
    if (sms <= 0) sms = 148;
    long long grid = static_cast<long long>(kCtasPerSm) * sms;
    if (grid > prm.total_items) grid = prm.total_items;
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // namespace
}  // namespace bsattn

namespace bsattn {
namespace {
// bytes of each workspace region (partial outputs sized for d = 128)
constexpr size_t kWsEntriesOff = kWsHeaderBytes;
constexpr size_t kWsTicketsOff = kWsEntriesOff + sizeof(int) * kMaxSlots * kEntryInts;
constexpr size_t kWsLseOff = kWsTicketsOff + sizeof(int) * kMaxSlots;
constexpr size_t kWsOpartOff = kWsLseOff + sizeof(float) * kMaxSlots * 64;
constexpr size_t kWsFullBytes = kWsOpartOff + sizeof(float) * kMaxSlots * 64 * 128;
constexpr size_t kWsMinBytes = 256;
}  // namespace
}  // namespace bsattn

extern "C" size_t bsattn_prefill_workspace_size(int, int, int, int) { return bsattn::kWsFullBytes; }

extern "C" int bsattn_prefill_bs(const void* q, const void* k, const void* v,
                                 const uint8_t* block_mask, int block_size, int is_causal, void* out,
                                 int B, int H, int Sq, int Sk, int d, bsattn_dtype dtype,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    using namespace bsattn;
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return BSATTN_ERR_INVALID_ARG;
    if (block_size != 64 && block_size != 128) return BSATTN_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return BSATTN_ERR_UNSUPPORTED;
    if (dtype != BSATTN_F16 && dtype != BSATTN_BF16) return BSATTN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < kWsMinBytes) return BSATTN_ERR_INVALID_ARG;
    const long long BH = static_cast<long long>(B) * H;
    if (BH == 0 || Sq == 0) return BSATTN_OK;
    if (!q || !k || !v || !out || !block_mask) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace))
        return BSATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Sk == 0) {
        // no keys at all: every row is exactly zero
        return cudaMemsetAsync(out, 0, static_cast<size_t>(BH) * Sq * d * 2, st) == cudaSuccess
                   ? BSATTN_OK
                   : BSATTN_ERR_CUDA;
    }
    const int nq = (Sq + 63) / 64, nk = (Sk + 63) / 64;
    if (nk > 4096 || BH * nq > 0x7fffffffLL || BH > 0x7fffffffLL) return BSATTN_ERR_UNSUPPORTED;
    if (block_size == 128 && nk < kSplitMinNk) {
        // both 64-row halves of a 128-token query block visit the same keys: full-rate M = 128
        // tiles, unless the mask rows do not fit that kernel's shared memory
        const int rc = prefill128_launch(q, k, v, block_mask, is_causal, out, B, H, Sq, Sk, d,
                                         dtype == BSATTN_BF16, workspace, st);
        if (rc != BSATTN_ERR_UNSUPPORTED) return rc;
    }
    PrefillParams prm{};
    prm.mask = block_mask;
    prm.ws = static_cast<int*>(workspace);
    prm.long_row = nk / 2 > 32 ? nk / 2 : 32;
    if (workspace_bytes >= kWsFullBytes && nk >= kSplitMinNk) {
        // room for the continuation queue and partial outputs, and rows long enough that one
        // of them could outlast the rest of the launch: a row visiting more than 96 key blocks
        // is split into parts of 64, run by whichever CTAs are free and merged by log-sum-exp
        uint8_t* w = static_cast<uint8_t*>(workspace);
        prm.split_min = 96;
        prm.split_len = 64;
        prm.entries = reinterpret_cast<int*>(w + kWsEntriesOff);
        prm.tickets = reinterpret_cast<int*>(w + kWsTicketsOff);
        prm.lse = reinterpret_cast<float*>(w + kWsLseOff);
        prm.opart = reinterpret_cast<float*>(w + kWsOpartOff);
    }
    prm.out = out;
    prm.B = B;
    prm.H = H;
    prm.Sq = Sq;
    prm.Sk = Sk;
    prm.nq = nq;
    prm.nk = nk;
    prm.bshift = block_size == 128 ? 1 : 0;
    prm.mq = (Sq + block_size - 1) / block_size;
    prm.mk = (Sk + block_size - 1) / block_size;
    prm.causal = is_causal ? 1 : 0;
    prm.total_items = static_cast<int>(BH * nq);
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    prm.budget_ns = wait_budget_ns();
    const bool bf16 = dtype == BSATTN_BF16;
    // the deeper rings, with P in TMEM, whenever they fit beside the mask-row lists (every width
    // up to 4096 key blocks at d = 64, up to 1304 at d = 128), else two stages (up to 2672 key
    // blocks at d = 128)
    static_assert(Layout<64, true>::bytes(4096) <= kSmemPerCtaMax, "d = 64 always runs the deeper rings");
    if (d == 64)
        return bf16 ? launch<64, true, true, true>(q, k, v, prm, st) : launch<64, false, true, true>(q, k, v, prm, st);
    if (Layout<128, true>::bytes(nk) <= kSmemPerCtaMax)
        return bf16 ? launch<128, true, true, true>(q, k, v, prm, st)
                    : launch<128, false, true, true>(q, k, v, prm, st);
    return bf16 ? launch<128, true, false>(q, k, v, prm, st) : launch<128, false, false>(q, k, v, prm, st);
}

extern "C" int bsattn_prefill(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                              int is_causal, void* out, int B, int H, int Sq, int Sk, int d,
                              bsattn_dtype dtype, void* workspace, size_t workspace_bytes,
                              void* stream) {
    return bsattn_prefill_bs(q, k, v, block_mask, 64, is_causal, out, B, H, Sq, Sk, d, dtype,
                             workspace, workspace_bytes, stream);
}

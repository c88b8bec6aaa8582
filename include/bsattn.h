/*
 * bsattn.h -- C ABI of the GB300 (sm_103a) block-sparse attention library.
 *
 * Sources of the operations (page title, section):
 *   [BSA] "TileLang 块稀疏 Flash-Attention 内核实现与实战指南" (TileLang block-sparse
 *         Flash-Attention kernel guide): 3.1 top-k mask, 3.2 threshold mask, 4.1-4.7 the
 *         prefill kernel, 5 the reference check, 6.1-6.3 GQA varlen sparse decode and the
 *         split heuristic, 7 paged KV decode.
 *   [FA]  "使用 TileLang 实现 FlashAttention ... 完整实战指南" (TileLang FlashAttention
 *         guide): online softmax, bottom-right causal alignment when seq_kv > seq_q.
 *   [XA]  "XAttention 算法实现指南" (XAttention algorithm guide): block selection
 *         (find_blocks_chunked) and its worked example.
 *
 * Conventions for every call:
 *   - Pointers marked (device) are caller-owned device memory; (host) caller-owned host
 *     memory.  The library never allocates, frees or retains any of them.
 *   - Tensors are dense, row-major (last index fastest), with no padding between rows.
 *   - GPU calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The return value only reports host-side argument checks and launch
 *     errors; faults found on the device (a bounded wait that expired, an out-of-range
 *     block index) are OR-ed into the status word at the start of the workspace and are
 *     read (and cleared) with bsattn_get_device_status().
 *   - Workspaces must be zero-filled once before their first use; every call leaves them
 *     ready for the next call (counters are reset by the kernels themselves).  After a
 *     call reports BSATTN_ERR_TIMEOUT the workspace must be zero-filled again.
 *   - Block size is 64 tokens (bsattn_prefill_bs also takes 128-token prefill masks);
 *     head dimension d is 64 or 128; dtype fp16 or bf16.
 */
#ifndef BSATTN_H_
#define BSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { BSATTN_F16 = 0, BSATTN_BF16 = 1 } bsattn_dtype;

typedef enum {
    BSATTN_OK = 0,
    BSATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned or too-small buffer */
    BSATTN_ERR_UNSUPPORTED = 2,  /* head dim / dtype / shape outside what is built */
    BSATTN_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
    BSATTN_ERR_TIMEOUT = 8,      /* device: a bounded wait expired (the kernel bailed out) */
    BSATTN_ERR_BAD_INDEX = 16    /* device: a block index past the sequence was skipped */
} bsattn_status;

#define BSATTN_BLOCK 64

/* Human-readable name of a status value (or of an OR of device status bits). */
const char* bsattn_status_string(int status);

/* Library version string. */
const char* bsattn_version(void);

/*
 * Block-sparse attention forward (prefill) -- [BSA] 4.1-4.7.
 *
 * For every (batch b, head h, 64-row query block qb) only key blocks kb with
 * block_mask[b][h][qb][kb] != 0 are visited; when is_causal, only key positions
 * j <= i + (Sk - Sq) are visible to query position i (bottom-right alignment, [FA]); keys
 * j >= Sk are never visible.  Computes out_i = softmax_j(q_i . k_j / sqrt(d)) v_j over the
 * visible keys with an exp2 online softmax in fp32, P rounded to the input dtype for the
 * second product; a query row with no visible key gets exactly 0.
 *
 *   q           (device) [B, H, Sq, d]  dtype
 *   k, v        (device) [B, H, Sk, d]  dtype
 *   block_mask  (device) [B, H, ceil(Sq/64), ceil(Sk/64)] uint8, nonzero = visit
 *   out         (device) [B, H, Sq, d]  dtype, fully written (rows with no work = 0)
 *   workspace   (device) >= 256 bytes, zero-filled once, 16-byte aligned: scheduler counters
 *               and the status word.  With bsattn_prefill_workspace_size() bytes (64 MiB) and
 *               rows that can span 1024+ key blocks, a row visiting more than 96 key blocks is
 *               split into 64-block parts run by different CTAs and merged by log-sum-exp
 *               (2048 partial slots; rows that do not fit run whole, so results are
 *               bit-reproducible only while the slots suffice).
 * q, k, v, out must be 16-byte aligned.  Returns BSATTN_OK or an error status; Sk beyond
 * 4096 key blocks at d = 64, or 2672 key blocks (171008 keys) at d = 128, returns
 * BSATTN_ERR_UNSUPPORTED (the per-CTA shared memory holds each item's mask-row list).
 */
int bsattn_prefill(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                   int is_causal, void* out, int B, int H, int Sq, int Sk, int d,
                   bsattn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * bsattn_prefill with a block mask of 64- or 128-token blocks -- [BSA] 4.1-4.7 with the
 * block size of [XA] "BSA (Block Sparse Attention)", block size requirement (the block-sparse
 * library that consumes XAttention's selection takes 128-token blocks only).
 *
 *   block_size  64 or 128 (else BSATTN_ERR_UNSUPPORTED)
 *   block_mask  (device) [B, H, ceil(Sq/block_size), ceil(Sk/block_size)] uint8: entry
 *               [qb][kb] != 0 makes query rows [qb*bs, qb*bs+bs) see keys [kb*bs, kb*bs+bs)
 *               (subject to the causal rule and to Sk, as in bsattn_prefill).
 * Every other argument, the result and the error behaviour are those of bsattn_prefill, which
 * is this call with block_size = 64.  The kernel works on 64-token tiles either way: a
 * 128-token entry stands for the four 64 x 64 tiles it covers.
 */
int bsattn_prefill_bs(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                      int block_size, int is_causal, void* out, int B, int H, int Sq, int Sk,
                      int d, bsattn_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Workspace bytes that enable splitting long rows (256 bytes is the minimum). */
size_t bsattn_prefill_workspace_size(int B, int H, int Sq, int Sk);

/*
 * GQA variable-length sparse decode -- [BSA] 6.1-6.2.
 *
 * One query token per sequence.  Query head h reads kv head g = h / (Hq / Hkv).  The keys
 * of (b, g) are the union over the slots t of block_indices[b][g][:] with t >= 0 of the
 * tokens [64 t, 64 t + 64) clipped to cache_seqlens[b]; out[b][h] = softmax attention of
 * q[b][h] over those keys (exactly 0 when there are none).  The selected blocks of each
 * (b, g) are cut into num_splits contiguous slices ([BSA] 6.2: the first len % num_splits
 * slices get one extra block) processed by separate CTAs and merged by log-sum-exp.
 *
 *   q              (device) [B, Hq, d]            dtype
 *   k, v           (device) [B, Smax, Hkv, d]     dtype (BSHD)
 *   cache_seqlens  (device) [B] int32, each in [0, Smax]
 *   block_indices  (device) [B, Hkv, max_sel] int32; -1 = empty slot; valid entries are
 *                  distinct and < ceil(cache_seqlens[b] / 64), in any order.  Entries at or
 *                  past the sequence end are skipped and flagged BSATTN_ERR_BAD_INDEX.
 *   num_splits     >= 1, or 0 to let the library choose (bsattn_decode_default_splits)
 *   out            (device) [B, Hq, d] dtype
 *   workspace      (device) >= bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, num_splits)
 *                  bytes, zero-filled once.
 * Requires Hq % Hkv == 0, 1 <= Hq / Hkv <= 8, d in {64, 128}; q, k, v, out 16-byte aligned.
 */
int bsattn_decode_varlen(const void* q, const void* k, const void* v,
                         const int32_t* cache_seqlens, const int32_t* block_indices,
                         int num_splits, void* out, int B, int Hq, int Hkv, int Smax, int d,
                         int max_sel, bsattn_dtype dtype, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * bsattn_decode_varlen without a workspace argument, for callers that cannot allocate
 * device memory when they attend (code running inside a custom allocator or memory pool,
 * runtimes that forbid allocation after start-up, hosts that only pass pointers to buffers
 * they own).  The pages have no counterpart: this is a deployment variant of the decode
 * above, with the same arguments (minus the workspace) and the same results.
 *
 * Its scratch is one fixed 8 MiB device array inside the library (held by every GPU that
 * loads the library until the process exits); shapes whose decode workspace
 * (bsattn_decode_workspace_size) exceeds it return BSATTN_ERR_UNSUPPORTED.  It allocates
 * nothing: no cudaMalloc / cudaFree, no allocating library routine.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  CUDA loads a library's device
 * code lazily by default, and that first call is also what loads this file's code and
 * reserves the array on the device: make one call per device before entering a context
 * that must not allocate (or run with CUDA_MODULE_LOADING=EAGER).  `stream` must belong to
 * the current device (else BSATTN_ERR_INVALID_ARG).  Each call clears the array's status
 * word and merge tickets with cudaMemsetAsync on `stream`.  All calls share the array, so
 * calls that overlap on the GPU (different streams, or threads) race and must be serialised
 * by the caller.  Device-detected conditions (a skipped out-of-range index, an expired
 * wait) go to the array's status word: read them with bsattn_decode_noalloc_status.
 */
int bsattn_decode_varlen_noalloc(const void* q, const void* k, const void* v,
                                 const int32_t* cache_seqlens, const int32_t* block_indices,
                                 int num_splits, void* out, int B, int Hq, int Hkv, int Smax,
                                 int d, int max_sel, bsattn_dtype dtype, void* stream);

/*
 * Reads and clears the device status word of bsattn_decode_varlen_noalloc on the current
 * device, after synchronising `stream` (which must belong to that device, else
 * BSATTN_ERR_INVALID_ARG).  Each allocation-free call clears the word when it starts, so the
 * result is the OR of the BSATTN_ERR_* bits (BSATTN_ERR_BAD_INDEX, BSATTN_ERR_TIMEOUT) that
 * the most recent call recorded (0 = none), or BSATTN_ERR_CUDA if the read itself failed.
 * It allocates nothing: a 4-byte copy into a host word.
 */
int bsattn_decode_noalloc_status(void* stream);

/*
 * GQA varlen sparse decode, block-mask form -- [BSA] 6 (the `_mask` example).  Identical to
 * bsattn_decode_varlen except that the selected blocks of (b, g) are given as
 *   block_mask (device) [B, Hkv, num_blocks] uint8, nonzero = block j selected;
 * slot j of the mask is block j, and the num_blocks slots are cut into num_splits slices as in
 * [BSA] 6.2.  Set entries at or past the sequence end select no tokens (not flagged).
 * Workspace: bsattn_decode_workspace_size(B, Hq, Hkv, d, num_blocks, num_splits) bytes.
 */
int bsattn_decode_varlen_mask(const void* q, const void* k, const void* v,
                              const int32_t* cache_seqlens, const uint8_t* block_mask,
                              int num_splits, void* out, int B, int Hq, int Hkv, int Smax, int d,
                              int num_blocks, bsattn_dtype dtype, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * GQA varlen sparse decode over a paged KV cache -- [BSA] 7.  As bsattn_decode_varlen, but
 *   k_pages, v_pages (device) [num_pages, page_size, Hkv, d] dtype
 *   block_table      (device) [B, max_pages_per_seq] int32: logical page p of sequence b is
 *                    physical page block_table[b][p]
 * Logical token position P of sequence b lives in page block_table[b][P / page_size], row
 * P % page_size.  page_size must be a multiple of 64 (a 64-token block never straddles two
 * pages; [BSA] 7 asserts the same).  Blocks whose page is out of range are skipped and flagged
 * BSATTN_ERR_BAD_INDEX.  Workspace as for bsattn_decode_varlen.
 */
int bsattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* cache_seqlens, const int32_t* block_indices,
                        const int32_t* block_table, int num_splits, void* out, int B, int Hq,
                        int Hkv, int num_pages, int page_size, int max_pages_per_seq, int d,
                        int max_sel, bsattn_dtype dtype, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Workspace bytes bsattn_decode_varlen needs (num_splits 0 = the library's choice). */
size_t bsattn_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_sel, int num_splits);

/*
 * The split count bsattn_decode_varlen uses when num_splits == 0: the decode is bound by HBM
 * bandwidth, so it takes as many splits as fill exactly one wave of resident CTAs (resident
 * CTAs per SM for head dim d x num_sms, divided over the B * Hkv groups), capped by max_sel
 * and 64.  num_sms <= 0 queries the current device.
 */
int bsattn_decode_default_splits(int B, int Hkv, int max_sel, int d, int num_sms);

/*
 * The split-count rule of [BSA] 6.3, bit-exact: if total_mblocks >= 0.8 num_SMs return 1
 * (or, when one kv head exceeds the assumed 50 MB L2, num_m_blocks > 2 num_SMs and not
 * causal/local, ceil(size / L2) capped at max_splits); if num_n_blocks <= 4 return 1;
 * otherwise the smallest s in [1, min(max_splits, num_SMs, num_n_blocks)] whose wave
 * efficiency w / ceil(w), w = total_mblocks s / num_SMs, is >= 0.85 of the best.
 * Pure host function.
 */
int bsattn_num_splits_heuristic(int total_mblocks, int num_SMs, int num_n_blocks,
                                int num_m_blocks, long long size_one_kv_head,
                                int is_causal_or_local, int max_splits);

/*
 * Host-side block-mask builders -- [BSA] 3.1 and 3.2.  scores (host) fp32
 * [B, H, nq, nk]; mask_out (host) uint8 of the same shape, fully written with 0 / 1.
 *   top-k:     per row keep the min(topk, nk) highest scores (ties: lower column first).
 *   threshold: keep score > threshold (strict).
 * Then, if use_dense_for_last_block, the last min(2, nq) rows are set all-1; then, if
 * apply_tril, entries with column > row are cleared.  NaN scores -> BSATTN_ERR_INVALID_ARG.
 */
int bsattn_mask_from_topk(const float* scores, int B, int H, int nq, int nk, int topk,
                          int use_dense_for_last_block, int apply_tril, uint8_t* mask_out);
int bsattn_mask_from_threshold(const float* scores, int B, int H, int nq, int nk,
                               float threshold, int use_dense_for_last_block, int apply_tril,
                               uint8_t* mask_out);

/*
 * Cumulative-threshold block mask -- [XA] "block selection (find_blocks_chunked)".  attn_sum
 * (host) fp32 [B, H, nq, nk] holds per (query block, key block) attention weight sums.  Per
 * row: block 0 (the sink) is kept and, when causal, the diagonal block i (if i < nk); the other
 * blocks are visited from the largest weight down (ties: lower column first) and taken while
 * the sum of the weights already taken is below threshold * (row total), so the block whose
 * addition reaches the threshold is taken too.  Sums are in double, left to right.
 * mask_out (host) uint8 [B, H, nq, nk].  NaN weights -> BSATTN_ERR_INVALID_ARG.
 */
int bsattn_mask_from_cumulative_threshold(const float* attn_sum, int B, int H, int nq, int nk,
                                          double threshold, int causal, uint8_t* mask_out);

/*
 * Reads and clears the device status word at the start of `workspace` (device), after
 * synchronising `stream`.  Returns the OR of the BSATTN_ERR_* bits the kernels recorded
 * since the last read (0 = none), or BSATTN_ERR_CUDA if the read itself failed.
 */
int bsattn_get_device_status(void* workspace, void* stream);

/*
 * Budget, in nanoseconds, of every bounded wait inside the kernels launched after this
 * call (default 2e9).  Exists so tests can make a wait expire on purpose and check that
 * the kernel reports BSATTN_ERR_TIMEOUT and leaves the context usable.
 */
void bsattn_set_wait_budget_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* BSATTN_H_ */

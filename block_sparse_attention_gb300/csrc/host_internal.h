// host_internal.h -- helpers shared by the launchers (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsattn {

// Budget of every bounded device wait, set by bsattn_set_wait_budget_ns.
unsigned long long wait_budget_ns();

// Encodes a 3-D tiled TMA descriptor over 16-bit elements (bf16 if `bf16`, else fp16):
// dims {dim0 (innermost), dim1, dim2}, byte strides of dims 1 and 2, box {box0, box1, box2},
// optional 128-byte swizzle, zero fill out of bounds.  Returns a bsattn_status.
int encode_3d(CUtensorMap* map, const void* base, int bf16, uint64_t dim0, uint64_t dim1,
              uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
              uint32_t box1, uint32_t box2, bool swizzle128);

// SM count of the current device (0 if it cannot be queried).
int num_sms_of_current_device();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The 128-row prefill for a 128-token block mask (prefill128.cu).  Arguments are checked by the
// caller; returns BSATTN_ERR_UNSUPPORTED when the mask rows do not fit its shared memory.
int prefill128_launch(const void* q, const void* k, const void* v, const uint8_t* block_mask,
                      int is_causal, void* out, int B, int H, int Sq, int Sk, int d, bool bf16,
                      void* workspace, cudaStream_t stream);

}  // namespace bsattn

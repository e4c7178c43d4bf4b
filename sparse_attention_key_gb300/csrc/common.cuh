// Shared device/host helpers of the Lightning Indexer CUDA library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lightning_indexer.h"

namespace lidx {

constexpr int kHeads = IDX_HEADS;   // 32 indexer heads
constexpr int kDim = IDX_DIM;       // 128 dims per head and per key
constexpr int kTopkMax = IDX_TOPK_MAX;

// ---------------------------------------------------------------------------
// Workspace layout. Every entry point's workspace starts with a 256-byte
// header holding the device status word; regions after it are 256-byte
// aligned.
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;

struct DeviceStatus {
    int32_t code;    // idx_status value: IDX_OK, IDX_ERR_DEVICE_ARG or IDX_ERR_TIMEOUT
    int32_t detail;  // first offending row, or a wait-site code
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record the first error of a call; later errors keep the first one.
__device__ inline void report_error(DeviceStatus* st, int32_t code, int32_t detail) {
    if (atomicCAS(&st->code, 0, code) == 0) atomicExch(&st->detail, detail);
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

// Programmatic dependent launch. Every kernel of this library is launched so
// that it may start while the previous kernel on the stream is finishing; it
// calls pdl_wait() before it reads or writes any global data (this returns
// once every grid it depends on has completed and its writes are visible; at
// once when there is none), then pdl_launch_dependents() so that the next
// kernel may be scheduled in turn. Because each kernel waits before it lets
// the next one start, a kernel's completion implies that of all kernels
// before it on the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Two fp32 -> packed bf16x2 (lo in bits 0..15), round to nearest even: one
// hardware conversion (equal to f32_to_bf16_rn on finite inputs).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
    uint32_t u = __float_as_uint(x);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// Order-preserving map of an fp32 score to uint32: a > b (numerically) iff
// score_key(a) > score_key(b). Adding +0 first turns -0 into +0, so the two
// zeros share one key; then negative values have all bits flipped and
// non-negative ones the sign bit set.
__device__ __forceinline__ uint32_t score_key(float x) {
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// Bins of the first radix digit of the exact top-K (key bits 31..20).
constexpr int kTopkDigit1Bins = 4096;

}  // namespace lidx

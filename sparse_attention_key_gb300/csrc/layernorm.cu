// Key LayerNorm of the Lightning Indexer.
//
// "Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph: indexer keys
// come from the attention input and pass a LayerNorm of width 128 that has a
// weight and a bias. Standard LayerNorm: biased variance, eps inside the square root,
// fp32 arithmetic, bf16 (nearest-even) output for the 16-bit key cache.
//
// HBM-bound: 256 B read + 256 B written per key row. Half a warp per row: each
// of its 16 lanes owns 8 consecutive features (one 16-byte load and store), and
// a warp keeps 4 row pairs in flight (64 bytes per lane outstanding) before
// reducing. Mean and variance are half-warp shuffle reductions (two passes over
// registers). The grid is persistent: 4 blocks of 8 warps per SM. The
// arithmetic runs on packed fp32 pairs (FADD2 / FMUL2 / FFMA2), with a hardware
// rsqrt and packed bf16x2 conversion, to keep the instruction count per row
// low enough that the kernel is bound by memory rather than issue.
#include "common.cuh"
#include "launch.h"
#include "ln_row.cuh"

namespace lidx {

constexpr int kLnWarpsPerBlock = 8;
constexpr int kLnRowsInFlight = 4;   // row pairs per warp per iteration

// kScatter: row r of the output is row slot[r] of y (a key cache of
// `y_rows` rows); slots outside [0, y_rows) (-1 marks padding) write nothing.
template <bool kF32Params, bool kScatter>
__global__ void __launch_bounds__(kLnWarpsPerBlock * 32)
key_layernorm_kernel(const uint4* x, const void* __restrict__ ln_w, const void* __restrict__ ln_b,
                     float eps, uint4* y, int64_t n_rows, const int64_t* __restrict__ slot,
                     int64_t y_rows) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;          // which row of the pair
    const int hl = lane & 15;            // lane within the half-warp: features 8*hl .. 8*hl+7
    float2 g[4], b[4];   // features 8*hl + 2k, 8*hl + 2k + 1
    ln_params_half_warp(ln_w, ln_b, kF32Params, hl, g, b);
    const int64_t warp_id = (int64_t)blockIdx.x * kLnWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * kLnWarpsPerBlock;
    constexpr int kRowsPerIter = 2 * kLnRowsInFlight;
    for (int64_t r0 = warp_id * kRowsPerIter; r0 < n_rows; r0 += n_warps * kRowsPerIter) {
        uint4 v[kLnRowsInFlight];
        int64_t dst[kLnRowsInFlight];
#pragma unroll
        for (int i = 0; i < kLnRowsInFlight; ++i) {   // loads first
            const int64_t row = r0 + 2 * i + half;
            // raw keys are read once: streaming loads (evict first), so the
            // LayerNorm output stays in L2 for a scorer that follows
            v[i] = row < n_rows ? __ldcs(x + row * 16 + hl) : make_uint4(0u, 0u, 0u, 0u);
            dst[i] = row;
            if (kScatter) {
                const int64_t sr = row < n_rows ? __ldg(slot + row) : -1;
                dst[i] = sr >= 0 && sr < y_rows ? sr : -1;
            }
        }
#pragma unroll
        for (int i = 0; i < kLnRowsInFlight; ++i) {
            const int64_t row = r0 + 2 * i + half;
            uint32_t o16[4];
            ln_row_half_warp(v[i], g, b, eps, o16);
            if (row < n_rows && dst[i] >= 0) y[dst[i] * 16 + hl] = make_uint4(o16[0], o16[1], o16[2], o16[3]);
        }
    }
}

cudaError_t launch_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                                 bool f32_params, float eps, uint16_t* k_out, int64_t n_rows,
                                 cudaStream_t stream, const int64_t* slot, int64_t out_rows) {
    const DeviceInfo& dev = device_info();
    constexpr int64_t kRowsPerBlock = kLnWarpsPerBlock * 2 * kLnRowsInFlight;
    const int64_t blocks_needed = (n_rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)dev.sm_count * 4;
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    const uint4* x = reinterpret_cast<const uint4*>(k_raw);
    uint4* y = reinterpret_cast<uint4*>(k_out);
    auto kern = slot != nullptr
                    ? (f32_params ? key_layernorm_kernel<true, true> : key_layernorm_kernel<false, true>)
                    : (f32_params ? key_layernorm_kernel<true, false> : key_layernorm_kernel<false, false>);
    return launch_kernel(kern, dim3(grid), dim3(kLnWarpsPerBlock * 32), 0, stream, 1, x, ln_w, ln_b,
                         eps, y, n_rows, slot, slot != nullptr ? out_rows : n_rows);
}

}  // namespace lidx

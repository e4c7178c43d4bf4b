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
// registers). The grid is persistent: 4 blocks of 8 warps per SM.
#include "common.cuh"
#include "launch.h"

namespace lidx {

constexpr int kLnWarpsPerBlock = 8;
constexpr int kLnRowsInFlight = 4;   // row pairs per warp per iteration

template <bool kF32Params>
__global__ void __launch_bounds__(kLnWarpsPerBlock * 32)
key_layernorm_kernel(const uint4* x, const void* __restrict__ ln_w, const void* __restrict__ ln_b,
                     float eps, uint4* y, int64_t n_rows) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;          // which row of the pair
    const int hl = lane & 15;            // lane within the half-warp: features 8*hl .. 8*hl+7
    float g[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int d = hl * 8 + j;
        if (kF32Params) {
            g[j] = static_cast<const float*>(ln_w)[d];
            b[j] = static_cast<const float*>(ln_b)[d];
        } else {
            g[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(ln_w)[d]) << 16);
            b[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(ln_b)[d]) << 16);
        }
    }
    const int64_t warp_id = (int64_t)blockIdx.x * kLnWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * kLnWarpsPerBlock;
    constexpr int kRowsPerIter = 2 * kLnRowsInFlight;
    for (int64_t r0 = warp_id * kRowsPerIter; r0 < n_rows; r0 += n_warps * kRowsPerIter) {
        uint4 v[kLnRowsInFlight];
#pragma unroll
        for (int i = 0; i < kLnRowsInFlight; ++i) {   // loads first
            const int64_t row = r0 + 2 * i + half;
            v[i] = row < n_rows ? x[row * 16 + hl] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kLnRowsInFlight; ++i) {
            const int64_t row = r0 + 2 * i + half;
            float f[8] = {bf16_lo(v[i].x), bf16_hi(v[i].x), bf16_lo(v[i].y), bf16_hi(v[i].y),
                          bf16_lo(v[i].z), bf16_hi(v[i].z), bf16_lo(v[i].w), bf16_hi(v[i].w)};
            float s = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const float mean = s * (1.0f / kDim);
            float c[8], ss = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = f[j] - mean;
                ss = fmaf(c[j], c[j], ss);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = 1.0f / sqrtf(ss * (1.0f / kDim) + eps);
            uint32_t o16[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o16[j] = f32_to_bf16_rn(fmaf(c[j] * inv, g[j], b[j]));
            if (row < n_rows)
                y[row * 16 + hl] = make_uint4(o16[0] | (o16[1] << 16), o16[2] | (o16[3] << 16),
                                              o16[4] | (o16[5] << 16), o16[6] | (o16[7] << 16));
        }
    }
}

cudaError_t launch_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                                 bool f32_params, float eps, uint16_t* k_out, int64_t n_rows,
                                 cudaStream_t stream) {
    const DeviceInfo& dev = device_info();
    constexpr int64_t kRowsPerBlock = kLnWarpsPerBlock * 2 * kLnRowsInFlight;
    const int64_t blocks_needed = (n_rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)dev.sm_count * 4;
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    const uint4* x = reinterpret_cast<const uint4*>(k_raw);
    uint4* y = reinterpret_cast<uint4*>(k_out);
    if (f32_params)
        key_layernorm_kernel<true><<<grid, kLnWarpsPerBlock * 32, 0, stream>>>(x, ln_w, ln_b, eps, y,
                                                                              n_rows);
    else
        key_layernorm_kernel<false><<<grid, kLnWarpsPerBlock * 32, 0, stream>>>(x, ln_w, ln_b, eps, y,
                                                                               n_rows);
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

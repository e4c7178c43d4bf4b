// Key LayerNorm of the Lightning Indexer.
//
// "Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph: indexer keys
// come from the attention input and pass a LayerNorm of width 128 that has a
// weight and a bias. Standard LayerNorm: biased variance, eps inside the square root,
// fp32 arithmetic, bf16 (nearest-even) output for the 16-bit key cache.
//
// HBM-bound: 256 B read + 256 B written per key row. One warp per row; each
// lane owns 4 consecutive features (one 8-byte load and store), so a warp
// moves a whole 256-byte row per instruction. The grid is a multiple of the
// SM count and strides over rows.
#include "common.cuh"
#include "launch.h"

namespace lidx {

constexpr int kLnWarpsPerBlock = 8;

template <bool kF32Params>
__global__ void __launch_bounds__(kLnWarpsPerBlock * 32)
key_layernorm_kernel(const uint2* x, const void* __restrict__ ln_w,
                     const void* __restrict__ ln_b, float eps, uint2* y,
                     int64_t n_rows) {
    const int lane = threadIdx.x & 31;
    float g[4], b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int d = lane * 4 + j;
        if (kF32Params) {
            g[j] = static_cast<const float*>(ln_w)[d];
            b[j] = static_cast<const float*>(ln_b)[d];
        } else {
            g[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(ln_w)[d]) << 16);
            b[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(ln_b)[d]) << 16);
        }
    }
    const int64_t warps = (int64_t)gridDim.x * kLnWarpsPerBlock;
    for (int64_t row = (int64_t)blockIdx.x * kLnWarpsPerBlock + (threadIdx.x >> 5); row < n_rows;
         row += warps) {
        const uint2 v = x[row * 32 + lane];
        float f[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
        float s = (f[0] + f[1]) + (f[2] + f[3]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float mean = s * (1.0f / kDim);
        float c[4], ss = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c[j] = f[j] - mean;
            ss = fmaf(c[j], c[j], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float var = ss * (1.0f / kDim);
        const float inv = 1.0f / sqrtf(var + eps);
        uint16_t o16[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o16[j] = f32_to_bf16_rn(fmaf(c[j] * inv, g[j], b[j]));
        uint2 out;
        out.x = uint32_t(o16[0]) | (uint32_t(o16[1]) << 16);
        out.y = uint32_t(o16[2]) | (uint32_t(o16[3]) << 16);
        y[row * 32 + lane] = out;
    }
}

cudaError_t launch_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                                 bool f32_params, float eps, uint16_t* k_out, int64_t n_rows,
                                 cudaStream_t stream) {
    const DeviceInfo& dev = device_info();
    const int64_t blocks_needed = (n_rows + kLnWarpsPerBlock - 1) / kLnWarpsPerBlock;
    const int64_t cap = (int64_t)dev.sm_count * 8;  // 8 blocks (64 warps) per SM
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    if (f32_params)
        key_layernorm_kernel<true><<<grid, kLnWarpsPerBlock * 32, 0, stream>>>(
            reinterpret_cast<const uint2*>(k_raw), ln_w, ln_b, eps, reinterpret_cast<uint2*>(k_out),
            n_rows);
    else
        key_layernorm_kernel<false><<<grid, kLnWarpsPerBlock * 32, 0, stream>>>(
            reinterpret_cast<const uint2*>(k_raw), ln_w, ln_b, eps, reinterpret_cast<uint2*>(k_out),
            n_rows);
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

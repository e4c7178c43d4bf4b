// The key LayerNorm of one 128-wide row by a half warp, shared by the
// LayerNorm kernels (layernorm.cu) and the projections' finishing kernel
// (project.cu), so that both give the same bits.
//
// "Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph: keys pass a
// 128-wide LayerNorm with a weight and a bias. Biased variance, eps inside the
// square root, fp32 arithmetic on packed pairs, bf16 (nearest-even) output.
#pragma once

#include "common.cuh"

namespace lidx {

// Lane hl (0..15) of a half warp holds features 8*hl .. 8*hl+7 of the row as
// four packed bf16 pairs (x), and the matching LayerNorm weights g and biases
// b as float pairs (features 8*hl + 2k, 8*hl + 2k + 1). Writes the lane's 8
// outputs as four packed bf16 pairs. Both half warps of a warp call it
// together (shuffles span 16 lanes).
__device__ __forceinline__ void ln_row_half_warp(const uint4& x, const float2 (&g)[4],
                                                 const float2 (&b)[4], float eps, uint32_t (&o16)[4]) {
    const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
    float2 f[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) f[k] = make_float2(bf16_lo(wv[k]), bf16_hi(wv[k]));
    const float2 s2 = __fadd2_rn(__fadd2_rn(f[0], f[1]), __fadd2_rn(f[2], f[3]));
    float s = s2.x + s2.y;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s * (1.0f / kDim);
    const float2 nm = make_float2(-mean, -mean);
    float2 c[4];
    float2 q = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        c[k] = __fadd2_rn(f[k], nm);
        q = __ffma2_rn(c[k], c[k], q);
    }
    float ss = q.x + q.y;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(fmaf(ss, 1.0f / kDim, eps));
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 o = __ffma2_rn(__fmul2_rn(c[k], inv2), g[k], b[k]);
        o16[k] = f32x2_to_bf16x2_rn(o.x, o.y);
    }
}

// LayerNorm weight and bias pairs of lane hl (features 8*hl .. 8*hl+7).
__device__ __forceinline__ void ln_params_half_warp(const void* ln_w, const void* ln_b, bool f32,
                                                    int hl, float2 (&g)[4], float2 (&b)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int d = hl * 8 + 2 * k;
        if (f32) {
            g[k] = make_float2(static_cast<const float*>(ln_w)[d], static_cast<const float*>(ln_w)[d + 1]);
            b[k] = make_float2(static_cast<const float*>(ln_b)[d], static_cast<const float*>(ln_b)[d + 1]);
        } else {
            const uint16_t* w16 = static_cast<const uint16_t*>(ln_w);
            const uint16_t* b16 = static_cast<const uint16_t*>(ln_b);
            g[k] = make_float2(__uint_as_float(uint32_t(w16[d]) << 16), __uint_as_float(uint32_t(w16[d + 1]) << 16));
            b[k] = make_float2(__uint_as_float(uint32_t(b16[d]) << 16), __uint_as_float(uint32_t(b16[d + 1]) << 16));
        }
    }
}

}  // namespace lidx

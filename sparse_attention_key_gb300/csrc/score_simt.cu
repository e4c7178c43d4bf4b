// CUDA-core scorer of the Lightning Indexer.
//
//   S[t,s] = sum_h w[t,h] * max(q[t,h,:] . k[s,:], 0)     for s < n(t) = q_pos[t] + 1
//
// ("Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph; no rotary,
// item (3) of its list.)
//
// One block = one query x 128 consecutive keys; one thread = one key. The
// query's 32x128 block is staged once in shared memory as fp32 and read back
// as warp-wide broadcasts; each thread holds its key row (256 B, sixteen
// 16-byte loads) as 128 fp32 registers and runs the 32 dot products. The
// accumulation order per head is the d order, fp32 FMA.
//
// This kernel is bound by the fp32 FMA rate (4096 FMAs per key), which caps it
// near a third of HBM bandwidth on decode; the tensor-core scorer replaces it
// on the hot path. It stays as the reference-free baseline for that ceiling.
#include "common.cuh"
#include "launch.h"

namespace lidx {

constexpr int kSimtKeys = 128;  // keys per block (one per thread)

__device__ __forceinline__ int find_sequence(const int32_t* cu_q, int B, int t) {
    // largest b with cu_q[b] <= t (cu_q non-decreasing, cu_q[0] = 0, cu_q[B] = T)
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kSimtKeys)
score_simt_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                  const float* __restrict__ w, const int32_t* __restrict__ q_pos,
                  const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B,
                  int T, int64_t n_keys, int64_t max_len, float* __restrict__ scores, int64_t ld,
                  DeviceStatus* status) {
    __shared__ __align__(16) float qs[kHeads * kDim];  // 16 KB
    __shared__ float ws[kHeads];

    const int64_t s0 = (int64_t)blockIdx.x * kSimtKeys;
    for (int t = blockIdx.y; t < T; t += gridDim.y) {
        const int b = find_sequence(cu_q, B, t);
        const int64_t key0 = __ldg(cu_k + b);
        const int64_t len_k = (int64_t)__ldg(cu_k + b + 1) - key0;
        const int64_t n = (int64_t)__ldg(q_pos + t) + 1;
        if (n < 1 || n > len_k || n > max_len || key0 < 0 || key0 + len_k > n_keys) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report_error(status, IDX_ERR_DEVICE_ARG, t);
            continue;
        }
        if (s0 >= n) continue;  // block-uniform

        __syncthreads();  // previous query's qs reads are done
        const uint4* qv = reinterpret_cast<const uint4*>(q + (int64_t)t * kHeads * kDim);
        for (int i = threadIdx.x; i < kHeads * kDim / 8; i += kSimtKeys) {
            const uint4 v = __ldg(qv + i);
            float4* dst = reinterpret_cast<float4*>(qs + i * 8);
            dst[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
            dst[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
        }
        if (threadIdx.x < kHeads) ws[threadIdx.x] = __ldg(w + (int64_t)t * kHeads + threadIdx.x);
        __syncthreads();

        const int64_t s = s0 + threadIdx.x;
        if (s < n) {
            float kf[kDim];
            const uint4* kv = reinterpret_cast<const uint4*>(k + (key0 + s) * kDim);
#pragma unroll
            for (int i = 0; i < kDim / 8; ++i) {
                const uint4 v = __ldg(kv + i);
                kf[i * 8 + 0] = bf16_lo(v.x);
                kf[i * 8 + 1] = bf16_hi(v.x);
                kf[i * 8 + 2] = bf16_lo(v.y);
                kf[i * 8 + 3] = bf16_hi(v.y);
                kf[i * 8 + 4] = bf16_lo(v.z);
                kf[i * 8 + 5] = bf16_hi(v.z);
                kf[i * 8 + 6] = bf16_lo(v.w);
                kf[i * 8 + 7] = bf16_hi(v.w);
            }
            float S = 0.f;
#pragma unroll 1
            for (int h = 0; h < kHeads; ++h) {
                const float4* qh = reinterpret_cast<const float4*>(qs + h * kDim);
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < kDim / 4; ++i) {
                    const float4 qq = qh[i];
                    dot = fmaf(qq.x, kf[4 * i + 0], dot);
                    dot = fmaf(qq.y, kf[4 * i + 1], dot);
                    dot = fmaf(qq.z, kf[4 * i + 2], dot);
                    dot = fmaf(qq.w, kf[4 * i + 3], dot);
                }
                S = fmaf(ws[h], fmaxf(dot, 0.f), S);
            }
            scores[(int64_t)t * ld + s] = S;
        }
    }
}

cudaError_t launch_score_simt(const ScoreArgs& a, cudaStream_t stream) {
    const int64_t tiles = (a.max_len + kSimtKeys - 1) / kSimtKeys;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    dim3 grid((unsigned)tiles, (unsigned)(a.T < 65535 ? a.T : 65535));
    score_simt_kernel<<<grid, kSimtKeys, 0, stream>>>(a.q, a.k, a.w, a.q_pos, a.cu_q, a.cu_k, a.B,
                                                      a.T, a.n_keys, a.max_len, a.scores, a.ld,
                                                      a.status);
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

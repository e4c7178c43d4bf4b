// Exact top-K of each score row with the tie/order rule of the Lightning Indexer.
//
// "Notes from an NVFP4 port of Kimi K3.1 Pro": the selection of the top 2048
// positions is exact (indexer paragraph); scores equal to the threshold at the
// K boundary form a tie group, and the output gives the kept above-threshold
// positions by increasing position, then the kept part of the tie group by
// increasing position from its lowest (item (4) of "Details that silently
// change the answer"); a history of K or fewer keys keeps every position
// (closing paragraph).
//
// Per row (one 1024-thread block):
//   1. n <= K: emit 0..n-1, pad with -1.
//   2. Radix select of the K-th largest key over order-preserving uint32 keys of
//      the fp32 scores (-0 folded onto +0), most significant digit first, digits
//      of 11/11/10 bits. Each pass builds a shared-memory histogram of the
//      elements that match the digits chosen so far; lanes of a warp that hit
//      the same bin are merged with a match-any vote so ties cost one atomic.
//      After the last pass the threshold tau is exact, count_above = #(key >
//      tau) and need = K - count_above.
//   3. Stable compaction: one ordered sweep in chunks of 4096 positions; a block
//      scan gives each thread its offsets into the "above" list and into the tie
//      list; ties past `need` are dropped. The sweep stops once both lists are
//      complete.
// Rows that fit in shared memory are read from global memory once (pass 1 runs
// on the way in); longer rows are re-read (from L2) by each pass.
#include "common.cuh"
#include "launch.h"

namespace lidx {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kBins = 2048;                 // 11-bit digit
constexpr int kChunk = kTopkThreads * 4;    // compaction chunk (4 positions per thread)

struct TopkShared {
    uint32_t hist[kBins];
    uint32_t warp_tot[kTopkWarps];
    uint32_t sel_bin;
    uint32_t sel_rank;
};

// Add the elements of `u` that match (prefix, mask) into hist[(u >> shift) & (bins-1)].
// All 32 lanes of the warp must call this together.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t u, bool valid, uint32_t prefix,
                                         uint32_t mask, int shift, uint32_t bin_mask) {
    const bool match = valid && ((u & mask) == prefix);
    const uint32_t bin = match ? ((u >> shift) & bin_mask) : 0xFFFFFFFFu;
    if (__any_sync(0xffffffffu, match)) {
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        const int lane = threadIdx.x & 31;
        if (match && (__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], __popc(peers));
    }
}

// Warp 0 finds the bin (scanning from the top) holding the rank-`rank` element
// (1-based from the largest). Writes sel_bin and the rank inside that bin.
__device__ __forceinline__ void find_bin(TopkShared& sh, int nbins, uint32_t rank) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int per = nbins / 32;               // bins per lane, lane 0 owns the top ones
    const int top = nbins - 1 - lane * per;   // this lane's highest bin
    uint32_t sum = 0;
    for (int i = 0; i < per; ++i) sum += sh.hist[top - i];
    // exclusive prefix over lanes (lane 0 first = largest bins)
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - sum;
    if (excl < rank && rank <= incl) {        // exactly one lane
        uint32_t acc = excl;
        for (int i = 0; i < per; ++i) {
            const uint32_t c = sh.hist[top - i];
            if (acc + c >= rank) {
                sh.sel_bin = (uint32_t)(top - i);
                sh.sel_rank = rank - acc;
                break;
            }
            acc += c;
        }
    }
}

__device__ __forceinline__ void zero_hist(TopkShared& sh) {
    for (int i = threadIdx.x; i < kBins; i += kTopkThreads) sh.hist[i] = 0;
}

// Exclusive block scan of one packed counter per thread; returns the exclusive
// prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(TopkShared& sh, uint32_t v,
                                                         uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) sh.warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t wt = sh.warp_tot[lane];
        uint32_t wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        sh.warp_tot[lane] = wi - wt;  // exclusive warp offsets
        if (lane == 31) sh.sel_rank = wi;  // reuse as the block total
    }
    __syncthreads();
    const uint32_t res = sh.warp_tot[warp] + incl - v;
    *total = sh.sel_rank;
    __syncthreads();  // warp_tot / sel_rank are reused by the next call
    return res;
}

template <bool kRowInSmem>
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
            bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
            int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
            const int32_t* __restrict__ cu_k, int B) {
    __shared__ TopkShared sh;
    extern __shared__ __align__(16) uint32_t row_keys[];  // used when kRowInSmem

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int64_t n = (int64_t)__ldg(n_valid + t) + (n_from_pos ? 1 : 0);
        int32_t* out = idx + (int64_t)t * K;
        bool bad = n < 0 || n > max_len || n > ld;
        if (cu_q != nullptr) {  // fused call: the row must lie inside its sequence
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
            }
            const int64_t len_k = (int64_t)__ldg(cu_k + lo + 1) - __ldg(cu_k + lo);
            bad = bad || n < 1 || n > len_k;
        }
        if (bad) {
            if (threadIdx.x == 0) report_error(status, IDX_ERR_DEVICE_ARG, t);
            for (int i = threadIdx.x; i < K; i += kTopkThreads) out[i] = -1;
            if (cnt && threadIdx.x == 0) cnt[t] = 0;
            continue;
        }
        if (n <= K) {  // dormant selection
            for (int i = threadIdx.x; i < K; i += kTopkThreads) out[i] = i < n ? i : -1;
            if (cnt && threadIdx.x == 0) cnt[t] = (int32_t)n;
            continue;
        }
        const float* row = scores + (int64_t)t * ld;
        const float4* row4 = reinterpret_cast<const float4*>(row);

        // ---- pass 1: top 11 bits (fused with the staging copy when the row fits)
        __syncthreads();
        zero_hist(sh);
        __syncthreads();
        for (int64_t base = 0; base < n; base += kChunk) {
            const int64_t i = base + 4 * threadIdx.x;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i + 3 < n) v = __ldg(row4 + (i >> 2));
            else if (i < n) {
                v.x = row[i];
                if (i + 1 < n) v.y = row[i + 1];
                if (i + 2 < n) v.z = row[i + 2];
            }
            const uint32_t u[4] = {score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w)};
            if (kRowInSmem && i < n) {
                if (i + 3 < n) *reinterpret_cast<uint4*>(row_keys + i) = make_uint4(u[0], u[1], u[2], u[3]);
                else for (int j = 0; j < 4 && i + j < n; ++j) row_keys[i + j] = u[j];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) hist_add(sh.hist, u[j], i + j < n, 0u, 0u, 21, kBins - 1);
        }
        __syncthreads();
        find_bin(sh, kBins, (uint32_t)K);
        __syncthreads();
        uint32_t prefix = sh.sel_bin << 21;
        uint32_t mask = 0xFFE00000u;
        uint32_t rank = sh.sel_rank;

        // ---- passes 2 and 3: bits 20..10, then 9..0, among matching elements
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 10 : 0;
            const int nbins = pass == 0 ? 2048 : 1024;
            __syncthreads();
            zero_hist(sh);
            __syncthreads();
            for (int64_t base = 0; base < n; base += kChunk) {
                const int64_t i = base + 4 * threadIdx.x;
                uint32_t u[4] = {0u, 0u, 0u, 0u};
                if (kRowInSmem) {
                    if (i + 3 < n) {
                        const uint4 x = *reinterpret_cast<const uint4*>(row_keys + i);
                        u[0] = x.x; u[1] = x.y; u[2] = x.z; u[3] = x.w;
                    } else {
                        for (int j = 0; j < 4; ++j) if (i + j < n) u[j] = row_keys[i + j];
                    }
                } else {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (i + 3 < n) v = __ldg(row4 + (i >> 2));
                    else if (i < n) {
                        v.x = row[i];
                        if (i + 1 < n) v.y = row[i + 1];
                        if (i + 2 < n) v.z = row[i + 2];
                    }
                    u[0] = score_key(v.x); u[1] = score_key(v.y);
                    u[2] = score_key(v.z); u[3] = score_key(v.w);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    hist_add(sh.hist, u[j], i + j < n, prefix, mask, shift, (uint32_t)nbins - 1);
            }
            __syncthreads();
            find_bin(sh, nbins, rank);
            __syncthreads();
            prefix |= sh.sel_bin << shift;
            mask |= (uint32_t)(nbins - 1) << shift;
            rank = sh.sel_rank;
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;                     // members of the tie group to keep
        const uint32_t n_above = (uint32_t)K - need;    // every key > tau is kept

        // ---- stable compaction in position order
        uint32_t done_above = 0, done_tie = 0;
        for (int64_t base = 0; base < n; base += kChunk) {
            const int64_t i = base + 4 * threadIdx.x;
            uint32_t u[4] = {0u, 0u, 0u, 0u};
            if (kRowInSmem) {
                if (i + 3 < n) {
                    const uint4 x = *reinterpret_cast<const uint4*>(row_keys + i);
                    u[0] = x.x; u[1] = x.y; u[2] = x.z; u[3] = x.w;
                } else {
                    for (int j = 0; j < 4; ++j) if (i + j < n) u[j] = row_keys[i + j];
                }
            } else {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i + 3 < n) v = __ldg(row4 + (i >> 2));
                else if (i < n) {
                    v.x = row[i];
                    if (i + 1 < n) v.y = row[i + 1];
                    if (i + 2 < n) v.z = row[i + 2];
                }
                u[0] = score_key(v.x); u[1] = score_key(v.y);
                u[2] = score_key(v.z); u[3] = score_key(v.w);
            }
            uint32_t a = 0, e = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = i + j < n;
                a += (ok && u[j] > tau) ? 1u : 0u;
                e += (ok && u[j] == tau) ? 1u : 0u;
            }
            uint32_t total;
            const uint32_t off = block_exclusive_scan(sh, a | (e << 16), &total);
            uint32_t pa = done_above + (off & 0xFFFFu);
            uint32_t pe = done_tie + (off >> 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = i + j < n;
                if (ok && u[j] > tau) out[pa++] = (int32_t)(i + j);
                else if (ok && u[j] == tau) {
                    if (pe < need) out[n_above + pe] = (int32_t)(i + j);
                    ++pe;
                }
            }
            done_above += total & 0xFFFFu;
            done_tie += total >> 16;
            if (done_above >= n_above && done_tie >= need) break;  // block-uniform
        }
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

// Largest row (in elements) staged in shared memory.
static int64_t smem_row_cap(const DeviceInfo& dev) {
    const int64_t avail = (int64_t)dev.max_smem_optin - (int64_t)sizeof(TopkShared) - 1024;
    return avail > 0 ? avail / 4 : 0;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
    const DeviceInfo& dev = device_info();
    const int64_t row_cap = a.max_len < a.ld ? a.max_len : a.ld;
    const int64_t padded = align_up((size_t)row_cap, 4);
    const int grid = a.T < dev.sm_count * 64 ? a.T : dev.sm_count * 64;
    if (grid <= 0) return cudaSuccess;
    if (padded <= smem_row_cap(dev)) {
        const size_t smem = (size_t)padded * 4;
        cudaError_t e = ensure_smem_optin((const void*)topk_kernel<true>, smem_row_cap(dev) * 4);
        if (e != cudaSuccess) return e;
        topk_kernel<true><<<grid, kTopkThreads, smem, stream>>>(a.scores, a.ld, a.n_valid,
                                                                a.n_from_pos, a.T, a.max_len,
                                                                a.topk, a.idx, a.cnt, a.status,
                                                                a.cu_q, a.cu_k, a.B);
    } else {
        topk_kernel<false><<<grid, kTopkThreads, 0, stream>>>(a.scores, a.ld, a.n_valid,
                                                              a.n_from_pos, a.T, a.max_len,
                                                              a.topk, a.idx, a.cnt, a.status,
                                                                a.cu_q, a.cu_k, a.B);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

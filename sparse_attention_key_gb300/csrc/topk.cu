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
// Scores become order-preserving uint32 keys (-0 folded onto +0). The K-th
// largest key tau is found by most-significant-digit radix select over three
// digits: bits 31..(32-D1), (31-D1)..10 and 9..0. One block per row, with the
// row's positions tracked in bitmaps (one bit per position):
//
//   pass A   histogram of the first digit; the bin b1 holding rank K (counted
//            from the top) follows.
//   split    positions whose first digit is above b1 are certainly kept (fewer
//            than K of them) -> "above" bits; positions in bin b1 are the
//            candidates -> "cand" bits (set as 4-bit masks, one per thread and
//            4-position vector).
//   digits   2 and 3 are histogrammed over the candidates only -> tau, and
//            need = the number of tau-valued keys kept.
//   mark     candidates above tau join the "above" bits, candidates equal to
//            tau get "tie" bits.
//   emit     one ordered scan of the bitmaps (each thread owns a contiguous word
//            range; a block scan of packed bit counts gives offsets): all above
//            positions in increasing order, then the first `need` tie positions
//            in increasing order.
// Short rows (staged kernel) are copied into shared memory as keys during pass
// A; every later step reads that copy. Long rows (streamed kernel) are read
// twice from global memory (pass A and the split); the candidates' keys are
// gathered from global memory again where needed. No block waits on another.
#include "common.cuh"
#include "launch.h"

namespace lidx {

namespace {

constexpr int kD3Bits = 10;                 // last digit: bits 9..0
constexpr int kStagedThreads = 256;
constexpr int kStreamThreads = 512;         // two blocks per SM overlap their phases
constexpr int64_t kStageCap = 12288;        // longest row staged in shared memory
constexpr int kUnroll = 4;                  // independent 16-byte loads per thread in flight
constexpr int kScratchBlocks = 512;         // blocks when the bitmaps live in global scratch

template <int THREADS, int D1BITS>
struct TopkSmem {
    static constexpr int kWarps = THREADS / 32;
    uint32_t hist[1 << D1BITS];
    uint32_t scan[THREADS / 32 + 1];
    uint64_t scan64[THREADS / 32];
    uint32_t sel_bin, sel_rank, cand_count;
};

// Exclusive block scan of one value per thread (sh.scan as scratch).
template <int THREADS, class S>
__device__ __forceinline__ uint32_t block_excl_scan(S& sh, uint32_t v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    __syncthreads();   // sh.scan may still be read after a previous scan
    if (lane == 31) sh.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t x0 = lane < S::kWarps ? sh.scan[lane] : 0u;
        uint32_t wi = x0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        if (lane < S::kWarps) sh.scan[lane] = wi - x0;
    }
    __syncthreads();
    return sh.scan[warp] + incl - v;
}

// Exclusive block scan of one 64-bit value per thread (sh.scan64 as scratch).
template <int THREADS, class S>
__device__ __forceinline__ uint64_t block_excl_scan64(S& sh, uint64_t v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    __syncthreads();
    if (lane == 31) sh.scan64[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint64_t x0 = lane < S::kWarps ? sh.scan64[lane] : 0ull;
        uint64_t wi = x0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        if (lane < S::kWarps) sh.scan64[lane] = wi - x0;
    }
    __syncthreads();
    return sh.scan64[warp] + incl - v;
}

// The bin (counting from the highest) holding the element of rank `rank`
// (1-based from the largest) in hist[0..nbins); writes sh.sel_bin and the rank
// inside that bin to sh.sel_rank.
template <int THREADS, class S>
__device__ __forceinline__ void select_bin(S& sh, int nbins, uint32_t rank) {
    const int per = (nbins + THREADS - 1) / THREADS;       // bins per thread
    const int hi = nbins - 1 - (int)threadIdx.x * per;     // this thread's highest bin
    uint32_t sum = 0;
    for (int i = 0; i < per; ++i)
        if (hi - i >= 0) sum += sh.hist[hi - i];
    const uint32_t excl = block_excl_scan<THREADS>(sh, sum);
    if (excl < rank && rank <= excl + sum) {   // exactly one thread
        uint32_t acc = excl;
        for (int i = 0; i < per; ++i) {
            const uint32_t c = sh.hist[hi - i];
            if (acc + c >= rank) {
                sh.sel_bin = (uint32_t)(hi - i);
                sh.sel_rank = rank - acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

template <int THREADS>
__device__ __forceinline__ void zero(uint32_t* p, int64_t n) {
    for (int64_t i = threadIdx.x; i < n; i += THREADS) p[i] = 0;
}

// Order-preserving key of a score: a > b (numerically) iff fkey(a) > fkey(b).
// Adding +0 turns -0 into +0 first, so the two zeros share one key.
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// Keys of the 4 scores of vector v (elements 4v..4v+3) of a row, from global.
__device__ __forceinline__ uint4 gkeys(const float* row, int32_t v) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(row) + v);
    return make_uint4(fkey(x.x), fkey(x.y), fkey(x.z), fkey(x.w));
}

__device__ __forceinline__ uint32_t comp(const uint4& k, int j) {
    return j == 0 ? k.x : j == 1 ? k.y : j == 2 ? k.z : k.w;
}

__device__ __forceinline__ void set_bit(uint32_t* bits, int64_t pos) {
    atomicOr(bits + (pos >> 5), 1u << (pos & 31));
}

// Ordered output from the two bitmaps: the set positions of `above` in
// increasing order to out[0..n_above), then the first `need` set positions of
// `tie` in increasing order to out[n_above..). Each thread owns a contiguous
// range of words; one block scan of packed (above, tie) counts gives offsets.
template <int THREADS, class S>
__device__ __forceinline__ void emit_ordered(S& sh, const uint32_t* above, const uint32_t* tie,
                                             int32_t nw, int32_t* out, uint32_t n_above,
                                             uint32_t need) {
    const int32_t per = (nw + THREADS - 1) / THREADS;
    const int32_t w0 = threadIdx.x * per;
    const int32_t w1 = w0 + per < nw ? w0 + per : nw;
    uint32_t ca = 0, ct = 0;
    for (int32_t w = w0; w < w1; ++w) {
        ca += __popc(above[w]);
        ct += __popc(tie[w]);
    }
    ct = ct < need ? ct : need;   // ties past `need` are never emitted
    const uint64_t off = block_excl_scan64<THREADS>(sh, (uint64_t)ca | ((uint64_t)ct << 32));
    uint32_t pa = (uint32_t)off, pt = (uint32_t)(off >> 32);
    for (int32_t w = w0; w < w1; ++w) {
        uint32_t m = above[w];
        while (m) {
            out[pa++] = w * 32 + (__ffs(m) - 1);
            m &= m - 1u;
        }
        m = tie[w];
        while (m && pt < need) {
            out[n_above + pt++] = w * 32 + (__ffs(m) - 1);
            m &= m - 1u;
        }
    }
}

// Row checks shared by both kernels. Returns the row length, or -1 after
// writing the output of a bad row (-1s, cnt 0, status) or of a row that keeps
// every position (n <= K).
template <int THREADS>
__device__ __forceinline__ int64_t row_prologue(int t, const int32_t* __restrict__ n_valid,
                                                bool n_from_pos, int64_t max_len, int64_t ld,
                                                int K, int32_t* out, int32_t* __restrict__ cnt,
                                                DeviceStatus* status,
                                                const int32_t* __restrict__ cu_q,
                                                const int32_t* __restrict__ cu_k, int B) {
    const int64_t n = (int64_t)__ldg(n_valid + t) + (n_from_pos ? 1 : 0);
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
        for (int i = threadIdx.x; i < K; i += THREADS) out[i] = -1;
        if (cnt && threadIdx.x == 0) cnt[t] = 0;
        return -1;
    }
    if (n <= K) {  // dormant selection: every position
        for (int i = threadIdx.x; i < K; i += THREADS) out[i] = i < n ? i : -1;
        if (cnt && threadIdx.x == 0) cnt[t] = (int32_t)n;
        return -1;
    }
    return n;
}

// ---------------------------------------------------------------------------
// Short rows: staged in shared memory as keys.
// ---------------------------------------------------------------------------
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 4)
topk_staged_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                   bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
                   int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ cu_k, int B, int32_t stage_cap) {
    constexpr int D1 = 11;                      // digits: bits 31..21, 20..10, 9..0
    constexpr int kD1Shift = 32 - D1;
    using S = TopkSmem<THREADS, D1>;
    __shared__ S sh;
    // dynamic: keys[stage_cap] | above[nw_cap] | tie[nw_cap]
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t* keys = dyn;
    const int32_t nw_cap = (stage_cap + 31) >> 5;
    uint32_t* above = dyn + stage_cap;
    uint32_t* tie = above + nw_cap;

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int32_t* out = idx + (int64_t)t * K;
        const int64_t n64 = row_prologue<THREADS>(t, n_valid, n_from_pos, max_len, ld, K, out, cnt,
                                                  status, cu_q, cu_k, B);
        if (n64 < 0) continue;
        const int32_t n = (int32_t)n64;
        const int32_t nvec = n >> 2, tail0 = nvec << 2;
        const int32_t nw = (n + 31) >> 5;
        const float* row = scores + (int64_t)t * ld;

        // ---- pass A: stage keys, first digit
        __syncthreads();
        zero<THREADS>(sh.hist, 1 << D1);
        zero<THREADS>(above, nw);
        zero<THREADS>(tie, nw);
        __syncthreads();
        for (int32_t vb = 0; vb < nvec; vb += kUnroll * THREADS) {
            uint4 k[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {   // loads first
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v < nvec) k[u] = gkeys(row, v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v >= nvec) break;
                reinterpret_cast<uint4*>(keys)[v] = k[u];
                atomicAdd(&sh.hist[k[u].x >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].y >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].z >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].w >> kD1Shift], 1u);
            }
        }
        if (threadIdx.x < n - tail0) {
            const uint32_t kk = fkey(__ldg(row + tail0 + threadIdx.x));
            keys[tail0 + threadIdx.x] = kk;
            atomicAdd(&sh.hist[kk >> kD1Shift], 1u);
        }
        __syncthreads();
        select_bin<THREADS>(sh, 1 << D1, (uint32_t)K);
        uint32_t prefix = sh.sel_bin << kD1Shift;
        uint32_t rank = sh.sel_rank;

        // ---- digits 2 and 3 among the keys that match the digits so far
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? kD3Bits : 0;
            const int bits = d == 0 ? 22 - D1 : kD3Bits;
            const uint32_t mask_hi = d == 0 ? (0xFFFFFFFFu << kD1Shift) : (0xFFFFFFFFu << kD3Bits);
            const uint32_t bin_mask = (1u << bits) - 1u;
            __syncthreads();
            zero<THREADS>(sh.hist, 1 << bits);
            __syncthreads();
            auto add = [&](uint32_t kk) {
                if ((kk & mask_hi) == prefix) atomicAdd(&sh.hist[(kk >> shift) & bin_mask], 1u);
            };
            for (int32_t v = threadIdx.x; v < nvec; v += THREADS) {
                const uint4 k = reinterpret_cast<const uint4*>(keys)[v];
                add(k.x); add(k.y); add(k.z); add(k.w);
            }
            if (threadIdx.x < n - tail0) add(keys[tail0 + threadIdx.x]);
            __syncthreads();
            select_bin<THREADS>(sh, 1 << bits, rank);
            prefix |= sh.sel_bin << shift;
            rank = sh.sel_rank;
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;                   // tau-valued keys kept
        const uint32_t n_above = (uint32_t)K - need;  // every key above tau is kept

        // ---- mark: one thread per 32-position word, no atomics
        for (int32_t w = threadIdx.x; w < nw; w += THREADS) {
            uint32_t a = 0, e = 0;
            const int32_t p0 = w << 5;
            const int32_t m = n - p0 < 32 ? n - p0 : 32;
            for (int32_t b = 0; b < m; ++b) {
                const uint32_t kk = keys[p0 + b];
                a |= (kk > tau ? 1u : 0u) << b;
                e |= (kk == tau ? 1u : 0u) << b;
            }
            above[w] = a;
            tie[w] = e;
        }
        __syncthreads();

        // ---- emit: above positions ascending, then the first `need` ties ascending
        emit_ordered<THREADS>(sh, above, tie, nw, out, n_above, need);
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

// ---------------------------------------------------------------------------
// Long rows: streamed from global memory (L2), bitmaps in shared memory, or in
// per-block global scratch when a row's bitmaps do not fit.
// ---------------------------------------------------------------------------
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 2)
topk_stream_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                   bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
                   int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ cu_k, int B, int64_t nw_cap,
                   uint32_t* __restrict__ gbits) {
    constexpr int D1 = 12;                      // digits: bits 31..20, 19..10, 9..0
    constexpr int kD1Shift = 32 - D1;
    using S = TopkSmem<THREADS, D1>;
    __shared__ S sh;
    extern __shared__ __align__(16) uint32_t dyn[];   // above | tie | cand bitmaps
    uint32_t* above = gbits ? gbits + (int64_t)blockIdx.x * 3 * nw_cap : dyn;
    uint32_t* tie = above + nw_cap;
    uint32_t* cand = tie + nw_cap;

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int32_t* out = idx + (int64_t)t * K;
        const int64_t n64 = row_prologue<THREADS>(t, n_valid, n_from_pos, max_len, ld, K, out, cnt,
                                                  status, cu_q, cu_k, B);
        if (n64 < 0) continue;
        const int32_t n = (int32_t)n64;
        const int32_t nvec = n >> 2, tail0 = nvec << 2;
        const int32_t nw = (n + 31) >> 5;
        const float* row = scores + (int64_t)t * ld;

        // ---- pass A: first digit
        __syncthreads();
        zero<THREADS>(sh.hist, 1 << D1);
        zero<THREADS>(above, nw);
        zero<THREADS>(tie, nw);
        zero<THREADS>(cand, nw);
        __syncthreads();
        for (int32_t vb = 0; vb < nvec; vb += kUnroll * THREADS) {
            uint4 k[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v < nvec) k[u] = gkeys(row, v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (vb + u * THREADS + threadIdx.x >= nvec) break;
                atomicAdd(&sh.hist[k[u].x >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].y >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].z >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].w >> kD1Shift], 1u);
            }
        }
        if (threadIdx.x < n - tail0)
            atomicAdd(&sh.hist[fkey(__ldg(row + tail0 + threadIdx.x)) >> kD1Shift], 1u);
        __syncthreads();
        select_bin<THREADS>(sh, 1 << D1, (uint32_t)K);
        const uint32_t b1 = sh.sel_bin;
        uint32_t prefix = b1 << kD1Shift;
        uint32_t rank = sh.sel_rank;

        // ---- split: above b1 -> above bits, in b1 -> cand bits (4-bit masks)
        for (int32_t vb = 0; vb < nvec; vb += kUnroll * THREADS) {
            uint4 k[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v < nvec) k[u] = gkeys(row, v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v >= nvec) break;
                uint32_t ma = 0, mc = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t d = comp(k[u], j) >> kD1Shift;
                    ma |= (d > b1 ? 1u : 0u) << j;
                    mc |= (d == b1 ? 1u : 0u) << j;
                }
                const uint32_t sh4 = (uint32_t)(v & 7) * 4;   // 4 positions of word v/8
                if (ma) atomicOr(above + (v >> 3), ma << sh4);
                if (mc) atomicOr(cand + (v >> 3), mc << sh4);
            }
        }
        if (threadIdx.x < n - tail0) {
            const int32_t p = tail0 + threadIdx.x;
            const uint32_t d = fkey(__ldg(row + p)) >> kD1Shift;
            if (d > b1) set_bit(above, p);
            else if (d == b1) set_bit(cand, p);
        }
        __syncthreads();

        // ---- digits 2 and 3 over the candidates (keys gathered from the row)
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? kD3Bits : 0;
            const int bits = d == 0 ? 22 - D1 : kD3Bits;
            const uint32_t mask_hi = d == 0 ? (0xFFFFFFFFu << kD1Shift) : (0xFFFFFFFFu << kD3Bits);
            const uint32_t bin_mask = (1u << bits) - 1u;
            __syncthreads();
            zero<THREADS>(sh.hist, 1 << bits);
            __syncthreads();
            for (int32_t w = threadIdx.x; w < nw; w += THREADS) {
                uint32_t m = cand[w];
                while (m) {
                    const int32_t p = (w << 5) + (__ffs(m) - 1);
                    m &= m - 1u;
                    const uint32_t kk = fkey(__ldg(row + p));
                    if ((kk & mask_hi) == prefix) atomicAdd(&sh.hist[(kk >> shift) & bin_mask], 1u);
                }
            }
            __syncthreads();
            select_bin<THREADS>(sh, 1 << bits, rank);
            prefix |= sh.sel_bin << shift;
            rank = sh.sel_rank;
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;                   // tau-valued keys kept
        const uint32_t n_above = (uint32_t)K - need;  // every key above tau is kept

        // ---- mark: candidates above tau -> above bits, equal -> tie bits
        for (int32_t w = threadIdx.x; w < nw; w += THREADS) {
            uint32_t m = cand[w];
            if (!m) continue;
            uint32_t a = 0, e = 0;
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1u;
                const uint32_t kk = fkey(__ldg(row + (w << 5) + b));
                a |= (kk > tau ? 1u : 0u) << b;
                e |= (kk == tau ? 1u : 0u) << b;
            }
            above[w] |= a;   // this thread owns word w in this step
            tie[w] = e;
        }
        __syncthreads();

        // ---- emit
        emit_ordered<THREADS>(sh, above, tie, nw, out, n_above, need);
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

// Shared memory a block may use in total (GB300 opt-in limit, 227 KB), and a
// bound on the streamed kernel's static part (histogram, scans, counters, with
// alignment padding).
constexpr int64_t kBlockSmem = 227 * 1024;
constexpr int64_t kStreamStaticBound = (int64_t)sizeof(TopkSmem<kStreamThreads, 12>) + 256;

bool bitmaps_fit_in_smem(int64_t row_cap) {
    const int64_t nw_cap = (row_cap + 31) / 32;
    return 3 * nw_cap * 4 + kStreamStaticBound <= kBlockSmem;
}

}  // namespace

size_t topk_scratch_bytes(int32_t T, int64_t max_len) {
    if (T <= 0 || max_len <= kStageCap || bitmaps_fit_in_smem(max_len)) return 0;
    return (size_t)kScratchBlocks * 3 * (size_t)((max_len + 31) / 32) * 4;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
    if (a.T <= 0) return cudaSuccess;
    const int64_t row_cap = a.max_len < a.ld ? a.max_len : a.ld;
    const int64_t nw_cap = (row_cap + 31) / 32;
    const int grid = a.T < 65535 ? a.T : 65535;
    if (row_cap <= kStageCap) {
        const int32_t stage = (int32_t)align_up((size_t)row_cap, 4);
        const size_t smem = ((size_t)stage + 2 * (size_t)nw_cap) * 4;
        auto kern = topk_staged_kernel<kStagedThreads>;
        cudaError_t e = ensure_smem_optin(
            (const void*)kern, (kStageCap + 2 * ((kStageCap + 31) / 32)) * 4);
        if (e != cudaSuccess) return e;
        kern<<<grid, kStagedThreads, smem, stream>>>(a.scores, a.ld, a.n_valid, a.n_from_pos, a.T,
                                                     a.max_len, a.topk, a.idx, a.cnt, a.status,
                                                     a.cu_q, a.cu_k, a.B, stage);
    } else {
        const bool in_smem = bitmaps_fit_in_smem(row_cap);
        if (!in_smem && a.bits_scratch == nullptr) return cudaErrorInvalidValue;
        const size_t smem = in_smem ? (size_t)(3 * nw_cap * 4) : 0;
        const int g = in_smem ? grid : (grid < kScratchBlocks ? grid : kScratchBlocks);
        auto kern = topk_stream_kernel<kStreamThreads>;
        const int64_t st = kernel_static_smem((const void*)kern);
        if (st < 0 || st > kStreamStaticBound) return cudaErrorInvalidValue;
        cudaError_t e = ensure_smem_optin((const void*)kern, kBlockSmem - kStreamStaticBound);
        if (e != cudaSuccess) return e;
        kern<<<g, kStreamThreads, smem, stream>>>(a.scores, a.ld, a.n_valid, a.n_from_pos, a.T,
                                                  a.max_len, a.topk, a.idx, a.cnt, a.status,
                                                  a.cu_q, a.cu_k, a.B, nw_cap,
                                                  in_smem ? nullptr : a.bits_scratch);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

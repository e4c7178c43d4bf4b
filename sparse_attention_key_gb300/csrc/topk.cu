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
// digits: bits 31..(32-D1), (31-D1)..10 and 9..0. One block per row:
//
//   pass A   histogram of the first digit; the bin b1 holding rank K (counted
//            from the top) follows. Short rows are copied into shared memory
//            on the way and every later pass reads that copy.
//   pass B   (long rows) one more read of the row: positions whose first digit
//            is above b1 are certainly kept (fewer than K of them) and get a bit
//            in the "above" bitmap; keys and positions of bin b1 go to a shared
//            candidate list.
//   digits   2 and 3 are histogrammed over bin b1 only (the candidate list, or a
//            rescan of the row if the list overflowed) -> tau, and need = the
//            number of tau-valued keys to keep.
//   mark     keys of bin b1 above tau get an "above" bit, keys equal to tau a
//            "tie" bit (short rows mark every key above tau here).
//   emit     two ordered scans of the bitmaps (n/32 words each; each thread owns
//            a contiguous word range, a block scan of bit counts gives offsets):
//            all above positions in increasing order, then the first `need` tie
//            positions in increasing order.
// The full row is read twice at most (once for short rows); everything after
// that touches only bin b1 and the bitmaps. No block waits on another.
#include "common.cuh"
#include "launch.h"

namespace lidx {

namespace {

constexpr int kD3Bits = 10;                 // last digit: bits 9..0
constexpr int kStagedThreads = 256;
constexpr int kStreamThreads = 1024;
constexpr int64_t kStageCap = 12288;        // longest row staged in shared memory
constexpr int kCandCap = 8192;              // long rows: candidates kept in shared memory
constexpr int kUnroll = 4;                  // independent 16-byte loads per thread in flight
constexpr int kScratchBlocks = 512;         // blocks when the bitmaps live in global scratch

template <int THREADS, int D1BITS>
struct TopkSmem {
    static constexpr int kWarps = THREADS / 32;
    uint32_t hist[1 << D1BITS];
    uint32_t scan[THREADS / 32 + 1];
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

// Keys of vector v, from the staged copy or from global.
template <bool STAGED>
__device__ __forceinline__ uint4 vkeys(const float* row, const uint32_t* staged, int32_t v) {
    if (STAGED) return reinterpret_cast<const uint4*>(staged)[v];
    return gkeys(row, v);
}

__device__ __forceinline__ uint32_t comp(const uint4& k, int j) {
    return j == 0 ? k.x : j == 1 ? k.y : j == 2 ? k.z : k.w;
}

__device__ __forceinline__ void set_bit(uint32_t* bits, int64_t pos) {
    atomicOr(bits + (pos >> 5), 1u << (pos & 31));
}

// Write the positions of the set bits of bits[0..nw) in increasing order to
// out[0..limit) (set bits past the first `limit` are dropped).
template <int THREADS, class S>
__device__ __forceinline__ void emit_ordered(S& sh, const uint32_t* bits, int64_t nw, int32_t* out,
                                             uint32_t limit) {
    const int64_t per = (nw + THREADS - 1) / THREADS;
    const int64_t w0 = threadIdx.x * per;
    const int64_t w1 = w0 + per < nw ? w0 + per : nw;
    uint32_t c = 0;
    for (int64_t w = w0; w < w1; ++w) c += __popc(bits[w]);
    uint32_t pos = block_excl_scan<THREADS>(sh, c);
    for (int64_t w = w0; w < w1 && pos < limit; ++w) {
        uint32_t m = bits[w];
        while (m && pos < limit) {
            const int b = __ffs(m) - 1;
            out[pos++] = (int32_t)(w * 32 + b);
            m &= m - 1u;
        }
    }
}

template <int THREADS, int D1BITS, bool STAGED>
__global__ void __launch_bounds__(THREADS, STAGED ? 4 : 1)
topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
            bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
            int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
            const int32_t* __restrict__ cu_k, int B, int64_t stage_cap, int64_t nw_cap,
            int cand_cap, uint32_t* __restrict__ gbits) {
    using S = TopkSmem<THREADS, D1BITS>;
    constexpr int kD1Shift = 32 - D1BITS;
    constexpr int kD2Bits = 22 - D1BITS;        // bits (31-D1)..10
    static_assert(kD2Bits <= D1BITS, "histogram holds the second digit");
    __shared__ S sh;
    // dynamic: [staged row: stage_cap][bitmaps: 2*nw_cap, unless global][cand keys][cand pos]
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t* staged = dyn;
    uint32_t* bits_sm = dyn + (STAGED ? stage_cap : 0);
    uint32_t* above_bits = gbits ? gbits + (int64_t)blockIdx.x * 2 * nw_cap : bits_sm;
    uint32_t* tie_bits = above_bits + nw_cap;
    uint32_t* cand_key = bits_sm + (gbits ? 0 : 2 * nw_cap);
    int32_t* cand_pos = reinterpret_cast<int32_t*>(cand_key + cand_cap);

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int64_t n64 = (int64_t)__ldg(n_valid + t) + (n_from_pos ? 1 : 0);
        int32_t* out = idx + (int64_t)t * K;
        bool bad = n64 < 0 || n64 > max_len || n64 > ld;
        if (cu_q != nullptr) {  // fused call: the row must lie inside its sequence
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
            }
            const int64_t len_k = (int64_t)__ldg(cu_k + lo + 1) - __ldg(cu_k + lo);
            bad = bad || n64 < 1 || n64 > len_k;
        }
        if (bad) {
            if (threadIdx.x == 0) report_error(status, IDX_ERR_DEVICE_ARG, t);
            for (int i = threadIdx.x; i < K; i += THREADS) out[i] = -1;
            if (cnt && threadIdx.x == 0) cnt[t] = 0;
            continue;
        }
        if (n64 <= K) {  // dormant selection: every position
            for (int i = threadIdx.x; i < K; i += THREADS) out[i] = i < n64 ? i : -1;
            if (cnt && threadIdx.x == 0) cnt[t] = (int32_t)n64;
            continue;
        }
        const int32_t n = (int32_t)n64;           // max_len < 2^31
        const int32_t nvec = n >> 2;              // full 4-element vectors
        const int32_t tail0 = nvec << 2;          // first element of the (< 4) tail
        const float* row = scores + (int64_t)t * ld;
        const int32_t nw = (n + 31) >> 5;

        // ---- pass A: first digit (short rows: staged on the way)
        __syncthreads();
        zero<THREADS>(sh.hist, 1 << D1BITS);
        zero<THREADS>(above_bits, nw);
        zero<THREADS>(tie_bits, nw);
        if (threadIdx.x == 0) sh.cand_count = 0;
        __syncthreads();
        for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += kUnroll * THREADS) {
            uint4 k[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)   // all loads first
                if (v0 + u * THREADS < nvec) k[u] = gkeys(row, v0 + u * THREADS);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (v0 + u * THREADS >= nvec) break;
                if (STAGED) reinterpret_cast<uint4*>(staged)[v0 + u * THREADS] = k[u];
                atomicAdd(&sh.hist[k[u].x >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].y >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].z >> kD1Shift], 1u);
                atomicAdd(&sh.hist[k[u].w >> kD1Shift], 1u);
            }
        }
        if (threadIdx.x < n - tail0) {
            const uint32_t kk = fkey(__ldg(row + tail0 + threadIdx.x));
            if (STAGED) staged[tail0 + threadIdx.x] = kk;
            atomicAdd(&sh.hist[kk >> kD1Shift], 1u);
        }
        __syncthreads();
        select_bin<THREADS>(sh, 1 << D1BITS, (uint32_t)K);
        const uint32_t b1 = sh.sel_bin;
        uint32_t rank = sh.sel_rank;
        uint32_t prefix = b1 << kD1Shift;

        // ---- pass B (long rows): certain positions -> bits, bin b1 -> candidates
        bool use_cand = false;
        if (!STAGED) {
            auto visit = [&](uint32_t kk, int32_t pos) {
                const uint32_t d = kk >> kD1Shift;
                if (d > b1) {
                    set_bit(above_bits, pos);
                } else if (d == b1) {
                    const uint32_t slot = atomicAdd(&sh.cand_count, 1u);
                    if (slot < (uint32_t)cand_cap) {
                        cand_key[slot] = kk;
                        cand_pos[slot] = pos;
                    }
                }
            };
            for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += kUnroll * THREADS) {
                uint4 k[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    if (v0 + u * THREADS < nvec) k[u] = gkeys(row, v0 + u * THREADS);
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int32_t v = v0 + u * THREADS;
                    if (v >= nvec) break;
                    // one test per vector: most vectors hold nothing >= b1
                    const uint32_t mx = max(max(k[u].x, k[u].y), max(k[u].z, k[u].w));
                    if ((mx >> kD1Shift) < b1) continue;
                    visit(k[u].x, 4 * v);
                    visit(k[u].y, 4 * v + 1);
                    visit(k[u].z, 4 * v + 2);
                    visit(k[u].w, 4 * v + 3);
                }
            }
            if (threadIdx.x < n - tail0)
                visit(fkey(__ldg(row + tail0 + threadIdx.x)), tail0 + threadIdx.x);
            __syncthreads();
            use_cand = sh.cand_count <= (uint32_t)cand_cap;
        }
        const int n_cand = use_cand ? (int)sh.cand_count : 0;

        // ---- digits 2 and 3 among keys that match the digits chosen so far
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? kD3Bits : 0;
            const int bits = d == 0 ? kD2Bits : kD3Bits;
            const uint32_t mask_hi = d == 0 ? (0xFFFFFFFFu << kD1Shift) : (0xFFFFFFFFu << kD3Bits);
            const uint32_t bin_mask = (1u << bits) - 1u;
            __syncthreads();
            zero<THREADS>(sh.hist, 1 << bits);
            __syncthreads();
            auto add = [&](uint32_t kk) {
                if ((kk & mask_hi) == prefix) atomicAdd(&sh.hist[(kk >> shift) & bin_mask], 1u);
            };
            if (use_cand) {
                for (int i = threadIdx.x; i < n_cand; i += THREADS) add(cand_key[i]);
            } else {
                for (int32_t v = threadIdx.x; v < nvec; v += THREADS) {
                    const uint4 k = vkeys<STAGED>(row, staged, v);
                    add(k.x); add(k.y); add(k.z); add(k.w);
                }
                if (threadIdx.x < n - tail0)
                    add(STAGED ? staged[tail0 + threadIdx.x] : fkey(__ldg(row + tail0 + threadIdx.x)));
            }
            __syncthreads();
            select_bin<THREADS>(sh, 1 << bits, rank);
            prefix |= sh.sel_bin << shift;
            rank = sh.sel_rank;
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;                   // members of the tie group kept
        const uint32_t n_above = (uint32_t)K - need;  // every key > tau is kept

        // ---- mark keys above / equal to tau not marked yet
        if (use_cand) {
            for (int i = threadIdx.x; i < n_cand; i += THREADS) {
                const uint32_t kk = cand_key[i];
                if (kk > tau) set_bit(above_bits, cand_pos[i]);
                else if (kk == tau) set_bit(tie_bits, cand_pos[i]);
            }
        } else {
            // staged rows never ran pass B, so every key above tau is marked here;
            // streamed rows marked first digits above b1 in pass B already
            auto mark = [&](uint32_t kk, int32_t pos) {
                if (kk > tau) {
                    if (STAGED || (kk >> kD1Shift) == b1) set_bit(above_bits, pos);
                } else if (kk == tau) {
                    set_bit(tie_bits, pos);
                }
            };
            for (int32_t v = threadIdx.x; v < nvec; v += THREADS) {
                const uint4 k = vkeys<STAGED>(row, staged, v);
                const uint32_t mx = max(max(k.x, k.y), max(k.z, k.w));
                if (mx < tau) continue;
                mark(k.x, 4 * v); mark(k.y, 4 * v + 1); mark(k.z, 4 * v + 2); mark(k.w, 4 * v + 3);
            }
            if (threadIdx.x < n - tail0)
                mark(STAGED ? staged[tail0 + threadIdx.x] : fkey(__ldg(row + tail0 + threadIdx.x)),
                     tail0 + threadIdx.x);
        }
        __syncthreads();

        // ---- emit: above positions ascending, then the first `need` ties ascending
        emit_ordered<THREADS>(sh, above_bits, nw, out, n_above);
        emit_ordered<THREADS>(sh, tie_bits, nw, out + n_above, need);
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

constexpr size_t kStreamStatic = sizeof(TopkSmem<kStreamThreads, 12>);

// Shared memory a block may use in total (GB300 opt-in limit, 227 KB).
constexpr int64_t kBlockSmem = 227 * 1024;

bool bitmaps_fit_in_smem(int64_t row_cap) {
    const int64_t nw_cap = (row_cap + 31) / 32;
    return (int64_t)kCandCap * 8 + 2 * nw_cap * 4 + (int64_t)kStreamStatic <= kBlockSmem;
}

}  // namespace

size_t topk_scratch_bytes(int32_t T, int64_t max_len) {
    if (T <= 0 || max_len <= kStageCap || bitmaps_fit_in_smem(max_len)) return 0;
    return (size_t)kScratchBlocks * 2 * (size_t)((max_len + 31) / 32) * 4;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
    if (a.T <= 0) return cudaSuccess;
    const int64_t row_cap = a.max_len < a.ld ? a.max_len : a.ld;
    const int64_t nw_cap = (row_cap + 31) / 32;
    const int grid = a.T < 65535 ? a.T : 65535;
    if (row_cap <= kStageCap) {
        const int64_t stage = (int64_t)align_up((size_t)row_cap, 4);
        const size_t smem = (size_t)(stage + 2 * nw_cap) * 4;
        auto kern = topk_kernel<kStagedThreads, 11, true>;
        cudaError_t e = ensure_smem_optin(
            (const void*)kern, (kStageCap + 2 * ((kStageCap + 31) / 32)) * 4);
        if (e != cudaSuccess) return e;
        kern<<<grid, kStagedThreads, smem, stream>>>(a.scores, a.ld, a.n_valid, a.n_from_pos, a.T,
                                                     a.max_len, a.topk, a.idx, a.cnt, a.status,
                                                     a.cu_q, a.cu_k, a.B, stage, nw_cap, 0, nullptr);
    } else {
        const bool in_smem = bitmaps_fit_in_smem(row_cap);
        if (!in_smem && a.bits_scratch == nullptr) return cudaErrorInvalidValue;
        const size_t smem = (size_t)kCandCap * 8 + (in_smem ? (size_t)(2 * nw_cap * 4) : 0);
        const int g = in_smem ? grid : (grid < kScratchBlocks ? grid : kScratchBlocks);
        auto kern = topk_kernel<kStreamThreads, 12, false>;
        cudaError_t e = ensure_smem_optin((const void*)kern, kBlockSmem - (int64_t)kStreamStatic);
        if (e != cudaSuccess) return e;
        kern<<<g, kStreamThreads, smem, stream>>>(a.scores, a.ld, a.n_valid, a.n_from_pos, a.T,
                                                  a.max_len, a.topk, a.idx, a.cnt, a.status,
                                                  a.cu_q, a.cu_k, a.B, 0, nw_cap, kCandCap,
                                                  in_smem ? nullptr : a.bits_scratch);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace lidx

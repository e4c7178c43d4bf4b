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
// digits: bits 31..(32-D1), (31-D1)..10 and 9..0. One block per row (for a
// few long rows, a thread-block cluster per row; beyond 2^21 positions,
// slice-parallel kernels), with the row's positions tracked in bitmaps (one
// bit per position):
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
// A; every later step reads that copy. Long rows (streamed kernel) are first
// requested into L2 as a whole (bulk prefetch), then read twice: pass A counts
// the first digit of the scores' own bits (moved into key order afterwards)
// and the split compares the scores as floats with the bounds of bin b1, so
// neither converts every score to its key; the candidates' keys are gathered
// once into a shared-memory list that digits 2-3 and the mark read (or, when
// the list would overflow, gathered again at each step). No block waits on
// another except through the cluster barriers, which every CTA of a cluster
// reaches.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace lidx {

namespace cg = cooperative_groups;

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
    alignas(16) uint32_t hist[1 << D1BITS];
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
// (1-based from the largest) in sh.hist[0..nbins); writes sh.sel_bin and the
// rank inside that bin to sh.sel_rank. Thread j sums the nbins/THREADS bins
// just below the top j*nbins/THREADS ones; an exclusive block scan of those
// sums gives every thread the count above its bins, and the one thread whose
// range holds the rank finds the bin. nbins is a multiple of THREADS. When the
// histogram holds fewer than `rank` elements (only for inputs outside the
// contract, such as scores an aborted scorer left half-written), bin 0 and
// rank 0 are returned.
template <int THREADS, class S>
__device__ __forceinline__ void select_bin(S& sh, int nbins, uint32_t rank) {
    const int per = nbins / THREADS;
    const int top = nbins - 1 - (int)threadIdx.x * per;   // this thread's highest bin
    uint32_t s = 0;
    if ((per & 3) == 0) {
        const uint4* h4 = reinterpret_cast<const uint4*>(sh.hist + (top + 1 - per));
        for (int i = 0; i < per / 4; ++i) {
            const uint4 v = h4[i];
            s += (v.x + v.y) + (v.z + v.w);
        }
    } else {
        for (int i = 0; i < per; ++i) s += sh.hist[top - i];
    }
    // (the scan's first barrier also separates the callers' reads of the
    // previous sel_bin / sel_rank from the writes below)
    const uint32_t excl = block_excl_scan<THREADS>(sh, s);
    if (threadIdx.x == THREADS - 1 && excl + s < rank) {   // fewer elements than rank
        sh.sel_bin = 0;
        sh.sel_rank = 0;
    }
    if (excl < rank && rank <= excl + s) {
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
    __syncthreads();
}

// Shared-memory slot of histogram bin b in a swizzled histogram: the low five
// bits are XORed with the next five, a bijection that sends bins 32 apart to
// different banks. Integer-valued scores leave the low key bits zero, so
// their second and third digits are multiples of 32 or 64; unswizzled, all of
// them would hit one bank.
__device__ __forceinline__ uint32_t swz(uint32_t b) { return b ^ ((b >> 5) & 31u); }

// select_bin over a histogram stored at swizzled slots (scalar reads).
template <int THREADS, class S>
__device__ __forceinline__ void select_bin_swz(S& sh, int nbins, uint32_t rank) {
    const int per = nbins / THREADS;
    const int top = nbins - 1 - (int)threadIdx.x * per;
    uint32_t s = 0;
    for (int i = 0; i < per; ++i) s += sh.hist[swz((uint32_t)(top - i))];
    const uint32_t excl = block_excl_scan<THREADS>(sh, s);
    if (threadIdx.x == THREADS - 1 && excl + s < rank) {
        sh.sel_bin = 0;
        sh.sel_rank = 0;
    }
    if (excl < rank && rank <= excl + s) {
        uint32_t acc = excl;
        for (int i = 0; i < per; ++i) {
            const uint32_t c = sh.hist[swz((uint32_t)(top - i))];
            if (acc + c >= rank) {
                sh.sel_bin = (uint32_t)(top - i);
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

__device__ __forceinline__ uint32_t fkey(float x) { return score_key(x); }

// Smallest non-NaN float whose order key is >= z (keys are monotone in the
// value, with -0 == +0): every float if z is at or below the key of -inf; no
// float (NaN, so that every comparison is false) if z is above the key of
// +inf. Otherwise the float whose key is exactly z: positive for
// z >= 0x80000000, negative below (z is never 0x7FFFFFFF, the key -0 would
// have before folding). For non-NaN x: fkey(x) >= z  <=>  x >= key_floor(z),
// denormals included (no flush to zero in this library).
__device__ __forceinline__ float key_floor(uint64_t z) {
    if (z <= 0x007FFFFFull) return -__int_as_float(0x7f800000);
    if (z > 0xFF800000ull) return __int_as_float(0x7fffffff);
    const uint32_t zz = (uint32_t)z;
    return __uint_as_float(zz >= 0x80000000u ? (zz ^ 0x80000000u) : ~zz);
}

// Keys of the 4 scores of vector v (elements 4v..4v+3) of a row, from global.
__device__ __forceinline__ uint4 gkeys(const float* row, int32_t v) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(row) + v);
    return make_uint4(fkey(x.x), fkey(x.y), fkey(x.z), fkey(x.w));
}

// Ask L2 to fetch [p, p + bytes) ahead of the reads (p 16-byte aligned, bytes
// a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The first n scores of a 16-byte aligned row (rows hold ld scores, ld a
// multiple of 4, so the rounded-up request stays inside the row), in 16 KB
// requests spread over the block's threads.
template <int THREADS>
__device__ __forceinline__ void prefetch_row_l2(const float* row, int64_t n) {
    const int64_t bytes = (n * 4 + 15) & ~(int64_t)15;
    constexpr int64_t kChunk = 16384;
    for (int64_t off = (int64_t)threadIdx.x * kChunk; off < bytes; off += (int64_t)THREADS * kChunk) {
        const int64_t sz = bytes - off < kChunk ? bytes - off : kChunk;
        prefetch_l2_bulk(reinterpret_cast<const char*>(row) + off, (uint32_t)sz);
    }
}

__device__ __forceinline__ void set_bit(uint32_t* bits, int64_t pos) {
    atomicOr(bits + (pos >> 5), 1u << (pos & 31));
}

// Ordered output from the two bitmaps: the set positions of `above` in
// increasing order to out[0..K-need), then the first `need` set positions of
// `tie` in increasing order to out[K-need..K). Each thread owns a contiguous
// range of words; one block scan of packed (above, tie) counts gives offsets.
// Writes stay inside out[0..K) even when the bitmaps disagree with the counts
// (scores that an aborted scorer left half-written): surplus positions are
// dropped.
template <int THREADS, class S>
__device__ __forceinline__ void emit_ordered(S& sh, const uint32_t* above, const uint32_t* tie,
                                             int32_t nw, int32_t* out, uint32_t K, uint32_t need) {
    need = need < K ? need : K;
    const uint32_t n_above = K - need;
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
        while (m && pa < n_above) {
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

// emit_ordered with warps instead of threads: warp w owns a contiguous range
// of words; its lanes count their words' bits, one exchange of the warps'
// totals through shared memory (cnt_a / cnt_t: THREADS / 32 words each) gives
// every warp its offsets, and the warp then walks its words one at a time,
// one bit per lane, so that consecutive lanes write consecutive outputs. One
// block barrier instead of a block scan's three. Writes stay inside out[0..K).
template <int THREADS>
__device__ __forceinline__ void emit_ordered_warps(const uint32_t* above, const uint32_t* tie, int32_t nw,
                                                   int32_t* out, uint32_t K, uint32_t need,
                                                   uint32_t* cnt_a, uint32_t* cnt_t) {
    constexpr int kWarps = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    need = need < K ? need : K;
    const uint32_t n_above = K - need;
    const int32_t per = (nw + kWarps - 1) / kWarps;
    const int32_t w0 = warp * per < nw ? warp * per : nw;
    const int32_t w1 = w0 + per < nw ? w0 + per : nw;
    uint32_t ca = 0, ct = 0;
    for (int32_t w = w0 + lane; w < w1; w += 32) {
        ca += __popc(above[w]);
        ct += __popc(tie[w]);
    }
    ca = __reduce_add_sync(0xffffffffu, ca);
    ct = __reduce_add_sync(0xffffffffu, ct);
    if (lane == 0) {
        cnt_a[warp] = ca;
        cnt_t[warp] = ct;
    }
    __syncthreads();
    uint32_t pa = __reduce_add_sync(0xffffffffu, lane < warp ? cnt_a[lane] : 0u);
    uint32_t pt = __reduce_add_sync(0xffffffffu, lane < warp ? cnt_t[lane] : 0u);
    const uint32_t lt = (1u << lane) - 1u;
    for (int32_t w = w0; w < w1; ++w) {   // warp-uniform
        const uint32_t a = above[w], e = tie[w];
        const int32_t p = (w << 5) + lane;
        const uint32_t oa = pa + __popc(a & lt), ot = pt + __popc(e & lt);
        if (((a >> lane) & 1u) && oa < n_above) out[oa] = p;
        if (((e >> lane) & 1u) && ot < need) out[n_above + ot] = p;
        pa += __popc(a);
        pt += __popc(e);
    }
}

// True when a bounded wait of the scorer that ran before this kernel in the
// same call gave up: its staged scores are then incomplete, and every row of
// the call is written as skipped (-1s, cnt 0) instead of being selected from
// them. Read after pdl_wait(), when the scorer has completed.
__device__ __forceinline__ bool scorer_gave_up(const DeviceStatus* status) {
    return *reinterpret_cast<const volatile int32_t*>(&status->code) == IDX_ERR_TIMEOUT;
}

// Row checks shared by both kernels. Returns the row length, or -1 after
// writing the output of a bad row (-1s, cnt 0, status), of every row of a
// call whose scorer gave up (-1s, cnt 0; `gave_up`), or of a row that keeps
// every position (n <= K).
template <int THREADS>
__device__ __forceinline__ int64_t row_prologue(int t, const int32_t* __restrict__ n_valid,
                                                bool n_from_pos, int64_t max_len, int64_t ld,
                                                int K, int32_t* out, int32_t* __restrict__ cnt,
                                                DeviceStatus* status,
                                                const int32_t* __restrict__ cu_q,
                                                const int32_t* __restrict__ cu_k, int B,
                                                bool gave_up) {
    if (gave_up) {
        for (int i = threadIdx.x; i < K; i += THREADS) out[i] = -1;
        if (cnt && threadIdx.x == 0) cnt[t] = 0;
        return -1;
    }
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
__global__ void __launch_bounds__(THREADS, 5)
topk_staged_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                   bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
                   int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ cu_k, int B, int32_t stage_cap) {
    pdl_wait();
    pdl_launch_dependents();
    const bool gave_up = scorer_gave_up(status);
    constexpr int D1 = 11;                      // digits: bits 31..21, 20..10, 9..0
    constexpr int kD1Shift = 32 - D1;
    using S = TopkSmem<THREADS, D1>;
    __shared__ S sh;
    __shared__ uint32_t s_d3_and[THREADS / 32], s_d3_or[THREADS / 32];
    __shared__ uint32_t s_cnt_a[THREADS / 32], s_cnt_t[THREADS / 32];
    // dynamic: keys[stage_cap] | above[nw_cap] | tie[nw_cap]
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t* keys = dyn;
    const int32_t nw_cap = (stage_cap + 31) >> 5;
    uint32_t* above = dyn + stage_cap;
    uint32_t* tie = above + nw_cap;

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int32_t* out = idx + (int64_t)t * K;
        const int64_t n64 = row_prologue<THREADS>(t, n_valid, n_from_pos, max_len, ld, K, out, cnt,
                                                  status, cu_q, cu_k, B, gave_up);
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

        // ---- digits 2 and 3 among the keys that match the digits so far.
        // The second digit's pass also ANDs and ORs the third digit of the
        // keys it counts; when those agree, every key sharing the first two
        // digits is the same key (integer scores, for instance, leave the
        // low key bits equal), and the third round is skipped.
        constexpr uint32_t kD3Mask = (1u << kD3Bits) - 1u;
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? kD3Bits : 0;
            const int bits = d == 0 ? 22 - D1 : kD3Bits;
            const uint32_t mask_hi = d == 0 ? (0xFFFFFFFFu << kD1Shift) : (0xFFFFFFFFu << kD3Bits);
            const uint32_t bin_mask = (1u << bits) - 1u;
            __syncthreads();
            zero<THREADS>(sh.hist, 1 << bits);
            __syncthreads();
            uint32_t d3_and = kD3Mask, d3_or = 0u;
            auto add = [&](uint32_t kk) {
                if ((kk & mask_hi) == prefix) {
                    atomicAdd(&sh.hist[swz((kk >> shift) & bin_mask)], 1u);
                    d3_and &= kk;
                    d3_or |= kk;
                }
            };
            for (int32_t v = threadIdx.x; v < nvec; v += THREADS) {
                const uint4 k = reinterpret_cast<const uint4*>(keys)[v];
                add(k.x); add(k.y); add(k.z); add(k.w);
            }
            if (threadIdx.x < n - tail0) add(keys[tail0 + threadIdx.x]);
            if (d == 0) {
                d3_and = __reduce_and_sync(0xffffffffu, d3_and);
                d3_or = __reduce_or_sync(0xffffffffu, d3_or);
                if ((threadIdx.x & 31) == 0) {
                    s_d3_and[threadIdx.x >> 5] = d3_and;
                    s_d3_or[threadIdx.x >> 5] = d3_or;
                }
            }
            __syncthreads();
            select_bin_swz<THREADS>(sh, 1 << bits, rank);
            prefix |= sh.sel_bin << shift;
            rank = sh.sel_rank;
            if (d == 0) {   // (the barriers above ordered the per-warp values; the same outcome everywhere)
                uint32_t a = kD3Mask, o = 0u;
#pragma unroll
                for (int i = 0; i < THREADS / 32; ++i) {
                    a &= s_d3_and[i];
                    o |= s_d3_or[i];
                }
                if ((a & kD3Mask) == (o & kD3Mask) && rank > 0) {
                    prefix |= o & kD3Mask;
                    break;
                }
            }
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;   // tau-valued keys kept; every key above tau is kept

        // ---- mark: a warp per 32-position word, one key per lane (consecutive
        // keys, no bank conflicts); the two ballots are the word's bits
        for (int32_t w = threadIdx.x >> 5; w < nw; w += THREADS / 32) {
            const int32_t p = (w << 5) + (threadIdx.x & 31);
            const uint32_t kk = p < n ? keys[p] : 0u;
            const uint32_t a = __ballot_sync(0xffffffffu, p < n && kk > tau);
            const uint32_t e = __ballot_sync(0xffffffffu, p < n && kk == tau);
            if ((threadIdx.x & 31) == 0) {
                above[w] = a;
                tie[w] = e;
            }
        }
        __syncthreads();

        // ---- emit: above positions ascending, then the first `need` ties ascending
        emit_ordered_warps<THREADS>(above, tie, nw, out, (uint32_t)K, need, s_cnt_a, s_cnt_t);
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

// ---------------------------------------------------------------------------
// Long rows: streamed from L2 after a bulk prefetch of the row; bitmaps in
// shared memory (or in per-block global scratch when a row's bitmaps do not
// fit), then a shared-memory list of the candidates: positions in increasing
// order from a block scan of the cand bits' counts, then their keys.
// ---------------------------------------------------------------------------
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 2)
topk_stream_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                   bool n_from_pos, int T, int64_t max_len, int K, int32_t* __restrict__ idx,
                   int32_t* __restrict__ cnt, DeviceStatus* status, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ cu_k, int B, int64_t nw_cap,
                   uint32_t* __restrict__ gbits, int32_t list_cap) {
    pdl_wait();
    pdl_launch_dependents();
    const bool gave_up = scorer_gave_up(status);
    constexpr int D1 = 12;                      // digits: bits 31..20, 19..10, 9..0
    constexpr int kD1Shift = 32 - D1;
    using S = TopkSmem<THREADS, D1>;
    __shared__ S sh;
    // above | tie | cand bitmaps, then (16-byte aligned) list_cap (key, position) pairs
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t* above = gbits ? gbits + (int64_t)blockIdx.x * 3 * nw_cap : dyn;
    uint32_t* tie = above + nw_cap;
    uint32_t* cand = tie + nw_cap;
    uint2* list = reinterpret_cast<uint2*>(dyn + (gbits ? 0 : (3 * nw_cap + 3) / 4 * 4));

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int32_t* out = idx + (int64_t)t * K;
        const int64_t n64 = row_prologue<THREADS>(t, n_valid, n_from_pos, max_len, ld, K, out, cnt,
                                                  status, cu_q, cu_k, B, gave_up);
        if (n64 < 0) continue;
        const int32_t n = (int32_t)n64;
        const int32_t nvec = n >> 2, tail0 = nvec << 2;
        const int32_t nw = (n + 31) >> 5;
        const float* row = scores + (int64_t)t * ld;
        prefetch_row_l2<THREADS>(row, n);

        // ---- pass A: first digit
        __syncthreads();
        zero<THREADS>(sh.hist, 1 << D1);
        zero<THREADS>(above, nw);
        zero<THREADS>(tie, nw);
        zero<THREADS>(cand, nw);
        __syncthreads();
        // Counted by the top 12 bits of the score itself (after -0 -> +0),
        // which spares the key conversion of every score; the counts are then
        // moved to key order: a non-negative score's key digit is its bits'
        // digit + 2048, a negative one's 4095 - its bits' digit.
        static_assert(D1 == 12 && (1 << D1) % THREADS == 0, "raw-digit histogram");
        for (int32_t vb = 0; vb < nvec; vb += kUnroll * THREADS) {
            float4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v < nvec) x[u] = __ldg(reinterpret_cast<const float4*>(row) + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (vb + u * THREADS + threadIdx.x >= nvec) break;
                atomicAdd(&sh.hist[__float_as_uint(__fadd_rn(x[u].x, 0.0f)) >> kD1Shift], 1u);
                atomicAdd(&sh.hist[__float_as_uint(__fadd_rn(x[u].y, 0.0f)) >> kD1Shift], 1u);
                atomicAdd(&sh.hist[__float_as_uint(__fadd_rn(x[u].z, 0.0f)) >> kD1Shift], 1u);
                atomicAdd(&sh.hist[__float_as_uint(__fadd_rn(x[u].w, 0.0f)) >> kD1Shift], 1u);
            }
        }
        if (threadIdx.x < n - tail0)
            atomicAdd(&sh.hist[__float_as_uint(__fadd_rn(__ldg(row + tail0 + threadIdx.x), 0.0f)) >> kD1Shift],
                      1u);
        __syncthreads();
        {
            constexpr int kPer = (1 << D1) / THREADS;
            uint32_t c[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) c[i] = sh.hist[threadIdx.x + i * THREADS];
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const uint32_t rb = threadIdx.x + i * THREADS;
                sh.hist[rb < 2048u ? rb + 2048u : 4095u - rb] = c[i];
            }
        }
        __syncthreads();
        select_bin<THREADS>(sh, 1 << D1, (uint32_t)K);
        const uint32_t b1 = sh.sel_bin;
        uint32_t prefix = b1 << kD1Shift;
        uint32_t rank = sh.sel_rank;

        // ---- split: above b1 -> above bits, in b1 -> cand bits (4-bit masks).
        // Compared as floats against the smallest values of bins b1 and b1+1
        // (finite scores: x >= key_floor(z) exactly when key(x) >= z), which
        // spares the key conversion of every score.
        const float f_lo = key_floor((uint64_t)b1 << kD1Shift);         // bin b1 or above
        const float f_hi = key_floor((uint64_t)(b1 + 1) << kD1Shift);   // above bin b1
        for (int32_t vb = 0; vb < nvec; vb += kUnroll * THREADS) {
            float4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v < nvec) x[u] = __ldg(reinterpret_cast<const float4*>(row) + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int32_t v = vb + u * THREADS + threadIdx.x;
                if (v >= nvec) break;
                const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                uint32_t ma = 0, mc = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool a = xs[j] >= f_hi;
                    ma |= (a ? 1u : 0u) << j;
                    mc |= (!a && xs[j] >= f_lo ? 1u : 0u) << j;
                }
                const uint32_t sh4 = (uint32_t)(v & 7) * 4;   // 4 positions of word v/8
                if (ma) atomicOr(above + (v >> 3), ma << sh4);
                if (mc) atomicOr(cand + (v >> 3), mc << sh4);
            }
        }
        if (threadIdx.x < n - tail0) {
            const int32_t p = tail0 + threadIdx.x;
            const float xf = __ldg(row + p);
            if (xf >= f_hi) set_bit(above, p);
            else if (xf >= f_lo) set_bit(cand, p);
        }
        __syncthreads();

        // ---- compact: candidate positions in order (block scan of counts), then their keys
        const int32_t per = (nw + THREADS - 1) / THREADS;
        const int32_t w0 = threadIdx.x * per < nw ? threadIdx.x * per : nw;
        const int32_t w1 = w0 + per < nw ? w0 + per : nw;
        uint32_t mine = 0;
        for (int32_t w = w0; w < w1; ++w) mine += __popc(cand[w]);
        const uint32_t off0 = block_excl_scan<THREADS>(sh, mine);
        if (threadIdx.x == THREADS - 1) sh.cand_count = off0 + mine;
        __syncthreads();
        const uint32_t n_cand = sh.cand_count;
        const bool listed = n_cand <= (uint32_t)list_cap;
        if (listed) {
            uint32_t o = off0;
            for (int32_t w = w0; w < w1; ++w) {
                uint32_t m = cand[w];
                while (m) {
                    list[o++].y = (uint32_t)((w << 5) + (__ffs(m) - 1));
                    m &= m - 1u;
                }
            }
            __syncthreads();
            for (uint32_t i = threadIdx.x; i < n_cand; i += 4 * THREADS) {
                float x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t ii = i + u * THREADS;
                    x[u] = ii < n_cand ? __ldg(row + list[ii].y) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t ii = i + u * THREADS;
                    if (ii < n_cand) list[ii].x = fkey(x[u]);
                }
            }
        }

        // ---- digits 2 and 3 over the candidates (from the list, else gathered from the row)
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? kD3Bits : 0;
            const int bits = d == 0 ? 22 - D1 : kD3Bits;
            const uint32_t mask_hi = d == 0 ? (0xFFFFFFFFu << kD1Shift) : (0xFFFFFFFFu << kD3Bits);
            const uint32_t bin_mask = (1u << bits) - 1u;
            __syncthreads();
            zero<THREADS>(sh.hist, 1 << bits);
            __syncthreads();
            if (listed) {
                for (uint32_t i = threadIdx.x; i < n_cand; i += THREADS) {
                    const uint32_t kk = list[i].x;
                    if ((kk & mask_hi) == prefix) atomicAdd(&sh.hist[(kk >> shift) & bin_mask], 1u);
                }
            } else {
                for (int32_t w = threadIdx.x; w < nw; w += THREADS) {
                    uint32_t m = cand[w];
                    while (m) {
                        const int32_t p = (w << 5) + (__ffs(m) - 1);
                        m &= m - 1u;
                        const uint32_t kk = fkey(__ldg(row + p));
                        if ((kk & mask_hi) == prefix) atomicAdd(&sh.hist[(kk >> shift) & bin_mask], 1u);
                    }
                }
            }
            __syncthreads();
            select_bin<THREADS>(sh, 1 << bits, rank);
            prefix |= sh.sel_bin << shift;
            rank = sh.sel_rank;
        }
        const uint32_t tau = prefix;
        const uint32_t need = rank;   // tau-valued keys kept; every key above tau is kept

        // ---- mark: candidates above tau -> above bits, equal -> tie bits
        if (listed) {
            for (uint32_t i = threadIdx.x; i < n_cand; i += THREADS) {
                const uint2 e = list[i];
                if (e.x > tau) atomicOr(above + (e.y >> 5), 1u << (e.y & 31));
                else if (e.x == tau) atomicOr(tie + (e.y >> 5), 1u << (e.y & 31));
            }
        } else {
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
        }
        __syncthreads();

        // ---- emit
        emit_ordered<THREADS>(sh, above, tie, nw, out, (uint32_t)K, need);
        if (cnt && threadIdx.x == 0) cnt[t] = K;
    }
}

// ---------------------------------------------------------------------------
// Few long rows (decode): each row is split into slices handled by separate
// blocks, so that T rows keep T x slices blocks busy instead of T. Three
// kernels share per-row scratch in global memory: first-digit histogram
// [4096], second-digit histogram of the candidates [1024], and the above /
// tie / cand bitmaps.
//   split_hist   per slice: first-digit histogram, added into the row's;
//   split_mark   per slice: select b1 from the row histogram, write whole
//                bitmap words (above b1, in b1), add the candidates' second
//                digits into the row's second histogram;
//   split_finish per row: digits 2 and 3 (the third over the candidates'
//                keys, gathered from the row), mark, ordered emit.
// ---------------------------------------------------------------------------
constexpr int kSplitThreads = 256;
constexpr int kSplitSlice = 4096;           // positions per block (multiple of 128)
constexpr int kFinishThreads = 1024;
constexpr int kFinishCand = 8192;           // candidates listed in (dynamic) shared memory
constexpr int32_t kSplitMaxRows = 128;      // fewer rows than GB300 has SMs

struct SplitScratch {
    uint32_t* hist1;   // [T][4096]
    uint32_t* hist2;   // [T][1024]
    uint32_t* bits;    // [T][3][nw_cap]: above | tie | cand
    int64_t nw_cap;
};

__host__ __device__ inline size_t split_hist_bytes(int32_t T) {
    return (size_t)T * (4096 + 1024) * 4;
}

__device__ __forceinline__ SplitScratch split_scratch(uint32_t* base, int32_t T, int64_t nw_cap) {
    SplitScratch sc;
    sc.hist1 = base;
    sc.hist2 = base + (size_t)T * 4096;
    sc.bits = base + (size_t)T * 5120;
    sc.nw_cap = nw_cap;
    return sc;
}

// Row length when the row needs a selection (n > K and valid), else -1; no
// side effects (the finishing kernel writes the other rows' output).
__device__ __forceinline__ int64_t selecting_row(int t, const int32_t* __restrict__ n_valid,
                                                 bool n_from_pos, int64_t max_len, int64_t ld, int K,
                                                 const int32_t* __restrict__ cu_q,
                                                 const int32_t* __restrict__ cu_k, int B) {
    const int64_t n = (int64_t)__ldg(n_valid + t) + (n_from_pos ? 1 : 0);
    bool bad = n < 0 || n > max_len || n > ld;
    if (cu_q != nullptr) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
        }
        const int64_t len_k = (int64_t)__ldg(cu_k + lo + 1) - __ldg(cu_k + lo);
        bad = bad || n < 1 || n > len_k;
    }
    return (bad || n <= K) ? -1 : n;
}

// Bits of the 4 positions held by each lane (4 consecutive positions per lane,
// lanes in order) gathered into the 32-bit word of their 32-position group:
// lanes 8j..8j+7 hold word j of the warp's 128 positions; returns that word
// in every lane of the group.
__device__ __forceinline__ uint32_t word_of_masks(uint32_t mask4) {
    const int lane = threadIdx.x & 31;
    uint32_t v = mask4 << ((lane & 7) * 4);
    v |= __shfl_xor_sync(0xffffffffu, v, 1);
    v |= __shfl_xor_sync(0xffffffffu, v, 2);
    v |= __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

__global__ void __launch_bounds__(kSplitThreads)
topk_split_hist_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                       bool n_from_pos, int64_t max_len, int K, const int32_t* __restrict__ cu_q,
                       const int32_t* __restrict__ cu_k, int B, int slices, uint32_t* scratch,
                       int32_t T, int64_t nw_cap) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint32_t hist[4096];
    const int t = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int64_t n64 = selecting_row(t, n_valid, n_from_pos, max_len, ld, K, cu_q, cu_k, B);
    const int32_t p0 = sl * kSplitSlice;
    if (n64 < 0 || p0 >= n64) return;                       // block-uniform
    const int32_t p1 = (int32_t)(n64 < p0 + kSplitSlice ? n64 : p0 + kSplitSlice);
    const SplitScratch sc = split_scratch(scratch, T, nw_cap);
    zero<kSplitThreads>(hist, 4096);
    __syncthreads();
    const float* row = scores + (int64_t)t * ld;
    const int32_t v0 = p0 >> 2, v1 = p1 >> 2;               // whole vectors, then the tail
    for (int32_t vb = v0; vb < v1; vb += kUnroll * kSplitThreads) {
        uint4 k[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t v = vb + u * kSplitThreads + threadIdx.x;
            if (v < v1) k[u] = gkeys(row, v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (vb + u * kSplitThreads + threadIdx.x >= v1) break;
            atomicAdd(&hist[k[u].x >> 20], 1u);
            atomicAdd(&hist[k[u].y >> 20], 1u);
            atomicAdd(&hist[k[u].z >> 20], 1u);
            atomicAdd(&hist[k[u].w >> 20], 1u);
        }
    }
    if (threadIdx.x < p1 - (v1 << 2)) atomicAdd(&hist[fkey(__ldg(row + (v1 << 2) + threadIdx.x)) >> 20], 1u);
    __syncthreads();
    uint32_t* g = sc.hist1 + (size_t)t * 4096;
    for (int b = threadIdx.x; b < 4096; b += kSplitThreads)
        if (hist[b]) atomicAdd(g + b, hist[b]);
}

__global__ void __launch_bounds__(kSplitThreads)
topk_split_mark_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                       bool n_from_pos, int64_t max_len, int K, const int32_t* __restrict__ cu_q,
                       const int32_t* __restrict__ cu_k, int B, int slices, uint32_t* scratch,
                       int32_t T, int64_t nw_cap) {
    pdl_wait();
    pdl_launch_dependents();
    using S = TopkSmem<kSplitThreads, 12>;
    __shared__ S sh;
    __shared__ uint32_t hist2[1024];
    const int t = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int64_t n64 = selecting_row(t, n_valid, n_from_pos, max_len, ld, K, cu_q, cu_k, B);
    const int32_t p0 = sl * kSplitSlice;
    if (n64 < 0 || p0 >= n64) return;                       // block-uniform
    const int32_t n = (int32_t)n64;
    const int32_t p1 = n < p0 + kSplitSlice ? n : p0 + kSplitSlice;
    const SplitScratch sc = split_scratch(scratch, T, nw_cap);
    const uint32_t* g1 = sc.hist1 + (size_t)t * 4096;
    for (int b = threadIdx.x; b < 4096; b += kSplitThreads) sh.hist[b] = g1[b];
    zero<kSplitThreads>(hist2, 1024);
    __syncthreads();
    select_bin<kSplitThreads>(sh, 4096, (uint32_t)K);
    const uint32_t b1 = sh.sel_bin;

    uint32_t* above = sc.bits + (size_t)t * 3 * nw_cap;
    uint32_t* tie = above + nw_cap;
    uint32_t* cand = tie + nw_cap;
    const float* row = scores + (int64_t)t * ld;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kSplitThreads / 32;
    // each warp: 128 consecutive positions per step (4 per lane), 4 steps in flight
    for (int32_t c0 = p0 + warp * 128; c0 < p1; c0 += kWarps * 128 * kUnroll) {
        float4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t p = c0 + u * kWarps * 128 + 4 * lane;
            x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p + 3 < p1) x[u] = __ldg(reinterpret_cast<const float4*>(row + p));
            else if (p < p1) {
                x[u].x = __ldg(row + p);
                if (p + 1 < p1) x[u].y = __ldg(row + p + 1);
                if (p + 2 < p1) x[u].z = __ldg(row + p + 2);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t cb = c0 + u * kWarps * 128;          // warp-uniform
            if (cb >= p1) break;
            const int32_t p = cb + 4 * lane;
            const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
            uint32_t ma = 0, mc = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (p + j >= p1) break;
                const uint32_t kk = fkey(xs[j]);
                const uint32_t d = kk >> 20;
                ma |= (d > b1 ? 1u : 0u) << j;
                if (d == b1) {
                    mc |= 1u << j;
                    atomicAdd(&hist2[(kk >> 10) & 1023u], 1u);
                }
            }
            const uint32_t wa = word_of_masks(ma), wc = word_of_masks(mc);
            if ((lane & 7) == 0) {
                const int32_t w = (cb >> 5) + (lane >> 3);
                if ((w << 5) < p1) {
                    above[w] = wa;
                    cand[w] = wc;
                    tie[w] = 0u;
                }
            }
        }
    }
    __syncthreads();
    uint32_t* g2 = sc.hist2 + (size_t)t * 1024;
    for (int b = threadIdx.x; b < 1024; b += kSplitThreads)
        if (hist2[b]) atomicAdd(g2 + b, hist2[b]);
}

__global__ void __launch_bounds__(kFinishThreads)
topk_split_finish_kernel(const float* __restrict__ scores, int64_t ld,
                         const int32_t* __restrict__ n_valid, bool n_from_pos, int T,
                         int64_t max_len, int K, int32_t* __restrict__ idx,
                         int32_t* __restrict__ cnt, DeviceStatus* status,
                         const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B,
                         uint32_t* scratch, int64_t nw_cap) {
    pdl_wait();
    pdl_launch_dependents();
    using S = TopkSmem<kFinishThreads, 12>;
    __shared__ S sh;
    extern __shared__ __align__(16) uint32_t dyn_list[];   // [kFinishCand] keys, positions
    uint32_t* cand_key = dyn_list;
    int32_t* cand_pos = reinterpret_cast<int32_t*>(dyn_list + kFinishCand);
    const int t = blockIdx.x;
    int32_t* out = idx + (int64_t)t * K;
    const int64_t n64 = row_prologue<kFinishThreads>(t, n_valid, n_from_pos, max_len, ld, K, out,
                                                     cnt, status, cu_q, cu_k, B,
                                                     scorer_gave_up(status));
    if (n64 < 0) return;
    const int32_t n = (int32_t)n64;
    const int32_t nw = (n + 31) >> 5;
    const SplitScratch sc = split_scratch(scratch, T, nw_cap);
    const float* row = scores + (int64_t)t * ld;
    uint32_t* above = sc.bits + (size_t)t * 3 * nw_cap;
    uint32_t* tie = above + nw_cap;
    const uint32_t* cand = tie + nw_cap;

    // digit 1 and digit 2 from the row histograms
    const uint32_t* g1 = sc.hist1 + (size_t)t * 4096;
    for (int b = threadIdx.x; b < 4096; b += kFinishThreads) sh.hist[b] = g1[b];
    __syncthreads();
    select_bin<kFinishThreads>(sh, 4096, (uint32_t)K);
    uint32_t prefix = sh.sel_bin << 20;
    uint32_t rank = sh.sel_rank;
    const uint32_t* g2 = sc.hist2 + (size_t)t * 1024;
    for (int b = threadIdx.x; b < 1024; b += kFinishThreads) sh.hist[b] = g2[b];
    __syncthreads();
    select_bin<kFinishThreads>(sh, 1024, rank);
    prefix |= sh.sel_bin << 10;
    rank = sh.sel_rank;

    // list the candidates' positions in shared memory (block scan of counts)
    const int32_t per = (nw + kFinishThreads - 1) / kFinishThreads;
    const int32_t w0 = threadIdx.x * per, w1 = w0 + per < nw ? w0 + per : nw;
    uint32_t mine = 0;
    for (int32_t w = w0; w < w1; ++w) mine += __popc(cand[w]);
    const uint32_t off = block_excl_scan<kFinishThreads>(sh, mine);
    if (threadIdx.x == kFinishThreads - 1) sh.cand_count = off + mine;
    __syncthreads();
    const uint32_t n_cand = sh.cand_count;
    const bool listed = n_cand <= (uint32_t)kFinishCand;
    if (listed) {
        uint32_t slot = off;
        for (int32_t w = w0; w < w1; ++w)
            for (uint32_t m = cand[w]; m; m &= m - 1u) cand_pos[slot++] = (w << 5) + (__ffs(m) - 1);
    }
    __syncthreads();
    // their keys, loads batched; digit 3 over them
    zero<kFinishThreads>(sh.hist, 1024);
    __syncthreads();
    if (listed) {
        for (uint32_t i0 = threadIdx.x; i0 < n_cand; i0 += 4 * kFinishThreads) {
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t i = i0 + u * kFinishThreads;
                x[u] = i < n_cand ? __ldg(row + cand_pos[i]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t i = i0 + u * kFinishThreads;
                if (i >= n_cand) break;
                const uint32_t kk = fkey(x[u]);
                cand_key[i] = kk;
                if ((kk & 0xFFFFFC00u) == prefix) atomicAdd(&sh.hist[kk & 1023u], 1u);
            }
        }
    } else {   // very many candidates: walk the bitmap, gathering per word
        for (int32_t w = threadIdx.x; w < nw; w += kFinishThreads) {
            for (uint32_t m = cand[w]; m; m &= m - 1u) {
                const uint32_t kk = fkey(__ldg(row + (w << 5) + (__ffs(m) - 1)));
                if ((kk & 0xFFFFFC00u) == prefix) atomicAdd(&sh.hist[kk & 1023u], 1u);
            }
        }
    }
    __syncthreads();
    select_bin<kFinishThreads>(sh, 1024, rank);
    const uint32_t tau = prefix | sh.sel_bin;
    const uint32_t need = sh.sel_rank;

    // mark candidates above tau (above bits) and equal to tau (tie bits), then emit
    if (listed) {
        for (uint32_t i = threadIdx.x; i < n_cand; i += kFinishThreads) {
            const uint32_t kk = cand_key[i];
            if (kk > tau) set_bit(above, cand_pos[i]);
            else if (kk == tau) set_bit(tie, cand_pos[i]);
        }
    } else {   // this thread owns word w
        for (int32_t w = threadIdx.x; w < nw; w += kFinishThreads) {
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
            above[w] |= a;
            tie[w] = e;
        }
    }
    __syncthreads();
    emit_ordered<kFinishThreads>(sh, above, tie, nw, out, (uint32_t)K, need);
    if (cnt && threadIdx.x == 0) cnt[t] = K;
}

// ---------------------------------------------------------------------------
// Few long rows: one cluster of C CTAs per row (C = 8, 4 or 2, chosen so that
// all rows fit in one wave). CTA r owns the slice [r*sl, (r+1)*sl) of the row
// (sl = ceil(n/C) rounded up to 128) and keeps that slice's above / tie / cand
// bitmaps and candidate list in its own shared memory.
//   digit 1  from hist1[t] (the scorer's epilogue histogram), or counted over
//            the slices and summed in the leader CTA (rank 0) through
//            distributed shared memory (DSMEM).
//   split    one pass over the slice. Lane l of a warp takes positions
//            cb + l + 32j of a 128-position chunk, so the warp's ballot of a
//            predicate is directly the bitmap word of positions
//            cb + 32j .. cb + 32j + 31. Scores are compared with the float
//            bounds of bin b1 (no key arithmetic for non-candidates).
//            Candidates (keys, positions) go to the CTA's list.
//   select   normally the leader gathers every CTA's candidate keys through
//            DSMEM, finds digits 2 and 3 alone, counts per CTA the candidates
//            above and equal to tau, and writes tau, need and each CTA's
//            output offsets into that CTA's shared memory. When a list
//            overflows (a large tie group), the CTAs instead sum their digit
//            counts in the leader and each walks its own cand bitmap.
//   emit     each CTA marks its candidates and writes its own positions at
//            its offsets: above positions first, then the first `need` tie
//            positions, both in increasing order across the cluster.
// ---------------------------------------------------------------------------
constexpr int kClusterMax = 8;
constexpr int kClThreads = 512;
constexpr int kClCand = 2048;            // candidates listed per CTA
constexpr int kClGather = 8192;          // candidate keys the leader gathers
constexpr int64_t kClSliceCap = 262144;  // longest slice (bitmaps in shared memory)
constexpr int64_t kClusterRowCap = kClusterMax * kClSliceCap;   // longest row of the cluster kernel

struct ClusterTopkSmem : TopkSmem<kClThreads, 12> {
    uint32_t h2[1024];                 // this CTA's candidates: second-digit counts
    uint32_t h3[1024];                 // this CTA's candidates: third-digit counts
    uint32_t m2[1024];                 // leader: the cluster's second-digit counts
    uint32_t m3[1024];                 // leader: the cluster's third-digit counts
    uint32_t n_above_b1;               // positions of this slice above bin b1
    uint32_t cta_cand[kClusterMax];    // every CTA's candidate count
    uint32_t cta_above[kClusterMax];   // every CTA's count above b1
    uint32_t ext_above[kClusterMax];   // leader: candidates above tau per CTA
    uint32_t ext_tie[kClusterMax];     // leader: candidates equal to tau per CTA
    uint32_t n_above[kClusterMax];     // leader (overflow path): marked positions per CTA
    uint32_t n_tie[kClusterMax];
    uint32_t seg[kClusterMax + 1];     // leader: first gathered key of each CTA
    uint32_t tau, need, a_off, t_off;  // written by the leader
};

__global__ void __launch_bounds__(kClThreads)
topk_cluster_kernel(const float* __restrict__ scores, int64_t ld,
                    const int32_t* __restrict__ n_valid, bool n_from_pos, int64_t max_len, int K,
                    int32_t* __restrict__ idx, int32_t* __restrict__ cnt, DeviceStatus* status,
                    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B,
                    const uint32_t* __restrict__ hist1, int32_t nw_slice_cap) {
    __shared__ ClusterTopkSmem sh;
    extern __shared__ __align__(16) uint32_t dyn_cl[];
    uint32_t* cand_key = dyn_cl;
    int32_t* cand_pos = reinterpret_cast<int32_t*>(dyn_cl + kClCand);
    uint32_t* g_key = dyn_cl + 2 * kClCand;          // leader: gathered keys
    uint32_t* above = g_key + kClGather;
    uint32_t* tie = above + nw_slice_cap;
    uint32_t* cand = tie + nw_slice_cap;
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int r = (int)cl.block_rank();
    const int t = blockIdx.x / C;
    int32_t* out = idx + (int64_t)t * K;
    if (hist1 == nullptr) zero<kClThreads>(sh.hist, 4096);
    zero<kClThreads>(sh.h2, 1024);
    zero<kClThreads>(sh.h3, 1024);
    zero<kClThreads>(sh.m2, 1024);
    zero<kClThreads>(sh.m3, 1024);
    if (threadIdx.x < kClusterMax) {
        sh.ext_above[threadIdx.x] = 0;
        sh.ext_tie[threadIdx.x] = 0;
        sh.n_above[threadIdx.x] = 0;
        sh.n_tie[threadIdx.x] = 0;
        sh.seg[threadIdx.x + 1] = 0;
    }
    if (threadIdx.x == 0) {
        sh.cand_count = 0;
        sh.n_above_b1 = 0;
        sh.seg[0] = 0;
    }
    // The row check reads only the call's inputs, which the kernels before
    // this one on the stream no longer write (each waits for its predecessor
    // before it lets its successor start), so it runs before pdl_wait;
    // outputs and the scores are touched after it. Every CTA of the cluster
    // takes the same decision; only the leader writes the output of a bad or
    // dormant row.
    const int64_t n64 = selecting_row(t, n_valid, n_from_pos, max_len, ld, K, cu_q, cu_k, B);
    pdl_wait();
    pdl_launch_dependents();
    // (the same in every CTA: only the scorer before this kernel writes a timeout)
    const bool gave_up = scorer_gave_up(status);
    if (n64 < 0 || gave_up) {   // the whole cluster returns, before any cluster barrier
        if (r == 0) row_prologue<kClThreads>(t, n_valid, n_from_pos, max_len, ld, K, out, cnt, status,
                                             cu_q, cu_k, B, gave_up);
        return;
    }
    if (hist1 != nullptr) {   // the row's first-digit histogram, from the scorer
        const uint4* g1 = reinterpret_cast<const uint4*>(hist1 + (size_t)t * 4096);
        uint4* h4 = reinterpret_cast<uint4*>(sh.hist);
        for (int b = threadIdx.x; b < 1024; b += kClThreads) h4[b] = g1[b];
    }
    const int32_t n = (int32_t)n64;
    const int32_t sl = (int32_t)((((int64_t)n + C - 1) / C + 127) / 128 * 128);
    const int32_t p0 = (int32_t)((int64_t)r * sl < n ? (int64_t)r * sl : n);
    const int32_t p1 = (int32_t)((int64_t)p0 + sl < n ? (int64_t)p0 + sl : n);
    const int32_t nwl = (p1 - p0 + 31) >> 5;          // this slice's bitmap words
    const float* row = scores + (int64_t)t * ld;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kClThreads / 32;
    ClusterTopkSmem* lead = cl.map_shared_rank(&sh, 0);
    __syncthreads();
    // Remote accesses come after the cluster barrier that ends the split pass
    // (every CTA has started and cleared its shared memory by then); only the
    // first-digit count below adds into the leader earlier, after a barrier.

    if (hist1 == nullptr) {   // digit 1: count the slice, sum in the leader
        cl.sync();
        // a non-empty slice starts at a multiple of 128; an empty one (p0 == n)
        // must not round p0 down into the previous slice
        const int32_t v_end = p0 < p1 ? (p1 + 3) >> 2 : (p0 >> 2);
        for (int32_t v = (p0 >> 2) + threadIdx.x; v < v_end; v += kClThreads) {
            const int32_t p = v << 2;
            if (p + 3 < p1) {
                const uint4 k = gkeys(row, v);
                atomicAdd(&sh.hist[k.x >> 20], 1u);
                atomicAdd(&sh.hist[k.y >> 20], 1u);
                atomicAdd(&sh.hist[k.z >> 20], 1u);
                atomicAdd(&sh.hist[k.w >> 20], 1u);
            } else {
                for (int32_t q = p; q < p1; ++q) atomicAdd(&sh.hist[fkey(__ldg(row + q)) >> 20], 1u);
            }
        }
        __syncthreads();
        if (r != 0)
            for (int b = threadIdx.x; b < 4096; b += kClThreads)
                if (sh.hist[b]) atomicAdd(&lead->hist[b], sh.hist[b]);
        cl.sync();
        if (r != 0)
            for (int b = threadIdx.x; b < 4096; b += kClThreads) sh.hist[b] = lead->hist[b];
        __syncthreads();
    }
    select_bin<kClThreads>(sh, 4096, (uint32_t)K);
    const uint32_t b1 = sh.sel_bin;
    uint32_t rank = sh.sel_rank;
    const float f_lo = key_floor((uint64_t)b1 << 20);          // bin b1 or above
    const float f_hi = key_floor((uint64_t)(b1 + 1) << 20);    // above bin b1

    // ---- split: one pass over the slice
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t my_above = 0;   // lane 0: above-b1 positions seen by this warp
    for (int32_t c0 = p0 + warp * 128; c0 < p1; c0 += kWarps * 128 * kUnroll) {
        float x[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int32_t p = c0 + u * kWarps * 128 + 32 * j + lane;
                x[u][j] = p < p1 ? __ldg(row + p) : __int_as_float(0x7fffffff);   // NaN: never kept
            }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t cb = c0 + u * kWarps * 128;          // warp-uniform
            if (cb >= p1) break;
            uint32_t ba[4], bc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool a = x[u][j] >= f_hi;
                ba[j] = __ballot_sync(0xffffffffu, a);
                bc[j] = __ballot_sync(0xffffffffu, !a && x[u][j] >= f_lo);
            }
            const int32_t w = (cb - p0) >> 5;                   // p0 is a multiple of 128
            if (lane < 4 && w + lane < nwl) {
                above[w + lane] = lane == 0 ? ba[0] : lane == 1 ? ba[1] : lane == 2 ? ba[2] : ba[3];
                cand[w + lane] = lane == 0 ? bc[0] : lane == 1 ? bc[1] : lane == 2 ? bc[2] : bc[3];
                tie[w + lane] = 0u;
            }
            if (lane == 0) my_above += __popc(ba[0]) + __popc(ba[1]) + __popc(ba[2]) + __popc(ba[3]);
            if ((bc[0] | bc[1] | bc[2] | bc[3]) != 0u) {      // warp-uniform
                const uint32_t tot = __popc(bc[0]) + __popc(bc[1]) + __popc(bc[2]) + __popc(bc[3]);
                uint32_t base = 0;
                if (lane == 0) base = atomicAdd(&sh.cand_count, tot);
                base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if ((bc[j] >> lane) & 1u) {
                        const uint32_t slot = base + __popc(bc[j] & lt_mask);
                        const uint32_t kk = fkey(x[u][j]);
                        if (slot < (uint32_t)kClCand) {
                            cand_key[slot] = kk;
                            cand_pos[slot] = cb + 32 * j + lane;
                        }
                        atomicAdd(&sh.h2[(kk >> 10) & 1023u], 1u);
                    }
                    base += __popc(bc[j]);
                }
            }
        }
    }
    if (lane == 0 && my_above) atomicAdd(&sh.n_above_b1, my_above);
    __syncthreads();
    cl.sync();   // every CTA's bitmaps, list and counts are complete

    if (warp == 0 && lane < C) {
        const ClusterTopkSmem* rs = cl.map_shared_rank(&sh, lane);
        sh.cta_cand[lane] = rs->cand_count;
        sh.cta_above[lane] = rs->n_above_b1;
    }
    __syncthreads();
    uint32_t total_cand = 0;
    bool fits = true;
    for (int i = 0; i < C; ++i) {
        total_cand += sh.cta_cand[i];
        fits = fits && sh.cta_cand[i] <= (uint32_t)kClCand;
    }
    const bool gathered = fits && total_cand <= (uint32_t)kClGather;   // same in every CTA
    const uint32_t n_cand = sh.cand_count;
    const bool listed = n_cand <= (uint32_t)kClCand;

    uint32_t tau, need, a_base, t_base;
    if (gathered) {
        if (r == 0) {
            // the cluster's candidate keys, CTA by CTA
            if (threadIdx.x == 0)
                for (int i = 0; i < C; ++i) sh.seg[i + 1] = sh.seg[i] + sh.cta_cand[i];
            __syncthreads();
            for (uint32_t e = threadIdx.x; e < total_cand; e += kClThreads) {   // one round trip
                int i = 0;
                while (i + 1 < C && e >= sh.seg[i + 1]) ++i;
                g_key[e] = cl.map_shared_rank(cand_key, i)[e - sh.seg[i]];
            }
            zero<kClThreads>(sh.hist, 1024);
            __syncthreads();
            for (uint32_t e = threadIdx.x; e < total_cand; e += kClThreads)
                atomicAdd(&sh.hist[(g_key[e] >> 10) & 1023u], 1u);
            __syncthreads();
            select_bin<kClThreads>(sh, 1024, rank);
            const uint32_t prefix = (b1 << 20) | (sh.sel_bin << 10);
            const uint32_t rank3 = sh.sel_rank;
            __syncthreads();
            zero<kClThreads>(sh.hist, 1024);
            __syncthreads();
            for (uint32_t e = threadIdx.x; e < total_cand; e += kClThreads) {
                const uint32_t kk = g_key[e];
                if ((kk & 0xFFFFFC00u) == prefix) atomicAdd(&sh.hist[kk & 1023u], 1u);
            }
            __syncthreads();
            select_bin<kClThreads>(sh, 1024, rank3);
            const uint32_t tau0 = prefix | sh.sel_bin;
            const uint32_t need0 = sh.sel_rank < (uint32_t)K ? sh.sel_rank : (uint32_t)K;
            for (uint32_t e = threadIdx.x; e < total_cand; e += kClThreads) {
                const uint32_t kk = g_key[e];
                if (kk < tau0) continue;
                int i = 0;
                while (i + 1 < C && e >= sh.seg[i + 1]) ++i;
                atomicAdd(kk > tau0 ? &sh.ext_above[i] : &sh.ext_tie[i], 1u);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t a = 0, e = 0;
                for (int i = 0; i < C; ++i) {
                    ClusterTopkSmem* rs = cl.map_shared_rank(&sh, i);
                    rs->tau = tau0;
                    rs->need = need0;
                    rs->a_off = a;
                    rs->t_off = e;
                    a += sh.cta_above[i] + sh.ext_above[i];
                    e += sh.ext_tie[i];
                }
            }
        }
        cl.sync();   // tau, need and offsets are in every CTA; no DSMEM access after this
        tau = sh.tau;
        need = sh.need;
        a_base = sh.a_off;
        t_base = sh.t_off;
        for (uint32_t i = threadIdx.x; i < n_cand; i += kClThreads) {
            const uint32_t kk = cand_key[i];
            if (kk > tau) set_bit(above, cand_pos[i] - p0);
            else if (kk == tau) set_bit(tie, cand_pos[i] - p0);
        }
    } else {
        // digit 2 from the cluster's summed counts
        for (int b = threadIdx.x; b < 1024; b += kClThreads)
            if (sh.h2[b]) atomicAdd(&lead->m2[b], sh.h2[b]);
        cl.sync();
        for (int b = threadIdx.x; b < 1024; b += kClThreads) sh.hist[b] = lead->m2[b];
        __syncthreads();
        select_bin<kClThreads>(sh, 1024, rank);
        const uint32_t prefix = (b1 << 20) | (sh.sel_bin << 10);
        rank = sh.sel_rank;
        // digit 3 over this slice's candidates that share the first two digits
        if (listed) {
            for (uint32_t i = threadIdx.x; i < n_cand; i += kClThreads) {
                const uint32_t kk = cand_key[i];
                if ((kk & 0xFFFFFC00u) == prefix) atomicAdd(&sh.h3[kk & 1023u], 1u);
            }
        } else {
            for (int32_t w = threadIdx.x; w < nwl; w += kClThreads)
                for (uint32_t m = cand[w]; m; m &= m - 1u) {
                    const uint32_t kk = fkey(__ldg(row + p0 + (w << 5) + (__ffs(m) - 1)));
                    if ((kk & 0xFFFFFC00u) == prefix) atomicAdd(&sh.h3[kk & 1023u], 1u);
                }
        }
        __syncthreads();
        for (int b = threadIdx.x; b < 1024; b += kClThreads)
            if (sh.h3[b]) atomicAdd(&lead->m3[b], sh.h3[b]);
        cl.sync();
        for (int b = threadIdx.x; b < 1024; b += kClThreads) sh.hist[b] = lead->m3[b];
        __syncthreads();
        select_bin<kClThreads>(sh, 1024, rank);
        tau = prefix | sh.sel_bin;
        need = sh.sel_rank < (uint32_t)K ? sh.sel_rank : (uint32_t)K;
        // mark this slice's candidates
        if (listed) {
            for (uint32_t i = threadIdx.x; i < n_cand; i += kClThreads) {
                const uint32_t kk = cand_key[i];
                if (kk > tau) set_bit(above, cand_pos[i] - p0);
                else if (kk == tau) set_bit(tie, cand_pos[i] - p0);
            }
        } else {   // this thread owns word w
            for (int32_t w = threadIdx.x; w < nwl; w += kClThreads) {
                uint32_t m = cand[w];
                if (!m) continue;
                uint32_t a = 0, e = 0;
                while (m) {
                    const int b = __ffs(m) - 1;
                    m &= m - 1u;
                    const uint32_t kk = fkey(__ldg(row + p0 + (w << 5) + b));
                    a |= (kk > tau ? 1u : 0u) << b;
                    e |= (kk == tau ? 1u : 0u) << b;
                }
                above[w] |= a;
                tie[w] = e;
            }
        }
        // per-CTA totals of marked positions, summed in the leader
        __syncthreads();
        uint32_t ca = 0, ct = 0;
        for (int32_t w = threadIdx.x; w < nwl; w += kClThreads) {
            ca += __popc(above[w]);
            ct += __popc(tie[w]);
        }
        if (ca) atomicAdd(&lead->n_above[r], ca);
        if (ct) atomicAdd(&lead->n_tie[r], ct);
        cl.sync();
        a_base = 0;
        t_base = 0;
        for (int i = 0; i < r; ++i) {
            a_base += lead->n_above[i];
            t_base += lead->n_tie[i];
        }
    }
    __syncthreads();

    // ---- emit: offsets inside the CTA from a block scan of packed counts
    const uint32_t n_above_all = (uint32_t)K - need;
    const int32_t per = (nwl + kClThreads - 1) / kClThreads;
    const int32_t w0 = threadIdx.x * per < nwl ? threadIdx.x * per : nwl;
    const int32_t w1 = w0 + per < nwl ? w0 + per : nwl;
    uint32_t ca = 0, ct = 0;
    for (int32_t w = w0; w < w1; ++w) {
        ca += __popc(above[w]);
        ct += __popc(tie[w]);
    }
    const uint64_t off = block_excl_scan64<kClThreads>(sh, (uint64_t)ca | ((uint64_t)ct << 32));
    uint32_t pa = a_base + (uint32_t)off, pt = t_base + (uint32_t)(off >> 32);
    for (int32_t w = w0; w < w1; ++w) {
        uint32_t m = above[w];
        while (m && pa < n_above_all) {
            out[pa++] = p0 + w * 32 + (__ffs(m) - 1);
            m &= m - 1u;
        }
        m = tie[w];
        while (m && pt < need) {
            out[n_above_all + pt++] = p0 + w * 32 + (__ffs(m) - 1);
            m &= m - 1u;
        }
    }
    if (r == 0 && cnt && threadIdx.x == 0) cnt[t] = K;
    if (!gathered) cl.sync();   // the leader's counters were read until here
}

// Shared memory a block may use in total (GB300 opt-in limit, 227 KB), and a
// bound on the streamed kernel's static part (histogram, scans, counters, with
// alignment padding).
constexpr int64_t kBlockSmem = 227 * 1024;
constexpr int64_t kStreamStaticBound = (int64_t)sizeof(TopkSmem<kStreamThreads, 12>) + 256;
constexpr int64_t kStreamList = 8192;   // candidates listed in shared memory (64 KB)

// The three bitmaps, rounded up to 16 bytes (the candidate list follows them).
bool bitmaps_fit_in_smem(int64_t row_cap) {
    const int64_t nw_cap = (row_cap + 31) / 32;
    return (3 * nw_cap + 3) / 4 * 16 + kStreamStaticBound <= kBlockSmem;
}

}  // namespace

// CTAs per row for the cluster kernel: the largest of 8, 4, 2 that keeps all
// T rows in one wave at two CTAs per SM, raised again (up to 8) while a slice
// would exceed kClSliceCap positions. Rows up to kClusterRowCap always fit.
static int cluster_ctas(int32_t T, int64_t row_cap) {
    const int64_t slots = 2 * (int64_t)(device_info().sm_count > 0 ? device_info().sm_count : 1);
    int c = (int64_t)T * 8 <= slots ? 8 : (int64_t)T * 4 <= slots ? 4 : 2;
    while (c < kClusterMax && ((row_cap + c - 1) / c + 127) / 128 * 128 > kClSliceCap) c *= 2;
    return c;
}

static bool uses_split(const TopkArgs& a) {
    const int64_t row_cap = a.max_len < a.ld ? a.max_len : a.ld;
    return a.T > 0 && a.T <= kSplitMaxRows && row_cap > kStageCap && a.bits_scratch != nullptr;
}

uint32_t* topk_split_row_hist(const TopkArgs& a) { return uses_split(a) ? a.bits_scratch : nullptr; }

void topk_prepare(TopkArgs* a, void** ptr, size_t* bytes) {
    *ptr = nullptr;
    *bytes = 0;
    if (!uses_split(*a) || a->hist_state != 0) return;
    *ptr = a->bits_scratch;
    *bytes = split_hist_bytes(a->T);
    a->hist_state = 1;
}

size_t topk_scratch_bytes(int32_t T, int64_t max_len) {
    if (T <= 0 || max_len <= kStageCap) return 0;
    const size_t nw_cap = (size_t)((max_len + 31) / 32);
    if (T <= kSplitMaxRows)
        return split_hist_bytes(T) + (max_len <= kClusterRowCap ? 0 : (size_t)T * 3 * nw_cap * 4);
    if (bitmaps_fit_in_smem(max_len)) return 0;
    return (size_t)kScratchBlocks * 3 * nw_cap * 4;
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
        e = launch_kernel(kern, dim3(grid), dim3(kStagedThreads), smem, stream, 1, a.scores, a.ld,
                          a.n_valid, a.n_from_pos, a.T, a.max_len, a.topk, a.idx, a.cnt, a.status,
                          a.cu_q, a.cu_k, a.B, stage);
        if (e != cudaSuccess) return e;
    } else if (a.T <= kSplitMaxRows && row_cap <= kClusterRowCap) {
        const int C = cluster_ctas(a.T, row_cap);
        const int64_t sl_cap = ((row_cap + C - 1) / C + 127) / 128 * 128;
        const int32_t nw_slice_cap = (int32_t)(sl_cap / 32);
        const size_t smem = ((size_t)2 * kClCand + kClGather + 3 * (size_t)nw_slice_cap) * 4;
        cudaError_t e = ensure_smem_optin((const void*)topk_cluster_kernel,
                                          ((int64_t)2 * kClCand + kClGather + 3 * (kClSliceCap / 32)) * 4);
        if (e != cudaSuccess) return e;
        const uint32_t* h1 = a.hist_state == 2 ? a.bits_scratch : nullptr;
        e = launch_kernel(topk_cluster_kernel, dim3((unsigned)(a.T * C)), dim3(kClThreads), smem, stream,
                          C, a.scores, a.ld, a.n_valid, a.n_from_pos, a.max_len, a.topk, a.idx, a.cnt,
                          a.status, a.cu_q, a.cu_k, a.B, h1, nw_slice_cap);
        if (e != cudaSuccess) return e;
    } else if (a.T <= kSplitMaxRows) {
        if (a.bits_scratch == nullptr) return cudaErrorInvalidValue;
        if (a.hist_state == 0) {
            cudaError_t e = cudaMemsetAsync(a.bits_scratch, 0, split_hist_bytes(a.T), stream);
            if (e != cudaSuccess) return e;
        }
        const int slices = (int)((row_cap + kSplitSlice - 1) / kSplitSlice);
        const int64_t blocks = (int64_t)a.T * slices;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
        if (a.hist_state != 2) {   // the scorer did not histogram the rows
            cudaError_t e = launch_kernel(topk_split_hist_kernel, dim3((unsigned)blocks), dim3(kSplitThreads),
                                          0, stream, 1, a.scores, a.ld, a.n_valid, a.n_from_pos,
                                          a.max_len, a.topk, a.cu_q, a.cu_k, a.B, slices,
                                          a.bits_scratch, a.T, nw_cap);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e1 = launch_kernel(topk_split_mark_kernel, dim3((unsigned)blocks), dim3(kSplitThreads),
                                       0, stream, 1, a.scores, a.ld, a.n_valid, a.n_from_pos,
                                       a.max_len, a.topk, a.cu_q, a.cu_k, a.B, slices, a.bits_scratch,
                                       a.T, nw_cap);
        if (e1 != cudaSuccess) return e1;
        const int64_t list_bytes = (int64_t)kFinishCand * 8;
        cudaError_t e2 = ensure_smem_optin((const void*)topk_split_finish_kernel, list_bytes);
        if (e2 != cudaSuccess) return e2;
        e2 = launch_kernel(topk_split_finish_kernel, dim3(a.T), dim3(kFinishThreads), (size_t)list_bytes,
                           stream, 1, a.scores, a.ld, a.n_valid, a.n_from_pos, a.T, a.max_len, a.topk,
                           a.idx, a.cnt, a.status, a.cu_q, a.cu_k, a.B, a.bits_scratch, nw_cap);
        if (e2 != cudaSuccess) return e2;
    } else {
        const bool in_smem = bitmaps_fit_in_smem(row_cap);
        if (!in_smem && a.bits_scratch == nullptr) return cudaErrorInvalidValue;
        const int64_t bm_bytes = in_smem ? (3 * nw_cap + 3) / 4 * 16 : 0;
        const int64_t room = in_smem ? (kBlockSmem - kStreamStaticBound - bm_bytes) / 8 : 0;
        const int32_t list_cap = (int32_t)(room < 0 ? 0 : room < kStreamList ? room : kStreamList);
        const size_t smem = (size_t)(bm_bytes + (int64_t)list_cap * 8);
        const int g = in_smem ? grid : (grid < kScratchBlocks ? grid : kScratchBlocks);
        auto kern = topk_stream_kernel<kStreamThreads>;
        const int64_t st = kernel_static_smem((const void*)kern);
        if (st < 0 || st > kStreamStaticBound) return cudaErrorInvalidValue;
        cudaError_t e = ensure_smem_optin((const void*)kern, kBlockSmem - kStreamStaticBound);
        if (e != cudaSuccess) return e;
        e = launch_kernel(kern, dim3(g), dim3(kStreamThreads), smem, stream, 1, a.scores, a.ld,
                          a.n_valid, a.n_from_pos, a.T, a.max_len, a.topk, a.idx, a.cnt, a.status,
                          a.cu_q, a.cu_k, a.B, nw_cap, in_smem ? nullptr : a.bits_scratch, list_cap);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace lidx

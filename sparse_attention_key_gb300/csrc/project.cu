// Indexer projections: the inputs of the indexer from the layer's activations.
//
// "Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph: the query
// comes off the normalised q-LoRA projection, the key from the attention input
// through the 128-wide LayerNorm with weight and bias, and a per-head weight
// vector sums the heads. Read plainly, per token t:
//   q[t]      = W_q  . qlora[t]      W_q  [32*128, rank]   -> bf16 [32,128]
//   k_pre[t]  = W_k  . x[t]          W_k  [128, hidden]    -> bf16 [128]
//   k[slot t] = LayerNorm(k_pre[t])  (the key cache)       -> bf16 [128]
//   w[t]      = W_w  . x[t]          W_w  [32, hidden]     -> fp32 [32]
// (weights in the [out, in] layout of a linear layer; any scale of w is part
// of W_w).
//
// All three products have the form C[M,N] = A[M,K] . B[N,K]^T with both
// operands K-major (rows of K contiguous bf16), which is the operand layout of
// the tensor core's MMA. One persistent, warp-specialised tcgen05 kernel runs
// them:
//   warp 0      TMA producer: per 64-wide K block, the A tile [128 rows, 64]
//               and the B tile [BN rows, 64] (128-byte swizzle) into a ring
//               of STAGES shared-memory stages;
//   warp 1      TMEM allocator and MMA issuer (one thread): 4 MMAs of
//               M=128 x N=BN x K=16 per K block into one of two accumulators;
//   warps 2..5  epilogue: tcgen05.ld of 32 columns at a time (one output row
//               per thread), then bf16 stores (round to nearest even) or fp32
//               partial sums.
// CTAs run in clusters of two that compute two adjacent row tiles of the same
// column tile: each CTA loads its own A tile and half of the shared B tile,
// which TMA multicasts into both CTAs' shared memory, so each SM reads 3/4 of
// the bytes it would alone. An MMA's completion is committed to the "stage
// empty" barriers of both CTAs (count 2): neither CTA refills a stage before
// both have consumed it. Work items are (row-tile pair, column tile, K split),
// dealt round-robin to the clusters, so the epilogue of one item overlaps the
// MMAs of the next. The key and weight products share one item of N = 128 + 32
// = 160 columns (the B tile is filled from W_k and W_w), so x is read once. When there
// are fewer row/column tiles than SMs (few tokens: the weights must stream
// from every SM), K is split and a second kernel sums the fp32 partials. The
// key/weight product always ends in one finishing kernel: it sums the splits,
// rounds k_pre to bf16, writes w (fp32) and appends LayerNorm(k_pre) to the
// cache with the same arithmetic as idx_key_layernorm_append (bit-identical).
//
// Every wait is bounded (idx_set_wait_limit_ns); a timeout records
// IDX_ERR_TIMEOUT in the status word at the start of the workspace (read it
// with idx_get_status), stops all roles, drains copies and MMAs already issued
// (100 ms bound) and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ln_row.cuh"
#include "tc_primitives.cuh"

namespace lidx {

namespace {

// Splits the finishing kernel loads per round (each round is a dependent
// memory round trip): 8, or 4 when no product has more splits (fewer
// registers, so all of a large T's tokens are resident at once).
constexpr int kFinishRound = 8;

constexpr int kGemmBM = 128;   // rows of A per tile (TMEM lanes)
constexpr int kGemmBK = 64;    // K per stage: one 128-byte swizzled row
constexpr int kGemmThreads = 6 * 32;
constexpr uint64_t kGemmDrainNs = 100000000ull;
constexpr int kGemmStages = 4;
constexpr int kGemmBNMax = 256;                              // columns per item, at most
constexpr int kGemmABytes = kGemmBM * kGemmBK * 2;           // 16 KB
constexpr int kGemmStage = kGemmABytes + kGemmBNMax * kGemmBK * 2;   // 48 KB
// epilogue staging: per epilogue warp two buffers of a 32 x 32 fp32 sub-tile
constexpr int kGemmOutBuf = 32 * 32 * 4;
constexpr int kGemmOutOff = kGemmStages * kGemmStage;
constexpr int kGemmBarOff = kGemmOutOff + 4 * 2 * kGemmOutBuf;
constexpr int kGemmSmem = kGemmBarOff + 8 * (2 * kGemmStages + 5) + 16;
constexpr int kGemmTmemCols = 2 * kGemmBNMax;               // two accumulators
static_assert(kGemmSmem <= 227 * 1024, "shared memory");
static_assert(kGemmABytes % 1024 == 0 && kGemmStage % 1024 == 0, "swizzled tiles stay 1024-byte aligned");

// Rows of the B tile that one CTA of the pair loads (and multicasts): from
// tensor map `map` of the problem, rows nt*BN + src_row .. + rows, to tile
// rows dst_row ..
struct BSeg {
    int map, src_row, dst_row, rows;
};

// One product C[M,N] = A[M,K] . B[N,K]^T of a grouped launch.
struct GemmProblem {
    int M, N;          // output rows (tokens) and columns
    int KB;            // 64-wide K blocks
    int m_pairs, n_tiles, splits;
    int BN;            // columns per item (multiple of 32, <= kGemmBNMax)
    int items;         // m_pairs * n_tiles * splits
    int out_bf16;      // 1: bf16 result [M, N]; 0: fp32 partials [splits, M, N]
    int nseg[2];       // B segments of cluster rank 0 and 1
    BSeg seg[2][2];
};

struct GemmGroup {
    GemmProblem p[2];
    int n_problems;    // 1 or 2
    int items;         // all problems' items
};

struct GemmMaps {   // CUtensorMap's own alignment keeps every map 64-byte aligned
    CUtensorMap a[2];      // A of each problem
    CUtensorMap b[2][3];   // B maps of each problem (BSeg::map)
    CUtensorMap out[2];    // output (bf16 2-D, or fp32 partials 3-D)
};
static_assert(alignof(GemmMaps) >= 64 && sizeof(CUtensorMap) % 64 == 0, "tensor maps 64-byte aligned");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Item g of the group: problem and item within it. The two problems' items
// are interleaved evenly (problem 0 takes item g when floor((g+1) I0 / I)
// grows), so every cluster gets a similar mix of both.
__device__ __forceinline__ void group_item(const GemmGroup& G, int g, int& p, int& i) {
    if (G.n_problems == 1) {
        p = 0;
        i = g;
        return;
    }
    const int64_t I = G.items, I0 = G.p[0].items;
    const int64_t before = (int64_t)g * I0 / I, upto = (int64_t)(g + 1) * I0 / I;
    if (upto > before) {
        p = 0;
        i = (int)before;
    } else {
        p = 1;
        i = (int)(g - upto);
    }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmGroup G, DeviceStatus* status,
               uint64_t wait_ns) {
    using namespace ptx;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // (the same outcome in both CTAs of a cluster: they return together)
    if ((smem_addr(smem_raw) & 1023u) != 0) {   // swizzled tiles need 1024-byte alignment
        pdl_wait();
        if (threadIdx.x == 0) report_error(status, IDX_ERR_UNSUPPORTED, 1024);
        return;
    }
    const int rank = (int)cluster_rank();           // 0 or 1
    const int cluster = (int)blockIdx.x >> 1, clusters = (int)gridDim.x >> 1;
    constexpr uint16_t kPair = 0x3;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + kGemmBarOff);
    uint64_t* empty = full + kGemmStages;
    uint64_t* acc_full = empty + kGemmStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;        // [2]
    uint64_t* done_bar = acc_empty + 2;        // the MMA issuer's final drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 2);   // the MMA commits of both CTAs of the pair
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full + a, 1);
            mbar_init(acc_empty + a, 4);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < G.n_problems; ++p) {
            prefetch_tmap(&maps.a[p]);
            for (int m = 0; m < 3; ++m) prefetch_tmap(&maps.b[p][m]);
            prefetch_tmap(&maps.out[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kGemmTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    // both CTAs' barriers are initialised before either multicasts into the other
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    bool aborted = false;
    auto give_up = [&](int site) {
        if (!*abort_flag) report_error(status, IDX_ERR_TIMEOUT, site);
        *abort_flag = 1;
        aborted = true;
    };
    // item i of problem P -> (row tile, column tile, split, K blocks [kb0, kb1))
    auto decode = [&](const GemmProblem& P, int i, int& mt, int& nt, int& sp, int& kb0, int& kb1) {
        sp = i % P.splits;
        const int rest = i / P.splits;
        nt = rest % P.n_tiles;
        mt = 2 * (rest / P.n_tiles) + rank;   // may pass the last row tile: rows read as zero
        kb0 = (int)((int64_t)P.KB * sp / P.splits);
        kb1 = (int)((int64_t)P.KB * (sp + 1) / P.splits);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued[kGemmStages];
#pragma unroll
            for (int s = 0; s < kGemmStages; ++s) issued[s] = 0;
            for (int g = cluster; g < G.items && !aborted; g += clusters) {
                int p, i, mt, nt, sp, kb0, kb1;
                group_item(G, g, p, i);
                const GemmProblem& P = G.p[p];
                decode(P, i, mt, nt, sp, kb0, kb1);
                const uint32_t bytes = (uint32_t)(kGemmABytes + P.BN * kGemmBK * 2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty + stage, phase ^ 1, abort_flag, wait_ns)) {
                        give_up(11);
                        break;
                    }
                    uint8_t* dst = smem_raw + stage * kGemmStage;
                    mbar_arrive_expect_tx(full + stage, bytes);
                    tma_load_2d(smem_addr(dst), &maps.a[p], full + stage, kb * kGemmBK, mt * kGemmBM);
                    // this CTA's share of the B tile, into both CTAs of the pair
                    for (int s = 0; s < P.nseg[rank]; ++s) {
                        const BSeg sg = P.seg[rank][s];
                        tma_load_2d_multicast(smem_addr(dst + kGemmABytes + sg.dst_row * 128),
                                              &maps.b[p][sg.map], full + stage, kb * kGemmBK,
                                              nt * P.BN + sg.src_row, kPair);
                    }
                    ++issued[stage];
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // let every copy this lane issued (and the other CTA's halves) land
            for (int s = 0; s < kGemmStages; ++s)
                if (issued[s] > 0) mbar_wait(full + s, (issued[s] - 1) & 1, nullptr, kGemmDrainNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_addr(smem_raw);
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            for (int g = cluster; g < G.items && !aborted; g += clusters) {
                int p, i, mt, nt, sp, kb0, kb1;
                group_item(G, g, p, i);
                const GemmProblem& P = G.p[p];
                decode(P, i, mt, nt, sp, kb0, kb1);
                const uint32_t idesc = idesc_bf16_f32(kGemmBM, P.BN);
                if (!mbar_wait(acc_empty + acc, aphase ^ 1, abort_flag, wait_ns)) {
                    give_up(12);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kGemmBNMax;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full + stage, phase, abort_flag, wait_ns)) {
                        give_up(13);
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = base + stage * kGemmStage;
                    const uint32_t b_addr = a_addr + kGemmABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + kk * 32),
                                    smem_desc_sw128(b_addr + kk * 32), idesc,
                                    (kb > kb0 || kk > 0) ? 1u : 0u);
                    tc_commit_multicast(empty + stage, kPair);   // frees the stage in both CTAs
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (aborted) break;
                tc_commit(acc_full + acc);
                if (++acc == 2) {
                    acc = 0;
                    aphase ^= 1;
                }
            }
            // wait for every MMA issued (and thereby for the arrivals of the
            // commits before this one) before shared and tensor memory go
            tc_commit(done_bar);
            mbar_wait(done_bar, 0, nullptr, kGemmDrainNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Each thread holds one output row; per 32-column chunk the warp
        // stages its 32 x 32 sub-tile in shared memory (row-major) and one
        // lane writes it with a TMA store, so global writes are whole boxes.
        const int quarter = warp & 3;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        uint8_t* obuf = smem_raw + kGemmOutOff + (warp - 2) * 2 * kGemmOutBuf;
        int acc = 0, nbuf = 0;
        uint32_t aphase = 0;
        for (int g = cluster; g < G.items && !aborted; g += clusters) {
            int p, i, mt, nt, sp, kb0, kb1;
            group_item(G, g, p, i);
            const GemmProblem& P = G.p[p];
            decode(P, i, mt, nt, sp, kb0, kb1);
            if (!mbar_wait(acc_full + acc, aphase, abort_flag, wait_ns)) {
                give_up(14);
                break;
            }
            tc_fence_after_sync();
            const int row0 = mt * kGemmBM + quarter * 32;   // this warp's first row
            const bool rows_ok = row0 < P.M;                  // warp-uniform
#pragma unroll 1
            for (int c = 0; c < P.BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld_x32(lane_base + acc * kGemmBNMax + c * 32, v);
                tmem_ld_wait(v);
                const int col = nt * P.BN + c * 32;
                if (!rows_ok || col >= P.N) continue;         // warp-uniform
                uint8_t* buf = obuf + (nbuf & 1) * kGemmOutBuf;
                if (lane == 0) bulk_wait_group_read<1>();    // the store that last used buf has read it
                __syncwarp();
                if (P.out_bf16) {
                    uint4* d = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d[j] = make_uint4(
                            f32x2_to_bf16x2_rn(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
                            f32x2_to_bf16x2_rn(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                            f32x2_to_bf16x2_rn(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                            f32x2_to_bf16x2_rn(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
                } else {
                    uint4* d = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
                    for (int j = 0; j < 8; ++j) d[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (P.out_bf16) tma_store_2d(&maps.out[p], smem_addr(buf), col, row0);
                    else tma_store_3d(&maps.out[p], smem_addr(buf), col, row0, sp);
                    bulk_commit_group();
                }
                ++nbuf;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + acc);
            if (++acc == 2) {
                acc = 0;
                aphase ^= 1;
            }
        }
        if (lane == 0) bulk_wait_group<0>();   // every store written before the CTA exits
    }

    // ---------------------------------------------------------------- teardown
    // (each CTA has drained its own copies, which include the other CTA's
    // multicast halves, and its MMAs, whose commits reach both CTAs; after the
    // cluster barrier neither CTA writes into the other's shared memory)
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kGemmTmemCols);
    }
}

// The end of a projection call (after the grouped GEMM):
//   blocks [0, q_blocks): when the q product was split, the sum of its K
//     splits' partials [splits][T][4096] in split order, rounded once to bf16
//     into q (one thread per 4 columns);
//   the other blocks: the key/weight product, per token (a half warp each):
//     the sum of its splits' partials [splits][T][160] in split order, k_pre =
//     that sum rounded to bf16 (the 16-bit activation), w = columns 128..159
//     (fp32), and the key LayerNorm of k_pre into row slot[t] of the cache
//     (ln_row_half_warp, as idx_key_layernorm_append: the same bits; slots
//     outside [0, cache_rows) write nothing).
// Loads of up to kB splits are in flight at a time; the additions keep the
// split order.
template <bool kF32Params, int kB>
__global__ void __launch_bounds__(256, kB <= 4 ? 3 : 2)
project_finish_kernel(const float* __restrict__ q_partial, int q_splits, uint16_t* __restrict__ q,
                      int q_blocks, const float* __restrict__ kw_partial, int kw_splits, int T,
                      const void* __restrict__ ln_w, const void* __restrict__ ln_b, float eps,
                      uint4* __restrict__ k_cache, int64_t cache_rows,
                      const int64_t* __restrict__ slot, float* __restrict__ w_out) {
    pdl_wait();
    pdl_launch_dependents();
    if ((int)blockIdx.x < q_blocks) {
        constexpr int kNq4 = IDX_HEADS * IDX_DIM / 4;
        const int64_t vecs = (int64_t)T * kNq4;
        const float4* part = reinterpret_cast<const float4*>(q_partial);
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs;
             i += (int64_t)q_blocks * blockDim.x) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < q_splits; s0 += kB) {
                float4 v[kB];
#pragma unroll
                for (int u = 0; u < kB; ++u)
                    v[u] = s0 + u < q_splits ? __ldg(part + (int64_t)(s0 + u) * vecs + i)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    if (s0 + u >= q_splits) break;
                    acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
                }
            }
            *reinterpret_cast<uint2*>(q + 4 * i) =
                make_uint2(f32x2_to_bf16x2_rn(acc.x, acc.y), f32x2_to_bf16x2_rn(acc.z, acc.w));
        }
        return;
    }
    const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
    const int64_t warp_id = ((int64_t)(blockIdx.x - q_blocks) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)(gridDim.x - q_blocks) * blockDim.x) >> 5;
    constexpr int kN = IDX_DIM + IDX_HEADS;
    for (int64_t t0 = 2 * warp_id; t0 < T; t0 += 2 * n_warps) {   // warp-uniform
        const int64_t t = t0 + half;
        const bool ok = t < T;
        float4 ka = make_float4(0.f, 0.f, 0.f, 0.f), kb = ka;
        float2 wv = make_float2(0.f, 0.f);
        const int64_t sr = ok ? __ldg(slot + t) : -1;   // (issued early: used at the end)
        if (ok) {
            for (int s0 = 0; s0 < kw_splits; s0 += kB) {
                float4 a[kB], c[kB];
                float2 u2[kB];
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    if (s0 + u < kw_splits) {
                        const float* p = kw_partial + ((int64_t)(s0 + u) * T + t) * kN;
                        a[u] = __ldg(reinterpret_cast<const float4*>(p + 8 * hl));
                        c[u] = __ldg(reinterpret_cast<const float4*>(p + 8 * hl + 4));
                        u2[u] = __ldg(reinterpret_cast<const float2*>(p + IDX_DIM + 2 * hl));
                    }
                }
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    if (s0 + u >= kw_splits) break;
                    ka.x += a[u].x; ka.y += a[u].y; ka.z += a[u].z; ka.w += a[u].w;
                    kb.x += c[u].x; kb.y += c[u].y; kb.z += c[u].z; kb.w += c[u].w;
                    wv.x += u2[u].x; wv.y += u2[u].y;
                }
            }
        }
        const uint4 kpre = make_uint4(f32x2_to_bf16x2_rn(ka.x, ka.y), f32x2_to_bf16x2_rn(ka.z, ka.w),
                                      f32x2_to_bf16x2_rn(kb.x, kb.y), f32x2_to_bf16x2_rn(kb.z, kb.w));
        float2 g[4], b[4];   // (loaded here: not live across the split loads)
        ln_params_half_warp(ln_w, ln_b, kF32Params, hl, g, b);
        uint32_t o16[4];
        ln_row_half_warp(kpre, g, b, eps, o16);   // both half warps take part
        if (ok) {
            *reinterpret_cast<float2*>(w_out + t * IDX_HEADS + 2 * hl) = wv;
            if (sr >= 0 && sr < cache_rows) k_cache[sr * 16 + hl] = make_uint4(o16[0], o16[1], o16[2], o16[3]);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 matrix [rows, K] (row stride K elements), loaded as {64, box_rows}
// boxes with the 128-byte swizzle; elements outside the matrix read as zero.
bool make_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGemmBK, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    const DeviceInfo& d = device_info();
    return d.sm_count > 0 ? d.sm_count : 1;
}

int64_t cluster_count() { return sm_count() / 2 > 0 ? sm_count() / 2 : 1; }

// The most K splits of `pairs` items: two waves of items over the clusters.
int max_splits(int64_t pairs) {
    const int64_t c = cluster_count(), p = pairs > 0 ? pairs : 1;
    const int64_t s = (2 * c + p - 1) / p;
    return (int)(s < 1 ? 1 : s);
}

// K splits for `pairs` row-tile pairs x column tiles of a product with KB K
// blocks: the smallest split with the least estimated time, counting waves of
// items over the clusters (K blocks per item), the partial sums' extra
// traffic (rows x cols x 8 bytes per split, at about 4 K blocks' worth per
// 512 KB per cluster) and the finishing kernel's dependent rounds of loads
// (about 3 K blocks' worth each; measured: 56 splits of a few tokens took
// 19.5 us to sum in rounds of 4, against 17.9 us for the whole GEMM). Each
// split keeps at least 2 K blocks when K allows, and there are at most
// max_splits(pairs) (the workspace holds that many).
int choose_splits(int64_t pairs, int KB, int64_t rows, int cols) {
    const int64_t clusters = cluster_count();
    int cap = KB >= 4 ? KB / 2 : (KB > 0 ? KB : 1);
    if (cap > max_splits(pairs)) cap = max_splits(pairs);
    int best = 1;
    double best_cost = 1e300;
    for (int s = 1; s <= cap; ++s) {
        const int64_t items = pairs * s;
        const double waves = (double)((items + clusters - 1) / clusters);
        const double kb = (double)((KB + s - 1) / s);
        const double extra = s > 1 ? (double)s * rows * cols * 8.0 / (512.0 * 1024.0) * 4.0 / clusters +
                                         3.0 * ((s + kFinishRound - 1) / kFinishRound)
                                   : 0.0;
        const double cost = waves * kb + extra;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

constexpr int kNq = IDX_HEADS * IDX_DIM;   // 4096 query features
constexpr int kNkw = IDX_DIM + IDX_HEADS;  // 160: key features, then head weights

int64_t pairs_of(int32_t T, int N, int BN) {
    const int64_t m_tiles = (T + kGemmBM - 1) / kGemmBM;
    return (m_tiles + 1) / 2 * ((N + BN - 1) / BN);
}

constexpr int kBNq = 256;    // W_q rows per item (two 128-row halves)
constexpr int kBNkw = 160;   // W_k (128) and W_w (32) rows per item

// Bytes of fp32 partials for T tokens (for the most splits any K can take):
// the key/weight product's, then the q product's when it can be split.
size_t kw_partial_bytes(int32_t T) {
    const int64_t t = T > 0 ? T : 0;
    return align_up((size_t)max_splits(pairs_of(T, kNkw, kBNkw)) * t * kNkw * 4, 256);
}
size_t q_partial_bytes(int32_t T) {
    const int64_t t = T > 0 ? T : 0;
    const int sq = max_splits(pairs_of(T, kNq, kBNq));
    return sq > 1 ? align_up((size_t)sq * t * kNq * 4, 256) : 0;
}

// Output maps of the epilogue's TMA stores: 32 x 32 boxes, no swizzle.
// bf16 [M, N] (row stride N), or fp32 partials [splits, M, N].
bool make_out_map_bf16(CUtensorMap* map, void* base, int64_t M, int64_t N) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_out_map_f32(CUtensorMap* map, void* base, int64_t splits, int64_t M, int64_t N) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)splits};
    const cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)(M * N * 4)};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

idx_status proj_fail(idx_status code, const char* msg) {
    set_last_error_text(msg);
    return code;
}

bool is_aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace
}  // namespace lidx

using namespace lidx;

extern "C" {

size_t idx_indexer_project_workspace_size(int32_t T) {
    return kWsHeader + kw_partial_bytes(T) + q_partial_bytes(T);
}

idx_status idx_indexer_project(const uint16_t* x, const uint16_t* q_lora, const uint16_t* w_q,
                               const uint16_t* w_k, const uint16_t* w_w, const void* ln_w,
                               const void* ln_b, int ln_dtype, float eps, int32_t T, int32_t hidden,
                               int32_t q_rank, uint16_t* q, uint16_t* k_cache, int64_t cache_rows,
                               const int64_t* slot, float* w, void* ws, size_t ws_bytes,
                               void* stream) {
    set_last_error_text("");
    TraceRange trace("idx_indexer_project");
    if (T < 0 || hidden < 8 || q_rank < 8 || hidden % 8 != 0 || q_rank % 8 != 0 || cache_rows < 0)
        return proj_fail(IDX_ERR_INVALID_ARG,
                         "T >= 0, hidden and q_rank positive multiples of 8, cache_rows >= 0");
    if (ln_dtype != IDX_PARAM_BF16 && ln_dtype != IDX_PARAM_F32)
        return proj_fail(IDX_ERR_INVALID_ARG, "ln_dtype must be IDX_PARAM_BF16 or IDX_PARAM_F32");
    if (!(eps >= 0.f) || eps > 1e30f) return proj_fail(IDX_ERR_INVALID_ARG, "eps must be finite, >= 0");
    if (T == 0) return IDX_OK;
    if (!x || !q_lora || !w_q || !w_k || !w_w || !ln_w || !ln_b || !q || !k_cache || !slot || !w)
        return proj_fail(IDX_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!is_aligned(x, 16) || !is_aligned(q_lora, 16) || !is_aligned(w_q, 16) ||
        !is_aligned(w_k, 16) || !is_aligned(w_w, 16) || !is_aligned(q, 16) ||
        !is_aligned(k_cache, 16) || !is_aligned(w, 16) || !is_aligned(slot, 8) ||
        !is_aligned(ln_w, 4) || !is_aligned(ln_b, 4))
        return proj_fail(IDX_ERR_INVALID_ARG, "matrices 16-byte aligned, slot 8-byte, LN params 4-byte");
    if (!ws || !is_aligned(ws, 256))
        return proj_fail(IDX_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
    if (ws_bytes < idx_indexer_project_workspace_size(T))
        return proj_fail(IDX_ERR_WORKSPACE, "workspace smaller than idx_indexer_project_workspace_size(T)");
    const DeviceInfo& dev = device_info();
    if (dev.device < 0) return proj_fail(IDX_ERR_CUDA, "no current CUDA device");
    if (!(dev.cc_major == 10 && dev.cc_minor == 3))
        return proj_fail(IDX_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    cudaStream_t s = (cudaStream_t)stream;
    DeviceStatus* status = static_cast<DeviceStatus*>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s);
    if (e != cudaSuccess) return proj_fail(IDX_ERR_CUDA, cudaGetErrorString(e));

    float* kw_partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
    float* q_partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader + kw_partial_bytes(T));

    // Problem 0: [k_pre | w] = x . [W_k ; W_w]^T, always as fp32 partials (the
    // finishing kernel writes k_pre's LayerNorm and w). Problem 1: q = q_lora .
    // W_q^T, bf16 straight from the accumulators, or split K. B tiles are
    // loaded in halves, one per CTA of a pair: [W_k ; W_w] as rows 0..79 of
    // W_k (rank 0), then rows 80..127 of W_k and the 32 rows of W_w (rank 1);
    // W_q as two 128-row boxes.
    GemmGroup G{};
    G.n_problems = 2;
    GemmProblem& kw = G.p[0];
    kw.M = T;
    kw.N = kNkw;
    kw.KB = (hidden + kGemmBK - 1) / kGemmBK;
    kw.m_pairs = ((T + kGemmBM - 1) / kGemmBM + 1) / 2;
    kw.n_tiles = 1;
    kw.BN = kBNkw;
    kw.splits = choose_splits(kw.m_pairs, kw.KB, T, kNkw);
    kw.out_bf16 = 0;
    kw.nseg[0] = 1;
    kw.seg[0][0] = BSeg{0, 0, 0, 80};
    kw.nseg[1] = 2;
    kw.seg[1][0] = BSeg{1, 80, 80, IDX_DIM - 80};
    kw.seg[1][1] = BSeg{2, 0, IDX_DIM, IDX_HEADS};
    GemmProblem& pq = G.p[1];
    pq.M = T;
    pq.N = kNq;
    pq.KB = (q_rank + kGemmBK - 1) / kGemmBK;
    pq.m_pairs = ((T + kGemmBM - 1) / kGemmBM + 1) / 2;
    pq.n_tiles = kNq / kBNq;
    pq.BN = kBNq;
    pq.splits = choose_splits((int64_t)pq.m_pairs * pq.n_tiles, pq.KB, T, kNq);
    pq.items = pq.m_pairs * pq.n_tiles * pq.splits;
    if (pq.items >= cluster_count()) {
        // q alone fills the clusters: cut the key/weight product (bound by
        // reading x) into at most 4 items per row-tile pair, of at least 16 K
        // blocks, interleaved with the q items, so that every cluster gets a
        // similar share of both
        const int fine = (kw.KB + 15) / 16;
        const int cap = max_splits(kw.m_pairs) < 4 ? max_splits(kw.m_pairs) : 4;
        kw.splits = fine < 1 ? 1 : (fine > cap ? cap : fine);
    }
    kw.items = kw.m_pairs * kw.n_tiles * kw.splits;
    pq.out_bf16 = pq.splits == 1;
    pq.nseg[0] = pq.nseg[1] = 1;
    pq.seg[0][0] = BSeg{0, 0, 0, kBNq / 2};
    pq.seg[1][0] = BSeg{0, kBNq / 2, kBNq / 2, kBNq / 2};
    G.items = kw.items + pq.items;

    GemmMaps maps;
    memset(&maps, 0, sizeof maps);
    if (!make_kmajor_map(&maps.a[0], x, T, hidden, kGemmBM) ||
        !make_kmajor_map(&maps.b[0][0], w_k, IDX_DIM, hidden, 80) ||
        !make_kmajor_map(&maps.b[0][1], w_k, IDX_DIM, hidden, IDX_DIM - 80) ||
        !make_kmajor_map(&maps.b[0][2], w_w, IDX_HEADS, hidden, IDX_HEADS) ||
        !make_out_map_f32(&maps.out[0], kw_partial, kw.splits, T, kNkw) ||
        !make_kmajor_map(&maps.a[1], q_lora, T, q_rank, kGemmBM) ||
        !make_kmajor_map(&maps.b[1][0], w_q, kNq, q_rank, kBNq / 2) ||
        !(pq.out_bf16 ? make_out_map_bf16(&maps.out[1], q, T, kNq)
                      : make_out_map_f32(&maps.out[1], q_partial, pq.splits, T, kNq)))
        return proj_fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    maps.b[1][1] = maps.b[1][0];   // (unused map slots repeat a valid map)
    maps.b[1][2] = maps.b[1][0];

    e = ensure_smem_optin((const void*)gemm_tc_kernel, kGemmSmem);
    if (e != cudaSuccess) return proj_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    const int64_t clusters = cluster_count();
    const int grid = 2 * (int)(G.items < clusters ? G.items : clusters);
    e = launch_kernel(gemm_tc_kernel, dim3(grid), dim3(kGemmThreads), (size_t)kGemmSmem, s, 2, maps, G,
                      status, wait_limit_ns());
    if (e != cudaSuccess) return proj_fail(IDX_ERR_CUDA, cudaGetErrorString(e));

    // the finishing kernel: q's split sum (if any) and the key/weight end
    const int sms = sm_count();
    const int64_t q_vecs = (int64_t)T * kNq / 4;
    const int q_blocks = pq.out_bf16 ? 0 : (int)((q_vecs + 255) / 256 < 2 * sms ? (q_vecs + 255) / 256 : 2 * sms);
    const int64_t kw_blocks_need = (((int64_t)T + 1) / 2 + 7) / 8;   // a half warp per token
    const int kw_blocks = (int)(kw_blocks_need < 4 * sms ? kw_blocks_need : 4 * sms);
    const bool round4 = kw.splits <= 4 && (pq.out_bf16 || pq.splits <= 4);
    auto fin = ln_dtype == IDX_PARAM_F32 ? (round4 ? project_finish_kernel<true, 4> : project_finish_kernel<true, kFinishRound>)
                                         : (round4 ? project_finish_kernel<false, 4> : project_finish_kernel<false, kFinishRound>);
    e = launch_kernel(fin, dim3(q_blocks + kw_blocks), dim3(256), 0, s, 1, (const float*)q_partial,
                      pq.splits, q, q_blocks, (const float*)kw_partial, kw.splits, T, ln_w, ln_b, eps,
                      reinterpret_cast<uint4*>(k_cache), cache_rows, slot, w);
    if (e != cudaSuccess) return proj_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    return IDX_OK;
}

}  // extern "C"

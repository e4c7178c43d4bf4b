// Sparse NoPE MLA attention over the indexer's selected positions (decode).
//
// Port notes ("Notes from an NVFP4 port of Kimi K3.1 Pro", opening paragraph
// and item (5)): the indexer keeps the best 2048 keys per query for every
// full-attention layer, and those layers are NoPE multi-head latent attention
// (the 64 "rope" dims are ordinary key dims). TokenSpeed's Kimi K3 post
// (section 2, MLA): each cached token holds a shared 512-wide latent and a
// 64-wide key part, there are 96 heads, and decode works with the query moved
// into that compressed space. Per query row t and head h:
//     l_s = scale * (q_h . c_s) over the selected rows c_s (576 wide),
//     out_h = sum_s softmax(l)_s c_s[0..512),  lse_h = log sum_s exp(l_s).
//
// One CTA per (query row, range of 32-row tiles of its selection), on the
// 5th-generation tensor cores:
//   warp 0     TMEM allocation; one lane issues MMA1:
//                S[128 heads (rows >= H unused), 32 rows] = Q . C^T, K = 576
//                (Q resident in shared memory, 128-byte swizzle, K-major)
//   warp 9     one lane issues MMA2:
//                O^T[512 dims, H] += C^T . P^T, K = 32 rows: the gathered tile
//                read a second time as an MN-major operand, P (bf16, 64-byte
//                swizzle) from shared memory; O^T stays in TMEM (4 x H columns)
//   warps 1-4  gather the selected rows with 16-byte cp.async into the swizzled
//              tile layout (three stages; 8 threads per row, so a warp copies
//              4 rows x 128 contiguous bytes per instruction); each tile's
//              barrier tracks the copies' landing (cp.async.mbarrier.arrive
//              .noinc); one lane loads Q by TMA
//   warps 5-8  softmax: a TMEM lane is a head, so each thread owns one row of S:
//              running maximum in the log2 domain, P = 2^(S - m), sum l.
//              O is rescaled (in TMEM) only when a head's maximum grows by more
//              than 2^kRescaleLog2 (2^20), so the scale of O and l may lag the
//              true maximum; both carry the same factor, and the result is
//              unchanged. Weights stay below 2^20, so O stays finite for cache
//              values below about 1e29 (fp32 sums of 2048 weighted rows).
// With one CTA per query row the kernel writes out/lse; with several it writes
// (O, m, l) partials that sparse_mla_merge_kernel combines.
// Every wait is bounded; a timeout or an out-of-range position is recorded in
// the status word.
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "tc_primitives.cuh"

namespace lidx {

namespace {

constexpr int kMlaDim = 576;                    // cache row: 512 latent + 64 key dims
constexpr int kMlaV = 512;                      // latent (value) dims
constexpr int kChunks = kMlaDim / 64;           // 64-dim (128-byte) chunks of a row
constexpr int kTileRows = 32;                   // selected rows per tile
constexpr int kChunkBytes = kTileRows * 128;    // one chunk of a tile
constexpr int kStageBytes = kChunks * kChunkBytes;
constexpr int kStages = 3;
constexpr int kThreads = 320;                   // warp 0 MMA1, 1-4 gather, 5-8 softmax, 9 MMA2
constexpr int kGather = 128;                    // warps 1-4
constexpr int kSoft = 128;                      // warps 5-8
constexpr uint32_t kTmemCols = 512;
constexpr int kSoftBar = 1;                     // named barrier of the softmax warps
constexpr uint64_t kMlaDrainNs = 100000000ull;  // 100 ms to drain after an abort
// A head's reference maximum (log2 domain) moves, and O and l are rescaled,
// only when the tile maximum exceeds it by more than this. Measured: a
// threshold of 8 rescaled on most tiles of rows whose logits spread widely,
// at up to a few microseconds per rescale.
constexpr float kRescaleLog2 = 20.f;

constexpr int kRow8 = kMlaDim;                  // an FP8 cache row: 576 bytes

template <int H, bool kFp8 = false>
struct MlaLayout {
    // swizzled bf16 tile stages (the FP8 path converts into the same stages)
    static constexpr int kNStages = kStages;
    static constexpr int kQChunk = H * 128;     // a 64-dim chunk of Q (H rows)
    static constexpr int kQBytes = kChunks * kQChunk;
    static constexpr int kC = kQBytes;          // 1024-byte aligned since H % 8 == 0
    static constexpr int kP = kC + kNStages * kStageBytes;   // 1024-byte aligned
    static constexpr int kPBytes = H * 64;      // P: a 64-byte row (32 bf16) per head, 64-byte swizzle
    static constexpr int kF = kP + kPBytes;     // per-head rescale factors [2][128]
    static constexpr int kM = kF + 1024;        // per-head m [128]
    static constexpr int kL = kM + 512;         // per-head l [128]
    static constexpr int kSc = kL + 512;        // FP8: row scales of each stage's tile [kNStages][32]
    static constexpr int kBar = kSc + kNStages * kTileRows * 4;
    static constexpr int kBytes = kBar + 24 * 8 + 16;   // barriers, TMEM slot, flags, masks
    static constexpr uint32_t kOCols = 4 * H;   // O^T: 4 tiles of 128 dims, H columns each
    static constexpr uint32_t kSCol = kOCols;   // S: two buffers of 32 columns
    static_assert(H % 32 == 0 && H >= 32 && H <= 96, "heads: 32, 64 or 96");
    static_assert(kOCols + 2 * kTileRows <= kTmemCols, "TMEM columns");
    static_assert(kBytes <= 227 * 1024, "shared memory");
    static_assert(kP % 1024 == 0, "alignment");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// 16 bytes of zeros (a source size of 0 reads nothing from global memory).
__device__ __forceinline__ void cp_async16_zero(uint32_t dst, const void* any_global) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(dst), "l"(any_global) : "memory");
}
// Arrive on `bar` once every cp.async this thread has issued so far has landed
// (the arrival is counted against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Make this thread's shared-memory writes (st.shared, cp.async) visible to the
// async proxy that tcgen05.mma reads operands through.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 bytes from global memory, read-only, not kept in L1 (rows are read once).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two E4M3 codes (low byte first) -> two bf16 values (low half first), exactly:
// every E4M3 value is an fp16 and a bf16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_codes));
    const float lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    const float hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
    return f32x2_to_bf16x2_rn(lo, hi);
}

// 2^x by the hardware approximation (ex2.approx: relative error near 2^-22,
// well inside the bf16 rounding the weights get next; 2^-inf = +0).
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Barrier `id` over `threads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(int id, int threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// each 128-byte row holds 64 consecutive M (or N) elements of one K index,
// rows of consecutive K are 128 B apart inside 1024-byte atoms; `lbo` is the
// distance between atoms along M/N (the next 64 elements), `sbo` between atoms
// along K (the next 8 K indices).
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Shared-memory descriptor of a K-major operand with the 64-byte swizzle: rows
// of 64 B (32 bf16), 8-row groups 512 B apart; the 16-byte pieces of row r sit
// at piece ^ ((r >> 1) & 3).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                      // leading byte offset (unused here), 16 B
    d |= (uint64_t)(512 >> 4) << 32;             // stride byte offset: 512 B per 8 rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;                      // layout: 64-byte swizzle
    return d;
}

// Store 32 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// kFp8: the cache rows are 576 E4M3 codes (cache8) with one fp32 scale each
// (row_scale); the row is c = row_scale x e4m3(code). The gather warps load
// the selected rows' codes into registers and convert them to bf16 (exact)
// into the swizzled tile the MMAs read, and the softmax applies the row scale in fp32: to the
// logits (scale x row_scale x q.e) and to P before its bf16 rounding
// (O accumulates p x row_scale x e; l sums p).
template <int H, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_q, const uint16_t* __restrict__ cache,
                  const uint8_t* __restrict__ cache8, const float* __restrict__ row_scale,
                  int64_t cache_rows, const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt,
                  const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B, int topk,
                  float scale_log2, int tiles_per_split, int n_split, float* __restrict__ out,
                  float* __restrict__ lse, float* __restrict__ part_o, float* __restrict__ part_ml,
                  DeviceStatus* status, uint64_t wait_ns) {
    using namespace ptx;
    using Lay = MlaLayout<H, kFp8>;
    constexpr int NST = Lay::kNStages;
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_addr(smem) & 1023u) != 0) {   // the swizzled tiles need 1024-byte alignment
        pdl_wait();
        if (threadIdx.x == 0) report_error(status, IDX_ERR_UNSUPPORTED, 1024);
        return;
    }
    uint8_t* q_s = smem;
    uint8_t* c_s = smem + Lay::kC;
    uint8_t* p_s = smem + Lay::kP;
    float* fac = reinterpret_cast<float*>(smem + Lay::kF);
    float* m_s = reinterpret_cast<float*>(smem + Lay::kM);
    float* l_s = reinterpret_cast<float*>(smem + Lay::kL);
    float* sc_s = reinterpret_cast<float*>(smem + Lay::kSc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
    uint64_t* q_full = bars;
    uint64_t* c_full = bars + 1;    // [kStages]: a tile gathered (kGather arrivals)
    uint64_t* c_empty = bars + 4;   // [kStages]: MMA2 done with the tile
    uint64_t* s_full = bars + 7;    // [2]: MMA1 wrote S
    uint64_t* p_full = bars + 9;    // P written (kSoft arrivals)
    uint64_t* o_done = bars + 10;   // MMA2 of a tile complete
    uint64_t* end_bar = bars + 11;  // every MMA1 issued has completed
    uint64_t* s_free = bars + 12;   // [2]: the softmax has read S (kSoft arrivals)
    uint64_t* end_bar2 = bars + 14; // every MMA2 issued has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* seq_of_row = reinterpret_cast<int*>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(c_full + s, kGather);
            mbar_init(c_empty + s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_full + 1, 1);
        mbar_init(p_full, kSoft);
        mbar_init(o_done, 1);
        mbar_init(end_bar, 1);
        mbar_init(s_free, kSoft);
        mbar_init(s_free + 1, kSoft);
        mbar_init(end_bar2, 1);
        *abort_flag = 0;
        *seq_of_row = 0;
        fence_mbar_init();
    }
    if (warp == 1 && lane == 0) prefetch_tmap(&tmap_q);
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    // ---- this CTA's query row, its sequence, and its tiles
    const int t = blockIdx.x / n_split, sp = blockIdx.x % n_split;
    // the sequence holding row t, found by all threads in one round of loads
    // (no dependent chain as in a binary search)
    for (int j = threadIdx.x; j < B; j += kThreads)
        if (__ldg(cu_q + j) <= t && t < __ldg(cu_q + j + 1)) *seq_of_row = j;
    __syncthreads();
    const int b = *seq_of_row;
    const int64_t k0 = __ldg(cu_k + b);
    const int64_t len_k = (int64_t)__ldg(cu_k + b + 1) - k0;
    int32_t n_sel = __ldg(cnt + t);
    bool bad = n_sel < 0 || n_sel > topk || k0 < 0 || len_k < 0 || k0 + len_k > cache_rows ||
               __ldg(cu_q + b) > t || __ldg(cu_q + b + 1) <= t;
    if (bad) {
        if (threadIdx.x == 0 && sp == 0) report_error(status, IDX_ERR_DEVICE_ARG, t);
        n_sel = 0;
    }
    const int tiles = (n_sel + kTileRows - 1) / kTileRows;
    const int tile0 = sp * tiles_per_split;
    const int nt = tiles - tile0 < tiles_per_split ? (tiles - tile0 > 0 ? tiles - tile0 : 0) : tiles_per_split;

    bool aborted = false;
    auto give_up = [&](int site) {
        if (!*abort_flag) report_error(status, IDX_ERR_TIMEOUT, site);
        *abort_flag = 1;
        aborted = true;
    };
    // position of selected entry j of this row (sequence-local), or -1
    auto position = [&](int32_t j) -> int32_t {
        if (j >= n_sel) return -1;
        const int32_t p = __ldg(idx + (int64_t)t * topk + j);
        return p >= 0 && p < len_k ? p : -1;
    };

    constexpr uint32_t kI1 = idesc_bf16_f32(128, kTileRows);
    constexpr uint32_t kI2 = idesc_bf16_f32(128, H) | (1u << 15);   // A is MN-major
    if (warp == 0) {
        // ---------------------------------------------------- MMA1 issuer: S = Q . C^T
        if (lane == 0 && nt > 0) {
            const uint32_t qa = smem_addr(q_s), ca = smem_addr(c_s);
            bool ok = mbar_wait(q_full, 0, abort_flag, wait_ns);
            if (!ok) give_up(20);
            for (int i = 0; i < nt && ok; ++i) {
                const int st = i % NST, s = i & 1;
                // tile i landed, and S buffer s read by the softmax of tile i-2
                if (!mbar_wait(c_full + st, (i / NST) & 1, abort_flag, wait_ns) ||
                    (i >= 2 && !mbar_wait(s_free + s, ((i >> 1) - 1) & 1, abort_flag, wait_ns))) {
                    give_up(21);
                    break;
                }
                // the tile was written through cp.async (generic proxy); the MMA
                // reads it through the async proxy
                fence_proxy_async_smem();
                tc_fence_after_sync();
                const uint32_t d = tmem_base + Lay::kSCol + kTileRows * s;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t a = smem_desc_sw128(qa + c * Lay::kQChunk + k * 32);
                        const uint64_t bd = smem_desc_sw128(ca + st * kStageBytes + c * kChunkBytes + k * 32);
                        tc_mma_bf16(d, a, bd, kI1, (c | k) != 0 ? 1u : 0u);
                    }
                tc_commit(s_full + s);
            }
            tc_commit(end_bar);   // every MMA1 issued has completed before teardown
            mbar_wait(end_bar, 0, nullptr, kMlaDrainNs);
        }
    } else if (warp == 9) {
        // --------------------------------------------------- MMA2 issuer: O^T += C^T . P^T
        if (lane == 0 && nt > 0) {
            const uint32_t ca = smem_addr(c_s), pa = smem_addr(p_s);
            for (int i = 0; i < nt; ++i) {
                // P(i) written (the softmax of tile i saw S(i): MMA1(i) is complete)
                if (!mbar_wait(p_full, i & 1, abort_flag, wait_ns)) {
                    give_up(22);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t cbase = ca + (i % NST) * kStageBytes;
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        // dims 128m .. 128m+127 = chunks 2m, 2m+1; rows 16k .. 16k+15
                        const uint64_t a = smem_desc_sw128_mn(cbase + 2 * m * kChunkBytes + k * 2048,
                                                              kChunkBytes, 1024);
                        const uint64_t bd = smem_desc_sw64(pa + k * 32);
                        tc_mma_bf16(tmem_base + m * H, a, bd, kI2, (i > 0 || k > 0) ? 1u : 0u);
                    }
                tc_commit(c_empty + (i % NST));
                tc_commit(o_done);
            }
            tc_commit(end_bar2);
            mbar_wait(end_bar2, 0, nullptr, kMlaDrainNs);
        }
    } else if (warp <= 4 && kFp8) {
        // ------------------------------------------------- gather (FP8 rows)
        // Each thread owns 9 of a tile's 32 x 36 16-byte pieces of codes. It
        // loads them into registers two tiles ahead (tile i+1 in flight while
        // tile i is converted), converts 16 codes into two 16-byte bf16 pieces
        // (exact) and stores them at their swizzled places in stage i % NST;
        // rows left out load nothing and convert to zeros. No shared-memory
        // staging: the three bf16 stages of the bf16 path fit beside Q.
        const int g = threadIdx.x - 32;   // 0 .. 127
        if (g == 0 && nt > 0) {
            mbar_arrive_expect_tx(q_full, Lay::kQBytes);
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c)
                tma_load_2d(smem_addr(q_s + c * Lay::kQChunk), &tmap_q, q_full, c * 64, t * H);
        }
        constexpr int kPcs = kRow8 / 16;                        // 36 pieces per row
        constexpr int kPer = kTileRows * kPcs / kGather;        // 9 pieces per thread
        static_assert(kTileRows * kPcs % kGather == 0, "pieces per thread");
        // positions of this thread's rows, fetched two tiles ahead: pe for the
        // even tiles, po for the odd ones
        int32_t pe[kPer], po[kPer];
        auto fetch_positions = [&](int i, int32_t (&P)[kPer]) {
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                P[j] = i < nt ? position((tile0 + i) * kTileRows + (g + kGather * j) / kPcs) : -1;
        };
        // issue the loads of tile i (positions in P; the thread holding a row's
        // first piece also loads that row's scale), then fetch the positions
        // of tile i+2 into P
        auto load_tile = [&](int i, int32_t (&P)[kPer], uint4 (&R)[kPer], float (&S)[kPer]) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int pc = g + kGather * j, r = pc / kPcs, w = pc - r * kPcs;
                if (w == 0 && i < nt && (tile0 + i) * kTileRows + r < n_sel && P[j] < 0)
                    report_error(status, IDX_ERR_DEVICE_ARG, t);
                R[j] = P[j] >= 0 ? ld_nc_v4(cache8 + (k0 + P[j]) * kRow8 + w * 16) : make_uint4(0u, 0u, 0u, 0u);
                S[j] = w == 0 && P[j] >= 0 ? __ldg(row_scale + k0 + P[j]) : 0.f;
            }
            fetch_positions(i + 2, P);
        };
        // tile i from R into stage i % NST (false: a wait gave up)
        auto store_tile = [&](int i, const uint4 (&R)[kPer], const float (&S)[kPer]) -> bool {
            const int st = i % NST;
            if (i >= NST && !mbar_wait(c_empty + st, (i / NST - 1) & 1, abort_flag, wait_ns)) return false;
            uint8_t* dst = c_s + st * kStageBytes;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int pc = g + kGather * j, r = pc / kPcs, w = pc - r * kPcs;
                if (w == 0) sc_s[st * kTileRows + r] = S[j];
                const int c = w >> 2, q0 = (w & 3) * 2;   // chunk; first 16-byte piece in its 128-byte row
                const uint4 lo = make_uint4(e4m3x2_to_bf16x2(R[j].x & 0xFFFFu), e4m3x2_to_bf16x2(R[j].x >> 16),
                                            e4m3x2_to_bf16x2(R[j].y & 0xFFFFu), e4m3x2_to_bf16x2(R[j].y >> 16));
                const uint4 hi = make_uint4(e4m3x2_to_bf16x2(R[j].z & 0xFFFFu), e4m3x2_to_bf16x2(R[j].z >> 16),
                                            e4m3x2_to_bf16x2(R[j].w & 0xFFFFu), e4m3x2_to_bf16x2(R[j].w >> 16));
                uint8_t* row = dst + c * kChunkBytes + r * 128;
                *reinterpret_cast<uint4*>(row + ((q0 ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4*>(row + (((q0 + 1) ^ (r & 7)) << 4)) = hi;
            }
            fence_proxy_async_smem();   // the MMAs read the tile through the async proxy
            mbar_arrive(c_full + st);
            return true;
        };
        uint4 ra[kPer], rb[kPer];
        float sa[kPer], sb[kPer];
        fetch_positions(0, pe);
        fetch_positions(1, po);
        if (nt > 0) load_tile(0, pe, ra, sa);
        for (int i = 0; i < nt; i += 2) {
            if (i + 1 < nt) load_tile(i + 1, po, rb, sb);
            if (!store_tile(i, ra, sa)) {
                give_up(27);
                break;
            }
            if (i + 1 >= nt) break;
            if (i + 2 < nt) load_tile(i + 2, pe, ra, sa);
            if (!store_tile(i + 1, rb, sb)) {
                give_up(27);
                break;
            }
        }
        if (g == 0 && nt > 0) mbar_wait(q_full, 0, nullptr, kMlaDrainNs);   // Q landed before exit
    } else if (warp <= 4) {
        // ------------------------------------------------------------ gather
        const int g = threadIdx.x - 32;   // 0 .. 127
        if (g == 0 && nt > 0) {
            mbar_arrive_expect_tx(q_full, Lay::kQBytes);
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c)
                tma_load_2d(smem_addr(q_s + c * Lay::kQChunk), &tmap_q, q_full, c * 64, t * H);
        }
        // Every write of a tile (rows, and zeros for rows left out) is a cp.async
        // whose landing the tile's barrier tracks (arrive.noinc): the producer
        // never waits for its own copies, only for a free stage. (Bulk L2
        // prefetches of the rows of later tiles were measured slower: they
        // compete with the gathers.)
        // 8 threads per row: a warp copies 4 rows x 128 contiguous bytes per instruction
        const int r8 = g >> 3, q8 = g & 7;   // rows r8 and r8 + 16
        int32_t pn0 = nt > 0 ? position(tile0 * kTileRows + r8) : -1;
        int32_t pn1 = nt > 0 ? position(tile0 * kTileRows + r8 + 16) : -1;
        for (int i = 0; i < nt; ++i) {
            const int s = i % NST;
            const int32_t p0 = pn0, p1 = pn1;
            pn0 = i + 1 < nt ? position((tile0 + i + 1) * kTileRows + r8) : -1;
            pn1 = i + 1 < nt ? position((tile0 + i + 1) * kTileRows + r8 + 16) : -1;
            if (i >= NST && !mbar_wait(c_empty + s, (i / NST - 1) & 1, abort_flag, wait_ns)) {
                give_up(23);
                break;
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int rr = r8 + 16 * h2;
                const int32_t pos = h2 == 0 ? p0 : p1;
                const int32_t j = (tile0 + i) * kTileRows + rr;
                if (j < n_sel && pos < 0 && q8 == 0) report_error(status, IDX_ERR_DEVICE_ARG, t);
                const uint8_t* src =
                    pos >= 0 ? reinterpret_cast<const uint8_t*>(cache + (k0 + pos) * kMlaDim) : nullptr;
                uint8_t* row_dst = c_s + s * kStageBytes + rr * 128;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const uint32_t dst = smem_addr(row_dst + c * kChunkBytes + ((q8 ^ (rr & 7)) << 4));
                    if (src) cp_async16(dst, src + c * 128 + q8 * 16);
                    else cp_async16_zero(dst, cache);
                }
            }
            cp_async_arrive_noinc(c_full + s);
        }
        cp_async_wait_all();   // nothing of this thread in flight when the CTA ends
        if (g == 0 && nt > 0) mbar_wait(q_full, 0, nullptr, kMlaDrainNs);   // Q landed before exit
    } else if (warp <= 8) {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;   // head = TMEM lane of S
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        int done = 0;
        for (int i = 0; i < nt; ++i) {
            const int s = i & 1;
            const bool vc = position((tile0 + i) * kTileRows + lane) >= 0;
            const uint32_t vmask = __ballot_sync(0xffffffffu, vc);
            // every wait's outcome is agreed by the whole group (bar.red.or),
            // so the group's barriers always see all of its threads. FP8: the
            // tile's barrier (complete before its S) also orders the gather
            // threads' row scales before the reads below.
            const bool s_ok = mbar_wait(s_full + s, (i >> 1) & 1, abort_flag, wait_ns) &&
                              (!kFp8 || mbar_wait(c_full + i % NST, (i / NST) & 1, abort_flag, wait_ns));
            if (bar_red_or(kSoftBar, kSoft, !s_ok)) {
                give_up(24);
                break;
            }
            tc_fence_after_sync();
            uint32_t v[32];
            tmem_ld_x32(lane_base + Lay::kSCol + kTileRows * s, v);
            tmem_ld_wait(v);
            tc_fence_before_sync();
            mbar_arrive(s_free + s);   // MMA1 of tile i+2 may overwrite this buffer
            // logits in the log2 domain (FP8: times the row's scale)
            const float sc_cur = kFp8 ? sc_s[(i % NST) * kTileRows + lane] : 1.f;
            float sc[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                sc[c] = kFp8 ? __shfl_sync(0xffffffffu, sc_cur, c) : 1.f;
                v[c] = __float_as_uint(__uint_as_float(v[c]) * scale_log2 * sc[c]);
            }
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if ((vmask >> c) & 1u) tmax = fmaxf(tmax, __uint_as_float(v[c]));
            // new reference maximum: the first finite one, or one that grew past 2^kRescaleLog2
            bool need = false;
            float f = 1.f;
            if (tmax > -INFINITY && (m_used == -INFINITY || tmax > m_used + kRescaleLog2)) {
                f = m_used == -INFINITY ? 0.f : exp2f(m_used - tmax);
                need = i > 0;   // before the first MMA2, O holds nothing to rescale
                m_used = tmax;
                l *= f;
            }
            float p[32];
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                p[c] = ((vmask >> c) & 1u) && m_used > -INFINITY
                           ? ex2_fast(__uint_as_float(v[c]) - m_used)
                           : 0.f;
                psum += p[c];
                if (kFp8) p[c] *= sc[c];   // O gathers p x row scale x code; l sums p
            }
            l += psum;
            // factors of tile i in buffer i & 1: the barrier of tile i+1 lies
            // between this tile's reads and the next writes of the same buffer
            float* fac_i = fac + 128 * (i & 1);
            if (h < H) fac_i[h] = f;
            const bool any = bar_red_or(kSoftBar, kSoft, need && h < H);
            if (i > 0) {   // MMA2 of the previous tile is done: O is quiet and P is free
                const bool o_ok = mbar_wait(o_done, (i - 1) & 1, abort_flag, wait_ns);
                if (bar_red_or(kSoftBar, kSoft, !o_ok)) {
                    give_up(25);
                    break;
                }
                tc_fence_after_sync();
            }
            if (any) {   // O^T: a lane is a dim, a column a head
#pragma unroll 1
                for (int m = 0; m < 4; ++m)
#pragma unroll 1
                    for (int cb = 0; cb < H / 32; ++cb) {
                        uint32_t o[32];
                        const uint32_t ta = lane_base + m * H + 32 * cb;
                        tmem_ld_x32(ta, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * fac_i[32 * cb + k]);
                        tmem_st_x32(ta, o);
                    }
                tmem_st_wait();
            }
            if (h < H) {   // P row h: 32 bf16 = four 16-byte pieces of a 64-byte swizzled row
                uint8_t* prow = p_s + h * 64;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint4 w = make_uint4(f32x2_to_bf16x2_rn(p[8 * jj + 0], p[8 * jj + 1]),
                                               f32x2_to_bf16x2_rn(p[8 * jj + 2], p[8 * jj + 3]),
                                               f32x2_to_bf16x2_rn(p[8 * jj + 4], p[8 * jj + 5]),
                                               f32x2_to_bf16x2_rn(p[8 * jj + 6], p[8 * jj + 7]));
                    *reinterpret_cast<uint4*>(prow + ((jj ^ ((h >> 1) & 3)) << 4)) = w;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(p_full);
            done = i + 1;
        }
        bool have_o = false;
        if (!aborted && done == nt && nt > 0) {   // uniform: every thread ran every tile
            const bool o_ok = mbar_wait(o_done, (nt - 1) & 1, abort_flag, wait_ns);
            have_o = !bar_red_or(kSoftBar, kSoft, !o_ok);
            if (!have_o) give_up(26);
            else tc_fence_after_sync();
        }
        if (h < H) {
            m_s[h] = m_used;
            l_s[h] = have_o ? l : 0.f;
        }
        named_bar_sync(kSoftBar, kSoft);
        // results: a thread owns dim 128m + 32*quarter + lane of every head
        if (n_split == 1) {
            if (h < H) {
                const float lh = l_s[h];
                lse[(int64_t)t * H + h] = lh > 0.f ? (m_s[h] + log2f(lh)) * 0.69314718055994531f : -INFINITY;
            }
        } else {
            if (h < H) {
                float* ml = part_ml + (((int64_t)t * n_split + sp) * H + h) * 2;
                ml[0] = m_s[h];
                ml[1] = l_s[h];
            }
        }
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
            const int d = 128 * m + 32 * quarter + lane;
#pragma unroll 1
            for (int cb = 0; cb < H / 32; ++cb) {
                uint32_t o[32];
                if (have_o) {
                    tmem_ld_x32(lane_base + m * H + 32 * cb, o);
                    tmem_ld_wait(o);
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int hh = 32 * cb + k;
                    if (n_split == 1) {
                        const float lh = l_s[hh];
                        out[((int64_t)t * H + hh) * kMlaV + d] =
                            have_o && lh > 0.f ? __uint_as_float(o[k]) / lh : 0.f;
                    } else if (have_o) {
                        part_o[(((int64_t)t * n_split + sp) * H + hh) * kMlaV + d] = __uint_as_float(o[k]);
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// out[t,h,:] and lse[t,h] from the splits' (O, m, l): weights 2^(m_s - M)
// with M the largest m among the splits that saw any row (l_s > 0). One block
// per (t, h); the first warp finds the weights, then each thread sums one
// float4 of dims over the splits with independent loads.
constexpr int kMaxSplits = 32;

__global__ void __launch_bounds__(128)
sparse_mla_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int n_split,
                        int H, float* __restrict__ out, float* __restrict__ lse) {
    __shared__ float wts[kMaxSplits];
    __shared__ float inv_l;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t th = blockIdx.x;   // t * H + h
    const int64_t t = th / H, h = th % H;
    if (threadIdx.x < 32) {
        const int s = threadIdx.x;
        float m = -INFINITY, l = 0.f;
        if (s < n_split) {
            const float2 ml = *reinterpret_cast<const float2*>(part_ml + ((t * n_split + s) * H + h) * 2);
            if (ml.y > 0.f) {
                m = ml.x;
                l = ml.y;
            }
        }
        float M = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = l > 0.f ? exp2f(m - M) : 0.f;
        float L = w * l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        wts[s] = w;
        if (s == 0) {
            inv_l = L > 0.f ? 1.f / L : 0.f;
            lse[th] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
    }
    __syncthreads();
    const int d4 = threadIdx.x;   // dims 4*d4 .. 4*d4+3
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < n_split; ++s) {
        const float w = wts[s];
        if (w != 0.f) {
            const float4 o = *reinterpret_cast<const float4*>(part_o + ((t * n_split + s) * H + h) * kMlaV + 4 * d4);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
        }
    }
    const float il = inv_l;
    *reinterpret_cast<float4*>(out + th * kMlaV + 4 * d4) = make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn mla_encode_fn() {
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

template <int H, bool kFp8>
cudaError_t launch_h(const MlaArgs& a, const CUtensorMap& map, int tps, int n_split, float* part_o,
                     float* part_ml, cudaStream_t stream) {
    using Lay = MlaLayout<H, kFp8>;
    auto kern = sparse_mla_kernel<H, kFp8>;
    cudaError_t e = ensure_smem_optin((const void*)kern, Lay::kBytes);
    if (e != cudaSuccess) return e;
    const float scale_log2 = a.scale * 1.4426950408889634f;
    e = launch_kernel(kern, dim3((unsigned)((int64_t)a.T * n_split)), dim3(kThreads), (size_t)Lay::kBytes,
                      stream, 1, map, a.cache, a.cache8, a.row_scale, a.cache_rows, a.idx, a.cnt, a.cu_q,
                      a.cu_k, a.B, a.topk, scale_log2, tps, n_split, a.out, a.lse, part_o, part_ml, a.status,
                      wait_limit_ns());
    if (e != cudaSuccess || n_split == 1) return e;
    return launch_kernel(sparse_mla_merge_kernel, dim3((unsigned)((int64_t)a.T * H)), dim3(128), 0, stream, 1,
                         (const float*)part_o, (const float*)part_ml, n_split, H, a.out, a.lse);
}

}  // namespace

// Splits per query row: the fewest that minimise waves x (tiles per split + 2),
// one CTA per SM and about two tiles' worth of fixed cost per CTA (Q load,
// pipeline fill, result write); at least two tiles per split.
int mla_splits(int32_t T, int32_t topk) {
    const int64_t tiles = (topk + kTileRows - 1) / kTileRows;
    const int64_t sms = device_info().sm_count > 0 ? device_info().sm_count : 1;
    if (T <= 0) return 1;
    int64_t cap = tiles / 2 > 0 ? tiles / 2 : 1;
    if (cap > kMaxSplits) cap = kMaxSplits;
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t s = 1; s <= cap; ++s) {
        const int64_t waves = ((int64_t)T * s + sms - 1) / sms;
        const int64_t cost = waves * ((tiles + s - 1) / s + 2);
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return (int)best;
}

size_t mla_partial_bytes(int32_t T, int32_t heads, int32_t topk) {
    const int s = mla_splits(T, topk);
    if (s <= 1) return 0;
    return align_up((size_t)T * s * heads * kMlaV * 4, 256) + align_up((size_t)T * s * heads * 2 * 4, 256);
}

cudaError_t launch_sparse_mla(const MlaArgs& a, void* partials, cudaStream_t stream) {
    if (a.T <= 0) return cudaSuccess;
    EncodeTiledFn enc = mla_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)kMlaDim, (cuuint64_t)a.T * a.heads};
    const cuuint64_t strides[1] = {(cuuint64_t)kMlaDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)a.heads};
    const cuuint32_t elem[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.q), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int n_split = mla_splits(a.T, a.topk);
    const int tiles = (a.topk + kTileRows - 1) / kTileRows;
    const int tps = (tiles + n_split - 1) / n_split;
    float* part_o = nullptr;
    float* part_ml = nullptr;
    if (n_split > 1) {
        part_o = static_cast<float*>(partials);
        part_ml = reinterpret_cast<float*>(static_cast<char*>(partials) +
                                           align_up((size_t)a.T * n_split * a.heads * kMlaV * 4, 256));
    }
    const bool fp8 = a.cache8 != nullptr;
    switch (a.heads) {
        case 32: return fp8 ? launch_h<32, true>(a, map, tps, n_split, part_o, part_ml, stream)
                            : launch_h<32, false>(a, map, tps, n_split, part_o, part_ml, stream);
        case 64: return fp8 ? launch_h<64, true>(a, map, tps, n_split, part_o, part_ml, stream)
                            : launch_h<64, false>(a, map, tps, n_split, part_o, part_ml, stream);
        case 96: return fp8 ? launch_h<96, true>(a, map, tps, n_split, part_o, part_ml, stream)
                            : launch_h<96, false>(a, map, tps, n_split, part_o, part_ml, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lidx

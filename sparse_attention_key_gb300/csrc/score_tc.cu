// Tensor-core scorer of the Lightning Indexer (tcgen05 + TMEM + TMA, sm_103a).
//
//   S[t,s] = sum_h w[t,h] * max(q[t,h,:] . k[s,:], 0)     for s < n(t) = q_pos[t] + 1
//
// ("Notes from an NVFP4 port of Kimi K3.1 Pro", indexer paragraph; no rotary,
// item (3) of "Details that silently change the answer".)
//
// The per-head dot products are one dense contraction per (query group, key
// tile): D[key, (query, head)] = K_tile[128 x 128] . Q_group[(query,head) x 128]^T,
// i.e. M = 128 keys, N = 32 heads x NQ queries, K = 128 dims. Keys are the M
// side so that one TMEM lane holds one key and the relu / head-weighted sum of
// a query is a loop over 32 consecutive accumulator columns inside one thread:
// the [T,32,L] intermediate never leaves TMEM and registers.
//
// Work decomposition. Queries of a sequence form groups of GQ = NQ * NSUB
// consecutive rows; a group needs ceil(max n(t) / 128) key tiles ("steps"). A
// plan kernel lists the groups and prefix-sums their steps; the scorer runs
// one CTA per SM and gives each CTA a contiguous range of steps of equal cost
// (a step costs 1, the start of a group kGroupStartCost more), so a CTA streams
// key tiles of one group while the group's queries stay resident in shared
// memory. With one or four queries per group and a large cache,
// score_tc_dyn_kernel starts from the same ranges but claims them in chunks
// and takes chunks from the CTA with the most steps left: some SMs pull keys
// from HBM more slowly than others, and static ranges leave them last.
//
// Roles inside a CTA (warp specialisation):
//   warp 0        TMA producer: the group's Q tile once per group, then key
//                 tiles into a STAGES-deep ring (128-byte swizzle).
//   warp 1        TMEM allocator and MMA issuer (one thread): per key tile and
//                 sub-group, 8 MMAs of K = 16 into one of NACC accumulators.
//   warps 2..     epilogue: tcgen05.ld of 32 columns per query, relu, weight,
//                 head sum, coalesced store of the fp32 score (masked to the
//                 causal length).
// Every wait is bounded (globaltimer); a timeout records IDX_ERR_TIMEOUT in
// the status word, raises a shared abort flag that ends all roles, waits for
// copies and MMAs still in flight (bounded) and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc_primitives.cuh"

namespace lidx {

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
struct TcPlanHeader {
    int32_t n_groups;
    int32_t total_steps;
    int32_t pad[2];
};

constexpr int kMaxScorerCtas = 1024;   // per-CTA start descriptors in the plan
// Steps per claim of the work-stealing scorers (score_tc_dyn_kernel). The plan
// hands each CTA its first chunk: its counter starts at kDynChunk.
constexpr int kDynChunk = 4;
// Key tiles of the cache per CTA from which the decode and verification
// scorers steal work (measured: a 250K-key decode batch, 13 tiles per CTA, is
// faster with static ranges; 64 histories of 64K-128K keys gain 11%).
constexpr int kDynMinTilesPerCta = 32;

size_t tc_plan_bytes(int32_t B, int32_t T) {
    const size_t g = (size_t)T + (size_t)B + 1;  // >= number of groups for any GQ >= 1
    return align_up(sizeof(TcPlanHeader), 256) + align_up(g * sizeof(int4), 256) +
           align_up((g + 1) * sizeof(int32_t), 256) + 2 * kMaxScorerCtas * sizeof(int4) +
           kMaxScorerCtas * sizeof(int32_t);
}

struct TcPlan {
    TcPlanHeader* hdr;
    int4* groups;        // {sequence, first query row, queries, key tiles}
    int32_t* step_begin; // [n_groups + 1]
    // Per scorer CTA c: [2c] = {group of its first step, key tile of that
    // step within the group, first step of the next group, end of the CTA's
    // range}, [2c+1] = that group's entry of `groups`.
    int4* cta_desc;
    // Per scorer CTA c: steps of its range already handed out (chunks are
    // claimed by atomicAdd; see score_tc_dyn_kernel). Set by the plan.
    int32_t* claim;
    int32_t capacity;    // entries of groups
};

static TcPlan plan_layout(void* base, int32_t B, int32_t T) {
    const size_t g = (size_t)T + (size_t)B + 1;
    char* p = static_cast<char*>(base);
    TcPlan pl;
    pl.hdr = reinterpret_cast<TcPlanHeader*>(p);
    pl.groups = reinterpret_cast<int4*>(p + align_up(sizeof(TcPlanHeader), 256));
    pl.step_begin = reinterpret_cast<int32_t*>(p + align_up(sizeof(TcPlanHeader), 256) +
                                               align_up(g * sizeof(int4), 256));
    pl.cta_desc = reinterpret_cast<int4*>(p + align_up(sizeof(TcPlanHeader), 256) +
                                          align_up(g * sizeof(int4), 256) +
                                          align_up((g + 1) * sizeof(int32_t), 256));
    pl.claim = reinterpret_cast<int32_t*>(pl.cta_desc + 2 * kMaxScorerCtas);
    pl.capacity = (int32_t)g;
    return pl;
}

// Descriptor of scorer CTA c of `grid`, which takes the steps between its
// boundary and the next CTA's; its first group is found by binary search in
// sb[0..n_groups] (shared or global memory; sb[n_groups] == total > 0).
// Extra cost of starting a group, in key tiles, for the scorers: loading the
// group's queries (one buffer: the MMAs wait) and the epilogue's per-group
// set-up (and, with one query per group, its first-digit histogram flush).
constexpr int kGroupStartCost = 2;

// First step of scorer CTA c of `grid` when the CTAs share the steps by cost:
// a step costs 1, and the first step of a group kGroupStartCost more. CTA c
// starts at the first step s whose cost before it, s + kGroupStartCost * (group
// starts before s), reaches total_cost * c / grid. sb[0..n_groups] are the
// groups' first steps (sb[n_groups] = total).
__device__ __forceinline__ int32_t cost_boundary(const int32_t* sb, int n_groups, int64_t total,
                                                 int grid, int c) {
    if (c >= grid) return (int32_t)total;
    const int64_t total_cost = total + (int64_t)kGroupStartCost * n_groups;
    const int64_t target = total_cost * c / grid;
    // the last group g whose first step's cost-before (sb[g] + K*g) is <= target
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)sb[mid] + (int64_t)kGroupStartCost * mid <= target) lo = mid; else hi = mid - 1;
    }
    const int64_t at = (int64_t)sb[lo] + (int64_t)kGroupStartCost * lo;
    if (target <= at) return sb[lo];
    // inside group lo the step sb[lo] + j (j >= 1) has cost-before at + K + j
    int64_t j = target - at - kGroupStartCost;
    if (j < 1) j = 1;
    const int64_t s = (int64_t)sb[lo] + j;
    return (int32_t)(s < sb[lo + 1] ? s : sb[lo + 1]);
}


// by_cost: boundaries by cost (sb in shared memory), else uniform in steps.
__device__ __forceinline__ void write_cta_desc(const TcPlan& plan, const int32_t* sb, int n_groups,
                                               int64_t total, int grid, int c, bool by_cost) {
    const int64_t beg = by_cost ? cost_boundary(sb, n_groups, total, grid, c) : total * c / grid;
    const int64_t end = by_cost ? cost_boundary(sb, n_groups, total, grid, c + 1) : total * (c + 1) / grid;
    int lo = 0, hi = n_groups - 1;   // the last group whose first step is <= beg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sb[mid] <= beg) lo = mid; else hi = mid - 1;
    }
    plan.cta_desc[2 * c] = make_int4(lo, (int)(beg - sb[lo]), sb[lo + 1], (int)end);
    plan.cta_desc[2 * c + 1] = plan.groups[lo];
    plan.claim[c] = kDynChunk;
}

// Descriptors of a plan with no steps: every CTA has an empty range.
__device__ __forceinline__ void write_empty_descs(const TcPlan& plan, int grid) {
    for (int c = threadIdx.x; c < grid; c += blockDim.x) {
        plan.cta_desc[2 * c] = make_int4(0, 0, 0, 0);
        plan.cta_desc[2 * c + 1] = make_int4(0, 0, 0, 0);
        plan.claim[c] = 0;
    }
}

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int block_exclusive_sum(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        warp_sums[lane] = wi - ws;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const int res = warp_sums[warp] + incl - v;
    *total = warp_sums[32];
    __syncthreads();
    return res;
}

// Block 0 builds the plan (after clearing the status word when asked); any
// further blocks clear `zero_bytes` at `zero_ptr` (the selection histograms
// that the scorer's epilogue adds into).
template <int GQ>
__global__ void __launch_bounds__(kPlanThreads)
tc_plan_kernel(const int32_t* __restrict__ q_pos, const int32_t* __restrict__ cu_q,
               const int32_t* __restrict__ cu_k, int B, int T, int64_t n_keys, int64_t max_len,
               TcPlan plan, DeviceStatus* status, bool zero_status, uint4* zero_ptr,
               int64_t zero_vec, int grid) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x > 0) {
        for (int64_t i = (int64_t)(blockIdx.x - 1) * kPlanThreads + threadIdx.x; i < zero_vec;
             i += (int64_t)(gridDim.x - 1) * kPlanThreads)
            zero_ptr[i] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    if (zero_status && threadIdx.x == 0) {
        status->code = 0;
        status->detail = 0;
    }
    __shared__ int warp_sums[33];
    __shared__ int overflow;
    if (threadIdx.x == 0) overflow = 0;
    __syncthreads();

    // groups of each sequence
    int carry = 0;
    for (int base = 0; base < B; base += kPlanThreads) {
        const int b = base + threadIdx.x;
        int cnt = 0, nq = 0, q0 = 0;
        if (b < B) {
            q0 = __ldg(cu_q + b);
            nq = __ldg(cu_q + b + 1) - q0;
            if (q0 < 0 || nq < 0 || (int64_t)q0 + nq > T) {
                report_error(status, IDX_ERR_DEVICE_ARG, -1 - b);
                nq = 0;
            }
            cnt = (nq + GQ - 1) / GQ;
        }
        int total;
        const int off = carry + block_exclusive_sum(cnt, warp_sums, &total);
        for (int j = 0; j < cnt; ++j) {
            if (off + j < plan.capacity)
                plan.groups[off + j] = make_int4(b, q0 + j * GQ, min(GQ, nq - j * GQ), 0);
            else
                overflow = 1;
        }
        carry += total;
    }
    __syncthreads();
    if (overflow || carry >= plan.capacity) {  // cu_q is not a partition of 0..T
        if (threadIdx.x == 0) {
            report_error(status, IDX_ERR_DEVICE_ARG, -1);
            plan.hdr->n_groups = 0;
            plan.hdr->total_steps = 0;
            plan.step_begin[0] = 0;
        }
        write_empty_descs(plan, grid);
        return;
    }
    const int n_groups = carry;

    // key tiles of each group: the longest valid causal history among its queries
    for (int g = threadIdx.x; g < n_groups; g += kPlanThreads) {
        int4 d = plan.groups[g];
        const int64_t k0 = __ldg(cu_k + d.x), k1 = __ldg(cu_k + d.x + 1);
        const bool seq_ok = k0 >= 0 && k1 >= k0 && k1 <= n_keys;
        int64_t nmax = 0;
        for (int i = 0; i < d.z; ++i) {
            const int t = d.y + i;
            const int64_t n = (int64_t)__ldg(q_pos + t) + 1;
            if (!seq_ok || n < 1 || n > k1 - k0 || n > max_len) {
                report_error(status, IDX_ERR_DEVICE_ARG, t);
                continue;
            }
            nmax = n > nmax ? n : nmax;
        }
        d.w = (int)((nmax + 127) / 128);
        plan.groups[g] = d;
    }
    __syncthreads();

    // prefix sum of steps
    carry = 0;
    for (int base = 0; base < n_groups; base += kPlanThreads) {
        const int g = base + threadIdx.x;
        const int v = g < n_groups ? plan.groups[g].w : 0;
        int total;
        const int off = carry + block_exclusive_sum(v, warp_sums, &total);
        if (g < n_groups) plan.step_begin[g] = off;
        carry += total;
    }
    if (threadIdx.x == 0) {
        plan.step_begin[n_groups] = carry;
        plan.hdr->n_groups = n_groups;
        plan.hdr->total_steps = carry;
    }
    // per-CTA start descriptors, one thread per CTA
    if (carry == 0) {
        write_empty_descs(plan, grid);
        return;
    }
    __syncthreads();   // step_begin and groups are complete
    if constexpr (GQ > 4) {   // several queries per group: CTA c's first step, steps shared uniformly
        for (int c = threadIdx.x; c < grid; c += kPlanThreads)
            plan.cta_desc[2 * c].x = (int32_t)((int64_t)carry * c / grid);
    } else {
        for (int c = threadIdx.x; c < grid; c += kPlanThreads)
            write_cta_desc(plan, plan.step_begin, n_groups, carry, grid, c, false);
    }
}

// Fast plan for up to kPlanSeqs sequences: one thread per sequence reads its
// bounds and counts its groups (a block scan places them), then each thread
// takes a contiguous run of groups, finds their sequence in shared memory,
// reads the queries' positions (all at once) and counts the key tiles; a
// second block scan gives the groups' first steps. Two rounds of global reads
// in all, instead of a chain of dependent ones. Argument checks and error
// reports are those of tc_plan_kernel.
constexpr int kPlanSeqs = 2048;
constexpr int kPlanSbShared = 2048;   // groups whose first steps are kept in shared memory
constexpr int kPlanRegGroups = 8;     // groups per thread kept in registers

template <int GQ>
__global__ void __launch_bounds__(kPlanThreads)
tc_plan_fast_kernel(const int32_t* __restrict__ q_pos, const int32_t* __restrict__ cu_q,
                    const int32_t* __restrict__ cu_k, int B, int T, int64_t n_keys,
                    int64_t max_len, TcPlan plan, DeviceStatus* status, bool zero_status,
                    uint4* zero_ptr, int64_t zero_vec, int grid) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x > 0) {
        for (int64_t i = (int64_t)(blockIdx.x - 1) * kPlanThreads + threadIdx.x; i < zero_vec;
             i += (int64_t)(gridDim.x - 1) * kPlanThreads)
            zero_ptr[i] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    __shared__ int s_q0[kPlanSeqs], s_nq[kPlanSeqs], s_lk[kPlanSeqs], s_gofs[kPlanSeqs + 1];
    __shared__ int s_sb[kPlanSbShared + 1];   // groups' first steps, when they fit
    __shared__ int warp_sums[33];
    // Up to kPlanThreads query rows: their positions are read in the same
    // round of loads as the sequences' bounds (one dependent round trip less).
    __shared__ int s_qp[kPlanThreads];
    const bool qp_pre = T <= kPlanThreads;
    if (qp_pre && (int)threadIdx.x < T) s_qp[threadIdx.x] = __ldg(q_pos + threadIdx.x);
    if (zero_status && threadIdx.x == 0) {
        status->code = 0;
        status->detail = 0;
    }
    __syncthreads();

    // sequences: bounds, validity and group counts
    int carry = 0;
    for (int base = 0; base < B; base += kPlanThreads) {
        const int b = base + threadIdx.x;
        int cnt = 0;
        if (b < B) {
            const int q0 = __ldg(cu_q + b), q1 = __ldg(cu_q + b + 1);
            const int64_t k0 = __ldg(cu_k + b), k1 = __ldg(cu_k + b + 1);
            int nq = q1 - q0;
            if (q0 < 0 || nq < 0 || (int64_t)q0 + nq > T) {
                report_error(status, IDX_ERR_DEVICE_ARG, -1 - b);
                nq = 0;
            }
            const bool seq_ok = k0 >= 0 && k1 >= k0 && k1 <= n_keys;
            cnt = (nq + GQ - 1) / GQ;
            s_q0[b] = q0;
            s_nq[b] = nq;
            s_lk[b] = seq_ok ? (int)(k1 - k0 < 0x7fffffffLL ? k1 - k0 : 0x7fffffffLL) : -1;
        }
        int total;
        const int off = carry + block_exclusive_sum(cnt, warp_sums, &total);
        if (b < B) s_gofs[b] = off;
        carry += total;
    }
    if (threadIdx.x == 0) s_gofs[B] = carry;
    __syncthreads();
    const int n_groups = carry;
    if (n_groups >= plan.capacity) {   // cu_q is not a partition of 0..T
        if (threadIdx.x == 0) {
            report_error(status, IDX_ERR_DEVICE_ARG, -1);
            plan.hdr->n_groups = 0;
            plan.hdr->total_steps = 0;
            plan.step_begin[0] = 0;
        }
        write_empty_descs(plan, grid);
        return;
    }

    // groups: a contiguous run per thread
    const int per = (n_groups + kPlanThreads - 1) / kPlanThreads;
    const int g0 = min(n_groups, (int)threadIdx.x * per), g1 = min(n_groups, g0 + per);
    int b = 0;
    if (g0 < g1) {   // the sequence of group g0: the last b with s_gofs[b] <= g0
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_gofs[mid] <= g0) lo = mid; else hi = mid - 1;
        }
        b = lo;
    }
    int steps_r[kPlanRegGroups];
    int my_steps = 0;
    for (int g = g0, k = 0; g < g1; ++g, ++k) {
        while (g >= s_gofs[b + 1]) ++b;   // empty sequences own no group
        const int j = g - s_gofs[b];
        const int q0 = s_q0[b] + j * GQ;
        const int nq = min(GQ, s_nq[b] - j * GQ);
        const int lk = s_lk[b];
        int qp[GQ];
#pragma unroll
        for (int i = 0; i < GQ; ++i) qp[i] = i < nq ? (qp_pre ? s_qp[q0 + i] : __ldg(q_pos + q0 + i)) : 0;
        int64_t nmax = 0;
#pragma unroll
        for (int i = 0; i < GQ; ++i) {
            if (i >= nq) break;
            const int64_t n = (int64_t)qp[i] + 1;
            if (lk < 0 || n < 1 || n > lk || n > max_len) {
                report_error(status, IDX_ERR_DEVICE_ARG, q0 + i);
                continue;
            }
            nmax = n > nmax ? n : nmax;
        }
        const int steps = (int)((nmax + 127) / 128);
        plan.groups[g] = make_int4(b, q0, nq, steps);
        if (k < kPlanRegGroups) steps_r[k] = steps;
        my_steps += steps;
    }
    int total;
    int sb = block_exclusive_sum(my_steps, warp_sums, &total);
    const bool sb_shared = n_groups <= kPlanSbShared;
    for (int g = g0, k = 0; g < g1; ++g, ++k) {
        plan.step_begin[g] = sb;
        if (sb_shared) s_sb[g] = sb;
        const int4 d = k < kPlanRegGroups ? make_int4(0, 0, 0, steps_r[k]) : plan.groups[g];
        sb += d.w;
    }
    if (threadIdx.x == 0) {
        plan.step_begin[n_groups] = total;
        if (sb_shared) s_sb[n_groups] = total;
        plan.hdr->n_groups = n_groups;
        plan.hdr->total_steps = total;
    }
    if (total == 0) {
        write_empty_descs(plan, grid);
        return;
    }
    __syncthreads();   // step offsets and groups are complete
    if constexpr (GQ > 4) {
        // several queries per group: [2c].x = the first step of CTA c, the
        // steps shared by cost (uniform when the group starts are not in
        // shared memory)
        for (int c = threadIdx.x; c < grid; c += kPlanThreads)
            plan.cta_desc[2 * c].x = sb_shared ? cost_boundary(s_sb, n_groups, total, grid, c)
                                               : (int32_t)((int64_t)total * c / grid);
    } else {
        for (int c = threadIdx.x; c < grid; c += kPlanThreads)
            write_cta_desc(plan, sb_shared ? s_sb : plan.step_begin, n_groups, total, grid, c,
                           sb_shared);
    }
}

// ---------------------------------------------------------------------------
// scorer
// ---------------------------------------------------------------------------
template <int NQ_, int NSUB_, int NACC_, int STAGES_, int EPI_WARPS_>
struct TcCfg {
    static constexpr int NQ = NQ_;          // queries per MMA
    static constexpr int NSUB = NSUB_;      // MMAs (sub-groups) per key tile
    static constexpr int NACC = NACC_;      // TMEM accumulators in flight
    static constexpr int STAGES = STAGES_;  // key-tile ring depth
    static constexpr int EPI_WARPS = EPI_WARPS_;
    static constexpr int N = NQ * 32;
    static constexpr int GQ = NQ * NSUB;
    static constexpr int QROWS = GQ * 32;
    static constexpr int Q_HALF = QROWS * 128;       // bytes of one 64-dim half of Q
    static constexpr int Q_BYTES = 2 * Q_HALF;
    static constexpr int K_HALF = 128 * 128;
    static constexpr int K_STAGE = 2 * K_HALF;        // 32 KB per key tile
    static constexpr int Q_BOX_ROWS = QROWS < 256 ? QROWS : 256;
    static constexpr int TMEM_COLS = NACC * N;
    static constexpr int THREADS = (2 + EPI_WARPS) * 32;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * NACC + 4) + 16;
    // Epilogue copy of the current group: weights [GQ][32] fp32, causal length
    // (0 = no output) and score row pointer per query.
    static constexpr int EPI_BYTES = (GQ * 32 * 4 + GQ * 8 + GQ * 4 + 15) / 16 * 16;
    static constexpr int EPI_THREADS = EPI_WARPS * 32;
    // The dynamic shared-memory window starts 1024-byte aligned (the kernel has
    // no static shared memory); the kernel checks this before using it.
    // One query per group (decode): the epilogue also histograms the first
    // radix digit of each written score for the exact top-K that follows.
    static constexpr int HIST_BINS = NQ * NSUB == 1 ? kTopkDigit1Bins : 0;
    static constexpr int HIST_OFF = (Q_BYTES + STAGES * K_STAGE + EPI_BYTES + BAR_BYTES + 15) / 16 * 16;
    static constexpr int SMEM = HIST_OFF + HIST_BINS * 4;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(N % 16 == 0 && N >= 32 && N <= 256, "MMA N");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
    static_assert(EPI_WARPS == 4 || EPI_WARPS == 8 || EPI_WARPS == 16,
                  "epilogue warps cover the 4 TMEM lane quarters evenly");
    static_assert(NQ % (EPI_WARPS / 4) == 0, "queries split evenly over a quarter's warps");
    static_assert(QROWS % Q_BOX_ROWS == 0, "Q box");
};

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s: no legitimate wait comes close

// Bound of every wait in the scorer (idx_set_wait_limit_ns changes it for tests).
static std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

uint64_t set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 100 ms to drain after an abort

// Walks the steps [beg, end) of a CTA: which group, which key tile.
struct StepCursor {
    int g;
    int j;                 // key tile within the group
    int32_t next_begin;    // first step of the next group
    int4 desc;

    // From a CTA's start descriptor (see TcPlan::cta_desc).
    __device__ __forceinline__ void init(int4 start, int4 group) {
        g = start.x;
        j = start.y;
        next_begin = start.z;
        desc = group;
    }
    // By binary search for step s among the groups' first steps.
    __device__ __forceinline__ void init(int32_t s, const TcPlan& p, int n_groups) {
        int lo = 0, hi = n_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.step_begin + mid) <= s) lo = mid; else hi = mid - 1;
        }
        g = lo;
        desc = p.groups[g];
        j = s - __ldg(p.step_begin + g);
        next_begin = __ldg(p.step_begin + g + 1);
    }
    // Move to step s (= previous + 1); true when the group changed.
    __device__ __forceinline__ bool advance(int32_t s, const TcPlan& p) {
        ++j;
        if (s < next_begin) return false;
        do {
            ++g;
            next_begin = __ldg(p.step_begin + g + 1);
        } while (s >= next_begin);
        desc = p.groups[g];
        j = s - __ldg(p.step_begin + g);
        return true;
    }
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                const float* __restrict__ w, const int32_t* __restrict__ q_pos,
                const int32_t* __restrict__ cu_k, int64_t max_len, float* __restrict__ scores,
                int64_t ld, TcPlan plan, DeviceStatus* status, uint32_t* __restrict__ row_hist,
                uint64_t wait_ns) {
    using namespace ptx;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_addr(smem_raw) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
        pdl_wait();
        if (threadIdx.x == 0) report_error(status, IDX_ERR_UNSUPPORTED, 1024);
        return;
    }
    uint8_t* smem = smem_raw;
    uint8_t* q_smem = smem;
    uint8_t* k_smem = smem + C::Q_BYTES;
    float* epi_w = reinterpret_cast<float*>(k_smem + C::STAGES * C::K_STAGE);
    float** epi_row = reinterpret_cast<float**>(epi_w + C::GQ * 32);
    int32_t* epi_n = reinterpret_cast<int32_t*>(epi_row + C::GQ);
    // mbarriers: 16-byte aligned, after the epilogue area
    uint64_t* bars = reinterpret_cast<uint64_t*>(k_smem + C::STAGES * C::K_STAGE + C::EPI_BYTES);
    static_assert((C::Q_BYTES + C::STAGES * C::K_STAGE + C::EPI_BYTES) % 16 == 0, "barrier alignment");
    uint64_t* k_full = bars;
    uint64_t* k_empty = bars + C::STAGES;
    uint64_t* acc_full = bars + 2 * C::STAGES;
    uint64_t* acc_empty = acc_full + C::NACC;
    uint64_t* q_full = acc_empty + C::NACC;
    uint64_t* q_empty = q_full + 1;
    uint64_t* done_bar = q_empty + 1;
    uint64_t* epi_bar = done_bar + 1;   // epilogue warps' own barrier (bounded waits)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + C::HIST_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (int a = 0; a < C::NACC; ++a) {
            mbar_init(acc_full + a, 1);
            mbar_init(acc_empty + a, C::EPI_WARPS);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(done_bar, 1);
        mbar_init(epi_bar, C::EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Set-up above touches only this CTA's shared and tensor memory; the plan,
    // the inputs and the outputs are used after the previous kernel completes.
    pdl_wait();
    pdl_launch_dependents();

    // This CTA's steps [beg, end). A few queries per group (decode and
    // verification, where the start-up latency matters): from the CTA's start
    // descriptor. Otherwise the cursors search the plan (measured faster for
    // the 16-query configuration, whose start-up is negligible against its
    // work).
    int4 start = make_int4(0, 0, 0, 0), start_group = make_int4(0, 0, 0, 0);
    int n_groups = 0;
    int32_t beg, end;
    if (C::GQ <= 4) {
        start = plan.cta_desc[2 * blockIdx.x];
        start_group = plan.cta_desc[2 * blockIdx.x + 1];
        end = start.w;
        beg = start.z - start_group.w + start.y;
    } else {
        n_groups = plan.hdr->n_groups;
        const int64_t total = plan.hdr->total_steps;
        // the plan's cost-weighted boundaries (see cost_boundary)
        beg = plan.cta_desc[2 * blockIdx.x].x;
        end = blockIdx.x + 1 < gridDim.x ? plan.cta_desc[2 * (blockIdx.x + 1)].x : (int32_t)total;
    }
    auto start_cursor = [&](StepCursor& c) {
        if (C::GQ <= 4) c.init(start, start_group);
        else c.init(beg, plan, n_groups);
    };

    bool aborted = false;
    auto give_up = [&](int site) {
        if (!*abort_flag) report_error(status, IDX_ERR_TIMEOUT, site);
        *abort_flag = 1;
        aborted = true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && beg < end) {
            int stage = 0;
            uint32_t phase = 0;
            int q_loads = 0;
            int issued[C::STAGES];
#pragma unroll
            for (int s = 0; s < C::STAGES; ++s) issued[s] = 0;
            StepCursor cur;
            start_cursor(cur);
            bool new_group = true;
            const uint64_t key_policy = C::GQ <= 4 ? l2_policy_evict_first() : 0ull;
            for (int32_t s = beg; s < end; ++s) {
                if (s > beg) new_group = cur.advance(s, plan);
                if (new_group) {
                    if (q_loads > 0 && !mbar_wait(q_empty, (q_loads - 1) & 1, abort_flag, wait_ns)) {
                        give_up(1);
                        break;
                    }
                    mbar_arrive_expect_tx(q_full, C::Q_BYTES);
                    const int32_t qrow0 = cur.desc.y * 32;
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int r = 0; r < C::QROWS; r += C::Q_BOX_ROWS)
                            tma_load_2d(smem_addr(q_smem + half * C::Q_HALF + r * 128), &tmap_q,
                                        q_full, half * 64, qrow0 + r);
                    ++q_loads;
                }
                if (!mbar_wait(k_empty + stage, phase ^ 1, abort_flag, wait_ns)) {
                    give_up(2);
                    break;
                }
                mbar_arrive_expect_tx(k_full + stage, C::K_STAGE);
                const int32_t key_row = __ldg(cu_k + cur.desc.x) + cur.j * 128;
                uint8_t* dst = k_smem + stage * C::K_STAGE;
                if (C::GQ <= 4) {
                    // a few queries per sequence: each key tile is read about
                    // once, so it should not push the staged scores out of L2
                    tma_load_2d_hint(smem_addr(dst), &tmap_k, k_full + stage, 0, key_row, key_policy);
                    tma_load_2d_hint(smem_addr(dst + C::K_HALF), &tmap_k, k_full + stage, 64, key_row,
                                     key_policy);
                } else {
                    tma_load_2d(smem_addr(dst), &tmap_k, k_full + stage, 0, key_row);
                    tma_load_2d(smem_addr(dst + C::K_HALF), &tmap_k, k_full + stage, 64, key_row);
                }
                ++issued[stage];
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // Let every copy this lane issued land before the CTA may exit.
            // Normally the MMA warp has consumed them all already; after an
            // abort (here or, later, in another role) some may be in flight.
            {
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued[s] > 0) mbar_wait(k_full + s, (issued[s] - 1) & 1, nullptr, kDrainLimitNs);
                if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, nullptr, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && beg < end) {
            constexpr uint32_t kIdesc = idesc_bf16_f32(128, C::N);
            const uint32_t q_base = smem_addr(q_smem), k_base = smem_addr(k_smem);
            int stage = 0, acc = 0, q_uses = 0;
            uint32_t phase = 0, aphase = 0;
            StepCursor cur;
            start_cursor(cur);
            bool new_group = true;
            for (int32_t s = beg; s < end && !aborted; ++s) {
                if (s > beg) new_group = cur.advance(s, plan);
                if (new_group) {
                    if (!mbar_wait(q_full, q_uses & 1, abort_flag, wait_ns)) {
                        give_up(3);
                        break;
                    }
                    ++q_uses;
                }
                if (!mbar_wait(k_full + stage, phase, abort_flag, wait_ns)) {
                    give_up(4);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t k_addr = k_base + stage * C::K_STAGE;
#pragma unroll 1
                for (int sub = 0; sub < C::NSUB; ++sub) {
                    if (!mbar_wait(acc_empty + acc, aphase ^ 1, abort_flag, wait_ns)) {
                        give_up(5);
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + acc * C::N;
                    const uint32_t b_addr = q_base + sub * C::N * 128;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk & 3) * 32;
                        const uint64_t a_desc = smem_desc_sw128(k_addr + (kk >> 2) * C::K_HALF + koff);
                        const uint64_t b_desc = smem_desc_sw128(b_addr + (kk >> 2) * C::Q_HALF + koff);
                        tc_mma_bf16(d_tmem, a_desc, b_desc, kIdesc, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(acc_full + acc);
                    if (++acc == C::NACC) {
                        acc = 0;
                        aphase ^= 1;
                    }
                }
                if (aborted) break;
                tc_commit(k_empty + stage);
                if (s + 1 == end || s + 1 >= cur.next_begin) tc_commit(q_empty);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // Wait for every MMA issued so far (and thereby for the arrivals of
            // the commits before this one) before shared memory is released.
            tc_commit(done_bar);
            mbar_wait(done_bar, 0, nullptr, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int kSplit = C::EPI_WARPS / 4;      // warps sharing a TMEM lane quarter
        constexpr int kQpw = C::NQ / kSplit;          // queries per warp per sub-group
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;              // 0 .. EPI_THREADS-1
        const int qoff = ((warp - 2) / 4) * kQpw;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int acc = 0;
        uint32_t aphase = 0, ephase = 0;
        const bool hist_on = C::HIST_BINS > 0 && row_hist != nullptr;
        // Barrier of the epilogue warps; false when the CTA is giving up.
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            const bool ok = mbar_wait(epi_bar, ephase, abort_flag, wait_ns);
            ephase ^= 1;
            if (!ok) give_up(7);
            return ok;
        };
        // Add the shared first-digit histogram into row `t`'s and clear it.
        auto flush_hist = [&](int t) {
            uint32_t* g = row_hist + (int64_t)t * C::HIST_BINS;
            for (int b = et; b < C::HIST_BINS; b += C::EPI_THREADS) {
                const uint32_t v = hist_s[b];
                if (v) {
                    atomicAdd(g + b, v);
                    hist_s[b] = 0;
                }
            }
        };
        if (hist_on)
            for (int b = et; b < C::HIST_BINS; b += C::EPI_THREADS) hist_s[b] = 0;
        int hist_row = -1;
        if (beg < end) {
            StepCursor cur;
            start_cursor(cur);
            bool new_group = true;
            for (int32_t s = beg; s < end && !aborted; ++s) {
                if (s > beg) new_group = cur.advance(s, plan);
                if (new_group) {
                    // copy the group's weights, causal lengths and row pointers
                    if (!epi_sync()) break;
                    if (hist_on && hist_row >= 0) flush_hist(hist_row);
                    const int q0 = cur.desc.y, nq = cur.desc.z;
                    hist_row = q0;
                    for (int i = et; i < C::GQ * 32; i += C::EPI_THREADS) {
                        const int qi = i >> 5;
                        epi_w[i] = qi < nq ? __ldg(w + (int64_t)(q0 + qi) * 32 + (i & 31)) : 0.f;
                    }
                    if (et < C::GQ) {
                        const int64_t k0 = __ldg(cu_k + cur.desc.x);
                        const int64_t len_k = (int64_t)__ldg(cu_k + cur.desc.x + 1) - k0;
                        int32_t ne = 0;
                        if (et < nq) {
                            const int64_t n = (int64_t)__ldg(q_pos + q0 + et) + 1;
                            if (n >= 1 && n <= len_k && n <= max_len) ne = (int32_t)n;
                        }
                        epi_n[et] = ne;
                        epi_row[et] = scores + (int64_t)(q0 + et) * ld;
                    }
                    if (!epi_sync()) break;
                }
                const int32_t key = cur.j * 128 + quarter * 32 + lane;
#pragma unroll 1
                for (int sub = 0; sub < C::NSUB; ++sub) {
                    if (!mbar_wait(acc_full + acc, aphase, abort_flag, wait_ns)) {
                        give_up(6);
                        break;
                    }
                    tc_fence_after_sync();
                    uint32_t v[kQpw][32];
#pragma unroll
                    for (int qi = 0; qi < kQpw; ++qi)
                        tmem_ld_x32(lane_base + acc * C::N + (qoff + qi) * 32, v[qi]);
                    tmem_ld_wait(v[0]);
#pragma unroll
                    for (int qi = 1; qi < kQpw; ++qi) reg_fence(v[qi]);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty + acc);
                    if (++acc == C::NACC) {
                        acc = 0;
                        aphase ^= 1;
                    }
#pragma unroll
                    for (int qi = 0; qi < kQpw; ++qi) {
                        const int q = sub * C::NQ + qoff + qi;
                        if (key >= epi_n[q]) continue;
                        const float4* w4 = reinterpret_cast<const float4*>(epi_w + q * 32);
                        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const float4 ww = w4[h4];
                            const float2 r0 = make_float2(fmaxf(__uint_as_float(v[qi][4 * h4 + 0]), 0.f),
                                                          fmaxf(__uint_as_float(v[qi][4 * h4 + 1]), 0.f));
                            const float2 r1 = make_float2(fmaxf(__uint_as_float(v[qi][4 * h4 + 2]), 0.f),
                                                          fmaxf(__uint_as_float(v[qi][4 * h4 + 3]), 0.f));
                            acc2 = __ffma2_rn(make_float2(ww.x, ww.y), r0, acc2);
                            acc2 = __ffma2_rn(make_float2(ww.z, ww.w), r1, acc2);
                        }
                        const float S = acc2.x + acc2.y;
                        epi_row[q][key] = S;
                        if (hist_on) atomicAdd(&hist_s[score_key(S) >> 20], 1u);
                    }
                }
            }
            if (hist_on && !aborted && hist_row >= 0 && epi_sync()) flush_hist(hist_row);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// scorer with work stealing (a few queries per group: decode, verification)
// ---------------------------------------------------------------------------
// The SMs of a GB300 do not stream keys at one rate: some are 10-20% slower
// than the median, always the same ones, so equal static ranges end at
// different times. Here a CTA takes its (cost-balanced) range in chunks of
// kDynChunk steps from its own counter, and once the range is used up takes
// chunks from the CTA with the most steps left. Warp 0 schedules: it claims a
// chunk, cuts it at group boundaries into segments, hands each segment to the
// MMA issuer and the epilogue through a ring of descriptors in shared memory,
// and issues the segment's TMA loads. A group's queries are loaded when the
// group changes, into the other of two buffers, so that they land while the
// previous group still computes. The plan gives every CTA its first chunk,
// and the claim of the next own chunk is issued before the current chunk's
// loads, so the counters' latency stays off the stream of key tiles.
constexpr int kDynSegs = 8;      // segment descriptors in flight

struct DynSeg {
    int32_t s0, n;      // n steps from step s0; n == 0: no more work
    int32_t j;          // key tile of s0 within its group
    int32_t qb;         // bit 0: query buffer; bit 1: the queries are new here
    int4 desc;          // the group's entry of plan.groups
};

template <class C>
struct DynLayout {
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = 2 * C::Q_BYTES;
    static constexpr int EPI_OFF = K_OFF + C::STAGES * C::K_STAGE;
    static constexpr int BAR_OFF = EPI_OFF + C::EPI_BYTES;
    static constexpr int NBARS = 2 * C::STAGES + 2 * C::NACC + 4 + 2 * kDynSegs + 2;
    static constexpr int SEG_OFF = (BAR_OFF + NBARS * 8 + 16 + 15) / 16 * 16;
    static constexpr int HIST_OFF = SEG_OFF + kDynSegs * (int)sizeof(DynSeg);
    static constexpr int SMEM = HIST_OFF + C::HIST_BINS * 4;
    static_assert(C::Q_BYTES % 1024 == 0 && K_OFF % 1024 == 0, "swizzled tiles are 1024-byte aligned");
    static_assert(BAR_OFF % 16 == 0, "barrier alignment");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
score_tc_dyn_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                    const float* __restrict__ w, const int32_t* __restrict__ q_pos,
                    const int32_t* __restrict__ cu_k, int64_t max_len, float* __restrict__ scores,
                    int64_t ld, TcPlan plan, DeviceStatus* status, uint32_t* __restrict__ row_hist,
                    uint64_t wait_ns) {
    using namespace ptx;
    using Ly = DynLayout<C>;
    static_assert(C::GQ <= 4, "work stealing is for a few queries per group");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_addr(smem_raw) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
        pdl_wait();
        if (threadIdx.x == 0) report_error(status, IDX_ERR_UNSUPPORTED, 1024);
        return;
    }
    uint8_t* smem = smem_raw;
    uint8_t* q_smem = smem + Ly::Q_OFF;
    uint8_t* k_smem = smem + Ly::K_OFF;
    float* epi_w = reinterpret_cast<float*>(smem + Ly::EPI_OFF);
    float** epi_row = reinterpret_cast<float**>(epi_w + C::GQ * 32);
    int32_t* epi_n = reinterpret_cast<int32_t*>(epi_row + C::GQ);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::BAR_OFF);
    uint64_t* k_full = bars;
    uint64_t* k_empty = bars + C::STAGES;
    uint64_t* acc_full = bars + 2 * C::STAGES;
    uint64_t* acc_empty = acc_full + C::NACC;
    uint64_t* q_full = acc_empty + C::NACC;     // [2]
    uint64_t* q_empty = q_full + 2;             // [2]
    uint64_t* seg_full = q_empty + 2;           // [kDynSegs]
    uint64_t* seg_empty = seg_full + kDynSegs;  // [kDynSegs]
    uint64_t* done_bar = seg_empty + kDynSegs;
    uint64_t* epi_bar = done_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    DynSeg* segs = reinterpret_cast<DynSeg*>(smem + Ly::SEG_OFF);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + Ly::HIST_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
        }
        for (int a = 0; a < C::NACC; ++a) {
            mbar_init(acc_full + a, 1);
            mbar_init(acc_empty + a, C::EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(q_full + b, 1);
            mbar_init(q_empty + b, 1);
        }
        for (int i = 0; i < kDynSegs; ++i) {
            mbar_init(seg_full + i, 1);
            mbar_init(seg_empty + i, 1 + C::EPI_WARPS);
        }
        mbar_init(done_bar, 1);
        mbar_init(epi_bar, C::EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
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

    if (warp == 0) {
        // ------------------------------------------------------- scheduler + TMA
        const int me = blockIdx.x;
        const int4 st = plan.cta_desc[2 * me], sg = plan.cta_desc[2 * me + 1];
        const int32_t my_beg = st.z - sg.w + st.y, my_end = st.w;
        int own_g = st.x;            // cursor over the own range (claims only move forward)
        int32_t own_next = st.z;
        int4 own_desc = sg;
        bool own = true;
        int32_t own_off = 0;         // the first own chunk needs no claim
        int32_t own_claim = 0;       // lane 0: the claim issued for the next own chunk
        int seg_slot = 0, stage = 0, qb = 1, last_g = -1;
        uint32_t seg_phase = 0, phase = 0;
        int q_uses[2] = {0, 0};
        int issued[C::STAGES];
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) issued[s] = 0;
        const uint64_t key_policy = l2_policy_evict_first();
        while (!aborted) {
            // ---- claim a chunk [c0, c1) and the cursor at the group holding c0
            int32_t c0 = 0, c1 = 0, nxt = 0;
            int g = 0;
            int4 d = make_int4(0, 0, 0, 0);
            if (own) {
                if (own_off < my_end - my_beg) {
                    c0 = my_beg + own_off;
                    c1 = min(c0 + kDynChunk, my_end);
                    g = own_g;
                    nxt = own_next;
                    d = own_desc;
                    // claim the next own chunk now; its offset is read after this
                    // chunk's loads are issued, so the atomic's latency is hidden
                    if (lane == 0) own_claim = atomicAdd(plan.claim + me, kDynChunk);
                } else {
                    own = false;
                }
            }
            if (!own) {   // the CTA with the most steps left
                bool got = false;
                for (int attempt = 0; attempt < 4 && !got; ++attempt) {
                    int best_v = -1;
                    int32_t best_rem = 0;
                    for (int v = lane; v < (int)gridDim.x; v += 32) {
                        const int4 vs = plan.cta_desc[2 * v];
                        const int32_t len = vs.w - (vs.z - plan.cta_desc[2 * v + 1].w + vs.y);
                        const int32_t rem = len - *reinterpret_cast<volatile const int32_t*>(plan.claim + v);
                        if (rem > best_rem) {
                            best_rem = rem;
                            best_v = v;
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const int32_t r2 = __shfl_xor_sync(0xffffffffu, best_rem, o);
                        const int v2 = __shfl_xor_sync(0xffffffffu, best_v, o);
                        if (r2 > best_rem || (r2 == best_rem && v2 < best_v)) {
                            best_rem = r2;
                            best_v = v2;
                        }
                    }
                    if (best_rem <= 0 || best_v < 0) break;   // nothing left anywhere
                    int32_t off = 0;
                    if (lane == 0) off = atomicAdd(plan.claim + best_v, kDynChunk);
                    off = __shfl_sync(0xffffffffu, off, 0);
                    const int4 vs = plan.cta_desc[2 * best_v], vg = plan.cta_desc[2 * best_v + 1];
                    const int32_t vbeg = vs.z - vg.w + vs.y;
                    if (off < vs.w - vbeg) {
                        got = true;
                        c0 = vbeg + off;
                        c1 = min(c0 + kDynChunk, vs.w);
                        g = vs.x;
                        nxt = vs.z;
                        d = vg;
                    }
                }
                if (!got) break;
            }
            // ---- cut the chunk at group boundaries; publish and load each segment
            int32_t s = c0;
            while (s < c1 && !aborted) {
                while (s >= nxt) {   // the group holding step s
                    ++g;
                    d = plan.groups[g];
                    nxt = __ldg(plan.step_begin + g + 1);
                }
                const int32_t e = min(c1, nxt);
                const int32_t j0 = s - (nxt - d.w);
                const bool new_q = g != last_g;
                if (new_q) {
                    qb ^= 1;
                    last_g = g;
                }
                if (lane == 0) {
                    if (!mbar_wait(seg_empty + seg_slot, seg_phase ^ 1, abort_flag, wait_ns)) give_up(11);
                    if (!aborted) {
                        DynSeg sd;
                        sd.s0 = s;
                        sd.n = e - s;
                        sd.j = j0;
                        sd.qb = qb | (new_q ? 2 : 0);
                        sd.desc = d;
                        segs[seg_slot] = sd;
                        mbar_arrive(seg_full + seg_slot);
                    }
                    if (!aborted && new_q) {
                        if (q_uses[qb] > 0 && !mbar_wait(q_empty + qb, (q_uses[qb] - 1) & 1, abort_flag, wait_ns))
                            give_up(12);
                        if (!aborted) {
                            mbar_arrive_expect_tx(q_full + qb, C::Q_BYTES);
                            const int32_t qrow0 = d.y * 32;
                            uint8_t* qdst = q_smem + qb * C::Q_BYTES;
#pragma unroll
                            for (int half = 0; half < 2; ++half)
#pragma unroll
                                for (int r = 0; r < C::QROWS; r += C::Q_BOX_ROWS)
                                    tma_load_2d(smem_addr(qdst + half * C::Q_HALF + r * 128), &tmap_q,
                                                q_full + qb, half * 64, qrow0 + r);
                            ++q_uses[qb];
                        }
                    }
                    const int32_t key0 = __ldg(cu_k + d.x);
                    for (int32_t i = 0; i < e - s && !aborted; ++i) {
                        if (!mbar_wait(k_empty + stage, phase ^ 1, abort_flag, wait_ns)) {
                            give_up(13);
                            break;
                        }
                        mbar_arrive_expect_tx(k_full + stage, C::K_STAGE);
                        const int32_t key_row = key0 + (j0 + i) * 128;
                        uint8_t* dst = k_smem + stage * C::K_STAGE;
                        tma_load_2d_hint(smem_addr(dst), &tmap_k, k_full + stage, 0, key_row, key_policy);
                        tma_load_2d_hint(smem_addr(dst + C::K_HALF), &tmap_k, k_full + stage, 64, key_row,
                                         key_policy);
                        ++issued[stage];
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
                if (++seg_slot == kDynSegs) {
                    seg_slot = 0;
                    seg_phase ^= 1;
                }
                aborted = __shfl_sync(0xffffffffu, aborted ? 1 : 0, 0) != 0;
                s = e;
            }
            if (own) {
                own_g = g;
                own_next = nxt;
                own_desc = d;
                own_off = __shfl_sync(0xffffffffu, own_claim, 0);
            }
        }
        if (lane == 0) {
            if (!aborted) {   // the end marker
                if (mbar_wait(seg_empty + seg_slot, seg_phase ^ 1, abort_flag, wait_ns)) {
                    segs[seg_slot].n = 0;
                    mbar_arrive(seg_full + seg_slot);
                } else {
                    give_up(14);
                }
            }
            // let every copy this lane issued land before the CTA may exit
            for (int s = 0; s < C::STAGES; ++s)
                if (issued[s] > 0) mbar_wait(k_full + s, (issued[s] - 1) & 1, nullptr, kDrainLimitNs);
            for (int b = 0; b < 2; ++b)
                if (q_uses[b] > 0) mbar_wait(q_full + b, (q_uses[b] - 1) & 1, nullptr, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdesc = idesc_bf16_f32(128, C::N);
            const uint32_t q_base = smem_addr(q_smem), k_base = smem_addr(k_smem);
            int seg_slot = 0, stage = 0, acc = 0, cur_qb = -1;
            uint32_t seg_phase = 0, phase = 0, aphase = 0;
            int q_uses[2] = {0, 0};
            while (!aborted) {
                if (!mbar_wait(seg_full + seg_slot, seg_phase, abort_flag, wait_ns)) {
                    give_up(15);
                    break;
                }
                const DynSeg sd = segs[seg_slot];
                mbar_arrive(seg_empty + seg_slot);
                if (++seg_slot == kDynSegs) {
                    seg_slot = 0;
                    seg_phase ^= 1;
                }
                if (sd.n == 0) break;
                const int qb = sd.qb & 1;
                if (sd.qb & 2) {   // new queries: the previous buffer is free once its MMAs are done
                    if (cur_qb >= 0) tc_commit(q_empty + cur_qb);
                    if (!mbar_wait(q_full + qb, q_uses[qb] & 1, abort_flag, wait_ns)) {
                        give_up(16);
                        break;
                    }
                    ++q_uses[qb];
                    cur_qb = qb;
                }
                for (int32_t i = 0; i < sd.n && !aborted; ++i) {
                    if (!mbar_wait(k_full + stage, phase, abort_flag, wait_ns)) {
                        give_up(17);
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t k_addr = k_base + stage * C::K_STAGE;
#pragma unroll 1
                    for (int sub = 0; sub < C::NSUB; ++sub) {
                        if (!mbar_wait(acc_empty + acc, aphase ^ 1, abort_flag, wait_ns)) {
                            give_up(18);
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t d_tmem = tmem_base + acc * C::N;
                        const uint32_t b_addr = q_base + qb * C::Q_BYTES + sub * C::N * 128;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t koff = (kk & 3) * 32;
                            const uint64_t a_desc = smem_desc_sw128(k_addr + (kk >> 2) * C::K_HALF + koff);
                            const uint64_t b_desc = smem_desc_sw128(b_addr + (kk >> 2) * C::Q_HALF + koff);
                            tc_mma_bf16(d_tmem, a_desc, b_desc, kIdesc, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(acc_full + acc);
                        if (++acc == C::NACC) {
                            acc = 0;
                            aphase ^= 1;
                        }
                    }
                    if (aborted) break;
                    tc_commit(k_empty + stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every MMA issued so far (and the arrivals of the commits before) completes
            tc_commit(done_bar);
            mbar_wait(done_bar, 0, nullptr, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int kSplit = C::EPI_WARPS / 4;
        constexpr int kQpw = C::NQ / kSplit;
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;
        const int qoff = ((warp - 2) / 4) * kQpw;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int acc = 0, seg_slot = 0;
        uint32_t aphase = 0, ephase = 0, seg_phase = 0;
        const bool hist_on = C::HIST_BINS > 0 && row_hist != nullptr;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            const bool ok = mbar_wait(epi_bar, ephase, abort_flag, wait_ns);
            ephase ^= 1;
            if (!ok) give_up(19);
            return ok;
        };
        auto flush_hist = [&](int t) {
            uint32_t* gh = row_hist + (int64_t)t * C::HIST_BINS;
            for (int b = et; b < C::HIST_BINS; b += C::EPI_THREADS) {
                const uint32_t v = hist_s[b];
                if (v) {
                    atomicAdd(gh + b, v);
                    hist_s[b] = 0;
                }
            }
        };
        if (hist_on)
            for (int b = et; b < C::HIST_BINS; b += C::EPI_THREADS) hist_s[b] = 0;
        int hist_row = -1, cur_q0 = -1;
        while (!aborted) {
            if (!mbar_wait(seg_full + seg_slot, seg_phase, abort_flag, wait_ns)) {
                give_up(20);
                break;
            }
            const DynSeg sd = segs[seg_slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(seg_empty + seg_slot);
            if (++seg_slot == kDynSegs) {
                seg_slot = 0;
                seg_phase ^= 1;
            }
            if (sd.n == 0) break;
            if (sd.desc.y != cur_q0) {   // a new group: its weights, causal lengths, row pointers
                if (!epi_sync()) break;
                if (hist_on && hist_row >= 0) flush_hist(hist_row);
                const int q0 = sd.desc.y, nq = sd.desc.z;
                hist_row = q0;
                cur_q0 = q0;
                for (int i = et; i < C::GQ * 32; i += C::EPI_THREADS) {
                    const int qi = i >> 5;
                    epi_w[i] = qi < nq ? __ldg(w + (int64_t)(q0 + qi) * 32 + (i & 31)) : 0.f;
                }
                if (et < C::GQ) {
                    const int64_t k0 = __ldg(cu_k + sd.desc.x);
                    const int64_t len_k = (int64_t)__ldg(cu_k + sd.desc.x + 1) - k0;
                    int32_t ne = 0;
                    if (et < nq) {
                        const int64_t n = (int64_t)__ldg(q_pos + q0 + et) + 1;
                        if (n >= 1 && n <= len_k && n <= max_len) ne = (int32_t)n;
                    }
                    epi_n[et] = ne;
                    epi_row[et] = scores + (int64_t)(q0 + et) * ld;
                }
                if (!epi_sync()) break;
            }
            for (int32_t i = 0; i < sd.n && !aborted; ++i) {
                const int32_t key = (sd.j + i) * 128 + quarter * 32 + lane;
#pragma unroll 1
                for (int sub = 0; sub < C::NSUB; ++sub) {
                    if (!mbar_wait(acc_full + acc, aphase, abort_flag, wait_ns)) {
                        give_up(21);
                        break;
                    }
                    tc_fence_after_sync();
                    uint32_t v[kQpw][32];
#pragma unroll
                    for (int qi = 0; qi < kQpw; ++qi)
                        tmem_ld_x32(lane_base + acc * C::N + (qoff + qi) * 32, v[qi]);
                    tmem_ld_wait(v[0]);
#pragma unroll
                    for (int qi = 1; qi < kQpw; ++qi) reg_fence(v[qi]);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty + acc);
                    if (++acc == C::NACC) {
                        acc = 0;
                        aphase ^= 1;
                    }
#pragma unroll
                    for (int qi = 0; qi < kQpw; ++qi) {
                        const int q = sub * C::NQ + qoff + qi;
                        if (key >= epi_n[q]) continue;
                        const float4* w4 = reinterpret_cast<const float4*>(epi_w + q * 32);
                        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const float4 ww = w4[h4];
                            const float2 r0 = make_float2(fmaxf(__uint_as_float(v[qi][4 * h4 + 0]), 0.f),
                                                          fmaxf(__uint_as_float(v[qi][4 * h4 + 1]), 0.f));
                            const float2 r1 = make_float2(fmaxf(__uint_as_float(v[qi][4 * h4 + 2]), 0.f),
                                                          fmaxf(__uint_as_float(v[qi][4 * h4 + 3]), 0.f));
                            acc2 = __ffma2_rn(make_float2(ww.x, ww.y), r0, acc2);
                            acc2 = __ffma2_rn(make_float2(ww.z, ww.w), r1, acc2);
                        }
                        const float S = acc2.x + acc2.y;
                        epi_row[q][key] = S;
                        if (hist_on) atomicAdd(&hist_s[score_key(S) >> 20], 1u);
                    }
                }
            }
        }
        if (hist_on && !aborted && hist_row >= 0 && epi_sync()) flush_hist(hist_row);
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
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

// 2-D bf16 tensor [rows, 128] with 256-byte rows, loaded as {64, box_rows}
// boxes with the 128-byte swizzle; rows past the end read as zero.
static bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {128, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prefill: 16 queries per group as 2 MMAs of N = 256, two 256-column TMEM
// accumulators, 3-stage key ring, 16 epilogue warps (4 per TMEM lane quarter,
// 2 queries each per MMA).
using PrefillCfg = TcCfg<8, 2, 2, 3, 16>;
// Decode: one query per group, N = 32, four accumulators, 6-stage key ring.
using DecodeCfg = TcCfg<1, 1, 4, 6, 4>;
// Speculative verification (a few queries per sequence): 4 queries per group
// as one MMA of N = 128, four 128-column accumulators, 5-stage key ring, 8
// epilogue warps (2 per TMEM lane quarter, 2 queries each).
using VerifyCfg = TcCfg<4, 1, 4, 5, 8>;

template <class C>
static cudaError_t launch_cfg(const ScoreArgs& a, const TcPlan& plan, cudaStream_t stream,
                             bool* hist_filled) {
    uint32_t* row_hist = C::HIST_BINS > 0 ? a.row_hist : nullptr;
    if (hist_filled) *hist_filled = row_hist != nullptr;
    CUtensorMap tk, tq;
    if (!make_tmap(&tk, a.k, a.n_keys, 128) || !make_tmap(&tq, a.q, (int64_t)a.T * 32, C::Q_BOX_ROWS))
        return cudaErrorInvalidValue;
    const int64_t zero_vec = a.zero_ptr != nullptr ? (int64_t)(a.zero_bytes / 16) : 0;
    const int64_t zero_blocks = zero_vec > 0 ? (zero_vec + 4 * kPlanThreads - 1) / (4 * kPlanThreads) : 0;
    const int plan_grid = 1 + (int)(zero_blocks < 64 ? zero_blocks : 64);
    const DeviceInfo& dev = device_info();
    if (dev.sm_count < 1 || dev.sm_count > kMaxScorerCtas) return cudaErrorInvalidValue;
    cudaError_t e = launch_kernel(a.B <= kPlanSeqs ? tc_plan_fast_kernel<C::GQ> : tc_plan_kernel<C::GQ>,
                                  dim3(plan_grid), dim3(kPlanThreads), 0, stream, 1, a.q_pos, a.cu_q,
                                  a.cu_k, a.B, a.T, a.n_keys, a.max_len, plan, a.status,
                                  a.zero_status, reinterpret_cast<uint4*>(a.zero_ptr), zero_vec,
                                  dev.sm_count);
    if (e != cudaSuccess) return e;
    // A few queries per group and enough key tiles per CTA (the keys of the
    // cache bound the steps): work stealing between the CTAs. With less work
    // per CTA the claims and the final search for work would cost more than
    // the imbalance they remove.
    const bool steal = C::GQ <= 4 && (a.n_keys + 127) / 128 >= (int64_t)kDynMinTilesPerCta * dev.sm_count;
    if constexpr (C::GQ <= 4) if (steal) {
        constexpr int kSmem = DynLayout<C>::SMEM;
        e = ensure_smem_optin((const void*)score_tc_dyn_kernel<C>, kSmem);
        if (e != cudaSuccess) return e;
        return launch_kernel(score_tc_dyn_kernel<C>, dim3(dev.sm_count), dim3(C::THREADS), (size_t)kSmem,
                             stream, 1, tk, tq, a.w, a.q_pos, a.cu_k, a.max_len, a.scores, a.ld, plan,
                             a.status, row_hist, g_wait_limit_ns.load());
    }
    e = ensure_smem_optin((const void*)score_tc_kernel<C>, C::SMEM);
    if (e != cudaSuccess) return e;
    return launch_kernel(score_tc_kernel<C>, dim3(dev.sm_count), dim3(C::THREADS), (size_t)C::SMEM,
                         stream, 1, tk, tq, a.w, a.q_pos, a.cu_k, a.max_len, a.scores, a.ld, plan,
                         a.status, row_hist, g_wait_limit_ns.load());
}

cudaError_t launch_score_tc(const ScoreArgs& a, void* plan_ws, cudaStream_t stream,
                            bool* hist_filled) {
    const TcPlan plan = plan_layout(plan_ws, a.B, a.T);
    // Mostly one query per sequence (decode), a few (speculative
    // verification), or many (prefill / chunks).
    if ((int64_t)a.T <= 2 * (int64_t)a.B) return launch_cfg<DecodeCfg>(a, plan, stream, hist_filled);
    if ((int64_t)a.T <= 4 * (int64_t)a.B) return launch_cfg<VerifyCfg>(a, plan, stream, hist_filled);
    return launch_cfg<PrefillCfg>(a, plan, stream, hist_filled);
}

}  // namespace lidx

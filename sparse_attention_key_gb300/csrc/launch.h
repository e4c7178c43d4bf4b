// Host-side launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "common.cuh"

namespace lidx {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;   // bytes of shared memory a block may opt in to
    size_t l2_bytes = 0;
};

// A named NVTX range around one entry point's host work (argument checks and
// launches), shown on Nsight timelines; NVTX does nothing when no tool is
// attached.
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

// Set the calling thread's idx_last_error() text.
void set_last_error_text(const char* msg);

// Count one kernel launch (reported by idx_kernel_launches).
void count_launch(int n = 1);

// After a kernel was enqueued on `stream`: record the calling thread's next
// measurement event there, if idx_set_kernel_events armed any.
void after_launch(cudaStream_t stream);

// Properties of the current device (cached per device).
const DeviceInfo& device_info();

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per device.
cudaError_t ensure_smem_optin(const void* kernel, int64_t bytes);

// Static shared memory of `kernel` as compiled (bytes), or -1.
int64_t kernel_static_smem(const void* kernel);

// Launch `kernel` on `stream` as a programmatic dependent launch (it may be
// scheduled while the previous kernel finishes; the kernel itself waits with
// pdl_wait() before touching global data), optionally as clusters of
// `cluster` CTAs along x. Counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    count_launch();
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) after_launch(stream);
    return e;
}

// slot == NULL: row r of k_raw -> row r of k_out. Otherwise row r -> row
// slot[r] of k_out ([out_rows,128]); out-of-range slots write nothing.
cudaError_t launch_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                                 bool f32_params, float eps, uint16_t* k_out, int64_t n_rows,
                                 cudaStream_t stream, const int64_t* slot = nullptr,
                                 int64_t out_rows = 0);

// Arguments of one scoring call (device pointers, host sizes).
struct ScoreArgs {
    const uint16_t* q;
    const uint16_t* k;
    const float* w;
    const int32_t* q_pos;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t B, T;
    int64_t n_keys;    // rows of k
    int64_t max_len;
    float* scores;
    int64_t ld;
    DeviceStatus* status;
    // Optional [T][kTopkDigit1Bins] first-digit histograms of the written
    // scores (zeroed before the scorer runs), filled by scorers that support it.
    uint32_t* row_hist = nullptr;
    // Device memory the plan kernel clears before anything else of the call
    // runs: the status word (when zero_status) and zero_bytes (a multiple of
    // 16) at zero_ptr (16-byte aligned; may be NULL).
    bool zero_status = false;
    void* zero_ptr = nullptr;
    size_t zero_bytes = 0;
};

// Tensor-core scorer (tcgen05/TMEM/TMA): a plan kernel, then the persistent
// scorer. `plan_ws` holds tc_plan_bytes(B, T) bytes of device scratch.
size_t tc_plan_bytes(int32_t B, int32_t T);
// Bound of every wait in the tensor-core kernels, in ns; returns the previous one.
uint64_t set_wait_limit_ns(uint64_t ns);
uint64_t wait_limit_ns();

// *hist_filled (may be NULL) tells whether a.row_hist was filled.
cudaError_t launch_score_tc(const ScoreArgs& a, void* plan_ws, cudaStream_t stream,
                            bool* hist_filled = nullptr);

// Arguments of one top-K call.
struct TopkArgs {
    const float* scores;
    int64_t ld;
    const int32_t* n_valid;   // per-row count, or q_pos when n_from_pos
    bool n_from_pos;          // n(t) = n_valid[t] + 1
    int32_t T;
    int64_t max_len;
    int32_t topk;
    int32_t* idx;
    int32_t* cnt;
    DeviceStatus* status;
    // Optional (fused call): the batch layout, used to skip rows whose query
    // position lies outside its sequence. NULL when the caller gives n_valid.
    const int32_t* cu_q = nullptr;
    const int32_t* cu_k = nullptr;
    int32_t B = 0;
    // Global scratch (topk_scratch_bytes; NULL when that size is 0): position
    // bitmaps of very long rows, or the split path's row histograms and bitmaps.
    uint32_t* bits_scratch = nullptr;
    // Split path only: 0 = row histograms not prepared, 1 = zeroed,
    // 2 = first-digit histograms already filled by the scorer.
    int hist_state = 0;
};

// Device scratch launch_topk needs for rows of up to max_len (often 0).
size_t topk_scratch_bytes(int32_t T, int64_t max_len);
// Split path (few long rows): its [T][kTopkDigit1Bins] first-digit row
// histograms inside bits_scratch, or NULL when the call does not take it.
uint32_t* topk_split_row_hist(const TopkArgs& a);
// The split path's row histograms must start at zero: returns the region to
// clear (and sets a->hist_state = 1), or sets *bytes = 0 when there is none.
void topk_prepare(TopkArgs* a, void** ptr, size_t* bytes);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

// Arguments of one sparse MLA call (device pointers, host sizes).
struct MlaArgs {
    const uint16_t* q;       // bf16 [T, heads, 576]
    const uint16_t* cache;   // bf16 [cache_rows, 576]
    int64_t cache_rows;
    const int32_t* idx;      // [T, topk]
    const int32_t* cnt;      // [T]
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t B, T, heads, topk;
    float scale;
    float* out;              // fp32 [T, heads, 512]
    float* lse;              // fp32 [T, heads]
    DeviceStatus* status;
    // FP8 cache (instead of `cache`): E4M3 codes [cache_rows, 576] and one
    // fp32 scale per row; NULL for the bf16 cache.
    const uint8_t* cache8 = nullptr;
    const float* row_scale = nullptr;
};

// Key splits per query row (1: the kernel writes out/lse itself).
int mla_splits(int32_t T, int32_t topk);
// Device scratch for the splits' partial results (0 when there is one split).
size_t mla_partial_bytes(int32_t T, int32_t heads, int32_t topk);
// The attention kernel, then (several splits) the merge; `partials` holds
// mla_partial_bytes(T, heads, topk) bytes, 256-byte aligned.
cudaError_t launch_sparse_mla(const MlaArgs& a, void* partials, cudaStream_t stream);

}  // namespace lidx

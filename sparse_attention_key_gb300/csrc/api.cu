// C ABI of the Lightning Indexer library: argument checks, workspace layout and
// kernel dispatch. Declarations and the contract of each call are in
// include/lightning_indexer.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace lidx {

static thread_local char g_last_error[512] = "";

static idx_status fail(idx_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

// Lets other translation units of the library report through idx_last_error().
void set_last_error_text(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

static idx_status cuda_fail(cudaError_t e, const char* where) {
    return fail(IDX_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Measurement events of the calling thread (idx_set_kernel_events).
constexpr int kMaxKernelEvents = 16;
static thread_local cudaEvent_t g_kernel_events[kMaxKernelEvents];
static thread_local int g_kernel_events_n = 0;
static thread_local int g_kernel_events_next = 0;

void after_launch(cudaStream_t stream) {
    if (g_kernel_events_next < g_kernel_events_n)
        cudaEventRecord(g_kernel_events[g_kernel_events_next++], stream);
}

static constexpr int kMaxDevices = 64;

const DeviceInfo& device_info() {
    static DeviceInfo infos[kMaxDevices];
    static std::once_flag flags[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        static DeviceInfo none;
        return none;
    }
    std::call_once(flags[dev], [dev]() {
        DeviceInfo d;
        d.device = dev;
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        int l2 = 0;
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        d.l2_bytes = (size_t)l2;
        infos[dev] = d;
    });
    return infos[dev];
}

// Static shared memory of a kernel (as compiled), cached per kernel.
int64_t kernel_static_smem(const void* kernel) {
    static std::mutex mu;
    static const void* keys[256];
    static int64_t vals[256];
    static int n = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (keys[i] == kernel) return vals[i];
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess) return -1;
    if (n < 256) {
        keys[n] = kernel;
        vals[n] = (int64_t)attr.sharedSizeBytes;
        ++n;
    }
    return (int64_t)attr.sharedSizeBytes;
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t ensure_smem_optin(const void* kernel, int64_t bytes) {
    static std::mutex mu;
    static const void* done_kernel[256];
    static int done_dev[256];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_kernel[i] == kernel && done_dev[i] == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (n_done < 256) {
        done_kernel[n_done] = kernel;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return cudaSuccess;
}

static idx_status check_device() {
    const DeviceInfo& d = device_info();
    if (d.device < 0) return fail(IDX_ERR_CUDA, "no current CUDA device");
    if (!(d.cc_major == 10 && d.cc_minor == 3))
        return fail(IDX_ERR_UNSUPPORTED, "device compute capability %d.%d: this library is built "
                    "for sm_103a (GB300) only", d.cc_major, d.cc_minor);
    return IDX_OK;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Staged-score row stride used inside a fused call's workspace.
static int64_t staged_ld(int64_t max_len) { return (int64_t)align_up((size_t)max_len, 4); }

static size_t score_plan_bytes(int32_t B, int32_t T) { return tc_plan_bytes(B, T); }

static idx_status check_batch(const void* q, const void* k, const void* w, const void* q_pos,
                              const void* cu_q, const void* cu_k, int32_t B, int32_t T,
                              int64_t n_keys, int64_t max_len) {
    if (B < 1) return fail(IDX_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
    if (T < 0) return fail(IDX_ERR_INVALID_ARG, "T must be >= 0 (got %d)", T);
    if (n_keys < 0 || n_keys > 0x7fffffffLL)
        return fail(IDX_ERR_INVALID_ARG, "n_keys must be in [0, 2^31-1] (got %lld)",
                    (long long)n_keys);
    if (max_len < 1 || max_len > 0x7fffffffLL)
        return fail(IDX_ERR_INVALID_ARG, "max_len must be in [1, 2^31-1] (got %lld)",
                    (long long)max_len);
    if (!cu_q || !cu_k) return fail(IDX_ERR_INVALID_ARG, "cu_q / cu_k must not be NULL");
    if (T > 0 && (!q || !k || !w || !q_pos))
        return fail(IDX_ERR_INVALID_ARG, "q, k, w and q_pos must not be NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 16) || !aligned(q_pos, 4) ||
        !aligned(cu_q, 4) || !aligned(cu_k, 4))
        return fail(IDX_ERR_INVALID_ARG, "q, k, w must be 16-byte aligned; int32 arrays 4-byte");
    return IDX_OK;
}

static idx_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (!ws) return fail(IDX_ERR_WORKSPACE, "workspace must not be NULL");
    if (!aligned(ws, 256)) return fail(IDX_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(IDX_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", ws_bytes,
                    need);
    return IDX_OK;
}

static idx_status clear_status(void* ws, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(DeviceStatus), s);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "cudaMemsetAsync(status)");
}

}  // namespace lidx

using namespace lidx;

extern "C" {

int32_t idx_version(void) { return 100; }

const char* idx_last_error(void) { return g_last_error; }

uint64_t idx_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t idx_set_wait_limit_ns(uint64_t limit_ns) { return set_wait_limit_ns(limit_ns); }

int32_t idx_set_kernel_events(void* const* events, int32_t n) {
    if (n < 0 || n > kMaxKernelEvents || (n > 0 && events == nullptr)) {
        fail(IDX_ERR_INVALID_ARG, "idx_set_kernel_events: n must be in [0, %d] with non-NULL events",
             kMaxKernelEvents);
        return -1;
    }
    for (int i = 0; i < n; ++i) g_kernel_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_kernel_events_n = n;
    g_kernel_events_next = 0;
    return n;
}

idx_status idx_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                             int ln_dtype, float eps, uint16_t* k_out, int64_t n_rows,
                             void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_key_layernorm");
    if (n_rows < 0) return fail(IDX_ERR_INVALID_ARG, "n_rows must be >= 0");
    if (ln_dtype != IDX_PARAM_BF16 && ln_dtype != IDX_PARAM_F32)
        return fail(IDX_ERR_INVALID_ARG, "ln_dtype must be IDX_PARAM_BF16 or IDX_PARAM_F32");
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(IDX_ERR_INVALID_ARG, "eps must be finite, >= 0");
    if (n_rows == 0) return IDX_OK;
    if (!k_raw || !ln_w || !ln_b || !k_out)
        return fail(IDX_ERR_INVALID_ARG, "k_raw, ln_w, ln_b, k_out must not be NULL");
    if (!aligned(k_raw, 16) || !aligned(k_out, 16) || !aligned(ln_w, 4) || !aligned(ln_b, 4))
        return fail(IDX_ERR_INVALID_ARG, "k_raw/k_out must be 16-byte aligned");
    if (idx_status st = check_device()) return st;
    cudaError_t e = launch_key_layernorm(k_raw, ln_w, ln_b, ln_dtype == IDX_PARAM_F32, eps, k_out,
                                         n_rows, (cudaStream_t)stream);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "key_layernorm launch");
}

idx_status idx_key_layernorm_append(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                                    int ln_dtype, float eps, uint16_t* k_cache, int64_t cache_rows,
                                    const int64_t* slot, int64_t n_rows, void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_key_layernorm_append");
    if (n_rows < 0 || cache_rows < 0) return fail(IDX_ERR_INVALID_ARG, "n_rows and cache_rows must be >= 0");
    if (ln_dtype != IDX_PARAM_BF16 && ln_dtype != IDX_PARAM_F32)
        return fail(IDX_ERR_INVALID_ARG, "ln_dtype must be IDX_PARAM_BF16 or IDX_PARAM_F32");
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(IDX_ERR_INVALID_ARG, "eps must be finite, >= 0");
    if (n_rows == 0) return IDX_OK;
    if (!k_raw || !ln_w || !ln_b || !k_cache || !slot)
        return fail(IDX_ERR_INVALID_ARG, "k_raw, ln_w, ln_b, k_cache, slot must not be NULL");
    if (!aligned(k_raw, 16) || !aligned(k_cache, 16) || !aligned(ln_w, 4) || !aligned(ln_b, 4) ||
        !aligned(slot, 8))
        return fail(IDX_ERR_INVALID_ARG, "k_raw/k_cache must be 16-byte aligned, slot 8-byte aligned");
    if (idx_status st = check_device()) return st;
    cudaError_t e = launch_key_layernorm(k_raw, ln_w, ln_b, ln_dtype == IDX_PARAM_F32, eps, k_cache,
                                         n_rows, (cudaStream_t)stream, slot, cache_rows);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "key_layernorm_append launch");
}

size_t idx_score_workspace_size(int32_t B, int32_t T, int64_t /*max_len*/) {
    if (B < 1 || T < 0) return kWsHeader;   // arguments the call rejects
    return kWsHeader + align_up(score_plan_bytes(B, T), 256);
}

idx_status idx_score(const uint16_t* q, const uint16_t* k, const float* w, const int32_t* q_pos,
                     const int32_t* cu_q, const int32_t* cu_k, int32_t B, int32_t T,
                     int64_t n_keys, int64_t max_len, float* scores, int64_t ld, void* ws,
                     size_t ws_bytes, void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_score");
    if (idx_status st = check_batch(q, k, w, q_pos, cu_q, cu_k, B, T, n_keys, max_len)) return st;
    if (ld < max_len || ld % 4 != 0)
        return fail(IDX_ERR_INVALID_ARG, "ld must be >= max_len and a multiple of 4");
    if (T > 0 && (!scores || !aligned(scores, 16)))
        return fail(IDX_ERR_INVALID_ARG, "scores must be non-NULL and 16-byte aligned");
    if (idx_status st = check_ws(ws, ws_bytes, idx_score_workspace_size(B, T, max_len))) return st;
    if (idx_status st = check_device()) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) return clear_status(ws, s);
    ScoreArgs a{q, k, w, q_pos, cu_q, cu_k, B, T, n_keys, max_len, scores, ld, (DeviceStatus*)ws};
    a.zero_status = true;   // the plan kernel, first of the call, clears the status word
    cudaError_t e = launch_score_tc(a, (char*)ws + kWsHeader, s);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "score launch");
}

size_t idx_topk_workspace_size(int32_t T, int64_t max_len, int32_t /*topk*/) {
    return kWsHeader + align_up(topk_scratch_bytes(T, max_len), 256);
}

idx_status idx_topk(const float* scores, int64_t ld, const int32_t* n_valid, int32_t T,
                    int64_t max_len, int32_t topk, int32_t* idx, int32_t* cnt, void* ws,
                    size_t ws_bytes, void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_topk");
    if (T < 0) return fail(IDX_ERR_INVALID_ARG, "T must be >= 0");
    if (topk < 1 || topk > IDX_TOPK_MAX)
        return fail(IDX_ERR_INVALID_ARG, "topk must be in [1, %d] (got %d)", IDX_TOPK_MAX, topk);
    if (max_len < 1 || max_len > 0x7fffffffLL)
        return fail(IDX_ERR_INVALID_ARG, "max_len must be in [1, 2^31-1]");
    if (ld < 1 || ld % 4 != 0) return fail(IDX_ERR_INVALID_ARG, "ld must be a positive multiple of 4");
    if (T > 0 && (!scores || !n_valid || !idx))
        return fail(IDX_ERR_INVALID_ARG, "scores, n_valid and idx must not be NULL");
    if (!aligned(scores, 16) || !aligned(n_valid, 4) || !aligned(idx, 4) || !aligned(cnt, 4))
        return fail(IDX_ERR_INVALID_ARG, "scores must be 16-byte aligned, int32 arrays 4-byte");
    if (idx_status st = check_ws(ws, ws_bytes, idx_topk_workspace_size(T, max_len, topk))) return st;
    if (idx_status st = check_device()) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (idx_status st = clear_status(ws, s)) return st;
    if (T == 0) return IDX_OK;
    TopkArgs a{scores, ld, n_valid, false, T, max_len, topk, idx, cnt, (DeviceStatus*)ws};
    a.bits_scratch = topk_scratch_bytes(T, max_len) ? (uint32_t*)((char*)ws + kWsHeader) : nullptr;
    cudaError_t e = launch_topk(a, s);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "topk launch");
}

size_t idx_score_topk_workspace_size(int32_t B, int32_t T, int64_t max_len, int32_t /*topk*/) {
    if (B < 1 || T < 0 || max_len < 1) return kWsHeader;   // arguments the call rejects
    return kWsHeader + align_up(score_plan_bytes(B, T), 256) +
           align_up((size_t)T * (size_t)staged_ld(max_len) * sizeof(float), 256) +
           align_up(topk_scratch_bytes(T, max_len), 256);
}

idx_status idx_score_topk(const uint16_t* q, const uint16_t* k, const float* w,
                          const int32_t* q_pos, const int32_t* cu_q, const int32_t* cu_k,
                          int32_t B, int32_t T, int64_t n_keys, int64_t max_len, int32_t topk,
                          int32_t* idx, int32_t* cnt, void* ws, size_t ws_bytes, void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_score_topk");
    if (idx_status st = check_batch(q, k, w, q_pos, cu_q, cu_k, B, T, n_keys, max_len)) return st;
    if (topk < 1 || topk > IDX_TOPK_MAX)
        return fail(IDX_ERR_INVALID_ARG, "topk must be in [1, %d] (got %d)", IDX_TOPK_MAX, topk);
    if (T > 0 && !idx) return fail(IDX_ERR_INVALID_ARG, "idx must not be NULL");
    if (!aligned(idx, 4) || !aligned(cnt, 4))
        return fail(IDX_ERR_INVALID_ARG, "idx/cnt must be 4-byte aligned");
    if (idx_status st = check_ws(ws, ws_bytes, idx_score_topk_workspace_size(B, T, max_len, topk)))
        return st;
    if (idx_status st = check_device()) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) return clear_status(ws, s);
    const int64_t ld = staged_ld(max_len);
    char* base = (char*)ws + kWsHeader + align_up(score_plan_bytes(B, T), 256);
    float* scores = (float*)base;
    DeviceStatus* status = (DeviceStatus*)ws;
    TopkArgs ta{scores, ld, q_pos, true, T, max_len, topk, idx, cnt, status, cu_q, cu_k, B};
    if (topk_scratch_bytes(T, max_len))
        ta.bits_scratch = (uint32_t*)((char*)scores +
                                      align_up((size_t)T * (size_t)ld * sizeof(float), 256));
    ScoreArgs sa{q, k, w, q_pos, cu_q, cu_k, B, T, n_keys, max_len, scores, ld, status};
    // The plan kernel, first of the call, clears the status word and the few-
    // rows selection histograms (which the scorer's epilogue may fill).
    sa.zero_status = true;
    topk_prepare(&ta, &sa.zero_ptr, &sa.zero_bytes);
    sa.row_hist = topk_split_row_hist(ta);
    bool hist_filled = false;
    cudaError_t e = launch_score_tc(sa, (char*)ws + kWsHeader, s, &hist_filled);
    if (e != cudaSuccess) return cuda_fail(e, "score launch");
    if (hist_filled) ta.hist_state = 2;
    e = launch_topk(ta, s);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "topk launch");
}

idx_status idx_get_status(const void* ws, void* stream, int32_t* detail) {
    if (!ws) return fail(IDX_ERR_INVALID_ARG, "workspace must not be NULL");
    DeviceStatus h{0, 0};
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (detail) *detail = h.detail;
    return (idx_status)h.code;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Sparse MLA attention over the selected positions
// ---------------------------------------------------------------------------
extern "C" {

size_t idx_sparse_mla_workspace_size(int32_t T, int32_t heads, int32_t topk) {
    if (T < 0 || (heads != 32 && heads != 64 && heads != 96) || topk < 1 || topk > IDX_TOPK_MAX)
        return kWsHeader;
    return kWsHeader + mla_partial_bytes(T, heads, topk);
}

static idx_status sparse_mla_common(const uint16_t* q, const uint16_t* cache, const uint8_t* cache8,
                                    const float* row_scale, int64_t cache_rows, const int32_t* idx,
                                    const int32_t* cnt, const int32_t* cu_q, const int32_t* cu_k,
                                    int32_t B, int32_t T, int32_t heads, int32_t topk, float scale,
                                    float* out, float* lse, void* ws, size_t ws_bytes, void* stream);

idx_status idx_sparse_mla(const uint16_t* q, const uint16_t* cache, int64_t cache_rows,
                          const int32_t* idx, const int32_t* cnt, const int32_t* cu_q,
                          const int32_t* cu_k, int32_t B, int32_t T, int32_t heads, int32_t topk,
                          float scale, float* out, float* lse, void* ws, size_t ws_bytes,
                          void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_sparse_mla");
    if (T > 0 && cache_rows > 0 && !cache) return fail(IDX_ERR_INVALID_ARG, "cache must not be NULL");
    if (!aligned(cache, 16)) return fail(IDX_ERR_INVALID_ARG, "cache must be 16-byte aligned");
    return sparse_mla_common(q, cache, nullptr, nullptr, cache_rows, idx, cnt, cu_q, cu_k, B, T, heads,
                             topk, scale, out, lse, ws, ws_bytes, stream);
}

idx_status idx_sparse_mla_fp8(const uint16_t* q, const uint8_t* cache8, const float* row_scale,
                              int64_t cache_rows, const int32_t* idx, const int32_t* cnt,
                              const int32_t* cu_q, const int32_t* cu_k, int32_t B, int32_t T,
                              int32_t heads, int32_t topk, float scale, float* out, float* lse,
                              void* ws, size_t ws_bytes, void* stream) {
    g_last_error[0] = 0;
    TraceRange trace("idx_sparse_mla_fp8");
    if (T > 0 && cache_rows > 0 && (!cache8 || !row_scale))
        return fail(IDX_ERR_INVALID_ARG, "cache8 and row_scale must not be NULL");
    if (!aligned(cache8, 16) || !aligned(row_scale, 4))
        return fail(IDX_ERR_INVALID_ARG, "cache8 must be 16-byte aligned, row_scale 4-byte");
    return sparse_mla_common(q, nullptr, cache8, row_scale, cache_rows, idx, cnt, cu_q, cu_k, B, T,
                             heads, topk, scale, out, lse, ws, ws_bytes, stream);
}

static idx_status sparse_mla_common(const uint16_t* q, const uint16_t* cache, const uint8_t* cache8,
                                    const float* row_scale, int64_t cache_rows, const int32_t* idx,
                                    const int32_t* cnt, const int32_t* cu_q, const int32_t* cu_k,
                                    int32_t B, int32_t T, int32_t heads, int32_t topk, float scale,
                                    float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
    if (B < 1) return fail(IDX_ERR_INVALID_ARG, "B must be >= 1 (got %d)", B);
    if (T < 0) return fail(IDX_ERR_INVALID_ARG, "T must be >= 0 (got %d)", T);
    if (heads != 32 && heads != 64 && heads != 96)
        return fail(IDX_ERR_INVALID_ARG, "heads must be 32, 64 or 96 (got %d)", heads);
    if (topk < 1 || topk > IDX_TOPK_MAX)
        return fail(IDX_ERR_INVALID_ARG, "topk must be in [1, %d] (got %d)", IDX_TOPK_MAX, topk);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(IDX_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (cache_rows < 0) return fail(IDX_ERR_INVALID_ARG, "cache_rows must be >= 0");
    if (!cu_q || !cu_k) return fail(IDX_ERR_INVALID_ARG, "cu_q / cu_k must not be NULL");
    if (T > 0 && (!q || !idx || !cnt || !out || !lse))
        return fail(IDX_ERR_INVALID_ARG, "q, idx, cnt, out and lse must not be NULL");
    if (!aligned(q, 16) || !aligned(idx, 4) || !aligned(cnt, 4) ||
        !aligned(out, 16) || !aligned(lse, 4) || !aligned(cu_q, 4) || !aligned(cu_k, 4))
        return fail(IDX_ERR_INVALID_ARG,
                    "q, cache and out must be 16-byte aligned; int32 and lse arrays 4-byte");
    if ((int64_t)T * heads > 0x7fffffffLL)
        return fail(IDX_ERR_INVALID_ARG, "T * heads must be below 2^31");
    if (idx_status st = check_ws(ws, ws_bytes, idx_sparse_mla_workspace_size(T, heads, topk))) return st;
    if (idx_status st = check_device()) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (idx_status st = clear_status(ws, s)) return st;
    if (T == 0) return IDX_OK;
    MlaArgs a{q, cache, cache_rows, idx, cnt, cu_q, cu_k, B, T, heads, topk, scale, out, lse,
              (DeviceStatus*)ws};
    a.cache8 = cache8;
    a.row_scale = row_scale;
    cudaError_t e = launch_sparse_mla(a, (char*)ws + kWsHeader, s);
    return e == cudaSuccess ? IDX_OK : cuda_fail(e, "sparse_mla launch");
}

}  // extern "C"

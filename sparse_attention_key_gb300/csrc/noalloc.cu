// idx_score_topk_noalloc: the whole indexer without a caller-provided workspace.
//
// Some callers cannot hand this library any device memory beyond the tensors
// they already own: an inference engine that plans every device allocation up
// front and forbids cudaMalloc on its request path (cudaMalloc can synchronise
// the device and can fail under memory pressure mid-request), or a plugin
// that is given only its input and output buffers by a host framework that
// owns the allocator. For them this entry point keeps its scratch — the staged
// fp32 scores and the device status word — in one fixed array that lives in
// this library's own device memory, and allocates nothing.
//
// Limits and sharing:
//   - The scratch array holds kNoAllocScoreBytes (32 MiB) of staged scores:
//     T * round_up(max_len, 4) * 4 bytes must fit, e.g. 64 queries with up to
//     131,072 keys each; 1 MiB of tile plan: T + B <= 40,000; and 6 MiB of
//     selection scratch (histograms and position bitmaps of decode-sized
//     batches). Larger calls are rejected on the host (IDX_ERR_WORKSPACE).
//   - Every GPU that loads the library reserves the array (39 MiB + 256 B)
//     until the process exits.
//   - All calls on a device share the one array and it keeps the contents of
//     the last call: calls that can overlap on the GPU (different streams, or
//     different host threads without ordering) race on it. Serialise them.
//   - The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current); make that first call
//     before any stream capture. The address is cached per device and CUDA
//     context: the first call in a new context of a device (after
//     cudaDeviceReset, say) looks it up again.
//   - There is no status word to read back. A row skipped for a device-side
//     argument error shows cnt[t] == 0 and an idx row of -1; when a bounded
//     wait inside the scorer gives up (IDX_ERR_TIMEOUT in the workspace entry
//     point), every row of the call is written that way. A valid row always
//     keeps at least one position, so cnt[t] == 0 marks the failure.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace lidx {

constexpr size_t kNoAllocScoreBytes = size_t(32) << 20;  // staged fp32 scores
constexpr size_t kNoAllocPlanBytes = size_t(1) << 20;    // tile plan of the scorer
constexpr size_t kNoAllocTopkBytes = size_t(6) << 20;    // selection scratch
constexpr size_t kNoAllocScratchBytes =
    kWsHeader + kNoAllocPlanBytes + kNoAllocScoreBytes + kNoAllocTopkBytes;

// Library-owned scratch. Host code must not use this name as a pointer: on the
// host it only stands for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kNoAllocMaxDevices = 64;

idx_status noalloc_fail(idx_status code, const char* msg) {
    set_last_error_text(msg);
    return code;
}

// Id of the calling thread's current CUDA context (unique for the life of
// the process; a context made after cudaDeviceReset gets a new one), or 0
// when there is none or the driver does not say.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of the scratch array in the current device's context. It is
// looked up with cudaGetSymbolAddress, with that device current, the first
// time a context calls, and cached per device together with the context's id:
// a later context on the same device (the module is loaded again there, for
// instance after cudaDeviceReset) looks it up anew instead of using a stale
// address. Returns nullptr and fills `err` on failure.
void* noalloc_scratch(cudaError_t* err) {
    static std::mutex mu;
    static void* addr[kNoAllocMaxDevices] = {};
    static unsigned long long ctx_of[kNoAllocMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = current_context_id();   // the lookup made the context current if needed
    }
    *err = cudaSuccess;
    return addr[dev];
}

bool is_aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace
}  // namespace lidx

using namespace lidx;

extern "C" IDX_API idx_status idx_score_topk_noalloc(
    const uint16_t* q, const uint16_t* k, const float* w, const int32_t* q_pos,
    const int32_t* cu_q, const int32_t* cu_k, int32_t B, int32_t T, int64_t n_keys,
    int64_t max_len, int32_t topk, int32_t* idx, int32_t* cnt, void* stream) {
    set_last_error_text("");
    TraceRange trace("idx_score_topk_noalloc");
    if (B < 1 || T < 0) return noalloc_fail(IDX_ERR_INVALID_ARG, "B must be >= 1 and T >= 0");
    if (n_keys < 0 || n_keys > 0x7fffffffLL)
        return noalloc_fail(IDX_ERR_INVALID_ARG, "n_keys must be in [0, 2^31-1]");
    if (max_len < 1 || max_len > 0x7fffffffLL)
        return noalloc_fail(IDX_ERR_INVALID_ARG, "max_len must be in [1, 2^31-1]");
    if (topk < 1 || topk > IDX_TOPK_MAX)
        return noalloc_fail(IDX_ERR_INVALID_ARG, "topk must be in [1, 2048]");
    if (!cu_q || !cu_k || (T > 0 && (!q || !k || !w || !q_pos || !idx)))
        return noalloc_fail(IDX_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!is_aligned(q, 16) || !is_aligned(k, 16) || !is_aligned(w, 16) || !is_aligned(q_pos, 4) ||
        !is_aligned(cu_q, 4) || !is_aligned(cu_k, 4) || !is_aligned(idx, 4) || !is_aligned(cnt, 4))
        return noalloc_fail(IDX_ERR_INVALID_ARG, "q, k, w must be 16-byte aligned; int32 arrays 4-byte");
    const int64_t ld = (int64_t)align_up((size_t)max_len, 4);
    if ((size_t)T * (size_t)ld * sizeof(float) > kNoAllocScoreBytes)
        return noalloc_fail(IDX_ERR_WORKSPACE,
                            "T * round_up(max_len, 4) * 4 bytes exceeds the 32 MiB scratch of "
                            "idx_score_topk_noalloc; use idx_score_topk with a workspace");
    if (topk_scratch_bytes(T, max_len) > kNoAllocTopkBytes)
        return noalloc_fail(IDX_ERR_WORKSPACE,
                            "the selection scratch for this T and max_len exceeds the 6 MiB of "
                            "idx_score_topk_noalloc; use idx_score_topk with a workspace");
    if (tc_plan_bytes(B, T) > kNoAllocPlanBytes || (int64_t)T + B > 40000)
        return noalloc_fail(IDX_ERR_WORKSPACE,
                            "T + B exceeds the 40,000 query rows and sequences that the 1 MiB plan "
                            "of idx_score_topk_noalloc holds; use idx_score_topk with a workspace");
    const DeviceInfo& dev = device_info();
    if (dev.device < 0) return noalloc_fail(IDX_ERR_CUDA, "no current CUDA device");
    if (!(dev.cc_major == 10 && dev.cc_minor == 3))
        return noalloc_fail(IDX_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    cudaError_t e = cudaSuccess;
    unsigned char* scratch = static_cast<unsigned char*>(noalloc_scratch(&e));
    if (!scratch) return noalloc_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) return IDX_OK;
    // Only the status word and the selection histograms must start at zero
    // (the plan kernel, first of the call, clears them); every staged score is
    // written before it is read within the same call.
    DeviceStatus* status = reinterpret_cast<DeviceStatus*>(scratch);
    void* plan = scratch + kWsHeader;
    float* scores = reinterpret_cast<float*>(scratch + kWsHeader + kNoAllocPlanBytes);
    TopkArgs ta{scores, ld, q_pos, true, T, max_len, topk, idx, cnt, status, cu_q, cu_k, B};
    if (topk_scratch_bytes(T, max_len))
        ta.bits_scratch = reinterpret_cast<uint32_t*>(scratch + kWsHeader + kNoAllocPlanBytes +
                                                      kNoAllocScoreBytes);
    ScoreArgs sa{q, k, w, q_pos, cu_q, cu_k, B, T, n_keys, max_len, scores, ld, status};
    sa.zero_status = true;
    topk_prepare(&ta, &sa.zero_ptr, &sa.zero_bytes);
    sa.row_hist = topk_split_row_hist(ta);
    bool hist_filled = false;
    e = launch_score_tc(sa, plan, s, &hist_filled);
    if (e != cudaSuccess) return noalloc_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    if (hist_filled) ta.hist_state = 2;
    e = launch_topk(ta, s);
    if (e != cudaSuccess) return noalloc_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    return IDX_OK;
}

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
// of W_w). The three products are plain GEMMs and run on cuBLASLt with the
// caller's workspace; the LayerNorm writes straight into the cache rows.
#include <cublasLt.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace lidx {

namespace {

cublasLtHandle_t lt_handle(cublasStatus_t* st) {
    static std::once_flag once;
    static cublasLtHandle_t h = nullptr;
    static cublasStatus_t status = CUBLAS_STATUS_SUCCESS;
    std::call_once(once, [] { status = cublasLtCreate(&h); });
    *st = status;
    return h;
}

// One GEMM shape's cuBLASLt objects: descriptors and the algorithm chosen by
// the heuristic, built once per (M, N, K, output type, workspace size) and
// kept for the life of the process.
struct GemmPlan {
    int M, N, K;
    cudaDataType_t ctype;
    size_t ws_bytes;
    cublasLtMatmulDesc_t op;
    cublasLtMatrixLayout_t la, lb, lc;
    cublasLtMatmulAlgo_t algo;
};

cublasStatus_t make_plan(cublasLtHandle_t h, GemmPlan* p) {
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    cublasLtMatmulPreference_t pref = nullptr;
    cublasLtMatmulHeuristicResult_t heur = {};
    int found = 0;
    p->op = nullptr;
    p->la = p->lb = p->lc = nullptr;
    cublasStatus_t st = cublasLtMatmulDescCreate(&p->op, CUBLAS_COMPUTE_32F, CUDA_R_32F);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasLtMatmulDescSetAttribute(p->op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb);
    if (st == CUBLAS_STATUS_SUCCESS) st = cublasLtMatrixLayoutCreate(&p->la, CUDA_R_16BF, p->K, p->N, p->K);
    if (st == CUBLAS_STATUS_SUCCESS) st = cublasLtMatrixLayoutCreate(&p->lb, CUDA_R_16BF, p->K, p->M, p->K);
    if (st == CUBLAS_STATUS_SUCCESS) st = cublasLtMatrixLayoutCreate(&p->lc, p->ctype, p->N, p->M, p->N);
    if (st == CUBLAS_STATUS_SUCCESS) st = cublasLtMatmulPreferenceCreate(&pref);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                  &p->ws_bytes, sizeof p->ws_bytes);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasLtMatmulAlgoGetHeuristic(h, p->op, p->la, p->lb, p->lc, p->lc, pref, 1, &heur, &found);
    if (st == CUBLAS_STATUS_SUCCESS && found == 0) st = CUBLAS_STATUS_NOT_SUPPORTED;
    if (st == CUBLAS_STATUS_SUCCESS) p->algo = heur.algo;
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (st != CUBLAS_STATUS_SUCCESS) {
        if (p->lc) cublasLtMatrixLayoutDestroy(p->lc);
        if (p->lb) cublasLtMatrixLayoutDestroy(p->lb);
        if (p->la) cublasLtMatrixLayoutDestroy(p->la);
        if (p->op) cublasLtMatmulDescDestroy(p->op);
    }
    return st;
}

// C[M,N] (row-major) = A[M,K] (row-major) . B[N,K]^T (row-major), bf16 inputs,
// fp32 accumulation, C of type ctype (bf16 or fp32). In cuBLASLt's
// column-major terms: C^T [N,M] = op_T(B as [K,N]) . (A as [K,M]).
cublasStatus_t gemm_tn(const void* A, const void* B, void* C, cudaDataType_t ctype, int M, int N,
                       int K, void* ws, size_t ws_bytes, cudaStream_t stream) {
    cublasStatus_t st = CUBLAS_STATUS_SUCCESS;
    cublasLtHandle_t h = lt_handle(&st);
    if (st != CUBLAS_STATUS_SUCCESS) return st;
    static std::mutex mu;
    static std::vector<GemmPlan> plans;
    GemmPlan plan{};
    bool cached = false;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const GemmPlan& p : plans)
            if (p.M == M && p.N == N && p.K == K && p.ctype == ctype && p.ws_bytes == ws_bytes) {
                plan = p;
                cached = true;
                break;
            }
        if (!cached) {
            plan = GemmPlan{M, N, K, ctype, ws_bytes, nullptr, nullptr, nullptr, nullptr, {}};
            st = make_plan(h, &plan);
            if (st != CUBLAS_STATUS_SUCCESS) return st;
            if (plans.size() < 256) {   // beyond that many shapes, plans are built per call
                plans.push_back(plan);
                cached = true;
            }
        }
    }
    const float alpha = 1.f, beta = 0.f;
    st = cublasLtMatmul(h, plan.op, &alpha, B, plan.la, A, plan.lb, &beta, C, plan.lc, C, plan.lc,
                        &plan.algo, ws, ws_bytes, stream);
    if (!cached) {
        cublasLtMatrixLayoutDestroy(plan.lc);
        cublasLtMatrixLayoutDestroy(plan.lb);
        cublasLtMatrixLayoutDestroy(plan.la);
        cublasLtMatmulDescDestroy(plan.op);
    }
    return st;
}

constexpr size_t kGemmWorkspace = size_t(32) << 20;   // cuBLASLt's share of the workspace

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
    const size_t t = T > 0 ? (size_t)T : 0;
    return align_up(t * IDX_DIM * sizeof(uint16_t), 256) + kGemmWorkspace;
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
    uint16_t* k_pre = static_cast<uint16_t*>(ws);
    void* gws = static_cast<char*>(ws) + align_up((size_t)T * IDX_DIM * sizeof(uint16_t), 256);
    cublasStatus_t st = gemm_tn(q_lora, w_q, q, CUDA_R_16BF, T, IDX_HEADS * IDX_DIM, q_rank, gws,
                                kGemmWorkspace, s);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = gemm_tn(x, w_k, k_pre, CUDA_R_16BF, T, IDX_DIM, hidden, gws, kGemmWorkspace, s);
    if (st == CUBLAS_STATUS_SUCCESS)
        st = gemm_tn(x, w_w, w, CUDA_R_32F, T, IDX_HEADS, hidden, gws, kGemmWorkspace, s);
    if (st != CUBLAS_STATUS_SUCCESS) return proj_fail(IDX_ERR_CUDA, "cuBLASLt matmul failed");
    cudaError_t e = launch_key_layernorm(k_pre, ln_w, ln_b, ln_dtype == IDX_PARAM_F32, eps, k_cache, T,
                                         s, slot, cache_rows);
    if (e != cudaSuccess) return proj_fail(IDX_ERR_CUDA, cudaGetErrorString(e));
    return IDX_OK;
}

}  // extern "C"

/*
 * lightning_indexer.h — C ABI of the GB300 (sm_103a) Lightning Indexer library.
 *
 * The Lightning Indexer is described in the Hugging Face discussion "Notes from
 * an NVFP4 port of Kimi K3.1 Pro" (moonshotai/Kimi-K3.1-Pro, discussion 7):
 *   - the indexer paragraph: each query has 32 heads of width 128; every key of
 *     its causal past gets relu(q_h . k) per head, the heads are combined with
 *     a per-head weight vector, and the 2048 highest-scoring positions are kept
 *     with no approximation; keys are normalised by a 128-wide LayerNorm that
 *     has a weight and a bias;
 *   - list "Details that silently change the answer", item (3): the indexer
 *     uses no rotary embedding (index_rope_dim = 0); item (4): the output
 *     order and the tie rule at the top-K boundary;
 *   - the closing paragraph: when a query's history holds no more than 2048
 *     keys, nothing is dropped and every position is kept.
 *
 * Conventions shared by every entry point
 *   Memory     All data pointers are DEVICE pointers to caller-owned memory on the
 *              current CUDA device. The library never allocates device memory,
 *              never frees, and never synchronises: all work is enqueued on
 *              `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *              stream) and completes asynchronously.
 *   bf16       bfloat16 tensors are arrays of uint16_t bit patterns.
 *   Layout     Row-major, contiguous, with 16-byte aligned base pointers.
 *   Batches    A packed ragged batch of B sequences: sequence b owns query rows
 *              cu_q[b] .. cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1 (both
 *              int32 [B+1], non-decreasing, cu_q[0] = cu_k[0] = 0, cu_q[B] = T).
 *              q_pos[t] is query t's position inside its sequence; the query
 *              sees keys 0 .. q_pos[t] (its causal length is n(t) = q_pos[t]+1,
 *              which must not exceed the sequence's key count).
 *              Output positions are sequence-local (0-based within the sequence).
 *   Errors     Arguments are checked on the host before anything is enqueued; a
 *              failed check returns a non-zero idx_status and enqueues nothing.
 *              Values that live on the device (cu_q, cu_k, q_pos, n_valid) are
 *              checked by the kernels, which skip the offending row and record
 *              IDX_ERR_DEVICE_ARG in the workspace's status word; read it with
 *              idx_get_status. A CUDA launch failure returns IDX_ERR_CUDA.
 *              idx_last_error() gives a message for the calling thread's last
 *              failure.
 *   Workspace  ws / ws_bytes: caller-owned device scratch, at least the size the
 *              matching *_workspace_size function returns, 256-byte aligned. It
 *              holds the status word, the tile plan and staged scores. Calls that
 *              may overlap on the GPU need separate workspaces. For arguments
 *              that the call itself rejects (B < 1, T < 0, max_len < 1) the size
 *              functions return the 256-byte header size.
 */
#ifndef LIGHTNING_INDEXER_H
#define LIGHTNING_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IDX_API __attribute__((visibility("default")))
#else
#define IDX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IDX_OK = 0,
    IDX_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad alignment, topk out of range */
    IDX_ERR_UNSUPPORTED = 2,  /* the current device is not an sm_103 (GB300) GPU */
    IDX_ERR_WORKSPACE = 3,    /* ws_bytes below the required size, or ws misaligned */
    IDX_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (text in idx_last_error) */
    IDX_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (status word) */
    IDX_ERR_DEVICE_ARG = 6    /* a device-resident argument was out of range (status word) */
} idx_status;

enum {
    IDX_HEADS = 32,      /* indexer heads */
    IDX_DIM = 128,       /* head dimension = key width = LayerNorm width */
    IDX_TOPK_MAX = 2048  /* positions kept per query */
};

enum { IDX_PARAM_BF16 = 0, IDX_PARAM_F32 = 1 };

/*
 * Key LayerNorm (indexer paragraph: indexer keys pass a 128-wide LayerNorm
 * with a weight and a bias). For every row x of k_raw:
 *     y = (x - mean(x)) / sqrt(var(x) + eps) * ln_w + ln_b
 * with the biased variance, computed in fp32 and rounded to bf16
 * (nearest-even) into k_out. Runs once per key when the indexer's key cache is
 * filled; the scoring entry points take its output.
 *   k_raw   bf16 [n_rows,128]        k_out  bf16 [n_rows,128] (may equal k_raw)
 *   ln_w, ln_b  [128], bf16 (ln_dtype = IDX_PARAM_BF16) or fp32 (IDX_PARAM_F32)
 *   n_rows  >= 0 (0 enqueues nothing)
 */
IDX_API idx_status idx_key_layernorm(const uint16_t* k_raw, const void* ln_w, const void* ln_b,
                             int ln_dtype, float eps, uint16_t* k_out, int64_t n_rows,
                             void* stream);

/*
 * Key LayerNorm fused into the key-cache append: the same LayerNorm as
 * idx_key_layernorm (bit-identical results), each output row written
 * straight into its slot of the key cache instead of a staging buffer
 * (port notes, indexer paragraph: new keys pass the LayerNorm before they
 * are cached; "Kimi K3 on AMD Instinct GPUs with TokenSpeed", section 2.2
 * "Fused cache writes and output processing": the cache rows are prepared,
 * normalisation included, by one kernel rather than several small ones).
 *   k_raw      bf16 [n_rows,128], new raw keys (must not overlap the cache
 *              rows being written)
 *   ln_w, ln_b [128], bf16 or fp32 as ln_dtype
 *   k_cache    bf16 [cache_rows,128]; row slot[r] receives LN(k_raw[r])
 *   slot       int64 [n_rows], device memory: destination row of each new
 *              key, distinct among the rows written; -1 marks a padding row.
 *              Any slot outside [0, cache_rows) writes nothing (no error).
 *   n_rows     >= 0 (0 enqueues nothing)
 * Rows of k_cache that no slot names are left untouched. Asynchronous on
 * `stream`; allocates nothing.
 */
IDX_API idx_status idx_key_layernorm_append(const uint16_t* k_raw, const void* ln_w,
                                            const void* ln_b, int ln_dtype, float eps,
                                            uint16_t* k_cache, int64_t cache_rows,
                                            const int64_t* slot, int64_t n_rows, void* stream);

/*
 * Indexer projections from the layer's activations (port notes, indexer
 * paragraph: the query comes off the normalised q-LoRA projection, the key
 * from the attention input through the key LayerNorm, and a per-head weight
 * vector sums the heads). Per token t (weights in the [out, in] layout of a
 * linear layer; bf16 products accumulated in fp32):
 *   q[t]             = W_q . q_lora[t]   W_q [32*128, q_rank]  -> q bf16 [T,32,128]
 *   k_pre[t]         = W_k . x[t]        W_k [128, hidden]     -> bf16 (workspace)
 *   k_cache[slot[t]] = LayerNorm(k_pre[t]) as idx_key_layernorm_append
 *   w[t]             = W_w . x[t]        W_w [32, hidden]      -> w fp32 [T,32]
 * Any scale of the per-head weights is part of W_w. The products run on the
 * library's own tensor-core GEMM (the key and weight products in one pass over
 * x); with few tokens K is split over the SMs and the fp32 partial sums are
 * added by a second kernel, which for the key also rounds k_pre to bf16 and
 * appends its LayerNorm to the cache (bit-identical to
 * idx_key_layernorm_append). ws: 256-byte aligned, at least
 * idx_indexer_project_workspace_size(T) bytes (a size that depends on the
 * current device's SM count); it holds the status word (idx_get_status reads
 * it: IDX_ERR_TIMEOUT if a bounded wait of the GEMM gave up) and the partial
 * sums. The library allocates nothing. x [T,hidden] and q_lora
 * [T,q_rank] are bf16 row-major; hidden and q_rank are multiples of 8;
 * matrices 16-byte aligned. slot and the LayerNorm parameters are as for
 * idx_key_layernorm_append.
 */
IDX_API size_t idx_indexer_project_workspace_size(int32_t T);
IDX_API idx_status idx_indexer_project(const uint16_t* x, const uint16_t* q_lora,
                                       const uint16_t* w_q, const uint16_t* w_k,
                                       const uint16_t* w_w, const void* ln_w, const void* ln_b,
                                       int ln_dtype, float eps, int32_t T, int32_t hidden,
                                       int32_t q_rank, uint16_t* q, uint16_t* k_cache,
                                       int64_t cache_rows, const int64_t* slot, float* w, void* ws,
                                       size_t ws_bytes, void* stream);

/*
 * Head scores (indexer paragraph: per-head relu of q_h . k over the causal
 * past, combined with a per-head weight; item (3): no rotary):
 *     scores[t*ld + s] = sum_h w[t,h] * max(sum_d q[t,h,d] * k[cu_k[b]+s, d], 0)
 * for every query t (of sequence b) and every s < n(t), bf16 products with
 * fp32 accumulation. Entries s >= n(t) of a row are left untouched.
 *   q      bf16 [T,32,128]     k  bf16 [n_keys,128] (post-LayerNorm key cache)
 *   w      fp32 [T,32]         q_pos, cu_q, cu_k: int32 (see Batches)
 *   n_keys rows of k (>= cu_k[B]); bounds every key read
 *   max_len  an upper bound on n(t) over the batch (host value, >= 1)
 *   scores fp32 [T,ld], ld >= max_len and a multiple of 4
 */
IDX_API idx_status idx_score(const uint16_t* q, const uint16_t* k, const float* w,
                     const int32_t* q_pos, const int32_t* cu_q, const int32_t* cu_k,
                     int32_t B, int32_t T, int64_t n_keys, int64_t max_len, float* scores,
                     int64_t ld,
                     void* ws, size_t ws_bytes, void* stream);
IDX_API size_t idx_score_workspace_size(int32_t B, int32_t T, int64_t max_len);

/*
 * Exact top-K of score rows under the order rule (indexer paragraph: the
 * selection is exact; item (4): scores equal to the threshold at the K
 * boundary form a tie group; the output first lists the kept positions whose
 * score exceeds the threshold, by increasing position, then the kept members
 * of the tie group, also by increasing position, the group being cut from its
 * low-position end; it is not sorted by score; closing paragraph: a history of
 * K or fewer keys keeps every position, in increasing order).
 * Threshold: tau is the K-th score in (score descending, position ascending)
 * order; -0.0 and +0.0 compare equal. Scores must be finite.
 *   scores  fp32 [T,ld] (row t holds n_valid[t] scores)
 *   n_valid int32 [T], 0 <= n_valid[t] <= min(ld, max_len)
 *   topk    1 .. 2048
 *   idx     int32 [T,topk]: the kept positions, then -1 padding
 *   cnt     int32 [T] number kept (= min(n_valid, topk)), or NULL
 */
IDX_API idx_status idx_topk(const float* scores, int64_t ld, const int32_t* n_valid, int32_t T,
                    int64_t max_len, int32_t topk, int32_t* idx, int32_t* cnt,
                    void* ws, size_t ws_bytes, void* stream);
IDX_API size_t idx_topk_workspace_size(int32_t T, int64_t max_len, int32_t topk);

/*
 * The whole indexer in one call: idx_score followed by idx_topk with
 * n_valid[t] = q_pos[t] + 1, staging the fp32 scores inside the workspace.
 * Arguments as for idx_score and idx_topk. When a bounded wait inside the
 * scorer gives up (IDX_ERR_TIMEOUT in the status word) no row is selected
 * from the incomplete scores: every row gets idx -1 and cnt 0.
 */
IDX_API idx_status idx_score_topk(const uint16_t* q, const uint16_t* k, const float* w,
                          const int32_t* q_pos, const int32_t* cu_q, const int32_t* cu_k,
                          int32_t B, int32_t T, int64_t n_keys, int64_t max_len, int32_t topk,
                          int32_t* idx,
                          int32_t* cnt, void* ws, size_t ws_bytes, void* stream);
IDX_API size_t idx_score_topk_workspace_size(int32_t B, int32_t T, int64_t max_len, int32_t topk);

/*
 * idx_score_topk without a workspace argument. The port notes have no
 * counterpart: this entry point exists for callers that cannot give the
 * library any extra device memory — an engine that plans all of its device
 * memory ahead and bans cudaMalloc while serving (it may synchronise the device
 * and may fail under memory pressure), or a plugin that its host framework
 * hands only input and output buffers. Same arguments and results as
 * idx_score_topk, minus ws/ws_bytes; it allocates nothing.
 *   Scratch   a fixed 39 MiB (+256 B) array inside the library's device image,
 *             reserved on every GPU that loads the library until process exit.
 *   Limit     T * round_up(max_len, 4) * 4 <= 32 MiB (e.g. 64 queries of up to
 *             131,072 keys), T + B <= 40,000, and at most 6 MiB of selection
 *             scratch (histograms and bitmaps of batches of up to 128
 *             queries with long histories); larger calls return
 *             IDX_ERR_WORKSPACE, enqueue nothing, and idx_last_error() says why.
 *   Sharing   every call on a device uses the same array, which keeps the last
 *             call's contents; calls that can overlap on the GPU (other streams,
 *             unordered host threads) race on it and must be serialised.
 *   Set-up    the first call on each device looks up the array's device address
 *             (cudaGetSymbolAddress, with that device current); make that first
 *             call before any stream capture. The address is kept per device and
 *             CUDA context, so the first call in a new context of a device
 *             (after cudaDeviceReset, say) looks it up again.
 *   Errors    host checks as idx_score_topk. There is no status word to read: a
 *             row skipped for a device-side argument error shows cnt[t] == 0 and
 *             idx -1, and when a bounded wait inside the scorer gives up (the
 *             workspace entry point's IDX_ERR_TIMEOUT) every row of the call is
 *             written that way. A valid row keeps at least one position, so
 *             cnt[t] == 0 always marks a failed row.
 */
IDX_API idx_status idx_score_topk_noalloc(const uint16_t* q, const uint16_t* k, const float* w,
                                          const int32_t* q_pos, const int32_t* cu_q,
                                          const int32_t* cu_k, int32_t B, int32_t T,
                                          int64_t n_keys, int64_t max_len, int32_t topk,
                                          int32_t* idx,
                                          int32_t* cnt, void* stream);

/*
 * Sparse NoPE MLA attention over the selected positions (decode; the step that
 * consumes the indexer's output). The port notes (opening paragraph and item
 * (5)) say the indexer keeps the best 2048 keys for each full-attention layer
 * and that those layers are NoPE multi-head latent attention; the TokenSpeed
 * post on Kimi K3 (section 2, MLA) gives the cache row (a shared 512-wide
 * latent and a 64-wide key part per token), 96 heads, and decode's query moved
 * into the compressed space. For query row t of sequence b and head h, with
 * S_t = idx[t, 0 .. cnt[t]) (sequence-local positions, as idx_score_topk
 * writes them) and c_s = cache row cu_k[b] + s:
 *   l_s  = scale * (q[t,h,:] . c_s)   over the 576 dims, s in S_t
 *   out[t,h,:] = sum_s softmax(l)_s * c_s[0..512)      (fp32 [T,heads,512])
 *   lse[t,h]   = log sum_s exp(l_s)                   (fp32 [T,heads], natural log)
 * An empty selection gives out = 0 and lse = -infinity. Arguments:
 *   q        bf16 [T, heads, 576], the absorbed queries
 *   cache    bf16 [cache_rows, 576], rows packed by sequence as cu_k says
 *   idx      int32 [T, topk]; cnt int32 [T] (0 .. topk) valid entries per row
 *   heads    32, 64 or 96;  topk 1 .. 2048;  scale > 0 and finite
 * A position outside its sequence is left out of the softmax and reported as
 * IDX_ERR_DEVICE_ARG in the status word. Queries are split over key ranges
 * when T is small (partial results in the workspace, merged by a second
 * kernel); ws is 256-byte aligned and holds idx_sparse_mla_workspace_size(T,
 * heads, topk) bytes, a size that depends on the current device's SM count.
 * q and cache are 16-byte aligned. Asynchronous on `stream`; allocates nothing.
 */
IDX_API size_t idx_sparse_mla_workspace_size(int32_t T, int32_t heads, int32_t topk);
IDX_API idx_status idx_sparse_mla(const uint16_t* q, const uint16_t* cache, int64_t cache_rows,
                                  const int32_t* idx, const int32_t* cnt, const int32_t* cu_q,
                                  const int32_t* cu_k, int32_t B, int32_t T, int32_t heads,
                                  int32_t topk, float scale, float* out, float* lse, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * idx_sparse_mla over an FP8 cache. The TokenSpeed post on Kimi K3 (section 2,
 * MLA, and the TL;DR's precision list) keeps the MLA cache in FP8; here a
 * cache row is 576 E4M3 codes (OCP FP8: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, subnormals, one NaN code per sign, no infinities) and one
 * fp32 scale, and stands for the row
 *   c_s[d] = row_scale[s] * e4m3(cache8[s, d]).
 * The result is that of idx_sparse_mla on these rows. Arguments as there, but:
 *   cache8     uint8 [cache_rows, 576], 16-byte aligned (rows packed by
 *              sequence as cu_k says); codes 0x7F and 0xFF (NaN) make the row's
 *              contributions NaN
 *   row_scale  fp32 [cache_rows], finite, 4-byte aligned
 * The workspace is idx_sparse_mla_workspace_size(T, heads, topk) bytes.
 * Asynchronous on `stream`; allocates nothing.
 */
IDX_API idx_status idx_sparse_mla_fp8(const uint16_t* q, const uint8_t* cache8, const float* row_scale,
                                      int64_t cache_rows, const int32_t* idx, const int32_t* cnt,
                                      const int32_t* cu_q, const int32_t* cu_k, int32_t B, int32_t T,
                                      int32_t heads, int32_t topk, float scale, float* out, float* lse,
                                      void* ws, size_t ws_bytes, void* stream);

/*
 * Device status word of a workspace, written by the kernels of the last call
 * that used it: IDX_OK, IDX_ERR_DEVICE_ARG or IDX_ERR_TIMEOUT. Synchronises
 * `stream` (a blocking read of 8 bytes). *detail (may be NULL) receives the
 * first offending row or a wait-site code.
 */
IDX_API idx_status idx_get_status(const void* ws, void* stream, int32_t* detail);

/* Message for the calling thread's last failed call ("" if none). */
IDX_API const char* idx_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
IDX_API int32_t idx_version(void);

/*
 * Number of CUDA kernels this library has enqueued in this process (all
 * devices, all threads), for launch accounting in benchmarks. Memsets are not
 * counted.
 */
IDX_API uint64_t idx_kernel_launches(void);

/*
 * Test hook for failure detection: sets the bound, in nanoseconds, of every
 * wait inside the tensor-core kernels (the scorer, the projection GEMM and the sparse MLA
 * attention; default 2,000,000,000) for launches enqueued from now on, and
 * returns the previous bound. When a wait runs out
 * the kernel records IDX_ERR_TIMEOUT in the status word, stops all its roles,
 * lets copies and tensor-core work already issued finish (within 100 ms),
 * frees its tensor memory and returns, leaving the CUDA context usable. The
 * selection kernels of the same fused call then select nothing from the
 * partly written scores: every row gets idx -1 and cnt 0. A bound of 0 makes
 * the first wait that is not already satisfied give up.
 */
IDX_API uint64_t idx_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Measurement hook (no counterpart in the port notes): arms n CUDA events
 * (cudaEvent_t handles passed as void*, created by the caller, n <= 16) for
 * the calling thread. The next n kernels that any entry point enqueues from
 * this thread each get events[i] recorded on their stream right after the
 * i-th of them, so that a benchmark can time every kernel of one real fused
 * call (event i-1 to event i). A recorded event sits between two kernels
 * that would otherwise overlap their start-up (programmatic dependent
 * launch), so the per-kernel times add up to a little more than the call
 * alone. n = 0 disarms. Returns n, or -1 for n outside [0, 16] or NULL
 * events (message in idx_last_error). The events are not owned.
 */
IDX_API int32_t idx_set_kernel_events(void* const* events, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* LIGHTNING_INDEXER_H */

/*
 * maxsim.h -- C ABI of libmaxsim.so, late-interaction MaxSim scoring on
 * NVIDIA GB300 (sm_103a).
 *
 * The operator ("TileMaxSim: IO-Aware GPU MaxSim Scoring with Dimension
 * Tiling and Fused Product Quantization", §1; "FLASH-MAXSIM: IO-Aware Fused
 * Kernels for Late-Interaction Scoring", Abstract):
 *
 *     score(Q, D_b) = sum_{i < nq} max_{j < L_b} <q_i, d_j>
 *
 * for a query Q of nq token embeddings and a document D_b of L_b token
 * embeddings, all of dimension d. Inputs are taken as given: the library
 * does not normalise them (the "cosine" of the pages is the dot product of
 * L2-normalised embeddings).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, row-major
 *    and contiguous. The library allocates and frees no device memory;
 *    where an operation needs scratch space the caller passes a workspace
 *    sized by the matching *_workspace_size() query.
 *  - Element pointers must be 16-byte aligned (TMA and vector loads).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every call is asynchronous on that stream and returns as soon
 *    as its kernels are enqueued; outputs are valid once the stream reaches
 *    that point.
 *  - Errors: argument problems found on the host return
 *    MAXSIM_ERR_INVALID_ARG or MAXSIM_ERR_UNSUPPORTED before anything is
 *    launched. A failed launch returns MAXSIM_ERR_CUDA. Problems found on
 *    the device (inconsistent CSR offsets or lengths, a pipeline wait that
 *    gave up) cannot be returned by the asynchronous call; the kernel
 *    records them in a per-device status word, treats a bad document as
 *    empty, and maxsim_device_status() reports them. No kernel traps, asserts
 *    or spins without a bound. No C++ exception crosses this ABI.
 *  - Outputs are fp32 (scores, gradients) or int32 (indices). An empty
 *    document (L_b = 0) scores 0.0 and has argmax -1.
 *  - The argmax of query token i in document b is the LOWEST doc-local token
 *    index j attaining the maximum similarity.
 *  - Per-device state: on its first call on a device the library looks up
 *    the device addresses of its own global variables (the status word, the
 *    table of maxsim_score_pq_noalloc) and keeps them for the life of the
 *    process. cudaDeviceReset() invalidates them: do not reset a device
 *    between calls into this library.
 */
#ifndef MAXSIM_H_
#define MAXSIM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum maxsim_status {
    MAXSIM_OK = 0,
    MAXSIM_ERR_INVALID_ARG = 1,  /* NULL/misaligned pointer, negative size, bad lengths/offsets */
    MAXSIM_ERR_UNSUPPORTED = 2,  /* valid arguments the library does not handle (e.g. d % 64 != 0 on the tensor-core path) */
    MAXSIM_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    MAXSIM_ERR_TIMEOUT = 4,      /* a device pipeline wait gave up after its time bound */
    MAXSIM_ERR_WORKSPACE = 5     /* workspace NULL or smaller than the size query returned */
} maxsim_status;

typedef enum maxsim_dtype {
    MAXSIM_BF16 = 0,   /* bf16 in, fp32 accumulate (tcgen05 tensor cores) */
    MAXSIM_FP16 = 1,   /* fp16 in, fp32 accumulate (tcgen05 tensor cores) */
    MAXSIM_FP32 = 2    /* fp32 in, fp32 FFMA on the CUDA cores */
} maxsim_dtype;

/* Bits of the device status word (see maxsim_device_status). */
#define MAXSIM_DEVERR_TIMEOUT    0x1u  /* a pipeline wait exceeded its time bound */
#define MAXSIM_DEVERR_BAD_INPUT  0x2u  /* a document's offsets/length were out of range */

/*
 * maxsim_debug_set_faults -- TEST-ONLY switches of the failure-detection
 * path; not part of the operator, never needed in normal use. Applies to the
 * current device, to every kernel launched after the call returns (the call
 * is synchronous).
 *   flags          MAXSIM_DEBUG_STALL_FWD_LOADER: the loader role of the
 *                  tensor-core forward kernel (maxsim_score / _varlen with
 *                  bf16 or fp16 and queries below 256 tokens) issues no copy,
 *                  so the kernel's other roles wait on barriers nothing will
 *                  complete; their bounded waits run out, record
 *                  MAXSIM_DEVERR_TIMEOUT and the kernel exits with no copy or
 *                  MMA in flight (its outputs are then undefined). 0 = off.
 *   wait_limit_ns  bound of every pipeline wait; 0 restores the default (2 s).
 * Call maxsim_debug_set_faults(0, 0) to return to normal operation. Unknown
 * flag bits return MAXSIM_ERR_INVALID_ARG; a failed copy MAXSIM_ERR_CUDA.
 */
#define MAXSIM_DEBUG_STALL_FWD_LOADER 0x1u
maxsim_status maxsim_debug_set_faults(unsigned int flags, uint64_t wait_limit_ns);

/* Library version: major*10000 + minor*100 + patch. */
int maxsim_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *maxsim_status_string(maxsim_status status);

/*
 * maxsim_device_status -- synchronises `stream`, then reads and clears the
 * status word of the current device. *flags (may be NULL) receives the
 * MAXSIM_DEVERR_* bits seen since the last call. Returns MAXSIM_ERR_TIMEOUT
 * if the timeout bit was set, else MAXSIM_ERR_INVALID_ARG if the bad-input
 * bit was set, else MAXSIM_OK (or MAXSIM_ERR_CUDA if the stream failed).
 */
maxsim_status maxsim_device_status(void *stream, unsigned int *flags);

/*
 * maxsim_score -- padded layout, one or more queries.
 *
 * Follows TileMaxSim §1 (operator), §2(1) (every document byte streamed
 * from HBM once, the per-query-token maximum kept on chip), §2(2)
 * (dimension tiling: partial dot products over d-chunks are summed before
 * the maximum) and §5 (fixed-Nd padding with a length mask); FLASH-MAXSIM
 * Figure 1 / Algorithm 2 (running maximum from -inf, only the scalar score
 * written back).
 *
 *   Q          [n_queries, nq, d]  dtype
 *   D          [B, nd, d]          dtype; document b's tokens are rows
 *                                  0 .. L_b-1 of D[b]; rows L_b .. nd-1 are
 *                                  never read by the tensor-core path beyond
 *                                  a 32-row granule and never contribute
 *   doc_len    [B] int32 or NULL   L_b (0 <= L_b <= nd); NULL means L_b = nd
 *   out        [n_queries, B] fp32 out[q*B + b] = score(Q[q], D_b)
 *   argmax_out [n_queries, B, nq] int32 or NULL
 *
 * Limits: nq >= 1, n_queries >= 1, nd >= 1, B >= 0 (B = 0 is a no-op).
 * BF16/FP16: d % 64 == 0 and 64 <= d <= 1024. FP32: d % 4 == 0, d <= 1024.
 */
maxsim_status maxsim_score(const void *Q, int n_queries, int nq, int d,
                           const void *D, int64_t B, int nd, const int32_t *doc_len,
                           maxsim_dtype dtype, float *out, int32_t *argmax_out,
                           void *stream);

/*
 * maxsim_length_order -- length-bucketed document order (TileMaxSim §5:
 * fixed-Nd padding wastes token compute on variable-length corpora, and
 * batching documents of similar length recovers the throughput). Writes the
 * permutation order_out[B] that sorts the documents by their number of 8-row
 * granules, ceil(L_b / 8), ascending and stably (equal keys keep index
 * order). It depends only on the lengths: compute it once per corpus and
 * pass it to maxsim_score_ordered for every query.
 *   doc_len    [B] int32, 0 <= L_b <= nd (padded layout), or
 *   offsets    [B+1] int64 (CSR layout; nd ignored, lengths above 8176
 *              tokens share the last bucket) -- exactly one of the two, or
 *              neither (every document has nd tokens: the identity order)
 *   workspace  >= maxsim_length_order_workspace_size(B, nd, csr) bytes,
 *              16-byte aligned (per-warp bucket counts)
 * A length outside [0, nd] (or a decreasing offset) counts as 0 and sets
 * MAXSIM_DEVERR_BAD_INPUT. B <= INT32_MAX.
 */
size_t maxsim_length_order_workspace_size(int64_t B, int nd, int csr);
maxsim_status maxsim_length_order(const int32_t *doc_len, const int64_t *offsets, int64_t B, int nd,
                                  int32_t *order_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * maxsim_score_ordered -- maxsim_score with the documents walked in the order
 * doc_order (a permutation of [0, B), e.g. from maxsim_length_order), so each
 * thread block scores documents of similar length. Results are written at
 * the documents' own indices and are identical to maxsim_score's: a
 * document's result depends only on its own rows. An entry outside [0, B)
 * is skipped and sets MAXSIM_DEVERR_BAD_INPUT; duplicates leave the missing
 * documents' outputs unwritten. Same arguments and limits as maxsim_score,
 * bf16/fp16 only, and queries shorter than 256 tokens (longer ones, and fp32,
 * return MAXSIM_ERR_UNSUPPORTED).
 */
maxsim_status maxsim_score_ordered(const void *Q, int n_queries, int nq, int d,
                                   const void *D, int64_t B, int nd, const int32_t *doc_len,
                                   const int32_t *doc_order, maxsim_dtype dtype, float *out,
                                   int32_t *argmax_out, void *stream);

/*
 * maxsim_score_varlen -- variable-length, padding-free documents in CSR
 * form (FLASH-MAXSIM, Abstract: variable-length padding-free scoring;
 * TileMaxSim §5: the padding waste it removes).
 *
 *   D_packed   [total_tokens, d] dtype; document b owns rows
 *              offsets[b] .. offsets[b+1]-1
 *   offsets    [B+1] int64, offsets[0] = 0, non-decreasing,
 *              offsets[B] = total_tokens (checked on the device: a document
 *              whose range falls outside [0, total_tokens] is scored as
 *              empty and sets MAXSIM_DEVERR_BAD_INPUT)
 *   out        [n_queries, B] fp32; argmax_out [n_queries, B, nq] int32 or NULL
 *
 * Same dtype and d limits as maxsim_score.
 */
maxsim_status maxsim_score_varlen(const void *Q, int n_queries, int nq, int d,
                                  const void *D_packed, const int64_t *offsets,
                                  int64_t B, int64_t total_tokens,
                                  maxsim_dtype dtype, float *out, int32_t *argmax_out,
                                  void *stream);

/*
 * maxsim_score_pq -- fused product-quantisation scoring (TileMaxSim §2(3)):
 * the per-query table T[i,m,k] = q_i[m*(d/M) .. (m+1)*(d/M)) . C[m,k,:] is
 * built once into the workspace, then each token's similarity is
 * sum_m T[i, m, codes[j,m]] by table lookup; decoded vectors never exist.
 *
 *   Q          [nq, d] fp32
 *   codebooks  [M, K, d/M] fp32 (d % M == 0, K <= 256)
 *   codes      [total_tokens, M] uint8, CSR documents as in maxsim_score_varlen
 *   out        [B] fp32; argmax_out [B, nq] int32 or NULL
 *   workspace  >= maxsim_score_pq_workspace_size(nq, M, K) bytes, 16-byte
 *              aligned; holds the table (groups of 8 query tokens, fp32);
 *              contents on entry are ignored, the call overwrites it.
 *
 * Limits: 1 <= nq <= 1024; M % 4 == 0, 4 <= M <= 64; 1 <= K <= 256;
 * d % M == 0, d <= 1024; one 8-token table group (M * K * 32 bytes) plus
 * 64 KB of code staging must fit in shared memory (M * K <= 5056), else
 * MAXSIM_ERR_UNSUPPORTED. A code >= K is clamped to K-1 and sets
 * MAXSIM_DEVERR_BAD_INPUT. Missing or short workspace: MAXSIM_ERR_WORKSPACE.
 */
size_t maxsim_score_pq_workspace_size(int nq, int M, int K);
maxsim_status maxsim_score_pq(const float *Q, int nq, int d,
                              const float *codebooks, int M, int K,
                              const uint8_t *codes, const int64_t *offsets,
                              int64_t B, int64_t total_tokens,
                              float *out, int32_t *argmax_out,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * maxsim_score_pq_noalloc -- maxsim_score_pq for callers that cannot
 * allocate device memory. The source pages have no counterpart: this is a
 * library convenience, not part of the method.
 *
 * Some callers have no way to hand over a workspace: code that runs where a
 * device allocation is forbidden or unavailable (a host callback, a hook
 * inside another library, a plugin without an allocator). This variant keeps
 * the PQ table in a fixed 1 MiB device array compiled into the library
 * (present on every GPU that loads it, until the process exits) and
 * allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *
 *   Arguments, layouts, results and other limits: as maxsim_score_pq,
 *   without the workspace.
 *   Limit: the table, ceil(nq/8)*8 * M * K * 4 bytes, must fit in 1 MiB
 *   (e.g. nq <= 64 at M = 16, K = 256); larger requests return
 *   MAXSIM_ERR_WORKSPACE before anything is launched.
 *   Set-up: the first call on each device looks up the array's device
 *   address with that device current; make that first call before any
 *   stream capture. A failed lookup returns MAXSIM_ERR_CUDA. The address is
 *   kept until the process exits, so the device must not be reset
 *   (cudaDeviceReset) between calls.
 *   Sharing: every call uses the same array, and it keeps the previous
 *   call's table. Each call rewrites every entry it reads, so no clearing is
 *   needed; but calls whose kernels overlap on the GPU (for example on two
 *   streams) race on the array and give wrong results -- serialise them.
 */
maxsim_status maxsim_score_pq_noalloc(const float *Q, int nq, int d,
                                      const float *codebooks, int M, int K,
                                      const uint8_t *codes, const int64_t *offsets,
                                      int64_t B, int64_t total_tokens,
                                      float *out, int32_t *argmax_out, void *stream);

/*
 * maxsim_score_streamed -- maxsim_score for documents that stay in host
 * memory, e.g. a corpus larger than GPU memory (TileMaxSim deep reading §5
 * names it as an open limitation). Same operator and outputs as
 * maxsim_score; per-document results are identical to scoring the same
 * documents from device memory.
 *   Q            device [n_queries, nq, d] (as maxsim_score)
 *   D_host       HOST [B, nd, d] in dtype; page-locked memory (cudaHostAlloc /
 *                torch pin_memory) lets copies overlap scoring, pageable
 *                memory works but serialises each copy
 *   doc_len_host HOST int32 [B] or NULL (as doc_len of maxsim_score)
 *   out, argmax_out  device, as maxsim_score
 *   workspace    device, 16-byte aligned, >= the size returned below
 *   chunk_docs   documents per chunk (>= 1); two chunks of device buffers
 *                alternate: the copy of chunk k + 1 (on a library-owned
 *                copy stream) runs while chunk k is scored on `stream`.
 * Returns after enqueueing; D_host, doc_len_host and the workspace must
 * stay valid and unchanged until `stream` has completed. Errors as
 * maxsim_score; a short workspace returns MAXSIM_ERR_WORKSPACE. On any other
 * error return, the copies the call had queued have finished (the call waits
 * for them), though kernels already queued on `stream` may still run.
 */
size_t maxsim_score_streamed_workspace_size(int n_queries, int nq, int nd, int d, maxsim_dtype dtype,
                                            int64_t chunk_docs);
maxsim_status maxsim_score_streamed(const void *Q, int n_queries, int nq, int d, const void *D_host,
                                    int64_t B, int nd, const int32_t *doc_len_host, maxsim_dtype dtype,
                                    float *out, int32_t *argmax_out, void *workspace,
                                    size_t workspace_bytes, int64_t chunk_docs, void *stream);

/*
 * maxsim_score_i8 -- INT8 x INT8 scoring (FLASH-MAXSIM, Abstract) with
 * per-token symmetric scales:
 *   dot(i,j) = sum_k Q[i,k] * D[j,k]        exact int32
 *   sim(i,j) = (float)dot(i,j) * d_scale[j] one fp32 multiply
 *   m_i      = max_j sim(i,j)
 *   out[b]   = sum_i q_scale[i] * m_i       fp32
 *
 *   Q [nq, d] int8, q_scale [nq] fp32 (> 0)
 *   D [total_tokens, d] int8, d_scale [total_tokens] fp32 (> 0); CSR as above
 *   out [B] fp32; maxv_out [B, nq] fp32 (m_i), maxdot_out [B, nq] int32
 *   (dot at the argmax), argmax_out [B, nq] int32 -- each of the last three
 *   may be NULL.
 *
 * sm_103a has no tcgen05 8-bit integer MMA. For nq <= 32 and d <= 192 the
 * int8 operands are converted to fp16 on chip and multiplied on tcgen05:
 * int8 values and products are exact in fp16 and the partial sums (|.| <=
 * 2^22) in the fp32 accumulator, so the dots are exact. Other shapes run on
 * the warp-level IMMA path (mma.sync m16n8k32 s8).
 *
 * Limits: 1 <= nq <= 256; d in {64, 128, 192, 256, 384, 512, 768, 1024}
 * (so |dot| < 2^24 and (float)dot is exact); Q and D 16-byte aligned.
 */
maxsim_status maxsim_score_i8(const int8_t *Q, const float *q_scale, int nq, int d,
                              const int8_t *D, const float *d_scale,
                              const int64_t *offsets, int64_t B, int64_t total_tokens,
                              float *out, float *maxv_out, int32_t *maxdot_out,
                              int32_t *argmax_out, void *stream);

/*
 * maxsim_backward -- gradients through the forward argmax (FLASH-MAXSIM,
 * Abstract: the backward pass reuses the forward argmax, with an
 * inverse-grid CSR construction and an atomic-free, destination-owned
 * gradient reduction). With loss = sum_{q,b} dS[q,b] * score[q,b] and
 * a = argmax[q,b,i]:
 *   dQ[q,i,:] = sum_b dS[q,b] * D[b, a, :]
 *   dD[b,j,:] = sum_q dS[q,b] * sum_{i : a = j} Q[q,i,:]
 * Each output row is written by exactly one thread block (no atomics); for
 * dD every document's argmax entries are grouped by token (a counting sort
 * on chip: the inverse CSR) before the sums.
 *
 *   Q [n_queries, nq, d], D [B, nd, d] (dtype BF16 or FP16), doc_len as in
 *   maxsim_score; argmax [n_queries, B, nq] int32 from maxsim_score
 *   (-1 = empty document); dS [n_queries, B] fp32.
 *   dQ [n_queries, nq, d] fp32 and dD [B, nd, d] fp32 are fully written
 *   (rows no argmax points at are 0).
 *   workspace >= maxsim_backward_workspace_size(...) bytes (see below).
 *
 * Limits: d % 64 == 0, d <= 1024; n_queries * nq <= 65536; the per-document
 * sort must fit in shared memory: about (10 * nd + 2 * n_queries * nq) * 2
 * bytes <= ~227 KB (e.g. nd <= 8192 with n_queries * nq = 16384). FP32 inputs
 * return MAXSIM_ERR_UNSUPPORTED. An argmax entry outside [0, L_b) (or -1 for
 * a non-empty document) is skipped and sets MAXSIM_DEVERR_BAD_INPUT.
 * The inverse CSR lives in shared memory, one document at a time. For
 * B >= 2048 the dQ sweep is split into up to 8 document ranges whose
 * partial sums go to the workspace (maxsim_backward_workspace_size bytes,
 * 16-byte aligned; 0 bytes -- NULL allowed -- for smaller B) and are added
 * in range order, so results do not depend on scheduling. A missing or
 * short workspace returns MAXSIM_ERR_WORKSPACE.
 */
size_t maxsim_backward_workspace_size(int n_queries, int nq, int d, int64_t B, int nd);
maxsim_status maxsim_backward(const void *Q, int n_queries, int nq, int d,
                              const void *D, int64_t B, int nd, const int32_t *doc_len,
                              maxsim_dtype dtype, const int32_t *argmax, const float *dS,
                              float *dQ, float *dD,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * maxsim_backward_dq -- the dQ half of maxsim_backward alone, for training
 * with a frozen document side (pre-encoded documents: no dD is wanted).
 * Same formula, arguments, limits, workspace and errors as maxsim_backward,
 * without Q (dQ does not depend on it) and without dD. Runs the same kernels
 * as the dQ half of maxsim_backward, so dQ is identical to that call's.
 */
maxsim_status maxsim_backward_dq(int n_queries, int nq, int d,
                                 const void *D, int64_t B, int nd, const int32_t *doc_len,
                                 maxsim_dtype dtype, const int32_t *argmax, const float *dS,
                                 float *dQ, void *workspace, size_t workspace_bytes, void *stream);

/*
 * maxsim_backward_dd -- the dD half of maxsim_backward alone (the inverse-grid
 * CSR and the destination-owned dD rows), for training with a frozen query
 * side. Same formula, arguments, limits and errors as maxsim_backward,
 * without D (dD does not depend on it), dQ and the workspace (dD needs none).
 * dD is identical to that of maxsim_backward.
 */
maxsim_status maxsim_backward_dd(const void *Q, int n_queries, int nq, int d,
                                 int64_t B, int nd, const int32_t *doc_len,
                                 maxsim_dtype dtype, const int32_t *argmax, const float *dS,
                                 float *dD, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAXSIM_H_ */

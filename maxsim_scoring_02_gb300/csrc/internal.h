// internal.h -- declarations shared between the kernel translation units and
// the C-ABI layer. Not installed; the public interface is include/maxsim.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "maxsim.h"

namespace msim {

// Per-device facts the launchers need (cached by the C-ABI layer).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  unsigned* status;  // device address of the per-device status word
};

// Returns nullptr if the device could not be queried.
const DeviceInfo* device_info();

// Forward scoring on tcgen05 tensor cores (bf16 / fp16 inputs).
// Documents are given either padded (csr = 0: rows b*nd .. b*nd+L_b-1, L_b
// from doc_len or nd) or CSR (csr = 1: rows offsets[b] .. offsets[b+1]-1).
// `order` (a permutation of [0, B), or null) is the order in which documents
// are walked; outputs always land at the documents' own indices. Not
// supported by the long-query kernel (MAXSIM_ERR_UNSUPPORTED).
maxsim_status launch_fwd_tc(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows,
                            int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                            int is_bf16, float* out, int32_t* argmax, cudaStream_t stream,
                            const int32_t* order = nullptr);

// Length-bucketed document order: a stable counting sort of documents by
// their number of 8-row granules ceil(L_b / 8), ascending, into order[B].
size_t length_order_workspace_bytes(int64_t B, int nd);
maxsim_status launch_length_order(const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                                  int32_t* order, void* workspace, cudaStream_t stream);

// Query-major forward for long queries (a few hundred to 1024 tokens); same
// arguments and outputs as launch_fwd_tc, which calls it when applicable.
bool fwd_qm_applicable(int nq, int d, int64_t total_rows);
maxsim_status launch_fwd_qm(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows,
                            int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                            int is_bf16, float* out, int32_t* argmax, cudaStream_t stream);

// Forward scoring with fp32 inputs on the tensor cores, each value split on
// chip into three bf16 parts (one query of at most 64 tokens, d % 64 == 0,
// the stacked query parts <= 48 KB); fwd_x3_applicable says whether it
// takes a shape.
bool fwd_x3_applicable(int n_queries, int nq, int d, int64_t total_rows);
maxsim_status launch_fwd_x3(const float* Q, int nq, int d, const float* D, int64_t total_rows, int csr,
                            const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd, float* out,
                            int32_t* argmax, cudaStream_t stream);

// fp32 forward: the tensor-core split kernel where it applies, else FFMA.
maxsim_status launch_fwd_fp32(const float* Q, int n_queries, int nq, int d, const float* D, int64_t total_rows,
                              int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                              float* out, int32_t* argmax, cudaStream_t stream);

// Forward scoring with fp32 inputs on the CUDA cores (FFMA).
maxsim_status launch_fwd_f32(const float* Q, int n_queries, int nq, int d, const float* D, int64_t total_rows,
                             int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                             float* out, int32_t* argmax, cudaStream_t stream);

// Product-quantisation scoring: table build into `table` (pq_workspace_bytes
// of device memory, 16-byte aligned), then table-lookup scoring.
size_t pq_workspace_bytes(int nq, int M, int K);
maxsim_status launch_pq(const float* Q, int nq, int d, const float* C, int M, int K, const uint8_t* codes,
                        const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, int32_t* argmax,
                        float* table, cudaStream_t stream);

// INT8 x INT8 scoring (warp-level IMMA, exact int32 dots).
maxsim_status launch_i8(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D, const float* d_scale,
                        const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, float* maxv,
                        int32_t* maxdot, int32_t* argmax, cudaStream_t stream);

// INT8 x INT8 scores only, on tcgen05 with the documents on the MMA's M
// dimension (int8 converted to fp16 on chip; exact for d <= 192).
bool i8x_applicable(int nq, int d, int64_t total_tokens);
maxsim_status launch_i8x(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D, const float* d_scale,
                         const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, cudaStream_t stream);

// INT8 x INT8 on tcgen05 (int8 converted to fp16 on chip; exact for d <= 256).
bool i8tc_applicable(int nq, int d);
maxsim_status launch_i8tc(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D,
                          const float* d_scale, const int64_t* offsets, int64_t B, int64_t total_tokens,
                          float* out, float* maxv, int32_t* maxdot, int32_t* argmax, cudaStream_t stream);

// Scoring of documents held in host memory, in chunks through two device
// buffers (copies overlapped with scoring). dtype: 0 bf16, 1 fp16, 2 fp32.
size_t streamed_workspace_bytes(int n_queries, int nq, int nd, int d, int dtype, int64_t chunk_docs);
maxsim_status launch_streamed(const void* Q, int n_queries, int nq, int d, const void* D_host, int64_t B, int nd,
                              const int32_t* doc_len_host, int dtype, float* out, int32_t* argmax, void* workspace,
                              size_t workspace_bytes, int64_t chunk, cudaStream_t stream);

// Backward through the saved argmax: dD (inverse CSR, destination-owned) and
// dQ. `parts` selects the gradients to compute (kBackwardDD | kBackwardDQ);
// the pointers of a part not selected are not read.
constexpr int kBackwardDD = 1;
constexpr int kBackwardDQ = 2;
size_t backward_workspace_bytes(int n_queries, int nq, int d, int64_t B);
maxsim_status launch_backward(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                              const int32_t* doc_len, int is_bf16, const int32_t* argmax, const float* dS, float* dQ,
                              float* dD, float* workspace, int parts, cudaStream_t stream);

// Encodes a TMA tensor map through the driver entry point (no libcuda link).
// dtype_code: 0 fp16, 1 bf16, 2 uint8, 3 fp32; swizzle: 0 none, 1 128-byte,
// 2 64-byte. Returns false if the driver call is unavailable or rejects the
// arguments.
bool encode_tmap(void* tmap, int dtype_code, int rank, void* gaddr, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, int swizzle);

}  // namespace msim

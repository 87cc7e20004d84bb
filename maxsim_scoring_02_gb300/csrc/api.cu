// api.cu -- the extern "C" entry points of libmaxsim.so (include/maxsim.h):
// host-side argument validation, per-device facts, TMA descriptor encoding
// and the device status word. All arithmetic of the operator lives in the
// kernel translation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace msim {

// Per-device status block: word 0 is the status word written by kernels
// (timeouts, bad documents); word 1 holds test-only fault switches; words 2-3
// the bound of pipeline waits in ns (0 = the default). Kernels receive its
// address as their `status` pointer.
__device__ __align__(16) unsigned g_status_block[4];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CSR lengths are bucketed up to this many tokens (1023 8-row granules).
constexpr int kOrderCsrNd = 8 * 1023;
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[dev]) {
    DeviceInfo info;
    if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_block) != cudaSuccess) return nullptr;
    info.status = static_cast<unsigned*>(addr);
    if (cudaMemset(info.status, 0, 4 * sizeof(unsigned)) != cudaSuccess) return nullptr;
    g_dev[dev] = info;
    g_dev_ready[dev] = true;
  }
  return &g_dev[dev];
}

bool encode_tmap(void* tmap, int dtype_code, int rank, void* gaddr, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, int swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return false;
  CUtensorMapDataType dt;
  switch (dtype_code) {
    case 0: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; break;
    case 1: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; break;
    case 2: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;
    default: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; break;
  }
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  const CUresult r = g_encode(static_cast<CUtensorMap*>(tmap), dt, static_cast<cuuint32_t>(rank), gaddr, gd, gs, bx,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle == 1   ? CU_TENSOR_MAP_SWIZZLE_128B
                              : swizzle == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msim

using namespace msim;

extern "C" {

int maxsim_version(void) { return 100; }

const char* maxsim_status_string(maxsim_status status) {
  switch (status) {
    case MAXSIM_OK: return "MAXSIM_OK";
    case MAXSIM_ERR_INVALID_ARG: return "MAXSIM_ERR_INVALID_ARG: invalid argument";
    case MAXSIM_ERR_UNSUPPORTED: return "MAXSIM_ERR_UNSUPPORTED: shape or dtype not supported";
    case MAXSIM_ERR_CUDA: return "MAXSIM_ERR_CUDA: CUDA runtime or launch failure";
    case MAXSIM_ERR_TIMEOUT: return "MAXSIM_ERR_TIMEOUT: a device pipeline wait timed out";
    case MAXSIM_ERR_WORKSPACE: return "MAXSIM_ERR_WORKSPACE: workspace missing or too small";
  }
  return "MAXSIM_ERR_UNKNOWN";
}

maxsim_status maxsim_device_status(void* stream, unsigned int* flags) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned h = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MAXSIM_ERR_CUDA;
  if (cudaMemcpyAsync(&h, dev->status, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MAXSIM_ERR_CUDA;
  if (cudaMemsetAsync(dev->status, 0, sizeof(unsigned), s) != cudaSuccess) return MAXSIM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MAXSIM_ERR_CUDA;
  if (flags) *flags = h;
  if (h & MAXSIM_DEVERR_TIMEOUT) return MAXSIM_ERR_TIMEOUT;
  if (h & MAXSIM_DEVERR_BAD_INPUT) return MAXSIM_ERR_INVALID_ARG;
  return MAXSIM_OK;
}

maxsim_status maxsim_debug_set_faults(unsigned int flags, uint64_t wait_limit_ns) {
  if (flags & ~static_cast<unsigned>(MAXSIM_DEBUG_STALL_FWD_LOADER)) return MAXSIM_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  const unsigned words[3] = {flags, static_cast<unsigned>(wait_limit_ns & 0xffffffffu),
                             static_cast<unsigned>(wait_limit_ns >> 32)};
  // synchronous: visible to every kernel launched after this call returns
  if (cudaMemcpy(dev->status + 1, words, sizeof(words), cudaMemcpyHostToDevice) != cudaSuccess)
    return MAXSIM_ERR_CUDA;
  return MAXSIM_OK;
}

static maxsim_status check_common(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B,
                                  maxsim_dtype dtype, const float* out, const int32_t* argmax_out) {
  if (n_queries < 1 || nq < 1 || d < 1 || B < 0) return MAXSIM_ERR_INVALID_ARG;
  if (dtype != MAXSIM_BF16 && dtype != MAXSIM_FP16 && dtype != MAXSIM_FP32) return MAXSIM_ERR_INVALID_ARG;
  if (!Q) return MAXSIM_ERR_INVALID_ARG;
  if (B == 0) return MAXSIM_OK;  // nothing to score: D and out may be empty (NULL) buffers
  if (!D || !out) return MAXSIM_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(D) || !aligned4(out) || (argmax_out && !aligned4(argmax_out)))
    return MAXSIM_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_queries) * nq > INT_MAX / 2) return MAXSIM_ERR_UNSUPPORTED;
  if (dtype == MAXSIM_FP32) {
    if (d % 4 != 0 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  } else {
    if (d % 64 != 0 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  }
  return MAXSIM_OK;
}

maxsim_status maxsim_score(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                           const int32_t* doc_len, maxsim_dtype dtype, float* out, int32_t* argmax_out,
                           void* stream) {
  maxsim_status st = check_common(Q, n_queries, nq, d, D, B, dtype, out, argmax_out);
  if (st != MAXSIM_OK) return st;
  if (nd < 1 || (doc_len && !aligned4(doc_len))) return MAXSIM_ERR_INVALID_ARG;
  if (B == 0) return MAXSIM_OK;
  if (B > INT64_MAX / nd) return MAXSIM_ERR_INVALID_ARG;
  const int64_t rows = B * static_cast<int64_t>(nd);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == MAXSIM_FP32)
    return launch_fwd_fp32(static_cast<const float*>(Q), n_queries, nq, d, static_cast<const float*>(D), rows, 0,
                          doc_len, nullptr, B, nd, out, argmax_out, s);
  return launch_fwd_tc(Q, n_queries, nq, d, D, rows, 0, doc_len, nullptr, B, nd, dtype == MAXSIM_BF16 ? 1 : 0, out,
                       argmax_out, s);
}

size_t maxsim_length_order_workspace_size(int64_t B, int nd, int csr) {
  if (B < 0 || (!csr && nd < 1)) return 0;
  return length_order_workspace_bytes(B, csr ? kOrderCsrNd : nd);
}

maxsim_status maxsim_length_order(const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                                  int32_t* order_out, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || B > INT_MAX || (doc_len && offsets) || (!offsets && nd < 1)) return MAXSIM_ERR_INVALID_ARG;
  if (B == 0) return MAXSIM_OK;
  if (!order_out || !aligned4(order_out) || (doc_len && !aligned4(doc_len)) || (offsets && !aligned4(offsets)))
    return MAXSIM_ERR_INVALID_ARG;
  const int keys_nd = offsets ? kOrderCsrNd : nd;
  if (!workspace || !aligned16(workspace) || workspace_bytes < length_order_workspace_bytes(B, keys_nd))
    return MAXSIM_ERR_WORKSPACE;
  return launch_length_order(doc_len, offsets, B, keys_nd, order_out, workspace, static_cast<cudaStream_t>(stream));
}

maxsim_status maxsim_score_ordered(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                                   const int32_t* doc_len, const int32_t* doc_order, maxsim_dtype dtype, float* out,
                                   int32_t* argmax_out, void* stream) {
  maxsim_status st = check_common(Q, n_queries, nq, d, D, B, dtype, out, argmax_out);
  if (st != MAXSIM_OK) return st;
  if (nd < 1 || (doc_len && !aligned4(doc_len))) return MAXSIM_ERR_INVALID_ARG;
  if (B == 0) return MAXSIM_OK;
  if (!doc_order || !aligned4(doc_order) || B > INT_MAX || B > INT64_MAX / nd) return MAXSIM_ERR_INVALID_ARG;
  if (dtype == MAXSIM_FP32) return MAXSIM_ERR_UNSUPPORTED;
  const int64_t rows = B * static_cast<int64_t>(nd);
  return launch_fwd_tc(Q, n_queries, nq, d, D, rows, 0, doc_len, nullptr, B, nd, dtype == MAXSIM_BF16 ? 1 : 0, out,
                       argmax_out, static_cast<cudaStream_t>(stream), doc_order);
}

size_t maxsim_score_streamed_workspace_size(int n_queries, int nq, int nd, int d, maxsim_dtype dtype,
                                            int64_t chunk_docs) {
  if (dtype != MAXSIM_BF16 && dtype != MAXSIM_FP16 && dtype != MAXSIM_FP32) return 0;
  return streamed_workspace_bytes(n_queries, nq, nd, d, static_cast<int>(dtype), chunk_docs);
}

maxsim_status maxsim_score_streamed(const void* Q, int n_queries, int nq, int d, const void* D_host, int64_t B, int nd,
                                    const int32_t* doc_len_host, maxsim_dtype dtype, float* out,
                                    int32_t* argmax_out, void* workspace, size_t workspace_bytes,
                                    int64_t chunk_docs, void* stream) {
  // the device-side checks of maxsim_score (D_host is checked for presence only)
  maxsim_status st = check_common(Q, n_queries, nq, d, Q, B, dtype, out, argmax_out);
  if (st != MAXSIM_OK) return st;
  if (nd < 1 || chunk_docs < 1 || (doc_len_host && !aligned4(doc_len_host))) return MAXSIM_ERR_INVALID_ARG;
  if (B == 0) return MAXSIM_OK;
  if (!D_host || B > INT64_MAX / nd) return MAXSIM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MAXSIM_ERR_WORKSPACE;
  return launch_streamed(Q, n_queries, nq, d, D_host, B, nd, doc_len_host, static_cast<int>(dtype), out, argmax_out,
                         workspace, workspace_bytes, chunk_docs, static_cast<cudaStream_t>(stream));
}

maxsim_status maxsim_score_varlen(const void* Q, int n_queries, int nq, int d, const void* D_packed,
                                  const int64_t* offsets, int64_t B, int64_t total_tokens, maxsim_dtype dtype,
                                  float* out, int32_t* argmax_out, void* stream) {
  if (!offsets || !aligned4(offsets) || total_tokens < 0) return MAXSIM_ERR_INVALID_ARG;
  // No packed rows at all: D_packed may be an empty (NULL) buffer. It is never
  // read; Q (same dtype, aligned) stands in so the descriptors can be encoded.
  if (total_tokens == 0 && !D_packed) D_packed = Q;
  maxsim_status st = check_common(Q, n_queries, nq, d, D_packed, B, dtype, out, argmax_out);
  if (st != MAXSIM_OK) return st;
  if (B == 0) return MAXSIM_OK;
  // With total_tokens == 0 every document is empty: the kernels still run to
  // write score 0 / argmax -1, and never read D_packed.
  const int64_t rows = total_tokens > 0 ? total_tokens : 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == MAXSIM_FP32)
    return launch_fwd_fp32(static_cast<const float*>(Q), n_queries, nq, d, static_cast<const float*>(D_packed),
                          total_tokens, 1, nullptr, offsets, B, 0, out, argmax_out, s);
  return launch_fwd_tc(Q, n_queries, nq, d, D_packed, rows, 1, nullptr, offsets, B, 0,
                       dtype == MAXSIM_BF16 ? 1 : 0, out, argmax_out, s);
}

size_t maxsim_score_pq_workspace_size(int nq, int M, int K) { return pq_workspace_bytes(nq, M, K); }

maxsim_status maxsim_score_pq(const float* Q, int nq, int d, const float* codebooks, int M, int K,
                              const uint8_t* codes, const int64_t* offsets, int64_t B, int64_t total_tokens,
                              float* out, int32_t* argmax_out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (nq < 1 || nq > 1024 || d < 1 || d > 1024 || B < 0 || total_tokens < 0) return MAXSIM_ERR_INVALID_ARG;
  if (M < 4 || M > 64 || M % 4 != 0 || K < 1 || K > 256 || d % M != 0) return MAXSIM_ERR_UNSUPPORTED;
  if (B == 0) return MAXSIM_OK;
  if (!Q || !codebooks || !offsets || !out || (total_tokens > 0 && !codes)) return MAXSIM_ERR_INVALID_ARG;
  if (!aligned4(Q) || !aligned4(codebooks) || !aligned4(offsets) || !aligned4(out) ||
      (codes && !aligned4(codes)) || (argmax_out && !aligned4(argmax_out)))
    return MAXSIM_ERR_INVALID_ARG;
  const size_t need = pq_workspace_bytes(nq, M, K);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return MAXSIM_ERR_WORKSPACE;
  if (!codes) codes = reinterpret_cast<const uint8_t*>(Q);  // no tokens at all: never read
  return launch_pq(Q, nq, d, codebooks, M, K, codes, offsets, B, total_tokens, out, argmax_out,
                   static_cast<float*>(workspace), static_cast<cudaStream_t>(stream));
}

maxsim_status maxsim_score_i8(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D,
                              const float* d_scale, const int64_t* offsets, int64_t B, int64_t total_tokens,
                              float* out, float* maxv_out, int32_t* maxdot_out, int32_t* argmax_out,
                              void* stream) {
  if (nq < 1 || nq > 256 || d < 1 || B < 0 || total_tokens < 0) return MAXSIM_ERR_INVALID_ARG;
  switch (d) {
    case 64: case 128: case 192: case 256: case 384: case 512: case 768: case 1024: break;
    default: return MAXSIM_ERR_UNSUPPORTED;
  }
  if (B == 0) return MAXSIM_OK;
  if (!Q || !q_scale || !offsets || !out || (total_tokens > 0 && (!D || !d_scale))) return MAXSIM_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned4(q_scale) || !aligned4(offsets) || !aligned4(out) || (D && !aligned16(D)) ||
      (d_scale && !aligned4(d_scale)) || (maxv_out && !aligned4(maxv_out)) ||
      (maxdot_out && !aligned4(maxdot_out)) || (argmax_out && !aligned4(argmax_out)))
    return MAXSIM_ERR_INVALID_ARG;
  if (!D) {  // no tokens at all: never read
    D = Q;
    d_scale = q_scale;
  }
  return launch_i8(Q, q_scale, nq, d, D, d_scale, offsets, B, total_tokens, out, maxv_out, maxdot_out, argmax_out,
                   static_cast<cudaStream_t>(stream));
}

size_t maxsim_backward_workspace_size(int n_queries, int nq, int d, int64_t B, int nd) {
  (void)nd;  // the inverse CSR is built in shared memory, one document at a time
  if (n_queries < 1 || nq < 1 || d < 1 || B < 0) return 0;
  return backward_workspace_bytes(n_queries, nq, d, B);  // per-range dQ partials
}

// Shared checks of the three backward entry points; `parts` says which
// gradients are computed, and only their inputs and outputs are checked.
static maxsim_status backward_common(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                                     const int32_t* doc_len, maxsim_dtype dtype, const int32_t* argmax,
                                     const float* dS, float* dQ, float* dD, void* workspace, size_t workspace_bytes,
                                     int parts, void* stream) {
  const bool want_dd = parts & kBackwardDD, want_dq = parts & kBackwardDQ;
  if (n_queries < 1 || nq < 1 || d < 1 || B < 0 || nd < 1) return MAXSIM_ERR_INVALID_ARG;
  if (dtype != MAXSIM_BF16 && dtype != MAXSIM_FP16) return dtype == MAXSIM_FP32 ? MAXSIM_ERR_UNSUPPORTED
                                                                               : MAXSIM_ERR_INVALID_ARG;
  if (d % 64 != 0 || d > 1024 || static_cast<int64_t>(n_queries) * nq > 65536 || nd > 65535)
    return MAXSIM_ERR_UNSUPPORTED;
  if ((want_dd && !Q) || (want_dq && !dQ)) return MAXSIM_ERR_INVALID_ARG;
  if ((want_dd && !aligned16(Q)) || (want_dq && !aligned16(dQ))) return MAXSIM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0) {  // no documents: dQ is all zeros, dD is empty
    if (!want_dq) return MAXSIM_OK;
    return cudaMemsetAsync(dQ, 0, static_cast<size_t>(n_queries) * nq * d * sizeof(float), s) == cudaSuccess
               ? MAXSIM_OK
               : MAXSIM_ERR_CUDA;
  }
  if (!argmax || !dS || (want_dd && !dD) || (want_dq && !D)) return MAXSIM_ERR_INVALID_ARG;
  if (!aligned4(argmax) || !aligned4(dS) || (want_dd && !aligned16(dD)) || (want_dq && !aligned16(D)) ||
      (doc_len && !aligned4(doc_len)))
    return MAXSIM_ERR_INVALID_ARG;
  if (want_dq) {
    const size_t need = backward_workspace_bytes(n_queries, nq, d, B);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return MAXSIM_ERR_WORKSPACE;
  }
  return launch_backward(Q, n_queries, nq, d, D, B, nd, doc_len, dtype == MAXSIM_BF16 ? 1 : 0, argmax, dS, dQ, dD,
                         static_cast<float*>(workspace), parts, s);
}

maxsim_status maxsim_backward(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                              const int32_t* doc_len, maxsim_dtype dtype, const int32_t* argmax, const float* dS,
                              float* dQ, float* dD, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_common(Q, n_queries, nq, d, D, B, nd, doc_len, dtype, argmax, dS, dQ, dD, workspace,
                         workspace_bytes, kBackwardDD | kBackwardDQ, stream);
}

maxsim_status maxsim_backward_dq(int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                                 const int32_t* doc_len, maxsim_dtype dtype, const int32_t* argmax, const float* dS,
                                 float* dQ, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_common(nullptr, n_queries, nq, d, D, B, nd, doc_len, dtype, argmax, dS, dQ, nullptr, workspace,
                         workspace_bytes, kBackwardDQ, stream);
}

maxsim_status maxsim_backward_dd(const void* Q, int n_queries, int nq, int d, int64_t B, int nd,
                                 const int32_t* doc_len, maxsim_dtype dtype, const int32_t* argmax, const float* dS,
                                 float* dD, void* stream) {
  return backward_common(Q, n_queries, nq, d, nullptr, B, nd, doc_len, dtype, argmax, dS, nullptr, dD, nullptr, 0,
                         kBackwardDD, stream);
}

}  // extern "C"

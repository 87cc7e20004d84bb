// pq_noalloc.cu -- maxsim_score_pq_noalloc: product-quantisation scoring for
// callers that cannot allocate device memory.
//
// The regular maxsim_score_pq needs a caller-provided workspace for its
// lookup table. Some callers have no way to get one: code running where a
// device allocation is not allowed or not possible (inside a host callback
// or a library hook that must not call cudaMalloc, a framework whose memory
// pool is owned by someone else, a plugin with no allocator handle). This
// entry point instead keeps the table in a fixed array that is part of the
// library image, so the call itself allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine. The array exists on every GPU
// that loads the library, from load until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace msim {
namespace {

// Table capacity: 1 MiB of fp32 entries. The table takes
// ceil(nq/8)*8 * M * K * 4 bytes, e.g. nq <= 64 at M = 16, K = 256.
constexpr size_t kNoAllocTableBytes = size_t(1) << 20;

static __device__ __align__(256) float g_pq_noalloc_table[kNoAllocTableBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
float* g_table_addr[kMaxDevices];  // device address of the array, per device

// Resolves the array's device address on the current device (once per
// device). The name g_pq_noalloc_table in host code is only a host-side
// stand-in; kernels must be given this address.
float* table_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_table_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pq_noalloc_table) != cudaSuccess || !ptr) return nullptr;
    g_table_addr[dev] = static_cast<float*>(ptr);
  }
  return g_table_addr[dev];
}

}  // namespace
}  // namespace msim

extern "C" maxsim_status maxsim_score_pq_noalloc(const float* Q, int nq, int d, const float* codebooks, int M,
                                                 int K, const uint8_t* codes, const int64_t* offsets, int64_t B,
                                                 int64_t total_tokens, float* out, int32_t* argmax_out,
                                                 void* stream) {
  if (nq < 1 || M < 1 || K < 1) return MAXSIM_ERR_INVALID_ARG;
  // Tables larger than the fixed array are refused before anything runs.
  if (msim::pq_workspace_bytes(nq, M, K) > msim::kNoAllocTableBytes) return MAXSIM_ERR_WORKSPACE;
  float* table = msim::table_for_current_device();
  if (!table) return MAXSIM_ERR_CUDA;
  // Same checks and kernels as maxsim_score_pq; the table build writes every
  // entry the scoring kernel reads, so nothing left by an earlier call leaks in.
  return maxsim_score_pq(Q, nq, d, codebooks, M, K, codes, offsets, B, total_tokens, out, argmax_out, table,
                         msim::kNoAllocTableBytes, stream);
}

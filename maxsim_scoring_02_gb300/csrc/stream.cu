// stream.cu -- scoring of a corpus that stays in host memory (the pages name
// corpora larger than GPU memory as an open limitation: TileMaxSim deep
// reading §5). Host-side runtime only: the documents are copied in chunks
// into two device buffers that alternate, the copy of chunk k + 1 running on
// a library-owned copy stream while chunk k is scored on the caller's
// stream; events order each buffer's reuse, and the copy stream first waits
// for the work already queued on the caller's stream. Every chunk is scored by the
// same forward kernels as maxsim_score, so the per-document results are the
// same as scoring the whole corpus from device memory.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace msim {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_copy_mutex;
cudaStream_t g_copy_stream[kMaxDevices];

// The device's copy stream (created on first use, never blocking the legacy stream).
cudaStream_t copy_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_copy_mutex);
  if (!g_copy_stream[dev] && cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
    g_copy_stream[dev] = nullptr;
  return g_copy_stream[dev];
}

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

struct StreamLayout {
  size_t dbuf, lbuf, obuf, abuf;   // bytes of one D buffer, lengths buffer, score / argmax scratch
  size_t total;
};

StreamLayout layout_of(int n_queries, int nq, int nd, int d, size_t esz, int64_t chunk, bool lengths, bool argmax) {
  StreamLayout l;
  l.dbuf = round16(static_cast<size_t>(chunk) * nd * d * esz);
  l.lbuf = lengths ? round16(static_cast<size_t>(chunk) * 4) : 0;
  // scratch for a chunk's outputs, only when several queries need a strided scatter
  l.obuf = n_queries > 1 ? round16(static_cast<size_t>(n_queries) * chunk * 4) : 0;
  l.abuf = (n_queries > 1 && argmax) ? round16(static_cast<size_t>(n_queries) * chunk * nq * 4) : 0;
  l.total = 2 * (l.dbuf + l.lbuf) + l.obuf + l.abuf;
  return l;
}

}  // namespace

size_t streamed_workspace_bytes(int n_queries, int nq, int nd, int d, int dtype, int64_t chunk_docs) {
  if (n_queries < 1 || nq < 1 || nd < 1 || d < 1 || chunk_docs < 1) return 0;
  const size_t esz = dtype == 2 ? 4 : 2;
  // lengths and argmax scratch are always provided for: the size does not depend on the call's options
  return layout_of(n_queries, nq, nd, d, esz, chunk_docs, true, true).total;
}

maxsim_status launch_streamed(const void* Q, int n_queries, int nq, int d, const void* D_host, int64_t B, int nd,
                              const int32_t* doc_len_host, int dtype, float* out, int32_t* argmax, void* workspace,
                              size_t workspace_bytes, int64_t chunk, cudaStream_t stream) {
  const size_t esz = dtype == 2 ? 4 : 2;
  const StreamLayout l = layout_of(n_queries, nq, nd, d, esz, chunk, true, true);
  if (!workspace || workspace_bytes < l.total) return MAXSIM_ERR_WORKSPACE;
  cudaStream_t cs = copy_stream();
  if (!cs) return MAXSIM_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dbuf[2] = {ws, ws + l.dbuf};
  int32_t* lbuf[2] = {reinterpret_cast<int32_t*>(ws + 2 * l.dbuf), reinterpret_cast<int32_t*>(ws + 2 * l.dbuf + l.lbuf)};
  float* otmp = reinterpret_cast<float*>(ws + 2 * (l.dbuf + l.lbuf));
  int32_t* atmp = reinterpret_cast<int32_t*>(ws + 2 * (l.dbuf + l.lbuf) + l.obuf);

  cudaEvent_t copied[2] = {nullptr, nullptr}, consumed[2] = {nullptr, nullptr}, entry = nullptr;
  maxsim_status st = MAXSIM_OK;
  for (int i = 0; i < 2 && st == MAXSIM_OK; ++i)
    if (cudaEventCreateWithFlags(&copied[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&consumed[i], cudaEventDisableTiming) != cudaSuccess)
      st = MAXSIM_ERR_CUDA;
  // The copy stream starts after everything already queued on the caller's
  // stream: an earlier call's kernels may still be reading the workspace
  // buffers the first two chunks are about to overwrite.
  if (st == MAXSIM_OK && (cudaEventCreateWithFlags(&entry, cudaEventDisableTiming) != cudaSuccess ||
                          cudaEventRecord(entry, stream) != cudaSuccess ||
                          cudaStreamWaitEvent(cs, entry, 0) != cudaSuccess))
    st = MAXSIM_ERR_CUDA;
  const size_t doc_bytes = static_cast<size_t>(nd) * d * esz;
  const int64_t n_chunks = (B + chunk - 1) / chunk;
  for (int64_t k = 0; k < n_chunks && st == MAXSIM_OK; ++k) {
    const int buf = static_cast<int>(k & 1);
    const int64_t b0 = k * chunk;
    const int64_t nb = B - b0 < chunk ? B - b0 : chunk;
    // the copy into this buffer waits until chunk k - 2 has been scored out of it
    if (k >= 2 && cudaStreamWaitEvent(cs, consumed[buf], 0) != cudaSuccess) { st = MAXSIM_ERR_CUDA; break; }
    if (cudaMemcpyAsync(dbuf[buf], static_cast<const uint8_t*>(D_host) + b0 * doc_bytes, nb * doc_bytes,
                        cudaMemcpyHostToDevice, cs) != cudaSuccess) { st = MAXSIM_ERR_CUDA; break; }
    if (doc_len_host && cudaMemcpyAsync(lbuf[buf], doc_len_host + b0, nb * sizeof(int32_t), cudaMemcpyHostToDevice,
                                        cs) != cudaSuccess) { st = MAXSIM_ERR_CUDA; break; }
    if (cudaEventRecord(copied[buf], cs) != cudaSuccess || cudaStreamWaitEvent(stream, copied[buf], 0) != cudaSuccess) {
      st = MAXSIM_ERR_CUDA;
      break;
    }
    // one query: the chunk's outputs are contiguous in `out`; several: scratch, then a strided scatter
    float* o = n_queries == 1 ? out + b0 : otmp;
    int32_t* a = argmax ? (n_queries == 1 ? argmax + b0 * nq : atmp) : nullptr;
    const int32_t* L = doc_len_host ? lbuf[buf] : nullptr;
    st = dtype == 2 ? launch_fwd_fp32(static_cast<const float*>(Q), n_queries, nq, d,
                                     reinterpret_cast<const float*>(dbuf[buf]), nb * nd, 0, L, nullptr, nb, nd, o, a,
                                     stream)
                    : launch_fwd_tc(Q, n_queries, nq, d, dbuf[buf], nb * nd, 0, L, nullptr, nb, nd, dtype == 0 ? 1 : 0,
                                    o, a, stream);
    if (st != MAXSIM_OK) break;
    if (n_queries > 1) {
      if (cudaMemcpy2DAsync(out + b0, B * sizeof(float), otmp, nb * sizeof(float), nb * sizeof(float), n_queries,
                            cudaMemcpyDeviceToDevice, stream) != cudaSuccess) { st = MAXSIM_ERR_CUDA; break; }
      if (argmax && cudaMemcpy2DAsync(argmax + b0 * nq, B * nq * sizeof(int32_t), atmp, nb * nq * sizeof(int32_t),
                                      nb * nq * sizeof(int32_t), n_queries, cudaMemcpyDeviceToDevice,
                                      stream) != cudaSuccess) { st = MAXSIM_ERR_CUDA; break; }
    }
    if (cudaEventRecord(consumed[buf], stream) != cudaSuccess) st = MAXSIM_ERR_CUDA;
  }
  // On an error the caller's stream may not wait on every copy already queued
  // into the workspace: finish them before returning, so the caller can free it.
  if (st != MAXSIM_OK) cudaStreamSynchronize(cs);
  // destruction is deferred by the runtime until the recorded work completes
  for (int i = 0; i < 2; ++i) {
    if (copied[i]) cudaEventDestroy(copied[i]);
    if (consumed[i]) cudaEventDestroy(consumed[i]);
  }
  if (entry) cudaEventDestroy(entry);
  return st;
}

}  // namespace msim

// order.cu -- length-bucketed document order (TileMaxSim deep reading §5:
// padding wastes token compute on variable-length corpora, and batching
// documents of similar length recovers the throughput).
//
// The order is a stable counting sort of the documents by their number of
// 8-row granules, key(b) = min(ceil(L_b / 8), K - 1), ascending: documents of
// equal key keep their index order. It depends only on the lengths, so a
// corpus computes it once and scores every query in that order. Three
// kernels, no atomics, deterministic:
//   1. count:   each warp owns a contiguous range of documents and builds its
//               key histogram in shared memory (lanes with equal keys found
//               with __match_any_sync, one leader per key adds the count);
//   2. scan:    one CTA turns the [warp][key] counts into exclusive starts in
//               (key, warp) order, so a key's documents are ordered by warp
//               and, within a warp, by index;
//   3. scatter: each warp walks its range again and writes every document
//               index at its key's running start plus its rank among the
//               equal-key lanes of its 32-document batch.
#include <cuda_runtime.h>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kOrdWarps = 8;
constexpr int kOrdThreads = 32 * kOrdWarps;
constexpr int kOrdCtas = 32;
constexpr int kOrdW = kOrdCtas * kOrdWarps;   // warps, each owning a document range
constexpr int kOrdMaxKeys = 1024;
constexpr int kScanThreads = 1024;

struct OrdParams {
  const int32_t* doc_len;    // padded layout (L_b <= nd), or null
  const int64_t* offsets;    // CSR layout, or null
  int64_t B;
  int nd;
  int K;                     // number of keys
  int32_t* counts;           // [kOrdW][K] workspace: counts, then starts
  int32_t* order;            // [B]
  unsigned* status;
};

int keys_for(int nd) {
  const int64_t k = (static_cast<int64_t>(nd) + 7) / 8 + 1;
  return static_cast<int>(k < kOrdMaxKeys ? k : kOrdMaxKeys);
}

__device__ __forceinline__ int ord_key(const OrdParams& p, int64_t b, bool& bad) {
  int64_t L = p.nd;
  if (p.doc_len) {
    L = __ldg(p.doc_len + b);
    if (L < 0 || L > p.nd) {
      bad = true;
      L = 0;
    }
  } else if (p.offsets) {
    L = __ldg(p.offsets + b + 1) - __ldg(p.offsets + b);
    if (L < 0) {
      bad = true;
      L = 0;
    }
  }
  const int64_t k = (L + 7) / 8;
  return static_cast<int>(k < p.K - 1 ? k : p.K - 1);
}

__device__ __forceinline__ void warp_range(const OrdParams& p, int gw, int64_t& b0, int64_t& b1) {
  b0 = p.B * gw / kOrdW;
  b1 = p.B * (gw + 1) / kOrdW;
}

__global__ void __launch_bounds__(kOrdThreads) ord_count_kernel(const OrdParams p) {
  extern __shared__ int32_t hist[];   // [kOrdWarps][K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kOrdWarps * p.K; i += kOrdThreads) hist[i] = 0;
  __syncthreads();
  int32_t* h = hist + warp * p.K;
  int64_t b0, b1;
  const int gw = blockIdx.x * kOrdWarps + warp;
  warp_range(p, gw, b0, b1);
  bool bad = false;
  for (int64_t c = b0; c < b1; c += 32) {
    const int64_t b = c + lane;
    const int key = b < b1 ? ord_key(p, b, bad) : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(grp) - 1) h[key] += __popc(grp);
    __syncwarp();
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kDevErrBadInput);
  for (int k = lane; k < p.K; k += 32) p.counts[static_cast<int64_t>(gw) * p.K + k] = h[k];
}

// Exclusive scan of counts in (key, warp) order, in place.
__global__ void __launch_bounds__(kScanThreads) ord_scan_kernel(const OrdParams p) {
  __shared__ int32_t wsum[kScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = static_cast<int64_t>(p.K) * kOrdW;
  const int64_t per = (n + kScanThreads - 1) / kScanThreads;
  const int64_t i0 = tid * per, i1 = i0 + per < n ? i0 + per : n;
  // element x of the (key, warp) sequence: key x / W, warp x % W
  auto at = [&](int64_t x) -> int32_t& { return p.counts[(x % kOrdW) * p.K + x / kOrdW]; };
  int run = 0;
  for (int64_t x = i0; x < i1; ++x) run += at(x);
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  base += incl - run;
  for (int64_t x = i0; x < i1; ++x) {
    const int c = at(x);
    at(x) = base;
    base += c;
  }
}

__global__ void __launch_bounds__(kOrdThreads) ord_scatter_kernel(const OrdParams p) {
  extern __shared__ int32_t start[];   // [kOrdWarps][K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kOrdWarps + warp;
  int32_t* st = start + warp * p.K;
  for (int k = lane; k < p.K; k += 32) st[k] = p.counts[static_cast<int64_t>(gw) * p.K + k];
  __syncwarp();
  int64_t b0, b1;
  warp_range(p, gw, b0, b1);
  bool bad = false;
  for (int64_t c = b0; c < b1; c += 32) {
    const int64_t b = c + lane;
    const int key = b < b1 ? ord_key(p, b, bad) : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (key >= 0) p.order[st[key] + __popc(grp & ((1u << lane) - 1u))] = static_cast<int32_t>(b);
    __syncwarp();
    if (key >= 0 && lane == __ffs(grp) - 1) st[key] += __popc(grp);
    __syncwarp();
  }
}

}  // namespace

size_t length_order_workspace_bytes(int64_t B, int nd) {
  (void)B;
  return static_cast<size_t>(kOrdW) * keys_for(nd) * sizeof(int32_t);
}

maxsim_status launch_length_order(const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                                  int32_t* order, void* workspace, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  OrdParams p;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.nd = nd;
  p.K = keys_for(nd);
  p.counts = static_cast<int32_t*>(workspace);
  p.order = order;
  p.status = dev->status;
  const size_t smem = static_cast<size_t>(kOrdWarps) * p.K * sizeof(int32_t);
  ord_count_kernel<<<kOrdCtas, kOrdThreads, smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  ord_scan_kernel<<<1, kScanThreads, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  ord_scatter_kernel<<<kOrdCtas, kOrdThreads, smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  return MAXSIM_OK;
}

}  // namespace msim

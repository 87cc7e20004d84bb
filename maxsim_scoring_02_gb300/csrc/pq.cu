// pq.cu -- fused product-quantisation MaxSim scoring (TileMaxSim deep
// reading §2(3)): decoded document vectors never exist; each token's
// similarity to query token i is a sum of table lookups.
//
//   T[i,m,k]  = sum_{t < d/M} Q[i, m*(d/M) + t] * C[m,k,t]      (pq_table_kernel)
//   sim(i,j)  = sum_{m < M} T[i, m, codes[j,m]]
//   out[b]    = sum_i max_{j in doc b} sim(i,j)                  (pq_score_kernel)
//
// Workspace layout (the only scratch memory of this path): the table in
// groups of 8 query tokens, [ceil(nq/8)][M][K][8] fp32, entries for query
// tokens past nq zero. One group (M*K*8 floats; 128 KB at M=16, K=256) sits
// in shared memory while a CTA scores its document range; the CTA then
// moves to the next group and adds that group's maxima to out[b]. Codes are
// re-read once per group (16 B per token at M=16 -- small next to the table
// lookups, which bound this path: shared-memory load throughput).
//
// Scoring thread map: a warp owns one document at a time; lane = (token
// slot tk = lane/8, query token i = lane%8), so the 8 lanes of a token read
// 32 consecutive bytes of the table per subspace. Lowest token index wins
// ties, as in the other paths.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kPqThreads = 256;
constexpr int kGroup = 8;  // query tokens per table group

__global__ void pq_table_kernel(const float* __restrict__ Q, int nq, int d, const float* __restrict__ C, int M,
                                int K, float* __restrict__ T) {
  // one thread per (group slot i, m, k); i spans ceil(nq/8)*8 so padding is written as 0
  const int ds = d / M;
  const int64_t n = static_cast<int64_t>((nq + kGroup - 1) / kGroup) * kGroup * M * K;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(e % K);
    const int m = static_cast<int>((e / K) % M);
    const int i = static_cast<int>(e / (static_cast<int64_t>(K) * M));
    float s = 0.f;
    if (i < nq) {
      const float* q = Q + static_cast<int64_t>(i) * d + m * ds;
      const float* c = C + (static_cast<int64_t>(m) * K + k) * ds;
      for (int t = 0; t < ds; ++t) s = fmaf(q[t], c[t], s);
    }
    const int g = i / kGroup, ii = i % kGroup;
    T[((static_cast<int64_t>(g) * M + m) * K + k) * kGroup + ii] = s;
  }
}

struct PqParams {
  const float* T;          // workspace table
  const uint8_t* codes;    // [total_tokens, M]
  const int64_t* offsets;  // [B+1]
  int64_t B, total_tokens;
  int nq, M, K, n_groups;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

// Codes of one token as 32-bit words (M % 4 == 0); word w holds subspaces 4w..4w+3.
template <bool ARGMAX>
__global__ void __launch_bounds__(kPqThreads, 1) pq_score_kernel(const PqParams p) {
  extern __shared__ float4 pq_smem4[];
  float* Ts = reinterpret_cast<float*>(pq_smem4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tk = lane >> 3, ii = lane & 7;
  const int M = p.M, K = p.K, MW = M >> 2;
  const uint32_t kmax = static_cast<uint32_t>(K - 1);
  const int64_t b0 = (p.B * blockIdx.x) / gridDim.x, b1 = (p.B * (blockIdx.x + 1)) / gridDim.x;
  const int64_t tsize = static_cast<int64_t>(M) * K * kGroup;  // floats per group
  const uint32_t* codes32 = reinterpret_cast<const uint32_t*>(p.codes);

  for (int g = 0; g < p.n_groups; ++g) {
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(p.T + g * tsize);
    for (int64_t e = tid; e < tsize / 4; e += kPqThreads) pq_smem4[e] = __ldg(src + e);
    __syncthreads();
    const int qi = g * kGroup + ii;
    for (int64_t b = b0 + warp; b < b1; b += kPqThreads / 32) {
      const int64_t s0 = __ldg(p.offsets + b), e0 = __ldg(p.offsets + b + 1);
      const bool bad = s0 < 0 || e0 < s0 || e0 > p.total_tokens;
      if (bad && g == 0 && lane == 0) atomicOr(p.status, kDevErrBadInput);
      const int64_t L = bad ? 0 : e0 - s0;
      float rm = -INFINITY;
      int ra = INT_MAX;
      bool badc = false;
      // token j = 4*it + tk; codes of the next iteration are loaded before the current one is scored
      uint32_t cw[16], nw[16];
      const uint32_t* row = codes32 + (s0 + tk) * MW;
#pragma unroll
      for (int w = 0; w < 16; ++w)
        if (w < MW) cw[w] = (tk < L) ? __ldg(row + w) : 0u;
      for (int64_t j = tk; j < L; j += 4) {
        const int64_t jn = j + 4;
#pragma unroll
        for (int w = 0; w < 16; ++w)
          if (w < MW) nw[w] = (jn < L) ? __ldg(row + (jn - tk) * MW + w) : 0u;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          if (w < MW) {
#pragma unroll
            for (int sb = 0; sb < 4; ++sb) {
              const int m = 4 * w + sb;
              const uint32_t raw = (cw[w] >> (8 * sb)) & 0xFFu;
              badc |= raw > kmax;                       // a code outside the codebook is clamped and reported
              s += Ts[(m * K + static_cast<int>(min(raw, kmax))) * kGroup + ii];
            }
          }
        }
        if (s > rm) {  // tokens ascend per lane: strict > keeps the lowest index
          rm = s;
          ra = static_cast<int>(j);
        }
#pragma unroll
        for (int w = 0; w < 16; ++w)
          if (w < MW) cw[w] = nw[w];
      }
      if (__any_sync(0xffffffffu, badc) && lane == 0 && g == 0) atomicOr(p.status, kDevErrBadInput);
      // max over the 4 token slots (lanes ii, ii+8, ii+16, ii+24)
#pragma unroll
      for (int o = 8; o <= 16; o <<= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, rm, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, ra, o);
        if (v2 > rm || (v2 == rm && i2 < ra)) {
          rm = v2;
          ra = i2;
        }
      }
      float part = (L > 0 && qi < p.nq) ? rm : 0.f;
      if (ARGMAX && tk == 0 && qi < p.nq) p.argmax[b * p.nq + qi] = L > 0 ? ra : -1;
#pragma unroll
      for (int o = 1; o <= 4; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) p.out[b] = (g == 0 ? 0.f : p.out[b]) + part;
    }
  }
}

}  // namespace

size_t pq_workspace_bytes(int nq, int M, int K) {
  if (nq < 1 || M < 1 || K < 1) return 0;
  return static_cast<size_t>((nq + kGroup - 1) / kGroup) * kGroup * M * K * sizeof(float);
}

maxsim_status launch_pq(const float* Q, int nq, int d, const float* C, int M, int K, const uint8_t* codes,
                        const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, int32_t* argmax,
                        float* table, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  const size_t smem = static_cast<size_t>(M) * K * kGroup * sizeof(float);
  if (smem > static_cast<size_t>(dev->max_smem_optin)) return MAXSIM_ERR_UNSUPPORTED;
  const int n_groups = (nq + kGroup - 1) / kGroup;
  {
    const int64_t n = static_cast<int64_t>(n_groups) * kGroup * M * K;
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
    pq_table_kernel<<<grid, threads, 0, stream>>>(Q, nq, d, C, M, K, table);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  }
  PqParams p;
  p.T = table;
  p.codes = codes;
  p.offsets = offsets;
  p.B = B;
  p.total_tokens = total_tokens;
  p.nq = nq;
  p.M = M;
  p.K = K;
  p.n_groups = n_groups;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;
  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  cudaError_t e;
  if (argmax) {
    e = cudaFuncSetAttribute(pq_score_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) pq_score_kernel<true><<<grid, kPqThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(pq_score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) pq_score_kernel<false><<<grid, kPqThreads, smem, stream>>>(p);
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

// fwd_f32.cu -- MaxSim forward with fp32 inputs on the CUDA cores (FFMA).
//
// Same operator and outputs as the tensor-core path (TileMaxSim deep
// reading §1; FLASH-MAXSIM Figure 1 / Algorithm 2), for fp32 embeddings that
// must be scored at fp32 accuracy: TF32 tensor-core inputs would round every
// element to 10 mantissa bits, far outside an fp32 score tolerance, so the
// products are formed with FFMA.
//
// Block of 256 threads = 8 warps. For a 32-token query chunk and a 128-token
// document tile, warp w owns query tokens 4w..4w+3 and lane l owns document
// tokens l, l+32, l+64, l+96: a 4 x 4 register tile of fp32 dot products,
// accumulated over 128-wide d-chunks staged in padded shared memory (row
// pitch 132 floats, so the lane-strided float4 reads are conflict-free). The
// maximum over tokens is a per-thread running maximum across tiles followed
// by one warp butterfly; the sum over query tokens goes through shared
// memory. Each grid-stride step handles one document for every query.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kThreads = 256;
constexpr int kQC = 32;     // query tokens per chunk
constexpr int kTT = 128;    // document tokens per tile
constexpr int kKC = 128;    // d per chunk
constexpr int kPitch = kKC + 4;

struct F32Params {
  const float* Q;
  const float* D;
  const int32_t* doc_len;
  const int64_t* offsets;
  int64_t B;
  int64_t total_rows;
  int nd, csr, n_queries, nq, d;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

__device__ __forceinline__ int64_t f32_doc_rows(const F32Params& p, int64_t b, int64_t& start, bool& bad) {
  bad = false;
  if (p.csr) {
    const int64_t s = __ldg(p.offsets + b), e = __ldg(p.offsets + b + 1);
    if (s < 0 || e < s || e > p.total_rows || e - s > INT_MAX) {
      bad = true;
      start = 0;
      return 0;
    }
    start = s;
    return e - s;
  }
  start = b * static_cast<int64_t>(p.nd);
  const int64_t L = p.doc_len ? static_cast<int64_t>(__ldg(p.doc_len + b)) : static_cast<int64_t>(p.nd);
  if (L < 0 || L > p.nd) {
    bad = true;
    return 0;
  }
  return L;
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kThreads) fwd_f32_kernel(const F32Params p) {
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);          // [kQC][kPitch]
  float* Ds = Qs + kQC * kPitch;                         // [kTT][kPitch]
  float* red = Ds + kTT * kPitch;                        // [8]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_qchunks = (p.nq + kQC - 1) / kQC;
  const int n_kc = (p.d + kKC - 1) / kKC;

  for (int64_t b = blockIdx.x; b < p.B; b += gridDim.x) {
    int64_t start;
    bool bad;
    const int64_t L = f32_doc_rows(p, b, start, bad);
    if (bad && tid == 0) atomicOr(p.status, kDevErrBadInput);
    const int ntiles = static_cast<int>((L + kTT - 1) / kTT);
    for (int q = 0; q < p.n_queries; ++q) {
      float qsum = 0.f;
      for (int qc = 0; qc < n_qchunks; ++qc) {
        float rm[4];
        int ra[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          rm[r] = -INFINITY;
          ra[r] = INT_MAX;
        }
        for (int t = 0; t < ntiles; ++t) {
          float acc[4][4];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < 4; ++m) acc[r][m] = 0.f;
          for (int kc = 0; kc < n_kc; ++kc) {
            const int k0 = kc * kKC;
            const int kw = min(kKC, p.d - k0);   // multiple of 4
            const int kw4 = kw >> 2;
            __syncthreads();
            // stage the query chunk (rows past nq read as 0)
            for (int f = tid; f < kQC * kw4; f += kThreads) {
              const int r = f / kw4, c4 = f % kw4;
              const int qi = qc * kQC + r;
              float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
              if (qi < p.nq)
                v = __ldg(reinterpret_cast<const float4*>(p.Q + (static_cast<int64_t>(q) * p.nq + qi) * p.d + k0) + c4);
              *reinterpret_cast<float4*>(Qs + r * kPitch + c4 * 4) = v;
            }
            // stage the document tile (rows past L read as 0, masked below)
            for (int f = tid; f < kTT * kw4; f += kThreads) {
              const int r = f / kw4, c4 = f % kw4;
              const int64_t j = static_cast<int64_t>(t) * kTT + r;
              float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
              if (j < L) v = __ldg(reinterpret_cast<const float4*>(p.D + (start + j) * p.d + k0) + c4);
              *reinterpret_cast<float4*>(Ds + r * kPitch + c4 * 4) = v;
            }
            __syncthreads();
            for (int k = 0; k < kw; k += 4) {
              float4 qv[4], dv[4];
#pragma unroll
              for (int r = 0; r < 4; ++r) qv[r] = *reinterpret_cast<const float4*>(Qs + (warp * 4 + r) * kPitch + k);
#pragma unroll
              for (int m = 0; m < 4; ++m) dv[m] = *reinterpret_cast<const float4*>(Ds + (lane + 32 * m) * kPitch + k);
#pragma unroll
              for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  float s = acc[r][m];
                  s = fmaf(qv[r].x, dv[m].x, s);
                  s = fmaf(qv[r].y, dv[m].y, s);
                  s = fmaf(qv[r].z, dv[m].z, s);
                  s = fmaf(qv[r].w, dv[m].w, s);
                  acc[r][m] = s;
                }
            }
          }
          // fold the tile into the running maxima (tokens ascending per thread)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int64_t j = static_cast<int64_t>(t) * kTT + lane + 32 * m;
            if (j < L) {
#pragma unroll
              for (int r = 0; r < 4; ++r)
                if (acc[r][m] > rm[r]) {
                  rm[r] = acc[r][m];
                  ra[r] = static_cast<int>(j);
                }
            }
          }
        }
        // warp butterfly: max over the 32 lanes, lowest index on ties
#pragma unroll
        for (int r = 0; r < 4; ++r) {
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, rm[r], o);
            const int i2 = __shfl_xor_sync(0xffffffffu, ra[r], o);
            if (v2 > rm[r] || (v2 == rm[r] && i2 < ra[r])) {
              rm[r] = v2;
              ra[r] = i2;
            }
          }
        }
        float part = 0.f;
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int qi = qc * kQC + warp * 4 + r;
            if (qi < p.nq) {
              if (L > 0) part += rm[r];
              if (ARGMAX) p.argmax[(static_cast<int64_t>(q) * p.B + b) * p.nq + qi] = L > 0 ? ra[r] : -1;
            }
          }
          red[warp] = part;
        }
        __syncthreads();
        if (tid == 0) {
          float s = 0.f;
          for (int w = 0; w < 8; ++w) s += red[w];
          qsum += s;
        }
        __syncthreads();  // red[] is rewritten by the next chunk
      }
      if (tid == 0) p.out[static_cast<int64_t>(q) * p.B + b] = qsum;
    }
  }
}

}  // namespace

maxsim_status launch_fwd_f32(const float* Q, int n_queries, int nq, int d, const float* D, int64_t total_rows,
                             int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                             float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (d % 4 != 0 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  F32Params p;
  p.Q = Q;
  p.D = D;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = n_queries;
  p.nq = nq;
  p.d = d;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;
  const size_t smem = (static_cast<size_t>(kQC + kTT) * kPitch + 8) * sizeof(float);
  const int64_t want = static_cast<int64_t>(dev->sm_count) * 2;
  const int grid = static_cast<int>(B < want ? B : want);
  cudaError_t e;
  if (argmax) {
    e = cudaFuncSetAttribute(fwd_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_f32_kernel<true><<<grid, kThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(fwd_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_f32_kernel<false><<<grid, kThreads, smem, stream>>>(p);
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

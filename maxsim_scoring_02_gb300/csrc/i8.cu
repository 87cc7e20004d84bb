// i8.cu -- INT8 x INT8 MaxSim scoring (FLASH-MAXSIM, Abstract: INT8xINT8
// quantisation) with per-token symmetric scales:
//
//   dot(i,j) = sum_k Q[i,k] * D[j,k]            exact int32 (tensor-core IMMA)
//   sim(i,j) = (float)dot(i,j) * d_scale[j]     one fp32 multiply, round-to-nearest
//   m_i      = max_j sim(i,j)                   lowest j on ties
//   out[b]   = sum_i q_scale[i] * m_i           fp32
//
// The 5th-generation tensor-core instruction for 8-bit integers
// (tcgen05.mma kind::i8) is not available for sm_103a, so the integer
// contraction runs on the warp-level IMMA path, mma.sync m16n8k32
// s8 x s8 -> s32, which keeps the dot products exact.
//
// Thread map: a warp owns one document at a time and walks it in 16-token
// row tiles; A fragments are loaded from global memory directly into
// registers (rows past the document end read as 0 and are masked), the
// query's B fragments come from shared memory in groups of 32 query tokens
// (4 n-tiles of 8). Each lane keeps the running maximum, its token index and
// its integer dot for the two query columns x two rows it holds; at the
// document end the 8 row-lanes of each column are combined with shuffles.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kI8Threads = 256;

struct I8Params {
  const int8_t* Q;
  const float* q_scale;
  const int8_t* D;
  const float* d_scale;
  const int64_t* offsets;
  int64_t B, total_tokens;
  int nq, d;
  float* out;
  float* maxv;
  int32_t* maxdot;
  int32_t* argmax;
  unsigned* status;
};

__device__ __forceinline__ void imma_16832(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Running best of one (query column) slot: value, token index, integer dot.
struct Best {
  float v;
  int j;
  int dot;
};
__device__ __forceinline__ void take(Best& b, float v, int j, int dot) {
  if (v > b.v || (v == b.v && j < b.j)) {
    b.v = v;
    b.j = j;
    b.dot = dot;
  }
}

// KC = d / 32 k-chunks (compile-time so the A fragments stay in registers).
template <int KC, bool DETAIL>
__global__ void __launch_bounds__(kI8Threads) i8_score_kernel(const I8Params p) {
  extern __shared__ uint32_t qs32[];  // Q as [nq_pad][d/4] words, rows past nq zero
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nqp = (p.nq + 31) & ~31;
  const int dw = p.d >> 2;
  for (int e = tid; e < nqp * dw; e += kI8Threads) {
    const int r = e / dw;
    qs32[e] = r < p.nq ? __ldg(reinterpret_cast<const uint32_t*>(p.Q) + e) : 0u;
  }
  __syncthreads();

  const int nwarps = gridDim.x * (kI8Threads / 32);
  const int gw = blockIdx.x * (kI8Threads / 32) + warp;
  for (int64_t b = gw; b < p.B; b += nwarps) {
    const int64_t s0 = __ldg(p.offsets + b), e0 = __ldg(p.offsets + b + 1);
    const bool bad = s0 < 0 || e0 < s0 || e0 > p.total_tokens || e0 - s0 > INT_MAX;
    if (bad && lane == 0) atomicOr(p.status, kDevErrBadInput);
    const int L = bad ? 0 : static_cast<int>(e0 - s0);
    float score = 0.f;
    for (int qg = 0; qg < nqp; qg += 32) {   // groups of 32 query columns = 4 n-tiles
      Best best[4][2];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) best[n][h] = Best{-INFINITY, INT_MAX, 0};
      for (int r0 = 0; r0 < L; r0 += 16) {
        const int ra = r0 + g, rb = r0 + g + 8;
        const bool va = ra < L, vb = rb < L;
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(p.D + (s0 + ra) * p.d);
        const uint32_t* pb = reinterpret_cast<const uint32_t*>(p.D + (s0 + rb) * p.d);
        uint32_t af[KC][4];
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
          af[kc][0] = va ? __ldg(pa + kc * 8 + t) : 0u;
          af[kc][1] = vb ? __ldg(pb + kc * 8 + t) : 0u;
          af[kc][2] = va ? __ldg(pa + kc * 8 + 4 + t) : 0u;
          af[kc][3] = vb ? __ldg(pb + kc * 8 + 4 + t) : 0u;
        }
        const float sa = va ? __ldg(p.d_scale + s0 + ra) : 0.f;
        const float sb = vb ? __ldg(p.d_scale + s0 + rb) : 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          int c[4] = {0, 0, 0, 0};
          const uint32_t* qrow = qs32 + (qg + n * 8 + g) * dw;
#pragma unroll
          for (int kc = 0; kc < KC; ++kc) imma_16832(c, af[kc], qrow[kc * 8 + t], qrow[kc * 8 + 4 + t]);
          // c0,c1: row ra, columns 2t, 2t+1; c2,c3: row rb
          if (va) {
            take(best[n][0], __fmul_rn(static_cast<float>(c[0]), sa), ra, c[0]);
            take(best[n][1], __fmul_rn(static_cast<float>(c[1]), sa), ra, c[1]);
          }
          if (vb) {
            take(best[n][0], __fmul_rn(static_cast<float>(c[2]), sb), rb, c[2]);
            take(best[n][1], __fmul_rn(static_cast<float>(c[3]), sb), rb, c[3]);
          }
        }
      }
      // combine the 8 row-lanes (same t) of every column
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int o = 4; o <= 16; o <<= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, best[n][h].v, o);
            const int j2 = __shfl_xor_sync(0xffffffffu, best[n][h].j, o);
            const int d2 = __shfl_xor_sync(0xffffffffu, best[n][h].dot, o);
            take(best[n][h], v2, j2, d2);
          }
      if (g == 0) {
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int qi = qg + n * 8 + 2 * t + h;
            if (qi < p.nq) {
              const float mv = L > 0 ? best[n][h].v : 0.f;
              score = fmaf(__ldg(p.q_scale + qi), mv, score);
              if (DETAIL) {
                const int64_t o = b * p.nq + qi;
                if (p.maxv) p.maxv[o] = mv;
                if (p.maxdot) p.maxdot[o] = L > 0 ? best[n][h].dot : 0;
                if (p.argmax) p.argmax[o] = L > 0 ? best[n][h].j : -1;
              }
            }
          }
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) score += __shfl_xor_sync(0xffffffffu, score, o);
    if (lane == 0) p.out[b] = score;
  }
}

template <int KC>
cudaError_t launch_kc(const I8Params& p, bool detail, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e;
  if (detail) {
    e = cudaFuncSetAttribute(i8_score_kernel<KC, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8_score_kernel<KC, true><<<grid, kI8Threads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(i8_score_kernel<KC, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8_score_kernel<KC, false><<<grid, kI8Threads, smem, stream>>>(p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

maxsim_status launch_i8(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D, const float* d_scale,
                        const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, float* maxv,
                        int32_t* maxdot, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  I8Params p;
  p.Q = Q;
  p.q_scale = q_scale;
  p.D = D;
  p.d_scale = d_scale;
  p.offsets = offsets;
  p.B = B;
  p.total_tokens = total_tokens;
  p.nq = nq;
  p.d = d;
  p.out = out;
  p.maxv = maxv;
  p.maxdot = maxdot;
  p.argmax = argmax;
  p.status = dev->status;
  const size_t smem = static_cast<size_t>((nq + 31) & ~31) * d;
  if (smem > static_cast<size_t>(dev->max_smem_optin)) return MAXSIM_ERR_UNSUPPORTED;
  const int64_t want = static_cast<int64_t>(dev->sm_count) * 4;
  const int64_t warps = (B + 7) / 8;
  const int grid = static_cast<int>(warps < want ? (warps < 1 ? 1 : warps) : want);
  const bool detail = maxv || maxdot || argmax;
  cudaError_t e;
  switch (d / 32) {
    case 2: e = launch_kc<2>(p, detail, grid, smem, stream); break;
    case 4: e = launch_kc<4>(p, detail, grid, smem, stream); break;
    case 6: e = launch_kc<6>(p, detail, grid, smem, stream); break;
    case 8: e = launch_kc<8>(p, detail, grid, smem, stream); break;
    case 12: e = launch_kc<12>(p, detail, grid, smem, stream); break;
    case 16: e = launch_kc<16>(p, detail, grid, smem, stream); break;
    case 24: e = launch_kc<24>(p, detail, grid, smem, stream); break;
    case 32: e = launch_kc<32>(p, detail, grid, smem, stream); break;
    default: return MAXSIM_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

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
// Thread map: a warp owns one document at a time and walks it in 32-row
// pieces staged in shared memory (16-row IMMA tiles; rows past the document
// end read as 0 and are masked); the query's B fragments come from shared
// memory in groups of 32 query tokens (4 n-tiles of 8). Each lane keeps the
// running maximum, its token index and its integer dot for the two query
// columns x two rows it holds; at the document end the 8 row-lanes of each
// column are combined with shuffles.
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
  int piece_rows;  // rows staged per piece: 32 or 16 (chosen to fit shared memory)
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kMaxPieceRows = 32;  // document rows staged per piece (two 16-row IMMA tiles)

// One unit of a warp's work: rows [j0, j0 + n) of its k-th document, for
// query-column group qg (32 columns).
struct Step {
  int64_t k;
  int qg;
  int j0, n;
  int64_t b, row0;
  bool valid, first, last;   // first / last piece of (document, qg)
};

// KC = d / 32 k-chunks (compile-time so fragment loops unroll). Each warp
// stages 32-row pieces of its documents (rows padded to d + 16 bytes, so
// the A-fragment reads hit 32 distinct banks) and their scales into a
// per-warp double buffer with cp.async; the next piece is in flight while
// the current one is multiplied.
template <int KC, bool DETAIL>
__global__ void __launch_bounds__(kI8Threads) i8_score_kernel(const I8Params p) {
  extern __shared__ uint32_t qs32[];  // Q as [nq_pad][d/4] words, rows past nq zero; then the stages
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int d = p.d;
  const int nqp = (p.nq + 31) & ~31;
  const int dw = d >> 2;
  const int pitch = d + 16;                                  // bytes per staged row
  const int pr = p.piece_rows;
  const int stage_bytes = pr * pitch + pr * 4;
  const int nthreads = blockDim.x;
  for (int e = tid; e < nqp * dw; e += nthreads) {
    const int r = e / dw;
    qs32[e] = r < p.nq ? __ldg(reinterpret_cast<const uint32_t*>(p.Q) + e) : 0u;
  }
  uint8_t* stage = reinterpret_cast<uint8_t*>(qs32 + nqp * dw) + warp * 2 * stage_bytes;
  const uint32_t stage_s = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  __syncthreads();

  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (nthreads / 32);
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (nthreads / 32) + warp;
  // offsets of 32 of this warp's documents at a time (lane k holds document k)
  int64_t kbase = -64, s_reg = 0, e_reg = 0;
  auto doc_range = [&](int64_t k, int64_t& s0, int& L) -> bool {
    const int64_t b = gw + k * nwarps;
    if (b >= p.B) return false;
    if (k - kbase >= 32 || k < kbase) {
      kbase = k;
      const int64_t bl = gw + (k + lane) * nwarps;
      s_reg = e_reg = 0;
      if (bl < p.B) {
        s_reg = __ldg(p.offsets + bl);
        e_reg = __ldg(p.offsets + bl + 1);
      }
    }
    const int src = static_cast<int>(k - kbase);
    s0 = __shfl_sync(0xffffffffu, s_reg, src);
    const int64_t e0 = __shfl_sync(0xffffffffu, e_reg, src);
    const bool bad = s0 < 0 || e0 < s0 || e0 > p.total_tokens || e0 - s0 > INT_MAX;
    if (bad && lane == 0) atomicOr(p.status, kDevErrBadInput);
    L = bad ? 0 : static_cast<int>(e0 - s0);
    return true;
  };
  auto make_step = [&](int64_t k, int qg, int j0) -> Step {
    Step st;
    st.k = k;
    st.qg = qg;
    st.j0 = j0;
    int64_t s0 = 0;
    int L = 0;
    st.valid = doc_range(k, s0, L);
    st.b = gw + k * nwarps;
    st.row0 = s0 + j0;
    st.n = min(pr, max(0, L - j0));
    st.first = j0 == 0;
    st.last = j0 + pr >= L;
    return st;
  };
  auto next_step = [&](const Step& st) -> Step {
    if (!st.last) return make_step(st.k, st.qg, st.j0 + pr);
    if (st.qg + 32 < nqp) return make_step(st.k, st.qg + 32, 0);
    return make_step(st.k + 1, 0, 0);
  };
  auto issue = [&](const Step& st, int bufi) {
    const uint32_t dst = stage_s + static_cast<uint32_t>(bufi * stage_bytes);
    const int chunks = d >> 4;                                 // 16-byte chunks per row
    for (int c = lane; c < st.n * chunks; c += 32) {
      const int r = c / chunks, cc = c - r * chunks;
      cp_async16(dst + r * pitch + cc * 16, p.D + (st.row0 + r) * d + cc * 16);
    }
    if (lane < st.n) cp_async4(dst + pr * pitch + lane * 4, p.d_scale + st.row0 + lane);
    cp_async_commit();
  };

  Step cur = make_step(0, 0, 0);
  int bufi = 0;
  if (cur.valid) issue(cur, 0);
  Best best[4][2];
  float score = 0.f;
  while (cur.valid) {
    const Step nxt = next_step(cur);
    if (nxt.valid) {
      issue(nxt, bufi ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    if (cur.first) {
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) best[n][h] = Best{-INFINITY, INT_MAX, 0};
    }
    const uint8_t* sb = stage + bufi * stage_bytes;
    const float* sc = reinterpret_cast<const float*>(sb + pr * pitch);
    for (int r0 = 0; r0 < cur.n; r0 += 16) {
      const int ra = r0 + g, rb = r0 + g + 8;
      const bool va = ra < cur.n, vb = rb < cur.n;
      const uint32_t* pa = reinterpret_cast<const uint32_t*>(sb + ra * pitch);
      const uint32_t* pb = reinterpret_cast<const uint32_t*>(sb + rb * pitch);
      uint32_t af[KC][4];
#pragma unroll
      for (int kc = 0; kc < KC; ++kc) {
        af[kc][0] = va ? pa[kc * 8 + t] : 0u;
        af[kc][1] = vb ? pb[kc * 8 + t] : 0u;
        af[kc][2] = va ? pa[kc * 8 + 4 + t] : 0u;
        af[kc][3] = vb ? pb[kc * 8 + 4 + t] : 0u;
      }
      const float sa = va ? sc[ra] : 0.f;
      const float sbv = vb ? sc[rb] : 0.f;
      const int ja = cur.j0 + ra, jb = cur.j0 + rb;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        int c[4] = {0, 0, 0, 0};
        const uint32_t* qrow = qs32 + (cur.qg + n * 8 + g) * dw;
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) imma_16832(c, af[kc], qrow[kc * 8 + t], qrow[kc * 8 + 4 + t]);
        // c0,c1: row ra, columns 2t, 2t+1; c2,c3: row rb
        if (va) {
          take(best[n][0], __fmul_rn(static_cast<float>(c[0]), sa), ja, c[0]);
          take(best[n][1], __fmul_rn(static_cast<float>(c[1]), sa), ja, c[1]);
        }
        if (vb) {
          take(best[n][0], __fmul_rn(static_cast<float>(c[2]), sbv), jb, c[2]);
          take(best[n][1], __fmul_rn(static_cast<float>(c[3]), sbv), jb, c[3]);
        }
      }
    }
    __syncwarp();  // this buffer is refilled two steps later
    if (cur.last) {
      const int L = cur.j0 + cur.n;
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
            const int qi = cur.qg + n * 8 + 2 * t + h;
            if (qi < p.nq) {
              const float mv = L > 0 ? best[n][h].v : 0.f;
              score = fmaf(__ldg(p.q_scale + qi), mv, score);
              if (DETAIL) {
                const int64_t o = cur.b * p.nq + qi;
                if (p.maxv) p.maxv[o] = mv;
                if (p.maxdot) p.maxdot[o] = L > 0 ? best[n][h].dot : 0;
                if (p.argmax) p.argmax[o] = L > 0 ? best[n][h].j : -1;
              }
            }
          }
      }
      if (cur.qg + 32 >= nqp) {  // document finished: sum over the 4 lanes holding partial scores
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) score += __shfl_xor_sync(0xffffffffu, score, o);
        if (lane == 0) p.out[cur.b] = score;
        score = 0.f;
      }
    }
    cur = nxt;
    bufi ^= 1;
  }
}

template <int KC>
cudaError_t launch_kc(const I8Params& p, bool detail, int grid, int threads, size_t smem, cudaStream_t stream) {
  cudaError_t e;
  if (detail) {
    e = cudaFuncSetAttribute(i8_score_kernel<KC, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8_score_kernel<KC, true><<<grid, threads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(i8_score_kernel<KC, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8_score_kernel<KC, false><<<grid, threads, smem, stream>>>(p);
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
  // scores only: documents on the tensor core's M dimension (exact dots)
  if (!maxv && !maxdot && !argmax && i8x_applicable(nq, d, total_tokens))
    return launch_i8x(Q, q_scale, nq, d, D, d_scale, offsets, B, total_tokens, out, stream);
  // d <= 256: the tcgen05 path (fp16 operands converted on chip, exact dots)
  if (i8tc_applicable(nq, d))
    return launch_i8tc(Q, q_scale, nq, d, D, d_scale, offsets, B, total_tokens, out, maxv, maxdot, argmax, stream);
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
  // largest block / piece that fits: 256, 128 or 64 threads; 32 or 16 rows per piece
  const size_t qbytes = static_cast<size_t>((nq + 31) & ~31) * d;
  int threads = 0, rows = 0;
  size_t smem = 0;
  for (int th = kI8Threads; th >= 64 && !threads; th /= 2)
    for (int r = kMaxPieceRows; r >= 16 && !threads; r /= 2) {
      const size_t need = qbytes + static_cast<size_t>(th / 32) * 2 * (static_cast<size_t>(r) * (d + 16) + r * 4);
      if (need <= static_cast<size_t>(dev->max_smem_optin)) {
        threads = th;
        rows = r;
        smem = need;
      }
    }
  if (!threads) return MAXSIM_ERR_UNSUPPORTED;
  p.piece_rows = rows;
  const int64_t want = static_cast<int64_t>(dev->sm_count) * 2 * (kI8Threads / threads);
  const int64_t warps = (B + threads / 32 - 1) / (threads / 32);
  const int grid = static_cast<int>(warps < want ? (warps < 1 ? 1 : warps) : want);
  const bool detail = maxv || maxdot || argmax;
  cudaError_t e;
  switch (d / 32) {
    case 2: e = launch_kc<2>(p, detail, grid, threads, smem, stream); break;
    case 4: e = launch_kc<4>(p, detail, grid, threads, smem, stream); break;
    case 6: e = launch_kc<6>(p, detail, grid, threads, smem, stream); break;
    case 8: e = launch_kc<8>(p, detail, grid, threads, smem, stream); break;
    case 12: e = launch_kc<12>(p, detail, grid, threads, smem, stream); break;
    case 16: e = launch_kc<16>(p, detail, grid, threads, smem, stream); break;
    case 24: e = launch_kc<24>(p, detail, grid, threads, smem, stream); break;
    case 32: e = launch_kc<32>(p, detail, grid, threads, smem, stream); break;
    default: return MAXSIM_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

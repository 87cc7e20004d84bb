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
// 32 consecutive bytes of the table per subspace. A warp walks its
// documents as pieces of <= 2 KB of codes, staged into a per-warp double
// buffer in shared memory with cp.async, so the next piece is in flight
// while the current one is scored; document offsets come 32 at a time.
// Lowest token index wins ties, as in the other paths.
//
// At M = 16, K = 256 (every code valid) a faster map is used. Lanes are
// (token slot ts = lane/2 of 16, query half h = lane%2 of 4 tokens), and one
// 128-bit load of a table row serves four query tokens. A row (code c,
// subspace m) is 32 B; with rows in [m][c] order its bank group (address / 32
// mod 4) would be c mod 4 -- random -- and the four rows that one quarter-warp
// (8 lanes) reads would collide about half the time. In shared memory the
// rows are therefore placed at c*16 + 4*(m%4) + m/4, so the bank group is the
// subspace quadrant m/4. Lane pair p = ts%4 of a quarter-warp walks the
// quadrants in the order p, p+1, p+2, p+3 (mod 4), so at every step its four
// pairs read four distinct bank groups: one wavefront per quarter-warp. Each
// quadrant's four terms are summed in order m from the first, and the token's
// similarity is (Q0 + Q1) + (Q2 + Q3) whatever the lane, so equal codes give
// equal scores and ties still go to the lowest token index.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kPqThreads = 512;
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

constexpr int kPieceBytes = 2048;   // codes staged per warp per piece (double-buffered)

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A piece: up to kPieceBytes / M consecutive tokens of one document.
struct Piece {
  int64_t b;      // document (-1: none)
  int64_t row0;   // first token row in codes
  int j0;         // doc-local index of the first token
  int n;          // tokens in the piece (0 for an empty or rejected document)
  bool last;      // the document's last piece
};

// Per-warp walk over documents b_first, b_first + stride, ... < b_end, with
// offsets fetched 32 documents at a time into registers (lane k holds doc k).
struct DocWalk {
  int64_t b_first, b_end, stride;
  int64_t kbase;         // index k of the documents currently held in registers
  int64_t s_reg, e_reg;  // this lane's document (k = kbase + lane)
  int cap;               // tokens per piece
  unsigned* status;
  const int64_t* offsets;
  int64_t total;

  __device__ __forceinline__ void load(int64_t k0) {
    kbase = k0;
    const int lane = threadIdx.x & 31;
    const int64_t b = b_first + (k0 + lane) * stride;
    s_reg = e_reg = 0;
    if (b < b_end) {
      s_reg = __ldg(offsets + b);
      e_reg = __ldg(offsets + b + 1);
    }
  }
  // First piece of document index k (k-th document of this warp).
  __device__ __forceinline__ Piece doc_piece(int64_t k, int j0) {
    Piece pc;
    pc.b = b_first + k * stride;
    if (pc.b >= b_end) {
      pc.b = -1;
      return pc;
    }
    if (k - kbase >= 32) load(k);
    const int src = static_cast<int>(k - kbase);
    const int64_t s0 = __shfl_sync(0xffffffffu, s_reg, src), e0 = __shfl_sync(0xffffffffu, e_reg, src);
    const bool bad = s0 < 0 || e0 < s0 || e0 > total || e0 - s0 > INT_MAX;
    if (bad && j0 == 0 && (threadIdx.x & 31) == 0) atomicOr(status, kDevErrBadInput);
    const int64_t L = bad ? 0 : e0 - s0;
    pc.row0 = s0 + j0;
    pc.j0 = j0;
    const int64_t left = L - j0;
    pc.n = static_cast<int>(left < cap ? (left > 0 ? left : 0) : cap);
    pc.last = j0 + pc.n >= L;
    return pc;
  }
};

// MWT = M / 4 code words per token (0: runtime M); FULLK: K == 256, so every
// uint8 code is a valid centroid and needs no clamp.
template <int MWT, bool FULLK, bool ARGMAX>
__global__ void __launch_bounds__(kPqThreads, 1) pq_score_kernel(const PqParams p) {
  extern __shared__ float4 pq_smem4[];
  float* Ts = reinterpret_cast<float*>(pq_smem4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tk = lane >> 3, ii = lane & 7;
  const int M = p.M, MW = MWT > 0 ? MWT : (M >> 2);
  const int K = FULLK ? 256 : p.K;
  const uint32_t kmax = static_cast<uint32_t>(K - 1);
  const int64_t b0 = (p.B * blockIdx.x) / gridDim.x, b1 = (p.B * (blockIdx.x + 1)) / gridDim.x;
  const int64_t tsize = static_cast<int64_t>(M) * K * kGroup;  // floats per table group
  uint32_t* stage = reinterpret_cast<uint32_t*>(Ts + tsize) + warp * (2 * kPieceBytes / 4);
  const uint32_t stage_s = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
  const int cap = kPieceBytes / M;
  // 16-byte copies need 16-byte rows and a 16-byte aligned codes base
  const bool vec16 = (M & 15) == 0 && (reinterpret_cast<uintptr_t>(p.codes) & 15) == 0;

  for (int g = 0; g < p.n_groups; ++g) {
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(p.T + g * tsize);
    if constexpr (MWT == 4 && FULLK) {
      // shared row c*16 + s holds subspace m = 4 (s % 4) + s / 4 of code c
      for (int e = tid; e < 16 * 256 * 2; e += kPqThreads) {
        const int row = e >> 1, c = row >> 4, sl = row & 15;
        const int m = 4 * (sl & 3) + (sl >> 2);
        pq_smem4[e] = __ldg(src + (m * 256 + c) * 2 + (e & 1));
      }
    } else {
      for (int64_t e = tid; e < tsize / 4; e += kPqThreads) pq_smem4[e] = __ldg(src + e);
    }
    __syncthreads();
    const int qi = g * kGroup + ii;

    DocWalk walk;
    walk.b_first = b0 + warp;
    walk.b_end = b1;
    walk.stride = kPqThreads / 32;
    walk.cap = cap;
    walk.status = p.status;
    walk.offsets = p.offsets;
    walk.total = p.total_tokens;
    walk.load(0);

    // stage the codes of a piece into buffer `bufi` of this warp
    auto issue = [&](const Piece& pc, int bufi) {
      const uint32_t dst = stage_s + static_cast<uint32_t>(bufi * kPieceBytes);
      const uint8_t* srcb = p.codes + pc.row0 * M;
      const int bytes = pc.n * M;
      if (vec16) {
        for (int o = lane * 16; o < bytes; o += 512) cp_async16(dst + o, srcb + o);
      } else {
        for (int o = lane * 4; o < bytes; o += 128) cp_async4(dst + o, srcb + o);
      }
      cp_async_commit();
    };

    int64_t k = 0;
    Piece cur = walk.doc_piece(0, 0);
    int bufi = 0;
    if (cur.b >= 0) issue(cur, 0);
    float rm = -INFINITY;
    int ra = INT_MAX;
    float rm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    int ra4[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX};
    bool badc = false;
    while (cur.b >= 0) {
      // the next piece: rest of this document, or the next document
      Piece nxt;
      if (!cur.last) {
        nxt = walk.doc_piece(k, cur.j0 + cur.n);
      } else {
        nxt = walk.doc_piece(k + 1, 0);
      }
      if (nxt.b >= 0) {
        issue(nxt, bufi ^ 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      // score the staged piece: token t = 4*it + tk
      const uint32_t* cw_base = stage + bufi * (kPieceBytes / 4);
      if constexpr (MWT == 4 && FULLK) {
        // token t = 16 * it + ts; query tokens 4 h .. 4 h + 3 of the group
        const int ts = lane >> 1, h = lane & 1, pr = ts & 3;
        const bool odd = pr & 1;
        int jo[4];  // float offset of quadrant (i + pr) % 4 and this lane's half of the row
#pragma unroll
        for (int i = 0; i < 4; ++i) jo[i] = ((i + pr) & 3) * 8 + 4 * h;
        for (int t = ts; t < cur.n; t += 16) {
          const uint4 cw = *reinterpret_cast<const uint4*>(cw_base + t * 4);
          // word i of rw: the codes of quadrant (i + pr) % 4
          uint32_t rw0 = cw.x, rw1 = cw.y, rw2 = cw.z, rw3 = cw.w;
          if (pr & 1) {
            const uint32_t x = rw0;
            rw0 = rw1;
            rw1 = rw2;
            rw2 = rw3;
            rw3 = x;
          }
          if (pr & 2) {
            uint32_t x = rw0;
            rw0 = rw2;
            rw2 = x;
            x = rw1;
            rw1 = rw3;
            rw3 = x;
          }
          const uint32_t rw[4] = {rw0, rw1, rw2, rw3};
          float acc[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int c = static_cast<int>((rw[i] >> (8 * r)) & 0xFFu);
              const float4 tv = *reinterpret_cast<const float4*>(Ts + c * 128 + 32 * r + jo[i]);
              if (r == 0) {
                acc[i][0] = tv.x;
                acc[i][1] = tv.y;
                acc[i][2] = tv.z;
                acc[i][3] = tv.w;
              } else {
                acc[i][0] += tv.x;
                acc[i][1] += tv.y;
                acc[i][2] += tv.z;
                acc[i][3] += tv.w;
              }
            }
          // acc[i] holds quadrant (i + pr) % 4; both pairings below equal (Q0 + Q1) + (Q2 + Q3)
          float s4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            s4[e] = (acc[0][e] + (odd ? acc[3][e] : acc[1][e])) + (acc[2][e] + (odd ? acc[1][e] : acc[3][e]));
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (s4[e] > rm4[e]) {  // tokens ascend per lane: strict > keeps the lowest index
              rm4[e] = s4[e];
              ra4[e] = cur.j0 + t;
            }
        }
        __syncwarp();  // the buffer is refilled two pieces later
        if (cur.last) {
          // max over the 16 token slots (lanes with the same query half)
#pragma unroll
          for (int o = 2; o <= 16; o <<= 1)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float v2 = __shfl_xor_sync(0xffffffffu, rm4[e], o);
              const int i2 = __shfl_xor_sync(0xffffffffu, ra4[e], o);
              if (v2 > rm4[e] || (v2 == rm4[e] && i2 < ra4[e])) {
                rm4[e] = v2;
                ra4[e] = i2;
              }
            }
          const bool nonempty = cur.j0 + cur.n > 0;
          float pe[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = g * kGroup + 4 * h + e;
            pe[e] = (nonempty && q < p.nq) ? rm4[e] : 0.f;
            if (ARGMAX && ts == 0 && q < p.nq) p.argmax[cur.b * p.nq + q] = nonempty ? ra4[e] : -1;
          }
          // ((q0 + q1) + (q2 + q3)) + ((q4 + q5) + (q6 + q7))
          float part = (pe[0] + pe[1]) + (pe[2] + pe[3]);
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          if (lane == 0) p.out[cur.b] = (g == 0 ? 0.f : p.out[cur.b]) + part;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            rm4[e] = -INFINITY;
            ra4[e] = INT_MAX;
          }
          ++k;
        }
      } else {
        const float* Tl = Ts + ii;   // this lane's query token within the 8-token group
        for (int t = tk; t < cur.n; t += 4) {
          float s = 0.f;
          if (MWT > 0) {
            uint32_t cw[MWT > 0 ? MWT : 1];
            if (MWT % 4 == 0) {
#pragma unroll
              for (int w = 0; w < MWT; w += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(cw_base + t * MWT + w);
                cw[w] = v.x;
                cw[w + 1] = v.y;
                cw[w + 2] = v.z;
                cw[w + 3] = v.w;
              }
            } else {
#pragma unroll
              for (int w = 0; w < MWT; ++w) cw[w] = cw_base[t * MWT + w];
            }
#pragma unroll
            for (int w = 0; w < MWT; ++w) {
#pragma unroll
              for (int sb = 0; sb < 4; ++sb) {
                const int m = 4 * w + sb;
                uint32_t c = (cw[w] >> (8 * sb)) & 0xFFu;
                if (!FULLK) {
                  badc |= c > kmax;  // a code outside the codebook is clamped and reported
                  c = min(c, kmax);
                }
                s += Tl[(m * K) * kGroup + static_cast<int>(c) * kGroup];
              }
            }
          } else {
            for (int w = 0; w < MW; ++w) {
              const uint32_t word = cw_base[t * MW + w];
#pragma unroll
              for (int sb = 0; sb < 4; ++sb) {
                const int m = 4 * w + sb;
                uint32_t c = (word >> (8 * sb)) & 0xFFu;
                if (!FULLK) {
                  badc |= c > kmax;
                  c = min(c, kmax);
                }
                s += Tl[(m * K + static_cast<int>(c)) * kGroup];
              }
            }
          }
          if (s > rm) {  // tokens ascend per lane: strict > keeps the lowest index
            rm = s;
            ra = cur.j0 + t;
          }
        }
        __syncwarp();  // the buffer is refilled two pieces later
        if (cur.last) {
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
          const bool nonempty = cur.j0 + cur.n > 0;
          float part = (nonempty && qi < p.nq) ? rm : 0.f;
          if (ARGMAX && tk == 0 && qi < p.nq) p.argmax[cur.b * p.nq + qi] = nonempty ? ra : -1;
#pragma unroll
          for (int o = 1; o <= 4; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (lane == 0) p.out[cur.b] = (g == 0 ? 0.f : p.out[cur.b]) + part;
          rm = -INFINITY;
          ra = INT_MAX;
          ++k;
        }
      }
      cur = nxt;
      bufi ^= 1;
    }
    if (__any_sync(0xffffffffu, badc) && lane == 0 && g == 0) atomicOr(p.status, kDevErrBadInput);
  }
}

template <int MWT, bool FULLK, bool ARGMAX>
cudaError_t launch_pq_one(const PqParams& p, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(pq_score_kernel<MWT, FULLK, ARGMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  pq_score_kernel<MWT, FULLK, ARGMAX><<<grid, kPqThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int MWT>
cudaError_t launch_pq_kernel(const PqParams& p, bool fullk, bool argmax, int grid, size_t smem, cudaStream_t stream) {
  if (fullk) return argmax ? launch_pq_one<MWT, true, true>(p, grid, smem, stream)
                           : launch_pq_one<MWT, true, false>(p, grid, smem, stream);
  return argmax ? launch_pq_one<MWT, false, true>(p, grid, smem, stream)
                : launch_pq_one<MWT, false, false>(p, grid, smem, stream);
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
  const size_t smem = static_cast<size_t>(M) * K * kGroup * sizeof(float) +
                      static_cast<size_t>(kPqThreads / 32) * 2 * kPieceBytes;
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
  const bool fullk = K == 256;
  cudaError_t e;
  switch (M / 4) {
    case 1: e = launch_pq_kernel<1>(p, fullk, argmax != nullptr, grid, smem, stream); break;
    case 2: e = launch_pq_kernel<2>(p, fullk, argmax != nullptr, grid, smem, stream); break;
    case 4: e = launch_pq_kernel<4>(p, fullk, argmax != nullptr, grid, smem, stream); break;
    case 8: e = launch_pq_kernel<8>(p, fullk, argmax != nullptr, grid, smem, stream); break;
    case 16: e = launch_pq_kernel<16>(p, fullk, argmax != nullptr, grid, smem, stream); break;
    default: e = launch_pq_kernel<0>(p, fullk, argmax != nullptr, grid, smem, stream); break;
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

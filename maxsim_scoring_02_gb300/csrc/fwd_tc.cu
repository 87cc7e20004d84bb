// fwd_tc.cu -- MaxSim forward on the 5th-generation tensor cores (tcgen05).
//
// Computes, for every (query q, document b):
//   out[q,b]      = sum_i max_{j < L_b} <Q[q,i,:], D_b[j,:]>
//   argmax[q,b,i] = lowest j attaining that maximum
// (TileMaxSim deep reading §1; FLASH-MAXSIM Figure 1 / Algorithm 2).
//
// Design (GB300 / sm_103a):
//  * Persistent grid, one CTA per SM; CTA c owns a contiguous document range,
//    so it streams one contiguous slab of D and every document byte is read
//    from HBM exactly once per (query, query-chunk) -- with one query of up
//    to 256 tokens that is the single pass of TileMaxSim §2(1) (BQ = Nq).
//  * Warp 4 (one lane) is the TMA producer: 128-token x 64-dim boxes,
//    128-byte swizzled, into a ring of 16 KB stages. Partial tiles (the tail
//    of a document) load only ceil(rows/32)*32 rows, so padding beyond that
//    granule is never read (TileMaxSim §5, the padding waste).
//  * Warp 5 (one lane) issues tcgen05.mma kind::f16, M = 128 document tokens,
//    N = NC query tokens, K = 16 per instruction, accumulating every 64-wide
//    d-slice of the tile into the same TMEM accumulator before any maximum is
//    taken (TileMaxSim §2(2), dimension tiling). Several TMEM accumulators
//    let the tensor core run ahead of the epilogue.
//  * Warps 0-3 read the accumulator (TMEM lane = document token, column =
//    query token) with tcgen05.ld, mask tokens outside the document to -inf,
//    and reduce the 32 rows a warp holds with a transpose butterfly of
//    shuffles, leaving lane l with the maximum (and lowest argmax) of query
//    column l. Per-warp partial maxima persist across the document's tiles in
//    registers; at the document end the four warps combine through shared
//    memory and the per-token maxima are summed. The Nq x Nd similarity tile
//    exists only in TMEM and registers.
//  * Every mbarrier wait is bounded (see ptx.cuh); after an abort the
//    producer drains its in-flight TMA loads and the MMA warp waits for its
//    last MMA before TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kThreads = 192;        // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kStageBytes = 16384;   // 128 rows x 64 elements x 2 bytes
constexpr int kTileRows = 128;
constexpr int kRowGranule = 32;      // rows per TMA box for partial tiles
constexpr int kMaxAcc = 4;

struct FwdTcParams {
  const int32_t* doc_len;   // padded layout, may be null
  const int64_t* offsets;   // CSR layout
  int64_t B;
  int64_t total_rows;
  int nd;
  int csr;
  int n_queries;
  int nq;
  int KB;          // d / 64
  int n_chunks;    // ceil(nq / NC)
  int stages;
  int n_acc;
  int n_qslots;
  uint32_t idesc;
  uint32_t tmem_cols;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

// Rows of document b: returns L_b and sets start; a document whose
// description is out of range is reported as bad and treated as empty.
__device__ __forceinline__ int64_t doc_rows(const FwdTcParams& p, int64_t b, int64_t& start, bool& bad) {
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

struct Smem {
  uint8_t* q;         // n_qslots x KB boxes of NC rows x 128 B
  uint8_t* stages;    // stages x 16 KB
  uint64_t* full;
  uint64_t* empty;
  uint64_t* qfull;    // [2]
  uint64_t* qempty;   // [2]
  uint64_t* accfull;  // [n_acc]
  uint64_t* accempty; // [n_acc]
  uint64_t* done;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* red_v;       // [2][4][NC]
  int32_t* red_i;     // [2][4][NC]
  float* sred;        // [2][4]
};

__host__ __device__ inline size_t smem_bytes_for(int NC, int KB, int stages, int n_acc, int n_qslots) {
  size_t bytes = 1024;  // alignment slack for the dynamic region
  bytes += static_cast<size_t>(n_qslots) * KB * NC * 128;
  bytes += static_cast<size_t>(stages) * kStageBytes;
  bytes += static_cast<size_t>(2 * stages + 4 + 2 * n_acc + 1) * 8;
  bytes += 16;  // tmem slot + abort flag (+pad)
  bytes += static_cast<size_t>(2 * 4 * NC) * 8;  // red_v + red_i
  bytes += 2 * 4 * 4;
  return bytes;
}

__device__ __forceinline__ Smem carve(uint8_t* raw, const FwdTcParams& p, int NC) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.q = base;
  s.stages = s.q + static_cast<size_t>(p.n_qslots) * p.KB * NC * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.stages + static_cast<size_t>(p.stages) * kStageBytes);
  s.full = bars;
  s.empty = s.full + p.stages;
  s.qfull = s.empty + p.stages;
  s.qempty = s.qfull + 2;
  s.accfull = s.qempty + 2;
  s.accempty = s.accfull + p.n_acc;
  s.done = s.accempty + p.n_acc;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.done + 1);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.red_v = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.red_i = reinterpret_cast<int32_t*>(s.red_v + 2 * 4 * NC);
  s.sred = reinterpret_cast<float*>(s.red_i + 2 * 4 * NC);
  return s;
}

// ------------------------------------------------------------ producer warp
template <int NC>
__device__ void run_producer(const FwdTcParams& p, const Smem& sm, const CUtensorMap* tm_d128,
                             const CUtensorMap* tm_d32, const CUtensorMap* tm_q, int64_t b0, int64_t b1) {
  const int S = p.stages, KB = p.KB, NQS = p.n_qslots;
  const uint32_t qbytes = static_cast<uint32_t>(KB) * NC * 128;
  const uint64_t policy = l2_policy_evict_first();
  uint32_t fill = 0, quse = 0;
  int prev_key = -1;
  for (int64_t b = b0; b < b1; ++b) {
    int64_t start;
    bool bad;
    const int64_t L = doc_rows(p, b, start, bad);
    if (L == 0) continue;
    const int ntiles = static_cast<int>((L + kTileRows - 1) / kTileRows);
    for (int q = 0; q < p.n_queries; ++q) {
      for (int c = 0; c < p.n_chunks; ++c) {
        const int key = q * p.n_chunks + c;
        if (key != prev_key) {
          const int slot = static_cast<int>(quse % NQS);
          const uint32_t use = quse / NQS;
          if (use > 0 && !mbar_wait(&sm.qempty[slot], (use - 1) & 1u, sm.abort_flag, p.status)) goto drain;
          mbar_arrive_expect_tx(&sm.qfull[slot], qbytes);
          for (int kb = 0; kb < KB; ++kb)
            tma_load_3d(sm.q + (static_cast<size_t>(slot) * KB + kb) * NC * 128, tm_q, &sm.qfull[slot], kb * 64,
                        c * NC, q);
          ++quse;
          prev_key = key;
        }
        for (int t = 0; t < ntiles; ++t) {
          const int64_t row0 = start + static_cast<int64_t>(t) * kTileRows;
          const int64_t left = L - static_cast<int64_t>(t) * kTileRows;
          const int rows = left >= kTileRows ? kTileRows : static_cast<int>(left);
          const int rows_ld = rows == kTileRows ? kTileRows : ((rows + kRowGranule - 1) / kRowGranule) * kRowGranule;
          for (int kb = 0; kb < KB; ++kb) {
            const int s = static_cast<int>(fill % S);
            const uint32_t ph = (fill / S) & 1u;
            if (!mbar_wait(&sm.empty[s], ph ^ 1u, sm.abort_flag, p.status)) goto drain;
            mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(rows_ld) * 128u);
            uint8_t* dst = sm.stages + static_cast<size_t>(s) * kStageBytes;
            if (rows_ld == kTileRows) {
              tma_load_2d_hint(dst, tm_d128, &sm.full[s], kb * 64, static_cast<int>(row0), policy);
            } else {
              for (int r = 0; r < rows_ld; r += kRowGranule)
                tma_load_2d_hint(dst + r * 128, tm_d32, &sm.full[s], kb * 64, static_cast<int>(row0 + r), policy);
            }
            ++fill;
          }
        }
      }
    }
  }
  return;
drain:
  // After an abort: wait (bounded) for every load this warp may still have in flight.
  for (uint32_t f = fill > static_cast<uint32_t>(S) ? fill - S : 0; f < fill; ++f)
    mbar_wait_drain(&sm.full[f % S], (f / S) & 1u, p.status);
  for (uint32_t u = quse > static_cast<uint32_t>(NQS) ? quse - NQS : 0; u < quse; ++u)
    mbar_wait_drain(&sm.qfull[u % NQS], (u / NQS) & 1u, p.status);
}

// ----------------------------------------------------------------- MMA warp
template <int NC>
__device__ void run_mma(const FwdTcParams& p, const Smem& sm, uint32_t tmem_base, int64_t b0, int64_t b1) {
  const int S = p.stages, KB = p.KB, NQS = p.n_qslots, A = p.n_acc;
  uint32_t fill = 0, quse = 0, acc = 0;
  int prev_key = -1, slot = 0;
  for (int64_t b = b0; b < b1; ++b) {
    int64_t start;
    bool bad;
    const int64_t L = doc_rows(p, b, start, bad);
    if (L == 0) continue;
    const int ntiles = static_cast<int>((L + kTileRows - 1) / kTileRows);
    for (int q = 0; q < p.n_queries; ++q) {
      for (int c = 0; c < p.n_chunks; ++c) {
        const int key = q * p.n_chunks + c;
        if (key != prev_key) {
          if (prev_key >= 0) umma_commit(&sm.qempty[slot]);  // slot free once its MMAs retire
          slot = static_cast<int>(quse % NQS);
          if (!mbar_wait(&sm.qfull[slot], (quse / NQS) & 1u, sm.abort_flag, p.status)) goto drain;
          tc_fence_after();
          ++quse;
          prev_key = key;
        }
        const uint32_t qbase = smem_u32(sm.q + static_cast<size_t>(slot) * KB * NC * 128);
        for (int t = 0; t < ntiles; ++t) {
          const int a = static_cast<int>(acc % A);
          if (!mbar_wait(&sm.accempty[a], ((acc / A) & 1u) ^ 1u, sm.abort_flag, p.status)) goto drain;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * NC);
          for (int kb = 0; kb < KB; ++kb) {
            const int s = static_cast<int>(fill % S);
            if (!mbar_wait(&sm.full[s], (fill / S) & 1u, sm.abort_flag, p.status)) goto drain;
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm.stages + static_cast<size_t>(s) * kStageBytes);
            const uint32_t b_addr = qbase + static_cast<uint32_t>(kb * NC * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16(d_tmem, sdesc_k_sw128(a_addr + kk * 32), sdesc_k_sw128(b_addr + kk * 32), p.idesc,
                       (kb | kk) != 0 ? 1u : 0u);
            umma_commit(&sm.empty[s]);  // stage reusable once these MMAs have read it
            ++fill;
          }
          umma_commit(&sm.accfull[a]);  // accumulator ready for the epilogue
          ++acc;
        }
      }
    }
  }
drain:
  // Wait until every MMA issued by this thread has completed before TMEM is freed.
  umma_commit(sm.done);
  mbar_wait_drain(sm.done, 0, p.status);
}

// Max over the 32 lanes of a warp for each of 32 columns: on return lane l
// holds the maximum of column l (and, with ARGMAX, the lowest row index
// attaining it). 31 shuffle rounds per value array.
template <bool ARGMAX>
__device__ __forceinline__ void warp_column_max(float (&v)[32], int row, int lane, float& out_v, int& out_i) {
  int ix[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) ix[k] = row;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = upper ? v[k] : v[k + w];
      const float keep = upper ? v[k + w] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      if (ARGMAX) {
        const int isend = upper ? ix[k] : ix[k + w];
        const int ikeep = upper ? ix[k + w] : ix[k];
        const int irecv = __shfl_xor_sync(0xffffffffu, isend, w);
        const bool take = (recv > keep) || (recv == keep && irecv < ikeep);
        v[k] = take ? recv : keep;
        ix[k] = take ? irecv : ikeep;
      } else {
        v[k] = fmaxf(keep, recv);
      }
    }
  }
  out_v = v[0];
  out_i = ix[0];
}

// ------------------------------------------------------------ epilogue warps
template <int NG, bool ARGMAX>
__device__ void run_epilogue(const FwdTcParams& p, const Smem& sm, uint32_t tmem_base, int64_t b0, int64_t b1) {
  constexpr int NC = 32 * NG;
  const int tid = threadIdx.x;  // 0..127 == TMEM lane
  const int warp = tid >> 5, lane = tid & 31;
  const int A = p.n_acc;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  uint32_t acc = 0;
  int rb = 0;
  for (int64_t b = b0; b < b1; ++b) {
    int64_t start;
    bool bad;
    const int64_t L = doc_rows(p, b, start, bad);
    if (bad && tid == 0) atomicOr(p.status, kDevErrBadInput);
    const int ntiles = static_cast<int>((L + kTileRows - 1) / kTileRows);
    for (int q = 0; q < p.n_queries; ++q) {
      float qsum = 0.f;
      for (int c = 0; c < p.n_chunks; ++c) {
        if (L == 0) {
          if (ARGMAX)
            for (int col = tid; col < NC; col += 128) {
              const int qc = c * NC + col;
              if (qc < p.nq) p.argmax[(static_cast<int64_t>(q) * p.B + b) * p.nq + qc] = -1;
            }
          continue;
        }
        float rm[NG];
        int ra[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          rm[g] = -INFINITY;
          ra[g] = INT_MAX;
        }
        for (int t = 0; t < ntiles; ++t) {
          const int a = static_cast<int>(acc % A);
          if (!mbar_wait(&sm.accfull[a], (acc / A) & 1u, sm.abort_flag, p.status)) return;
          tc_fence_after();
          const int row = t * kTileRows + tid;
          const bool valid = row < L;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            float v[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(a * NC + g * 32), v);
            if (!valid) {
#pragma unroll
              for (int k = 0; k < 32; ++k) v[k] = -INFINITY;
            }
            float bv;
            int bi;
            warp_column_max<ARGMAX>(v, row, lane, bv, bi);
            if (ARGMAX) {
              if (bv > rm[g] || (bv == rm[g] && bi < ra[g])) {
                rm[g] = bv;
                ra[g] = bi;
              }
            } else {
              rm[g] = fmaxf(rm[g], bv);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.accempty[a]);
          ++acc;
        }
        // Combine the four warps' partial maxima, then sum the query tokens.
        float* rv = sm.red_v + rb * 4 * NC;
        int32_t* ri = sm.red_i + rb * 4 * NC;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          rv[warp * NC + g * 32 + lane] = rm[g];
          if (ARGMAX) ri[warp * NC + g * 32 + lane] = ra[g];
        }
        named_bar_sync(1, 128);
        float part = 0.f;
        for (int col = tid; col < NC; col += 128) {
          float bv = rv[col];
          int bi = ARGMAX ? ri[col] : 0;
#pragma unroll
          for (int w = 1; w < 4; ++w) {
            const float v2 = rv[w * NC + col];
            if (ARGMAX) {
              const int i2 = ri[w * NC + col];
              if (v2 > bv || (v2 == bv && i2 < bi)) {
                bv = v2;
                bi = i2;
              }
            } else {
              bv = fmaxf(bv, v2);
            }
          }
          const int qc = c * NC + col;
          if (qc < p.nq) {
            part += bv;
            if (ARGMAX) p.argmax[(static_cast<int64_t>(q) * p.B + b) * p.nq + qc] = bi;
          }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (NC <= 32) {
          if (tid == 0) qsum += part;
        } else {
          if (lane == 0) sm.sred[rb * 4 + warp] = part;
          named_bar_sync(2, 128);
          if (tid == 0) qsum += (sm.sred[rb * 4 + 0] + sm.sred[rb * 4 + 1]) + (sm.sred[rb * 4 + 2] + sm.sred[rb * 4 + 3]);
        }
        rb ^= 1;
      }
      if (tid == 0) p.out[static_cast<int64_t>(q) * p.B + b] = qsum;
    }
  }
}

template <int NG, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_d128, const __grid_constant__ CUtensorMap tm_d32,
                  const __grid_constant__ CUtensorMap tm_q, const FwdTcParams p) {
  constexpr int NC = 32 * NG;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve(smem_raw, p, NC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.qfull[i], 1);
      mbar_init(&sm.qempty[i], 1);
    }
    for (int a = 0; a < p.n_acc; ++a) {
      mbar_init(&sm.accfull[a], 1);
      mbar_init(&sm.accempty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(sm.done, 1);
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_d128);
    tma_prefetch_desc(&tm_d32);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 5) {
    tmem_alloc(sm.tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  const int64_t b0 = (p.B * blockIdx.x) / gridDim.x;
  const int64_t b1 = (p.B * (blockIdx.x + 1)) / gridDim.x;

  if (warp == 4) {
    if (lane == 0) run_producer<NC>(p, sm, &tm_d128, &tm_d32, &tm_q, b0, b1);
  } else if (warp == 5) {
    if (lane == 0) run_mma<NC>(p, sm, tmem_base, b0, b1);
  } else {
    run_epilogue<NG, ARGMAX>(p, sm, tmem_base, b0, b1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int NG, bool ARGMAX>
cudaError_t launch_variant(const CUtensorMap& d128, const CUtensorMap& d32, const CUtensorMap& tq,
                           const FwdTcParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = fwd_tc_kernel<NG, ARGMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(d128, d32, tq, p);
  return cudaGetLastError();
}

}  // namespace

maxsim_status launch_fwd_tc(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows,
                            int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                            int is_bf16, float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (d % 64 != 0 || d < 64 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  if (total_rows < 1 || total_rows > static_cast<int64_t>(INT_MAX)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;

  // Query chunk width NC = 32 * NG: as wide as nq needs (up to 256 columns,
  // the largest N of one MMA), but the resident query chunk stays <= 96 KB.
  int ng_need = (nq + 31) / 32;
  int ng_cap = static_cast<int>((96 * 1024) / (static_cast<size_t>(KB) * 4096));
  if (ng_cap < 1) ng_cap = 1;
  int NG = 1;
  while (NG < ng_need && NG < 8 && NG * 2 <= ng_cap) NG *= 2;
  const int NC = 32 * NG;
  const int n_chunks = (nq + NC - 1) / NC;
  const int n_acc = (512 / NC) < kMaxAcc ? (512 / NC) : kMaxAcc;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(n_acc * NC)) tmem_cols <<= 1;

  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  const size_t qslot = static_cast<size_t>(KB) * NC * 128;
  int n_qslots = 1;
  if (n_queries * n_chunks > 1 && smem_bytes_for(NC, KB, 6, n_acc, 2) <= budget) n_qslots = 2;
  int stages = 16;
  while (stages > 2 && smem_bytes_for(NC, KB, stages, n_acc, n_qslots) > budget) --stages;
  const size_t smem = smem_bytes_for(NC, KB, stages, n_acc, n_qslots);
  if (smem > budget) return MAXSIM_ERR_UNSUPPORTED;
  (void)qslot;

  // TMA descriptors: documents as a [total_rows, d] matrix (two box heights)
  // and queries as [n_queries, nq, d] so rows past nq read as zero.
  alignas(64) CUtensorMap tm_d128, tm_d32, tm_q;
  const int dt = is_bf16 ? 1 : 0;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_rows)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t box128[2] = {64, 128}, box32[2] = {64, 32};
  const uint64_t qdims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(nq), static_cast<uint64_t>(n_queries)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(nq) * d * 2};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(NC), 1};
  if (!encode_tmap(&tm_d128, dt, 2, const_cast<void*>(D), ddims, dstrides, box128, 1) ||
      !encode_tmap(&tm_d32, dt, 2, const_cast<void*>(D), ddims, dstrides, box32, 1) ||
      !encode_tmap(&tm_q, dt, 3, const_cast<void*>(Q), qdims, qstrides, qbox, 1))
    return MAXSIM_ERR_CUDA;

  FwdTcParams p;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = n_queries;
  p.nq = nq;
  p.KB = KB;
  p.n_chunks = n_chunks;
  p.stages = stages;
  p.n_acc = n_acc;
  p.n_qslots = n_qslots;
  p.idesc = idesc_f16(is_bf16, 128, NC);
  p.tmem_cols = tmem_cols;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  cudaError_t e;
  const bool am = argmax != nullptr;
  switch (NG) {
    case 1: e = am ? launch_variant<1, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream)
                   : launch_variant<1, false>(tm_d128, tm_d32, tm_q, p, grid, smem, stream); break;
    case 2: e = am ? launch_variant<2, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream)
                   : launch_variant<2, false>(tm_d128, tm_d32, tm_q, p, grid, smem, stream); break;
    case 4: e = am ? launch_variant<4, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream)
                   : launch_variant<4, false>(tm_d128, tm_d32, tm_q, p, grid, smem, stream); break;
    default: e = am ? launch_variant<8, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream)
                    : launch_variant<8, false>(tm_d128, tm_d32, tm_q, p, grid, smem, stream); break;
  }
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

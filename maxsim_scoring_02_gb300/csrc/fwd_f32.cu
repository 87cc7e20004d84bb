// fwd_f32.cu -- MaxSim forward with fp32 inputs on the CUDA cores (FFMA).
//
// Same operator and outputs as the tensor-core path (TileMaxSim deep
// reading §1; FLASH-MAXSIM Figure 1 / Algorithm 2), for fp32 embeddings that
// must be scored at fp32 accuracy: TF32 tensor-core inputs would round every
// element to 10 mantissa bits, far outside an fp32 score tolerance, so the
// products are formed with FFMA. At 16 FLOP per document byte the op sits
// above the FP32 ridge of the part (~12 FLOP/B), so the FFMA pipe bounds it.
//
// Work unit: a group of four documents (4 g .. 4 g + 3) scored against one
// 32-token query chunk; the CTA tile is the chunk x four 128-token document
// tiles (tile t of each document), accumulated over 32-dim slices of d.
//
// Roles (320 threads, one CTA per SM):
//  * Producer (warp 8, lane 0): TMA loads of the 32-dim slice of the four
//    document tiles (4 x 16 KB, 128-byte swizzle) into a ring of kStages
//    stages; a document with no tile t is not loaded.
//  * Query transposer (warp 9): writes the chunk's 32 x 32 query slice into
//    the same stage k-major (one 36-float row per dim), read from global
//    memory with coalesced loads (lane = dim).
//  * Consumers (warps 0-7): warps 2u and 2u + 1 own document u of the group,
//    64 tokens each; a thread holds an 8 x 8 register tile of dot products:
//    query rows 4 lm + r and 16 + 4 lm + r (r < 4), tokens 64 wn + ln + 8 m
//    (m < 8), lane = 8 lm + ln. Per 4-dim chunk it loads 8 float4 of the
//    k-major query slice and 8 float4 of document rows, then issues 256 FFMA
//    ordered (dim, token, row). With the query slice k-major, the changing
//    query operand of consecutive FFMAs alternates register banks with the
//    row, so each accumulator needs one fixed bank; with both operands
//    token-major it would clash on half of them (measured: 84 against 104
//    FMA/clk/SM in isolation). A 128-bit shared load costs two wavefronts
//    when each even/odd lane pair reads one address, four otherwise: 48
//    wavefronts per 256 FFMA per warp, under the 64 cycles of FMA pipe they
//    need. The chunk loop is not unrolled: larger bodies lose more to
//    instruction fetch than they save.
//  * After the last d-slice of a tile, each thread folds its tile into running
//    maxima (tokens ascending, so the lowest index wins ties); after the last
//    tile a butterfly over the 8 token lanes and a hand-off through shared
//    memory let warp 2u take the maximum over its document's two warps, write
//    the argmax and add the chunk's sum into the query's score.
// Every wait is a bounded mbarrier wait; a timeout sets MAXSIM_DEVERR_TIMEOUT
// and the kernel drains its loads in flight and exits.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kProducerWarp = kConsumerWarps;       // TMA of the document tiles
constexpr int kQWarp = kConsumerWarps + 1;          // k-major copy of the query slice
constexpr int kThreads = kConsumers + 64;
constexpr int kGroup = 4;                        // documents per work unit
constexpr int kQC = 32;                          // query tokens per chunk
constexpr int kTT = 128;                         // document tokens per tile
constexpr int kKC = 32;                          // d per stage (one 128-byte swizzle row)
constexpr int kStages = 3;
// Hand-off buffers for the per-document maximum: a consumer warp can finish up
// to kStages items ahead of the warp that combines (one stage per item), so
// kStages + 1 buffers keep every buffer's contents read before it is rewritten.
constexpr int kRed = kStages + 1;
// Query slice, k-major: kKC rows (one per k) of the chunk's 32 query tokens,
// padded to 36 floats so the transposing writes spread over the banks.
constexpr int kQPitch = kQC + 4;
constexpr uint32_t kQBytes = 5120;               // kKC x kQPitch x 4 = 4608, rounded up to 1 KB
constexpr uint32_t kDBytes = kTT * kKC * 4;      // 16 KB per document tile
constexpr uint32_t kStageBytes = kQBytes + kGroup * kDBytes;
static_assert(kKC * kQPitch * 4 <= kQBytes, "query slice");

struct F32Params {
  const int32_t* doc_len;
  const int64_t* offsets;
  int64_t B;
  int64_t n_groups;
  int64_t total_rows;
  int nd, csr, n_queries, nq, d;
  int evict_first;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

struct F32Smem {
  uint8_t* stage;     // kStages x (Q slice, 4 D slices), 1024-byte aligned
  float* red_v;       // [kRed][8 warps][32 rows]
  int* red_i;         // [kRed][8 warps][32 rows]
  uint64_t* full;     // [kStages]
  uint64_t* empty;    // [kStages]
  uint64_t* redfull;  // [kRed]
  int* abort_flag;
};

size_t f32_smem_bytes() {
  return 1024 + static_cast<size_t>(kStages) * kStageBytes + 2u * kRed * kConsumerWarps * 32 * 4 +
         (2u * kStages + kRed) * 8 + 16;
}

__device__ __forceinline__ F32Smem f32_carve(uint8_t* raw) {
  F32Smem s;
  s.stage = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.red_v = reinterpret_cast<float*>(s.stage + kStages * kStageBytes);
  s.red_i = reinterpret_cast<int*>(s.red_v + kRed * kConsumerWarps * 32);
  s.full = reinterpret_cast<uint64_t*>(s.red_i + kRed * kConsumerWarps * 32);
  s.empty = s.full + kStages;
  s.redfull = s.empty + kStages;
  s.abort_flag = reinterpret_cast<int*>(s.redfull + kRed);
  return s;
}

template <int OFF>
__device__ __forceinline__ float4 lds128(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4+%5];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}

// Tokens of document b and its first row; bad offsets / lengths give 0 tokens.
__device__ __forceinline__ int f32_doc_rows(const F32Params& p, int64_t b, int64_t& start, bool& bad) {
  bad = false;
  start = 0;
  if (b >= p.B) return 0;
  if (p.csr) {
    const int64_t s = __ldg(p.offsets + b), e = __ldg(p.offsets + b + 1);
    if (s < 0 || e < s || e > p.total_rows || e - s > INT_MAX) {
      bad = true;
      return 0;
    }
    start = s;
    return static_cast<int>(e - s);
  }
  start = b * static_cast<int64_t>(p.nd);
  const int64_t L = p.doc_len ? static_cast<int64_t>(__ldg(p.doc_len + b)) : static_cast<int64_t>(p.nd);
  if (L < 0 || L > p.nd) {
    bad = true;
    return 0;
  }
  return static_cast<int>(L);
}

// Producer: walks the same (group, query, chunk, tile, d-slice) sequence as the
// consumers and fills the ring with the document slices.
__device__ void f32_producer(const CUtensorMap* tm_d, const F32Params& p, const F32Smem& sm) {
  const int n_qc = (p.nq + kQC - 1) / kQC;
  const int KC = (p.d + kKC - 1) / kKC;
  const uint64_t policy = l2_policy_evict_first();
  const bool ef = p.evict_first != 0;
  const uint32_t stage0 = smem_u32(sm.stage), full0 = smem_u32(sm.full), empty0 = smem_u32(sm.empty);
  uint32_t slot = 0, phase = 0;
  int64_t issued = 0;
  bool ok = true;
  for (int64_t g = blockIdx.x; ok && g < p.n_groups; g += gridDim.x) {
    int64_t start[kGroup];
    int T[kGroup], Tmax = 0;
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      bool bad;
      const int L = f32_doc_rows(p, g * kGroup + u, start[u], bad);
      T[u] = (L + kTT - 1) / kTT;
      Tmax = T[u] > Tmax ? T[u] : Tmax;
    }
    if (Tmax == 0) continue;
    for (int q = 0; ok && q < p.n_queries; ++q)
      for (int qc = 0; ok && qc < n_qc; ++qc) {
        for (int t = 0; ok && t < Tmax; ++t) {
          uint32_t tx = 0;
#pragma unroll
          for (int u = 0; u < kGroup; ++u) tx += t < T[u] ? kDBytes : 0u;
          for (int kc = 0; kc < KC; ++kc) {
            if (!mbar_wait_a(empty0 + 8 * slot, phase ^ 1u, sm.abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t full = full0 + 8 * slot, dst = stage0 + slot * kStageBytes;
            mbar_arrive_expect_tx_a(full, tx);
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
              if (t >= T[u]) continue;
              const int drow = static_cast<int>(start[u] + static_cast<int64_t>(t) * kTT);
              const uint32_t ddst = dst + kQBytes + u * kDBytes;
              if (ef)
                tma_load_2d_a(ddst, tm_d, full, kc * kKC, drow, policy);
              else
                tma_load_2d_nohint_a(ddst, tm_d, full, kc * kKC, drow);
            }
            ++issued;
            if (++slot == kStages) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
      }
  }
  if (!ok) {
    // After an abort: wait (bounded) for every load still in flight into this CTA's ring.
    for (int64_t y = issued > kStages ? issued - kStages : 0; y < issued; ++y)
      mbar_wait_drain(sm.full + (y % kStages), static_cast<uint32_t>((y / kStages) & 1), p.status);
  }
}

// Query transposer (one warp): for every ring stage, the 32 x 32 query slice
// read from global memory (lane = k) and written k-major into the stage; its
// 32 arrivals complete the stage's full barrier together with the TMA bytes.
__device__ void f32_qwarp(const float* __restrict__ Q, const F32Params& p, const F32Smem& sm, int lane) {
  const int n_qc = (p.nq + kQC - 1) / kQC;
  const int KC = (p.d + kKC - 1) / kKC;
  const int64_t qrows = static_cast<int64_t>(p.n_queries) * p.nq;
  const uint32_t full0 = smem_u32(sm.full), empty0 = smem_u32(sm.empty);
  uint32_t slot = 0, phase = 0;
  for (int64_t g = blockIdx.x; g < p.n_groups; g += gridDim.x) {
    int Tmax = 0;
    for (int u = 0; u < kGroup; ++u) {
      int64_t st;
      bool bad;
      const int L = f32_doc_rows(p, g * kGroup + u, st, bad);
      Tmax = max(Tmax, (L + kTT - 1) / kTT);
    }
    if (Tmax == 0) continue;
    for (int q = 0; q < p.n_queries; ++q)
      for (int qc = 0; qc < n_qc; ++qc) {
        const int64_t row0 = static_cast<int64_t>(q) * p.nq + qc * kQC;
        for (int t = 0; t < Tmax; ++t)
          for (int kc = 0; kc < KC; ++kc) {
            const int k = kc * kKC + lane;
            float v[kQC];
#pragma unroll
            for (int r = 0; r < kQC; ++r)
              v[r] = (row0 + r < qrows && k < p.d) ? __ldg(Q + (row0 + r) * p.d + k) : 0.f;
            if (!mbar_wait_a(empty0 + 8 * slot, phase ^ 1u, sm.abort_flag, p.status)) return;
            float* dst = reinterpret_cast<float*>(sm.stage + slot * kStageBytes) + lane * kQPitch;
#pragma unroll
            for (int r = 0; r < kQC; r += 4) *reinterpret_cast<float4*>(dst + r) = make_float4(v[r], v[r + 1], v[r + 2], v[r + 3]);
            mbar_arrive_a(full0 + 8 * slot);
            if (++slot == kStages) {
              slot = 0;
              phase ^= 1u;
            }
          }
      }
  }
}

__device__ __forceinline__ float f4c(const float4& v, int c) { return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w; }

// One 32-dim slice: 8 chunks of 4 dims. Per chunk: 8 query loads (k-major:
// 4 dims x 2 groups of 4 rows) and 8 document loads (token-major, 4 dims of
// one token each), then 256 FFMA ordered (dim, token, row): the document
// value stays in the operand reuse cache and each accumulator's register bank
// only has to differ from its row's, which is one fixed choice per row.
__device__ __forceinline__ void f32_slice(float (&acc)[8][8], uint32_t qK, uint32_t dX) {
#pragma unroll 1
  for (int pc = 0; pc < 8; ++pc) {
    const uint32_t qq = qK + pc * (4 * kQPitch * 4), dd = dX ^ static_cast<uint32_t>(pc << 4);
    float4 qk[4][2], dv[8];
    qk[0][0] = lds128<0 * kQPitch * 4>(qq);
    qk[0][1] = lds128<0 * kQPitch * 4 + 64>(qq);
    qk[1][0] = lds128<1 * kQPitch * 4>(qq);
    qk[1][1] = lds128<1 * kQPitch * 4 + 64>(qq);
    qk[2][0] = lds128<2 * kQPitch * 4>(qq);
    qk[2][1] = lds128<2 * kQPitch * 4 + 64>(qq);
    qk[3][0] = lds128<3 * kQPitch * 4>(qq);
    qk[3][1] = lds128<3 * kQPitch * 4 + 64>(qq);
    dv[0] = lds128<0>(dd);
    dv[1] = lds128<1024>(dd);
    dv[2] = lds128<2048>(dd);
    dv[3] = lds128<3072>(dd);
    dv[4] = lds128<4096>(dd);
    dv[5] = lds128<5120>(dd);
    dv[6] = lds128<6144>(dd);
    dv[7] = lds128<7168>(dd);
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r][m] = fmaf(f4c(qk[c][r >> 2], r & 3), f4c(dv[m], c), acc[r][m]);
  }
}

template <bool ARGMAX>
__device__ void f32_consumer(const F32Params& p, const F32Smem& sm, int warp, int lane) {
  const int u = warp >> 1, wn = warp & 1, lm = lane >> 3, ln = lane & 7;
  // Query rows 4 lm + r and 16 + 4 lm + r (r < 4) from the k-major slice;
  // tokens 64 wn + ln + 8 m with the 128-byte swizzle (chunk c of row j sits
  // at chunk c ^ (j & 7), and (64 wn + ln + 8 m) & 7 = ln).
  const uint32_t qoff = static_cast<uint32_t>(lm * 16);
  const uint32_t doff = (kQBytes + u * kDBytes + static_cast<uint32_t>((wn * 64 + ln) * 128)) |
                        static_cast<uint32_t>(ln << 4);
  const int n_qc = (p.nq + kQC - 1) / kQC;
  const int KC = (p.d + kKC - 1) / kKC;
  const uint32_t stage0 = smem_u32(sm.stage);
  const uint32_t full0 = smem_u32(sm.full), empty0 = smem_u32(sm.empty), redfull0 = smem_u32(sm.redfull);
  uint32_t slot = 0, phase = 0, rslot = 0, rphase = 0;
  float qsum = 0.f;

  for (int64_t g = blockIdx.x; g < p.n_groups; g += gridDim.x) {
    const int64_t b = g * kGroup + u;            // this warp's document
    // this document's length and the group's tile count (every consumer warp
    // walks the same ring sequence)
    int L = 0, Tmax = 0;
    bool bad = false;
#pragma unroll
    for (int v = 0; v < kGroup; ++v) {
      int64_t s2;
      bool b2;
      const int Lv = f32_doc_rows(p, g * kGroup + v, s2, b2);
      Tmax = max(Tmax, (Lv + kTT - 1) / kTT);
      if (v == u) {
        L = Lv;
        bad = b2;
      }
    }
    if (bad && wn == 0 && lane == 0) atomicOr(p.status, kDevErrBadInput);
    if (Tmax == 0) {
      // every document of the group is empty (or rejected): score 0, argmax -1
      if (wn == 0 && b < p.B) {
        for (int q = lane; q < p.n_queries; q += 32) p.out[static_cast<int64_t>(q) * p.B + b] = 0.f;
        if (ARGMAX)
          for (int64_t i = lane; i < static_cast<int64_t>(p.n_queries) * p.nq; i += 32) {
            const int64_t q = i / p.nq, qi = i - q * p.nq;
            p.argmax[(q * p.B + b) * p.nq + qi] = -1;
          }
      }
      continue;
    }
    for (int q = 0; q < p.n_queries; ++q) {
      for (int qc = 0; qc < n_qc; ++qc) {
        float rm[8];
        int ra[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          rm[r] = -INFINITY;
          ra[r] = INT_MAX;
        }
        for (int t = 0; t < Tmax; ++t) {
          float acc[8][8];
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[r][m] = 0.f;
          // a warp whose 64 tokens of this tile all lie past L only keeps the ring moving
          const bool active = t * kTT + wn * 64 < L;
          for (int kc = 0; kc < KC; ++kc) {
            if (!mbar_wait_a(full0 + 8 * slot, phase, sm.abort_flag, p.status)) return;
            if (active) {
              const uint32_t st = stage0 + slot * kStageBytes;
              f32_slice(acc, st + qoff, st + doff);
            }
            mbar_arrive_a(empty0 + 8 * slot);
            if (++slot == kStages) {
              slot = 0;
              phase ^= 1u;
            }
          }
          if (active) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int j = t * kTT + wn * 64 + ln + 8 * m;
              if (j < L) {
#pragma unroll
                for (int r = 0; r < 8; ++r)
                  if (acc[r][m] > rm[r]) {
                    rm[r] = acc[r][m];
                    ra[r] = j;
                  }
              }
            }
          }
        }
        // maximum over the 8 token lanes, lowest index on ties
#pragma unroll
        for (int r = 0; r < 8; ++r) {
#pragma unroll
          for (int o = 1; o <= 4; o <<= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, rm[r], o);
            const int i2 = __shfl_xor_sync(0xffffffffu, ra[r], o);
            if (v2 > rm[r] || (v2 == rm[r] && i2 < ra[r])) {
              rm[r] = v2;
              ra[r] = i2;
            }
          }
        }
        float* rv = sm.red_v + (rslot * kConsumerWarps + warp) * 32;
        int* ri = sm.red_i + (rslot * kConsumerWarps + warp) * 32;
        if (ln == 0) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            rv[4 * lm + (r & 3) + 16 * (r >> 2)] = rm[r];
            ri[4 * lm + (r & 3) + 16 * (r >> 2)] = ra[r];
          }
        }
        mbar_arrive_a(redfull0 + 8 * rslot);
        if (wn == 0) {
          if (!mbar_wait_a(redfull0 + 8 * rslot, rphase, sm.abort_flag, p.status)) return;
          const float* v0 = sm.red_v + (rslot * kConsumerWarps + warp) * 32;
          const int* i0 = sm.red_i + (rslot * kConsumerWarps + warp) * 32;
          float v = v0[lane];
          int ix = i0[lane];
          const float v2 = v0[32 + lane];
          const int i2 = i0[32 + lane];
          if (v2 > v || (v2 == v && i2 < ix)) {
            v = v2;
            ix = i2;
          }
          const int qi = qc * kQC + lane;
          const bool valid = qi < p.nq && b < p.B;
          if (L == 0) {
            v = 0.f;
            ix = -1;
          }
          if (ARGMAX && valid) p.argmax[(static_cast<int64_t>(q) * p.B + b) * p.nq + qi] = ix;
          float s = valid ? v : 0.f;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          qsum = (qc == 0 ? 0.f : qsum) + s;
          if (lane == 0 && qc == n_qc - 1 && b < p.B) p.out[static_cast<int64_t>(q) * p.B + b] = qsum;
        }
        if (++rslot == kRed) {
          rslot = 0;
          rphase ^= 1u;
        }
      }
    }
  }
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_f32_kernel(const __grid_constant__ CUtensorMap tm_d, const float* __restrict__ Q, const F32Params p) {
  extern __shared__ uint8_t raw[];
  const F32Smem sm = f32_carve(raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sm.full + s, 1 + 32);
      mbar_init(sm.empty + s, kConsumers);
    }
    for (int s = 0; s < kRed; ++s) mbar_init(sm.redfull + s, kConsumers);
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) tma_prefetch_desc(&tm_d);
  __syncthreads();
  if (warp == kProducerWarp) {
    if (lane == 0) f32_producer(&tm_d, p, sm);
    return;
  }
  if (warp == kQWarp) {
    f32_qwarp(Q, p, sm, lane);
    return;
  }
  f32_consumer<ARGMAX>(p, sm, warp, lane);
}

}  // namespace

maxsim_status launch_fwd_f32(const float* Q, int n_queries, int nq, int d, const float* D, int64_t total_rows,
                             int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                             float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (d % 4 != 0 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  // TMA row coordinates are 32-bit: the same row limit as the tensor-core path
  if (total_rows > (static_cast<int64_t>(1) << 30)) return MAXSIM_ERR_UNSUPPORTED;
  F32Params p;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.n_groups = (B + kGroup - 1) / kGroup;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = n_queries;
  p.nq = nq;
  p.d = d;
  // one query chunk: each document tile is read once, so stream it past L2
  p.evict_first = (n_queries * ((nq + kQC - 1) / kQC) == 1) ? 1 : 0;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  // documents as a [rows, d] matrix in 32-dim x 128-row boxes with the
  // 128-byte swizzle; rows and dims past the ends read as zero
  alignas(64) CUtensorMap tm_d;
  const uint64_t map_rows = total_rows > 0 ? static_cast<uint64_t>(total_rows) : 1;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), map_rows};
  const uint64_t strides[1] = {static_cast<uint64_t>(d) * 4};
  const uint32_t dbox[2] = {kKC, kTT};
  if (!encode_tmap(&tm_d, 3, 2, const_cast<float*>(D), ddims, strides, dbox, 1))
    return MAXSIM_ERR_CUDA;

  const size_t smem = f32_smem_bytes();
  if (smem > static_cast<size_t>(dev->max_smem_optin)) return MAXSIM_ERR_UNSUPPORTED;
  const int64_t want = dev->sm_count;
  const int grid = static_cast<int>(p.n_groups < want ? p.n_groups : want);
  cudaError_t e;
  if (argmax) {
    e = cudaFuncSetAttribute(fwd_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_f32_kernel<true><<<grid, kThreads, smem, stream>>>(tm_d, Q, p);
  } else {
    e = cudaFuncSetAttribute(fwd_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) fwd_f32_kernel<false><<<grid, kThreads, smem, stream>>>(tm_d, Q, p);
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

// i8tc.cu -- INT8 x INT8 MaxSim scoring on the 5th-generation tensor cores
// (FLASH-MAXSIM, Abstract: INT8xINT8 quantisation), per-token symmetric scales:
//
//   dot(i,j) = sum_k Q[i,k] * D[j,k]            exact integer
//   sim(i,j) = (float)dot(i,j) * d_scale[j]     one fp32 multiply, round-to-nearest
//   m_i      = max_j sim(i,j)                   lowest j on ties
//   out[b]   = sum_i q_scale[i] * m_i           fp32
//
// tcgen05 has no 8-bit integer MMA on sm_103a, but every int8 value is exact
// in fp16 and so is every product (|q d| <= 2^14). With d <= 256 every partial
// sum is an integer of magnitude <= 2^22, exact in the fp32 accumulator, so an
// fp16 kind::f16 MMA yields the exact integer dot.
//
// Work: each CTA owns a contiguous range of CSR documents, cut into tiles of
// up to 128 token rows. The MMA puts the query tokens on the TMEM lanes
// (A = the query, M = 128 rows of which nq <= 32 are real) and the tile's
// document rows on the columns (B = the tile, N = its rows rounded up to 16),
// so one lane holds all of one query token's similarities and the maximum
// over the document is a serial scan in that lane: no cross-lane reduction.
// The MMA work on the padding rows is far below the tensor-core budget.
// Roles (288 threads):
//  * Producer (warp 6): one contiguous bulk copy per tile (rows x d int8: CSR
//    rows are contiguous) into a ring of stages, no padding rows fetched, the
//    tile's token scales beside it (4-byte cp.async per lane, arriving on the
//    same stage barrier) and the tile's description (document, tile, rows,
//    last-tile flag). It alone reads the CSR offsets, 32 documents at a time;
//    a final stage marks the end of the CTA's work.
//  * Converters (warps 1, 2, 3, 5): int8 -> fp16 of each tile into one of two
//    K-major, 128-byte-swizzled operand buffers. Per 4 bytes: an XOR makes
//    them biased bytes u = x + 128, PRMT places each under the fp16 exponent
//    of 1024 (value 1024 + u), and one packed fp16 subtract of 1152 gives x.
//  * MMA (lane 0 of warps 7 and 8, alternate tiles): S^T = Q (M = 128) x
//    D_tile^T (N = rows rounded up to 16) over K = d into one of four TMEM
//    accumulators. Each issuing thread owns one operand buffer and two
//    accumulators: a thread's barrier polls wait behind its own MMAs, and
//    with two threads those are the tile before last, usually complete.
//  * Epilogue (warps 0 and 4, both on TMEM lanes 0-31 = the query tokens):
//    documents alternate between the two warps (by index parity), so all of
//    a document's tiles meet in one warp's registers. Per tile each lane
//    scans its row: one fp32 multiply by the column's scale, strict-greater
//    update in ascending token order (lowest token wins ties). At the
//    document's last tile the lanes sum q_scale[i] * m_i and write the score
//    and the per-token outputs. Warp 0 also writes documents without tiles
//    (empty or rejected) as empty.
// Every wait is bounded (ptx.cuh); after a timeout the producer and the MMA
// thread drain their asynchronous operations before the CTA exits.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "i8_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kTcThreads = 288;
constexpr int kTcProducerWarp = 6;
constexpr int kTcMmaWarp = 7;      // and warp 8: the second MMA thread
constexpr int kTcRows = 128;       // document rows per tile (MMA N <= 128)
constexpr int kTcM = 128;          // MMA M: query rows, nq <= 32 real
constexpr int kTcAcc = 4;          // TMEM accumulators of kTcRows columns
constexpr int kTcMaxNq = 32;
constexpr int kTcMaxD = 256;
constexpr int kTcMetaBytes = 32;

// Description of one ring stage, written by the producer before its arrival.
struct TileMeta {
  int64_t b;     // document
  int rows;      // token rows in this tile
  int t;         // tile index within the document
  int L;         // document length
  int flags;     // 1: last tile of the document, 2: end of the CTA's work
};
static_assert(sizeof(TileMeta) <= kTcMetaBytes, "tile meta");

__host__ __device__ constexpr uint32_t stage_bytes_of(int d) {
  return static_cast<uint32_t>(kTcRows * d + kTcRows * 4 + kTcMetaBytes);
}

struct I8TcParams {
  const int8_t* Q;
  const float* q_scale;
  const int8_t* D;
  const float* d_scale;
  const int64_t* offsets;
  int64_t B, total_tokens;
  int nq, d, S8;
  float* out;
  float* maxv;
  int32_t* maxdot;
  int32_t* argmax;
  unsigned* status;
};

struct I8TcSmem {
  uint32_t q16, a16, s8;        // shared addresses: fp16 Q atoms, 2 fp16 tile buffers, ring stages
  float* qsc;                   // [32] q_scale
  int* arows;                   // [2] rows of the tile in each buffer (-1: end of work)
  uint32_t full8, empty8;       // [S8] each
  uint32_t afull, aempty;       // [2] each
  uint32_t accfull, accempty;   // [kTcAcc] each
  uint32_t* tmem_slot;
  int* abort_flag;
};

size_t i8tc_smem_bytes(int d, int S8) {
  const size_t q16 = static_cast<size_t>(kTcM) * d * 2;
  const size_t a16 = 2u * kTcRows * d * 2;
  const size_t s8 = static_cast<size_t>(S8) * stage_bytes_of(d);
  const size_t misc = kTcMaxNq * 4 + 2 * 4;
  const size_t bars = (2u * S8 + 2 * 2 + 2 * kTcAcc) * 8;
  return 1024 + q16 + a16 + s8 + misc + bars + 16;
}

__device__ I8TcSmem i8tc_carve(uint8_t* raw, const I8TcParams& p) {
  I8TcSmem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q16 = base;
  uint8_t* a16 = q16 + static_cast<size_t>(kTcM) * p.d * 2;
  uint8_t* s8 = a16 + 2u * kTcRows * p.d * 2;
  uint8_t* misc = s8 + static_cast<size_t>(p.S8) * stage_bytes_of(p.d);
  s.q16 = smem_u32(q16);
  s.a16 = smem_u32(a16);
  s.s8 = smem_u32(s8);
  s.qsc = reinterpret_cast<float*>(misc);
  s.arows = reinterpret_cast<int*>(s.qsc + kTcMaxNq);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.arows + 2);
  s.full8 = smem_u32(bars);
  s.empty8 = s.full8 + 8 * p.S8;
  s.afull = s.empty8 + 8 * p.S8;
  s.aempty = s.afull + 16;
  s.accfull = s.aempty + 16;
  s.accempty = s.accfull + 8 * kTcAcc;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * p.S8 + 2 * 2 + 2 * kTcAcc);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  return s;
}

// This CTA's documents: a contiguous share of [0, B).
__device__ __forceinline__ void i8tc_range(const I8TcParams& p, int64_t& b0, int64_t& b1) {
  b0 = p.B * blockIdx.x / gridDim.x;
  b1 = p.B * (blockIdx.x + 1) / gridDim.x;
}

__device__ __forceinline__ void cp_async4_a(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ const TileMeta* meta_of(const I8TcSmem& sm, uint32_t slot, int d) {
  return reinterpret_cast<const TileMeta*>(
      __cvta_shared_to_generic(sm.s8 + slot * stage_bytes_of(d) + static_cast<uint32_t>(kTcRows * d + kTcRows * 4)));
}

__device__ void i8tc_producer(const I8TcParams& p, const I8TcSmem& sm, int lane) {
  int64_t b0, b1;
  i8tc_range(p, b0, b1);
  const uint32_t sbytes = stage_bytes_of(p.d);
  uint32_t slot = 0, phase = 0;
  int64_t issued = 0;
  bool ok = true;
  // one stage per tile, then one end marker
  auto fill = [&](int64_t b, int64_t row0, int rows, int t, int L, int flags) -> bool {
    if (!mbar_wait_a(sm.empty8 + 8 * slot, phase ^ 1u, sm.abort_flag, p.status)) return false;
    const uint32_t dst = sm.s8 + slot * sbytes, bar = sm.full8 + 8 * slot;
    if (lane == 0) {
      TileMeta* m = const_cast<TileMeta*>(meta_of(sm, slot, p.d));
      m->b = b;
      m->rows = rows;
      m->t = t;
      m->L = L;
      m->flags = flags;
      const uint32_t bytes = static_cast<uint32_t>(rows) * p.d;
      mbar_arrive_expect_tx_a(bar, bytes);   // release: the description above is visible with the stage
      if (bytes) bulk_g2s_a(dst, p.D + row0 * p.d, bytes, bar);
    }
    for (int r = lane; r < rows; r += 32) cp_async4_a(dst + kTcRows * p.d + 4 * r, p.d_scale + row0 + r);
    cp_async_arrive_noinc(bar);
    ++issued;
    if (++slot == static_cast<uint32_t>(p.S8)) {
      slot = 0;
      phase ^= 1u;
    }
    return true;
  };
  for (int64_t cb = b0; ok && cb < b1; cb += 32) {
    // offsets of 32 documents at once; lane k holds document cb + k
    int64_t ls = 0, le = 0;
    if (cb + lane < b1) {
      ls = __ldg(p.offsets + cb + lane);
      le = __ldg(p.offsets + cb + lane + 1);
    }
    const bool lbad = cb + lane < b1 && (ls < 0 || le < ls || le > p.total_tokens || le - ls > INT_MAX);
    if (lbad) atomicOr(p.status, kDevErrBadInput);
    const int nk = static_cast<int>(min(static_cast<int64_t>(32), b1 - cb));
    for (int k = 0; ok && k < nk; ++k) {
      const int64_t s0 = __shfl_sync(0xffffffffu, ls, k), e0 = __shfl_sync(0xffffffffu, le, k);
      const bool bad = s0 < 0 || e0 < s0 || e0 > p.total_tokens || e0 - s0 > INT_MAX;
      const int L = bad ? 0 : static_cast<int>(e0 - s0);
      for (int t = 0; ok && t * kTcRows < L; ++t) {
        const int rows = min(kTcRows, L - t * kTcRows);
        ok = fill(cb + k, s0 + static_cast<int64_t>(t) * kTcRows, rows, t, L, (t + 1) * kTcRows >= L ? 1 : 0);
      }
    }
  }
  if (ok) ok = fill(b1, 0, 0, 0, 0, 2);
  if (!ok) {
    // After an abort: wait (bounded) for every copy still in flight into this CTA's ring.
    for (int64_t y = issued > p.S8 ? issued - p.S8 : 0; y < issued; ++y)
      mbar_wait_drain(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.full8 + 8 * (y % p.S8))),
                      static_cast<uint32_t>((y / p.S8) & 1), p.status);
  }
}

template <int D16>
__device__ void i8tc_converter(const I8TcParams& p, const I8TcSmem& sm, int ct) {
  constexpr int kD = D16 * 16;
  uint32_t slot = 0, phase = 0, ab = 0, aph = 0;
  for (;;) {
    if (!mbar_wait_a(sm.full8 + 8 * slot, phase, sm.abort_flag, p.status)) return;
    const TileMeta* m = meta_of(sm, slot, kD);
    const int rows = m->rows, flags = m->flags;
    if (!mbar_wait_a(sm.aempty + 8 * ab, aph ^ 1u, sm.abort_flag, p.status)) return;
    if (flags & 2) {
      // end of work: hand the marker to both MMA threads (this buffer, then the other)
      if (ct == 0) sm.arows[ab] = -1;
      mbar_arrive_a(sm.afull + 8 * ab);
      const uint32_t ob = ab ^ 1u, oph = ab ? aph ^ 1u : aph;
      if (!mbar_wait_a(sm.aempty + 8 * ob, oph ^ 1u, sm.abort_flag, p.status)) return;
      if (ct == 0) sm.arows[ob] = -1;
      mbar_arrive_a(sm.afull + 8 * ob);
      return;
    }
    const uint32_t src = sm.s8 + slot * stage_bytes_of(kD);
    const uint32_t dst = sm.a16 + ab * static_cast<uint32_t>(kTcRows * kD * 2);
    const int n = rows * D16;
    for (int i = ct; i < n; i += 128) {
      const int r = i / D16, ci = i - r * D16;
      cvt16(lds_u4(src + static_cast<uint32_t>(r * kD + ci * 16)), dst, r, ci, kTcRows * 128);
    }
    if (ct == 0) sm.arows[ab] = rows;
    fence_proxy_async_smem();   // generic-proxy writes, read by the tensor core
    mbar_arrive_a(sm.afull + 8 * ab);
    if (++slot == static_cast<uint32_t>(p.S8)) {
      slot = 0;
      phase ^= 1u;
    }
    if (++ab == 2) {
      ab = 0;
      aph ^= 1u;
    }
  }
}

// MMA thread `par` (0 or 1): tiles n = par, par + 2, ...; operand buffer par,
// accumulators par and par + 2.
__device__ void i8tc_mma(const I8TcParams& p, const I8TcSmem& sm, uint32_t tmem, uint32_t par) {
  const int ksteps = p.d / 16;
  const uint32_t a_bytes = static_cast<uint32_t>(kTcRows * p.d * 2);
  const volatile int* arows = sm.arows;
  const uint32_t ab = par;
  uint32_t aph = 0;
  int64_t done = 0;
  bool ok = true;
  for (uint32_t i = 0;; ++i) {
    // this thread's i-th tile is n = 2 i + par: accumulator n & 3, its (n >> 2)-th use
    const uint32_t n = 2 * i + par, acc = n & 3, cph = (n >> 2) & 1;
    if (!mbar_poll_a(sm.afull + 8 * ab, aph, sm.abort_flag, p.status)) {
      ok = false;
      break;
    }
    const int rows = arows[ab];
    if (rows < 0) break;
    if (!mbar_poll_a(sm.accempty + 8 * acc, cph ^ 1u, sm.abort_flag, p.status)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t idesc = idesc_f16(0, kTcM, (rows + 15) & ~15);
    const uint32_t bbase = sm.a16 + ab * a_bytes;
    for (int k = 0; k < ksteps; ++k) {
      const uint32_t off = static_cast<uint32_t>(k & 3) * 32;
      const uint64_t adesc = sdesc_k_sw128(sm.q16 + static_cast<uint32_t>(k >> 2) * (kTcM * 128) + off);
      const uint64_t bdesc = sdesc_k_sw128(bbase + static_cast<uint32_t>(k >> 2) * (kTcRows * 128) + off);
      umma_f16(tmem + acc * static_cast<uint32_t>(kTcRows), adesc, bdesc, idesc, k > 0 ? 1u : 0u);
    }
    umma_commit_a(sm.accfull + 8 * acc);
    umma_commit_a(sm.aempty + 8 * ab);
    ++done;
    aph ^= 1u;
  }
  if (!ok && done > 0) {
    // the tensor core must be done with TMEM and shared memory before the CTA exits
    mbar_wait_drain(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.aempty + 8 * ab)), aph ^ 1u, p.status);
  }
}

// Documents [from, to) have no tiles (empty or rejected): score 0, m_i 0,
// dot 0, argmax -1. Written by warp 0.
template <bool DETAIL>
__device__ void write_empty(const I8TcParams& p, int64_t from, int64_t to, int lane) {
  for (int64_t b = from; b < to; ++b) {
    if (lane == 0) p.out[b] = 0.f;
    if (DETAIL)
      for (int i = lane; i < p.nq; i += 32) {
        const int64_t o = b * p.nq + i;
        if (p.maxv) p.maxv[o] = 0.f;
        if (p.maxdot) p.maxdot[o] = 0;
        if (p.argmax) p.argmax[o] = -1;
      }
  }
}

template <bool DETAIL>
__device__ void i8tc_epilogue(const I8TcParams& p, const I8TcSmem& sm, uint32_t tmem, int warp, int lane) {
  int64_t b0, b1;
  i8tc_range(p, b0, b1);
  const int me = warp >> 2;                  // documents with (b & 1) == me
  const uint32_t sbytes = stage_bytes_of(p.d);
  uint32_t acc = 0, cph = 0, slot = 0, sph = 0;
  int64_t next_b = b0;                       // warp 0: first document not yet written
  float bv = -INFINITY;
  int bj = INT_MAX, bd = 0;
  const bool qlive = lane < p.nq;
  const float qs = qlive ? sm.qsc[lane] : 0.f;
  for (;;) {
    if (!mbar_wait_a(sm.full8 + 8 * slot, sph, sm.abort_flag, p.status)) return;
    const TileMeta* m = meta_of(sm, slot, p.d);
    const int64_t b = m->b;
    const int rows = m->rows, t = m->t, flags = m->flags;
    if (flags & 2) break;
    if (warp == 0 && t == 0) {
      write_empty<DETAIL>(p, next_b, b, lane);
      next_b = b + 1;
    }
    if (static_cast<int>(b & 1) == me) {
      if (t == 0) {
        bv = -INFINITY;
        bj = INT_MAX;
        bd = 0;
      }
      if (!mbar_wait_a(sm.accfull + 8 * acc, cph, sm.abort_flag, p.status)) return;
      tc_fence_after();
      const float* sc = reinterpret_cast<const float*>(
          __cvta_shared_to_generic(sm.s8 + slot * sbytes + static_cast<uint32_t>(kTcRows * p.d)));
      const int jbase = t * kTcRows;
#pragma unroll 1
      for (int c = 0; c * 32 < rows; ++c) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + acc * static_cast<uint32_t>(kTcRows) + 32 * c, v);
        const float4* sc4 = reinterpret_cast<const float4*>(sc + 32 * c);
        const int lim = rows - 32 * c;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 s4 = sc4[q4];
          const float ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * q4 + e;
            if (k < lim) {
              const float sim = __fmul_rn(v[k], ss[e]);
              if (sim > bv) {
                bv = sim;
                bj = jbase + 32 * c + k;
                if (DETAIL) bd = __float2int_rn(v[k]);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_a(sm.accempty + 8 * acc);
      if (flags & 1) {
        // document complete: the score and this lane's query-token outputs
        float sterm = qlive ? qs * bv : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sterm += __shfl_xor_sync(0xffffffffu, sterm, o);
        if (lane == 0) p.out[b] = sterm;
        if (DETAIL && qlive) {
          const int64_t o = b * p.nq + lane;
          if (p.maxv) p.maxv[o] = bv;
          if (p.maxdot) p.maxdot[o] = bd;
          if (p.argmax) p.argmax[o] = bj;
        }
      }
    }
    mbar_arrive_a(sm.empty8 + 8 * slot);     // both warps release every stage
    if (++acc == kTcAcc) {
      acc = 0;
      cph ^= 1u;
    }
    if (++slot == static_cast<uint32_t>(p.S8)) {
      slot = 0;
      sph ^= 1u;
    }
  }
  if (warp == 0) write_empty<DETAIL>(p, next_b, b1, lane);
}

template <int D16, bool DETAIL>
__global__ void __launch_bounds__(kTcThreads, 1) i8tc_kernel(const I8TcParams p) {
  extern __shared__ uint8_t raw[];
  const I8TcSmem sm = i8tc_carve(raw, p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.S8; ++s) {
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.full8 + 8 * s)), 1 + 32);
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.empty8 + 8 * s)), 64);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.afull + 8 * i)), 128);
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.aempty + 8 * i)), 1);
    }
    for (int i = 0; i < kTcAcc; ++i) {
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.accfull + 8 * i)), 1);
      mbar_init(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(sm.accempty + 8 * i)), 32);
    }
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  // the query, int8 -> fp16 in the K-major SW128 layout (rows past nq zero)
  {
    const int n = kTcM * D16;
    for (int i = threadIdx.x; i < n; i += kTcThreads) {
      const int r = i / D16, ci = i - r * D16;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (r < p.nq) w = __ldg(reinterpret_cast<const uint4*>(p.Q + static_cast<int64_t>(r) * p.d) + ci);
      cvt16(w, sm.q16, r, ci, kTcM * 128);
    }
    fence_proxy_async_smem();
    for (int i = threadIdx.x; i < p.nq; i += kTcThreads) sm.qsc[i] = __ldg(p.q_scale + i);
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(sm.tmem_slot, kTcAcc * kTcRows);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  if (warp == 0 || warp == 4) {
    i8tc_epilogue<DETAIL>(p, sm, tmem, warp, lane);
  } else if (warp <= 5) {
    i8tc_converter<D16>(p, sm, (warp == 5 ? 3 : warp - 1) * 32 + lane);
  } else if (warp == kTcProducerWarp) {
    i8tc_producer(p, sm, lane);
  } else if (lane == 0) {
    i8tc_mma(p, sm, tmem, static_cast<uint32_t>(warp - kTcMmaWarp));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcAcc * kTcRows);
  }
}

template <int D16>
cudaError_t i8tc_launch_d(const I8TcParams& p, bool detail, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e;
  if (detail) {
    e = cudaFuncSetAttribute(i8tc_kernel<D16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8tc_kernel<D16, true><<<grid, kTcThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(i8tc_kernel<D16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) i8tc_kernel<D16, false><<<grid, kTcThreads, smem, stream>>>(p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool i8tc_applicable(int nq, int d) {
  const DeviceInfo* dev = device_info();
  if (!dev || nq < 1 || nq > kTcMaxNq || d % 64 != 0 || d > kTcMaxD) return false;
  return i8tc_smem_bytes(d, 2) <= static_cast<size_t>(dev->max_smem_optin);
}

maxsim_status launch_i8tc(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D,
                          const float* d_scale, const int64_t* offsets, int64_t B, int64_t total_tokens,
                          float* out, float* maxv, int32_t* maxdot, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  I8TcParams p;
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
  // as many stages as fit (each holds one tile of up to 128 rows)
  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  int S8 = 12;
  while (S8 > 2 && i8tc_smem_bytes(d, S8) > budget) --S8;
  if (i8tc_smem_bytes(d, S8) > budget) return MAXSIM_ERR_UNSUPPORTED;
  p.S8 = S8;
  const size_t smem = i8tc_smem_bytes(d, S8);
  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  const bool detail = maxv || maxdot || argmax;
  cudaError_t e;
  switch (d / 16) {
    case 4: e = i8tc_launch_d<4>(p, detail, grid, smem, stream); break;
    case 8: e = i8tc_launch_d<8>(p, detail, grid, smem, stream); break;
    case 12: e = i8tc_launch_d<12>(p, detail, grid, smem, stream); break;
    case 16: e = i8tc_launch_d<16>(p, detail, grid, smem, stream); break;
    default: return MAXSIM_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

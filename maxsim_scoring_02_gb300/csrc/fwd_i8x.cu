// fwd_i8x.cu -- INT8 x INT8 MaxSim scores on the tcgen05 tensor cores, with
// document rows on the MMA's M dimension (the chunk-slot walk of fwd_tc.cu).
//
// Computes, per CSR document b (FLASH-MAXSIM, Abstract: INT8 x INT8 with
// per-token symmetric scales):
//   dot(i,j) = sum_k Q[i,k] * D[j,k]              exact integer
//   sim(i,j) = (float)dot(i,j) * d_scale[j]       one fp32 multiply
//   m_i      = max_{j < L_b} sim(i,j)
//   out[b]   = sum_i q_scale[i] * m_i
// for nq <= 64 and d in {64, 128, 192}; calls that ask for the per-token
// outputs (m_i, the dot at the argmax, the argmax) take i8tc.cu instead.
//
// Exactness: int8 values are exact in fp16 and so is every product
// (|q d| <= 2^14); with d <= 192 every partial sum is an integer below 2^22,
// exact in the fp32 accumulator, so an fp16 kind::f16 MMA returns the exact
// dot whatever order the tensor core adds in.
//
// Roles (16 warps), on the chunk-slot walk and group tables of
// fwd_common.cuh:
//  * Builder (warp 11): each group's slot table, one group ahead.
//  * Loader (warp 8, lane 0 issues): TMA loads of the int8 rows of a tile
//    (all d bytes of a row in one box row; one 128-row box for four
//    contiguous slots, else one 32-row box per slot) into a ring of raw
//    stages.
//  * Converters (warps 12-15): thread t converts tile row t of each raw
//    stage into a ring of fp16 operand stages, K-major with 128-byte
//    swizzling (the exponent-bias conversion of i8_common.cuh), walking the
//    row's 16-byte chunks from chunk t mod 8 so that a quarter warp's reads
//    and stores fall on distinct banks, then releases the raw stage.
//  * MMA (warp 9, an elected lane issues): M = 128 document rows, N = 32 or
//    64 query tokens, K = 16, d / 16 steps per tile into one of four TMEM
//    accumulators.
//  * Slot partials (warps 0-7, two groups of four taking tiles round-robin):
//    tcgen05.ld of a 32-row slot, each lane's row multiplied by its row's
//    d_scale (loaded before the accumulator is waited for), rows past the
//    slot's valid rows masked, then the column maxima of fwd_tc.cu. A
//    document whose slots all lie in one tile is finished by the group.
//  * Merge (warp 10): documents that span tiles, as in fwd_tc.cu, each
//    column weighted by q_scale in the sum.
// HBM bytes per document: L_b * (d + 4) (int8 rows and fp32 scales) + 8 of
// offsets, read once. Every wait is bounded (ptx.cuh); after an abort the
// loader drains its copies and the MMA warp waits for its last MMA before
// TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "fwd_common.cuh"
#include "i8_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kI8xBuilderWarp = kMergeWarp + 1;       // 11
constexpr int kI8xConvWarp0 = kMergeWarp + 2;         // 12-15
constexpr int kI8xConvWarps = 4;
constexpr int kI8xThreads = 32 * (kI8xConvWarp0 + kI8xConvWarps);
constexpr int kI8xSlice = 128 * 128;                  // a 64-dim fp16 slice of a 128-row tile
constexpr int kI8xMaxD = 192;
constexpr int kI8xMaxRaw = 12, kI8xOp = 2;

struct I8xSmem {
  uint8_t* q;            // KB slices x (NC rows x 128 B), fp16 swizzled
  uint8_t* raw;          // p.stages x (128 rows x d bytes); d = 64: 64-byte swizzled
  uint8_t* op;           // p.n_qslots x (KB slices x 16 KB)
  GroupTab* tab;         // [2]
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* part_v;         // [PB][4][NC]
  int32_t* part_i;       // [PB][4][NC]
  float* gsum;           // [kCapDocs] (multi-pass only; unused here)
};

__host__ __device__ inline size_t i8x_bars_count(int n_raw, int n_op, int n_acc, int n_part) {
  return 2 * n_raw + 2 * n_op + 2 * n_acc + 4 + 2 * n_part + 1;
}

__host__ __device__ inline size_t i8x_smem_bytes(int NC, int d, int n_raw, int n_op, int n_acc, int n_part) {
  const int KB = d / 64;
  size_t bytes = 1024;
  bytes += static_cast<size_t>(KB) * NC * 128;
  bytes += static_cast<size_t>(n_raw) * 128 * d;
  bytes += static_cast<size_t>(n_op) * KB * kI8xSlice;
  bytes += 2 * sizeof(GroupTab);
  bytes += i8x_bars_count(n_raw, n_op, n_acc, n_part) * 8 + 16;
  bytes += static_cast<size_t>(n_part * 4 * NC) * 8;
  bytes += kCapDocs * 4;
  return bytes;
}

__device__ __forceinline__ I8xSmem i8x_carve(uint8_t* raw, const FwdTcParams& p, int NC, int d) {
  I8xSmem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.q = base;
  // operand stages first: each starts on a 1024-byte boundary (swizzle atoms)
  s.op = s.q + static_cast<size_t>(p.KB) * NC * 128;
  s.raw = s.op + static_cast<size_t>(p.n_qslots) * p.KB * kI8xSlice;
  s.tab = reinterpret_cast<GroupTab*>(s.raw + static_cast<size_t>(p.stages) * 128 * d);
  s.bars = reinterpret_cast<uint64_t*>(s.tab + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + i8x_bars_count(p.stages, p.n_qslots, p.n_acc, p.n_part));
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.part_v = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.part_i = reinterpret_cast<int32_t*>(s.part_v + p.n_part * 4 * NC);
  s.gsum = reinterpret_cast<float*>(s.part_i + p.n_part * 4 * NC);
  return s;
}

// Barrier addresses (32-bit shared) in the order of i8x_bars_count.
struct I8xBars {
  uint32_t rawfull, rawempty, opfull, opempty, accfull, accempty, tabfull, tabempty, partfull, partempty, done;
  __device__ __forceinline__ I8xBars(const I8xSmem& sm, int NR, int NO, int A, int PB) {
    rawfull = smem_u32(sm.bars);
    rawempty = rawfull + 8 * NR;
    opfull = rawempty + 8 * NR;
    opempty = opfull + 8 * NO;
    accfull = opempty + 8 * NO;
    accempty = accfull + 8 * A;
    tabfull = accempty + 8 * A;
    tabempty = tabfull + 16;
    partfull = tabempty + 16;
    partempty = partfull + 8 * PB;
    done = partempty + 8 * PB;
  }
};

// --------------------------------------------------------------- loader
__device__ void i8x_loader(const FwdTcParams& p, const I8xSmem& sm, const I8xBars& br, const CUtensorMap* tm128,
                           const CUtensorMap* tm32, int d) {
  const int lane = threadIdx.x & 31;
  if (debug_faults(p.status) & kDebugStallFwdLoader) return;   // test-only switch (maxsim_debug_set_faults)
  const int NR = p.stages;
  const uint64_t policy = l2_policy_evict_first();
  const uint32_t raw0 = smem_u32(sm.raw);
  const uint32_t stage_bytes = 128u * static_cast<uint32_t>(d), slot_bytes = 32u * static_cast<uint32_t>(d);
  int s = 0;
  uint32_t ph = 0, fills = 0;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    const GroupTab* T = sm.tab + buf;
    {
      bool w = true;
      if (lane == 0) w = mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) { ok = false; break; }
    }
    if (T->n_docs < 0) break;
    if (lane == 0) {
      const int n_slots = T->n_slots;
      const int n_tiles = (n_slots + 3) >> 2;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int i0 = 4 * t;
        const int nslot = min(4, n_slots - i0);
        int rows[4];
        bool contiguous = nslot == 4;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          rows[w] = w < nslot ? T->slot_row[i0 + w] : 0;
          if (w > 0 && rows[w] != rows[0] + 32 * w) contiguous = false;
        }
        if (!mbar_wait_a(br.rawempty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = br.rawfull + 8 * s;
        const uint32_t dst = raw0 + static_cast<uint32_t>(s) * stage_bytes;
        mbar_arrive_expect_tx_a(fb, contiguous ? stage_bytes : static_cast<uint32_t>(nslot) * slot_bytes);
        if (contiguous) {
          tma_load_2d_a(dst, tm128, fb, 0, rows[0], policy);
        } else {
          for (int w = 0; w < nslot; ++w) tma_load_2d_a(dst + w * slot_bytes, tm32, fb, 0, rows[w], policy);
        }
        ++fills;
        if (++s == NR) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    if (ok && lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);   // slot rows read
  }
  if (!ok && lane == 0) {
    // After an abort: wait (bounded) for every load this warp may still have in flight.
    for (uint32_t f = fills > static_cast<uint32_t>(NR) ? fills - NR : 0; f < fills; ++f)
      mbar_wait_drain(sm.bars + (f % NR), (f / NR) & 1u, p.status);
  }
}

// ----------------------------------------------------------- converters
// Converter thread t (0..127) converts tile row t, 16 bytes (one chunk) at a
// time, into two 16-byte chunks of the operand stage (K-major, 128-byte
// swizzle). Thread t walks its row's n = d / 16 chunks starting at chunk
// t mod 8 (d = 128, 192; at d = 64 the raw rows carry the 64-byte swizzle,
// chunk j of row t at j ^ ((t >> 1) & 3), and every thread starts at 0), so
// the eight rows of a quarter warp fall on distinct banks in the stores and
// in the reads (two-way in the reads at d = 192). A thread loads its whole
// row before it converts, releases the raw stage, then stores.
template <int KB>
__device__ void i8x_converters(const FwdTcParams& p, const I8xSmem& sm, const I8xBars& br) {
  constexpr int kN = 4 * KB;                   // 16-byte chunks per row
  constexpr uint32_t kStage = 128u * 64u * KB, kOp = static_cast<uint32_t>(KB) * kI8xSlice;
  const int ct = threadIdx.x - 32 * kI8xConvWarp0, lane = threadIdx.x & 31;
  const int rot = KB == 1 ? 0 : (ct & 7);
  const uint32_t sw = KB == 1 ? static_cast<uint32_t>((ct >> 1) & 3) : 0u;
  const uint32_t row0 = smem_u32(sm.raw) + static_cast<uint32_t>(ct) * (64u * KB), op0 = smem_u32(sm.op);
  const int NR = p.stages, NO = p.n_qslots;
  int s = 0, o = 0;
  uint32_t ph = 0, oph = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    bool w = true;
    if (lane == 0) w = mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status);
    if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) return;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) return;
    const int n_tiles = (T->n_slots + 3) >> 2;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait_a(br.rawfull + 8 * s, ph, sm.abort_flag, p.status)) return;
      const uint32_t src = row0 + static_cast<uint32_t>(s) * kStage;
      uint4 w4[kN];
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        int j = c + rot;
        if (j >= kN) j -= kN;
        w4[c] = lds_u4(src + ((static_cast<uint32_t>(j) ^ sw) << 4));
      }
      mbar_arrive_a(br.rawempty + 8 * s);  // the row is in registers (the arrive orders the reads before it)
      if (!mbar_wait_a(br.opempty + 8 * o, oph ^ 1u, sm.abort_flag, p.status)) return;
      const uint32_t dst = op0 + static_cast<uint32_t>(o) * kOp;
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        int j = c + rot;
        if (j >= kN) j -= kN;
        cvt16(w4[c], dst, ct, j, kI8xSlice);
      }
      // generic-proxy writes, read by the tensor core, ordered before the async proxy's accesses
      fence_proxy_async_smem();
      mbar_arrive_a(br.opfull + 8 * o);    // every converter thread arrives after its own fence
      if (++s == NR) {
        s = 0;
        ph ^= 1u;
      }
      if (++o == NO) {
        o = 0;
        oph ^= 1u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

// ----------------------------------------------------------------- MMA
// The whole warp runs the loop (warp-uniform control flow); an elected lane
// issues. Per tile: one operand stage, KB slices x 4 K steps.
template <int NC>
__device__ void i8x_mma(const FwdTcParams& p, const I8xSmem& sm, const I8xBars& br, uint32_t tmem_base) {
  const int lane = threadIdx.x & 31;
  const int KB = p.KB, A = p.n_acc, NO = p.n_qslots;
  const uint32_t idesc = p.idesc;
  const uint64_t adesc0 = sdesc_k_sw128(smem_u32(sm.op));
  const uint64_t qdesc0 = sdesc_k_sw128(smem_u32(sm.q));
  int o = 0, a = 0;
  uint32_t oph = 0, aph = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!__all_sync(0xffffffffu, mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status))) break;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) break;
    const int n_tiles = (T->n_slots + 3) >> 2;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!__all_sync(0xffffffffu, mbar_wait_a(br.accempty + 8 * a, aph ^ 1u, sm.abort_flag, p.status)) ||
          !__all_sync(0xffffffffu, mbar_wait_a(br.opfull + 8 * o, oph, sm.abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * NC);
      const uint64_t od = adesc0 + static_cast<uint64_t>((o * KB * kI8xSlice) >> 4);
      for (int kb = 0; kb < KB; ++kb) {
        const uint64_t ad = od + static_cast<uint64_t>((kb * kI8xSlice) >> 4);
        const uint64_t bd = qdesc0 + static_cast<uint64_t>((kb * NC * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_f16_el(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      umma_commit_el(br.opempty + 8 * o);    // operand stage reusable once these MMAs have read it
      umma_commit_el(br.accfull + 8 * a);    // accumulator ready for the epilogue
      if (++o == NO) {
        o = 0;
        oph ^= 1u;
      }
      if (++a == A) {
        a = 0;
        aph ^= 1u;
      }
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
  // Wait until every MMA issued by this warp has completed before TMEM is freed.
  umma_commit_el(br.done);
  mbar_wait_drain(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(br.done)), 0, p.status);
}

// --------------------------------------------------------- slot partials
// As in fwd_tc.cu (single pass, scores only): warp w reduces slot w of the
// group's tiles; a document whose slots all lie in the tile is finished by
// one of its slots' warps, its columns weighted by q_scale.
template <int NG>
__device__ void i8x_partials(const FwdTcParams& p, const I8xSmem& sm, const I8xBars& br, uint32_t tmem_base) {
  constexpr int NC = 32 * NG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const uint32_t grp = warp >> 2;
  const int A = p.n_acc, PB = p.n_part;
  const int lgA = __ffs(A) - 1, lgPB = __ffs(PB) - 1;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  float qw[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) qw[g] = g * 32 + lane < p.nq ? __ldg(p.col_scale + g * 32 + lane) : 0.f;
  uint32_t tt = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) break;
    const int n_slots = T->n_slots;
    const int n_tiles = (n_slots + 3) >> 2;
    for (int t = 0; t < n_tiles; ++t, ++tt) {
      if (tt % kGroups != grp) continue;
      const int a = static_cast<int>(tt & static_cast<uint32_t>(A - 1));
      const uint32_t aph = (tt >> lgA) & 1u;
      const int pb = static_cast<int>(tt & static_cast<uint32_t>(PB - 1));
      const uint32_t pph = (tt >> lgPB) & 1u;
      const int i0 = 4 * t;
      const bool mine = quarter < n_slots - i0;
      // this lane's row scale, fetched before the accumulator is waited for
      int vrows = 0;
      float rs = 0.f;
      if (mine) {
        vrows = T->slot_info[i0 + quarter] & 63;
        if (lane < vrows) rs = __ldg(p.row_scale + T->slot_row[i0 + quarter] + lane);
      }
      if (!mbar_wait_a(br.partempty + 8 * pb, pph ^ 1u, sm.abort_flag, p.status)) return;
      if (!mbar_wait_a(br.accfull + 8 * a, aph, sm.abort_flag, p.status)) return;
      tc_fence_after();
      float own_v[NG];
      if (mine) {
        const int row = (T->slot_info[i0 + quarter] >> 6) * kSlotRows + lane;
        float* pv = sm.part_v + (pb * 4 + quarter) * NC;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float v[32];
          tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(a * NC + g * 32), v);
          if (g == NG - 1) {  // accumulator fully in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
          }
          // sim = (float)dot * d_scale[row]: one rounding, as in the definition
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = lane < vrows ? __fmul_rn(v[k], rs) : -INFINITY;
          float bv;
          int bi;
          warp_column_max<false>(v, row, lane, bv, bi);
          pv[g * 32 + lane] = bv;
          own_v[g] = bv;
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
      }
      mbar_arrive_a(br.partfull + 8 * pb);  // every thread of the group arrives (count 128)
      if (mine) {
        const int sd = T->slot_doc[i0 + quarter];
        if (sd & kSlotLocal) {
          const int info = T->slot_info[i0 + quarter];
          const int ncs = (sd >> 17) & 7;
          const int f0 = quarter - (info >> 6);
          const int fin = ncs == 1 ? f0 : f0 + static_cast<int>((tt >> 1) % static_cast<uint32_t>(ncs));
          if (quarter == fin) {
            if (ncs > 1 && !mbar_wait_a(br.partfull + 8 * pb, pph, sm.abort_flag, p.status)) return;
            const int64_t bd = doc_at(p, T->first_doc + (sd & kSlotDocMask));
            float sum = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              float m = own_v[g];
              if (ncs > 1) {
                m = -INFINITY;
                for (int j = 0; j < ncs; ++j) m = fmaxf(m, sm.part_v[(pb * 4 + f0 + j) * NC + g * 32 + lane]);
              }
              if (g * 32 + lane < p.nq) sum += qw[g] * m;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0 && bd >= 0) p.out[bd] = sum;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_a(br.partempty + 8 * pb);  // done reading this buffer
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

// The query as the MMA's B operand: per 64-dim slice, NC rows of fp16 (zero
// for tokens >= nq), K-major with 128-byte swizzling.
__device__ void i8x_query(const int8_t* Q, int nq, int d, const I8xSmem& sm, int NC) {
  const int cpr = d >> 4;
  const uint32_t q0 = smem_u32(sm.q);
  for (int u = threadIdx.x; u < NC * cpr; u += kI8xThreads) {
    const int r = u / cpr, ci = u - r * cpr;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (r < nq) w = __ldg(reinterpret_cast<const uint4*>(Q + static_cast<int64_t>(r) * d) + ci);
    cvt16(w, q0, r, ci, static_cast<uint32_t>(NC * 128));
  }
}

template <int NG>
__global__ void __launch_bounds__(kI8xThreads, 1)
    fwd_i8x_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm32,
                   const int8_t* __restrict__ Q, const FwdTcParams p, int d) {
  constexpr int NC = 32 * NG;
  extern __shared__ uint8_t smem_raw[];
  const I8xSmem sm = i8x_carve(smem_raw, p, NC, d);
  const I8xBars br(sm, p.stages, p.n_qslots, p.n_acc, p.n_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    uint64_t* b = sm.bars;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(b + s, 1);                               // rawfull: the loader's expect_tx
      mbar_init(b + p.stages + s, 32 * kI8xConvWarps);   // rawempty: every converter thread
    }
    b += 2 * p.stages;
    for (int s = 0; s < p.n_qslots; ++s) {
      mbar_init(b + s, 32 * kI8xConvWarps);              // opfull: every converter thread
      mbar_init(b + p.n_qslots + s, 1);                  // opempty: the MMA commit
    }
    b += 2 * p.n_qslots;
    for (int i = 0; i < p.n_acc; ++i) mbar_init(b + i, 1);             // accfull
    for (int i = 0; i < p.n_acc; ++i) mbar_init(b + p.n_acc + i, 4);   // accempty: the 4 warps of one group
    b += 2 * p.n_acc;
    for (int i = 0; i < 2; ++i) mbar_init(b + i, 1);                   // tabfull: the builder
    // tabempty: loader + MMA + partial warps + merge + converters
    for (int i = 0; i < 2; ++i) mbar_init(b + 2 + i, 4 * kGroups + 3 + kI8xConvWarps);
    b += 4;
    for (int i = 0; i < p.n_part; ++i) mbar_init(b + i, 128);            // partfull: the threads of one group
    for (int i = 0; i < p.n_part; ++i) mbar_init(b + p.n_part + i, 5);  // partempty: merge + the group's 4 warps
    mbar_init(b + 2 * p.n_part, 1);                                     // done
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  i8x_query(Q, p.nq, d, sm, NC);
  fence_proxy_async_smem();
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm128);
    tma_prefetch_desc(&tm32);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sm.tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  const int64_t b0 = (p.B * blockIdx.x) / gridDim.x;
  const int64_t b1 = (p.B * (blockIdx.x + 1)) / gridDim.x;

  if (warp == kProducerWarp) {
    i8x_loader(p, sm, br, &tm128, &tm32, d);
  } else if (warp == kMmaWarp) {
    i8x_mma<NC>(p, sm, br, tmem_base);
  } else if (warp == kMergeWarp) {
    run_merge<NG, false, true>(p, sm, br);   // one query, one chunk, one pass
  } else if (warp == kI8xBuilderWarp) {
    run_builder(p, sm, br, b0, b1);
  } else if (warp >= kI8xConvWarp0) {
    if (p.KB == 1) i8x_converters<1>(p, sm, br);
    else if (p.KB == 2) i8x_converters<2>(p, sm, br);
    else i8x_converters<3>(p, sm, br);
  } else {
    i8x_partials<NG>(p, sm, br, tmem_base);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int NG>
cudaError_t i8x_launch(const CUtensorMap& d128, const CUtensorMap& d32, const int8_t* Q, const FwdTcParams& p,
                       int d, int grid, size_t smem, cudaStream_t stream) {
  auto kern = fwd_i8x_kernel<NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, kI8xThreads, smem, stream>>>(d128, d32, Q, p, d);
  return cudaGetLastError();
}

}  // namespace

bool i8x_applicable(int nq, int d, int64_t total_tokens) {
  if (nq < 1 || nq > 64 || (d != 64 && d != 128 && d != kI8xMaxD)) return false;
  if (total_tokens < 1 || total_tokens > (static_cast<int64_t>(1) << 30)) return false;
  const DeviceInfo* dev = device_info();
  const int NC = nq <= 32 ? 32 : 64;
  return dev && i8x_smem_bytes(NC, d, 2, kI8xOp, 512 / NC < 4 ? 512 / NC : 4, 4) <=
                    static_cast<size_t>(dev->max_smem_optin);
}

maxsim_status launch_i8x(const int8_t* Q, const float* q_scale, int nq, int d, const int8_t* D, const float* d_scale,
                         const int64_t* offsets, int64_t B, int64_t total_tokens, float* out, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (!i8x_applicable(nq, d, total_tokens)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;
  const int NG = nq <= 32 ? 1 : 2, NC = 32 * NG;
  const int n_acc = 4, n_part = 4;
  // Two operand stages (the converters fill one while the MMAs read the
  // other) and as many raw stages as fit.
  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  int n_raw = kI8xMaxRaw;
  while (n_raw > 2 && i8x_smem_bytes(NC, d, n_raw, kI8xOp, n_acc, n_part) > budget) --n_raw;
  const size_t smem = i8x_smem_bytes(NC, d, n_raw, kI8xOp, n_acc, n_part);
  if (smem > budget) return MAXSIM_ERR_UNSUPPORTED;

  // documents as a [total_tokens, d] uint8 matrix: boxes of d bytes x 128
  // or 32 rows (64-byte swizzle at d = 64, none otherwise)
  alignas(64) CUtensorMap tm128, tm32;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_tokens)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d)};
  const uint32_t box128[2] = {static_cast<uint32_t>(d), 128}, box32[2] = {static_cast<uint32_t>(d), 32};
  const int swz = d == 64 ? 2 : 0;
  if (!encode_tmap(&tm128, 2, 2, const_cast<int8_t*>(D), ddims, dstrides, box128, swz) ||
      !encode_tmap(&tm32, 2, 2, const_cast<int8_t*>(D), ddims, dstrides, box32, swz))
    return MAXSIM_ERR_CUDA;

  FwdTcParams p;
  p.order = nullptr;
  p.doc_len = nullptr;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_tokens;
  p.nd = 0;
  p.csr = 1;
  p.n_queries = 1;
  p.nq = nq;
  p.KB = KB;
  p.n_chunks = 1;
  p.multipass = 0;
  p.local_finish = 1;
  p.col_scale = q_scale;
  p.row_scale = d_scale;
  p.stages = n_raw;      // raw int8 stages
  p.n_acc = n_acc;
  p.n_qslots = kI8xOp;   // fp16 operand stages
  p.n_part = n_part;
  p.idesc = idesc_f16(0, 128, NC);
  p.tmem_cols = static_cast<uint32_t>(n_acc * NC) <= 128 ? 128u : 256u;
  p.out = out;
  p.argmax = nullptr;
  p.status = dev->status;

  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  const cudaError_t e = NG == 1 ? i8x_launch<1>(tm128, tm32, Q, p, d, grid, smem, stream)
                                : i8x_launch<2>(tm128, tm32, Q, p, d, grid, smem, stream);
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

// fwd_x3.cu -- MaxSim forward for fp32 inputs on the tcgen05 tensor cores.
//
// Computes the same outputs as the fp32 FFMA kernel (fwd_f32.cu):
//   out[b]      = sum_i max_{j < L_b} <Q[i,:], D_b[j,:]>
//   argmax[b,i] = lowest j attaining that maximum
// (TileMaxSim deep reading §1; FLASH-MAXSIM Figure 1 / Algorithm 2), for one
// query of at most 64 tokens.
//
// Three-part bf16 split. A bf16 number holds 8 significant bits, an fp32
// one 24, so every fp32 value x is written on chip as x = x0 + x1 + x2 with
// x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1) (round to nearest
// each time; the differences are exact in fp32, and what x2 leaves out is
// below 2^-26 |x|). Every product of two bf16 numbers is exact in fp32, so
//   <q, d> = sum_{a,b} <q_b, d_a>
// is computed by the tensor core with nothing lost but fp32 accumulation.
// The query's three parts are stacked along the MMA's N dimension (rows
// b*NC .. b*NC+NC-1 of the B operand are part b), and per 16-wide K step
// three MMAs -- one per document part d_a, all into the same accumulator --
// form all nine products: accumulator column group b holds D Q_b^T. The
// epilogue adds the groups, S = G0 + (G1 + G2), before the maximum.
//
// Roles (15 warps), on the chunk-slot walk of fwd_tc.cu (fwd_common.cuh):
//  * Loader (warp 8, lane 0 issues): TMA loads of fp32 document rows into a
//    ring of raw stages, one stage per (tile, 64-dim slice): two 32-float
//    column halves of 128 rows (four contiguous slots: one box per half;
//    otherwise one 32-row box per slot and half).
//  * Converters (warps 11-14): split each raw stage into the three bf16
//    parts, written in the K-major 128-byte-swizzled layout of the MMA's A
//    operand, into a ring of operand stages; then release the raw stage.
//  * MMA (warp 9, lane 0 issues): kind::f16 bf16, M = 128 document rows,
//    N = 3 NC, K = 16: per operand stage 3 parts x 4 K steps.
//  * Slot partials (warps 0-7) and merge (warp 10): as in fwd_tc.cu, with the
//    three column groups added first.
// HBM bytes per document are L_b * d * 4, read once. Every wait is bounded;
// after an abort the loader drains its copies and the MMA thread waits for
// its last MMA before TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "fwd_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

constexpr int kX3ConvWarp0 = 4 * kGroups + 3;        // warps 11-14
constexpr int kX3ConvWarps = 4;
constexpr int kX3Threads = 32 * (4 * kGroups + 3 + kX3ConvWarps);
constexpr int kRawBytes = 128 * 64 * 4;              // one (tile, 64-dim slice) of fp32 rows
constexpr int kPartBytes = 128 * 128;                // one bf16 part of it, 128 B per row
constexpr int kOpBytes = 3 * kPartBytes;             // an operand stage: the three parts
constexpr int kX3MaxRaw = 4, kX3Op = 2;              // ring depths (chosen at launch: p.stages raw, p.n_qslots operand)
constexpr int kX3MaxQBytes = 48 * 1024;              // the stacked query parts (B operand)

struct X3Smem {
  uint8_t* q;            // KB slices x (3 NC rows x 128 B)
  uint8_t* raw;          // p.stages x 32 KB: [half][row][32 fp32]
  uint8_t* op;           // p.n_qslots x 48 KB operand stages: [part][row][64 bf16] swizzled
  GroupTab* tab;         // [2]
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* part_v;         // [PB][4][NC]
  int32_t* part_i;       // [PB][4][NC]
  float* gsum;           // [kCapDocs] (multi-pass only; unused here)
};

__host__ __device__ inline size_t x3_bars_count(int n_raw, int n_op, int n_acc, int n_part) {
  return 2 * n_raw + 2 * n_op + 2 * n_acc + 4 + 2 * n_part + 1;
}

__host__ __device__ inline size_t x3_smem_bytes(int NC, int KB, int n_raw, int n_op, int n_acc, int n_part) {
  size_t bytes = 1024;
  bytes += static_cast<size_t>(KB) * 3 * NC * 128;
  bytes += static_cast<size_t>(n_raw) * kRawBytes + static_cast<size_t>(n_op) * kOpBytes;
  bytes += 2 * sizeof(GroupTab);
  bytes += x3_bars_count(n_raw, n_op, n_acc, n_part) * 8 + 16;
  bytes += static_cast<size_t>(n_part * 4 * NC) * 8;
  bytes += kCapDocs * 4;
  return bytes;
}

__device__ __forceinline__ X3Smem x3_carve(uint8_t* raw, const FwdTcParams& p, int NC) {
  X3Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.q = base;
  s.raw = s.q + static_cast<size_t>(p.KB) * 3 * NC * 128;
  s.op = s.raw + static_cast<size_t>(p.stages) * kRawBytes;
  s.tab = reinterpret_cast<GroupTab*>(s.op + static_cast<size_t>(p.n_qslots) * kOpBytes);
  s.bars = reinterpret_cast<uint64_t*>(s.tab + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + x3_bars_count(p.stages, p.n_qslots, p.n_acc, p.n_part));
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.part_v = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.part_i = reinterpret_cast<int32_t*>(s.part_v + p.n_part * 4 * NC);
  s.gsum = reinterpret_cast<float*>(s.part_i + p.n_part * 4 * NC);
  return s;
}

// Barrier addresses (32-bit shared) in the order of x3_bars_count.
struct X3Bars {
  uint32_t rawfull, rawempty, opfull, opempty, accfull, accempty, tabfull, tabempty, partfull, partempty, done;
  __device__ __forceinline__ X3Bars(const X3Smem& sm, int NR, int NO, int A, int PB) {
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

// Two fp32 values -> their bf16 parts (x0 and the residual x - x0, exact),
// packed as one bf16x2 word (first value in the low half).
__device__ __forceinline__ uint32_t split2(float& a, float& b) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(b), "f"(a));
  a -= __uint_as_float(w << 16);
  b -= __uint_as_float(w & 0xffff0000u);
  return w;
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// Eight fp32 values (dims 8c .. 8c+7 of row r) -> the three bf16 parts, each
// 16 bytes stored at chunk c ^ (r & 7) of row r of its 128-byte-swizzled
// part (parts `part_bytes` apart).
__device__ __forceinline__ void split8_store(float (&v)[8], uint32_t row_addr, int c, int r, uint32_t part_bytes) {
  const uint32_t dst = row_addr + static_cast<uint32_t>((c ^ (r & 7)) << 4);
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = split2(v[2 * k], v[2 * k + 1]);
    sts128(dst + part * part_bytes, w[0], w[1], w[2], w[3]);
  }
}

// --------------------------------------------------------------- loader
__device__ void x3_loader(const FwdTcParams& p, const X3Smem& sm, const X3Bars& br, const CUtensorMap* tm128,
                          const CUtensorMap* tm32, int64_t b0, int64_t b1) {
  const int lane = threadIdx.x & 31;
  if (debug_faults(p.status) & kDebugStallFwdLoader) return;   // test-only switch (maxsim_debug_set_faults)
  const int KB = p.KB, NR = p.stages;
  const uint64_t policy = l2_policy_evict_first();
  const uint32_t raw0 = smem_u32(sm.raw);
  int s = 0;
  uint32_t ph = 0, fills = 0;
  int64_t nb = b0, carry = 0;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    GroupTab* T = sm.tab + buf;
    if (gi >= 2) {
      bool w = true;
      if (lane == 0) w = mbar_wait_a(br.tabempty + 8 * buf, ((gi >> 1) - 1) & 1u, sm.abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) { ok = false; break; }
    }
    if (nb >= b1) {
      if (lane == 0) T->n_docs = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive_a(br.tabfull + 8 * buf);
      break;
    }
    build_group(p, T, nb, b1, carry);
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabfull + 8 * buf);
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
        const uint32_t bytes = contiguous ? static_cast<uint32_t>(kRawBytes) : static_cast<uint32_t>(nslot) * 8192u;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_a(br.rawempty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = br.rawfull + 8 * s;
          const uint32_t dst = raw0 + static_cast<uint32_t>(s) * kRawBytes;
          mbar_arrive_expect_tx_a(fb, bytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int x = kb * 64 + 32 * h;
            if (contiguous) {
              tma_load_2d_a(dst + h * 16384u, tm128, fb, x, rows[0], policy);
            } else {
              for (int w = 0; w < nslot; ++w) tma_load_2d_a(dst + h * 16384u + w * 4096u, tm32, fb, x, rows[w], policy);
            }
          }
          ++fills;
          if (++s == NR) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  if (!ok && lane == 0) {
    // After an abort: wait (bounded) for every load this warp may still have in flight.
    for (uint32_t f = fills > static_cast<uint32_t>(NR) ? fills - NR : 0; f < fills; ++f)
      mbar_wait_drain(sm.bars + (f % NR), (f / NR) & 1u, p.status);
  }
}

// ----------------------------------------------------------- converters
// 128 threads; per stage each handles 8 units (row r, 16-byte chunk c of the
// 64-dim slice): thread t takes c = t % 8 and rows t / 8 + 16 k. Each unit's
// eight values are split into the three bf16 parts of the operand stage.
__device__ void x3_converters(const FwdTcParams& p, const X3Smem& sm, const X3Bars& br) {
  const int ct = threadIdx.x - 32 * kX3ConvWarp0, lane = threadIdx.x & 31;
  const int c = ct & 7, h = c >> 2, cw = c & 3;
  const uint32_t raw0 = smem_u32(sm.raw), op0 = smem_u32(sm.op);
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
    const int n_stages = ((T->n_slots + 3) >> 2) * p.KB;
    for (int st = 0; st < n_stages; ++st) {
      if (!mbar_wait_a(br.rawfull + 8 * s, ph, sm.abort_flag, p.status)) return;
      if (!mbar_wait_a(br.opempty + 8 * o, oph ^ 1u, sm.abort_flag, p.status)) return;
      const uint32_t src = raw0 + static_cast<uint32_t>(s) * kRawBytes + h * 16384u + cw * 32u;
      const uint32_t dst = op0 + static_cast<uint32_t>(o) * kOpBytes;
#pragma unroll 4
      for (int k = 0; k < 8; ++k) {
        const int r = ct / 8 + 16 * k;
        float v[8];
        const float4 a = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(src + r * 128u));
        const float4 b = *reinterpret_cast<const float4*>(__cvta_shared_to_generic(src + r * 128u + 16u));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        split8_store(v, dst + r * 128u, c, r, kPartBytes);
      }
      // generic-proxy writes (read by the tensor core) and reads (the raw
      // stage, next written by TMA) ordered before the async proxy's accesses
      fence_proxy_async_smem();
      mbar_arrive_a(br.opfull + 8 * o);    // every converter thread arrives after its own fence
      mbar_arrive_a(br.rawempty + 8 * s);
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
// Per operand stage (a 64-dim slice of a tile): for each document part a,
// four K steps of M = 128 rows x N = 3 NC stacked query parts.
template <int NC>
__device__ void x3_mma(const FwdTcParams& p, const X3Smem& sm, const X3Bars& br, uint32_t tmem_base) {
  constexpr int N = 3 * NC;
  const int KB = p.KB, A = p.n_acc, NO = p.n_qslots;
  const uint32_t idesc = p.idesc;
  const uint64_t adesc0 = sdesc_k_sw128(smem_u32(sm.op));
  const uint64_t qdesc0 = sdesc_k_sw128(smem_u32(sm.q));
  int o = 0, a = 0;
  uint32_t oph = 0, aph = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) break;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) break;
    const int n_tiles = (T->n_slots + 3) >> 2;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait_a(br.accempty + 8 * a, aph ^ 1u, sm.abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * N);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_a(br.opfull + 8 * o, oph, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t od = adesc0 + static_cast<uint64_t>((o * kOpBytes) >> 4);
        const uint64_t bd = qdesc0 + static_cast<uint64_t>((kb * N * 128) >> 4);
#pragma unroll
        for (int part = 0; part < 3; ++part)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(d_tmem, od + static_cast<uint64_t>((part * kPartBytes) >> 4) + 2 * kk, bd + 2 * kk, idesc,
                     (kb | part | kk) != 0 ? 1u : 0u);
        umma_commit_a(br.opempty + 8 * o);   // operand stage reusable once these MMAs have read it
        if (++o == NO) {
          o = 0;
          oph ^= 1u;
        }
      }
      if (!ok) break;
      umma_commit_a(br.accfull + 8 * a);     // accumulator ready for the epilogue
      if (++a == A) {
        a = 0;
        aph ^= 1u;
      }
    }
    if (!ok) break;
    mbar_arrive_a(br.tabempty + 8 * buf);
  }
  // Wait until every MMA issued by this thread has completed before TMEM is freed.
  umma_commit_a(br.done);
  mbar_wait_drain(reinterpret_cast<uint64_t*>(__cvta_shared_to_generic(br.done)), 0, p.status);
}

// ------------------------------------------------------- slot partials
// As in fwd_tc.cu; the accumulator row holds three column groups (D Q_b^T for
// the query parts b = 0, 1, 2), added before the maximum.
template <int NG, bool ARGMAX>
__device__ void x3_partials(const FwdTcParams& p, const X3Smem& sm, const X3Bars& br, uint32_t tmem_base) {
  constexpr int NC = 32 * NG, N = 3 * NC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const uint32_t grp = warp >> 2;
  const int A = p.n_acc, PB = p.n_part;
  const int lgA = __ffs(A) - 1, lgPB = __ffs(PB) - 1;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
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
      if (!mbar_wait_a(br.partempty + 8 * pb, pph ^ 1u, sm.abort_flag, p.status)) return;
      if (!mbar_wait_a(br.accfull + 8 * a, aph, sm.abort_flag, p.status)) return;
      tc_fence_after();
      const int i0 = 4 * t;
      if (quarter < n_slots - i0) {
        const int info = T->slot_info[i0 + quarter];
        const int vrows = info & 63;
        const int row = (info >> 6) * kSlotRows + lane;
        float* pv = sm.part_v + (pb * 4 + quarter) * NC;
        int32_t* pi = sm.part_i + (pb * 4 + quarter) * NC;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float v[32], v1[32], v2[32];
          const uint32_t col = tmem_base + lane_base + static_cast<uint32_t>(a * N + g * 32);
          tmem_ld_32x32b_x32(col, v);
          tmem_ld_32x32b_x32(col + NC, v1);
          tmem_ld_32x32b_x32(col + 2 * NC, v2);
          if (g == NG - 1) {  // accumulator fully in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
          }
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = lane < vrows ? v[k] + (v1[k] + v2[k]) : -INFINITY;
          float bv;
          int bi;
          warp_column_max<ARGMAX>(v, row, lane, bv, bi);
          pv[g * 32 + lane] = bv;
          if (ARGMAX) pi[g * 32 + lane] = bi;
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
      }
      mbar_arrive_a(br.partfull + 8 * pb);   // every thread of the group arrives (count 128)
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

// The query's three bf16 parts, stacked as the MMA's B operand: per 64-dim
// slice kb, rows b*NC + i (part b of query token i; zero for i >= nq), 128
// bytes each, 16-byte chunk c of row n stored at chunk c ^ (n & 7).
__device__ void x3_split_query(const FwdTcParams& p, const float* Q, const X3Smem& sm, int NC) {
  const int n = p.KB * NC * 8;   // units (kb, token, chunk)
  const uint32_t q0 = smem_u32(sm.q);
  for (int u = threadIdx.x; u < n; u += kX3Threads) {
    const int kb = u / (NC * 8), rem = u - kb * NC * 8, i = rem >> 3, c = rem & 7;
    float v[8];
    if (i < p.nq) {
      const float4* src = reinterpret_cast<const float4*>(Q + static_cast<int64_t>(i) * p.KB * 64 + kb * 64 + c * 8);
      const float4 a = __ldg(src), b = __ldg(src + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 0.f;
    }
    const uint32_t slice = q0 + static_cast<uint32_t>(kb * 3 * NC * 128);
    // row n = part * NC + i: the parts are NC rows (NC * 128 bytes) apart
    split8_store(v, slice + static_cast<uint32_t>(i * 128), c, i, static_cast<uint32_t>(NC * 128));
  }
}

template <int NG, bool ARGMAX>
__global__ void __launch_bounds__(kX3Threads, 1)
    fwd_x3_kernel(const __grid_constant__ CUtensorMap tm128, const __grid_constant__ CUtensorMap tm32,
                  const float* __restrict__ Q, const FwdTcParams p) {
  constexpr int NC = 32 * NG;
  extern __shared__ uint8_t smem_raw[];
  const X3Smem sm = x3_carve(smem_raw, p, NC);
  const X3Bars br(sm, p.stages, p.n_qslots, p.n_acc, p.n_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    uint64_t* b = sm.bars;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(b + s, 1);                            // rawfull: the loader's expect_tx
      mbar_init(b + p.stages + s, 32 * kX3ConvWarps); // rawempty: every converter thread
    }
    b += 2 * p.stages;
    for (int s = 0; s < p.n_qslots; ++s) {
      mbar_init(b + s, 32 * kX3ConvWarps);            // opfull: every converter thread
      mbar_init(b + p.n_qslots + s, 1);               // opempty: the MMA commit
    }
    b += 2 * p.n_qslots;
    for (int i = 0; i < p.n_acc; ++i) mbar_init(b + i, 1);               // accfull
    for (int i = 0; i < p.n_acc; ++i) mbar_init(b + p.n_acc + i, 4);     // accempty: the 4 warps of one group
    b += 2 * p.n_acc;
    // tabempty: MMA + partial warps + merge + converters
    for (int i = 0; i < 2; ++i) mbar_init(b + i, 1);
    for (int i = 0; i < 2; ++i) mbar_init(b + 2 + i, 4 * kGroups + 2 + kX3ConvWarps);
    b += 4;
    for (int i = 0; i < p.n_part; ++i) mbar_init(b + i, 128);            // partfull
    for (int i = 0; i < p.n_part; ++i) mbar_init(b + p.n_part + i, 1);   // partempty
    mbar_init(b + 2 * p.n_part, 1);                                     // done
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  x3_split_query(p, Q, sm, NC);
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
    x3_loader(p, sm, br, &tm128, &tm32, b0, b1);
  } else if (warp == kMmaWarp) {
    if (lane == 0) x3_mma<NC>(p, sm, br, tmem_base);
  } else if (warp == kMergeWarp) {
    run_merge<NG, ARGMAX>(p, sm, br);
  } else if (warp >= kX3ConvWarp0) {
    x3_converters(p, sm, br);
  } else {
    x3_partials<NG, ARGMAX>(p, sm, br, tmem_base);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int NG, bool ARGMAX>
cudaError_t x3_launch(const CUtensorMap& d128, const CUtensorMap& d32, const float* Q, const FwdTcParams& p, int grid,
                      size_t smem, cudaStream_t stream) {
  auto kern = fwd_x3_kernel<NG, ARGMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, kX3Threads, smem, stream>>>(d128, d32, Q, p);
  return cudaGetLastError();
}

}  // namespace

bool fwd_x3_applicable(int n_queries, int nq, int d, int64_t total_rows) {
  if (n_queries != 1 || nq < 1 || nq > 64 || d % 64 != 0 || d < 64) return false;
  if (total_rows < 1 || total_rows > (static_cast<int64_t>(1) << 30)) return false;
  const int NC = nq <= 32 ? 32 : 64;
  if ((d / 64) * 3 * NC * 128 > kX3MaxQBytes) return false;
  const DeviceInfo* dev = device_info();
  const int n_acc = NC == 32 ? 4 : 2, n_part = 4;
  return dev && x3_smem_bytes(NC, d / 64, 2, kX3Op, n_acc, n_part) <= static_cast<size_t>(dev->max_smem_optin);
}

maxsim_status launch_fwd_x3(const float* Q, int nq, int d, const float* D, int64_t total_rows, int csr,
                            const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd, float* out,
                            int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (!fwd_x3_applicable(1, nq, d, total_rows)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;
  const int NG = nq <= 32 ? 1 : 2, NC = 32 * NG, N = 3 * NC;
  const int n_acc = NG == 1 ? 4 : 2;     // 4 x 96 or 2 x 192 of the 512 TMEM columns
  const int n_part = 4;
  // Two operand stages, so the converters fill one while the MMAs read the
  // other, and as many raw stages (bytes in flight from HBM) as then fit,
  // two to four. Measured at d = 128 (two raw stages fit): one operand stage
  // with four raw stages, or a ring of single-part buffers with four raw
  // stages, both ran 18-25 % slower.
  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  int n_raw = kX3MaxRaw;
  const int n_op = kX3Op;
  while (n_raw > 2 && x3_smem_bytes(NC, KB, n_raw, n_op, n_acc, n_part) > budget) --n_raw;
  const size_t smem = x3_smem_bytes(NC, KB, n_raw, n_op, n_acc, n_part);
  if (smem > budget) return MAXSIM_ERR_UNSUPPORTED;

  // documents as a [total_rows, d] fp32 matrix: boxes of 32 floats (128 B,
  // no swizzle) x 128 or 32 rows
  alignas(64) CUtensorMap tm128, tm32;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_rows)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d) * 4};
  const uint32_t box128[2] = {32, 128}, box32[2] = {32, 32};
  if (!encode_tmap(&tm128, 3, 2, const_cast<float*>(D), ddims, dstrides, box128, 0) ||
      !encode_tmap(&tm32, 3, 2, const_cast<float*>(D), ddims, dstrides, box32, 0))
    return MAXSIM_ERR_CUDA;

  FwdTcParams p;
  p.order = nullptr;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = 1;
  p.nq = nq;
  p.KB = KB;
  p.n_chunks = 1;
  p.multipass = 0;
  p.local_finish = 0;
  p.col_scale = nullptr;
  p.row_scale = nullptr;
  p.stages = n_raw;      // raw fp32 stages
  p.n_acc = n_acc;
  p.n_qslots = n_op;     // bf16 operand stages
  p.n_part = n_part;
  p.idesc = idesc_f16(1, 128, N);
  p.tmem_cols = 512;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  cudaError_t e;
  if (NG == 1)
    e = argmax ? x3_launch<1, true>(tm128, tm32, Q, p, grid, smem, stream)
               : x3_launch<1, false>(tm128, tm32, Q, p, grid, smem, stream);
  else
    e = argmax ? x3_launch<2, true>(tm128, tm32, Q, p, grid, smem, stream)
               : x3_launch<2, false>(tm128, tm32, Q, p, grid, smem, stream);
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

maxsim_status launch_fwd_fp32(const float* Q, int n_queries, int nq, int d, const float* D, int64_t total_rows,
                              int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                              float* out, int32_t* argmax, cudaStream_t stream) {
  if (fwd_x3_applicable(n_queries, nq, d, total_rows))
    return launch_fwd_x3(Q, nq, d, D, total_rows, csr, doc_len, offsets, B, nd, out, argmax, stream);
  return launch_fwd_f32(Q, n_queries, nq, d, D, total_rows, csr, doc_len, offsets, B, nd, out, argmax, stream);
}

}  // namespace msim

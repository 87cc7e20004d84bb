// fwd_tc.cu -- MaxSim forward on the 5th-generation tensor cores (tcgen05).
//
// Computes, for every (query q, document b):
//   out[q,b]      = sum_i max_{j < L_b} <Q[q,i,:], D_b[j,:]>
//   argmax[q,b,i] = lowest j attaining that maximum
// (TileMaxSim deep reading §1; FLASH-MAXSIM Figure 1 / Algorithm 2).
//
// Design (GB300 / sm_103a):
//  * Documents are cut into 32-row chunks. A 128-row MMA tile holds four
//    chunk slots; slot w is TMEM lanes 32w..32w+31 and is reduced by epilogue
//    warp w, so a warp's 32 rows always belong to ONE document. Short
//    documents therefore share tiles (four 32-token documents per tile), long
//    ones span tiles, and padding beyond a document's last 32-row granule is
//    never loaded (TileMaxSim §5, the padding waste). Padded (length-masked)
//    and CSR layouts only differ in where a document's rows start.
//  * Persistent grid, one CTA per SM; CTA c owns a contiguous document range
//    and walks it in groups of up to 256 chunks. A builder warp writes each
//    group's slot table in shared memory one group ahead (32 lanes load the
//    document offsets of up to 256 documents at once), so no
//    role waits on a global load in its issue loop and the loader keeps
//    issuing copies across group boundaries.
//  * Loader (one lane issues): TMA loads of 64-dim x 32/128-row boxes,
//    128-byte swizzled, into a ring of 16 KB stages; four contiguous slots go
//    as one 128-row box. Every document byte is read from HBM once per
//    (query, query chunk) pass -- with one query of up to 256 tokens that is
//    the single pass of TileMaxSim §2(1) (BQ = Nq). With several queries or
//    query chunks, all passes run over one group (<= 256 chunks) before the
//    next, so the repeats are served by L2.
//  * MMA warp: tcgen05.mma kind::f16, M = 128 rows, N = NC query tokens,
//    K = 16; every 64-wide d-slice of a tile accumulates into the same TMEM
//    accumulator before any maximum is taken (TileMaxSim §2(2), dimension
//    tiling). Up to four accumulators let it run ahead. The whole warp runs
//    the issue loop and one elected lane issues each MMA: with the loop
//    warp-uniform, issuing costs about half the cycles per MMA of a loop run
//    by one lane alone.
//  * Slot partials (warps 0 .. 4G-1, G = 2 or 3 groups of four taking tiles
//    round-robin; warp w reads TMEM lane quarter w % 4; then come the loader,
//    MMA, merge and builder warps): tcgen05.ld of 32 lanes, rows past
//    the chunk's valid rows masked to -inf, a transpose butterfly of shuffles
//    leaves lane l with the maximum (and lowest argmax) of query column l
//    over the slot, handed over in a ring of shared-memory buffers. A
//    document whose slots all lie in one tile (every document of up to 128
//    tokens that starts on a tile boundary, e.g. Nd = 32 / 64 / 128) is
//    finished by the group itself: one of its slots' warps (in turn, tile by
//    tile) folds its slots, sums the per-token maxima and writes the score;
//    a one-slot document from registers, without waiting for the others.
//  * Merge warp: folds the slot partials of documents that span tiles,
//    in document order, and when such a document ends sums its per-token
//    maxima and writes the score (FLASH-MAXSIM Figure 1: only the scalar
//    score is written). Partial warps never wait for the merge except
//    through the buffer ring. The similarity tile exists only in TMEM and
//    registers.
//  * Every mbarrier wait is bounded (ptx.cuh); after an abort the producer
//    drains its in-flight TMA loads and the MMA thread waits for its last MMA
//    before TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "fwd_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {

// Roles by warp index for G groups of four slot-partial warps (warps
// 0 .. 4G-1): then the loader, the MMA warp, the merge warp and the table
// builder. G = 3 when the partial warps bind (argmax, or d = 64 with
// documents of at most 256 tokens), else 2.
template <int G> struct TcRoles {
  static constexpr int kLoader = 4 * G, kMma = 4 * G + 1, kMerge = 4 * G + 2, kBuilder = 4 * G + 3;
  static constexpr int kThreads = 32 * (4 * G + 4);
};

struct Smem {
  uint8_t* q;            // n_qslots x KB boxes of NC rows x 128 B
  uint8_t* stages;       // stages x 16 KB
  GroupTab* tab;         // [2]
  uint64_t* bars;        // full[S] empty[S] qfull[2] qempty[2] accfull[A] accempty[A] tabfull[2] tabempty[2]
                         // partfull[PB] partempty[PB] done
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* part_v;         // [PB][4][NC]
  int32_t* part_i;       // [PB][4][NC]
  float* gsum;           // [kCapDocs]
};

__host__ __device__ inline size_t bars_count(int stages, int n_acc, int n_part) {
  return 2 * stages + 4 + 2 * n_acc + 4 + 2 * n_part + 1;
}

__host__ __device__ inline size_t smem_bytes_for(int NC, int KB, int stages, int n_acc, int n_qslots, int n_part) {
  size_t bytes = 1024;  // alignment slack for the dynamic region
  bytes += static_cast<size_t>(n_qslots) * KB * NC * 128;
  bytes += static_cast<size_t>(stages) * kStageBytes;
  bytes += 2 * sizeof(GroupTab);
  bytes += bars_count(stages, n_acc, n_part) * 8;
  bytes += 16;
  bytes += static_cast<size_t>(n_part * 4 * NC) * 8;
  bytes += kCapDocs * 4;
  return bytes;
}

__device__ __forceinline__ Smem carve(uint8_t* raw, const FwdTcParams& p, int NC) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.q = base;
  s.stages = s.q + static_cast<size_t>(p.n_qslots) * p.KB * NC * 128;
  s.tab = reinterpret_cast<GroupTab*>(s.stages + static_cast<size_t>(p.stages) * kStageBytes);
  s.bars = reinterpret_cast<uint64_t*>(s.tab + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + bars_count(p.stages, p.n_acc, p.n_part));
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.part_v = reinterpret_cast<float*>(s.tmem_slot + 4);
  s.part_i = reinterpret_cast<int32_t*>(s.part_v + p.n_part * 4 * NC);
  s.gsum = reinterpret_cast<float*>(s.part_i + p.n_part * 4 * NC);
  return s;
}

// Barrier addresses (32-bit shared) in the order laid out by carve().
struct Bars {
  uint32_t full, empty, qfull, qempty, accfull, accempty, tabfull, tabempty, partfull, partempty, done;
  __device__ __forceinline__ Bars(const Smem& sm, int S, int A, int PB) {
    const uint32_t b0 = smem_u32(sm.bars);
    full = b0;
    empty = full + 8 * S;
    qfull = empty + 8 * S;
    qempty = qfull + 16;
    accfull = qempty + 16;
    accempty = accfull + 8 * A;
    tabfull = accempty + 8 * A;
    tabempty = tabfull + 16;
    partfull = tabempty + 16;
    partempty = partfull + 8 * PB;
    done = partempty + 8 * PB;
  }
};

template <int NC>
__device__ void run_producer(const FwdTcParams& p, const Smem& sm, const Bars& br, const CUtensorMap* tm_d128,
                             const CUtensorMap* tm_d32, const CUtensorMap* tm_q) {
  const int lane = threadIdx.x & 31;
  // Test-only fault switch (maxsim_debug_set_faults): the loader issues
  // nothing, so every other role's bounded wait runs out and the CTA aborts
  // with no copy or MMA in flight.
  if (debug_faults(p.status) & kDebugStallFwdLoader) return;
  const int S = p.stages, KB = p.KB, NQS = p.n_qslots;
  const uint32_t qbytes = static_cast<uint32_t>(KB) * NC * 128;
  const uint64_t policy = l2_policy_evict_first();
  const uint32_t stage0 = smem_u32(sm.stages);
  const uint32_t q0 = smem_u32(sm.q);
  int s = 0;
  uint32_t ph = 0, fills = 0, quse = 0;
  int prev_key = -1;
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
      for (int q = 0; q < p.n_queries && ok; ++q) {
        for (int c = 0; c < p.n_chunks && ok; ++c) {
          if (n_tiles == 0) continue;
          const int key = q * p.n_chunks + c;
          if (key != prev_key) {
            const int slot = static_cast<int>(quse % NQS);
            const uint32_t use = quse / NQS;
            if (use > 0 && !mbar_wait_a(br.qempty + 8 * slot, (use - 1) & 1u, sm.abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx_a(br.qfull + 8 * slot, qbytes);
            for (int kb = 0; kb < KB; ++kb)
              tma_load_3d_a(q0 + static_cast<uint32_t>((slot * KB + kb) * NC * 128), tm_q, br.qfull + 8 * slot,
                            kb * 64, c * NC, q);
            ++quse;
            prev_key = key;
          }
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
            const uint32_t bytes = contiguous ? 16384u : static_cast<uint32_t>(nslot) * 4096u;
            for (int kb = 0; kb < KB; ++kb) {
              if (!mbar_wait_a(br.empty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
                ok = false;
                break;
              }
              const uint32_t fb = br.full + 8 * s;
              const uint32_t dst = stage0 + static_cast<uint32_t>(s) * kStageBytes;
              mbar_arrive_expect_tx_a(fb, bytes);
              if (contiguous) {
                tma_load_2d_a(dst, tm_d128, fb, kb * 64, rows[0], policy);
              } else {
                for (int w = 0; w < nslot; ++w) tma_load_2d_a(dst + w * 4096u, tm_d32, fb, kb * 64, rows[w], policy);
              }
              ++fills;
              if (++s == S) {
                s = 0;
                ph ^= 1u;
              }
            }
          }
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    if (ok && lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);   // slot rows read
  }
  if (!ok && lane == 0) {
    // After an abort: wait (bounded) for every load this warp may still have in flight.
    for (uint32_t f = fills > static_cast<uint32_t>(S) ? fills - S : 0; f < fills; ++f)
      mbar_wait_drain(sm.bars + (f % S), (f / S) & 1u, p.status);
    for (uint32_t u = quse > static_cast<uint32_t>(NQS) ? quse - NQS : 0; u < quse; ++u)
      mbar_wait_drain(sm.bars + 2 * S + (u % NQS), (u / NQS) & 1u, p.status);
  }
}

// ----------------------------------------------------------------- MMA warp
// The whole warp runs the issue loop (warp-uniform control flow); one
// elected lane issues each MMA and commit.
template <int NC>
__device__ void run_mma(const FwdTcParams& p, const Smem& sm, const Bars& br, uint32_t tmem_base) {
  const int lane = threadIdx.x & 31;
  const int S = p.stages, KB = p.KB, NQS = p.n_qslots, A = p.n_acc;
  const uint32_t idesc = p.idesc;
  const uint64_t adesc0 = sdesc_k_sw128(smem_u32(sm.stages));
  const uint64_t qdesc0 = sdesc_k_sw128(smem_u32(sm.q));
  int s = 0, a = 0;
  uint32_t ph = 0, aph = 0, quse = 0;
  int prev_key = -1, slot = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!__all_sync(0xffffffffu, mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status))) break;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) break;
    const int n_tiles = (T->n_slots + 3) >> 2;
    bool ok = true;
    for (int q = 0; q < p.n_queries && ok; ++q) {
      for (int c = 0; c < p.n_chunks && ok; ++c) {
        if (n_tiles == 0) continue;
        const int key = q * p.n_chunks + c;
        if (key != prev_key) {
          if (prev_key >= 0) umma_commit_el(br.qempty + 8 * slot);  // slot free once its MMAs retire
          slot = static_cast<int>(quse % NQS);
          if (!__all_sync(0xffffffffu, mbar_wait_a(br.qfull + 8 * slot, (quse / NQS) & 1u, sm.abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          ++quse;
          prev_key = key;
        }
        const uint64_t qdesc = qdesc0 + static_cast<uint64_t>((slot * KB * NC * 128) >> 4);
        for (int t = 0; t < n_tiles; ++t) {
          if (!__all_sync(0xffffffffu, mbar_wait_a(br.accempty + 8 * a, aph ^ 1u, sm.abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * NC);
          for (int kb = 0; kb < KB; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait_a(br.full + 8 * s, ph, sm.abort_flag, p.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = adesc0 + static_cast<uint64_t>(s * (kStageBytes >> 4));
            const uint64_t bd = qdesc + static_cast<uint64_t>((kb * NC * 128) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_f16_el(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            umma_commit_el(br.empty + 8 * s);  // stage reusable once these MMAs have read it
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_el(br.accfull + 8 * a);  // accumulator ready for the epilogue
          if (++a == A) {
            a = 0;
            aph ^= 1u;
          }
        }
      }
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
  // Wait until every MMA issued by this warp has completed before TMEM is freed.
  umma_commit_el(br.done);
  mbar_wait_drain(sm.bars + (br.done - br.full) / 8, 0, p.status);
}

// --------------------------------------------------------- partial warps 0-3
// Warp w reduces slot w of every tile: TMEM lanes 32w..32w+31 hold 32 rows of
// one document; the butterfly leaves the slot's per-column maxima in
// part[pbuf][w][:], handed to the merge warp through partfull/partempty.
template <int NG, bool ARGMAX, int G>
__device__ void run_partials(const FwdTcParams& p, const Smem& sm, const Bars& br, uint32_t tmem_base) {
  constexpr int NC = 32 * NG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;            // slot index == TMEM lane quarter
  const uint32_t grp = warp >> 2;          // groups take tiles round-robin
  const int A = p.n_acc, PB = p.n_part;    // both multiples of G
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  uint32_t tt = 0;                         // global tile counter (same sequence as the MMA and merge)
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const GroupTab* T = sm.tab + buf;
    if (T->n_docs < 0) break;
    const int n_slots = T->n_slots;
    const int n_tiles = (n_slots + 3) >> 2;
    const int passes = p.n_queries * p.n_chunks;
    for (int pass = 0; pass < passes; ++pass) {
      for (int t = 0; t < n_tiles; ++t, ++tt) {
        if (tt % G != grp) continue;
        // tile tt uses entry tt % n of a ring of n (n = A or PB, a multiple of
        // G times a power of two): each entry is used by one group only, in
        // that group's tile order, so no wait can run two phases ahead
        const uint32_t tg = tt / G;
        const int a = static_cast<int>(tt % G) + G * static_cast<int>(tg & static_cast<uint32_t>(A / G - 1));
        const uint32_t aph = (tg >> (__ffs(A / G) - 1)) & 1u;
        const int pb = static_cast<int>(tt % G) + G * static_cast<int>(tg & static_cast<uint32_t>(PB / G - 1));
        const uint32_t pph = (tg >> (__ffs(PB / G) - 1)) & 1u;
        if (!mbar_wait_a(br.partempty + 8 * pb, pph ^ 1u, sm.abort_flag, p.status)) return;
        if (!mbar_wait_a(br.accfull + 8 * a, aph, sm.abort_flag, p.status)) return;
        tc_fence_after();
        const int i0 = 4 * t;
        float own_v[NG];
        int own_i[NG];
        if (quarter < n_slots - i0) {
          const int info = T->slot_info[i0 + quarter];
          const int vrows = info & 63;
          const int row = (info >> 6) * kSlotRows + lane;   // doc-local token index of this lane's row
          float* pv = sm.part_v + (pb * 4 + quarter) * NC;
          int32_t* pi = sm.part_i + (pb * 4 + quarter) * NC;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            float v[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(a * NC + g * 32), v);
            if (g == NG - 1) {  // accumulator fully in registers: hand it back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
            }
            if (lane >= vrows) {
#pragma unroll
              for (int k = 0; k < 32; ++k) v[k] = -INFINITY;
            }
            float bv;
            int bi;
            warp_column_max<ARGMAX>(v, row, lane, bv, bi);
            pv[g * 32 + lane] = bv;
            if (ARGMAX) pi[g * 32 + lane] = bi;
            own_v[g] = bv;
            own_i[g] = bi;
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
        }
        mbar_arrive_a(br.partfull + 8 * pb);  // every thread of the group arrives (count 128)
        // A document whose slots all lie in this tile is finished here, by one
        // of its slots' warps (taken in turn from tile to tile); a one-slot
        // document by its own warp from registers, a longer one once the whole
        // group has written its slots.
        if (quarter < n_slots - i0) {
          const int sd = T->slot_doc[i0 + quarter];
          if (sd & kSlotLocal) {
            const int info = T->slot_info[i0 + quarter];
            const int ncs = (sd >> 17) & 7;
            const int f0 = quarter - (info >> 6);            // the document's first slot in the tile
            const int fin = ncs == 1 ? f0 : f0 + static_cast<int>((tt >> 1) % static_cast<uint32_t>(ncs));
            if (quarter == fin) {
              if (ncs > 1 && !mbar_wait_a(br.partfull + 8 * pb, pph, sm.abort_flag, p.status)) return;
              const int64_t bd = doc_at(p, T->first_doc + (sd & kSlotDocMask));
              float sum = 0.f;
#pragma unroll
              for (int g = 0; g < NG; ++g) {
                float m = own_v[g];
                int mi = own_i[g];
                if (ncs > 1) {
                  m = -INFINITY;
                  mi = INT_MAX;
                  for (int j = 0; j < ncs; ++j) {
                    const int o = (pb * 4 + f0 + j) * NC + g * 32 + lane;
                    const float v2 = sm.part_v[o];
                    if (ARGMAX) {
                      const int i2 = sm.part_i[o];
                      if (v2 > m || (v2 == m && i2 < mi)) {
                        m = v2;
                        mi = i2;
                      }
                    } else {
                      m = fmaxf(m, v2);
                    }
                  }
                }
                const int qc = g * 32 + lane;
                if (qc < p.nq) {
                  sum += m;
                  if (ARGMAX && bd >= 0) p.argmax[bd * p.nq + qc] = mi;
                }
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

// SINGLE: one query, one column chunk, one pass (the merge's other paths
// are compiled out).
template <int NG, bool ARGMAX, int G, bool SINGLE = false>
__global__ void __launch_bounds__(TcRoles<G>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_d128, const __grid_constant__ CUtensorMap tm_d32,
                  const __grid_constant__ CUtensorMap tm_q, const FwdTcParams p) {
  constexpr int NC = 32 * NG;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve(smem_raw, p, NC);
  const Bars br(sm, p.stages, p.n_acc, p.n_part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(sm.bars + s, 1);                 // full
      mbar_init(sm.bars + p.stages + s, 1);      // empty
    }
    uint64_t* rest = sm.bars + 2 * p.stages;
    for (int i = 0; i < 4; ++i) mbar_init(rest + i, 1);                    // qfull[2], qempty[2]
    for (int i = 0; i < p.n_acc; ++i) mbar_init(rest + 4 + i, 1);          // accfull
    for (int i = 0; i < p.n_acc; ++i) mbar_init(rest + 4 + p.n_acc + i, 4);  // accempty: the 4 warps of one group
    for (int i = 0; i < 2; ++i) mbar_init(rest + 4 + 2 * p.n_acc + i, 1);  // tabfull
    for (int i = 0; i < 2; ++i) mbar_init(rest + 6 + 2 * p.n_acc + i, 4 * G + 3);  // tabempty: loader + MMA + partials + merge
    uint64_t* pr = rest + 8 + 2 * p.n_acc;
    for (int i = 0; i < p.n_part; ++i) mbar_init(pr + i, 128);             // partfull: the threads of one group
    for (int i = 0; i < p.n_part; ++i) mbar_init(pr + p.n_part + i, 5);    // partempty: merge warp + the group's 4 warps
    mbar_init(pr + 2 * p.n_part, 1);                                       // done
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TcRoles<G>::kLoader && lane == 0) {
    tma_prefetch_desc(&tm_d128);
    tma_prefetch_desc(&tm_d32);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == TcRoles<G>::kMma) {
    tmem_alloc(sm.tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  const int64_t b0 = (p.B * blockIdx.x) / gridDim.x;
  const int64_t b1 = (p.B * (blockIdx.x + 1)) / gridDim.x;

  if (warp == TcRoles<G>::kLoader) {
    run_producer<NC>(p, sm, br, &tm_d128, &tm_d32, &tm_q);
  } else if (warp == TcRoles<G>::kBuilder) {
    run_builder(p, sm, br, b0, b1);
  } else if (warp == TcRoles<G>::kMma) {
    run_mma<NC>(p, sm, br, tmem_base);
  } else if (warp == TcRoles<G>::kMerge) {
    run_merge<NG, ARGMAX, SINGLE>(p, sm, br);
  } else {
    run_partials<NG, ARGMAX, G>(p, sm, br, tmem_base);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TcRoles<G>::kMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <int NG, bool ARGMAX, int G, bool SINGLE = false>
cudaError_t launch_variant(const CUtensorMap& d128, const CUtensorMap& d32, const CUtensorMap& tq,
                           const FwdTcParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = fwd_tc_kernel<NG, ARGMAX, G, SINGLE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, TcRoles<G>::kThreads, smem, stream>>>(d128, d32, tq, p);
  return cudaGetLastError();
}

}  // namespace

maxsim_status launch_fwd_tc(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows,
                            int csr, const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd,
                            int is_bf16, float* out, int32_t* argmax, cudaStream_t stream, const int32_t* order) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (d % 64 != 0 || d < 64 || d > 1024) return MAXSIM_ERR_UNSUPPORTED;
  // rows are int32 TMA coordinates and chunk indices are packed above 6 bits
  if (total_rows < 1 || total_rows > (static_cast<int64_t>(1) << 30)) return MAXSIM_ERR_UNSUPPORTED;
  // long queries: query-major kernel (document tiles reused across 512 query rows)
  if (fwd_qm_applicable(nq, d, total_rows)) {
    if (order) return MAXSIM_ERR_UNSUPPORTED;   // the long-query kernel walks documents in index order
    return launch_fwd_qm(Q, n_queries, nq, d, D, total_rows, csr, doc_len, offsets, B, nd, is_bf16, out, argmax,
                         stream);
  }
  const int KB = d / 64;

  // Query chunk width NC = 32 * NG: as wide as nq needs (up to 256 columns,
  // the largest N of one MMA), with the resident query chunk <= 96 KB.
  const int ng_need = (nq + 31) / 32;
  int ng_cap = static_cast<int>((96 * 1024) / (static_cast<size_t>(KB) * 4096));
  if (ng_cap < 1) ng_cap = 1;
  int NG = 1;
  while (NG < ng_need && NG < 8 && NG * 2 <= ng_cap) NG *= 2;
  const int NC = 32 * NG;
  const int n_chunks = (nq + NC - 1) / NC;
  const int multipass = (n_queries * n_chunks > 1) ? 1 : 0;
  // multi-pass groups hold whole documents of at most 256 chunks
  if (multipass && !csr && nd > kCapSlots * kSlotRows) return MAXSIM_ERR_UNSUPPORTED;
  // Three groups of slot-partial warps where they bind (measured: argmax
  // +10 %, d = 64 with Nd <= 256 +3-8 %), two elsewhere; with three, the
  // accumulators and part buffers come in multiples of three (one set per
  // group), so N <= 128.
  const bool am = argmax != nullptr;
  const bool g3 = (am || (KB == 1 && !csr && nd <= 256)) && NC <= 128;
  const int n_acc = g3 ? 3 * ((512 / NC) / 3 >= 2 ? 2 : 1) : ((512 / NC) < kMaxAcc ? (512 / NC) : kMaxAcc);
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(n_acc * NC)) tmem_cols <<= 1;

  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  const int n_part = g3 ? 3 : (NC >= 128 ? 2 : 4);
  int n_qslots = 1;
  if (multipass && smem_bytes_for(NC, KB, 4, n_acc, 2, n_part) <= budget) n_qslots = 2;
  int stages = 16;
  while (stages > 2 && smem_bytes_for(NC, KB, stages, n_acc, n_qslots, n_part) > budget) --stages;
  const size_t smem = smem_bytes_for(NC, KB, stages, n_acc, n_qslots, n_part);
  if (smem > budget) return MAXSIM_ERR_UNSUPPORTED;

  // TMA descriptors: documents as a [total_rows, d] matrix (128- and 32-row
  // boxes) and queries as [n_queries, nq, d] so rows past nq read as zero.
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
  p.order = order;
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
  p.multipass = multipass;
  p.local_finish = multipass ? 0 : 1;
  p.col_scale = nullptr;
  p.row_scale = nullptr;
  p.stages = stages;
  p.n_acc = n_acc;
  p.n_qslots = n_qslots;
  p.n_part = n_part;
  p.idesc = idesc_f16(is_bf16, 128, NC);
  p.tmem_cols = tmem_cols;
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  const int grid = static_cast<int>(B < dev->sm_count ? B : dev->sm_count);
  cudaError_t e;
#define MAXSIM_TC_LAUNCH(NGv, AMv) \
  (g3 ? launch_variant<NGv, AMv, 3>(tm_d128, tm_d32, tm_q, p, grid, smem, stream) \
      : launch_variant<NGv, AMv, 2>(tm_d128, tm_d32, tm_q, p, grid, smem, stream))
  // Scores-only launches of one query (up to 32 tokens), one chunk and one
  // pass take the merge walk compiled for that case where documents end
  // inside tiles or span them (CSR, length-masked, d = 64): measured +3 %
  // length-masked and CSR, +9 % at d = 64 with 256-token documents. Full-length
  // documents at d >= 128, the cheapest walk, measured ~1 % slower with it
  // and keep the general build.
  const bool single = !am && NG == 1 && n_queries == 1 && !multipass && p.n_chunks == 1 &&
                      (csr || doc_len != nullptr || KB == 1);
  switch (NG) {
    case 1:
      if (single)
        e = g3 ? launch_variant<1, false, 3, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream)
               : launch_variant<1, false, 2, true>(tm_d128, tm_d32, tm_q, p, grid, smem, stream);
      else
        e = am ? MAXSIM_TC_LAUNCH(1, true) : MAXSIM_TC_LAUNCH(1, false);
      break;
    case 2: e = am ? MAXSIM_TC_LAUNCH(2, true) : MAXSIM_TC_LAUNCH(2, false); break;
    case 4: e = am ? MAXSIM_TC_LAUNCH(4, true) : MAXSIM_TC_LAUNCH(4, false); break;
    default: e = am ? MAXSIM_TC_LAUNCH(8, true) : MAXSIM_TC_LAUNCH(8, false); break;
  }
#undef MAXSIM_TC_LAUNCH
  return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

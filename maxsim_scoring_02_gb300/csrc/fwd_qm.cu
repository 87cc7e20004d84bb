// fwd_qm.cu -- MaxSim forward for long queries, query-major on tcgen05.
//
// Same operator and outputs as fwd_tc.cu (TileMaxSim deep reading §1;
// FLASH-MAXSIM Figure 1 / Algorithm 2), for queries of a few hundred to 1024
// tokens (ColPali-style Lq = 1024), where the contraction is tensor-bound:
//  * A = a resident set of up to four 128-row query blocks of one query
//    (M = 128 query tokens per MMA); B = a 128-token document tile streamed
//    by TMA (N = 128 document tokens). Every document tile in shared memory
//    is multiplied against all resident query blocks, so one tile fill feeds
//    up to 512 query rows (16 B of fill per SM clock at the tensor rate).
//  * TMEM lane = query row, column = document token: the maximum over the
//    document's tokens is thread-local (a 3-input max tree per 32-column
//    chunk); the argmax is searched only in a chunk that raises the running
//    maximum. No similarity value leaves the SM.
//  * Work items are (query set, document) pairs in set-major order, split
//    contiguously over a persistent grid; a set's partial score is added to
//    out[q, b] (zeroed first). A query has at most two sets, and a + b equals
//    b + a in floating point, so the result does not depend on which set
//    lands first.
//  * Warps: 0-3 epilogue (TMEM lanes 0-127), 4 producer (item tables, TMA),
//    5 MMA issuer. Every wait is a bounded mbarrier wait (ptx.cuh); there is
//    no named barrier, so an abort cannot strand a warp.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

#ifndef MAXSIM_QM_MIN_NQ
#define MAXSIM_QM_MIN_NQ 257
#endif

namespace msim {
namespace {

constexpr int kQmThreads = 192;
constexpr int kQmTile = 128;             // document tokens per tile (MMA N)
constexpr int kQmBlock = 128;            // query rows per block (MMA M)
constexpr int kQmMaxBlocks = 4;          // query blocks per resident set
constexpr int kQmMaxSets = 2;            // sets per query (keeps the sum order-free)
constexpr int kQmStage = kQmTile * 128;  // one 64-dim box of a tile: 16 KB
constexpr int kQmAcc = 4;                // TMEM accumulators of 128 columns
constexpr int kQmItems = 32;             // items per table

struct QmParams {
  const int32_t* doc_len;
  const int64_t* offsets;
  int64_t B, total_rows;
  int nd, csr;
  int n_queries, nq, KB;
  int set_blocks;  // query blocks per set (<= 4)
  int sets_per_query;
  int stages;
  uint32_t idesc;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

struct QmItem {
  int64_t b;
  int32_t start;  // first row of the document in D
  int32_t L;      // tokens (0: empty or rejected)
  int32_t set;
  int32_t pad;
};
struct ItemTab {
  int32_t n;  // items in the table; -1 = end of work
  int32_t pad;
  QmItem item[kQmItems];
};

// Barrier block: full[S] empty[S] qfull qempty accfull[4] accempty[4]
// tabfull[2] tabempty[2] redfull[2] redempty[2] done.
__host__ __device__ constexpr int qm_bars(int S) { return 2 * S + 2 + 2 * kQmAcc + 8 + 1; }
// Small structures first, then the 1024-byte aligned operand region (worst
// case padding counted).
__host__ __device__ constexpr size_t qm_small_bytes(int S) {
  return 2 * sizeof(ItemTab) + static_cast<size_t>(qm_bars(S)) * 8 + 16 + 8 * 4;
}
__host__ __device__ constexpr size_t qm_smem_bytes(int KB, int set_blocks, int S) {
  return qm_small_bytes(S) + 1023 + static_cast<size_t>(set_blocks) * KB * kQmBlock * 128 +
         static_cast<size_t>(S) * kQmStage;
}

struct QmSmem {
  ItemTab* tab;    // [2]
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* red;      // [2 slots][4 warps]
  uint8_t* q;      // [set_blocks][KB][128 rows][128 B], SW128
  uint8_t* stages; // [S][128 rows][128 B], SW128
};

__device__ __forceinline__ QmSmem qm_carve(uint8_t* raw, const QmParams& p) {
  QmSmem s;
  s.tab = reinterpret_cast<ItemTab*>(raw);
  s.bars = reinterpret_cast<uint64_t*>(s.tab + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + qm_bars(p.stages));
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.red = reinterpret_cast<float*>(s.tmem_slot + 4);
  const uintptr_t end = reinterpret_cast<uintptr_t>(raw) + qm_small_bytes(p.stages);
  s.q = reinterpret_cast<uint8_t*>((end + 1023) & ~uintptr_t(1023));
  s.stages = s.q + static_cast<size_t>(p.set_blocks) * p.KB * kQmBlock * 128;
  return s;
}

struct QmBars {
  uint32_t full, empty, qfull, qempty, accfull, accempty, tabfull, tabempty, redfull, redempty, done;
  __device__ __forceinline__ QmBars(const QmSmem& sm, int S) {
    full = smem_u32(sm.bars);
    empty = full + 8 * S;
    qfull = empty + 8 * S;
    qempty = qfull + 8;
    accfull = qempty + 8;
    accempty = accfull + 8 * kQmAcc;
    tabfull = accempty + 8 * kQmAcc;
    tabempty = tabfull + 16;
    redfull = tabempty + 16;
    redempty = redfull + 16;
    done = redempty + 16;
  }
};

// Query blocks of a set that hold at least one real query row.
__device__ __forceinline__ int qm_blocks_of_set(const QmParams& p, int set) {
  const int r0 = (set % p.sets_per_query) * p.set_blocks * kQmBlock;
  const int left = (p.nq - r0 + kQmBlock - 1) / kQmBlock;
  return left < p.set_blocks ? left : p.set_blocks;
}

// ------------------------------------------------------------ producer warp
// All lanes build item tables; lane 0 issues the query-set and tile loads.
__device__ void qm_producer(const QmParams& p, const QmSmem& sm, const QmBars& br, const CUtensorMap* tm_d,
                            const CUtensorMap* tm_q, int64_t i0, int64_t i1) {
  const int lane = threadIdx.x & 31;
  const int S = p.stages, KB = p.KB;
  const uint64_t policy = l2_policy_evict_first();
  const uint32_t stage0 = smem_u32(sm.stages), q0 = smem_u32(sm.q);
  int s = 0;
  uint32_t ph = 0, fills = 0, qloads = 0;
  int prev_set = -1;
  bool ok = true;
  int64_t it = i0;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    ItemTab* T = sm.tab + buf;
    if (gi >= 2) {
      bool w = true;
      if (lane == 0) w = mbar_wait_a(br.tabempty + 8 * buf, ((gi >> 1) - 1) & 1u, sm.abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
    }
    int n = 0;
    while (n < kQmItems && it + n < i1) {
      const int64_t item = it + n + lane;
      if (n + lane < kQmItems && item < i1) {
        const int set = static_cast<int>(item / p.B);
        const int64_t b = item - static_cast<int64_t>(set) * p.B;
        int64_t start = 0, L = 0;
        bool bad = false;
        if (p.csr) {
          const int64_t s0 = __ldg(p.offsets + b), e0 = __ldg(p.offsets + b + 1);
          bad = s0 < 0 || e0 < s0 || e0 > p.total_rows;
          start = bad ? 0 : s0;
          L = bad ? 0 : e0 - s0;
        } else {
          start = b * static_cast<int64_t>(p.nd);
          L = p.doc_len ? static_cast<int64_t>(__ldg(p.doc_len + b)) : static_cast<int64_t>(p.nd);
          bad = L < 0 || L > p.nd;
          if (bad) L = 0;
        }
        if (bad) atomicOr(p.status, kDevErrBadInput);
        QmItem& e = T->item[n + lane];
        e.b = b;
        e.start = static_cast<int32_t>(start);
        e.L = static_cast<int32_t>(L);
        e.set = set;
      }
      const int64_t left = i1 - (it + n);
      n += static_cast<int>(left < 32 ? left : 32);
      if (n > kQmItems) n = kQmItems;
    }
    it += n;
    if (lane == 0) T->n = n > 0 ? n : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabfull + 8 * buf);
    if (n == 0) break;
    if (lane == 0) {
      for (int k = 0; k < n && ok; ++k) {
        const QmItem e = T->item[k];
        const int ntiles = (e.L + kQmTile - 1) / kQmTile;
        if (ntiles == 0) continue;
        if (e.set != prev_set) {  // load the next query set once the last one's MMAs retired
          if (qloads > 0 && !mbar_wait_a(br.qempty, (qloads - 1) & 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int q = e.set / p.sets_per_query;
          const int r0 = (e.set % p.sets_per_query) * p.set_blocks * kQmBlock;
          const int nb = qm_blocks_of_set(p, e.set);
          mbar_arrive_expect_tx_a(br.qfull, static_cast<uint32_t>(nb * KB * kQmBlock * 128));
          for (int j = 0; j < nb; ++j)
            for (int kb = 0; kb < KB; ++kb)
              tma_load_3d_a(q0 + static_cast<uint32_t>((j * KB + kb) * kQmBlock * 128), tm_q, br.qfull, kb * 64,
                            r0 + j * kQmBlock, q);
          ++qloads;
          prev_set = e.set;
        }
        for (int t = 0; t < ntiles && ok; ++t) {
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_a(br.empty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx_a(br.full + 8 * s, kQmStage);
            tma_load_2d_a(stage0 + static_cast<uint32_t>(s) * kQmStage, tm_d, br.full + 8 * s, kb * 64,
                          e.start + t * kQmTile, policy);
            ++fills;
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  if (!ok && lane == 0) {  // let copies in flight land before the CTA exits
    for (uint32_t f = fills > static_cast<uint32_t>(S) ? fills - S : 0; f < fills; ++f)
      mbar_wait_drain(sm.bars + (f % S), (f / S) & 1u, p.status);
    if (qloads > 0) mbar_wait_drain(sm.bars + 2 * S, (qloads - 1) & 1u, p.status);
  }
}

// ----------------------------------------------------------------- MMA warp
// One thread. Per tile: wait for its KB stages, then for each query block j
// accumulate Q_j (128 x d) * tile^T into the next free accumulator.
__device__ void qm_mma(const QmParams& p, const QmSmem& sm, const QmBars& br, uint32_t tmem_base) {
  const int S = p.stages, KB = p.KB;
  const uint64_t ad0 = sdesc_k_sw128(smem_u32(sm.q)), bd0 = sdesc_k_sw128(smem_u32(sm.stages));
  int s = 0, a = 0;
  uint32_t ph = 0, aph = 0, quses = 0;
  int prev_set = -1;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) break;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) break;
    for (int k = 0; k < n && ok; ++k) {
      const QmItem e = T->item[k];
      const int ntiles = (e.L + kQmTile - 1) / kQmTile;
      if (ntiles == 0) continue;
      if (e.set != prev_set) {
        if (prev_set >= 0) umma_commit_a(br.qempty);  // the old set is free once its MMAs retire
        if (!mbar_wait_a(br.qfull, quses & 1u, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ++quses;
        prev_set = e.set;
      }
      const int nb = qm_blocks_of_set(p, e.set);
      for (int t = 0; t < ntiles && ok; ++t) {
        for (int kb = 0; kb < KB; ++kb) {  // the tile's KB stages stay resident for every block
          int si = s + kb;
          uint32_t phk = ph;
          if (si >= S) {
            si -= S;
            phk ^= 1u;
          }
          if (!mbar_wait_a(br.full + 8 * si, phk, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < nb; ++j) {
          if (!mbar_wait_a(br.accempty + 8 * a, aph ^ 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * kQmTile);
          for (int kb = 0; kb < KB; ++kb) {
            int si = s + kb;
            if (si >= S) si -= S;
            const uint64_t ad = ad0 + static_cast<uint64_t>(((j * KB + kb) * kQmBlock * 128) >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>((si * kQmStage) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16(d_tmem, ad + 2 * kk, bd + 2 * kk, p.idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_a(br.accfull + 8 * a);
          if (++a == kQmAcc) {
            a = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        for (int kb = 0; kb < KB; ++kb) {  // stages reusable once all blocks' MMAs have read them
          umma_commit_a(br.empty + 8 * s);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (ok) mbar_arrive_a(br.tabempty + 8 * buf);
  }
  umma_commit_a(br.done);  // TMEM is freed only after the last MMA completes
  mbar_wait_drain(sm.bars + qm_bars(p.stages) - 1, 0, p.status);
}

// ------------------------------------------------------------ epilogue warps
// Thread = query row of each block. Per (set, document): running maximum
// (and argmax) per row over the document's tiles, then the set's partial
// score: warp sums, folded in warp order by warp 0 through a 2-slot buffer.
template <bool ARGMAX>
__device__ void qm_epilogue(const QmParams& p, const QmSmem& sm, const QmBars& br, uint32_t tmem_base) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  int a = 0;
  uint32_t aph = 0, u = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) return;
    for (int k = 0; k < n; ++k, ++u) {
      const QmItem e = T->item[k];
      const int q = e.set / p.sets_per_query;
      const int r0 = (e.set % p.sets_per_query) * p.set_blocks * kQmBlock;
      const int nb = qm_blocks_of_set(p, e.set);
      const int ntiles = (e.L + kQmTile - 1) / kQmTile;
      float rm[kQmMaxBlocks];
      int ra[kQmMaxBlocks];
#pragma unroll
      for (int j = 0; j < kQmMaxBlocks; ++j) {
        rm[j] = -INFINITY;
        ra[j] = -1;
      }
      for (int t = 0; t < ntiles; ++t) {
        const int valid = min(kQmTile, e.L - t * kQmTile);
#pragma unroll
        for (int j = 0; j < kQmMaxBlocks; ++j) {
          if (j >= nb) break;
          if (!mbar_wait_a(br.accfull + 8 * a, aph, sm.abort_flag, p.status)) return;
          __syncwarp();  // tcgen05.ld is warp-collective
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kQmTile / 32; ++c) {
            float v[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(a * kQmTile + c * 32), v);
            if (c == kQmTile / 32 - 1) {  // accumulator fully read: hand it back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);
            }
            const int col0 = c * 32;
            if (col0 + 32 > valid) {
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (col0 + x >= valid) v[x] = -INFINITY;
            }
            float m1[11];
#pragma unroll
            for (int x = 0; x < 10; ++x)
              asm("max.f32 %0, %1, %2, %3;" : "=f"(m1[x]) : "f"(v[3 * x]), "f"(v[3 * x + 1]), "f"(v[3 * x + 2]));
            m1[10] = fmaxf(v[30], v[31]);
            float m2[4];
#pragma unroll
            for (int x = 0; x < 3; ++x)
              asm("max.f32 %0, %1, %2, %3;" : "=f"(m2[x]) : "f"(m1[3 * x]), "f"(m1[3 * x + 1]), "f"(m1[3 * x + 2]));
            m2[3] = fmaxf(m1[9], m1[10]);
            float cm;
            asm("max.f32 %0, %1, %2, %3;" : "=f"(cm) : "f"(m2[0]), "f"(m2[1]), "f"(m2[2]));
            cm = fmaxf(cm, m2[3]);
            if (cm > rm[j]) {  // columns ascend: strict > keeps the lowest index on ties
              rm[j] = cm;
              if (ARGMAX) {
                int idx = 31;
#pragma unroll
                for (int x = 31; x >= 0; --x)
                  if (v[x] == cm) idx = x;
                ra[j] = t * kQmTile + col0 + idx;
              }
            }
          }
          if (++a == kQmAcc) {
            a = 0;
            aph ^= 1u;
          }
        }
      }
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < kQmMaxBlocks; ++j) {
        if (j >= nb) break;
        const int row = r0 + j * kQmBlock + tid;
        if (row < p.nq) {
          if (e.L > 0) part += rm[j];
          if (ARGMAX) p.argmax[(static_cast<int64_t>(q) * p.B + e.b) * p.nq + row] = e.L > 0 ? ra[j] : -1;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const int slot = u & 1;
      const uint32_t rph = (u >> 1) & 1u;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait_a(br.redempty + 8 * slot, rph ^ 1u, sm.abort_flag, p.status);
        if (ok) {
          sm.red[slot * 4 + warp] = part;
          mbar_arrive_a(br.redfull + 8 * slot);
          if (warp == 0) {
            ok = mbar_wait_a(br.redfull + 8 * slot, rph, sm.abort_flag, p.status);
            if (ok) {
              const float* r = sm.red + slot * 4;
              atomicAdd(p.out + static_cast<int64_t>(q) * p.B + e.b, (r[0] + r[1]) + (r[2] + r[3]));
              mbar_arrive_a(br.redempty + 8 * slot);
            }
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kQmThreads, 1)
    fwd_qm_kernel(const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_q, const QmParams p) {
  extern __shared__ __align__(16) uint8_t qm_raw[];
  const QmSmem sm = qm_carve(qm_raw, p);
  const QmBars br(sm, p.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(sm.bars + s, 1);
      mbar_init(sm.bars + p.stages + s, 1);
    }
    uint64_t* r = sm.bars + 2 * p.stages;
    mbar_init(r + 0, 1);                                               // qfull
    mbar_init(r + 1, 1);                                               // qempty
    for (int i = 0; i < kQmAcc; ++i) mbar_init(r + 2 + i, 1);           // accfull
    for (int i = 0; i < kQmAcc; ++i) mbar_init(r + 2 + kQmAcc + i, 4);  // accempty: 4 epilogue warps
    r += 2 + 2 * kQmAcc;
    for (int i = 0; i < 2; ++i) mbar_init(r + i, 1);      // tabfull
    for (int i = 0; i < 2; ++i) mbar_init(r + 2 + i, 5);  // tabempty: MMA + 4 epilogue warps
    for (int i = 0; i < 2; ++i) mbar_init(r + 4 + i, 4);  // redfull: 4 epilogue warps
    for (int i = 0; i < 2; ++i) mbar_init(r + 6 + i, 1);  // redempty: warp 0
    mbar_init(r + 8, 1);                                  // done
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_d);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 5) {
    tmem_alloc(sm.tmem_slot, kQmAcc * kQmTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  const int64_t items = static_cast<int64_t>(p.n_queries) * p.sets_per_query * p.B;
  const int64_t i0 = (items * blockIdx.x) / gridDim.x, i1 = (items * (blockIdx.x + 1)) / gridDim.x;
  if (warp == 4) {
    qm_producer(p, sm, br, &tm_d, &tm_q, i0, i1);
  } else if (warp == 5) {
    if (lane == 0) qm_mma(p, sm, br, tmem_base);
  } else {
    qm_epilogue<ARGMAX>(p, sm, br, tmem_base);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kQmAcc * kQmTile);
  }
}

// Query blocks per set for head dimension d (KB boxes of 64), or 0 when not
// even one fits beside a double-buffered tile (2 * KB + 2 stages).
int qm_set_blocks(int KB, size_t budget) {
  for (int blocks = kQmMaxBlocks; blocks >= 1; --blocks)
    if (qm_smem_bytes(KB, blocks, 2 * KB + 2) <= budget) return blocks;
  return 0;
}

}  // namespace

bool fwd_qm_applicable(int nq, int d, int64_t total_rows) {
  const DeviceInfo* dev = device_info();
  if (!dev || nq < MAXSIM_QM_MIN_NQ || d % 64 != 0 || d < 64 || total_rows < 1 ||
      total_rows > (static_cast<int64_t>(1) << 30))
    return false;
  const int blocks = qm_set_blocks(d / 64, static_cast<size_t>(dev->max_smem_optin));
  // at least 2 blocks per set (tile reuse) and at most 2 sets per query
  return blocks >= 2 && nq <= kQmMaxSets * blocks * kQmBlock;
}

maxsim_status launch_fwd_qm(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows, int csr,
                            const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd, int is_bf16,
                            float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (!fwd_qm_applicable(nq, d, total_rows)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;
  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  const int blocks = qm_set_blocks(KB, budget);
  int stages = 16;
  while (stages > 2 * KB + 2 && qm_smem_bytes(KB, blocks, stages) > budget) --stages;
  const size_t smem = qm_smem_bytes(KB, blocks, stages);
  if (smem > budget) return MAXSIM_ERR_UNSUPPORTED;

  QmParams p;
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = n_queries;
  p.nq = nq;
  p.KB = KB;
  p.set_blocks = blocks;
  p.sets_per_query = (nq + blocks * kQmBlock - 1) / (blocks * kQmBlock);
  p.stages = stages;
  p.idesc = idesc_f16(is_bf16, kQmBlock, kQmTile);
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  // documents as a [total_rows, d] matrix in 128-row boxes; queries as
  // [n_queries, nq, d] so rows past nq read as zero
  alignas(64) CUtensorMap tm_d, tm_q;
  const int dt = is_bf16 ? 1 : 0;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_rows)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t dbox[2] = {64, kQmTile};
  const uint64_t qdims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(nq), static_cast<uint64_t>(n_queries)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(nq) * d * 2};
  const uint32_t qbox[3] = {64, kQmBlock, 1};
  if (!encode_tmap(&tm_d, dt, 2, const_cast<void*>(D), ddims, dstrides, dbox, 1) ||
      !encode_tmap(&tm_q, dt, 3, const_cast<void*>(Q), qdims, qstrides, qbox, 1))
    return MAXSIM_ERR_CUDA;
  if (cudaMemsetAsync(out, 0, static_cast<size_t>(n_queries) * B * sizeof(float), stream) != cudaSuccess)
    return MAXSIM_ERR_CUDA;
  const int64_t items = static_cast<int64_t>(n_queries) * p.sets_per_query * B;
  const int grid = static_cast<int>(items < dev->sm_count ? items : dev->sm_count);
  cudaError_t e;
  if (argmax) {
    e = cudaFuncSetAttribute(fwd_qm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_qm_kernel<true><<<grid, kQmThreads, smem, stream>>>(tm_d, tm_q, p);
  } else {
    e = cudaFuncSetAttribute(fwd_qm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_qm_kernel<false><<<grid, kQmThreads, smem, stream>>>(tm_d, tm_q, p);
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

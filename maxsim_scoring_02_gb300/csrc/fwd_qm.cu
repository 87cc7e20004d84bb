// fwd_qm.cu -- MaxSim forward for long queries, query-major on tcgen05.
//
// Same operator and outputs as fwd_tc.cu (TileMaxSim deep reading §1;
// FLASH-MAXSIM Figure 1 / Algorithm 2), for queries of a few hundred to 1024
// tokens (ColPali-style Lq = 1024), where the contraction is tensor-bound:
//  * A = a resident set of up to four 128-row query blocks of one query
//    (M = 128 query tokens per MMA); B = a document tile of N tokens
//    streamed by TMA. Every tile in shared memory is multiplied against all
//    resident query blocks, so one tile fill feeds up to 512 query rows.
//  * N is chosen per document (a multiple of 16, at most 192) so that its
//    tiles cover it evenly. An MMA of N >= 176 carries ~90 cycles or more of
//    tensor work, which hides the issuing thread's turnaround after a
//    barrier wait; narrower MMAs leave the pipe idle part of the time.
//  * Two TMEM accumulators (block j uses accumulator j % 2). TMEM lane =
//    query row, column = document token, so the maximum over the document
//    is thread-local (3-input max tree per 32-column chunk); the argmax is
//    searched only in a chunk that raises the running maximum.
//  * Eight epilogue warps: warps w and w + 4 share TMEM lane quarter w; the
//    first four own the even query blocks, the others the odd ones, so each
//    row's running maximum stays in one thread. setmaxnreg gives them 224
//    registers, enough to hold an accumulator row of 192 columns.
//  * Work items are (query set, document) pairs. CTAs form set lanes x
//    document partitions: the set lanes of a partition stream the same
//    documents at the same time, for different query sets, so most tile
//    fills hit L2. A query has at most two sets, whose partial scores are
//    added to out[q, b] (zeroed first); a + b equals b + a in floating point,
//    so the result does not depend on which set lands first.
//  * Warps: 0-7 epilogue, 8 producer (item tables, TMA), 9 MMA issuer,
//    10-11 idle (they complete the control warpgroup for setmaxnreg).
//    Every wait is a bounded mbarrier wait (ptx.cuh); there is no named
//    barrier, so an abort cannot strand a warp.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

#ifndef QM_SEARCH_FMA
#define QM_SEARCH_FMA 0
#endif
#ifndef MAXSIM_QM_MIN_NQ
#define MAXSIM_QM_MIN_NQ 256
#endif

namespace msim {
namespace {

constexpr int kQmEpiWarps = 8;
constexpr int kQmProducerWarp = 8;
constexpr int kQmMmaWarp = 9;
constexpr int kQmThreads = 384;    // 3 warpgroups: epilogue halves 0 and 1, control
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 fits the
// 64K file); the control warpgroup drops to 56 and the epilogue warpgroups
// rise to 224, which uses exactly the launch total (per SM sub-partition as
// well: one warp of each warpgroup sits on each).
constexpr int kQmRegsLaunch = 168, kQmRegsCtl = 56, kQmRegsEpi = 224;
static_assert(2 * 128 * kQmRegsEpi + 128 * kQmRegsCtl <= kQmThreads * kQmRegsLaunch, "register split");
constexpr int kQmBlock = 128;      // query rows per block (MMA M)
constexpr int kQmMaxBlocks = 4;    // query blocks per resident set
constexpr int kQmMaxSets = 2;      // sets per query (keeps the sum order-free)
constexpr int kQmAcc = 2;          // TMEM accumulators of nmax columns
constexpr int kQmItems = 32;       // items per table
constexpr int kQmMaxN = 192;       // widest tile: a whole accumulator row fits in registers
constexpr int kQmMaxChunks = kQmMaxN / 32;
constexpr int kQmMaxSetLanes = 16;

struct QmParams {
  const int32_t* doc_len;
  const int64_t* offsets;
  int64_t B, total_rows;
  int nd, csr;
  int n_queries, nq, KB;
  int set_blocks;      // query blocks per set (<= 4)
  int sets_per_query;
  int stages;
  int nmax;            // tile rows fetched per stage = widest MMA N
  int is_bf16;
  int set_lanes;       // CTAs that share one document partition
  int doc_parts;       // document partitions
  float* out;
  int32_t* argmax;
  unsigned* status;
};

struct QmItem {
  int64_t b;
  int32_t start;  // first row of the document in D
  int32_t L;      // tokens (0: empty or rejected)
  int32_t set;
  int32_t N;      // MMA N (tile width) for this document
};
struct ItemTab {
  int32_t n;  // items in the table; -1 = end of work
  int32_t pad;
  QmItem item[kQmItems];
};

// Barrier block: full[S] empty[S] qfull qempty accfull[2] accempty[2]
// tabfull[2] tabempty[2] redfull[2] redempty[2] done.
__host__ __device__ constexpr int qm_bars(int S) { return 2 * S + 2 + 2 * kQmAcc + 8 + 1; }
// Small structures first, then the 1024-byte aligned operand region (worst
// case padding counted).
__host__ __device__ constexpr size_t qm_small_bytes(int S) {
  return 2 * sizeof(ItemTab) + static_cast<size_t>(qm_bars(S)) * 8 + 16 + 2 * kQmEpiWarps * 4;
}
__host__ __device__ constexpr size_t qm_smem_bytes(int KB, int set_blocks, int S, int nmax) {
  return qm_small_bytes(S) + 1023 + static_cast<size_t>(set_blocks) * KB * kQmBlock * 128 +
         static_cast<size_t>(S) * nmax * 128;
}

struct QmSmem {
  ItemTab* tab;     // [2]
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* red;       // [2 slots][8 warps]
  uint8_t* q;       // [set_blocks][KB][128 rows][128 B], SW128
  uint8_t* stages;  // [S][nmax rows][128 B], SW128
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

// Tile width for a document of L tokens: its ceil(L / nmax) tiles as even as
// the 16-column MMA granularity allows (nmax is a multiple of 16).
__device__ __forceinline__ int qm_tile_n(int64_t L, int nmax) {
  if (L <= 0) return 16;
  const int64_t nt = (L + nmax - 1) / nmax;
  const int64_t n = (((L + nt - 1) / nt) + 15) & ~static_cast<int64_t>(15);
  return static_cast<int>(n);
}

// This CTA's item range: set lane ps handles sets ps, ps + set_lanes, ...
// over documents [b0, b0 + ndocs) of its partition; item k = (k / ndocs)-th
// of those sets, document b0 + k % ndocs.
struct QmRange {
  int ps;
  int64_t b0, ndocs, n;
};
__device__ __forceinline__ QmRange qm_range(const QmParams& p) {
  QmRange r;
  r.ps = static_cast<int>(blockIdx.x % p.set_lanes);
  const int64_t pd = blockIdx.x / p.set_lanes;
  r.b0 = (p.B * pd) / p.doc_parts;
  r.ndocs = (p.B * (pd + 1)) / p.doc_parts - r.b0;
  const int s_total = p.n_queries * p.sets_per_query;
  const int my_sets = r.ps < s_total ? (s_total - r.ps + p.set_lanes - 1) / p.set_lanes : 0;
  r.n = static_cast<int64_t>(my_sets) * r.ndocs;
  return r;
}

// ------------------------------------------------------------ producer warp
// All lanes build item tables; lane 0 issues the query-set and tile loads.
__device__ void qm_producer(const QmParams& p, const QmSmem& sm, const QmBars& br, const CUtensorMap* tm_d,
                            const CUtensorMap* tm_q) {
  const int lane = threadIdx.x & 31;
  const int S = p.stages, KB = p.KB;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.nmax) * 128;
  const QmRange rg = qm_range(p);
  const uint32_t stage0 = smem_u32(sm.stages), q0 = smem_u32(sm.q);
  int s = 0;
  uint32_t ph = 0, fills = 0, qloads = 0;
  int prev_set = -1;
  bool ok = true;
  int64_t it = 0;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    ItemTab* T = sm.tab + buf;
    if (gi >= 2) {
      bool w = true;
      if (lane == 0) w = mbar_wait_inl_a(br.tabempty + 8 * buf, ((gi >> 1) - 1) & 1u, sm.abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
    }
    int n = 0;
    while (n < kQmItems && it + n < rg.n) {
      const int64_t k = it + n + lane;
      if (n + lane < kQmItems && k < rg.n) {
        const int set = rg.ps + static_cast<int>(k / rg.ndocs) * p.set_lanes;
        const int64_t b = rg.b0 + k % rg.ndocs;
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
        e.N = qm_tile_n(L, p.nmax);
      }
      const int64_t left = rg.n - (it + n);
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
        if (e.L == 0) continue;
        const int ntiles = (e.L + e.N - 1) / e.N;
        if (e.set != prev_set) {  // load the next query set once the last one's MMAs retired
          if (qloads > 0 && !mbar_wait_inl_a(br.qempty, (qloads - 1) & 1u, sm.abort_flag, p.status)) {
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
            if (!mbar_wait_inl_a(br.empty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx_a(br.full + 8 * s, stage_bytes);
            // default L2 policy: the other set lanes of this partition read
            // the same tile shortly after
            tma_load_2d_nohint_a(stage0 + static_cast<uint32_t>(s) * stage_bytes, tm_d, br.full + 8 * s, kb * 64,
                                 e.start + t * e.N);
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
// accumulate Q_j (128 x d) * tile^T into the next free accumulator. Waits use
// the non-suspending poll so the next MMA issues as soon as it may.
__device__ void qm_mma(const QmParams& p, const QmSmem& sm, const QmBars& br, uint32_t tmem_base) {
  const int S = p.stages, KB = p.KB;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.nmax) * 128;
  const uint64_t ad0 = sdesc_k_sw128(smem_u32(sm.q)), bd0 = sdesc_k_sw128(smem_u32(sm.stages));
  int s = 0;
  uint32_t ph = 0, aphs = 0, quses = 0;  // aphs bit a: phase parity of accumulator a
  int prev_set = -1;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_inl_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) break;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) break;
    for (int k = 0; k < n && ok; ++k) {
      const QmItem e = T->item[k];
      if (e.L == 0) continue;
      const int ntiles = (e.L + e.N - 1) / e.N;
      if (e.set != prev_set) {
        if (prev_set >= 0) umma_commit_a(br.qempty);  // the old set is free once its MMAs retire
        if (!mbar_poll_inl_a(br.qfull, quses & 1u, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ++quses;
        prev_set = e.set;
      }
      const int nb = qm_blocks_of_set(p, e.set);
      const uint32_t idesc = idesc_f16(p.is_bf16, kQmBlock, e.N);
      for (int t = 0; t < ntiles && ok; ++t) {
        for (int kb = 0; kb < KB; ++kb) {  // the tile's KB stages stay resident for every block
          int si = s + kb;
          uint32_t phk = ph;
          if (si >= S) {
            si -= S;
            phk ^= 1u;
          }
          if (!mbar_poll_inl_a(br.full + 8 * si, phk, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < nb; ++j) {
          const int a = j & 1;  // block j always uses accumulator j % 2 (owned by epilogue half j % 2)
          if (!mbar_poll_inl_a(br.accempty + 8 * a, ((aphs >> a) & 1u) ^ 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * p.nmax);
          for (int kb = 0; kb < KB; ++kb) {
            int si = s + kb;
            if (si >= S) si -= S;
            const uint64_t ad = ad0 + static_cast<uint64_t>(((j * KB + kb) * kQmBlock * 128) >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>((si * stage_bytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_a(br.accfull + 8 * a);
          aphs ^= 1u << a;
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
// Maximum of 32 values held as fp32 bit patterns (3-input max tree).
__device__ __forceinline__ float qm_max32(const uint32_t (&r)[32]) {
  float m1[11];
#pragma unroll
  for (int x = 0; x < 10; ++x)
    asm("max.f32 %0, %1, %2, %3;"
        : "=f"(m1[x])
        : "f"(__uint_as_float(r[3 * x])), "f"(__uint_as_float(r[3 * x + 1])), "f"(__uint_as_float(r[3 * x + 2])));
  m1[10] = fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31]));
  float m2[4];
#pragma unroll
  for (int x = 0; x < 3; ++x)
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m2[x]) : "f"(m1[3 * x]), "f"(m1[3 * x + 1]), "f"(m1[3 * x + 2]));
  m2[3] = fmaxf(m1[9], m1[10]);
  float cm;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(cm) : "f"(m2[0]), "f"(m2[1]), "f"(m2[2]));
  return fmaxf(cm, m2[3]);
}

// Lowest index x with value x equal to m (m is one of the 32 values).
__device__ __forceinline__ int qm_first_eq(const uint32_t (&r)[32], float m) {
#if QM_SEARCH_FMA
  // w[x] = x where value x equals m, else >= 2^11 (or +inf): the difference
  // (m - v) * 2^100 is zero exactly when v == m and at least 2^-49 otherwise,
  // and scaling it by 2^60 before adding x leaves only exact matches below
  // 32. Two FMAs per value on the FMA pipe, a 3-input min tree on the ALU.
  const float s1 = 1.2676506002282294e30f;  // 2^100
  const float s2 = 1.152921504606846976e18f;  // 2^60
  const float ms = m * s1;
  float w[32];
#pragma unroll
  for (int x = 0; x < 32; ++x) w[x] = fmaf(fmaf(-__uint_as_float(r[x]), s1, ms), s2, static_cast<float>(x));
  float m1[11];
#pragma unroll
  for (int x = 0; x < 10; ++x)
    asm("min.f32 %0, %1, %2, %3;" : "=f"(m1[x]) : "f"(w[3 * x]), "f"(w[3 * x + 1]), "f"(w[3 * x + 2]));
  m1[10] = fminf(w[30], w[31]);
  float m2[4];
#pragma unroll
  for (int x = 0; x < 3; ++x)
    asm("min.f32 %0, %1, %2, %3;" : "=f"(m2[x]) : "f"(m1[3 * x]), "f"(m1[3 * x + 1]), "f"(m1[3 * x + 2]));
  m2[3] = fminf(m1[9], m1[10]);
  float mn;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(mn) : "f"(m2[0]), "f"(m2[1]), "f"(m2[2]));
  mn = fminf(mn, m2[3]);
  if (mn <= 31.0f) return static_cast<int>(mn);
  // |m| >= 2^28 overflows the scaled difference: plain search
#endif
  int idx = 31;
#pragma unroll
  for (int x = 31; x >= 0; --x)
    if (__uint_as_float(r[x]) == m) idx = x;
  return idx;
}

// Thread = query row (TMEM lane) of a block; warp half h (0: warps 0-3,
// 1: warps 4-7) owns the query blocks j with j % 2 == h, and block j always
// accumulates into accumulator j % 2, so each accumulator has one consumer
// that meets its phases in order (with alternating owners a consumer running
// ahead could take an older phase of the same parity for its own). Each row's
// running maximum lives in one thread. An accumulator is loaded in one go
// (all of its N columns) before it is handed back, so the MMA into it can
// resume while the maxima are taken. Per (set, document): running
// maximum (and argmax) per row over the document's tiles, then the argmax
// rows and the set's partial score (warp sums, added in warp order by
// warp 0 through a 2-slot buffer).
template <bool ARGMAX>
__device__ void qm_epilogue(const QmParams& p, const QmSmem& sm, const QmBars& br, uint32_t tmem_base) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row_in_block = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const int a = half;  // this half's accumulator (blocks j with j % 2 == half)
  uint32_t aph = 0, u = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_inl_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) return;
    for (int k = 0; k < n; ++k, ++u) {
      const QmItem e = T->item[k];
      const int q = e.set / p.sets_per_query;
      const int r0 = (e.set % p.sets_per_query) * p.set_blocks * kQmBlock;
      const int nb = qm_blocks_of_set(p, e.set);
      const int ntiles = e.L > 0 ? (e.L + e.N - 1) / e.N : 0;
      const int nch = (e.N + 31) / 32;
      // running maxima of this half's blocks (half, half + 2), kept in
      // scalars so the block loop need not be unrolled
      float rm0 = -INFINITY, rm1 = -INFINITY;
      int ra0 = -1, ra1 = -1;
      for (int t = 0; t < ntiles; ++t) {
        const int valid = min(e.N, e.L - t * e.N);
#pragma unroll 1
        for (int jj = 0; jj < kQmMaxBlocks / 2; ++jj) {
          if (2 * jj + half >= nb) break;
          if (!mbar_wait_inl_a(br.accfull + 8 * a, aph, sm.abort_flag, p.status)) return;
          aph ^= 1u;
          __syncwarp();  // tcgen05.ld is warp-collective
          tc_fence_after();
          uint32_t r[kQmMaxChunks][32];
          const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(a * p.nmax);
#pragma unroll
          for (int c = 0; c < kQmMaxChunks; ++c)
            if (c < nch) tmem_ld_32x32b_x32_issue(taddr + static_cast<uint32_t>(c * 32), r[c]);
          tmem_wait_ld_regs(r[0]);
#pragma unroll
          for (int c = 1; c < kQmMaxChunks; ++c) reg_order(r[c]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_a(br.accempty + 8 * a);  // accumulator read: hand it back
          float rmj = jj ? rm1 : rm0;
          int raj = jj ? ra1 : ra0;
#pragma unroll
          for (int c = 0; c < kQmMaxChunks; ++c) {
            if (c >= nch) break;
            const int col0 = c * 32;
            if (col0 + 32 > valid) {
              const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (col0 + x >= valid) r[c][x] = ninf;
            }
            const float cm = qm_max32(r[c]);
            if (cm > rmj) {  // columns ascend: strict > keeps the lowest index on ties
              rmj = cm;
              if (ARGMAX) raj = t * e.N + col0 + qm_first_eq(r[c], cm);
            }
          }
          if (jj) {
            rm1 = rmj;
            ra1 = raj;
          } else {
            rm0 = rmj;
            ra0 = raj;
          }
        }
      }
      float part = 0.f;
#pragma unroll
      for (int jj = 0; jj < kQmMaxBlocks / 2; ++jj) {
        const int j = 2 * jj + half;
        if (j >= nb) break;
        const int row = r0 + j * kQmBlock + row_in_block;
        if (row < p.nq) {
          if (e.L > 0) part += jj ? rm1 : rm0;
          if (ARGMAX)
            p.argmax[(static_cast<int64_t>(q) * p.B + e.b) * p.nq + row] = e.L > 0 ? (jj ? ra1 : ra0) : -1;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const int slot = u & 1;
      const uint32_t rph = (u >> 1) & 1u;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait_inl_a(br.redempty + 8 * slot, rph ^ 1u, sm.abort_flag, p.status);
        if (ok) {
          sm.red[slot * kQmEpiWarps + warp] = part;
          mbar_arrive_a(br.redfull + 8 * slot);
          if (warp == 0) {
            ok = mbar_wait_inl_a(br.redfull + 8 * slot, rph, sm.abort_flag, p.status);
            if (ok) {
              const float* r = sm.red + slot * kQmEpiWarps;
              const float sum = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
              atomicAdd(p.out + static_cast<int64_t>(q) * p.B + e.b, sum);
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
    mbar_init(r + 0, 1);                                                        // qfull
    mbar_init(r + 1, 1);                                                        // qempty
    for (int i = 0; i < kQmAcc; ++i) mbar_init(r + 2 + i, 1);                    // accfull
    for (int i = 0; i < kQmAcc; ++i) mbar_init(r + 2 + kQmAcc + i, 4);  // accempty: owning half
    r += 2 + 2 * kQmAcc;
    for (int i = 0; i < 2; ++i) mbar_init(r + i, 1);                    // tabfull
    for (int i = 0; i < 2; ++i) mbar_init(r + 2 + i, kQmEpiWarps + 1);  // tabempty: epilogue + MMA
    for (int i = 0; i < 2; ++i) mbar_init(r + 4 + i, kQmEpiWarps);      // redfull
    for (int i = 0; i < 2; ++i) mbar_init(r + 6 + i, 1);                // redempty: warp 0
    mbar_init(r + 8, 1);                                                // done
    *sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kQmProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_d);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kQmMmaWarp) {
    tmem_alloc(sm.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  if (warp >= kQmEpiWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kQmRegsCtl));
    if (warp == kQmProducerWarp) {
      qm_producer(p, sm, br, &tm_d, &tm_q);
    } else if (warp == kQmMmaWarp) {
      if (lane == 0) qm_mma(p, sm, br, tmem_base);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kQmRegsEpi));
    qm_epilogue<ARGMAX>(p, sm, br, tmem_base);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kQmMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Tile rows (widest MMA N) and stages for head dimension d = 64 * KB, or
// false when four query blocks and two tiles do not fit.
bool qm_shape(int KB, size_t budget, int* nmax, int* stages) {
  if (KB < 1 || KB > 2) return false;
  for (int n = kQmMaxN; n >= 128; n -= 16) {
    int S = 8;
    while (S > 2 * KB && qm_smem_bytes(KB, kQmMaxBlocks, S, n) > budget) --S;
    if (S >= 2 * KB && qm_smem_bytes(KB, kQmMaxBlocks, S, n) <= budget && kQmAcc * n <= 512) {
      *nmax = n;
      *stages = S;
      return true;
    }
  }
  return false;
}

// Set lanes x document partitions: the most balanced split of
// s_total sets x B documents over at most sm CTAs, preferring more set lanes
// (more CTAs reading the same documents at once) among near-equal splits.
void qm_grid(int s_total, int64_t B, int sm, int* set_lanes, int* doc_parts) {
  double best = 0.0;
  double eff[kQmMaxSetLanes + 1] = {0};
  const int hi = s_total < kQmMaxSetLanes ? s_total : kQmMaxSetLanes;
  for (int ps = 1; ps <= hi && ps <= sm; ++ps) {
    const int64_t pd = (sm / ps) < B ? (sm / ps) : B;
    const double per_cta = static_cast<double>((s_total + ps - 1) / ps) * static_cast<double>((B + pd - 1) / pd);
    eff[ps] = static_cast<double>(s_total) * static_cast<double>(B) / (static_cast<double>(sm) * per_cta);
    if (eff[ps] > best) best = eff[ps];
  }
  *set_lanes = 1;
  for (int ps = hi; ps >= 1; --ps)
    if (ps <= sm && eff[ps] >= 0.98 * best) {
      *set_lanes = ps;
      break;
    }
  const int64_t pd = (sm / *set_lanes) < B ? (sm / *set_lanes) : B;
  *doc_parts = static_cast<int>(pd);
}

}  // namespace

bool fwd_qm_applicable(int nq, int d, int64_t total_rows) {
  const DeviceInfo* dev = device_info();
  if (!dev || nq < MAXSIM_QM_MIN_NQ || nq > kQmMaxSets * kQmMaxBlocks * kQmBlock || d % 64 != 0 || total_rows < 1 ||
      total_rows > (static_cast<int64_t>(1) << 30))
    return false;
  int nmax = 0, stages = 0;
  return qm_shape(d / 64, static_cast<size_t>(dev->max_smem_optin), &nmax, &stages);
}

maxsim_status launch_fwd_qm(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows, int csr,
                            const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd, int is_bf16,
                            float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (!fwd_qm_applicable(nq, d, total_rows)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;
  int nmax = 0, stages = 0;
  if (!qm_shape(KB, static_cast<size_t>(dev->max_smem_optin), &nmax, &stages)) return MAXSIM_ERR_UNSUPPORTED;
  const size_t smem = qm_smem_bytes(KB, kQmMaxBlocks, stages, nmax);

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
  p.set_blocks = kQmMaxBlocks;
  p.sets_per_query = (nq + kQmMaxBlocks * kQmBlock - 1) / (kQmMaxBlocks * kQmBlock);
  p.stages = stages;
  p.nmax = nmax;
  p.is_bf16 = is_bf16;
  qm_grid(n_queries * p.sets_per_query, B, dev->sm_count, &p.set_lanes, &p.doc_parts);
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  // documents as a [total_rows, d] matrix in nmax-row boxes; queries as
  // [n_queries, nq, d] so rows past nq read as zero
  alignas(64) CUtensorMap tm_d, tm_q;
  const int dt = is_bf16 ? 1 : 0;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_rows)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t dbox[2] = {64, static_cast<uint32_t>(nmax)};
  const uint64_t qdims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(nq), static_cast<uint64_t>(n_queries)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(nq) * d * 2};
  const uint32_t qbox[3] = {64, kQmBlock, 1};
  if (!encode_tmap(&tm_d, dt, 2, const_cast<void*>(D), ddims, dstrides, dbox, 1) ||
      !encode_tmap(&tm_q, dt, 3, const_cast<void*>(Q), qdims, qstrides, qbox, 1))
    return MAXSIM_ERR_CUDA;
  if (cudaMemsetAsync(out, 0, static_cast<size_t>(n_queries) * B * sizeof(float), stream) != cudaSuccess)
    return MAXSIM_ERR_CUDA;
  const int grid = p.set_lanes * p.doc_parts;
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

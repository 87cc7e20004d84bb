// fwd_qm.cu -- MaxSim forward for long queries, query-major, on CTA pairs.
//
// Same operator and outputs as fwd_tc.cu (TileMaxSim deep reading §1;
// FLASH-MAXSIM Figure 1 / Algorithm 2), for queries of 256 to 1024 tokens
// (ColPali-style Lq = 1024), where the contraction is tensor-bound:
//  * Two CTAs on two SMs form a cluster and issue pair MMAs (tcgen05
//    cta_group::2, M = 256): each CTA holds up to four 128-row blocks of the
//    query (the pair covers up to 1024 query rows, so one pass per query),
//    and half of each document tile (N / 2 rows of N <= 256). Each SM thus
//    fetches half a tile per pass, and one MMA instruction carries 128 cycles
//    of work at N = 256, long enough to hide the issuing thread's turnaround
//    after a barrier wait.
//  * N is chosen per document (a multiple of 32, at most 256) so that its
//    tiles cover it evenly; 1024-token documents take four tiles of 256.
//  * Two TMEM accumulators (block pair j uses accumulator j % 2; a single
//    block pair alternates between them), each 256 columns in both CTAs. TMEM lane = query row, column = document token, so
//    the maximum over the document is thread-local (3-input max tree per
//    32-column chunk); the argmax is searched once per round of four chunks,
//    in the first chunk holding the round's maximum, when that maximum
//    raises the running one. No similarity value leaves the SM.
//  * Eight epilogue warps per CTA: warps w and w + 4 share TMEM lane quarter
//    w; the first four own the even block pairs (accumulator 0), the others
//    the odd ones, so each accumulator has one in-order consumer per CTA and
//    each row's running maximum stays in one thread. setmaxnreg gives them
//    224 registers; an accumulator row is read in two rounds of 128 columns.
//  * Work items are (query, document) pairs. Pairs form set lanes x document
//    partitions: the set lanes of a partition stream the same documents at
//    the same time for different queries, so tile fills mostly hit L2. Each
//    CTA adds its rows' partial score to out[q, b] (zeroed first); with two
//    addends the result does not depend on which lands first.
//  * Warps: 0-7 epilogue; 8 producer (item tables, TMA of this CTA's
//    operands); 9 in the even CTA issues the MMAs, in the odd CTA relays its
//    operand arrivals to the even CTA; 10-11 idle (they complete the control
//    warpgroup for setmaxnreg). The even CTA's commits arrive on both CTAs'
//    barriers (multicast); the odd CTA's epilogue releases accumulators on
//    the even CTA's barrier. Every wait is a bounded mbarrier wait (ptx.cuh);
//    the cluster barrier at exit keeps each CTA's barriers alive until the
//    other is done with them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

#ifndef MAXSIM_QM_MIN_NQ
#define MAXSIM_QM_MIN_NQ 256
#endif

namespace msim {
namespace {

constexpr int kQpEpiWarps = 8;
constexpr int kQpProducerWarp = 8;
constexpr int kQpMmaWarp = 9;
constexpr int kQpThreads = 384;    // 3 warpgroups: epilogue halves 0 and 1, control
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 fits the
// 64K file); the control warpgroup drops to 56 and the epilogue warpgroups
// rise to 224, which uses exactly the launch total (per SM sub-partition as
// well: one warp of each warpgroup sits on each).
constexpr int kQpRegsLaunch = 168, kQpRegsCtl = 56, kQpRegsEpi = 224;
static_assert(2 * 128 * kQpRegsEpi + 128 * kQpRegsCtl <= kQpThreads * kQpRegsLaunch, "register split");
constexpr int kQpBlock = 128;             // query rows per block (each CTA's half of M = 256)
constexpr int kQpMaxBlocks = 4;           // query blocks per CTA
constexpr int kQpAcc = 2;                 // accumulators of kQpMaxN columns
constexpr int kQpMaxN = 256;              // pair tile width (MMA N)
constexpr int kQpHalf = kQpMaxN / 2;      // tile rows held by each CTA (TMA box rows)
constexpr int kQpStageBytes = kQpHalf * 128;
constexpr int kQpRound = 4;               // 32-column chunks read per round
constexpr int kQpItems = 32;              // items per table
constexpr int kQpMaxSetLanes = 16;

struct QpParams {
  const int32_t* doc_len;
  const int64_t* offsets;
  int64_t B, total_rows;
  int nd, csr;
  int n_queries, nq, KB;
  int P;          // query blocks per CTA; block i of CTA r is query rows (r * P + i) * 128 ...
  int nbp;        // block pairs with real rows (= blocks of the even CTA that hold rows)
  int stages;
  int is_bf16;
  int set_lanes;  // pairs that share one document partition
  int doc_parts;  // document partitions
  float* out;
  int32_t* argmax;
  unsigned* status;
};

struct QpItem {
  int64_t b;
  int32_t start;  // first row of the document in D
  int32_t L;      // tokens (0: empty or rejected)
  int32_t q;      // query
  int32_t N;      // pair MMA N (tile width) for this document
};
struct ItemTab {
  int32_t n;  // items in the table; -1 = end of work
  int32_t pad;
  QpItem item[kQpItems];
};

// Barrier block: full[S] empty[S] full2[S] qfull qfull2 qempty accfull[2]
// accempty[2] tabfull[2] tabempty[2] redfull[2] redempty[2] done. full2,
// qfull2 and accempty are used in the even CTA only.
__host__ __device__ constexpr int qp_bars(int S) { return 3 * S + 3 + 2 * kQpAcc + 8 + 1; }
// Small structures first, then the 1024-byte aligned operand region (worst
// case padding counted). Both CTAs of a pair use the same offsets: the pair
// MMA addresses the odd CTA's operands by the even CTA's descriptors.
__host__ __device__ constexpr size_t qp_small_bytes(int S) {
  return 2 * sizeof(ItemTab) + static_cast<size_t>(qp_bars(S)) * 8 + 16 + 2 * kQpEpiWarps * 4;
}
__host__ __device__ constexpr size_t qp_smem_bytes(int KB, int P, int S) {
  return qp_small_bytes(S) + 1023 + static_cast<size_t>(P) * KB * kQpBlock * 128 +
         static_cast<size_t>(S) * kQpStageBytes;
}

struct QpSmem {
  ItemTab* tab;     // [2]
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* red;       // [2 slots][8 warps]
  uint8_t* q;       // [P][KB][128 rows][128 B], SW128
  uint8_t* stages;  // [S][128 rows][128 B], SW128
};

__device__ __forceinline__ QpSmem qp_carve(uint8_t* raw, const QpParams& p) {
  QpSmem s;
  s.tab = reinterpret_cast<ItemTab*>(raw);
  s.bars = reinterpret_cast<uint64_t*>(s.tab + 2);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + qp_bars(p.stages));
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.red = reinterpret_cast<float*>(s.tmem_slot + 4);
  const uintptr_t end = reinterpret_cast<uintptr_t>(raw) + qp_small_bytes(p.stages);
  s.q = reinterpret_cast<uint8_t*>((end + 1023) & ~uintptr_t(1023));
  s.stages = s.q + static_cast<size_t>(p.P) * p.KB * kQpBlock * 128;
  return s;
}

struct QpBars {
  uint32_t full, empty, full2, qfull, qfull2, qempty, accfull, accempty, tabfull, tabempty, redfull, redempty, done;
  __device__ __forceinline__ QpBars(const QpSmem& sm, int S) {
    full = smem_u32(sm.bars);
    empty = full + 8 * S;
    full2 = empty + 8 * S;
    qfull = full2 + 8 * S;
    qfull2 = qfull + 8;
    qempty = qfull2 + 8;
    accfull = qempty + 8;
    accempty = accfull + 8 * kQpAcc;
    tabfull = accempty + 8 * kQpAcc;
    tabempty = tabfull + 16;
    redfull = tabempty + 16;
    redempty = redfull + 16;
    done = redempty + 16;
  }
};

// Pair tile width for a document of L tokens: its ceil(L / 256) tiles as
// even as the 32-column granularity allows.
__device__ __forceinline__ int qp_tile_n(int64_t L) {
  if (L <= 0) return 32;
  const int64_t nt = (L + kQpMaxN - 1) / kQpMaxN;
  const int64_t n = (((L + nt - 1) / nt) + 31) & ~static_cast<int64_t>(31);
  return static_cast<int>(n);
}

// Accumulator of block pair i at accumulator use number `uses`: i % 2, so
// each accumulator has one consumer half; with a single block pair, uses
// alternate between the two (both consumed, in order, by half 0).
__device__ __forceinline__ int qp_acc_of(int nbp, int i, uint32_t uses) {
  return nbp == 1 ? static_cast<int>(uses & 1u) : (i & 1);
}

// This pair's item range: set lane ps handles queries ps, ps + set_lanes, ...
// over documents [b0, b0 + ndocs) of its partition; item k = (k / ndocs)-th
// of those queries, document b0 + k % ndocs.
struct QpRange {
  int ps;
  int64_t b0, ndocs, n;
};
__device__ __forceinline__ QpRange qp_range(const QpParams& p) {
  QpRange r;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  r.ps = pair % p.set_lanes;
  const int64_t pd = pair / p.set_lanes;
  r.b0 = (p.B * pd) / p.doc_parts;
  r.ndocs = (p.B * (pd + 1)) / p.doc_parts - r.b0;
  const int my_q = r.ps < p.n_queries ? (p.n_queries - r.ps + p.set_lanes - 1) / p.set_lanes : 0;
  r.n = static_cast<int64_t>(my_q) * r.ndocs;
  return r;
}

// ------------------------------------------------------------ producer warp
// All lanes build item tables (the same sequence in both CTAs of the pair);
// lane 0 issues this CTA's query-block and half-tile loads.
__device__ void qp_producer(const QpParams& p, const QpSmem& sm, const QpBars& br, const CUtensorMap* tm_d,
                            const CUtensorMap* tm_q, uint32_t rank) {
  const int lane = threadIdx.x & 31;
  const int S = p.stages, KB = p.KB;
  const QpRange rg = qp_range(p);
  const uint32_t stage0 = smem_u32(sm.stages), q0 = smem_u32(sm.q);
  int s = 0;
  uint32_t ph = 0, fills = 0, qloads = 0;
  int prev_q = -1;
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
    while (n < kQpItems && it + n < rg.n) {
      const int64_t k = it + n + lane;
      if (n + lane < kQpItems && k < rg.n) {
        const int q = rg.ps + static_cast<int>(k / rg.ndocs) * p.set_lanes;
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
        if (bad && rank == 0) atomicOr(p.status, kDevErrBadInput);
        QpItem& e = T->item[n + lane];
        e.b = b;
        e.start = static_cast<int32_t>(start);
        e.L = static_cast<int32_t>(L);
        e.q = q;
        e.N = qp_tile_n(L);
      }
      const int64_t left = rg.n - (it + n);
      n += static_cast<int>(left < 32 ? left : 32);
      if (n > kQpItems) n = kQpItems;
    }
    it += n;
    if (lane == 0) T->n = n > 0 ? n : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabfull + 8 * buf);
    if (n == 0) break;
    if (lane == 0) {
      for (int k = 0; k < n && ok; ++k) {
        const QpItem e = T->item[k];
        if (e.L == 0) continue;
        const int ntiles = (e.L + e.N - 1) / e.N;
        if (e.q != prev_q) {  // this CTA's query blocks, once the last query's MMAs retired
          if (qloads > 0 && !mbar_wait_inl_a(br.qempty, (qloads - 1) & 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          int nload = 0;
          for (int i = 0; i < p.P; ++i)
            if ((static_cast<int>(rank) * p.P + i) * kQpBlock < p.nq) ++nload;
          mbar_arrive_expect_tx_a(br.qfull, static_cast<uint32_t>(nload * KB * kQpBlock * 128));
          for (int i = 0; i < nload; ++i)
            for (int kb = 0; kb < KB; ++kb)
              tma_load_3d_a(q0 + static_cast<uint32_t>((i * KB + kb) * kQpBlock * 128), tm_q, br.qfull, kb * 64,
                            (static_cast<int>(rank) * p.P + i) * kQpBlock, e.q);
          ++qloads;
          prev_q = e.q;
        }
        const int row_off = static_cast<int>(rank) * (e.N / 2);
        for (int t = 0; t < ntiles && ok; ++t) {
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_inl_a(br.empty + 8 * s, ph ^ 1u, sm.abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx_a(br.full + 8 * s, kQpStageBytes);
            // default L2 policy: the other set lanes of this partition read
            // the same rows shortly after
            tma_load_2d_nohint_a(stage0 + static_cast<uint32_t>(s) * kQpStageBytes, tm_d, br.full + 8 * s, kb * 64,
                                 e.start + t * e.N + row_off);
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
    if (qloads > 0) mbar_wait_drain(sm.bars + 3 * S, (qloads - 1) & 1u, p.status);
  }
}

// ------------------------------------------------- MMA issuer (even CTA)
// One thread. Per tile: wait for both CTAs' halves of its KB stages, then for
// each block pair i accumulate Q_i (256 x d, 128 rows per CTA) * tile^T into
// accumulator i % 2 of both CTAs. Waits use the non-suspending poll so the
// next MMA issues as soon as it may.
__device__ void qp_mma(const QpParams& p, const QpSmem& sm, const QpBars& br, uint32_t tmem_base) {
  const int S = p.stages, KB = p.KB;
  const uint64_t ad0 = sdesc_k_sw128(smem_u32(sm.q)), bd0 = sdesc_k_sw128(smem_u32(sm.stages));
  const uint16_t both = 3;
  int s = 0;
  uint32_t ph = 0, aphs = 0, quses = 0, uses = 0;  // aphs bit a: phase parity of accumulator a
  int prev_q = -1;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_inl_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) break;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) break;
    for (int k = 0; k < n && ok; ++k) {
      const QpItem e = T->item[k];
      if (e.L == 0) continue;
      const int ntiles = (e.L + e.N - 1) / e.N;
      if (e.q != prev_q) {
        if (prev_q >= 0) umma_commit_pair(br.qempty, both);  // the old query is free once its MMAs retire
        if (!mbar_poll_inl_a(br.qfull, quses & 1u, sm.abort_flag, p.status) ||
            !mbar_poll_inl_a(br.qfull2, quses & 1u, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ++quses;
        prev_q = e.q;
      }
      const uint32_t idesc = idesc_f16(p.is_bf16, 2 * kQpBlock, e.N);
      for (int t = 0; t < ntiles && ok; ++t) {
        for (int kb = 0; kb < KB && ok; ++kb) {  // the tile's KB stages stay resident for every block pair
          int si = s + kb;
          uint32_t phk = ph;
          if (si >= S) {
            si -= S;
            phk ^= 1u;
          }
          ok = mbar_poll_inl_a(br.full + 8 * si, phk, sm.abort_flag, p.status) &&
               mbar_poll_inl_a(br.full2 + 8 * si, phk, sm.abort_flag, p.status);
        }
        if (!ok) break;
        tc_fence_after();
        for (int i = 0; i < p.nbp; ++i, ++uses) {
          const int a = qp_acc_of(p.nbp, i, uses);
          if (!mbar_poll_inl_a(br.accempty + 8 * a, ((aphs >> a) & 1u) ^ 1u, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * kQpMaxN);
          for (int kb = 0; kb < KB; ++kb) {
            int si = s + kb;
            if (si >= S) si -= S;
            const uint64_t ad = ad0 + static_cast<uint64_t>(((i * KB + kb) * kQpBlock * 128) >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>((si * kQpStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(br.accfull + 8 * a, both);
          aphs ^= 1u << a;
        }
        if (!ok) break;
        for (int kb = 0; kb < KB; ++kb) {  // both CTAs' stages reusable once the MMAs have read them
          umma_commit_pair(br.empty + 8 * s, both);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (ok) mbar_arrive_a(br.tabempty + 8 * buf);
  }
  umma_commit_pair(br.done, 1);  // TMEM is freed only after the last MMA completes
  mbar_wait_drain(sm.bars + qp_bars(p.stages) - 1, 0, p.status);
}

// ---------------------------------------------- operand relay (odd CTA)
// One thread, walking the same items as the issuer: each time this CTA's
// query blocks or half tile land, arrive on the even CTA's qfull2 / full2.
__device__ void qp_relay(const QpParams& p, const QpSmem& sm, const QpBars& br) {
  const int S = p.stages, KB = p.KB;
  const uint32_t full2_r = mapa_shared(br.full2, 0), qfull2_r = mapa_shared(br.qfull2, 0);
  int s = 0;
  uint32_t ph = 0, quses = 0;
  int prev_q = -1;
  bool ok = true;
  for (uint32_t gi = 0; ok; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_inl_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) break;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) break;
    for (int k = 0; k < n && ok; ++k) {
      const QpItem e = T->item[k];
      if (e.L == 0) continue;
      const int ntiles = (e.L + e.N - 1) / e.N;
      if (e.q != prev_q) {
        if (!mbar_wait_inl_a(br.qfull, quses & 1u, sm.abort_flag, p.status)) {
          ok = false;
          break;
        }
        mbar_arrive_cluster(qfull2_r);
        ++quses;
        prev_q = e.q;
      }
      for (int t = 0; t < ntiles && ok; ++t) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_inl_a(br.full + 8 * s, ph, sm.abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(full2_r + 8 * s);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (ok) mbar_arrive_a(br.tabempty + 8 * buf);
  }
}

// ------------------------------------------------------------ epilogue warps
// Maximum of 32 values held as fp32 bit patterns (3-input max tree).
__device__ __forceinline__ float qp_max32(const uint32_t (&r)[32]) {
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

// Running maximum / argmax of one row over chunks [c_base, c_base + nc) of a
// round held in r (columns past `valid` masked first). The argmax is searched
// once per round, and only when the round's maximum beats the running one:
// in the first chunk whose maximum equals the round's (columns ascend, so this
// is the lowest column holding it; ties with the running maximum keep the
// earlier column), its values selected from the round by the chunk index.
template <bool ARGMAX>
__device__ __forceinline__ void qp_scan_round(uint32_t (&r)[kQpRound][32], int c_base, int nc, int valid,
                                              int col_base, float& rm, int& ra) {
  float cm[kQpRound];
#pragma unroll
  for (int c = 0; c < kQpRound; ++c) {
    cm[c] = -INFINITY;
    if (c >= nc) continue;
    const int col0 = (c_base + c) * 32;
    if (col0 + 32 > valid) {
      const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
      for (int x = 0; x < 32; ++x)
        if (col0 + x >= valid) r[c][x] = ninf;
    }
    cm[c] = qp_max32(r[c]);
  }
  static_assert(kQpRound == 4, "round of four chunks");
  float rmax;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(rmax) : "f"(cm[0]), "f"(cm[1]), "f"(cm[2]));
  rmax = fmaxf(rmax, cm[3]);
  const bool better = rmax > rm;
  if (!ARGMAX) {
    if (better) rm = rmax;
    return;
  }
  if (__any_sync(0xffffffffu, better) && better) {
    const bool lo = !(cm[0] == rmax) && (cm[1] == rmax || !(cm[2] == rmax));   // first chunk: 1 or 3
    const bool hi = !(cm[0] == rmax) && !(cm[1] == rmax);                     // first chunk: 2 or 3
    int idx = 31;
#pragma unroll
    for (int x = 31; x >= 0; --x) {
      const uint32_t v = hi ? (lo ? r[3][x] : r[2][x]) : (lo ? r[1][x] : r[0][x]);
      if (__uint_as_float(v) == rmax) idx = x;
    }
    rm = rmax;
    ra = col_base + (c_base + (hi ? 2 : 0) + (lo ? 1 : 0)) * 32 + idx;
  }
}

// Thread = query row (TMEM lane) of this CTA's blocks; warp half h owns the
// block pairs i with i % 2 == h, whose accumulator is h. Per (query,
// document): running maximum (and argmax) per row over the document's tiles,
// then the argmax rows and this CTA's partial score (warp sums, added in warp
// order by warp 0 through a 2-slot buffer).
template <bool ARGMAX>
__device__ void qp_epilogue(const QpParams& p, const QpSmem& sm, const QpBars& br, uint32_t tmem_base,
                            uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row_in_block = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t accempty_r = mapa_shared(br.accempty, 0);  // on the even CTA
  uint32_t aphs = 0, uses = 0, u = 0;  // aphs bit a: phase parity of accumulator a
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_inl_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const ItemTab* T = sm.tab + buf;
    const int n = T->n;
    if (n < 0) return;
    for (int k = 0; k < n; ++k, ++u) {
      const QpItem e = T->item[k];
      const int ntiles = e.L > 0 ? (e.L + e.N - 1) / e.N : 0;
      const int nch = e.N / 32;
      const int nc1 = nch < kQpRound ? nch : kQpRound;
      // running maxima of this half's block pairs (half, half + 2)
      float rm0 = -INFINITY, rm1 = -INFINITY;
      int ra0 = -1, ra1 = -1;
      for (int t = 0; t < ntiles; ++t) {
        const int valid = min(e.N, e.L - t * e.N);
#pragma unroll 1
        for (int jj = 0; jj < kQpMaxBlocks / 2; ++jj) {
          if (2 * jj + half >= p.nbp) break;
          const int a = qp_acc_of(p.nbp, 2 * jj + half, uses++);
          if (!mbar_wait_inl_a(br.accfull + 8 * a, (aphs >> a) & 1u, sm.abort_flag, p.status)) return;
          aphs ^= 1u << a;
          const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(a * kQpMaxN);
          __syncwarp();  // tcgen05.ld is warp-collective
          tc_fence_after();
          float rmj = jj ? rm1 : rm0;
          int raj = jj ? ra1 : ra0;
          uint32_t r[kQpRound][32];
#pragma unroll
          for (int c = 0; c < kQpRound; ++c)
            if (c < nc1) tmem_ld_32x32b_x32_issue(taddr + static_cast<uint32_t>(c * 32), r[c]);
          tmem_wait_ld_regs(r[0]);
#pragma unroll
          for (int c = 1; c < kQpRound; ++c) reg_order(r[c]);
          if (nch > kQpRound) {  // second round of columns: read it before handing the accumulator back
            qp_scan_round<ARGMAX>(r, 0, nc1, valid, t * e.N, rmj, raj);
#pragma unroll
            for (int c = 0; c < kQpRound; ++c)
              if (c < nch - kQpRound)
                tmem_ld_32x32b_x32_issue(taddr + static_cast<uint32_t>((kQpRound + c) * 32), r[c]);
            tmem_wait_ld_regs(r[0]);
#pragma unroll
            for (int c = 1; c < kQpRound; ++c) reg_order(r[c]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {  // accumulator read: hand it back (on the even CTA)
            if (rank == 0)
              mbar_arrive_a(br.accempty + 8 * a);
            else
              mbar_arrive_remote(accempty_r + 8 * a);
          }
          if (nch > kQpRound)
            qp_scan_round<ARGMAX>(r, kQpRound, nch - kQpRound, valid, t * e.N, rmj, raj);
          else
            qp_scan_round<ARGMAX>(r, 0, nc1, valid, t * e.N, rmj, raj);
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
      for (int jj = 0; jj < kQpMaxBlocks / 2; ++jj) {
        const int i = 2 * jj + half;
        if (i >= p.nbp) break;
        const int row = (static_cast<int>(rank) * p.P + i) * kQpBlock + row_in_block;
        if (row < p.nq) {
          if (e.L > 0) part += jj ? rm1 : rm0;
          if (ARGMAX)
            p.argmax[(static_cast<int64_t>(e.q) * p.B + e.b) * p.nq + row] = e.L > 0 ? (jj ? ra1 : ra0) : -1;
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
          sm.red[slot * kQpEpiWarps + warp] = part;
          mbar_arrive_a(br.redfull + 8 * slot);
          if (warp == 0) {
            ok = mbar_wait_inl_a(br.redfull + 8 * slot, rph, sm.abort_flag, p.status);
            if (ok) {
              const float* r = sm.red + slot * kQpEpiWarps;
              const float sum = ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
              atomicAdd(p.out + static_cast<int64_t>(e.q) * p.B + e.b, sum);
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kQpThreads, 1)
    fwd_qm_kernel(const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_q, const QpParams p) {
  extern __shared__ __align__(16) uint8_t qp_raw[];
  const QpSmem sm = qp_carve(qp_raw, p);
  const QpBars br(sm, p.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    const int S = p.stages;
    for (int s = 0; s < S; ++s) {
      mbar_init(sm.bars + s, 1);          // full: this CTA's TMA
      mbar_init(sm.bars + S + s, 1);      // empty: multicast commit
      mbar_init(sm.bars + 2 * S + s, 1);  // full2: the odd CTA's relay
    }
    uint64_t* r = sm.bars + 3 * S;
    mbar_init(r + 0, 1);                                                // qfull
    mbar_init(r + 1, 1);                                                // qfull2
    mbar_init(r + 2, 1);                                                // qempty
    for (int i = 0; i < kQpAcc; ++i) mbar_init(r + 3 + i, 1);            // accfull
    for (int i = 0; i < kQpAcc; ++i) mbar_init(r + 3 + kQpAcc + i, 8);  // accempty: owning half, both CTAs
    r += 3 + 2 * kQpAcc;
    for (int i = 0; i < 2; ++i) mbar_init(r + i, 1);                    // tabfull
    for (int i = 0; i < 2; ++i) mbar_init(r + 2 + i, kQpEpiWarps + 1);  // tabempty: epilogue + issuer / relay
    for (int i = 0; i < 2; ++i) mbar_init(r + 4 + i, kQpEpiWarps);      // redfull
    for (int i = 0; i < 2; ++i) mbar_init(r + 6 + i, 1);                // redempty: warp 0
    mbar_init(r + 8, 1);                                                // done
    *sm.abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == kQpProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_d);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kQpMmaWarp) tmem_alloc_pair(sm.tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  if (warp >= kQpEpiWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kQpRegsCtl));
    if (warp == kQpProducerWarp) {
      qp_producer(p, sm, br, &tm_d, &tm_q, rank);
    } else if (warp == kQpMmaWarp && lane == 0) {
      if (rank == 0)
        qp_mma(p, sm, br, tmem_base);
      else
        qp_relay(p, sm, br);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kQpRegsEpi));
    qp_epilogue<ARGMAX>(p, sm, br, tmem_base, rank);
  }
  tc_fence_before();
  cluster_sync_all();  // neither CTA leaves while the other may still signal it
  if (warp == kQpMmaWarp) {
    __syncwarp();  // the MMA / relay thread rejoins its warp for the dealloc
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// Query blocks per CTA and stages for nq query rows and d = 64 * KB, or false
// when the blocks and two tiles of stages do not fit.
bool qp_shape(int nq, int KB, size_t budget, int* P, int* stages) {
  if (KB < 1 || KB > 2 || nq < 1 || nq > 2 * kQpMaxBlocks * kQpBlock) return false;
  const int nblk = (nq + kQpBlock - 1) / kQpBlock;
  *P = (nblk + 1) / 2;
  int S = 12;
  while (S > 2 * KB && qp_smem_bytes(KB, *P, S) > budget) --S;
  *stages = S;
  return S >= 2 * KB && qp_smem_bytes(KB, *P, S) <= budget;
}

// Set lanes x document partitions over `pairs` pairs: the most balanced
// split of n_queries x B items, preferring more set lanes (more pairs reading
// the same documents at once) among near-equal splits.
void qp_grid(int n_queries, int64_t B, int pairs, int* set_lanes, int* doc_parts) {
  double best = 0.0;
  double eff[kQpMaxSetLanes + 1] = {0};
  const int hi = n_queries < kQpMaxSetLanes ? n_queries : kQpMaxSetLanes;
  for (int ps = 1; ps <= hi && ps <= pairs; ++ps) {
    const int64_t pd = (pairs / ps) < B ? (pairs / ps) : B;
    const double per = static_cast<double>((n_queries + ps - 1) / ps) * static_cast<double>((B + pd - 1) / pd);
    eff[ps] = static_cast<double>(n_queries) * static_cast<double>(B) / (static_cast<double>(pairs) * per);
    if (eff[ps] > best) best = eff[ps];
  }
  *set_lanes = 1;
  for (int ps = hi; ps >= 1; --ps)
    if (ps <= pairs && eff[ps] >= 0.98 * best) {
      *set_lanes = ps;
      break;
    }
  const int64_t pd = (pairs / *set_lanes) < B ? (pairs / *set_lanes) : B;
  *doc_parts = static_cast<int>(pd);
}

}  // namespace

bool fwd_qm_applicable(int nq, int d, int64_t total_rows) {
  const DeviceInfo* dev = device_info();
  if (!dev || dev->sm_count < 2 || nq < MAXSIM_QM_MIN_NQ || d % 64 != 0 || total_rows < 1 ||
      total_rows > (static_cast<int64_t>(1) << 30))
    return false;
  int P = 0, stages = 0;
  return qp_shape(nq, d / 64, static_cast<size_t>(dev->max_smem_optin), &P, &stages);
}

maxsim_status launch_fwd_qm(const void* Q, int n_queries, int nq, int d, const void* D, int64_t total_rows, int csr,
                            const int32_t* doc_len, const int64_t* offsets, int64_t B, int nd, int is_bf16,
                            float* out, int32_t* argmax, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  if (!fwd_qm_applicable(nq, d, total_rows)) return MAXSIM_ERR_UNSUPPORTED;
  const int KB = d / 64;
  QpParams p;
  if (!qp_shape(nq, KB, static_cast<size_t>(dev->max_smem_optin), &p.P, &p.stages)) return MAXSIM_ERR_UNSUPPORTED;
  const size_t smem = qp_smem_bytes(KB, p.P, p.stages);
  p.doc_len = doc_len;
  p.offsets = offsets;
  p.B = B;
  p.total_rows = total_rows;
  p.nd = nd;
  p.csr = csr;
  p.n_queries = n_queries;
  p.nq = nq;
  p.KB = KB;
  const int nblk = (nq + kQpBlock - 1) / kQpBlock;
  p.nbp = nblk < p.P ? nblk : p.P;
  p.is_bf16 = is_bf16;
  qp_grid(n_queries, B, dev->sm_count / 2, &p.set_lanes, &p.doc_parts);
  p.out = out;
  p.argmax = argmax;
  p.status = dev->status;

  // documents as a [total_rows, d] matrix in 128-row boxes (half a pair
  // tile); queries as [n_queries, nq, d] so rows past nq read as zero
  alignas(64) CUtensorMap tm_d, tm_q;
  const int dt = is_bf16 ? 1 : 0;
  const uint64_t ddims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(total_rows)};
  const uint64_t dstrides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t dbox[2] = {64, static_cast<uint32_t>(kQpHalf)};
  const uint64_t qdims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(nq), static_cast<uint64_t>(n_queries)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(nq) * d * 2};
  const uint32_t qbox[3] = {64, kQpBlock, 1};
  if (!encode_tmap(&tm_d, dt, 2, const_cast<void*>(D), ddims, dstrides, dbox, 1) ||
      !encode_tmap(&tm_q, dt, 3, const_cast<void*>(Q), qdims, qstrides, qbox, 1))
    return MAXSIM_ERR_CUDA;
  if (cudaMemsetAsync(out, 0, static_cast<size_t>(n_queries) * B * sizeof(float), stream) != cudaSuccess)
    return MAXSIM_ERR_CUDA;
  const int grid = 2 * p.set_lanes * p.doc_parts;
  cudaError_t e;
  if (argmax) {
    e = cudaFuncSetAttribute(fwd_qm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_qm_kernel<true><<<grid, kQpThreads, smem, stream>>>(tm_d, tm_q, p);
  } else {
    e = cudaFuncSetAttribute(fwd_qm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) fwd_qm_kernel<false><<<grid, kQpThreads, smem, stream>>>(tm_d, tm_q, p);
  }
  if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

}  // namespace msim

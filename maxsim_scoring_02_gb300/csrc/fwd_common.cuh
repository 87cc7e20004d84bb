// fwd_common.cuh -- the parts of the tensor-core forward kernels that do not
// depend on how a tile reaches the tensor core: the launch parameters, the
// group tables of 32-row chunk slots built by the loader warp, the column
// maximum of a 32-row slot, and the merge warp that folds slot maxima in
// document order and writes scores and argmax (TileMaxSim deep reading §1,
// §2(1); FLASH-MAXSIM Figure 1 / Algorithm 2). Included by fwd_tc.cu (bf16 /
// fp16 tiles loaded straight into the MMA operand layout) and fwd_x3.cu
// (fp32 tiles split on chip into three bf16 parts).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {


// Two groups of four slot-partial warps take tiles round-robin (warp w reads
// TMEM lane quarter w % 4); then the producer, MMA and merge warps.
constexpr int kGroups = 2;
constexpr int kProducerWarp = 4 * kGroups, kMmaWarp = 4 * kGroups + 1, kMergeWarp = 4 * kGroups + 2;
constexpr int kThreads = 32 * (4 * kGroups + 3);
constexpr int kStageBytes = 16384;   // 128 rows x 64 elements x 2 bytes
constexpr int kSlotRows = 32;
constexpr int kCapSlots = 256;       // chunk slots per group table
constexpr int kCapDocs = 256;        // documents per group table
constexpr int kMaxAcc = 4;
constexpr int kMaxFin = 5;           // documents finished per tile (4 slots + pass end)
// slot_doc entries: bits 0-15 the local document index; bit 16 set when all
// the document's slots lie in this slot's tile (it starts and ends there), in
// which case bits 17-19 hold its slot count and the partial warps finish it.
constexpr int kSlotLocal = 1 << 16;
constexpr int kSlotDocMask = 0xffff;

struct FwdTcParams {
  const int32_t* order;     // walk position -> document index, or null (identity)
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
  int multipass;   // n_queries * n_chunks > 1
  int stages;
  int n_acc;
  int n_qslots;
  int n_part;      // slot-partial buffers between the partial warps and the merge warp
  int local_finish;  // single pass: the partial warps finish documents whose slots lie in one tile
  const float* col_scale;  // single pass, or null: the score sums col_scale[i] * m_i instead of m_i
  const float* row_scale;  // per document row, or null: similarities are dot * row_scale[row]
  uint32_t idesc;
  uint32_t tmem_cols;
  float* out;
  int32_t* argmax;
  unsigned* status;
};

// One group of documents, written by the producer warp, read by all roles.
struct GroupTab {
  int32_t n_docs;          // documents in the group (incl. empty ones); -1 = end of work
  int32_t n_slots;         // chunk slots used
  int64_t first_doc;       // global index of local document 0
  int32_t slot_row[kCapSlots];   // first row of the chunk in D
  int32_t slot_info[kCapSlots];  // (chunk index in doc << 6) | valid rows (1..32)
  int32_t slot_doc[kCapSlots];   // local document index and flags (kSlotLocal)
  int32_t doc_len[kCapDocs];     // 0 for empty (or rejected) documents
};

// Document scored at walk position `pos`: the identity, or order[pos] when a
// document order is given (-1 if that entry is outside [0, B)).
__device__ __forceinline__ int64_t doc_at(const FwdTcParams& p, int64_t pos) {
  if (!p.order) return pos;
  const int64_t b = __ldg(p.order + pos);
  return (b < 0 || b >= p.B) ? -1 : b;
}

// Rows of the document at walk position `pos` (start row and length);
// out-of-range descriptions are reported as bad and scored as empty documents.
__device__ __forceinline__ int64_t doc_rows(const FwdTcParams& p, int64_t pos, int64_t& start, bool& bad) {
  bad = false;
  const int64_t b = doc_at(p, pos);
  if (b < 0) {
    bad = true;
    start = 0;
    return 0;
  }
  if (p.csr) {
    const int64_t s = __ldg(p.offsets + b), e = __ldg(p.offsets + b + 1);
    if (s < 0 || e < s || e > p.total_rows) {
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

// ------------------------------------------------------------ producer warp
// Builds the slot table of the next group (all 32 lanes). `nb` / `carry` is
// the walk position: next document and, in single-pass mode, the number of
// its chunks already placed in earlier groups (a long document may be split
// across groups there; in multi-pass mode a group always holds whole
// documents).
__device__ void build_group(const FwdTcParams& p, GroupTab* T, int64_t& nb, int64_t b1, int64_t& carry) {
  const int lane = threadIdx.x & 31;
  int nslots = 0, ndocs = 0;
  if (lane == 0) T->first_doc = nb;
  const int64_t carry0 = carry;
  // Round `it` of the loop below looks at documents nb0 + 32 * it + lane
  // (every earlier round accepted 32); their descriptions are fetched up
  // front, so the rounds wait for one global-load latency, not one each.
  constexpr int kRounds = kCapDocs / 32;
  const int64_t nb0 = nb;
  int64_t pre_start[kRounds], pre_len[kRounds];
  bool pre_bad[kRounds];
#pragma unroll
  for (int it = 0; it < kRounds; ++it) {
    const int64_t b = nb0 + 32 * it + lane;
    pre_start[it] = 0;
    pre_len[it] = 0;
    pre_bad[it] = false;
    if (b < b1) pre_len[it] = doc_rows(p, b, pre_start[it], pre_bad[it]);
  }
#pragma unroll
  for (int it = 0; it < kRounds; ++it) {
    if (!(nb < b1 && ndocs < kCapDocs && nslots < kCapSlots)) break;
    const int64_t b = nb + lane;
    const bool in = b < b1 && ndocs + lane < kCapDocs;
    int64_t start = 0, L = 0;
    bool bad = false;
    if (in) {
      L = pre_len[it];
      start = pre_start[it];
      bad = pre_bad[it];
    }
    if (bad) atomicOr(p.status, kDevErrBadInput);
    const int64_t ck0 = (lane == 0) ? carry : 0;   // chunks of this doc already placed
    int64_t chunks = in ? (L + kSlotRows - 1) / kSlotRows - ck0 : 0;
    if (p.multipass && chunks > kCapSlots) {        // cannot fit a group: reject
      atomicOr(p.status, kDevErrBadInput);
      chunks = 0;
      L = 0;
    }
    // inclusive scan of chunk counts (saturated to the capacity)
    int c32 = static_cast<int>(chunks > kCapSlots ? kCapSlots + 1 : chunks);
    int incl = c32;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl = min(incl + v, 1 << 20);
    }
    const int pre = incl - c32;
    const int room = kCapSlots - nslots;
    // a lane's document is accepted whole if it fits; in single-pass mode the
    // first one that does not fit is placed partially (split)
    const bool whole = in && (pre + c32 <= room);
    const unsigned acc_mask = __ballot_sync(0xffffffffu, whole);
    const int n_whole = __popc(~acc_mask) == 0 ? 32 : __ffs(~acc_mask) - 1;  // accepted lanes form a prefix
    bool split = false;
    int placed = whole ? c32 : 0;
    if (!p.multipass && lane == n_whole && in && pre < room) {
      split = true;
      placed = room - pre;
    }
    const unsigned split_mask = __ballot_sync(0xffffffffu, split);
    if (whole || split) {
      const int dl = ndocs + lane;
      T->doc_len[dl] = static_cast<int32_t>(L);
      const int idx0 = nslots + pre;
      const bool local = p.local_finish && whole && ck0 == 0 && placed > 0 && (idx0 >> 2) == ((idx0 + placed - 1) >> 2);
      const int dflag = dl | (local ? (kSlotLocal | (placed << 17)) : 0);
      for (int k = 0; k < placed; ++k) {
        const int idx = nslots + pre + k;
        const int64_t ck = ck0 + k;
        const int64_t rowk = start + ck * kSlotRows;
        const int64_t left = L - ck * kSlotRows;
        T->slot_row[idx] = static_cast<int32_t>(rowk);
        T->slot_info[idx] = static_cast<int32_t>((ck << 6) | (left >= kSlotRows ? kSlotRows : left));
        T->slot_doc[idx] = dflag;
      }
    }
    // totals (from the last placing lane)
    const int last = split_mask ? (__ffs(split_mask) - 1) : (n_whole - 1);
    int tot = 0;
    if (last >= 0) tot = __shfl_sync(0xffffffffu, pre + placed, last);
    int split_placed = split_mask ? __shfl_sync(0xffffffffu, placed, __ffs(split_mask) - 1) : 0;
    nslots += tot;
    ndocs += n_whole + (split_mask ? 1 : 0);
    if (split_mask) {
      carry = (n_whole == 0 ? carry : 0) + split_placed;
      nb += n_whole;
      break;
    }
    if (n_whole > 0) carry = 0;
    nb += n_whole;
    if (n_whole < 32) break;   // capacity reached (docs or slots)
  }
  (void)carry0;
  if (lane == 0) {
    T->n_docs = ndocs;
    T->n_slots = nslots;
  }
  __syncwarp();
}

// ------------------------------------------------------------ table builder
// A warp of its own builds each group's slot table (all 32 lanes) one group
// ahead of the loader, so the loader never stops issuing copies to build one.
template <class SmemT, class BarsT>
__device__ void run_builder(const FwdTcParams& p, const SmemT& sm, const BarsT& br, int64_t b0, int64_t b1) {
  const int lane = threadIdx.x & 31;
  int64_t nb = b0, carry = 0;
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    GroupTab* T = sm.tab + buf;
    if (gi >= 2) {
      bool w = true;
      if (lane == 0) w = mbar_wait_a(br.tabempty + 8 * buf, ((gi >> 1) - 1) & 1u, sm.abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) return;
    }
    const bool end = nb >= b1;
    if (end) {
      if (lane == 0) T->n_docs = -1;
    } else {
      build_group(p, T, nb, b1, carry);
    }
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabfull + 8 * buf);
    if (end) return;
  }
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

// Appends (doc, sum) to the finished-document list without dynamic indexing.
__device__ __forceinline__ void fin_push(int64_t (&fd)[kMaxFin], float (&fs)[kMaxFin], int& n, int64_t doc,
                                         float sum) {
#pragma unroll
  for (int f = 0; f < kMaxFin; ++f)
    if (f == n) {
      fd[f] = doc;
      fs[f] = sum;
    }
  ++n;
}
// --------------------------------------------------------------- merge warp
// Merges slot partials in document order (lane l owns query columns
// l, l+32, ...), finishes documents (sum over query tokens, argmax), and
// writes empty documents' outputs. SINGLE: the launch is known to run one
// query, one column chunk and one pass, and the other paths are compiled out.
template <int NG, bool ARGMAX, bool SINGLE = false, class SmemT, class BarsT>
__device__ void run_merge(const FwdTcParams& p, const SmemT& sm, const BarsT& br) {
  constexpr int NC = 32 * NG;
  const int n_queries = SINGLE ? 1 : p.n_queries;
  const int n_chunks = SINGLE ? 1 : p.n_chunks;
  const bool multipass = SINGLE ? false : (p.multipass != 0);
  const int lane = threadIdx.x & 31;
  const int PB = p.n_part;
  int pb = 0;
  uint32_t pph = 0;
  int64_t cur = -1;
  float rm[NG], qw[NG];
  int ra[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    rm[g] = -INFINITY;
    ra[g] = INT_MAX;
    // weight of column g * 32 + lane in the score (single pass when scaled)
    qw[g] = (p.col_scale && g * 32 + lane < p.nq) ? __ldg(p.col_scale + g * 32 + lane) : 1.f;
  }
  auto doc_sum = [&](int c, int64_t doc, int q) -> float {
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int qc = c * NC + g * 32 + lane;
      if (qc < p.nq) {
        sum += p.col_scale ? qw[g] * rm[g] : rm[g];
        if (ARGMAX && doc >= 0) p.argmax[(static_cast<int64_t>(q) * p.B + doc) * p.nq + qc] = ra[g];
      }
    }
    return sum;
  };
  for (uint32_t gi = 0;; ++gi) {
    const int buf = gi & 1;
    if (!mbar_wait_a(br.tabfull + 8 * buf, (gi >> 1) & 1u, sm.abort_flag, p.status)) return;
    const GroupTab* T = sm.tab + buf;
    const int n_docs = T->n_docs;
    if (n_docs < 0) break;
    const int n_slots = T->n_slots;
    const int n_tiles = (n_slots + 3) >> 2;
    const int64_t first = T->first_doc;
    for (int q = 0; q < n_queries; ++q) {
      for (int c = 0; c < n_chunks; ++c) {
        const bool last_chunk = c == n_chunks - 1;
        // empty documents of the group: score 0, argmax -1 (no slots, no MMA)
        for (int dl = lane; dl < n_docs; dl += 32) {
          const int64_t b = doc_at(p, first + dl);
          if (T->doc_len[dl] == 0 && b >= 0) {
            if (ARGMAX)
              for (int col = 0; col < NC; ++col) {
                const int qc = c * NC + col;
                if (qc < p.nq) p.argmax[(static_cast<int64_t>(q) * p.B + b) * p.nq + qc] = -1;
              }
            if (last_chunk) p.out[static_cast<int64_t>(q) * p.B + b] = 0.f;
          }
        }
        if (multipass) cur = -1;
        for (int t = 0; t < n_tiles; ++t) {
          if (!mbar_wait_a(br.partfull + 8 * pb, pph, sm.abort_flag, p.status)) return;
          const int i0 = 4 * t;
          const int nslot = min(4, n_slots - i0);
          // one 16-byte read of the tile's four slot entries (i0 is a multiple of 4)
          const int4 sd4 = *reinterpret_cast<const int4*>(T->slot_doc + i0);
          const int sds[4] = {sd4.x, sd4.y, sd4.z, sd4.w};
          bool any = cur >= 0;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (w < nslot && !(sds[w] & kSlotLocal)) any = true;
          int nfin = 0;
          int64_t fin_doc[kMaxFin];
          float fin_sum[kMaxFin];
          const float* pv = sm.part_v + pb * 4 * NC;
          const int32_t* pi = sm.part_i + pb * 4 * NC;
          // a tile in the middle of the open document: fold its four slots
          const bool through = nslot == 4 && sds[0] == sds[1] && sds[1] == sds[2] && sds[2] == sds[3] &&
                               !(sds[0] & kSlotLocal) && first + (sds[0] & kSlotDocMask) == cur;
          if (through) {
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              float v4[4];
              int i4[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                v4[w] = pv[w * NC + g * 32 + lane];
                i4[w] = ARGMAX ? pi[w * NC + g * 32 + lane] : 0;
              }
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                if (ARGMAX) {
                  if (v4[w] > rm[g] || (v4[w] == rm[g] && i4[w] < ra[g])) {
                    rm[g] = v4[w];
                    ra[g] = i4[w];
                  }
                } else {
                  rm[g] = fmaxf(rm[g], v4[w]);
                }
              }
            }
          } else if (any) {
            // up to 64 query columns: all four slots' values first (independent
            // loads), then the walk; wider chunks load in the walk
            constexpr bool kPre = NG <= 2;
            float sv[4][NG];
            int si[4][NG];
            if (kPre) {
#pragma unroll
              for (int w = 0; w < 4; ++w)
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                  sv[w][g] = pv[w * NC + g * 32 + lane];
                  si[w][g] = ARGMAX ? pi[w * NC + g * 32 + lane] : 0;
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              if (w < nslot) {
                // slots of documents finished by the partial warps close the open document
                const bool loc = (sds[w] & kSlotLocal) != 0;
                const int64_t dg = loc ? -1 : first + (sds[w] & kSlotDocMask);
                if (dg != cur) {
                  if (cur >= 0) fin_push(fin_doc, fin_sum, nfin, cur, doc_sum(c, doc_at(p, cur), q));
                  cur = dg;
#pragma unroll
                  for (int g = 0; g < NG; ++g) {
                    rm[g] = -INFINITY;
                    ra[g] = INT_MAX;
                  }
                }
                if (!loc) {
#pragma unroll
                  for (int g = 0; g < NG; ++g) {
                    const float v2 = kPre ? sv[w][g] : pv[w * NC + g * 32 + lane];
                    if (ARGMAX) {
                      const int i2 = kPre ? si[w][g] : pi[w * NC + g * 32 + lane];
                      if (v2 > rm[g] || (v2 == rm[g] && i2 < ra[g])) {
                        rm[g] = v2;
                        ra[g] = i2;
                      }
                    } else {
                      rm[g] = fmaxf(rm[g], v2);
                    }
                  }
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_a(br.partempty + 8 * pb);
          if (++pb == PB) {
            pb = 0;
            pph ^= 1u;
          }
          if (multipass && t == n_tiles - 1 && cur >= 0) {
            fin_push(fin_doc, fin_sum, nfin, cur, doc_sum(c, doc_at(p, cur), q));
            cur = -1;
          }
          auto write_doc = [&](int64_t b, float total) {   // b is a walk position
            const int64_t bd = doc_at(p, b);
            const int64_t o = static_cast<int64_t>(q) * p.B + bd;
            if (n_chunks == 1) {
              if (bd >= 0) p.out[o] = total;
            } else {
              const int dl = static_cast<int>(b - first);
              const float g2 = (c == 0 ? 0.f : sm.gsum[dl]) + total;
              if (!last_chunk) sm.gsum[dl] = g2;
              else if (bd >= 0) p.out[o] = g2;
            }
          };
          if (nfin == 1) {   // the common case: one butterfly, lane 0 writes
            float s = fin_sum[0];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) write_doc(fin_doc[0], s);
          } else if (nfin > 1) {
#pragma unroll
            for (int f = 0; f < kMaxFin; ++f)
              if (f < nfin) {
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) fin_sum[f] += __shfl_xor_sync(0xffffffffu, fin_sum[f], o);
              }
            if (lane < nfin) {
              float total = 0.f;
              int64_t b = 0;
#pragma unroll
              for (int f = 0; f < kMaxFin; ++f)
                if (f == lane) {
                  total = fin_sum[f];
                  b = fin_doc[f];
                }
              write_doc(b, total);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_a(br.tabempty + 8 * buf);
  }
  // end of work: the last document of a single-pass walk is still open
  if (!multipass && cur >= 0) {
    const int64_t bd = doc_at(p, cur);
    float sum = doc_sum(0, bd, 0);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0 && bd >= 0) p.out[bd] = sum;
  }
}

}  // namespace
}  // namespace msim

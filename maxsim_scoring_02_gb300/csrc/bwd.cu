// bwd.cu -- MaxSim backward through the saved forward argmax (FLASH-MAXSIM,
// Abstract: the backward pass reuses the forward argmax, with an inverse-grid
// CSR construction and an atomic-free, destination-owned reduction).
//
// With loss = sum_{q,b} dS[q,b] * score[q,b] and a = argmax[q,b,i]:
//   dD[b,j,:] = sum_{(q,i) : a(q,b,i) = j} dS[q,b] * Q[q,i,:]     (dd_kernel)
//   dQ[q,i,:] = sum_b dS[q,b] * D[b, a(q,b,i), :]                   (dq_kernel)
//
// dd_kernel -- one CTA per document (persistent over documents). The
// document's nQ*nq argmax entries are grouped by token j with a counting
// sort in shared memory: each warp counts its chunk of entries into a
// private histogram (lanes holding the same key are found with one ballot
// per key bit and only their lowest lane updates the warp's counter, so no
// atomics are needed), a scan over (key, warp) gives the inverse CSR row
// pointers, and a second pass scatters the entries stably. Then groups of
// lanes (half-warps for d <= 256, else warps) each walk the sorted list over
// their own contiguous range of rows, balanced by entries + rows, in batches
// of entries that run across row boundaries; a row is written (zeros if
// nothing points at it) once its last entry has been added -- every row of
// dD[b] has exactly one writer and its entries are added in list order.
//
// dq_kernel -- each CTA owns a block of (q, i) destination rows; a thread
// holds 32 dimensions of one row as fp32 accumulators in registers and sweeps
// one contiguous range of documents in ascending order. Per document it
// copies its 64-byte slice of the selected D row into its own shared-memory
// slot with 16-byte cp.async, several documents ahead of the one it
// accumulates, and fetches the argmax entries and dS values further ahead
// into a register ring, so the dependent argmax -> row loads never stall the
// accumulation (no data is shared between threads, so no barrier is needed).
// The CTAs of a range sweep in the same order, so the gathered rows are
// re-served from L2. With several ranges each writes its own partial dQ to
// the workspace and dq_reduce_kernel adds them in range order -- still
// destination-owned, atomic-free and deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace msim {
namespace {


// Two packed 16-bit values (low half first) as floats, exactly.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
}

// (a0, a1) += g * (x0, x1) as one packed fp32x2 FMA: two IEEE round-to-nearest
// FMAs, bit-identical to two fmaf calls, in one issue slot.
__device__ __forceinline__ void fma2(float& a0, float& a1, float g, float2 x) {
  asm("{\n\t.reg .b64 acc, xv, gv;\n\t"
      "mov.b64 acc, {%0, %1};\n\t"
      "mov.b64 xv, {%2, %3};\n\t"
      "mov.b64 gv, {%4, %4};\n\t"
      "fma.rn.f32x2 acc, gv, xv, acc;\n\t"
      "mov.b64 {%0, %1}, acc;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x.x), "f"(x.y), "f"(g));
}

struct BwdParams {
  const void* Q;
  const void* D;
  const int32_t* doc_len;
  const int32_t* argmax;
  const float* dS;
  float* dQ;
  float* dD;
  int64_t B;
  int nQ, nq, d, nd;
  uint32_t nq_inv;   // ceil(2^32 / nq) for nq > 1 (0 for nq = 1): e / nq = umulhi(e, nq_inv) for e < 2^16
  int splits;        // dQ document ranges (partials summed in range order)
  float* partial;    // [splits][nQ][nq][d] workspace (splits > 1)
  unsigned* status;
};

// Query of argmax entry e = q * nq + i (e < 2^16): a multiply-high by the
// rounded-up reciprocal, exact here because with nq_inv * nq = 2^32 + eps
// (0 <= eps < nq) the excess e * eps / 2^32 stays below 1 (e, eps < 2^16).
__device__ __forceinline__ int entry_query(const BwdParams& p, int e) {
  const int q = static_cast<int>(__umulhi(static_cast<uint32_t>(e), p.nq_inv));
  return p.nq_inv ? q : e;   // nq = 1: the entry is the query
}

__device__ __forceinline__ int doc_length(const BwdParams& p, int64_t b) {
  if (!p.doc_len) return p.nd;
  const int L = __ldg(p.doc_len + b);
  return (L < 0 || L > p.nd) ? -1 : L;
}

// ------------------------------------------------------------------- dD
// NW warps per CTA; DPL = d / 32. The row walk takes entries in groups of
// G lanes (16 for d <= 256, else 32); lane l of a group owns the DL =
// 32 DPL / G consecutive dimensions [DL l, DL l + DL) of a row, so a group's
// load of a Q row is d * 2 contiguous bytes (whole 32-byte sectors).

// DPL 16-bit values at `src` (DPL * 2 bytes, aligned to that size up to 16)
// as DPL / 2 packed 32-bit words.
template <int DPL>
__device__ __forceinline__ void load_row_words(const void* src, uint32_t (&w)[DPL / 2]) {
  if constexpr (DPL % 8 == 0) {
#pragma unroll
    for (int c = 0; c < DPL / 8; ++c) {
      const uint4 v = __ldg(static_cast<const uint4*>(src) + c);
      w[4 * c] = v.x;
      w[4 * c + 1] = v.y;
      w[4 * c + 2] = v.z;
      w[4 * c + 3] = v.w;
    }
  } else if constexpr (DPL % 4 == 0) {
#pragma unroll
    for (int c = 0; c < DPL / 4; ++c) {
      const uint2 v = __ldg(static_cast<const uint2*>(src) + c);
      w[2 * c] = v.x;
      w[2 * c + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int c = 0; c < DPL / 2; ++c) w[c] = __ldg(static_cast<const uint32_t*>(src) + c);
  }
}

// Entries gathered per batch of the row walk: enough Q-row loads in flight
// per lane to cover L2 latency, within the register budget of two 16-warp
// CTAs per SM (64 registers a thread). For d <= 256 the batch is per group
// of 16 lanes: U entries of 2 DPL values each.
__host__ __device__ constexpr int dd_batch(int dpl) { return dpl <= 4 ? 8 : dpl <= 8 ? 4 : dpl <= 16 ? 2 : 1; }

// Lanes of the warp whose key equals this lane's key, for keys below
// 2^nbits (nbits warp-uniform): one ballot per key bit, keeping the lanes
// that agree with this lane on that bit.
__device__ __forceinline__ unsigned dd_peers(unsigned key, int nbits) {
  unsigned m = 0xffffffffu;
  for (int i = 0; i < nbits; ++i) {
    const unsigned bit = (key >> i) & 1u;
    const unsigned bal = __ballot_sync(0xffffffffu, bit != 0u);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__host__ __device__ constexpr size_t dd_smem_bytes(int nw, int nd, int nQ, int ne) {
  return (static_cast<size_t>(nd) + 1 + nQ + nw) * 4 + (static_cast<size_t>(nw) * nd + 2 * static_cast<size_t>(ne)) * 2;
}

template <typename T, int DPL, int NW>
__global__ void __launch_bounds__(NW * 32, 2) dd_kernel(const BwdParams p) {
  constexpr int NT = NW * 32;
  constexpr int U = dd_batch(DPL);
  extern __shared__ int32_t bsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nd = p.nd, ne = p.nQ * p.nq;
  // 16-bit storage: tokens < 65535, entries and positions < 65536
  int32_t* rowptr = bsm;                                                   // [nd + 1]
  float* dsv = reinterpret_cast<float*>(rowptr + nd + 1);                  // [nQ]
  int32_t* wsum = reinterpret_cast<int32_t*>(dsv + p.nQ);                  // [NW] scan scratch
  uint16_t* counts = reinterpret_cast<uint16_t*>(wsum + NW);               // [NW][nd] -> offsets
  uint16_t* list = counts + NW * nd;                                       // [ne] sorted entry ids
  uint16_t* keys = list + ne;                                              // [ne] token + 1 (0 = skip)
  const int chunk = (ne + NW - 1) / NW;
  const int e_lo = warp * chunk, e_hi = min(ne, e_lo + chunk);
  const uint32_t qrow_bytes = static_cast<uint32_t>(p.d) * 2;   // e * qrow_bytes < 2^16 * 2^11
  const int nbits = 32 - __clz(nd);                              // keys 0 .. nd

  for (int64_t b = blockIdx.x; b < p.B; b += gridDim.x) {
    int L = doc_length(p, b);
    if (L < 0) {
      if (tid == 0) atomicOr(p.status, kDevErrBadInput);
      L = 0;
    }
    for (int x = tid; x < NW * nd; x += NT) counts[x] = 0;
    for (int q = tid; q < p.nQ; q += NT) dsv[q] = __ldg(p.dS + static_cast<int64_t>(q) * p.B + b);
    // stage the document's argmax entries (coalesced per query row), validated:
    // -1 is only valid for an empty document; anything outside [0, L) is skipped
    bool bad = false;
#pragma unroll 8
    for (int e = tid; e < ne; e += NT) {
      const int q = entry_query(p, e), i = e - q * p.nq;
      int key = __ldg(p.argmax + (static_cast<int64_t>(q) * p.B + b) * p.nq + i);
      if (key < 0 || key >= L) {
        if (!(key == -1 && L == 0)) bad = true;
        key = -1;
      }
      keys[e] = static_cast<uint16_t>(key + 1);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kDevErrBadInput);
    __syncthreads();
    // pass 1: per-warp histograms of the argmax keys (key = token + 1, 0 = skip)
    for (int e0 = e_lo; e0 < e_hi; e0 += 32) {
      const int e = e0 + lane;
      const unsigned key = e < e_hi ? keys[e] : 0u;
      const unsigned grp = dd_peers(key, nbits);
      if (key != 0u && lane == __ffs(grp) - 1)
        counts[warp * nd + key - 1] = static_cast<uint16_t>(counts[warp * nd + key - 1] + __popc(grp));
      __syncwarp();
    }
    __syncthreads();
    // scan over (key, warp): offsets[w][j] = start[j] + sum_{w' < w} counts[w'][j]
    {
      const int per = (nd + NT - 1) / NT;
      const int j0 = tid * per, j1 = min(nd, j0 + per);
      int run = 0;
      for (int j = j0; j < j1; ++j)
        for (int w = 0; w < NW; ++w) run += counts[w * nd + j];
      // block-wide exclusive scan of the per-thread totals
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      int base = 0;
      for (int w = 0; w < warp; ++w) base += wsum[w];
      base += incl - run;
      for (int j = j0; j < j1; ++j) {
        rowptr[j] = base;
        for (int w = 0; w < NW; ++w) {
          const int c = counts[w * nd + j];
          counts[w * nd + j] = static_cast<uint16_t>(base);
          base += c;
        }
      }
      if (j1 == nd && j0 < j1) rowptr[nd] = base;
    }
    __syncthreads();
    // pass 2: stable scatter of entry ids into the inverse CSR list
    for (int e0 = e_lo; e0 < e_hi; e0 += 32) {
      const int e = e0 + lane;
      const unsigned key = e < e_hi ? keys[e] : 0u;
      const unsigned grp = dd_peers(key, nbits);
      int pos = 0;
      if (key != 0u) pos = counts[warp * nd + key - 1] + __popc(grp & ((1u << lane) - 1u));
      __syncwarp();
      if (key != 0u) {
        list[pos] = static_cast<uint16_t>(e);
        if (lane == __ffs(grp) - 1)
          counts[warp * nd + key - 1] = static_cast<uint16_t>(counts[warp * nd + key - 1] + __popc(grp));
      }
      __syncwarp();
    }
    __syncthreads();
    // Destination-owned rows. Entry groups of G lanes (half-warps for
    // d <= 256, else warps), lane l of a group owning the DL dimensions
    // [DL l, DL l + DL); group k walks the inverse CSR list over its own
    // contiguous range of rows [ja, jb), cut so that entries + rows are
    // balanced across groups, in batches of U entries that run across row
    // boundaries. A row is written (zeros if nothing points at it) when its
    // last entry has been added; its entries are added in list order, so the
    // sums are deterministic and each row has exactly one writer.
    {
      constexpr int G = DPL <= 8 ? 16 : 32;
      constexpr int DL = DPL * 32 / G;
      constexpr int NG = NT / G;
      const int grp = tid / G, sub = tid % G;
      const uint8_t* Qs = static_cast<const uint8_t*>(p.Q) + static_cast<size_t>(sub) * DL * 2;
      const int total = rowptr[nd];
      // first row j with rowptr[j] + j >= k (total + nd) / NG (strictly increasing in j)
      auto row_start = [&](int k) -> int {
        if (k <= 0) return 0;
        if (k >= NG) return nd;
        const int64_t target = (static_cast<int64_t>(total + nd) * k) / NG;
        int lo = 0, hi = nd;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (rowptr[mid] + mid >= target) hi = mid;
          else lo = mid + 1;
        }
        return lo;
      };
      const int ja = row_start(grp), jb = row_start(grp + 1);
      if (ja < jb) {
        float acc[DL];
#pragma unroll
        for (int k = 0; k < DL; ++k) acc[k] = 0.f;
        float* dbase = p.dD + b * nd * static_cast<int64_t>(p.d) + sub * DL;
        int j = ja, pos = rowptr[ja], end = rowptr[ja + 1];
        const int stop = rowptr[jb];
        auto write_row = [&]() {   // row j is complete: write it and move to row j + 1
          float* drow = dbase + static_cast<int64_t>(j) * p.d;
          if constexpr (DL % 4 == 0) {
#pragma unroll
            for (int k = 0; k < DL; k += 4)
              __stcs(reinterpret_cast<float4*>(drow + k), make_float4(acc[k], acc[k + 1], acc[k + 2], acc[k + 3]));
          } else {
#pragma unroll
            for (int k = 0; k < DL; k += 2) __stcs(reinterpret_cast<float2*>(drow + k), make_float2(acc[k], acc[k + 1]));
          }
#pragma unroll
          for (int k = 0; k < DL; ++k) acc[k] = 0.f;
          ++j;
        };
        for (;;) {
          while (pos == end) {   // rows whose lists are exhausted (or empty)
            write_row();
            if (j == jb) break;
            end = rowptr[j + 1];
          }
          if (j == jb) break;
          // pos < end <= stop: a batch of U entries from pos
          uint32_t x[U][DL / 2];
          float gq[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int e = list[min(pos + u, stop - 1)];
            gq[u] = dsv[entry_query(p, e)];
            load_row_words<DL>(Qs + static_cast<uint32_t>(e) * qrow_bytes, x[u]);   // Q[q, i, :], e = q*nq + i
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (pos + u < stop) {
              while (pos + u == end) {   // entry pos + u opens a later row (stays below jb)
                write_row();
                end = rowptr[j + 1];
              }
#pragma unroll
              for (int k = 0; k < DL / 2; ++k) fma2(acc[2 * k], acc[2 * k + 1], gq[u], unpack2<T>(x[u][k]));
            }
          }
          pos = min(pos + U, stop);
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------- dQ
// Each thread owns 32 dimensions of one destination row, so a CTA holds
// R = 256 / (d / 32) rows of one query. Documents are taken in blocks of
// K = 2048 / R: the block's argmax entries for the CTA's rows (K x R
// int32, contiguous per document), its dS values and document lengths are
// loaded into registers one block ahead (eight entries per thread) and
// staged in shared memory, so reading them never waits on memory. Per
// document a thread copies its 64-byte slice of the selected D row into its
// own shared-memory slot with 16-byte cp.async (zero-fill for a skipped
// entry), kDqDepth documents ahead of the one it accumulates. blockIdx.y
// picks one of `splits` contiguous document ranges; with one range the sum
// goes straight to dQ, otherwise to partial[range] for dq_reduce_kernel.
constexpr int kDqThreads = 256;
constexpr int kDqDepth = 6;                 // documents in flight per thread
constexpr int kDqStage = 2048;              // argmax entries staged per block (8 per thread)

__host__ __device__ constexpr int dq_rows(int d) { return kDqThreads / (d / 32); }
__host__ __device__ constexpr int dq_block_docs(int d) { return kDqStage / dq_rows(d); }
// [depth][4 x 16 B][thread] row slices (the v-th 16 bytes of all threads
// contiguous), then [2][kDqStage] argmax entries, [2][K] dS and [2][K] lengths
__host__ __device__ constexpr size_t dq_smem_bytes(int d) {
  return static_cast<size_t>(kDqDepth) * 4 * kDqThreads * 16 + 2 * kDqStage * 4 + 2 * 2 * dq_block_docs(d) * 4;
}

template <typename T>
__global__ void __launch_bounds__(kDqThreads, 2) dq_kernel(const BwdParams p) {
  extern __shared__ __align__(16) uint8_t dq_raw[];
  const int tid = threadIdx.x;
  const int d = p.d, tpr = d / 32, R = dq_rows(d), K = dq_block_docs(d);
  const int blocks_per_q = (p.nq + R - 1) / R;
  const int q = blockIdx.x / blocks_per_q;
  const int i0 = (blockIdx.x - q * blocks_per_q) * R;
  const int rr = tid / tpr, part = tid - rr * tpr;
  const int i = i0 + rr;
  const bool active = rr < R && i < p.nq;  // d / 32 need not divide the thread count
  const int64_t bs = (p.B * blockIdx.y) / p.splits, be = (p.B * (blockIdx.y + 1)) / p.splits;
  const int64_t n = be - bs;
  // The row is cut into 4 bands of d / 4 elements; the row's tpr threads take
  // 8 consecutive elements of each band, so the threads of a row copy a band's
  // bytes contiguously and every 16-byte copy instruction of a warp covers
  // whole 32-byte sectors. acc[8 v + h] is element v * band + 8 part + h.
  const int band = d / 4;
  const T* Dp = static_cast<const T*>(p.D) + part * 8;
  const uint32_t slot0 = smem_u32(dq_raw) + static_cast<uint32_t>(tid) * 16;
  int32_t* am_s = reinterpret_cast<int32_t*>(dq_raw + static_cast<size_t>(kDqDepth) * 4 * kDqThreads * 16);  // [2][K][R]
  float* ds_s = reinterpret_cast<float*>(am_s + 2 * kDqStage);                                               // [2][K]
  int32_t* len_s = reinterpret_cast<int32_t*>(ds_s + 2 * K);                                                 // [2][K]
  bool bad = false;

  // block staging: entry x = tid + 256 m is document x / R, row x % R of the block
  int sa[kDqStage / kDqThreads];
  float sg = 0.f;
  int sl = 0;
  auto load_block = [&](int64_t blk) {
    const int64_t b0 = bs + blk * K;
#pragma unroll
    for (int m = 0; m < kDqStage / kDqThreads; ++m) {
      const int x = tid + kDqThreads * m, kk = x / R, r = x - kk * R;
      sa[m] = -1;
      if (blk * K + kk < n && i0 + r < p.nq)
        sa[m] = __ldg(p.argmax + (static_cast<int64_t>(q) * p.B + b0 + kk) * p.nq + i0 + r);
    }
    if (tid < K && blk * K + tid < n) {
      sg = __ldg(p.dS + static_cast<int64_t>(q) * p.B + b0 + tid);
      sl = doc_length(p, b0 + tid);   // -1: the document's length itself is invalid
    }
  };
  auto store_block = [&](int buf) {
#pragma unroll
    for (int m = 0; m < kDqStage / kDqThreads; ++m) am_s[buf * kDqStage + tid + kDqThreads * m] = sa[m];
    if (tid < K) {
      ds_s[buf * K + tid] = sg;
      len_s[buf * K + tid] = sl;
    }
  };
  // argmax of entry j for this thread's row (staged at block position kk of
  // buffer buf), validated against the document's length (-1: nothing to
  // add; a bad entry also sets the bad-input bit)
  auto entry = [&](int64_t j, int kk, int buf) -> int {
    if (!active || j >= n) return -1;
    const int v = am_s[buf * kDqStage + kk * R + rr];
    const int L = len_s[buf * K + kk];
    if (v >= 0 && v < L) return v;
    if (v < -1 || v >= 0) bad = true;
    return -1;
  };

  load_block(0);
  store_block(0);
  __syncthreads();
  if (K < n) load_block(1);
  // issue pointer: entry ij at block position ikk of block iblk (buffer iblk & 1)
  int64_t ij = 0, iblk = 0;
  int ikk = 0;
  const T* dbase = Dp + bs * static_cast<int64_t>(p.nd) * d;   // document bs + ij's rows
  const int64_t doc_elems = static_cast<int64_t>(p.nd) * d;
  // The copy of an entry into ring slot `slot`; returns the weight to apply
  // when it is consumed (0 for nothing to add: the slot is then zero-filled,
  // so the consumer's FMAs add zeros and need no branch).
  auto issue_next = [&](int slot) -> float {
    if (ikk == 0 && iblk > 0 && ij < n) {
      // entering block iblk: stage it in the buffer block iblk - 2 used (every
      // thread has consumed that block: the consumer runs kDqDepth - 1 entries
      // behind, and K > kDqDepth), then start loading block iblk + 1
      __syncthreads();
      store_block(static_cast<int>(iblk & 1));
      __syncthreads();
      if ((iblk + 1) * K < n) load_block(iblk + 1);
    }
    const int buf = static_cast<int>(iblk & 1);
    const int a = entry(ij, ikk, buf);
    const float g = a >= 0 ? ds_s[buf * K + ikk] : 0.f;
    const uint32_t dst = slot0 + static_cast<uint32_t>(slot * 4 * kDqThreads * 16);
    const T* src = a >= 0 ? dbase + static_cast<uint32_t>(a) * static_cast<uint32_t>(d) : Dp;
#pragma unroll
    for (int v = 0; v < 4; ++v) cp_async16(dst + v * kDqThreads * 16, src + v * band, a >= 0 ? 16u : 0u);
    cp_async_commit();
    ++ij;
    dbase += doc_elems;
    if (++ikk == K) {
      ikk = 0;
      ++iblk;
    }
    return g;
  };
  float gw[kDqDepth];   // weight of the entry in each ring slot
#pragma unroll
  for (int k = 0; k < kDqDepth - 1; ++k) gw[k] = issue_next(k);
  float acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.f;
  for (int64_t j0 = 0; j0 < n; j0 += kDqDepth) {
#pragma unroll
    for (int k = 0; k < kDqDepth; ++k) {
      if (j0 + k >= n) break;
      gw[(k + kDqDepth - 1) % kDqDepth] = issue_next((k + kDqDepth - 1) % kDqDepth);   // entry j + depth - 1
      cp_async_wait<kDqDepth - 1>();  // entry j's copies have landed (zeros if there was nothing to copy)
      const float g = gw[k];
      const uint8_t* src = dq_raw + k * 4 * kDqThreads * 16 + tid * 16;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + v * kDqThreads * 16);
#pragma unroll
        for (int h = 0; h < 4; ++h)
          fma2(acc[v * 8 + 2 * h], acc[v * 8 + 2 * h + 1], g,
               unpack2<T>(h == 0 ? w.x : h == 1 ? w.y : h == 2 ? w.z : w.w));
      }
    }
  }
  cp_async_wait<0>();
  if (active) {
    float* out = (p.splits > 1 ? p.partial + static_cast<int64_t>(blockIdx.y) * p.nQ * p.nq * d : p.dQ) +
                 (static_cast<int64_t>(q) * p.nq + i) * d + part * 8;
#pragma unroll
    for (int v = 0; v < 4; ++v)
#pragma unroll
      for (int h = 0; h < 8; h += 4)
        *reinterpret_cast<float4*>(out + v * band + h) =
            make_float4(acc[8 * v + h], acc[8 * v + h + 1], acc[8 * v + h + 2], acc[8 * v + h + 3]);
  }
  if (bad) atomicOr(p.status, kDevErrBadInput);
}

// dQ = sum of the per-range partials, in range order (deterministic).
__global__ void dq_reduce_kernel(const BwdParams p) {
  const int64_t n4 = static_cast<int64_t>(p.nQ) * p.nq * p.d / 4;
  const float4* src = reinterpret_cast<const float4*>(p.partial);
  float4* dst = reinterpret_cast<float4*>(p.dQ);
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n4;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = src[e];
    for (int s = 1; s < p.splits; ++s) {
      const float4 v = src[s * n4 + e];
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    dst[e] = a;
  }
}

template <typename T, int NW>
maxsim_status launch_dd_nw(const BwdParams& p, size_t smem, int grid, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  switch (p.d / 32) {
#define MSIM_DD(DPL)                                                                                        \
  case DPL:                                                                                                 \
    e = cudaFuncSetAttribute(dd_kernel<T, DPL, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,           \
                             static_cast<int>(smem));                                                       \
    if (e == cudaSuccess) dd_kernel<T, DPL, NW><<<grid, NW * 32, smem, stream>>>(p);                        \
    break;
    MSIM_DD(2) MSIM_DD(4) MSIM_DD(6) MSIM_DD(8) MSIM_DD(10) MSIM_DD(12) MSIM_DD(14) MSIM_DD(16)
    MSIM_DD(18) MSIM_DD(20) MSIM_DD(22) MSIM_DD(24) MSIM_DD(26) MSIM_DD(28) MSIM_DD(30) MSIM_DD(32)
#undef MSIM_DD
    default: return MAXSIM_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  return MAXSIM_OK;
}

// dD: 16 warps per CTA and two CTAs per SM when the per-document sort fits
// twice in shared memory (the ColPali shape: 100 KB), else 8 warps.
template <typename T>
maxsim_status launch_dd(const BwdParams& p, const DeviceInfo* dev, cudaStream_t stream) {
  const int ne = p.nQ * p.nq;
  const size_t budget = static_cast<size_t>(dev->max_smem_optin);
  const size_t smem16 = dd_smem_bytes(16, p.nd, p.nQ, ne), smem8 = dd_smem_bytes(8, p.nd, p.nQ, ne);
  const int64_t want = static_cast<int64_t>(dev->sm_count) * 2;
  const int grid = static_cast<int>(p.B < want ? p.B : want);
  if (2 * smem16 + 2048 <= budget + 1024) return launch_dd_nw<T, 16>(p, smem16, grid, stream);
  if (smem8 > budget) return MAXSIM_ERR_UNSUPPORTED;
  return launch_dd_nw<T, 8>(p, smem8, grid, stream);
}

template <typename T>
maxsim_status launch_dq(const BwdParams& p, cudaStream_t stream) {
  const int R = dq_rows(p.d);
  const int blocks = p.nQ * ((p.nq + R - 1) / R);
  const size_t dq_smem = dq_smem_bytes(p.d);
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dq_smem));
  if (e == cudaSuccess) dq_kernel<T><<<dim3(blocks, p.splits), kDqThreads, dq_smem, stream>>>(p);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  if (p.splits > 1) {
    const int64_t n4 = static_cast<int64_t>(p.nQ) * p.nq * p.d / 4;
    const int64_t want = (n4 + 255) / 256;
    dq_reduce_kernel<<<static_cast<int>(want < 4096 ? want : 4096), 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
  }
  return MAXSIM_OK;
}

template <typename T>
maxsim_status launch_typed(const BwdParams& p, const DeviceInfo* dev, int parts, cudaStream_t stream) {
  if (parts & kBackwardDD) {
    const maxsim_status st = launch_dd<T>(p, dev, stream);
    if (st != MAXSIM_OK) return st;
  }
  return (parts & kBackwardDQ) ? launch_dq<T>(p, stream) : MAXSIM_OK;
}

}  // namespace

int backward_splits(int64_t B) {
  const int64_t s = B / 1024;  // at least ~1K documents per range
  return static_cast<int>(s < 1 ? 1 : (s > 8 ? 8 : s));
}

size_t backward_workspace_bytes(int n_queries, int nq, int d, int64_t B) {
  const int s = backward_splits(B);
  return s > 1 ? static_cast<size_t>(s) * n_queries * nq * d * sizeof(float) : 0;
}

maxsim_status launch_backward(const void* Q, int n_queries, int nq, int d, const void* D, int64_t B, int nd,
                              const int32_t* doc_len, int is_bf16, const int32_t* argmax, const float* dS, float* dQ,
                              float* dD, float* workspace, int parts, cudaStream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return MAXSIM_ERR_CUDA;
  BwdParams p;
  p.Q = Q;
  p.D = D;
  p.doc_len = doc_len;
  p.argmax = argmax;
  p.dS = dS;
  p.dQ = dQ;
  p.dD = dD;
  p.B = B;
  p.nQ = n_queries;
  p.nq = nq;
  p.d = d;
  p.nd = nd;
  p.nq_inv = nq > 1 ? static_cast<uint32_t>(((uint64_t(1) << 32) + nq - 1) / nq) : 0u;   // nq <= 65536
  p.splits = backward_splits(B);
  p.partial = workspace;
  p.status = dev->status;
  return is_bf16 ? launch_typed<__nv_bfloat16>(p, dev, parts, stream) : launch_typed<__half>(p, dev, parts, stream);
}

}  // namespace msim

// route.cu -- span scores and top-k selection.
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: every
// query scores the O(L^0.5) candidate spans and keeps the top k.  The router
// is fixed by the specification: score_j = q . summary_j in fp32, ties to
// the lower span index.  Candidates of a query at position t are the complete
// spans j < l = floor(t / S) (its own span l is always attended anyway).
//
// Each kernel computes a score in an order that depends only on the index
// of the dimension, never on the span's position in a tile, so spans with
// identical summaries get identical scores and tie exactly.  Scores never
// leave the chip: each kernel keeps, per query row, a running list of its
// best (score, span) pairs in registers or shared memory.
#include <cooperative_groups.h>

#include "decode_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace ssa {
namespace {

constexpr int kMaxK = 64;   // topk limit
constexpr int kCluster = 16; // CTAs splitting one kv-head's candidates in decode

// Order-preserving 32-bit key of a finite score: a higher score has a
// higher key; 0 is reserved for "no candidate".
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- decode
// A candidate of the decode router is one 64-bit entry: the score's key in
// the high word, the complement of the span in the low word.  One unsigned
// comparison then orders by score and, among equal scores, puts the lower
// span first; entries are distinct (spans are), and 0 means "none".
__device__ __forceinline__ uint64_t make_entry(float s, int64_t j) {
  return ((uint64_t)score_key(s) << 32) | (uint32_t)~(uint32_t)j;
}
__device__ __forceinline__ int entry_span(uint64_t e) { return (int)~(uint32_t)e; }
__device__ __forceinline__ float entry_score(uint64_t e) {
  const uint32_t k = (uint32_t)(e >> 32);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// The 16 bytes w as fp32 values: eight 16-bit or four fp32 elements.
template <int DT>
__device__ __forceinline__ void unpack16(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == DT_F32) {
      f[i] = __uint_as_float(u[i]);
    } else if constexpr (DT == DT_BF16) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
      const float2 v = __half22float2(h);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
}
__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Warp lists of 32 * E entries: element e = i * 32 + lane sits in register
// i of the lane.  Bitonic networks (Batcher): a compare-exchange stage of
// distance j inside runs of length k leaves the larger entry at the lower
// index when the run is to end descending ((e & k) == 0), else the smaller.
template <int E>
__device__ __forceinline__ void bitonic_stage(uint64_t (&a)[E], int j, int k, int lane) {
  if (j >= 32) {
    const int jj = j >> 5;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (i & jj) continue;
      const int i2 = i | jj;
      const bool desc = ((i * 32 + lane) & k) == 0;
      const uint64_t hi = umax64(a[i], a[i2]), lo = umin64(a[i], a[i2]);
      a[i] = desc ? hi : lo;
      a[i2] = desc ? lo : hi;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const uint64_t p = __shfl_xor_sync(0xffffffffu, a[i], j);
      const int e = i * 32 + lane;
      const bool take_max = ((e & j) == 0) == ((e & k) == 0);
      a[i] = take_max ? umax64(a[i], p) : umin64(a[i], p);
    }
  }
}

// Sorts the warp's 32 * E entries descending.
template <int E>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&a)[E], int lane) {
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) bitonic_stage<E>(a, j, k, lane);
}

// L <- the best 32 * E of L and B, both descending, descending.  The
// element-wise maximum of L and reversed B is a bitonic sequence that holds
// the best 32 * E of the two; one merge network sorts it.
template <int E>
__device__ __forceinline__ void merge_best_desc(uint64_t (&L)[E], const uint64_t (&B)[E], int lane) {
#pragma unroll
  for (int i = 0; i < E; ++i) L[i] = umax64(L[i], __shfl_sync(0xffffffffu, B[E - 1 - i], 31 - lane));
#pragma unroll
  for (int j = 16 * E; j > 0; j >>= 1) bitonic_stage<E>(L, j, 32 * E, lane);
}

// grid (kCluster, Hkv, B), one cluster of 16 CTAs per (b, kv-head), 256
// threads.  CTA `rank` owns candidates [rank*chunk, (rank+1)*chunk).
//  scores   blocks of 64 candidates, four lanes per candidate, every head
//           of the group per thread.  Lane quarter qq sums the dimensions d
//           with (d / 4) % 4 == qq in increasing order; the quarters are
//           added as (q0 + q1) + (q2 + q3).  The CTA's summaries are
//           prefetched into L2 before the kernel waits for its predecessor.
//  level 1  one warp per head sorts each block and merges it into its list
//           of the best LC = 32 * E >= k entries so far, kept in registers.
//  level 2  every CTA sends its list of head h to CTA h; after a cluster
//           barrier CTA h merges its 16 lists in a four-level tree.  The
//           best k of the result are its winners, written in ascending span
//           order.
// With PLAN (a whole decode step) the winners also go to CTA 0, which after
// a second cluster barrier builds the group's decode plan (decode_plan.cuh)
// for the attend kernel that follows.
// With GRP (group-shared selection) the CTAs score one query per kv-head,
// the sum of the group's g queries, each element summed over the heads in
// order in fp32 (the group router's own sum, so the selections are its
// bits), and the winners are every head's selection.
constexpr int kBlk = 64;

template <int G, int D, int E>
struct DecodeRouteSmem {
  static constexpr int kQS = D / 4 + 4;  // floats per lane quarter of a q row (padded)
  float q[G][4 * kQS];
  uint64_t sc[G][kBlk];                  // the block's entries per head (0 = none)
  uint64_t recv[kCluster][32 * E];       // the lists of this CTA's head, one per CTA
  dplan::PlanSmem ps;                    // winners in span order and plan scratch (CTA 0)
};

template <int DT, int D, int G, int E, bool PLAN, bool GRP>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(256, 1)
    route_decode_kernel(const void* __restrict__ Q, const float* __restrict__ summ,
                        int32_t* __restrict__ sel, float* __restrict__ sel_score, int Hq, int Hkv,
                        int64_t pos, int S, int topk, int64_t ns_cap, dplan::Plan plan, dplan::Geo geo) {
  using Sm = DecodeRouteSmem<G, D, E>;
  constexpr int kQS = Sm::kQS;
  constexpr int NL = D / 16;          // float4 loads per lane per candidate
  constexpr int HPW = (G + 7) / 8;    // heads per warp
  __shared__ __align__(16) Sm sm;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = Hq / Hkv;
  const int gs = GRP ? 1 : g;   // query rows scored: each head, or the group's sum
  const int64_t ell = pos / S;
  const int64_t chunk = (ell + kCluster - 1) / kCluster;
  const int64_t lo = min(ell, (int64_t)rank * chunk);
  const int64_t hi = min(ell, lo + chunk);
  const int qq = tid & 3, cj = tid >> 2;  // lane quarter, candidate of the block

  const float* sbase = summ + (int64_t)(b * Hkv + kvh) * ns_cap * D;
  // the summaries do not depend on the predecessor's results in a decode
  // step, but they may be its output in general: only warm L2 before the wait
  for (int64_t line = lo * (D / 32) + tid; line < hi * (D / 32); line += 256)
    ptx::prefetch_l2_evict_last(sbase + line * 32);
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();

  const uint64_t pol_keep = ptx::policy_evict_last();  // the summaries are read every step
  float4 sv[NL];
  auto load_block = [&](int64_t jb) {
    const int64_t j = jb + cj;
    if (j < hi) {
      const float4* src = reinterpret_cast<const float4*>(sbase + j * D);
#pragma unroll
      for (int i = 0; i < NL; ++i) sv[i] = ptx::ldg_hint(src + 4 * i + qq, pol_keep);
    }
  };
  if (lo < hi) load_block(lo);
  {
    // the group's g rows of Q are contiguous: 16-byte loads, all in flight
    constexpr int V = DT == DT_F32 ? 4 : 8;  // elements per 16 bytes
    const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(Q) +
                                                       (int64_t)(b * Hq + kvh * g) * D * (16 / V));
    const int nvec = g * D / V;
    uint4 raw[(G * D / V + 255) / 256];
#pragma unroll
    for (int u = 0; u < (G * D / V + 255) / 256; ++u)
      if (tid + 256 * u < nvec) raw[u] = qsrc[tid + 256 * u];
    if constexpr (PLAN && DT != DT_F32) {
      // the attend kernel reads the step's queries from this device copy, so
      // that Q may also be page-locked host memory read once over the link
      if (rank == 0) {
        uint4* qdst = reinterpret_cast<uint4*>(plan.q + (int64_t)(b * Hq + kvh * g) * D);
#pragma unroll
        for (int u = 0; u < (G * D / V + 255) / 256; ++u)
          if (tid + 256 * u < nvec) qdst[tid + 256 * u] = raw[u];
      }
    }
    if constexpr (GRP) {
      // the group's summed query, four dimensions per thread
      if (tid < D / 4) {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int h = 0; h < g; ++h) {
          const int64_t base = (int64_t)(b * Hq + kvh * g + h) * D + 4 * tid;
#pragma unroll
          for (int c = 0; c < 4; ++c) s4[c] += load_elem<DT>(Q, base + c);
        }
        *reinterpret_cast<float4*>(&sm.q[0][(tid & 3) * kQS + 4 * (tid >> 2)]) =
            make_float4(s4[0], s4[1], s4[2], s4[3]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < (G * D / V + 255) / 256; ++u) {
        const int x = tid + 256 * u;
        if (x < nvec) {
          float f[8];
          unpack16<DT>(raw[u], f);
#pragma unroll
          for (int c = 0; c < V; c += 4) {
            const int e = x * V + c, hl = e / D, d = e - hl * D, ff = d >> 2;
            *reinterpret_cast<float4*>(&sm.q[hl][(ff & 3) * kQS + 4 * (ff >> 2)]) =
                make_float4(f[c], f[c + 1], f[c + 2], f[c + 3]);
          }
        }
      }
    }
  }
  __syncthreads();

  uint64_t L[HPW][E];  // this warp's level-1 lists (heads warp, warp + 8)
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh)
#pragma unroll
    for (int i = 0; i < E; ++i) L[hh][i] = 0ull;

  for (int64_t jb = lo; jb < hi; jb += kBlk) {
    {
      const int64_t j = jb + cj;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
      if (j < hi) {
#pragma unroll
        for (int i = 0; i < NL; ++i) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (h < gs) {
              const float4 qv = *reinterpret_cast<const float4*>(&sm.q[h][qq * kQS + 4 * i]);
              acc[h] = fmaf(qv.x, sv[i].x, acc[h]);
              acc[h] = fmaf(qv.y, sv[i].y, acc[h]);
              acc[h] = fmaf(qv.z, sv[i].z, acc[h]);
              acc[h] = fmaf(qv.w, sv[i].w, acc[h]);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (h < gs) {
          float a = acc[h];
          a += __shfl_xor_sync(0xffffffffu, a, 1);
          a += __shfl_xor_sync(0xffffffffu, a, 2);
          if (qq == 0) sm.sc[h][cj] = j < hi ? make_entry(a, j) : 0ull;
        }
      }
    }
    if (jb + kBlk < hi) load_block(jb + kBlk);
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
      const int h = warp + 8 * hh;
      if (h < gs) {
        uint64_t blk[2] = {sm.sc[h][lane], sm.sc[h][lane + 32]};
        bitonic_sort_desc<2>(blk, lane);
        if constexpr (E == 1) {
          const uint64_t top[1] = {blk[0]};
          merge_best_desc<1>(L[hh], top, lane);
        } else {
          merge_best_desc<2>(L[hh], blk, lane);
        }
      }
    }
    __syncthreads();
  }
  // level 2: list of head h -> CTA h
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int h = warp + 8 * hh;
    if (h < gs) {
      uint64_t* dst = cluster.map_shared_rank(&sm.recv[rank][0], h);
#pragma unroll
      for (int i = 0; i < E; ++i) dst[i * 32 + lane] = L[hh][i];
    }
  }
  cluster.sync();
  if (rank < gs) {
    const int h = rank;
    for (int lev = 0; lev < 4; ++lev) {
      const int a = warp << (lev + 1), c = a + (1 << lev);
      if (c < kCluster) {
        uint64_t A[E], Bv[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
          A[i] = sm.recv[a][i * 32 + lane];
          Bv[i] = sm.recv[c][i * 32 + lane];
        }
        merge_best_desc<E>(A, Bv, lane);
#pragma unroll
        for (int i = 0; i < E; ++i) sm.recv[a][i * 32 + lane] = A[i];
      }
      __syncthreads();
    }
    if (warp == 0) {
      // the best k, in ascending span order (spans are distinct)
      const uint64_t* w = sm.recv[0];
      int n = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int x = lane + 32 * i;
        n += __popc(__ballot_sync(0xffffffffu, x < topk && w[x] != 0ull));
      }
      // the heads this selection belongs to: head h, or every head of the group
      const int h0 = GRP ? 0 : h, h1 = GRP ? g : h + 1;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int x = lane + 32 * i;
        if (x < n) {
          const int jx = entry_span(w[x]);
          int p = 0;
          for (int y = 0; y < n; ++y) p += entry_span(w[y]) < jx;
          for (int ht = h0; ht < h1; ++ht) {
            const int64_t row = (int64_t)b * Hq + kvh * g + ht;
            sel[row * topk + p] = jx;
            if (sel_score) sel_score[row * topk + p] = entry_score(w[x]);
            if constexpr (PLAN) *cluster.map_shared_rank(&sm.ps.sj[ht][p], 0) = jx;
          }
        } else if (x < topk) {
          for (int ht = h0; ht < h1; ++ht) {
            const int64_t row = (int64_t)b * Hq + kvh * g + ht;
            sel[row * topk + x] = -1;
            if (sel_score) sel_score[row * topk + x] = __int_as_float(0x7fc00000);
          }
        }
      }
      if constexpr (PLAN) {
        if (lane < h1 - h0) *cluster.map_shared_rank(&sm.ps.nv[h0 + lane], 0) = n;
      }
    }
  }
  if constexpr (PLAN) {
    cluster.sync();
    if (rank == 0) dplan::plan_build<8>(b * Hkv + kvh, sm.ps, plan, geo);
  }
}

// ---------------------------------------------------------------- prefill
// grid (ceil(n_q * g / 64), Hkv, B).  A CTA owns 64 rows of one kv-head:
// row r of the tile is query i = (row0 + r) / g, head kvh * g + (row0 + r) % g.
// It streams the candidate summaries in tiles of 64, computes the 64 x 64
// score tile with fp32 FMA (4 x 4 per thread, operands transposed in shared
// memory), and folds each tile into the rows' sorted lists.
constexpr int kRows = 64, kCols = 64, kPad = 68;

template <int D>
size_t prefill_smem_bytes(int topk) {
  return sizeof(float) * (2 * D * kPad + kRows * (kCols + 1) + kRows * topk) +
         sizeof(int) * kRows * topk;
}

template <int DT, int D>
__global__ void __launch_bounds__(256) route_prefill_kernel(
    const void* __restrict__ Q, const float* __restrict__ summ, int32_t* __restrict__ sel,
    float* __restrict__ sel_score, int Hq, int Hkv, int64_t n_q, int64_t q_pos0, int S, int topk,
    int64_t ns_cap) {
  extern __shared__ __align__(16) float smem[];
  float* qT = smem;                    // [D][kPad]
  float* sT = qT + D * kPad;           // [D][kPad]
  float* sc = sT + D * kPad;           // [kRows][kCols + 1]
  float* lsv = sc + kRows * (kCols + 1);  // [kRows][kMaxK]
  int* lsj = reinterpret_cast<int*>(lsv + kRows * topk);

  const int tid = threadIdx.x;
  const int g = Hq / Hkv;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int64_t rows_total = n_q * g;
  const int64_t row0 = (int64_t)blockIdx.x * kRows;
  const int64_t nrows = min((int64_t)kRows, rows_total - row0);

  for (int x = tid; x < kRows * D; x += 256) {
    int r = x / D, c = x - r * D;
    float v = 0.f;
    if (r < nrows) {
      int64_t fr = row0 + r, i = fr / g;
      int h = kvh * g + (int)(fr - i * g);
      v = load_elem<DT>(Q, ((int64_t)(b * Hq + h) * n_q + i) * D + c);
    }
    qT[c * kPad + r] = v;
  }
  for (int x = tid; x < kRows * topk; x += 256) {
    lsv[x] = -INFINITY;
    lsj[x] = kNoSpan;
  }
  const int64_t ell_max = (q_pos0 + (row0 + nrows - 1) / g) / S;
  __syncthreads();

  const float* sbase = summ + (int64_t)(b * Hkv + kvh) * ns_cap * D;
  const int tx = tid & 15, ty = tid >> 4;
  for (int64_t jb = 0; jb < ell_max; jb += kCols) {
    for (int x = tid; x < kCols * (D / 4); x += 256) {
      int c4 = x / kCols, jj = x - c4 * kCols;
      int64_t j = jb + jj;
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < ell_max) s = __ldg(reinterpret_cast<const float4*>(sbase + j * D) + c4);
      sT[(c4 * 4 + 0) * kPad + jj] = s.x;
      sT[(c4 * 4 + 1) * kPad + jj] = s.y;
      sT[(c4 * 4 + 2) * kPad + jj] = s.z;
      sT[(c4 * 4 + 3) * kPad + jj] = s.w;
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; ++c) {
      float4 qa = *reinterpret_cast<const float4*>(&qT[c * kPad + ty * 4]);
      float4 sb = *reinterpret_cast<const float4*>(&sT[c * kPad + tx * 4]);
      const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
      const float sv[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = fmaf(qv[a], sv[e], acc[a][e]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[(ty * 4 + a) * (kCols + 1) + tx * 4 + e] = acc[a][e];
    __syncthreads();
    if (tid < nrows) {
      const int r = tid;
      const int64_t ell = (q_pos0 + (row0 + r) / g) / S;
      const int64_t jend = min(jb + kCols, ell);
      float* lv = lsv + r * topk;
      int* lj = lsj + r * topk;
      for (int64_t j = jb; j < jend; ++j) {
        float s = sc[r * (kCols + 1) + (int)(j - jb)];
        if (!better(s, (int)j, lv[topk - 1], lj[topk - 1])) continue;
        int p = topk - 1;
        while (p > 0 && better(s, (int)j, lv[p - 1], lj[p - 1])) {
          lv[p] = lv[p - 1];
          lj[p] = lj[p - 1];
          --p;
        }
        lv[p] = s;
        lj[p] = (int)j;
      }
    }
    __syncthreads();
  }

  if (tid < nrows) {
    const int r = tid;
    const int64_t fr = row0 + r, i = fr / g;
    const int h = kvh * g + (int)(fr - i * g);
    const int64_t orow = (int64_t)(b * Hq + h) * n_q + i;
    float* lv = lsv + r * topk;
    int* lj = lsj + r * topk;
    int n = 0;
    while (n < topk && lj[n] != kNoSpan) ++n;
    // ascending span order (insertion sort of at most 32 entries)
    for (int a = 1; a < n; ++a) {
      int jv = lj[a];
      float sv = lv[a];
      int p = a;
      while (p > 0 && lj[p - 1] > jv) {
        lj[p] = lj[p - 1];
        lv[p] = lv[p - 1];
        --p;
      }
      lj[p] = jv;
      lv[p] = sv;
    }
    int32_t* out = sel + orow * topk;
    for (int s = 0; s < topk; ++s) out[s] = s < n ? lj[s] : -1;
    if (sel_score) {
      float* os = sel_score + orow * topk;
      for (int s = 0; s < topk; ++s) os[s] = s < n ? lv[s] : __int_as_float(0x7fc00000);
    }
  }
}

template <int DT, int D, int G, int E, bool PLAN, bool GRP>
cudaError_t launch_decode_route(const Problem& pr, const void* Q, int64_t q_pos0, const float* summ,
                                int32_t* sel, float* sel_score, const dplan::Plan& plan, const dplan::Geo& geo,
                                cudaStream_t st) {
  dim3 grid(kCluster, pr.Hkv, pr.B);
  // a cluster of 16 is above the portable size of 8: the kernel opts in once per device
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && !attr_done[dev]) {
    e = cudaFuncSetAttribute(route_decode_kernel<DT, D, G, E, PLAN, GRP>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_pdl(route_decode_kernel<DT, D, G, E, PLAN, GRP>, grid, dim3(256), 0, st, Q, summ, sel, sel_score,
                    pr.Hq, pr.Hkv, q_pos0, pr.S, pr.topk, pr.ns_cap, plan, geo);
}

template <int DT, int D, int G, bool PLAN, bool GRP>
cudaError_t decode_route_e(const Problem& pr, const void* Q, int64_t q_pos0, const float* summ, int32_t* sel,
                           float* sel_score, const dplan::Plan& plan, const dplan::Geo& geo, cudaStream_t st) {
  // level-1 lists of 32 entries hold the best k for k <= 32, else 64
  if (pr.topk <= 32)
    return launch_decode_route<DT, D, G, 1, PLAN, GRP>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  return launch_decode_route<DT, D, G, 2, PLAN, GRP>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
}

template <int DT, int D, bool PLAN, bool GRP = false>
cudaError_t decode_route_g(const Problem& pr, const void* Q, int64_t q_pos0, const float* summ, int32_t* sel,
                           float* sel_score, const dplan::Plan& plan, const dplan::Geo& geo, cudaStream_t st) {
  if (pr.g <= 4) return decode_route_e<DT, D, 4, PLAN, GRP>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  if (pr.g <= 8) return decode_route_e<DT, D, 8, PLAN, GRP>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  return decode_route_e<DT, D, 16, PLAN, GRP>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const float* summ, int32_t* sel, float* sel_score, cudaStream_t st) {
  if (n_q == 1) return decode_route_g<DT, D, false>(pr, Q, q_pos0, summ, sel, sel_score, {}, {}, st);
  const size_t smem = prefill_smem_bytes<D>(pr.topk);
  static bool attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_attr(route_prefill_kernel<DT, D>, prefill_smem_bytes<D>(kMaxK), attr_done);
  if (e != cudaSuccess) return e;
  int64_t tiles = (n_q * pr.g + kRows - 1) / kRows;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)tiles, pr.Hkv, pr.B);
  route_prefill_kernel<DT, D><<<grid, 256, smem, st>>>(Q, summ, sel, sel_score, pr.Hq, pr.Hkv,
                                                       n_q, q_pos0, pr.S, pr.topk, pr.ns_cap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const Problem& pr, const void* Q, int64_t pos, const float* summ, const void* K,
                               const void* V, int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st) {
  dplan::Plan plan;
  dplan::Geo geo;
  decode_plan_args(pr, pos, ws, &plan, &geo);
  cudaError_t e;
  if (pr.d == 128)
    e = pr.dtype == DT_BF16 ? decode_route_g<DT_BF16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  else
    e = pr.dtype == DT_BF16 ? decode_route_g<DT_BF16, 64, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 64, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  if (e != cudaSuccess) return e;
  return launch_attend_decode_planned(pr, plan.q, K, V, O, lse, plan, geo, ws_error(ws), st);
}

cudaError_t launch_decode_step_group(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                     const void* K, const void* V, int32_t* sel, void* O, float* lse, void* ws,
                                     cudaStream_t st) {
  dplan::Plan plan;
  dplan::Geo geo;
  decode_plan_args(pr, pos, ws, &plan, &geo, true);
  cudaError_t e;
  if (pr.d == 128)
    e = pr.dtype == DT_BF16 ? decode_route_g<DT_BF16, 128, true, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 128, true, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  else
    e = pr.dtype == DT_BF16 ? decode_route_g<DT_BF16, 64, true, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 64, true, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  if (e != cudaSuccess) return e;
  return launch_attend_decode_planned(pr, plan.q, K, V, O, lse, plan, geo, ws_error(ws), st);
}

cudaError_t launch_decode_step_q8(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                  const int8_t* Kq, const float* Ks, const int8_t* Vq, const float* Vs,
                                  int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st) {
  dplan::Plan plan;
  dplan::Geo geo;
  decode_plan_args(pr, pos, ws, &plan, &geo);
  const cudaError_t e = pr.dtype == DT_BF16
                            ? decode_route_g<DT_BF16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  if (e != cudaSuccess) return e;
  return launch_attend_decode_q8_planned(pr, plan.q, Kq, Ks, Vq, Vs, O, lse, plan, geo, ws_error(ws), st);
}

cudaError_t launch_decode_step_q4(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                  const uint32_t* Kq4, const float* Ks, const uint32_t* Vq4, const float* Vs,
                                  int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st) {
  dplan::Plan plan;
  dplan::Geo geo;
  decode_plan_args(pr, pos, ws, &plan, &geo);
  const cudaError_t e = pr.dtype == DT_BF16
                            ? decode_route_g<DT_BF16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st)
                            : decode_route_g<DT_F16, 128, true>(pr, Q, pos, summ, sel, nullptr, plan, geo, st);
  if (e != cudaSuccess) return e;
  return launch_attend_decode_q4_planned(pr, plan.q, Kq4, Ks, Vq4, Vs, O, lse, plan, geo, ws_error(ws), st);
}

cudaError_t launch_route(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const float* summ, int32_t* sel, float* sel_score, cudaStream_t st) {
  if (n_q == 0) return cudaSuccess;
  if (pr.d == 128) {
    switch (pr.dtype) {
      case DT_F32: return launch_typed<DT_F32, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
      case DT_BF16: return launch_typed<DT_BF16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
      default: return launch_typed<DT_F16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
    }
  }
  switch (pr.dtype) {
    case DT_F32: return launch_typed<DT_F32, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
    case DT_BF16: return launch_typed<DT_BF16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
    default: return launch_typed<DT_F16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, st);
  }
}

}  // namespace ssa

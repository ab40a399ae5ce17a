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
// best k (score, span) pairs in shared memory.
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

// Marks the k best of the warp's entries.  Entry (i, lane) is the i-th
// register of the lane; the entries' order (i major, lane minor) must be
// ascending span index, so that among equal keys the earlier entry is the
// lower span.  Finds the k-th largest key T by a bitwise search on the
// key's bits (one warp-wide count per bit), takes every key above T and the
// first entries equal to T.  Returns the lane's bitmask of chosen entries.
template <int NV>
__device__ __forceinline__ uint32_t warp_select(const uint32_t (&key)[NV], int k, int lane) {
  int nv = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) nv += key[i] != 0u;
  nv = __reduce_add_sync(0xffffffffu, nv);
  uint32_t chosen = 0u;
  if (nv <= k) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (key[i] != 0u) chosen |= 1u << i;
    return chosen;
  }
  uint32_t T = 0u;
#pragma unroll 1
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    int c = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) c += key[i] >= cand;
    if (__reduce_add_sync(0xffffffffu, c) >= k) T = cand;
  }
  int gt = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) gt += key[i] > T;
  int need = k - __reduce_add_sync(0xffffffffu, gt);
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t eq = __ballot_sync(0xffffffffu, key[i] == T);
    const bool take = key[i] > T || (key[i] == T && __popc(eq & lt_mask) < need);
    need -= min(need, __popc(eq));
    if (take) chosen |= 1u << i;
  }
  return chosen;
}

// Replaces a head's list (topk entries, ascending spans, invalid = kNoSpan)
// by the topk best of the list and one block of 128 scores (spans jb ..);
// NL = 0 when the list is still empty.
template <int NL>
__device__ __forceinline__ void fold_block(float* lsv, int* lsj, const float* sc, int64_t jb,
                                           int64_t hi, int lane, int topk) {
  constexpr int NV = NL + 4;
  float v[NV];
  int vj[NV];
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NL; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < topk ? lsv[e] : -INFINITY;
    vj[i] = e < topk ? lsj[e] : kNoSpan;
    key[i] = vj[i] == kNoSpan ? 0u : score_key(v[i]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t jj = jb + lane + 32 * i;
    const bool ok = jj < hi;
    v[NL + i] = ok ? sc[lane + 32 * i] : -INFINITY;
    vj[NL + i] = ok ? (int)jj : kNoSpan;
    key[NL + i] = ok ? score_key(v[NL + i]) : 0u;
  }
  const uint32_t chosen = warp_select<NV>(key, topk, lane);
  __syncwarp();
  int base = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const bool c = (chosen >> i) & 1u;
    const uint32_t bal = __ballot_sync(0xffffffffu, c);
    if (c) {
      const int p = base + __popc(bal & ((1u << lane) - 1u));
      lsv[p] = v[i];
      lsj[p] = vj[i];
    }
    base += __popc(bal);
  }
  for (int e = base + lane; e < topk; e += 32) {
    lsv[e] = -INFINITY;
    lsj[e] = kNoSpan;
  }
}

// ---------------------------------------------------------------- decode
// grid (kCluster, Hkv, B), one cluster per (b, kv-head).  CTA `rank` scores
// candidates [rank*chunk, (rank+1)*chunk) for all g heads of the group in
// blocks of 256: two lanes per candidate, each summing one half of d with
// all of its summary loads in flight at once, the two halves then added.
// Each block is folded into per-head lists; finally CTA `rank` merges head
// rank (+16) over the cluster's lists through distributed shared memory.
//
// With PLAN (a whole decode step), each final list is also pushed into CTA
// 0's shared memory, and CTA 0 then builds the group's decode plan
// (decode_plan.cuh) for the attend kernel that follows: the step needs no
// separate plan kernel.
constexpr int kBlk = 128;

template <int DT, int D, int G, int NE, bool PLAN>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(256)
    route_decode_kernel(const void* __restrict__ Q, const float* __restrict__ summ,
                        int32_t* __restrict__ sel, float* __restrict__ sel_score, int Hq, int Hkv,
                        int64_t pos, int S, int topk, int64_t ns_cap, dplan::Plan plan, dplan::Geo geo) {
  constexpr int HD = D / 2;          // dims per lane
  constexpr int HPAD = HD + 4;       // padded half stride, keeps the two halves in other banks
  constexpr int NL = HD / 4;         // float4 loads per lane
  __shared__ __align__(16) float q_s[G][2 * HPAD];
  __shared__ float sc_s[G][kBlk];
  __shared__ float lsv_s[G][kMaxK];
  __shared__ int lsj_s[G][kMaxK];
  __shared__ dplan::PlanSmem ps;     // CTA 0 of a PLAN cluster: the group's final lists and plan scratch

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = Hq / Hkv;
  const int64_t ell = pos / S;
  const int64_t chunk = (ell + kCluster - 1) / kCluster;
  const int64_t lo = min(ell, (int64_t)rank * chunk);
  const int64_t hi = min(ell, lo + chunk);

  for (int x = tid; x < G * kMaxK; x += 256) {
    lsv_s[x / kMaxK][x % kMaxK] = -INFINITY;
    lsj_s[x / kMaxK][x % kMaxK] = kNoSpan;
  }
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  for (int x = tid; x < g * D; x += 256) {
    const int hl = x / D, c = x - hl * D;
    q_s[hl][(c / HD) * HPAD + (c % HD)] = load_elem<DT>(Q, (int64_t)(b * Hq + kvh * g + hl) * D + c);
  }
  __syncthreads();

  const float* sbase = summ + (int64_t)(b * Hkv + kvh) * ns_cap * D;
  const int half = tid & 1;
  const uint64_t pol_keep = ptx::policy_evict_last();  // the summaries are read every step
  for (int64_t jb = lo; jb < hi; jb += kBlk) {
    {
      const int jj = tid >> 1;
      const int64_t j = jb + jj;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
      if (j < hi) {
        const float4* src = reinterpret_cast<const float4*>(sbase + j * D + half * HD);
        float4 sv[NL];
#pragma unroll
        for (int i = 0; i < NL; ++i) sv[i] = ptx::ldg_hint(src + i, pol_keep);
#pragma unroll
        for (int i = 0; i < NL; ++i) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (h < g) {
              const float4 qv = *reinterpret_cast<const float4*>(&q_s[h][half * HPAD + 4 * i]);
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
        if (h < g) {
          const float other = __shfl_xor_sync(0xffffffffu, acc[h], 1);
          if (half == 0) sc_s[h][jj] = j < hi ? acc[h] + other : -INFINITY;
        }
      }
    }
    __syncthreads();
    // fold this block into the head's list (list entries come first: their
    // spans are below every span of the block; the first block has no list)
    for (int h = warp; h < g; h += 8) {
      if (jb == lo)
        fold_block<0>(lsv_s[h], lsj_s[h], sc_s[h], jb, hi, lane, topk);
      else
        fold_block<2>(lsv_s[h], lsj_s[h], sc_s[h], jb, hi, lane, topk);
    }
    __syncthreads();
  }

  cluster.sync();
  // final: CTA `rank` selects head rank (+16) from the cluster's lists, which
  // concatenated in rank order are ascending in span index
  if (warp == 0) {
    for (int h = rank; h < g; h += kCluster) {
      float v[NE];
      int vj[NE];
      uint32_t key[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int e = i * 32 + lane;  // entry e = src * topk + s
        const int src = e / topk, s = e - src * topk;
        v[i] = -INFINITY;
        vj[i] = kNoSpan;
        if (src < kCluster) {
          v[i] = cluster.map_shared_rank(&lsv_s[h][0], src)[s];
          vj[i] = cluster.map_shared_rank(&lsj_s[h][0], src)[s];
        }
        key[i] = vj[i] == kNoSpan ? 0u : score_key(v[i]);
      }
      const uint32_t chosen = warp_select<NE>(key, topk, lane);
      const int64_t row = (int64_t)b * Hq + kvh * g + h;
      int32_t* out = sel + row * topk;
      float* osc = sel_score ? sel_score + row * topk : nullptr;
      int base = 0;
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const bool c = (chosen >> i) & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, c);
        if (c) {
          const int p = base + __popc(bal & ((1u << lane) - 1u));
          out[p] = vj[i];
          if (osc) osc[p] = v[i];
          if constexpr (PLAN) cluster.map_shared_rank(&ps.sj[h][0], 0)[p] = vj[i];
        }
        base += __popc(bal);
      }
      for (int e = base + lane; e < topk; e += 32) {
        out[e] = -1;
        if (osc) osc[e] = __int_as_float(0x7fc00000);
      }
      if constexpr (PLAN) {
        if (lane == 0) *cluster.map_shared_rank(&ps.nv[h], 0) = base;
      }
    }
  }
  cluster.sync();
  if constexpr (PLAN) {
    if (rank == 0) dplan::plan_build<8>(b * Hkv + kvh, ps, plan, geo);
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

template <int DT, int D, int G, int NE, bool PLAN>
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
    e = cudaFuncSetAttribute(route_decode_kernel<DT, D, G, NE, PLAN>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_pdl(route_decode_kernel<DT, D, G, NE, PLAN>, grid, dim3(256), 0, st, Q, summ, sel,
                    sel_score, pr.Hq, pr.Hkv, q_pos0, pr.S, pr.topk, pr.ns_cap, plan, geo);
}

template <int DT, int D, int G, bool PLAN>
cudaError_t decode_route_ne(const Problem& pr, const void* Q, int64_t q_pos0, const float* summ,
                            int32_t* sel, float* sel_score, const dplan::Plan& plan, const dplan::Geo& geo,
                            cudaStream_t st) {
  // entries per lane of the final cluster merge: kCluster * topk / 32
  if (pr.topk <= 16)
    return launch_decode_route<DT, D, G, 8, PLAN>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  return launch_decode_route<DT, D, G, 32, PLAN>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
}

template <int DT, int D, bool PLAN>
cudaError_t decode_route_g(const Problem& pr, const void* Q, int64_t q_pos0, const float* summ, int32_t* sel,
                           float* sel_score, const dplan::Plan& plan, const dplan::Geo& geo, cudaStream_t st) {
  if (pr.g <= 4) return decode_route_ne<DT, D, 4, PLAN>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  if (pr.g <= 8) return decode_route_ne<DT, D, 8, PLAN>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
  return decode_route_ne<DT, D, 16, PLAN>(pr, Q, q_pos0, summ, sel, sel_score, plan, geo, st);
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
  return launch_attend_decode_planned(pr, Q, K, V, O, lse, plan, geo, ws_error(ws), st);
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

// route.cu -- span scores and top-k selection.
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: every
// query scores the O(L^0.5) candidate spans and keeps the top k.  The router
// is fixed by the specification: score_j = q . summary_j in fp32, ties to
// the lower span index.  Candidates of a query at position t are the complete
// spans j < l = floor(t / S) (its own span l is always attended anyway).
//
// Both kernels compute a score as one fp32 FMA chain over c = 0 .. d-1,
// acc = fma(q[c], summary[c], acc), so a (query, span) pair gets the same
// bits in decode and in prefill, and identical spans tie exactly.  Scores
// never leave the chip: each kernel keeps, per query row, a running list of
// its best k (score, span) pairs in shared memory.
#include <cooperative_groups.h>

#include "internal.h"

namespace cg = cooperative_groups;

namespace ssa {
namespace {

constexpr int kMaxG = 16;   // query heads per kv-head
constexpr int kMaxK = 64;   // topk limit
constexpr int kCluster = 8; // CTAs splitting one kv-head's candidates in decode

// Warp-wide arg-max under `better`; every lane returns the winner.
__device__ __forceinline__ void warp_best(float& s, int& j) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float os = __shfl_xor_sync(0xffffffffu, s, off);
    int oj = __shfl_xor_sync(0xffffffffu, j, off);
    if (better(os, oj, s, j)) {
      s = os;
      j = oj;
    }
  }
}

// Writes the (at most topk) valid entries a warp holds, ascending by span,
// then -1.  Lane r holds the r-th best in slot A and the (r+32)-th best in
// slot B, as (score, span) or (-inf, kNoSpan).
__device__ __forceinline__ void warp_emit_sorted(float sa, int ja, float sb, int jb, int lane,
                                                 int topk, int32_t* sel_row, float* score_row) {
  int pa = 0, pb = 0, nvalid = 0;
  for (int src = 0; src < 32; ++src) {
    int oa = __shfl_sync(0xffffffffu, ja, src);
    int ob = __shfl_sync(0xffffffffu, jb, src);
    if (src < topk && oa != kNoSpan) {
      ++nvalid;
      pa += oa < ja;
      pb += oa < jb;
    }
    if (src + 32 < topk && ob != kNoSpan) {
      ++nvalid;
      pa += ob < ja;
      pb += ob < jb;
    }
  }
  const float nan = __int_as_float(0x7fc00000);
  if (lane < topk) {
    if (ja != kNoSpan) {
      sel_row[pa] = ja;
      if (score_row) score_row[pa] = sa;
    }
    if (lane >= nvalid) {
      sel_row[lane] = -1;
      if (score_row) score_row[lane] = nan;
    }
  }
  if (lane + 32 < topk) {
    if (jb != kNoSpan) {
      sel_row[pb] = jb;
      if (score_row) score_row[pb] = sb;
    }
    if (lane + 32 >= nvalid) {
      sel_row[lane + 32] = -1;
      if (score_row) score_row[lane + 32] = nan;
    }
  }
}

// Extracts the topk best of NV entries per lane (warp-wide) into slots A/B.
template <int NV>
__device__ __forceinline__ void warp_topk(float (&v)[NV], int (&vj)[NV], int lane, int topk,
                                          float& sa, int& ja, float& sb, int& jb) {
  sa = -INFINITY;
  ja = kNoSpan;
  sb = -INFINITY;
  jb = kNoSpan;
  for (int r = 0; r < topk; ++r) {
    float bs = -INFINITY;
    int bj = kNoSpan;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (better(v[i], vj[i], bs, bj)) {
        bs = v[i];
        bj = vj[i];
      }
    warp_best(bs, bj);
    if (bj == kNoSpan) break;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (vj[i] == bj) {
        v[i] = -INFINITY;
        vj[i] = kNoSpan;
      }
    if (lane == r) {
      sa = bs;
      ja = bj;
    } else if (lane + 32 == r) {
      sb = bs;
      jb = bj;
    }
  }
}

// ---------------------------------------------------------------- decode
// grid (kCluster, Hkv, B), one cluster per (b, kv-head).  CTA `rank` scores
// candidates [rank*chunk, (rank+1)*chunk) for all g heads of the group,
// 256 candidates at a time (one per thread), and folds each batch into
// per-head lists; then CTA `rank` merges head rank (+8) over the cluster's
// lists through distributed shared memory.
template <int DT, int D>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(256)
    route_decode_kernel(const void* __restrict__ Q, const float* __restrict__ summ,
                        int32_t* __restrict__ sel, float* __restrict__ sel_score, int Hq, int Hkv,
                        int64_t pos, int S, int topk, int64_t ns_cap) {
  __shared__ __align__(16) float q_s[kMaxG][D];
  __shared__ float sc_s[kMaxG][256];
  __shared__ float lsv_s[kMaxG][kMaxK];
  __shared__ int lsj_s[kMaxG][kMaxK];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = Hq / Hkv;
  const int64_t ell = pos / S;
  const int64_t chunk = (ell + kCluster - 1) / kCluster;
  const int64_t lo = min(ell, (int64_t)rank * chunk);
  const int64_t hi = min(ell, lo + chunk);

  for (int x = tid; x < g * D; x += 256) {
    int hl = x / D, c = x - hl * D;
    q_s[hl][c] = load_elem<DT>(Q, (int64_t)(b * Hq + kvh * g + hl) * D + c);
  }
  for (int x = tid; x < kMaxG * kMaxK; x += 256) {
    lsv_s[x / kMaxK][x % kMaxK] = -INFINITY;
    lsj_s[x / kMaxK][x % kMaxK] = kNoSpan;
  }
  __syncthreads();

  const float* sbase = summ + (int64_t)(b * Hkv + kvh) * ns_cap * D;
  for (int64_t jb = lo; jb < hi; jb += 256) {
    const int64_t j = jb + tid;
    float acc[kMaxG];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) acc[h] = 0.f;
    if (j < hi) {
      const float4* srow = reinterpret_cast<const float4*>(sbase + j * D);
#pragma unroll 4
      for (int c4 = 0; c4 < D / 4; ++c4) {
        float4 s = __ldg(srow + c4);
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          if (h < g) {
            float4 qv = *reinterpret_cast<const float4*>(&q_s[h][c4 * 4]);
            acc[h] = fmaf(qv.x, s.x, acc[h]);
            acc[h] = fmaf(qv.y, s.y, acc[h]);
            acc[h] = fmaf(qv.z, s.z, acc[h]);
            acc[h] = fmaf(qv.w, s.w, acc[h]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kMaxG; ++h)
      if (h < g) sc_s[h][tid] = j < hi ? acc[h] : -INFINITY;
    __syncthreads();
    // fold this batch into the head's list: topk rounds of warp arg-max
    for (int h = warp; h < g; h += 8) {
      float v[10];
      int vj[10];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int64_t jj = jb + lane + 32 * i;
        bool ok = jj < hi;
        v[i] = ok ? sc_s[h][lane + 32 * i] : -INFINITY;
        vj[i] = ok ? (int)jj : kNoSpan;
      }
      v[8] = lane < topk ? lsv_s[h][lane] : -INFINITY;
      vj[8] = lane < topk ? lsj_s[h][lane] : kNoSpan;
      v[9] = lane + 32 < topk ? lsv_s[h][lane + 32] : -INFINITY;
      vj[9] = lane + 32 < topk ? lsj_s[h][lane + 32] : kNoSpan;
      float sa, sb;
      int ja, jb2;
      warp_topk<10>(v, vj, lane, topk, sa, ja, sb, jb2);
      __syncwarp();
      if (lane < topk) {
        lsv_s[h][lane] = sa;
        lsj_s[h][lane] = ja;
      }
      if (lane + 32 < topk) {
        lsv_s[h][lane + 32] = sb;
        lsj_s[h][lane + 32] = jb2;
      }
    }
    __syncthreads();
  }

  cluster.sync();
  if (warp == 0) {
    constexpr int NE = kCluster * kMaxK / 32;  // entries per lane
    for (int h = rank; h < g; h += kCluster) {
      float v[NE];
      int vj[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        int e = lane + 32 * i;  // entry e of the concatenated lists
        int src = e / kMaxK, s = e % kMaxK;
        v[i] = -INFINITY;
        vj[i] = kNoSpan;
        if (s < topk) {
          const float* rv = cluster.map_shared_rank(&lsv_s[h][0], src);
          const int* rj = cluster.map_shared_rank(&lsj_s[h][0], src);
          v[i] = rv[s];
          vj[i] = rj[s];
        }
      }
      float sa, sb;
      int ja, jb2;
      warp_topk<NE>(v, vj, lane, topk, sa, ja, sb, jb2);
      const int64_t row = (int64_t)b * Hq + kvh * g + h;
      warp_emit_sorted(sa, ja, sb, jb2, lane, topk, sel + row * topk,
                       sel_score ? sel_score + row * topk : nullptr);
    }
  }
  cluster.sync();
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

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const float* summ, int32_t* sel, float* sel_score, cudaStream_t st) {
  if (n_q == 1) {
    dim3 grid(kCluster, pr.Hkv, pr.B);
    route_decode_kernel<DT, D><<<grid, 256, 0, st>>>(Q, summ, sel, sel_score, pr.Hq, pr.Hkv,
                                                     q_pos0, pr.S, pr.topk, pr.ns_cap);
    return cudaGetLastError();
  }
  const size_t smem = prefill_smem_bytes<D>(pr.topk);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(route_prefill_kernel<DT, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)prefill_smem_bytes<D>(kMaxK));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int64_t tiles = (n_q * pr.g + kRows - 1) / kRows;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)tiles, pr.Hkv, pr.B);
  route_prefill_kernel<DT, D><<<grid, 256, smem, st>>>(Q, summ, sel, sel_score, pr.Hq, pr.Hkv,
                                                       n_q, q_pos0, pr.S, pr.topk, pr.ns_cap);
  return cudaGetLastError();
}

}  // namespace

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

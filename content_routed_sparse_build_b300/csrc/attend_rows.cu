// attend_rows.cu -- exact attention over the selected spans, one warp per
// query row.  This is the fp32 path (and the path for shapes the tiled
// kernels do not take); it reads each attended key and value row once per
// query row.
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section:
// token-level attention inside the chosen spans; SubQ SSA page (stork.ai):
// exact attention over the content-selected token subset.  A query at
// position t attends the tokens of its selected spans and tokens
// [l*S, t] of its local span l = floor(t / S), with softmax weights
// exp(x - max x) / sum, x = scale * q . k.
//
// The running maximum / sum (online softmax) is kept in base 2: q is scaled
// by scale * log2(e) once, weights are exp2f(x2 - m2), and the returned lse
// is converted back to natural log.
#include "internal.h"

namespace ssa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int DT, int D>
struct RowState {
  static constexpr int E = D / 32;  // elements per lane
  float q[E], o[E];
  float m, l;
};

template <int DT, int D>
__device__ __forceinline__ void load_row(const void* base, int64_t row, int lane, float* out) {
  constexpr int E = D / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) out[e] = load_elem<DT>(base, row * D + lane * E + e);
}

// Attend tokens [t0, t1) of kv row block `kvrow0` (row index of token 0).
template <int DT, int D>
__device__ __forceinline__ void attend_range(RowState<DT, D>& st, const void* K, const void* V,
                                             int64_t kvrow0, int64_t t0, int64_t t1, int lane) {
  constexpr int E = D / 32;
  for (int64_t t = t0; t < t1; t += 4) {
    const int nt = (int)min((int64_t)4, t1 - t);
    float k[4][E], v[4][E], x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u < nt) {
        load_row<DT, D>(K, kvrow0 + t + u, lane, k[u]);
        load_row<DT, D>(V, kvrow0 + t + u, lane, v[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float p = 0.f;
      if (u < nt) {
#pragma unroll
        for (int e = 0; e < E; ++e) p = fmaf(st.q[e], k[u][e], p);
      }
      x[u] = p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] += __shfl_xor_sync(0xffffffffu, x[u], off);
    float mx = st.m;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (u < nt) mx = fmaxf(mx, x[u]);
    const float alpha = exp2f(st.m - mx);
    st.l *= alpha;
#pragma unroll
    for (int e = 0; e < E; ++e) st.o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u < nt) {
        const float p = exp2f(x[u] - mx);
        st.l += p;
#pragma unroll
        for (int e = 0; e < E; ++e) st.o[e] = fmaf(p, v[u][e], st.o[e]);
      }
    }
    st.m = mx;
  }
}

template <int DT, int D>
__global__ void __launch_bounds__(256) attend_rows_kernel(
    const void* __restrict__ Q, const void* __restrict__ K, const void* __restrict__ V,
    const int32_t* __restrict__ sel, void* __restrict__ O, float* __restrict__ lse,
    uint32_t* __restrict__ err, int Hq, int Hkv, int64_t n_q, int64_t q_pos0, int64_t L_cap, int S,
    int topk, float scale, int64_t n_rows) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const int64_t i = row % n_q;
  const int h = (int)((row / n_q) % Hq);
  const int64_t b = row / (n_q * Hq);
  const int g = Hq / Hkv;
  const int64_t kvrow0 = (b * Hkv + h / g) * L_cap;
  const int64_t t = q_pos0 + i;
  const int64_t ell = t / S;

  RowState<DT, D> st;
  load_row<DT, D>(Q, row, lane, st.q);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    st.q[e] *= scale * kLog2e;
    st.o[e] = 0.f;
  }
  st.m = -INFINITY;
  st.l = 0.f;

  // Selected spans: the row's leading strictly ascending run of complete
  // spans before the local one; anything after it other than -1 is flagged.
  const int32_t* srow = sel + row * topk;
  const int j0 = lane < topk ? srow[lane] : -1;
  const int j1 = lane + 32 < topk ? srow[lane + 32] : -1;
  bool bad;
  const int used = warp_sel_prefix(j0, j1, lane, topk, ell, &bad);
  if (bad && lane == 0) flag_error(err, SSA_DEVERR_BAD_SELECTION);
  for (int s = 0; s < used; ++s) {
    const int64_t j = __shfl_sync(0xffffffffu, s < 32 ? j0 : j1, s & 31);
    attend_range<DT, D>(st, K, V, kvrow0, j * S, (j + 1) * S, lane);
  }
  attend_range<DT, D>(st, K, V, kvrow0, ell * S, t + 1, lane);

  const float inv = 1.f / st.l;
#pragma unroll
  for (int e = 0; e < E; ++e) store_elem<DT>(O, row * D + lane * E + e, st.o[e] * inv);
  if (lse && lane == 0) lse[row] = st.m * kLn2 + logf(st.l);
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const void* K, const void* V, const int32_t* sel, void* O, float* lse,
                         uint32_t* err, cudaStream_t st) {
  const int64_t n_rows = (int64_t)pr.B * pr.Hq * n_q;
  const int64_t blocks = (n_rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attend_rows_kernel<DT, D><<<(unsigned)blocks, 256, 0, st>>>(
      Q, K, V, sel, O, lse, err, pr.Hq, pr.Hkv, n_q, q_pos0, pr.L_cap, pr.S, pr.topk, pr.scale,
      n_rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_rows(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                               const void* K, const void* V, const int32_t* sel, void* O,
                               float* lse, uint32_t* err, cudaStream_t st) {
  if (n_q == 0) return cudaSuccess;
  if (pr.d == 128) {
    switch (pr.dtype) {
      case DT_F32: return launch_typed<DT_F32, 128>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
      case DT_BF16: return launch_typed<DT_BF16, 128>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
      default: return launch_typed<DT_F16, 128>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
    }
  }
  switch (pr.dtype) {
    case DT_F32: return launch_typed<DT_F32, 64>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
    case DT_BF16: return launch_typed<DT_BF16, 64>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
    default: return launch_typed<DT_F16, 64>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, err, st);
  }
}

}  // namespace ssa

// summaries.cu -- span summaries: the mean of each span's keys.
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: the
// context is cut into O(L^0.5) spans and the spans are what gets scored; the
// summary itself is fixed by the specification as the mean of the keys.
//
// One CTA per (b*kv-head, span).  The span is one contiguous block of
// n_j * d elements, read once with 16-byte loads, four in flight per thread.
// Thread (row group r, column slice c) sums rows r, r + RPP, ... of its
// column slice in row order; the RPP partial sums are then added in fixed
// order 0 .. RPP-1.  The order depends on nothing but the row index inside
// the span, so two spans holding identical keys get bit-identical summaries.
#include "internal.h"

namespace ssa {
namespace {

template <int DT, int D>
__global__ void __launch_bounds__(256) summaries_kernel(const void* __restrict__ K,
                                                        float* __restrict__ summ, int64_t L_cap,
                                                        int64_t L, int S, int64_t span_begin,
                                                        int64_t ns_cap) {
  constexpr int kBytes = Elem<DT>::kBytes;
  constexpr int VEC = 16 / kBytes;  // elements per 16-byte load
  constexpr int TPR = D / VEC;      // threads per key row
  constexpr int RPP = 256 / TPR;    // rows per pass
  __shared__ float red[RPP * D];

  const int64_t bh = blockIdx.y;
  const int64_t j = span_begin + blockIdx.x;
  const int64_t t0 = j * S;
  const int64_t t1 = t0 + S < L ? t0 + S : L;
  const int n = (int)(t1 - t0);
  const int tr = threadIdx.x / TPR;
  const int tc = threadIdx.x % TPR;
  const char* base = static_cast<const char*>(K) + ((bh * L_cap + t0) * D + tc * VEC) * kBytes;
  constexpr int64_t kRow = (int64_t)D * kBytes;

  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;

  int r = tr;
  for (; r + 3 * RPP < n; r += 4 * RPP) {
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      x[u] = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)(r + u * RPP) * kRow));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float f[VEC];
      widen16<DT>(x[u], f);
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += f[v];
    }
  }
  for (; r < n; r += RPP) {
    uint4 x = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * kRow));
    float f[VEC];
    widen16<DT>(x, f);
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] += f[v];
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) red[tr * D + tc * VEC + v] = acc[v];
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < RPP; ++q) s += red[q * D + c];
    summ[(bh * ns_cap + j) * D + c] = s / (float)n;
  }
}

template <int DT, int D>
cudaError_t launch(const Problem& pr, const void* K, int64_t j0, int64_t j1, float* summ,
                   cudaStream_t st) {
  dim3 grid((unsigned)(j1 - j0), (unsigned)(pr.B * pr.Hkv));
  summaries_kernel<DT, D><<<grid, 256, 0, st>>>(K, summ, pr.L_cap, pr.L, pr.S, j0, pr.ns_cap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_summaries(const Problem& pr, const void* K, int64_t j0, int64_t j1, float* summ,
                             cudaStream_t st) {
  if (j1 <= j0) return cudaSuccess;
  // grid.x is limited to 2^31 - 1 and grid.y to 65535
  if (j1 - j0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (pr.d == 128) {
    switch (pr.dtype) {
      case DT_F32: return launch<DT_F32, 128>(pr, K, j0, j1, summ, st);
      case DT_BF16: return launch<DT_BF16, 128>(pr, K, j0, j1, summ, st);
      default: return launch<DT_F16, 128>(pr, K, j0, j1, summ, st);
    }
  }
  switch (pr.dtype) {
    case DT_F32: return launch<DT_F32, 64>(pr, K, j0, j1, summ, st);
    case DT_BF16: return launch<DT_BF16, 64>(pr, K, j0, j1, summ, st);
    default: return launch<DT_F16, 64>(pr, K, j0, j1, summ, st);
  }
}

}  // namespace ssa

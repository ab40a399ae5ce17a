// route_group.cu -- group-shared selection for grouped-query attention: one
// top-k per (b, kv-head, query), which every query head of the group uses.
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: each
// query keeps the top k of the O(L^0.5) candidate spans; the pages leave the
// router open.  This variant scores span j for the g query heads of a
// kv-head together: score_j = sum over the heads h of q_h . summary_j, and
// keeps the k best under (score desc, j asc) over the same candidates as the
// per-head router.  By linearity that is (sum_h q_h) . summary_j, so:
//
//  sum        q_sum[b, kvh, i] = sum over the group's heads of Q[b, h, i] (fp32)
//  route      the per-head fp32 router with one query head per kv-head
//  broadcast  each group's selection (and scores) to its g head rows
//
// With one selection per group, the g heads' spans coincide and the decode
// attention streams k spans plus the local span per kv-head instead of up to
// g k + 1.
#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct GroupLayout {
  size_t qsum, sel, score, total;
};

GroupLayout group_layout(const Problem& pr, int64_t n_q) {
  GroupLayout l;
  const size_t rows = (size_t)pr.B * pr.Hkv * n_q;
  size_t off = kWsHeader;
  l.qsum = off; off = align256(off + rows * pr.d * 4);
  l.sel = off; off = align256(off + rows * pr.topk * 4);
  l.score = off; off = align256(off + rows * pr.topk * 4);
  l.total = off;
  return l;
}

// grid-stride over the B * Hkv * n_q * D elements of q_sum
template <int DT, int D>
__global__ void __launch_bounds__(256) group_sum_kernel(const void* __restrict__ Q, float* __restrict__ qsum,
                                                        int Hq, int Hkv, int64_t n_q, int64_t total) {
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int g = Hq / Hkv;
  for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
    const int c = (int)(e % D);
    const int64_t i = (e / D) % n_q;
    const int64_t bk = e / ((int64_t)D * n_q);  // b * Hkv + kvh
    const int64_t b = bk / Hkv, kvh = bk - b * Hkv;
    float acc = 0.f;
    for (int h = 0; h < g; ++h) acc += load_elem<DT>(Q, ((b * Hq + kvh * g + h) * n_q + i) * D + c);
    qsum[e] = acc;
  }
}

// grid-stride over the B * Hq * n_q * topk entries of sel
__global__ void __launch_bounds__(256) group_broadcast_kernel(const int32_t* __restrict__ sel_g,
                                                              const float* __restrict__ score_g,
                                                              int32_t* __restrict__ sel, float* __restrict__ score,
                                                              int Hq, int Hkv, int64_t n_q, int topk,
                                                              int64_t total) {
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int g = Hq / Hkv;
  for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
    const int k = (int)(e % topk);
    const int64_t i = (e / topk) % n_q;
    const int64_t bh = e / ((int64_t)topk * n_q);  // b * Hq + h
    const int64_t b = bh / Hq, h = bh - b * Hq;
    const int64_t src = ((b * Hkv + h / g) * n_q + i) * topk + k;
    sel[e] = sel_g[src];
    if (score) score[e] = score_g[src];
  }
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                         int32_t* sel, float* sel_score, void* ws, cudaStream_t st) {
  const GroupLayout lay = group_layout(pr, n_q);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* qsum = reinterpret_cast<float*>(w8 + lay.qsum);
  int32_t* sel_g = reinterpret_cast<int32_t*>(w8 + lay.sel);
  float* score_g = reinterpret_cast<float*>(w8 + lay.score);
  const int sms = device_sm_count();
  const int64_t n_sum = (int64_t)pr.B * pr.Hkv * n_q * D;
  const int64_t blocks_sum = std::min<int64_t>((n_sum + 255) / 256, (int64_t)sms * 8);
  cudaError_t e = launch_pdl(group_sum_kernel<DT, D>, dim3((unsigned)blocks_sum), dim3(256), 0, st, Q, qsum,
                             pr.Hq, pr.Hkv, n_q, n_sum);
  if (e != cudaSuccess) return e;
  Problem p1 = pr;
  p1.Hq = pr.Hkv;
  p1.g = 1;
  p1.dtype = DT_F32;
  e = launch_route(p1, qsum, n_q, q_pos0, summ, sel_g, sel_score ? score_g : nullptr, st);
  if (e != cudaSuccess) return e;
  const int64_t n_sel = (int64_t)pr.B * pr.Hq * n_q * pr.topk;
  const int64_t blocks_sel = std::min<int64_t>((n_sel + 255) / 256, (int64_t)sms * 8);
  return launch_pdl(group_broadcast_kernel, dim3((unsigned)blocks_sel), dim3(256), 0, st, sel_g,
                    static_cast<const float*>(score_g), sel, sel_score, pr.Hq, pr.Hkv, n_q, pr.topk, n_sel);
}

}  // namespace

size_t route_group_ws_bytes(const Problem& pr, int64_t n_q) { return group_layout(pr, n_q).total - kWsHeader; }

cudaError_t launch_route_group(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                               int32_t* sel, float* sel_score, void* ws, cudaStream_t st) {
  if (n_q == 0) return cudaSuccess;
  if (pr.d == 128) {
    switch (pr.dtype) {
      case DT_F32: return launch_typed<DT_F32, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
      case DT_BF16: return launch_typed<DT_BF16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
      default: return launch_typed<DT_F16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
    }
  }
  switch (pr.dtype) {
    case DT_F32: return launch_typed<DT_F32, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
    case DT_BF16: return launch_typed<DT_BF16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
    default: return launch_typed<DT_F16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
  }
}

}  // namespace ssa

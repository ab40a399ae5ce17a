// decode_plan.cuh -- the plan of a decode step and the log-sum-exp merges of
// its partial outputs, shared by the decode attention kernels (decode.cu)
// and by the fused route + plan kernel of a whole decode step (route.cu).
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: each
// query attends the tokens of its chosen spans plus its own span.  In decode
// the g query heads of a kv-head group choose their spans independently;
// the plan lists the union U of those spans once, so that every key / value
// byte of the union is streamed once for all heads of the group:
//   span[u]    span index of entry u of U (ascending, the local span last)
//   mask[u]    the heads of the group that attend it
//   rank[u][h] its position in head h's sel row (topk for the local span)
// Work items are (group, entry of U, chunk of CH tokens); chunk c of entry u
// writes one partial (m, l, o) per head of mask[u] into slot
// [row][rank][c], row = b * Hq + head.
//
// The attend kernel leaves one partial per (head, rank, chunk); a merge
// kernel combines each head's partials in that order into O and lse, and
// skips the slots no item wrote (m = -inf: the plan empties them).
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace dplan {

constexpr int kMaxG = 16;
constexpr int kMaxK = 64;
constexpr int kPlanWords = 512;
constexpr int64_t kPlanBits = kPlanWords * 32;  // candidates the bitmap path covers

struct Plan {
  int* n_union;       // [n_grp]   |U| including the local span
  int* n_items;       // [n_grp]   work items of the group
  int* span;          // [n_grp][umax]
  uint32_t* mask;     // [n_grp][umax] heads (bit r = head kvh*g + r) that attend the span
  uint8_t* rank;      // [n_grp][umax][16] position of the span in each head's sel row (topk = local)
  int* counter;       // work-item counter of the attend kernel
  float* ml;          // [B*Hq][topk+1][C][2]  (m, l) per partial, base-2 m
  float* po;          // [B*Hq][topk+1][C][D]  unnormalised partial outputs
  uint16_t* q;        // [B*Hq][D]  the step's 16-bit queries, copied by the route of a whole step
};

struct Geo {
  int Hq, Hkv, g, topk, S, C, CH, umax, n_grp;
  int64_t pos, ell;
  float scale_log2e;
};

// Chunks of the local span [ell * S, pos].
__host__ __device__ __forceinline__ int local_chunks(const Geo& geo) {
  const int64_t n_local = geo.pos - geo.ell * geo.S + 1;
  return (int)((n_local + geo.CH - 1) / geo.CH);
}

// Shared-memory scratch of plan_build; the caller fills sj / nv (the used
// spans of each head of the group, ascending) before calling it.
struct PlanSmem {
  int sj[kMaxG][kMaxK];
  int nv[kMaxG];
  int cpref[kMaxG][kMaxK + 1];    // prefix counts of canonical entries
  uint8_t canon[kMaxG][kMaxK];
  uint32_t smask[kMaxG * kMaxK + 1];
  uint32_t bits[kPlanWords];      // selected spans (bitmap path)
  int wpref[kPlanWords + 1];      // popcount of the words below
  int nu;
};

// Builds group grp's plan from s.sj / s.nv with all NW warps of the CTA,
// empties the (m, l) slots of the group's partials (a slot that no item
// writes keeps m = -inf and the merge skips it) and, for group 0, resets the
// item counter.
// The position of span j in U is the number of distinct selected spans below
// j: up to kPlanBits candidates it is read off a bitmap of the selected spans
// (a prefix popcount over its words); beyond that, from binary searches in
// the heads' sorted lists.  Every thread of the CTA must call it.
template <int NW>
__device__ __forceinline__ void plan_build(int grp, PlanSmem& s, const Plan& plan, const Geo& geo) {
  constexpr int NT = NW * 32;
  const int g = geo.g, k = geo.topk, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int umax = geo.umax, gbase = grp * umax;
  const int b = grp / geo.Hkv, kvh = grp - b * geo.Hkv;
  const int row0 = b * geo.Hq + kvh * g;
  const uint32_t lt = (1u << lane) - 1u;
  if (grp == 0 && tid == 0) *plan.counter = 0;
  {
    const int nparts = g * (k + 1) * geo.C;
    float2* ml = reinterpret_cast<float2*>(plan.ml) + (int64_t)row0 * (k + 1) * geo.C;
    for (int x = tid; x < nparts; x += NT) ml[x] = make_float2(-INFINITY, 0.f);
  }
  for (int x = tid; x < kMaxG * kMaxK + 1; x += NT) s.smask[x] = 0u;
  const bool bitmap = geo.ell <= kPlanBits;
  const int nw = bitmap ? (int)((geo.ell + 31) >> 5) : 0;
  for (int x = tid; x < nw; x += NT) s.bits[x] = 0u;
  __syncthreads();
  if (bitmap) {
    for (int h = warp; h < g; h += NW) {
      if (lane < s.nv[h]) atomicOr(&s.bits[s.sj[h][lane] >> 5], 1u << (s.sj[h][lane] & 31));
      if (lane + 32 < s.nv[h]) atomicOr(&s.bits[s.sj[h][lane + 32] >> 5], 1u << (s.sj[h][lane + 32] & 31));
    }
    __syncthreads();
    if (warp == 0) {
      int run = 0;
      for (int base = 0; base < nw; base += 32) {
        const int c = base + lane < nw ? __popc(s.bits[base + lane]) : 0;
        int v = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += o;
        }
        if (base + lane < nw) s.wpref[base + lane] = run + v - c;
        run += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) s.nu = run;
    }
    __syncthreads();
    for (int h = warp; h < g; h += NW) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = lane + 32 * hh;
        if (r >= s.nv[h]) continue;
        const int j = s.sj[h][r];
        const int p = s.wpref[j >> 5] + __popc(s.bits[j >> 5] & ((1u << (j & 31)) - 1u));
        // the first head to claim the position writes the span
        if (atomicOr(&s.smask[p], 1u << h) == 0u) plan.span[gbase + p] = j;
        plan.rank[(size_t)(gbase + p) * 16 + h] = (uint8_t)r;
      }
    }
  } else {
    // canonical entry: no lower head of the group holds the same span
    for (int h = warp; h < g; h += NW) {
      uint32_t bal[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = lane + 32 * hh;
        bool c = false;
        if (r < s.nv[h]) {
          const int j = s.sj[h][r];
          bool dup = false;
          for (int h2 = 0; h2 < h; ++h2) {
            int lo = 0, hi = s.nv[h2];
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (s.sj[h2][mid] < j) lo = mid + 1; else hi = mid;
            }
            dup |= lo < s.nv[h2] && s.sj[h2][lo] == j;
          }
          c = !dup;
          s.canon[h][r] = c ? 1 : 0;
        }
        bal[hh] = __ballot_sync(0xffffffffu, c);
      }
      s.cpref[h][lane] = __popc(bal[0] & lt);
      s.cpref[h][lane + 32] = __popc(bal[0]) + __popc(bal[1] & lt);
      if (lane == 0) s.cpref[h][64] = __popc(bal[0]) + __popc(bal[1]);
    }
    __syncthreads();
    // position of span j in U = number of distinct spans below j
    for (int h = warp; h < g; h += NW) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = lane + 32 * hh;
        if (r >= s.nv[h]) continue;
        const int j = s.sj[h][r];
        int p = 0;
        for (int h2 = 0; h2 < g; ++h2) {
          int lo = 0, hi = s.nv[h2];
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s.sj[h2][mid] < j) lo = mid + 1; else hi = mid;
          }
          p += s.cpref[h2][lo];
        }
        if (s.canon[h][r]) plan.span[gbase + p] = j;
        atomicOr(&s.smask[p], 1u << h);
        plan.rank[(size_t)(gbase + p) * 16 + h] = (uint8_t)r;
      }
    }
    __syncthreads();
    if (tid == 0) {
      int n = 0;
      for (int h = 0; h < g; ++h) n += s.cpref[h][s.nv[h]];
      s.nu = n;
    }
  }
  __syncthreads();
  const int nu = s.nu;
  for (int p = tid; p < nu; p += NT) plan.mask[gbase + p] = s.smask[p];
  if (tid < g) plan.rank[(size_t)(gbase + nu) * 16 + tid] = (uint8_t)k;
  if (tid == 0) {
    plan.span[gbase + nu] = (int)geo.ell;
    plan.mask[gbase + nu] = (1u << g) - 1u;
    plan.n_union[grp] = nu + 1;
    plan.n_items[grp] = nu * geo.C + local_chunks(geo);
  }
}

}  // namespace dplan
}  // namespace ssa

namespace ssa {

// decode.cu: the plan pointers and geometry of a decode step at `pos` in the
// decode workspace ws, and the attend + merge launches (16-bit or 8-bit
// cache) of a step whose plan an earlier kernel on the stream has built.
// group: the plan of a group-shared step (its own item size).
void decode_plan_args(const Problem& pr, int64_t pos, void* ws, dplan::Plan* plan, dplan::Geo* geo,
                      bool group = false);
cudaError_t launch_attend_decode_planned(const Problem& pr, const void* Q, const void* K, const void* V, void* O,
                                         float* lse, const dplan::Plan& plan, const dplan::Geo& geo,
                                         uint32_t* err, cudaStream_t st);
cudaError_t launch_attend_decode_q4_planned(const Problem& pr, const void* Q, const uint32_t* Kq4, const float* Ks,
                                            const uint32_t* Vq4, const float* Vs, void* O, float* lse,
                                            const dplan::Plan& plan, const dplan::Geo& geo, uint32_t* err,
                                            cudaStream_t st);
cudaError_t launch_attend_decode_q8_planned(const Problem& pr, const void* Q, const int8_t* Kq, const float* Ks,
                                            const int8_t* Vq, const float* Vs, void* O, float* lse,
                                            const dplan::Plan& plan, const dplan::Geo& geo, uint32_t* err,
                                            cudaStream_t st);

}  // namespace ssa

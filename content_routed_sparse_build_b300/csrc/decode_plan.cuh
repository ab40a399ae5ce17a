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
// Merge.  The last item to finish a span of U (a per-span arrival count)
// combines that span's chunk partials in chunk order, per head, into the
// chunk-0 slot; the last span to finish a head (a per-head count) combines
// the head's span partials in rank order (ascending span, the local span
// last) into O and lse.  No warp ever waits for another: whoever finishes
// last does the work, so the merges need no barrier and cannot hang.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace dplan {

constexpr int kMaxG = 16;
constexpr int kMaxK = 64;
constexpr int kPlanWords = 512;
constexpr int64_t kPlanBits = kPlanWords * 32;  // candidates the bitmap path covers
constexpr float kLn2 = 0.6931471805599453f;

struct Plan {
  int* n_union;       // [n_grp]   |U| including the local span
  int* n_items;       // [n_grp]   work items of the group
  int* span;          // [n_grp][umax]
  uint32_t* mask;     // [n_grp][umax] heads (bit r = head kvh*g + r) that attend the span
  uint8_t* rank;      // [n_grp][umax][16] position of the span in each head's sel row (topk = local)
  int* counter;       // work-item counter of the attend kernel
  int* n_used;        // [B*Hq] used entries of each head's sel row
  int* span_done;     // [n_grp][umax] chunks of each entry of U finished
  int* head_done;     // [B*Hq] entries of U of each head merged
  float* ml;          // [B*Hq][topk+1][C][2]  (m, l) per partial, base-2 m
  float* po;          // [B*Hq][topk+1][C][D]  unnormalised partial outputs
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

// Builds group grp's plan from s.sj / s.nv with all NW warps of the CTA and
// resets the group's arrival counts (and, for group 0, the item counter).
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
  for (int p = tid; p <= nu; p += NT) plan.span_done[gbase + p] = 0;
  if (tid < g) {
    plan.rank[(size_t)(gbase + nu) * 16 + tid] = (uint8_t)k;
    plan.n_used[row0 + tid] = s.nv[tid];
    plan.head_done[row0 + tid] = 0;
  }
  if (tid == 0) {
    plan.span[gbase + nu] = (int)geo.ell;
    plan.mask[gbase + nu] = (1u << g) - 1u;
    plan.n_union[grp] = nu + 1;
    plan.n_items[grp] = nu * geo.C + local_chunks(geo);
  }
}

// ---------------------------------------------------------------- merges
// Partials are written during the attend kernel by other SMs, so they are
// read through L2 (ld.global.cg), never through a possibly stale L1 line.
template <int D>
__device__ __forceinline__ void load_part(const float* po, int64_t slot, int lane, float (&v)[D / 32]) {
  const float* src = po + slot * D + lane * (D / 32);
  if constexpr (D == 128) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = x.x; v[1] = x.y;
  }
}

// Folds partial slots slot_of(0 .. n) into (M, Ls, acc), in that order,
// with up to NB slots' loads in flight at once.
template <int D, int NB, typename F>
__device__ __forceinline__ void fold_slots(const Plan& plan, F slot_of, int n, int lane, float& M, float& Ls,
                                           float (&acc)[D / 32]) {
  constexpr int E = D / 32;
  constexpr int kMergeBatch = NB;
  const float2* ml = reinterpret_cast<const float2*>(plan.ml);
  for (int s0 = 0; s0 < n; s0 += kMergeBatch) {
    float2 mv[kMergeBatch];
    float ov[kMergeBatch][E];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (s0 + i < n) {
        const int64_t sl = slot_of(s0 + i);
        mv[i] = __ldcg(ml + sl);
        load_part<D>(plan.po, sl, lane, ov[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (s0 + i >= n || mv[i].x == -INFINITY) continue;
      const float Mn = fmaxf(M, mv[i].x);
      const float a = exp2f(M - Mn), bb = exp2f(mv[i].x - Mn);
      Ls = Ls * a + mv[i].y * bb;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = acc[e] * a + ov[i][e] * bb;
      M = Mn;
    }
  }
}

// Called by the warp whose item was the last of entry u of group grp's U
// (after a fence that made the other items' partials visible): merges the
// entry's chunks per head, then counts the entry for each of its heads and
// merges every head whose last entry this was into O and lse.  NB partials'
// loads are in flight at once.  It is a call, not inlined: it runs once per
// span, and inlined into the attend loop its registers would crowd the
// loop's.
template <int DT, int D, int NB>
__device__ __noinline__ void tail_merge(const Plan& plan, const Geo& geo, int grp, int u, int nch, uint32_t hmask,
                                        void* __restrict__ O, float* __restrict__ lse, int lane) {
  constexpr int E = D / 32;
  const int b = grp / geo.Hkv, kvh = grp - b * geo.Hkv;
  const int row0 = b * geo.Hq + kvh * geo.g;
  const int slot_idx = grp * geo.umax + u;
  const int kp1 = geo.topk + 1;
  float2* ml = reinterpret_cast<float2*>(plan.ml);
  if (nch > 1) {
    for (uint32_t hm = hmask; hm; hm &= hm - 1u) {
      const int r = __ffs(hm) - 1;
      const int rk = plan.rank[(size_t)slot_idx * 16 + r];
      const int64_t base = ((int64_t)(row0 + r) * kp1 + rk) * geo.C;
      float M = -INFINITY, Ls = 0.f, acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      fold_slots<D, NB>(plan, [&](int c) { return base + c; }, nch, lane, M, Ls, acc);
      float* dst = plan.po + base * D + lane * E;
      if constexpr (E == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
      }
      if (lane == 0) ml[base] = make_float2(M, Ls);
    }
    __threadfence();
    __syncwarp();
  }
  // count the entry for its heads; the heads it completes are merged here
  bool fin = false;
  if (lane < geo.g && ((hmask >> lane) & 1u)) {
    const int row = row0 + lane;
    const int old = atomicAdd(plan.head_done + row, 1);
    fin = old == __ldg(plan.n_used + row);  // entries per head: used spans + the local span
  }
  const uint32_t fm = __ballot_sync(0xffffffffu, fin);
  if (!fm) return;
  __threadfence();
  for (uint32_t m2 = fm; m2; m2 &= m2 - 1u) {
    const int r = __ffs(m2) - 1;
    const int64_t row = row0 + r;
    const int used = __ldg(plan.n_used + row);
    const int topk = geo.topk, C = geo.C;
    float M = -INFINITY, Ls = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    // the head's used spans in rank order (ascending span), then the local span
    fold_slots<D, NB>(plan, [&](int i) { return (row * kp1 + (i < used ? i : topk)) * C; }, used + 1, lane, M, Ls,
                  acc);
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < E; ++e) store_elem<DT>(O, row * D + lane * E + e, acc[e] * inv);
    if (lse && lane == 0) lse[row] = M * kLn2 + logf(Ls);
  }
}

}  // namespace dplan
}  // namespace ssa

namespace ssa {

// decode.cu: the plan pointers and geometry of a decode step at `pos` in the
// decode workspace ws, and the attend launch of a step whose plan an earlier
// kernel on the stream has built (O and lse written by its tail merges).
void decode_plan_args(const Problem& pr, int64_t pos, void* ws, dplan::Plan* plan, dplan::Geo* geo);
cudaError_t launch_attend_decode_planned(const Problem& pr, const void* Q, const void* K, const void* V, void* O,
                                         float* lse, const dplan::Plan& plan, const dplan::Geo& geo,
                                         uint32_t* err, cudaStream_t st);

}  // namespace ssa

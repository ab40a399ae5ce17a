// decode.cu -- decode attention: one query per head, split over the spans,
// log-sum-exp merge (16-bit K / V).
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section:
// token-level attention inside each query's chosen spans; SubQ SSA page
// (stork.ai): exact attention over the content-selected subset.  The local
// span [l*S, pos] is always attended.
//
// Three kernels (the plan itself is built by decode_plan.cuh, here or, for a
// whole decode step, inside the route kernel):
//  plan    one CTA per (b, kv-head): validates the g heads' selections and
//          builds their union U (ascending, local span last) with, per span,
//          the mask of heads that chose it and each head's rank for it.
//  attend  persistent, one CTA per SM, six independent warps.  Work items
//          are (group, span of U, chunk of CH tokens): a warp's first item
//          is fixed by its index, later ones come from an atomic counter.  Each warp runs its own two-stage ring of 32-token
//          K / V tiles loaded by TMA (128-byte swizzle, mbarrier completion),
//          each tile computed as two 16-token fragments.  The MMAs are
//          transposed so that the query group fits the n8 side of
//          mma.sync: S^T = K Q^T (tokens x heads) and O^T += V^T P^T
//          (d x heads), P^T turned into the B operand by movmatrix.  An
//          online softmax runs per head (column); at the end of an item the
//          warp writes one partial (m, l, o) per head that chose the span.
//          Every K / V byte of the union is read once.
//  merge   one CTA per (b, q-head): combines the head's partials (span
//          order, then chunk order) into O and lse.
// Softmax runs in base 2: scores are scaled by scale * log2(e).
#include "decode_plan.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

using dplan::Geo;
using dplan::Plan;
using dplan::kMaxG;
using dplan::kMaxK;

constexpr int kTile = 32;     // tokens per ring stage
constexpr int kSub = kTile / 16;  // m16 fragments per tile
constexpr int kWarps = 6;     // independent warps per CTA (6 x 2 stages x 16 KB of K / V ring)
constexpr int kThreads = kWarps * 32;
constexpr int kMaxGroups = 1024;
constexpr int kSmemLimit = 227 * 1024;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;            // 128-byte boxes per row
  static constexpr int kBox = kTile * 128;         // bytes per box
  static constexpr int kHalf = kBoxes * kBox;      // K (or V) bytes per stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr size_t kRing = (size_t)kWarps * kStages * kStage;
  static constexpr size_t kBars = (size_t)kWarps * kStages * 8;
  static constexpr size_t kMeta = (size_t)kWarps * kStages * 16;
  static constexpr size_t kMetaT = (size_t)kWarps * kStages * 16;  // the item's (t0, t1) per stage
  static constexpr size_t kFixed = 1024 + kRing + kBars + kMeta + kMetaT + (size_t)(2 * kMaxGroups + 1) * 4;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Tokens per work item, a power of two from 64 to 1024.  Per-head
// selection: about two items per warp of the GPU for the largest possible
// union (g k + 1 spans per group).  Group-shared selection, whose union is
// always k + 1 spans: the smallest size that gives at most one item per
// warp.
int chunk_tokens(const Problem& pr, int n_warps_total, bool group) {
  int c = 64;
  if (group) {
    const double work = (double)pr.B * pr.Hkv * (pr.topk + 1) * (double)pr.S;
    while (c < 1024 && (double)c * n_warps_total < work) c *= 2;
    return c;
  }
  const double work = (double)pr.B * pr.Hkv * (pr.g * pr.topk + 1) * (double)pr.S;
  const double ch = work / (2.0 * n_warps_total);
  while (c < 1024 && 2.0 * c <= ch) c *= 2;
  return c;
}

struct Layout {
  size_t n_union, n_items, span, mask, rank, counter, ml, po, q, total;
  int C, CH;
};

// The decode workspace holds the partial slots of either kind of step: the
// regions are sized for the smaller item size (more chunks per span), and a
// step's slots use its own C as the stride.
Layout layout(const Problem& pr, bool group = false) {
  Layout l;
  const int ch_head = chunk_tokens(pr, device_sm_count() * kWarps, false);
  const int ch_group = chunk_tokens(pr, device_sm_count() * kWarps, true);
  l.CH = group ? ch_group : ch_head;
  l.C = (pr.S + l.CH - 1) / l.CH;
  const int ch_min = ch_head < ch_group ? ch_head : ch_group;
  const size_t c_alloc = (size_t)((pr.S + ch_min - 1) / ch_min);
  const size_t n_grp = (size_t)pr.B * pr.Hkv;
  const size_t umax = (size_t)pr.g * pr.topk + 1;
  const size_t parts = (size_t)pr.B * pr.Hq * (pr.topk + 1) * c_alloc;
  size_t off = kWsHeader;
  l.n_union = off; off = align256(off + n_grp * 4);
  l.n_items = off; off = align256(off + n_grp * 4);
  l.span = off; off = align256(off + n_grp * umax * 4);
  l.mask = off; off = align256(off + n_grp * umax * 4);
  l.rank = off; off = align256(off + n_grp * umax * 16);
  l.counter = off; off = align256(off + 4);
  l.ml = off; off = align256(off + parts * 2 * 4);
  l.po = off; off = align256(off + parts * (size_t)pr.d * 4);
  l.q = off; off = align256(off + (size_t)pr.B * pr.Hq * pr.d * 2);
  l.total = off;
  return l;
}

// ---------------------------------------------------------------- plan
// One CTA per (b, kv-head), one warp per query head of the group: reads and
// validates the heads' sel rows, then builds the group's plan.
constexpr int kPlanThreads = kMaxG * 32;

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const int32_t* __restrict__ sel,
                                                                   Plan plan, Geo geo,
                                                                   uint32_t* __restrict__ err) {
  __shared__ dplan::PlanSmem ps;
  const int grp = blockIdx.x;
  const int b = grp / geo.Hkv, kvh = grp - b * geo.Hkv;
  const int g = geo.g, k = geo.topk, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  if (warp < g) {
    const int32_t* row = sel + (int64_t)(b * geo.Hq + kvh * g + warp) * k;
    const int j0 = lane < k ? __ldg(row + lane) : -1;
    const int j1 = lane + 32 < k ? __ldg(row + lane + 32) : -1;
    bool bad;
    const int used = warp_sel_prefix(j0, j1, lane, k, geo.ell, &bad);
    if (bad && lane == 0) flag_error(err, SSA_DEVERR_BAD_SELECTION);
    if (lane < used) ps.sj[warp][lane] = j0;
    if (lane + 32 < used) ps.sj[warp][lane + 32] = j1;
    if (lane == 0) ps.nv[warp] = used;
  }
  dplan::plan_build<kPlanThreads / 32>(grp, ps, plan, geo);
}

// ---------------------------------------------------------------- attend
// Where each warp reads the plan.  The tables stay in global memory (L1 /
// L2 hits): copying them into shared memory at kernel start delayed every
// warp's first load by several microseconds per step.
struct Tables {
  const int* gpref;       // [n_grp + 1] item prefix over groups
  const int* n_union;     // [n_grp]
  const int* span;        // [n_grp * umax]
  const uint32_t* mask;   // [n_grp * umax]
  const uint8_t* rank;    // [n_grp * umax * 16]
  const uint16_t* q;      // [B * Hq] rows of q_stride elements
  int q_stride;
};

struct Item {
  int grp, u, c, ntiles;
  int64_t t0, t1;
};

__device__ __forceinline__ void decode_item(int it, const Tables& tb, const Geo& geo, Item& x) {
  int lo = 0, hi = geo.n_grp - 1;  // last group with gpref[g] <= it
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.gpref[mid] <= it) lo = mid; else hi = mid - 1;
  }
  x.grp = lo;
  const int li = it - tb.gpref[lo];
  const int nu = tb.n_union[lo];
  if (li < (nu - 1) * geo.C) {
    x.u = li / geo.C;
    x.c = li - x.u * geo.C;
    const int64_t j = tb.span[lo * geo.umax + x.u];
    x.t0 = j * geo.S + (int64_t)x.c * geo.CH;
    x.t1 = min(x.t0 + geo.CH, (j + 1) * geo.S);
  } else {
    x.u = nu - 1;
    x.c = li - (nu - 1) * geo.C;
    x.t0 = geo.ell * geo.S + (int64_t)x.c * geo.CH;
    x.t1 = min(x.t0 + geo.CH, geo.pos + 1);
  }
  x.ntiles = (int)((x.t1 - x.t0 + kTile - 1) / kTile);
}

template <int DT, int D, int NG>
__global__ void __launch_bounds__(kThreads, 1)
    decode_attend_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const void* __restrict__ Q, Plan plan, Geo geo, uint32_t* __restrict__ err) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRing);
  int4* metas = reinterpret_cast<int4*>(bars + kWarps * C::kStages);
  int64_t* metats = reinterpret_cast<int64_t*>(metas + kWarps * C::kStages);
  int* s_gpref = reinterpret_cast<int*>(metats + 2 * kWarps * C::kStages);
  int* s_nunion = s_gpref + kMaxGroups + 1;   // the groups' union sizes, read once here

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  // ---- shared set-up: barriers, group prefix
  if (tid == 0) {
    for (int s = 0; s < kWarps * C::kStages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  Tables tb;
  tb.gpref = s_gpref;
  tb.n_union = s_nunion;
  tb.span = plan.span;
  tb.mask = plan.mask;
  tb.rank = plan.rank;
  tb.q = static_cast<const uint16_t*>(Q);
  tb.q_stride = D;
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < geo.n_grp; base += 32) {
      const int gi = base + lane;
      int v = gi < geo.n_grp ? plan.n_items[gi] : 0;
      if (gi < geo.n_grp) s_nunion[gi] = plan.n_union[gi];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (gi < geo.n_grp) s_gpref[gi + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_gpref[0] = 0;
  }
  __syncthreads();
  const int total = s_gpref[geo.n_grp];

  // ---- per-warp ring
  uint8_t* wring = ring + (size_t)warp * C::kStages * C::kStage;
  uint64_t* fb = bars + warp * C::kStages;
  int4* meta = metas + warp * C::kStages;
  int64_t* metat = metats + 2 * warp * C::kStages;

  // issue side (lane 0 drives, state kept warp-uniform)
  Item iss;
  iss.ntiles = 0;
  iss.grp = iss.u = iss.c = 0;
  iss.t0 = iss.t1 = 0;
  int iss_tile = 0;
  // Work items come from an atomic counter.  The claim for the next item is
  // made when two tiles of the current one remain to be issued, so that the
  // atomic's round trip is hidden without reserving work for long (which
  // would unbalance the tail).
  // the first item of every warp is fixed; later ones come from the counter
  const int n_static = (int)gridDim.x * (int)(blockDim.x >> 5);
  int it_next = (int)blockIdx.x * (int)(blockDim.x >> 5) + warp, it_claim = 0;
  bool have_next = true, claim_issued = false;
  bool exhausted = false;

  const uint64_t pol_stream = ptx::policy_evict_first();  // K / V are read once per step
  // Loads the next tile into `stage`; returns false when no work is left.
  auto issue = [&](int stage) -> bool {
    if (iss_tile == iss.ntiles) {
      if (!have_next) it_next = __shfl_sync(0xffffffffu, it_claim, 0);
      if (it_next >= total) {
        exhausted = true;
        return false;
      }
      decode_item(it_next, tb, geo, iss);
      iss_tile = 0;
      have_next = false;
      claim_issued = false;
    }
    if (lane == 0) {
      meta[stage] = make_int4(iss.grp, iss.u, iss.c, iss_tile);
      metat[2 * stage] = iss.t0;
      metat[2 * stage + 1] = iss.t1;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ptx::mbar_arrive_expect_tx(&fb[stage], C::kStage);
      uint8_t* dK = wring + (size_t)stage * C::kStage;
      uint8_t* dV = dK + C::kHalf;
      const int y = (int)(iss.t0 + (int64_t)iss_tile * kTile);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        ptx::tma_load_3d_hint(dK + bx * C::kBox, &tmK, &fb[stage], bx * 64, y, iss.grp, pol_stream);
        ptx::tma_load_3d_hint(dV + bx * C::kBox, &tmV, &fb[stage], bx * 64, y, iss.grp, pol_stream);
      }
    }
    ++iss_tile;
    if (!claim_issued && iss.ntiles - iss_tile <= 2) {
      if (lane == 0) it_claim = atomicAdd(plan.counter, 1) + n_static;
      claim_issued = true;
    }
    return true;
  };

  int inflight = 0;
#pragma unroll 1
  for (int s = 0; s < C::kStages; ++s) {
    if (exhausted || !issue(s)) break;
    ++inflight;
  }

  // Consumer state.  NG groups of 8 heads; lane holds, per group, heads
  // 2*q4 and 2*q4+1 of the group (columns of S^T and O^T) and tokens / d
  // rows r8 and r8 + 8 of each 16-row fragment.
  const int q4 = lane & 3, r8 = lane >> 2;
  const int mi = lane >> 3, rr = lane & 7;
  uint32_t qb[NG][D / 16][2];
  float o[NG][D / 16][4];
  float m[NG][2], l[NG][2];
  uint32_t hmask = 0u;          // the item's heads, and this thread's heads' ranks
  int rk[NG][2];
  Item cur;
  cur.grp = cur.u = cur.c = cur.ntiles = 0;
  cur.t0 = cur.t1 = 0;
  int stage = 0;
  uint32_t phase = 0;
#pragma unroll 1
  while (inflight > 0) {
    if (!ptx::mbar_wait(&fb[stage], phase)) {
      if (lane == 0) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const int4 mt = meta[stage];
    if (mt.w == 0) {
      cur.grp = mt.x;
      cur.u = mt.y;
      cur.c = mt.z;
      cur.t0 = metat[2 * stage];
      cur.t1 = metat[2 * stage + 1];
      cur.ntiles = (int)((cur.t1 - cur.t0 + kTile - 1) / kTile);
      {
        // the end-of-item tables, read now so that their latency overlaps
        const int slot_idx = cur.grp * geo.umax + cur.u;
        hmask = tb.mask[slot_idx];
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = ng * 8 + 2 * q4 + i;
            rk[ng][i] = r < geo.g ? tb.rank[(size_t)slot_idx * 16 + r] : 0;
          }
      }
      // B operand of S^T = K Q^T: thread holds Q[head r8][d pair] per k-step
      const int b = cur.grp / geo.Hkv, kvh = cur.grp - b * geo.Hkv;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        const int h = ng * 8 + r8;
        const bool ok = h < geo.g;
        const uint32_t* qr =
            reinterpret_cast<const uint32_t*>(tb.q + (int64_t)(b * geo.Hq + kvh * geo.g + h) * tb.q_stride);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          qb[ng][kk][0] = ok ? qr[kk * 8 + q4] : 0u;
          qb[ng][kk][1] = ok ? qr[kk * 8 + 4 + q4] : 0u;
        }
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) o[ng][mt2][0] = o[ng][mt2][1] = o[ng][mt2][2] = o[ng][mt2][3] = 0.f;
        m[ng][0] = m[ng][1] = -INFINITY;
        l[ng][0] = l[ng][1] = 0.f;
      }
    }
    const uint32_t aK = ptx::smem_u32(wring + (size_t)stage * C::kStage);
    const uint32_t aV = aK + C::kHalf;

    // S^T (kTile tokens x 8 heads per group), one m16 fragment per 16 tokens:
    // A = K tile rows, B = Q^T
    float s[NG][kSub][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int t = 0; t < kSub; ++t) s[ng][t][0] = s[ng][t][1] = s[ng][t][2] = s[ng][t][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const int row = t * 16 + (mi & 1) * 8 + rr;
        const int chunk = 2 * (kk & 3) + (mi >> 1);
        uint32_t a[4];
        ptx::ldsm_x4(aK + (kk >> 2) * C::kBox + ptx::sw128(row, chunk), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) ptx::mma16816<DT>(s[ng][t], a, qb[ng][kk][0], qb[ng][kk][1]);
      }
    }
    // mask tokens outside the item (partial tiles only)
    const int64_t tbase = cur.t0 + (int64_t)mt.w * kTile;
    if (tbase + kTile > cur.t1) {
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const bool v0 = tbase + t * 16 + r8 < cur.t1, v1 = tbase + t * 16 + r8 + 8 < cur.t1;
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          if (!v0) s[ng][t][0] = s[ng][t][1] = -INFINITY;
          if (!v1) s[ng][t][2] = s[ng][t][3] = -INFINITY;
        }
      }
    }
    // online softmax per head (column): reduce over the tile's tokens = the
    // lane's rows of every fragment and the eight lanes sharing q4
    const float c = geo.scale_log2e;
    uint32_t pb[NG][kSub][2];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      float mx[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float v = fmaxf(s[ng][0][i], s[ng][0][i + 2]);
#pragma unroll
        for (int t = 1; t < kSub; ++t) v = fmaxf(v, fmaxf(s[ng][t][i], s[ng][t][i + 2]));
        v *= c;
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mx[i] = fmaxf(m[ng][i], v);
      }
      float nb[2], alpha[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float bse = mx[i] == -INFINITY ? 0.f : mx[i];
        nb[i] = -bse;
        alpha[i] = exp2f(m[ng][i] - bse);
        m[ng][i] = mx[i];
      }
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const float p0 = ptx::ex2(fmaf(s[ng][t][0], c, nb[0]));
        const float p1 = ptx::ex2(fmaf(s[ng][t][1], c, nb[1]));
        const float p2 = ptx::ex2(fmaf(s[ng][t][2], c, nb[0]));
        const float p3 = ptx::ex2(fmaf(s[ng][t][3], c, nb[1]));
        ls0 += p0 + p2;
        ls1 += p1 + p3;
        // P^T rows (tokens) -> P rows (heads): the B operand of O^T += V^T P^T
        pb[ng][t][0] = ptx::movmatrix_trans(ptx::pack2<DT>(p0, p1));
        pb[ng][t][1] = ptx::movmatrix_trans(ptx::pack2<DT>(p2, p3));
      }
      l[ng][0] = l[ng][0] * alpha[0] + ls0;
      l[ng][1] = l[ng][1] * alpha[1] + ls1;
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          o[ng][mt2][0] *= alpha[0];
          o[ng][mt2][1] *= alpha[1];
          o[ng][mt2][2] *= alpha[0];
          o[ng][mt2][3] *= alpha[1];
        }
      }
    }
    // O^T (d x heads) += V^T (d x kTile tokens) P^T, one k16 step per fragment
#pragma unroll
    for (int mt2 = 0; mt2 < D / 16; ++mt2) {
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const int row = t * 16 + (mi >> 1) * 8 + rr;
        const int chunk = 2 * mt2 + (mi & 1);
        uint32_t a[4];
        ptx::ldsm_x4_t(aV + (chunk >> 3) * C::kBox + ptx::sw128(row, chunk & 7), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) ptx::mma16816<DT>(o[ng][mt2], a, pb[ng][t][0], pb[ng][t][1]);
      }
    }
    __syncwarp();
    --inflight;
    const bool last = mt.w == cur.ntiles - 1;
    if (!exhausted && issue(stage)) ++inflight;
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (!last) continue;

    // ---- item epilogue: one partial per head that attends this span
    const int b = cur.grp / geo.Hkv, kvh = cur.grp - b * geo.Hkv;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float lt = l[ng][i];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int r = ng * 8 + 2 * q4 + i;  // head within the group
        if (r >= geo.g || !((hmask >> r) & 1u)) continue;
        const int64_t slot =
            ((int64_t)(b * geo.Hq + kvh * geo.g + r) * (geo.topk + 1) + rk[ng][i]) * geo.C + cur.c;
        float* dst = plan.po + slot * D + r8;
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          dst[mt2 * 16] = o[ng][mt2][i];
          dst[mt2 * 16 + 8] = o[ng][mt2][i + 2];
        }
        if (r8 == 0) *reinterpret_cast<float2*>(plan.ml + slot * 2) = make_float2(m[ng][i], lt);
      }
    }
  }
}

// ---------------------------------------------------------------- attend, 8-bit cache
// The same work items, plan and merge as the 16-bit kernel, over the 8-bit
// cache of quant.cu (d = 128).  Each ring stage holds one 32-token tile: the
// K rows (TMA, 128-byte swizzle), the d-major V tile and the tile's K and V
// scales (bulk copies).  Tiles are 32-token aligned; tokens of a tile
// outside the item are masked.  The MMAs run in fp16 on exact values: each
// code q enters as the fp16 subnormal (q + 128) 2^-24 (an XOR and a byte
// permute, no conversion arithmetic), and Q is rounded to fp16 once per kv
// group.  The factor and the offset are folded out:
//   S^T = ks * (2^24 (Kq' Q^T) - 128 sum_d Q)         (tokens x heads)
//   O^T += 2^24 (Vq'^T (vs P)^T - 128 * 1^T (vs P)^T), l += sum of P
// where the last term is one more MMA against a fragment of 2^-24s, so it
// sums the same rounded (vs P) values the main MMA used.
// The k order of the K fragments is permuted: thread quad c reads 8
// consecutive bytes d = 32 J + 8 c .. + 7 of a row, bytes 0-3 feeding k-step
// 2 J and bytes 4-7 k-step 2 J + 1; Q's fragments are built with the same
// d-to-k map, so every product still pairs K[t][d] with Q[h][d].
namespace q8 {
// Twelve warps of two stages: an 8-bit tile is half the bytes of a 16-bit
// one, so the same ring holds twice the warps, which hide the conversion
// and MMA latency of each tile.
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kKBytes = kTile * 128;   // 32 rows of 128 int8
constexpr int kVBytes = kTile * 128;   // 128 d-rows of 32 tokens
constexpr int kSBytes = 2 * kTile * 4; // ks then vs
constexpr size_t kRingK = (size_t)kWarps * kStages * kKBytes;
constexpr size_t kRingV = (size_t)kWarps * kStages * kVBytes;
constexpr size_t kRingS = (size_t)kWarps * kStages * kSBytes;
constexpr size_t kBars = (size_t)kWarps * kStages * 8;
constexpr size_t kMeta = (size_t)kWarps * kStages * 16;
constexpr size_t kMetaT = (size_t)kWarps * kStages * 16;
constexpr size_t kFixed =
    1024 + kRingK + kRingV + kRingS + kBars + kMeta + kMetaT + (size_t)(2 * kMaxGroups + 1) * 4;
static_assert(kFixed <= (size_t)kSmemLimit, "8-bit ring does not fit in shared memory");

// First 32-aligned tile start and tile count of tokens [t0, t1).
__device__ __forceinline__ int64_t tile_base(int64_t t0) { return t0 & ~(int64_t)(kTile - 1); }
__device__ __forceinline__ int tiles(int64_t t0, int64_t t1) {
  return (int)((t1 - tile_base(t0) + kTile - 1) / kTile);
}
}  // namespace q8

template <int DT, int NG>
__global__ void __launch_bounds__(q8::kThreads, 1)
    decode_attend_q8_kernel(const __grid_constant__ CUtensorMap tmK, const int8_t* __restrict__ Vq,
                            const float* __restrict__ Ks, const float* __restrict__ Vs, int64_t L_cap,
                            const void* __restrict__ Q, Plan plan, Geo geo, uint32_t* __restrict__ err) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ringK = smem;
  uint8_t* ringV = ringK + q8::kRingK;
  uint8_t* ringS = ringV + q8::kRingV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ringS + q8::kRingS);
  int4* metas = reinterpret_cast<int4*>(bars + q8::kWarps * q8::kStages);
  int64_t* metats = reinterpret_cast<int64_t*>(metas + q8::kWarps * q8::kStages);
  int* s_gpref = reinterpret_cast<int*>(metats + 2 * q8::kWarps * q8::kStages);
  int* s_nunion = s_gpref + kMaxGroups + 1;   // the groups' union sizes, read once here

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < q8::kWarps * q8::kStages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmK);
  }
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  Tables tb;
  tb.gpref = s_gpref;
  tb.n_union = s_nunion;
  tb.span = plan.span;
  tb.mask = plan.mask;
  tb.rank = plan.rank;
  tb.q = static_cast<const uint16_t*>(Q);
  tb.q_stride = D;
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < geo.n_grp; base += 32) {
      const int gi = base + lane;
      int v = gi < geo.n_grp ? plan.n_items[gi] : 0;
      if (gi < geo.n_grp) s_nunion[gi] = plan.n_union[gi];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (gi < geo.n_grp) s_gpref[gi + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_gpref[0] = 0;
  }
  __syncthreads();
  const int total = s_gpref[geo.n_grp];

  uint8_t* wK = ringK + (size_t)warp * q8::kStages * q8::kKBytes;
  uint8_t* wV = ringV + (size_t)warp * q8::kStages * q8::kVBytes;
  uint8_t* wS = ringS + (size_t)warp * q8::kStages * q8::kSBytes;
  uint64_t* fb = bars + warp * q8::kStages;
  int4* meta = metas + warp * q8::kStages;
  int64_t* metat = metats + 2 * warp * q8::kStages;
  const int64_t tiles_per_head = L_cap / kTile;

  Item iss;
  iss.ntiles = 0;
  iss.grp = iss.u = iss.c = 0;
  iss.t0 = iss.t1 = 0;
  int iss_tile = 0;
  // the first item of every warp is fixed; later ones come from the counter
  const int n_static = (int)gridDim.x * (int)(blockDim.x >> 5);
  // the first item of every warp is fixed; later ones come from the counter,
  // which is not touched at all when the fixed items cover the step
  const bool may_claim = total > n_static;
  int it_next = (int)blockIdx.x * (int)(blockDim.x >> 5) + warp, it_claim = total;
  bool have_next = true, claim_issued = false;
  bool exhausted = false;
  const uint64_t pol_stream = ptx::policy_evict_first();  // K rows are read once per step

  auto issue = [&](int stage) -> bool {
    if (iss_tile == iss.ntiles) {
      if (!have_next) it_next = __shfl_sync(0xffffffffu, it_claim, 0);
      if (it_next >= total) {
        exhausted = true;
        return false;
      }
      decode_item(it_next, tb, geo, iss);
      iss.ntiles = q8::tiles(iss.t0, iss.t1);
      iss_tile = 0;
      have_next = false;
      claim_issued = false;
    }
    if (lane == 0) {
      meta[stage] = make_int4(iss.grp, iss.u, iss.c, iss_tile);
      metat[2 * stage] = iss.t0;
      metat[2 * stage + 1] = iss.t1;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ptx::mbar_arrive_expect_tx(&fb[stage], q8::kKBytes + q8::kVBytes + q8::kSBytes);
      const int64_t y = q8::tile_base(iss.t0) + (int64_t)iss_tile * kTile;
      uint8_t* dS = wS + stage * q8::kSBytes;
      ptx::tma_load_3d_hint(wK + stage * q8::kKBytes, &tmK, &fb[stage], 0, (int)y, iss.grp, pol_stream);
      ptx::bulk_load(wV + stage * q8::kVBytes, Vq + ((int64_t)iss.grp * tiles_per_head + y / kTile) * (D * kTile),
                     q8::kVBytes, &fb[stage]);
      ptx::bulk_load(dS, Ks + (int64_t)iss.grp * L_cap + y, kTile * 4, &fb[stage]);
      ptx::bulk_load(dS + kTile * 4, Vs + (int64_t)iss.grp * L_cap + y, kTile * 4, &fb[stage]);
    }
    ++iss_tile;
    if (may_claim && !claim_issued && iss.ntiles - iss_tile <= 2) {
      if (lane == 0) it_claim = atomicAdd(plan.counter, 1) + n_static;
      claim_issued = true;
    }
    return true;
  };

  int inflight = 0, first_grp = -1;
#pragma unroll 1
  for (int s = 0; s < q8::kStages; ++s) {
    if (exhausted || !issue(s)) break;
    if (s == 0) first_grp = iss.grp;
    ++inflight;
  }

  const int q4 = lane & 3, r8 = lane >> 2;
  // Q of head r8 (+8 ng), d = 32 J + 8 q4 .. + 7, fp16 pairs, and 128 times
  // the sum of each of this thread's two heads' rounded Q.  They depend on
  // the kv group only: loaded for the first item while its tiles are in
  // flight, and again only when an item of another group starts.
  uint32_t qf[NG][D / 32][4];
  float qs128[NG][2];
  int q_grp = -1;
  auto load_q = [&](int grp) {
    const int b = grp / geo.Hkv, kvh = grp - b * geo.Hkv;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int h = ng * 8 + r8;
      const bool ok = h < geo.g;
      const uint16_t* qr = tb.q + (int64_t)(b * geo.Hq + kvh * geo.g + h) * tb.q_stride;
      // a thread's dimensions 32 J + 8 q4 .. + 7 are 16 contiguous bytes
      uint4 qv[D / 32];
#pragma unroll
      for (int J = 0; J < D / 32; ++J)
        qv[J] = ok ? *reinterpret_cast<const uint4*>(qr + 32 * J + 8 * q4) : make_uint4(0u, 0u, 0u, 0u);
      float qsum = 0.f;
#pragma unroll
      for (int J = 0; J < D / 32; ++J) {
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          const uint32_t w = pr == 0 ? qv[J].x : pr == 1 ? qv[J].y : pr == 2 ? qv[J].z : qv[J].w;
          uint32_t v = w;
          if constexpr (DT == DT_BF16) {
            const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
            v = ptx::pack2<DT_F16>(lo, hi);
          }
          const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&v));
          qsum += r.x + r.y;
          qf[ng][J][pr] = v;
        }
      }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
      // lanes 4 h .. 4 h + 3 hold head h's sum; this thread's columns are
      // heads 2 q4 and 2 q4 + 1
      qs128[ng][0] = 128.f * __shfl_sync(0xffffffffu, qsum, 8 * q4);
      qs128[ng][1] = 128.f * __shfl_sync(0xffffffffu, qsum, 8 * q4 + 4);
    }
    q_grp = grp;
  };
  if (first_grp >= 0) load_q(first_grp);

  float o[NG][D / 16][4];
  float oc[NG][4];              // sum_t (P vs)'_t 2^-24 of heads 2 q4, 2 q4 + 1
  float m[NG][2], l[NG][2];
  constexpr float kTwo24 = 16777216.f;
  const float2 kTwo24x2 = make_float2(kTwo24, kTwo24);
  uint32_t hmask = 0u;          // the item's heads, and this thread's heads' ranks
  int rk[NG][2];
  Item cur;
  cur.grp = cur.u = cur.c = cur.ntiles = 0;
  cur.t0 = cur.t1 = 0;
  int stage = 0;
  uint32_t phase = 0;
#pragma unroll 1
  while (inflight > 0) {
    if (!ptx::mbar_wait(&fb[stage], phase)) {
      if (lane == 0) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const int4 mt = meta[stage];
    if (mt.w == 0) {
      cur.grp = mt.x;
      cur.u = mt.y;
      cur.c = mt.z;
      cur.t0 = metat[2 * stage];
      cur.t1 = metat[2 * stage + 1];
      cur.ntiles = q8::tiles(cur.t0, cur.t1);
      {
        // the end-of-item tables, read now so that their latency overlaps
        const int slot_idx = cur.grp * geo.umax + cur.u;
        hmask = tb.mask[slot_idx];
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = ng * 8 + 2 * q4 + i;
            rk[ng][i] = r < geo.g ? tb.rank[(size_t)slot_idx * 16 + r] : 0;
          }
      }
      if (cur.grp != q_grp) load_q(cur.grp);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) o[ng][mt2][0] = o[ng][mt2][1] = o[ng][mt2][2] = o[ng][mt2][3] = 0.f;
        oc[ng][0] = oc[ng][1] = oc[ng][2] = oc[ng][3] = 0.f;
        m[ng][0] = m[ng][1] = -INFINITY;
        l[ng][0] = l[ng][1] = 0.f;
      }
    }
    const uint32_t aK = ptx::smem_u32(wK + stage * q8::kKBytes);
    const uint32_t aV = ptx::smem_u32(wV + stage * q8::kVBytes);
    const float* sks = reinterpret_cast<const float*>(wS + stage * q8::kSBytes);
    const float* svs = sks + kTile;

    // S^T = Kq Q^T per 16-token fragment t
    float s[NG][kSub][4], s2[NG][kSub][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int t = 0; t < kSub; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[ng][t][i] = s2[ng][t][i] = 0.f;
#pragma unroll
    for (int J = 0; J < D / 32; ++J) {
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const int ra = t * 16 + r8, rb = ra + 8;
        const int chunk = 2 * J + (q4 >> 1);
        const uint2 wa = ptx::lds64(aK + ptx::sw128(ra, chunk) + 8 * (q4 & 1));
        const uint2 wb = ptx::lds64(aK + ptx::sw128(rb, chunk) + 8 * (q4 & 1));
        uint32_t a0[4], a1[4];
        ptx::s8x4_to_f16x2_sub(wa.x, a0[0], a0[2]);
        ptx::s8x4_to_f16x2_sub(wb.x, a0[1], a0[3]);
        ptx::s8x4_to_f16x2_sub(wa.y, a1[0], a1[2]);
        ptx::s8x4_to_f16x2_sub(wb.y, a1[1], a1[3]);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          ptx::mma16816<DT_F16>(s[ng][t], a0, qf[ng][J][0], qf[ng][J][1]);
          ptx::mma16816<DT_F16>(s2[ng][t], a1, qf[ng][J][2], qf[ng][J][3]);
        }
      }
    }
    // the odd k-steps accumulated apart (two independent MMA chains per fragment)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int t = 0; t < kSub; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[ng][t][i] += s2[ng][t][i];
    // rows (tokens) r8 and r8 + 8 of each fragment: K / V scales, validity
    const int64_t tbase = q8::tile_base(cur.t0) + (int64_t)mt.w * kTile;
    float ksc[kSub][2], vsc[kSub][2];
    bool valid[kSub][2];
#pragma unroll
    for (int t = 0; t < kSub; ++t)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = t * 16 + r8 + 8 * i;
        const int64_t tok = tbase + row;
        valid[t][i] = tok >= cur.t0 && tok < cur.t1;
        ksc[t][i] = sks[row];
        vsc[t][i] = svs[row];
      }
    // the MMA summed q'_d (q_d + 128) 2^-24 over d: the score is
    // 2^24 acc - 128 sum_d q'_d, times the token's K scale
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const float2 nq = make_float2(-qs128[ng][0], -qs128[ng][1]);
        const float2 a = __fmul2_rn(__ffma2_rn(make_float2(s[ng][t][0], s[ng][t][1]), kTwo24x2, nq),
                                    make_float2(ksc[t][0], ksc[t][0]));
        const float2 b = __fmul2_rn(__ffma2_rn(make_float2(s[ng][t][2], s[ng][t][3]), kTwo24x2, nq),
                                    make_float2(ksc[t][1], ksc[t][1]));
        s[ng][t][0] = valid[t][0] ? a.x : -INFINITY;
        s[ng][t][1] = valid[t][0] ? a.y : -INFINITY;
        s[ng][t][2] = valid[t][1] ? b.x : -INFINITY;
        s[ng][t][3] = valid[t][1] ? b.y : -INFINITY;
      }
    const float c = geo.scale_log2e;
    uint32_t pb[NG][kSub][2];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      float mx[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float v = fmaxf(s[ng][0][i], s[ng][0][i + 2]);
#pragma unroll
        for (int t = 1; t < kSub; ++t) v = fmaxf(v, fmaxf(s[ng][t][i], s[ng][t][i + 2]));
        v *= c;
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mx[i] = fmaxf(m[ng][i], v);
      }
      float nb[2], alpha[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float bse = mx[i] == -INFINITY ? 0.f : mx[i];
        nb[i] = -bse;
        alpha[i] = exp2f(m[ng][i] - bse);
        m[ng][i] = mx[i];
      }
      // the two rows of a fragment (heads 2 c and 2 c + 1) side by side in
      // packed fp32 operations, each lane rounded as its scalar form
      const float2 c2 = make_float2(c, c), nb2 = make_float2(nb[0], nb[1]);
      float2 ls = make_float2(0.f, 0.f);
#pragma unroll
      for (int t = 0; t < kSub; ++t) {
        const float2 e01 = __ffma2_rn(make_float2(s[ng][t][0], s[ng][t][1]), c2, nb2);
        const float2 e23 = __ffma2_rn(make_float2(s[ng][t][2], s[ng][t][3]), c2, nb2);
        const float2 p01 = make_float2(ptx::ex2(e01.x), ptx::ex2(e01.y));
        const float2 p23 = make_float2(ptx::ex2(e23.x), ptx::ex2(e23.y));
        ls = __fadd2_rn(ls, __fadd2_rn(p01, p23));
        // the V scale of each token weights its P (0 for masked tokens,
        // whose scale slot may hold anything)
        const float v0 = valid[t][0] ? vsc[t][0] : 0.f, v1 = valid[t][1] ? vsc[t][1] : 0.f;
        const float2 w01 = __fmul2_rn(p01, make_float2(v0, v0));
        const float2 w23 = __fmul2_rn(p23, make_float2(v1, v1));
        pb[ng][t][0] = ptx::movmatrix_trans(ptx::pack2<DT_F16>(w01.x, w01.y));
        pb[ng][t][1] = ptx::movmatrix_trans(ptx::pack2<DT_F16>(w23.x, w23.y));
      }
      l[ng][0] = l[ng][0] * alpha[0] + ls.x;
      l[ng][1] = l[ng][1] * alpha[1] + ls.y;
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
        const float2 al = make_float2(alpha[0], alpha[1]);
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          const float2 x = __fmul2_rn(make_float2(o[ng][mt2][0], o[ng][mt2][1]), al);
          const float2 y = __fmul2_rn(make_float2(o[ng][mt2][2], o[ng][mt2][3]), al);
          o[ng][mt2][0] = x.x;
          o[ng][mt2][1] = x.y;
          o[ng][mt2][2] = y.x;
          o[ng][mt2][3] = y.y;
        }
        const float2 x = __fmul2_rn(make_float2(oc[ng][0], oc[ng][1]), al);
        const float2 y = __fmul2_rn(make_float2(oc[ng][2], oc[ng][3]), al);
        oc[ng][0] = x.x;
        oc[ng][1] = x.y;
        oc[ng][2] = y.x;
        oc[ng][3] = y.y;
      }
    }
    // O^T += Vq^T (vs P)^T: d-rows r8 and r8 + 8 of each m16 slice, one
    // 8-byte load per row covering both 16-token fragments
#pragma unroll
    for (int mt2 = 0; mt2 < D / 16; ++mt2) {
      const uint2 va = ptx::lds64(aV + (mt2 * 16 + r8) * 32 + 8 * q4);
      const uint2 vb = ptx::lds64(aV + (mt2 * 16 + r8 + 8) * 32 + 8 * q4);
      uint32_t a0[4], a1[4];
      ptx::s8x4_to_f16x2_sub(va.x, a0[0], a0[2]);
      ptx::s8x4_to_f16x2_sub(vb.x, a0[1], a0[3]);
      ptx::s8x4_to_f16x2_sub(va.y, a1[0], a1[2]);
      ptx::s8x4_to_f16x2_sub(vb.y, a1[1], a1[3]);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        ptx::mma16816<DT_F16>(o[ng][mt2], a0, pb[ng][0][0], pb[ng][0][1]);
        ptx::mma16816<DT_F16>(o[ng][mt2], a1, pb[ng][1][0], pb[ng][1][1]);
      }
    }
    {
      // a row of 1s at the fields' scale 2^-24: sum_t (P vs)'_t 2^-24 per head
      const uint32_t one[4] = {0x00010001u, 0x00010001u, 0x00010001u, 0x00010001u};
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        ptx::mma16816<DT_F16>(oc[ng], one, pb[ng][0][0], pb[ng][0][1]);
        ptx::mma16816<DT_F16>(oc[ng], one, pb[ng][1][0], pb[ng][1][1]);
      }
    }
    __syncwarp();
    --inflight;
    const bool last = mt.w == cur.ntiles - 1;
    if (!exhausted && issue(stage)) ++inflight;
    if (++stage == q8::kStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (!last) continue;

    const int b = cur.grp / geo.Hkv, kvh = cur.grp - b * geo.Hkv;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float lt = l[ng][i];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int r = ng * 8 + 2 * q4 + i;
        if (r >= geo.g || !((hmask >> r) & 1u)) continue;
        const int64_t slot =
            ((int64_t)(b * geo.Hq + kvh * geo.g + r) * (geo.topk + 1) + rk[ng][i]) * geo.C + cur.c;
        float* dst = plan.po + slot * D + r8;
        // 2^24 (acc - 128 * sum_t (P vs)' 2^-24): the codes' offset removed
        const float corr = -128.f * kTwo24 * oc[ng][i];
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          dst[mt2 * 16] = fmaf(o[ng][mt2][i], kTwo24, corr);
          dst[mt2 * 16 + 8] = fmaf(o[ng][mt2][i + 2], kTwo24, corr);
        }
        if (r8 == 0) *reinterpret_cast<float2*>(plan.ml + slot * 2) = make_float2(m[ng][i], lt);
      }
    }
  }
}

// ---------------------------------------------------------------- attend, 4-bit cache
// The same work items, plan and merge over the 4-bit cache of quant.cu
// (d = 128).  A ring stage holds 64 tokens: two consecutive 32-token blocks
// of K (4 KB) and of V (4 KB), both laid out for the fragments (quant.cu),
// and their K and V scales, all by bulk copies; four independent 16-token
// fragments per stage give each warp four S chains and amortise the
// per-stage wait, issue and max reduction over 64 tokens.  A thread reads one 32-bit word per
// fragment row and masks its eight nibbles n = code + 8 into four fp16 pairs
// of subnormals, n * 2^-24 or (second and fourth pair) 16 n * 2^-24, with no
// arithmetic; the MMAs then see exact values and the rest is folded:
//   K: Q's dimensions that meet a 16 n field are taken at Q / 16, so every
//      product is q' n 2^-24 with q' the Q value the MMA used; the score is
//      2^24 acc - 8 sum_d q'_d, the sum taken once per item and head;
//   V: the tokens stored as 16 n fields (those with bit 3 of the tile index
//      set) carry P * vs / 16, and one more MMA against a constant fragment
//      of 1s at the same scales accumulates sum_t (P vs)' 2^-24 per head, so
//      the output is 2^24 (acc - 8 * that), all of it in the same rounded
//      products the MMA summed.
// The dimension and token orders of the words are those of the 8-bit
// kernel's fragments, so Q's fragments and the softmax are the 8-bit kernel's.
namespace q4 {
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kT = 64;                 // tokens per ring stage
constexpr int kSubT = kT / 16;         // m16 fragments per stage
constexpr int kBlk = 32;               // tokens per stored block
constexpr int kBlkBytes = 2048;        // 32 tokens x 128 nibbles, of K or of V
constexpr int kKBytes = 2 * kBlkBytes;
constexpr int kVBytes = 2 * kBlkBytes;
constexpr int kSBytes = 2 * kT * 4;    // ks then vs
constexpr size_t kRingK = (size_t)kWarps * kStages * kKBytes;
constexpr size_t kRingV = (size_t)kWarps * kStages * kVBytes;
constexpr size_t kRingS = (size_t)kWarps * kStages * kSBytes;
constexpr size_t kBars = (size_t)kWarps * kStages * 8;
constexpr size_t kMeta = (size_t)kWarps * kStages * 16;   // (grp, u, c, tile) per stage
constexpr size_t kMetaT = (size_t)kWarps * kStages * 16;  // the item's (t0, t1) per stage
constexpr size_t kFixed =
    1024 + kRingK + kRingV + kRingS + kBars + kMeta + kMetaT + (size_t)(2 * kMaxGroups + 1) * 4;
static_assert(kFixed <= (size_t)kSmemLimit, "4-bit ring does not fit in shared memory");

__device__ __forceinline__ int64_t tile_base(int64_t t0) { return t0 & ~(int64_t)(kT - 1); }
__device__ __forceinline__ int tiles(int64_t t0, int64_t t1) {
  return (int)((t1 - tile_base(t0) + kT - 1) / kT);
}
}  // namespace q4

template <int DT, int NG>
__global__ void __launch_bounds__(q4::kThreads, 1)
    decode_attend_q4_kernel(const uint32_t* __restrict__ Kq4, const uint32_t* __restrict__ Vq4,
                            const float* __restrict__ Ks, const float* __restrict__ Vs, int64_t L_cap,
                            const void* __restrict__ Q, Plan plan, Geo geo, uint32_t* __restrict__ err) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ringK = smem;
  uint8_t* ringV = ringK + q4::kRingK;
  uint8_t* ringS = ringV + q4::kRingV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ringS + q4::kRingS);
  int4* metas = reinterpret_cast<int4*>(bars + q4::kWarps * q4::kStages);
  int64_t* metats = reinterpret_cast<int64_t*>(metas + q4::kWarps * q4::kStages);
  int* s_gpref = reinterpret_cast<int*>(metats + 2 * q4::kWarps * q4::kStages);
  int* s_nunion = s_gpref + kMaxGroups + 1;   // the groups' union sizes, read once here

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < q4::kWarps * q4::kStages; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
  }
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  Tables tb;
  tb.gpref = s_gpref;
  tb.n_union = s_nunion;
  tb.span = plan.span;
  tb.mask = plan.mask;
  tb.rank = plan.rank;
  tb.q = static_cast<const uint16_t*>(Q);
  tb.q_stride = D;
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < geo.n_grp; base += 32) {
      const int gi = base + lane;
      int v = gi < geo.n_grp ? plan.n_items[gi] : 0;
      if (gi < geo.n_grp) s_nunion[gi] = plan.n_union[gi];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (gi < geo.n_grp) s_gpref[gi + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_gpref[0] = 0;
  }
  __syncthreads();
  const int total = s_gpref[geo.n_grp];

  uint8_t* wK = ringK + (size_t)warp * q4::kStages * q4::kKBytes;
  uint8_t* wV = ringV + (size_t)warp * q4::kStages * q4::kVBytes;
  uint8_t* wS = ringS + (size_t)warp * q4::kStages * q4::kSBytes;
  uint64_t* fb = bars + warp * q4::kStages;
  int4* meta = metas + warp * q4::kStages;
  int64_t* metat = metats + 2 * warp * q4::kStages;
  const int64_t blocks_per_head = L_cap / q4::kBlk;

  Item iss;
  iss.ntiles = 0;
  iss.grp = iss.u = iss.c = 0;
  iss.t0 = iss.t1 = 0;
  int iss_tile = 0;
  // the first item of every warp is fixed; later ones come from the counter,
  // which is not touched at all when the fixed items cover the step
  const int n_static = (int)gridDim.x * (int)(blockDim.x >> 5);
  const bool may_claim = total > n_static;
  int it_next = (int)blockIdx.x * (int)(blockDim.x >> 5) + warp, it_claim = total;
  bool have_next = true, claim_issued = false;
  bool exhausted = false;

  auto issue = [&](int stage) -> bool {
    if (iss_tile == iss.ntiles) {
      if (!have_next) it_next = __shfl_sync(0xffffffffu, it_claim, 0);
      if (it_next >= total) {
        exhausted = true;
        return false;
      }
      decode_item(it_next, tb, geo, iss);
      iss.ntiles = q4::tiles(iss.t0, iss.t1);
      iss_tile = 0;
      have_next = false;
      claim_issued = false;
    }
    if (lane == 0) {
      meta[stage] = make_int4(iss.grp, iss.u, iss.c, iss_tile);
      metat[2 * stage] = iss.t0;
      metat[2 * stage + 1] = iss.t1;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const int64_t y = q4::tile_base(iss.t0) + (int64_t)iss_tile * q4::kT;
      // the head's last 32-token block may stand alone (L_cap is a multiple
      // of 32, not of 64); the stage's other half is then never unmasked
      const uint32_t nb = y + q4::kT <= L_cap ? 2u : 1u;
      ptx::mbar_arrive_expect_tx(&fb[stage], nb * (2 * q4::kBlkBytes + 2 * q4::kBlk * 4));
      uint8_t* dS = wS + stage * q4::kSBytes;
      const int64_t blk = ((int64_t)iss.grp * blocks_per_head + y / q4::kBlk) * 512;
      ptx::bulk_load(wK + stage * q4::kKBytes, Kq4 + blk, nb * q4::kBlkBytes, &fb[stage]);
      ptx::bulk_load(wV + stage * q4::kVBytes, Vq4 + blk, nb * q4::kBlkBytes, &fb[stage]);
      ptx::bulk_load(dS, Ks + (int64_t)iss.grp * L_cap + y, nb * q4::kBlk * 4, &fb[stage]);
      ptx::bulk_load(dS + q4::kT * 4, Vs + (int64_t)iss.grp * L_cap + y, nb * q4::kBlk * 4, &fb[stage]);
    }
    ++iss_tile;
    if (may_claim && !claim_issued && iss.ntiles - iss_tile <= 2) {
      if (lane == 0) it_claim = atomicAdd(plan.counter, 1) + n_static;
      claim_issued = true;
    }
    return true;
  };

  int inflight = 0, first_grp = -1;
#pragma unroll 1
  for (int s = 0; s < q4::kStages; ++s) {
    if (exhausted || !issue(s)) break;
    if (s == 0) first_grp = iss.grp;
    ++inflight;
  }

  const int q4 = lane & 3, r8 = lane >> 2;
  // Q of head r8 (+8 ng), d = 32 J + 8 q4 .. + 7, fp16 pairs; pairs 1 and 3
  // (d + 2, 3 and d + 6, 7) divided by 16.  They depend on the kv group
  // only: loaded for the first item while its tiles are in flight, and
  // again only when an item of another group starts.
  uint32_t qf[NG][D / 32][4];
  float qs8[NG][2];             // 8 sum_d q'_d of heads 2 q4 and 2 q4 + 1
  int q_grp = -1;
  auto load_q = [&](int grp) {
    const int b = grp / geo.Hkv, kvh = grp - b * geo.Hkv;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int h = ng * 8 + r8;
      const bool ok = h < geo.g;
      const uint16_t* qr = tb.q + (int64_t)(b * geo.Hq + kvh * geo.g + h) * tb.q_stride;
      // a thread's dimensions 32 J + 8 q4 .. + 7 are 16 contiguous bytes:
      // four 16-byte loads, all in flight at once
      uint4 qv[D / 32];
#pragma unroll
      for (int J = 0; J < D / 32; ++J)
        qv[J] = ok ? *reinterpret_cast<const uint4*>(qr + 32 * J + 8 * q4) : make_uint4(0u, 0u, 0u, 0u);
      float qsum = 0.f;
#pragma unroll
      for (int J = 0; J < D / 32; ++J) {
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          uint32_t v = 0u;
          if (ok) {
            const uint32_t w = pr == 0 ? qv[J].x : pr == 1 ? qv[J].y : pr == 2 ? qv[J].z : qv[J].w;
            float lo, hi;
            if constexpr (DT == DT_BF16) {
              lo = __uint_as_float(w << 16);
              hi = __uint_as_float(w & 0xffff0000u);
            } else {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
              lo = f.x;
              hi = f.y;
            }
            const float sc = (pr & 1) ? 0.0625f : 1.f;
            v = ptx::pack2<DT_F16>(lo * sc, hi * sc);
            // q' as the MMA sees it: the rounded fp16 value, times 16 back
            const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&v));
            qsum += (r.x + r.y) * ((pr & 1) ? 16.f : 1.f);
          }
          qf[ng][J][pr] = v;
        }
      }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
      // lanes 4 h .. 4 h + 3 hold head h's sum; this thread's columns are
      // heads 2 q4 and 2 q4 + 1
      qs8[ng][0] = 8.f * __shfl_sync(0xffffffffu, qsum, 8 * q4);
      qs8[ng][1] = 8.f * __shfl_sync(0xffffffffu, qsum, 8 * q4 + 4);
    }
    q_grp = grp;
  };
  if (first_grp >= 0) load_q(first_grp);

  float o[NG][D / 16][4];
  float oc[NG][4];              // sum_t (P vs)'_t 2^-24 of heads 2 q4, 2 q4 + 1
  float m[NG][2], l[NG][2];
  uint32_t hmask = 0u;          // the item's heads, and this thread's heads' ranks
  int rk[NG][2];
  Item cur;
  cur.grp = cur.u = cur.c = cur.ntiles = 0;
  cur.t0 = cur.t1 = 0;
  int stage = 0;
  uint32_t phase = 0;
  constexpr float kTwo24 = 16777216.f;
  const float2 kTwo24x2 = make_float2(kTwo24, kTwo24);
#pragma unroll 1
  while (inflight > 0) {
    if (!ptx::mbar_wait(&fb[stage], phase)) {
      if (lane == 0) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const int4 mt = meta[stage];
    if (mt.w == 0) {
      cur.grp = mt.x;
      cur.u = mt.y;
      cur.c = mt.z;
      cur.t0 = metat[2 * stage];
      cur.t1 = metat[2 * stage + 1];
      cur.ntiles = q4::tiles(cur.t0, cur.t1);
      // the end-of-item tables, read now so that their latency overlaps
      const int slot_idx = cur.grp * geo.umax + cur.u;
      hmask = tb.mask[slot_idx];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = ng * 8 + 2 * q4 + i;
          rk[ng][i] = r < geo.g ? tb.rank[(size_t)slot_idx * 16 + r] : 0;
        }
      if (cur.grp != q_grp) load_q(cur.grp);
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) o[ng][mt2][0] = o[ng][mt2][1] = o[ng][mt2][2] = o[ng][mt2][3] = 0.f;
        oc[ng][0] = oc[ng][1] = oc[ng][2] = oc[ng][3] = 0.f;
        m[ng][0] = m[ng][1] = -INFINITY;
        l[ng][0] = l[ng][1] = 0.f;
      }
    }
    const uint32_t aK = ptx::smem_u32(wK + stage * q4::kKBytes);
    const uint32_t aV = ptx::smem_u32(wV + stage * q4::kVBytes);
    const float* sks = reinterpret_cast<const float*>(wS + stage * q4::kSBytes);
    const float* svs = sks + q4::kT;

    // S^T = Kq Q^T per 16-token fragment t (block t / 2, rows 16 (t % 2) ..)
    float s[NG][q4::kSubT][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int t = 0; t < q4::kSubT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[ng][t][i] = 0.f;
#pragma unroll
    for (int J = 0; J < D / 32; ++J) {
#pragma unroll
      for (int t = 0; t < q4::kSubT; ++t) {
        const uint32_t aB = aK + (t >> 1) * q4::kBlkBytes;
        const int ra = (t & 1) * 16 + r8, rb = ra + 8;
        const uint32_t wa = ptx::lds32(aB + ((J * q4::kBlk + ra) * 4 + q4) * 4);
        const uint32_t wb = ptx::lds32(aB + ((J * q4::kBlk + rb) * 4 + q4) * 4);
        uint32_t a0[4], a1[4];
        ptx::u4x8_to_f16x2_sub(wa, a0[0], a0[2], a1[0], a1[2]);
        ptx::u4x8_to_f16x2_sub(wb, a0[1], a0[3], a1[1], a1[3]);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          ptx::mma16816<DT_F16>(s[ng][t], a0, qf[ng][J][0], qf[ng][J][1]);
          ptx::mma16816<DT_F16>(s[ng][t], a1, qf[ng][J][2], qf[ng][J][3]);
        }
      }
    }
    // rows (tokens) r8 and r8 + 8 of each fragment: the K scale, and the V
    // scale with the 1/16 of the rows stored as 16 n fields (row + 8)
    float vsc[q4::kSubT][2];
#pragma unroll
    for (int t = 0; t < q4::kSubT; ++t) {
      const float k0 = sks[t * 16 + r8], k1 = sks[t * 16 + r8 + 8];
      vsc[t][0] = svs[t * 16 + r8];
      vsc[t][1] = svs[t * 16 + r8 + 8] * 0.0625f;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
        const float2 nq = make_float2(-qs8[ng][0], -qs8[ng][1]);
        const float2 a = __fmul2_rn(__ffma2_rn(make_float2(s[ng][t][0], s[ng][t][1]), kTwo24x2, nq),
                                    make_float2(k0, k0));
        const float2 b = __fmul2_rn(__ffma2_rn(make_float2(s[ng][t][2], s[ng][t][3]), kTwo24x2, nq),
                                    make_float2(k1, k1));
        s[ng][t][0] = a.x;
        s[ng][t][1] = a.y;
        s[ng][t][2] = b.x;
        s[ng][t][3] = b.y;
      }
    }
    // a tile the item covers only in part: its other tokens get no weight
    // (their scale slots may hold anything)
    const int64_t tbase = q4::tile_base(cur.t0) + (int64_t)mt.w * q4::kT;
    if (tbase < cur.t0 || tbase + q4::kT > cur.t1) {
      const int lo = (int)(cur.t0 > tbase ? cur.t0 - tbase : 0);
      const int hi = (int)(cur.t1 - tbase < q4::kT ? cur.t1 - tbase : q4::kT);
#pragma unroll
      for (int t = 0; t < q4::kSubT; ++t)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int row = t * 16 + r8 + 8 * i;
          if (row >= lo && row < hi) continue;
          vsc[t][i] = 0.f;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) s[ng][t][2 * i] = s[ng][t][2 * i + 1] = -INFINITY;
        }
    }
    const float c = geo.scale_log2e;
    uint32_t pb[NG][q4::kSubT][2];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      float mx[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float v = fmaxf(s[ng][0][i], s[ng][0][i + 2]);
#pragma unroll
        for (int t = 1; t < q4::kSubT; ++t) v = fmaxf(v, fmaxf(s[ng][t][i], s[ng][t][i + 2]));
        v *= c;
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        mx[i] = fmaxf(m[ng][i], v);
      }
      float nb[2], alpha[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float bse = mx[i] == -INFINITY ? 0.f : mx[i];
        nb[i] = -bse;
        alpha[i] = exp2f(m[ng][i] - bse);
        m[ng][i] = mx[i];
      }
      // the two rows of a fragment side by side in packed fp32 operations
      const float2 c2 = make_float2(c, c), nb2 = make_float2(nb[0], nb[1]);
      float2 ls = make_float2(0.f, 0.f);
#pragma unroll
      for (int t = 0; t < q4::kSubT; ++t) {
        const float2 e01 = __ffma2_rn(make_float2(s[ng][t][0], s[ng][t][1]), c2, nb2);
        const float2 e23 = __ffma2_rn(make_float2(s[ng][t][2], s[ng][t][3]), c2, nb2);
        const float2 p01 = make_float2(ptx::ex2(e01.x), ptx::ex2(e01.y));
        const float2 p23 = make_float2(ptx::ex2(e23.x), ptx::ex2(e23.y));
        ls = __fadd2_rn(ls, __fadd2_rn(p01, p23));
        // the V scale of each token weights its P (0 for masked tokens)
        const float2 w01 = __fmul2_rn(p01, make_float2(vsc[t][0], vsc[t][0]));
        const float2 w23 = __fmul2_rn(p23, make_float2(vsc[t][1], vsc[t][1]));
        pb[ng][t][0] = ptx::movmatrix_trans(ptx::pack2<DT_F16>(w01.x, w01.y));
        pb[ng][t][1] = ptx::movmatrix_trans(ptx::pack2<DT_F16>(w23.x, w23.y));
      }
      l[ng][0] = l[ng][0] * alpha[0] + ls.x;
      l[ng][1] = l[ng][1] * alpha[1] + ls.y;
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
        const float2 al = make_float2(alpha[0], alpha[1]);
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          const float2 x = __fmul2_rn(make_float2(o[ng][mt2][0], o[ng][mt2][1]), al);
          const float2 y = __fmul2_rn(make_float2(o[ng][mt2][2], o[ng][mt2][3]), al);
          o[ng][mt2][0] = x.x;
          o[ng][mt2][1] = x.y;
          o[ng][mt2][2] = y.x;
          o[ng][mt2][3] = y.y;
        }
        const float2 x = __fmul2_rn(make_float2(oc[ng][0], oc[ng][1]), al);
        const float2 y = __fmul2_rn(make_float2(oc[ng][2], oc[ng][3]), al);
        oc[ng][0] = x.x;
        oc[ng][1] = x.y;
        oc[ng][2] = y.x;
        oc[ng][3] = y.y;
      }
    }
    // O^T += Vq^T (vs P)^T: d-rows r8 and r8 + 8 of each m16 slice, one
    // 4-byte load per row covering both 16-token fragments
#pragma unroll
    for (int mt2 = 0; mt2 < D / 16; ++mt2) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t aB = aV + b * q4::kBlkBytes;
        const uint32_t va = ptx::lds32(aB + ((mt2 * 16 + r8) * 4 + q4) * 4);
        const uint32_t vb = ptx::lds32(aB + ((mt2 * 16 + r8 + 8) * 4 + q4) * 4);
        uint32_t a0[4], a1[4];
        ptx::u4x8_to_f16x2_sub(va, a0[0], a0[2], a1[0], a1[2]);
        ptx::u4x8_to_f16x2_sub(vb, a0[1], a0[3], a1[1], a1[3]);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          ptx::mma16816<DT_F16>(o[ng][mt2], a0, pb[ng][2 * b][0], pb[ng][2 * b][1]);
          ptx::mma16816<DT_F16>(o[ng][mt2], a1, pb[ng][2 * b + 1][0], pb[ng][2 * b + 1][1]);
        }
      }
    }
    {
      // rows of 1s at the scales of the fields: 2^-24 for tokens 2 q4 (+1)
      // of each 16-token fragment, 16 * 2^-24 for tokens 2 q4 + 8 (+9)
      const uint32_t one[4] = {0x00010001u, 0x00010001u, 0x00100010u, 0x00100010u};
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int t = 0; t < q4::kSubT; ++t) ptx::mma16816<DT_F16>(oc[ng], one, pb[ng][t][0], pb[ng][t][1]);
    }
    __syncwarp();
    --inflight;
    const bool last = mt.w == cur.ntiles - 1;
    if (!exhausted && issue(stage)) ++inflight;
    if (++stage == q4::kStages) {
      stage = 0;
      phase ^= 1u;
    }
    if (!last) continue;

    const int b = cur.grp / geo.Hkv, kvh = cur.grp - b * geo.Hkv;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float lt = l[ng][i];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int r = ng * 8 + 2 * q4 + i;
        if (r >= geo.g || !((hmask >> r) & 1u)) continue;
        const int64_t slot =
            ((int64_t)(b * geo.Hq + kvh * geo.g + r) * (geo.topk + 1) + rk[ng][i]) * geo.C + cur.c;
        float* dst = plan.po + slot * D + r8;
        const float corr = -8.f * kTwo24 * oc[ng][i];
#pragma unroll
        for (int mt2 = 0; mt2 < D / 16; ++mt2) {
          dst[mt2 * 16] = fmaf(o[ng][mt2][i], kTwo24, corr);
          dst[mt2 * 16 + 8] = fmaf(o[ng][mt2][i + 2], kTwo24, corr);
        }
        if (r8 == 0) *reinterpret_cast<float2*>(plan.ml + slot * 2) = make_float2(m[ng][i], lt);
      }
    }
  }
}

// ---------------------------------------------------------------- merge
// One CTA per (b, q-head): its (topk + 1) * C partial slots, in (span rank,
// chunk) order, split into 8 contiguous runs, one per warp; empty slots
// (m = -inf) are skipped.  The warps' results are then combined in order.
constexpr int kMergeWarps = 8;
constexpr int kBatch = 8;

template <int DT, int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    decode_merge_kernel(Plan plan, Geo geo, void* __restrict__ O, float* __restrict__ lse) {
  constexpr int E = D / 32;  // columns per lane
  __shared__ float wm[kMergeWarps], wl[kMergeWarps];
  __shared__ float wo[kMergeWarps][D];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int nslots = (geo.topk + 1) * geo.C;
  const int per = (nslots + kMergeWarps - 1) / kMergeWarps;
  const int s0 = warp * per, s1 = min(s0 + per, nslots);
  const int64_t base = (int64_t)row * nslots;
  const float2* ml = reinterpret_cast<const float2*>(plan.ml);
  float M = -INFINITY, Ls = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int sb = s0; sb < s1; sb += 32) {
    const int sl = sb + lane;
    const float2 mlv = sl < s1 ? ml[base + sl] : make_float2(-INFINITY, 0.f);
    uint32_t nz = __ballot_sync(0xffffffffu, mlv.x != -INFINITY);
    while (nz) {
      int ids[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        ids[i] = nz ? __ffs(nz) - 1 : -1;
        nz &= nz ? nz - 1u : 0u;
      }
      float po[kBatch][E];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (ids[i] >= 0) {
          const float* src = plan.po + (base + sb + ids[i]) * D + lane * E;
          if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            po[i][0] = v.x; po[i][1] = v.y; po[i][2] = v.z; po[i][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            po[i][0] = v.x; po[i][1] = v.y;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (ids[i] < 0) continue;
        const float pm = __shfl_sync(0xffffffffu, mlv.x, ids[i]);
        const float pl = __shfl_sync(0xffffffffu, mlv.y, ids[i]);
        const float Mn = fmaxf(M, pm);
        const float a = exp2f(M - Mn), bb = exp2f(pm - Mn);
        Ls = Ls * a + pl * bb;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * a + po[i][e] * bb;
        M = Mn;
      }
    }
  }
  if (lane == 0) {
    wm[warp] = M;
    wl[warp] = Ls;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) wo[warp][lane * E + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    const int col = threadIdx.x;
    float Mt = -INFINITY;
    for (int w = 0; w < kMergeWarps; ++w) Mt = fmaxf(Mt, wm[w]);
    float Lt = 0.f, ot = 0.f;
    for (int w = 0; w < kMergeWarps; ++w) {
      if (wm[w] == -INFINITY) continue;
      const float f = exp2f(wm[w] - Mt);
      Lt += wl[w] * f;
      ot += wo[w][col] * f;
    }
    store_elem<DT>(O, (int64_t)row * D + col, ot / Lt);
    if (lse && col == 0) lse[row] = Mt * kLn2 + logf(Lt);
  }
}


// The plan's workspace pointers and the geometry of a decode step.
void plan_geo(const Problem& pr, int64_t pos, void* ws, Plan& plan, Geo& geo, bool group = false) {
  const Layout lay = layout(pr, group);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  plan.n_union = reinterpret_cast<int*>(w8 + lay.n_union);
  plan.n_items = reinterpret_cast<int*>(w8 + lay.n_items);
  plan.span = reinterpret_cast<int*>(w8 + lay.span);
  plan.mask = reinterpret_cast<uint32_t*>(w8 + lay.mask);
  plan.rank = w8 + lay.rank;
  plan.counter = reinterpret_cast<int*>(w8 + lay.counter);
  plan.ml = reinterpret_cast<float*>(w8 + lay.ml);
  plan.po = reinterpret_cast<float*>(w8 + lay.po);
  plan.q = reinterpret_cast<uint16_t*>(w8 + lay.q);
  geo.Hq = pr.Hq;
  geo.Hkv = pr.Hkv;
  geo.g = pr.g;
  geo.topk = pr.topk;
  geo.S = pr.S;
  geo.C = lay.C;
  geo.CH = lay.CH;
  geo.umax = pr.g * pr.topk + 1;
  geo.n_grp = pr.B * pr.Hkv;
  geo.pos = pos;
  geo.ell = pos / pr.S;
  geo.scale_log2e = pr.scale * kLog2e;
}

template <int DT>
cudaError_t attend_q8(const Problem& pr, const void* Q, const int8_t* Kq, const float* Ks, const int8_t* Vq,
                      const float* Vs, void* O, float* lse, const Plan& plan, const Geo& geo, uint32_t* err,
                      cudaStream_t st) {
  constexpr int D = 128;
  CUtensorMap tmK;
  cudaError_t e = make_q8_tmap(&tmK, Kq, D, pr.L, pr.L_cap, (int64_t)pr.B * pr.Hkv, kTile);
  if (e != cudaSuccess) return e;
  auto attend = pr.g <= 8 ? decode_attend_q8_kernel<DT, 1> : decode_attend_q8_kernel<DT, 2>;
  static bool attr_done[2][kMaxDevices] = {};
  e = ensure_smem_attr(attend, kSmemLimit, attr_done[pr.g <= 8 ? 0 : 1]);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attend, dim3(device_sm_count()), dim3(q8::kThreads), q8::kFixed, st, tmK, Vq, Ks, Vs, pr.L_cap, Q,
                 plan, geo, err);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<DT, D>, dim3(pr.B * pr.Hq), dim3(kMergeWarps * 32), 0, st, plan, geo, O,
                    lse);
}

template <int DT>
cudaError_t attend_q4(const Problem& pr, const void* Q, const uint32_t* Kq4, const float* Ks, const uint32_t* Vq4,
                      const float* Vs, void* O, float* lse, const Plan& plan, const Geo& geo, uint32_t* err,
                      cudaStream_t st) {
  constexpr int D = 128;
  auto attend = pr.g <= 8 ? decode_attend_q4_kernel<DT, 1> : decode_attend_q4_kernel<DT, 2>;
  static bool attr_done[2][kMaxDevices] = {};
  cudaError_t e = ensure_smem_attr(attend, q4::kFixed, attr_done[pr.g <= 8 ? 0 : 1]);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attend, dim3(device_sm_count()), dim3(q4::kThreads), q4::kFixed, st, Kq4, Vq4, Ks, Vs, pr.L_cap,
                 Q, plan, geo, err);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<DT, D>, dim3(pr.B * pr.Hq), dim3(kMergeWarps * 32), 0, st, plan, geo, O,
                    lse);
}

template <int DT, int D>
cudaError_t attend_16(const Problem& pr, const void* Q, const void* K, const void* V, void* O, float* lse,
                      const Plan& plan, const Geo& geo, uint32_t* err, cudaStream_t st) {
  using Cf = Cfg<D>;
  CUtensorMap tmK, tmV;
  cudaError_t e = make_kv_tmap(&tmK, K, pr.dtype, D, pr.L, pr.L_cap, (int64_t)pr.B * pr.Hkv, kTile);
  if (e != cudaSuccess) return e;
  e = make_kv_tmap(&tmV, V, pr.dtype, D, pr.L, pr.L_cap, (int64_t)pr.B * pr.Hkv, kTile);
  if (e != cudaSuccess) return e;
  auto attend = pr.g <= 8 ? decode_attend_kernel<DT, D, 1> : decode_attend_kernel<DT, D, 2>;
  static bool attr_done[2][kMaxDevices] = {};
  e = ensure_smem_attr(attend, kSmemLimit, attr_done[pr.g <= 8 ? 0 : 1]);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attend, dim3(device_sm_count()), dim3(kThreads), Cf::kFixed, st, tmK, tmV, Q, plan, geo, err);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<DT, D>, dim3(pr.B * pr.Hq), dim3(kMergeWarps * 32), 0, st, plan, geo, O,
                    lse);
}

}  // namespace

cudaError_t launch_attend_decode_q8(const Problem& pr, const void* Q, int64_t pos, const int8_t* Kq,
                                    const float* Ks, const int8_t* Vq, const float* Vs, const int32_t* sel,
                                    void* O, float* lse, void* ws, cudaStream_t st) {
  Plan plan;
  Geo geo;
  plan_geo(pr, pos, ws, plan, geo);
  uint32_t* err = ws_error(ws);
  cudaError_t e = launch_pdl(decode_plan_kernel, dim3(geo.n_grp), dim3(kPlanThreads), 0, st, sel, plan, geo, err);
  if (e != cudaSuccess) return e;
  if (pr.dtype == DT_BF16) return attend_q8<DT_BF16>(pr, Q, Kq, Ks, Vq, Vs, O, lse, plan, geo, err, st);
  return attend_q8<DT_F16>(pr, Q, Kq, Ks, Vq, Vs, O, lse, plan, geo, err, st);
}

cudaError_t launch_attend_decode_q4(const Problem& pr, const void* Q, int64_t pos, const uint32_t* Kq4,
                                    const float* Ks, const uint32_t* Vq4, const float* Vs, const int32_t* sel,
                                    void* O, float* lse, void* ws, cudaStream_t st) {
  Plan plan;
  Geo geo;
  plan_geo(pr, pos, ws, plan, geo);
  uint32_t* err = ws_error(ws);
  cudaError_t e = launch_pdl(decode_plan_kernel, dim3(geo.n_grp), dim3(kPlanThreads), 0, st, sel, plan, geo, err);
  if (e != cudaSuccess) return e;
  if (pr.dtype == DT_BF16) return attend_q4<DT_BF16>(pr, Q, Kq4, Ks, Vq4, Vs, O, lse, plan, geo, err, st);
  return attend_q4<DT_F16>(pr, Q, Kq4, Ks, Vq4, Vs, O, lse, plan, geo, err, st);
}

cudaError_t launch_attend_decode_q4_planned(const Problem& pr, const void* Q, const uint32_t* Kq4, const float* Ks,
                                            const uint32_t* Vq4, const float* Vs, void* O, float* lse,
                                            const dplan::Plan& plan, const dplan::Geo& geo, uint32_t* err,
                                            cudaStream_t st) {
  if (pr.dtype == DT_BF16) return attend_q4<DT_BF16>(pr, Q, Kq4, Ks, Vq4, Vs, O, lse, plan, geo, err, st);
  return attend_q4<DT_F16>(pr, Q, Kq4, Ks, Vq4, Vs, O, lse, plan, geo, err, st);
}

bool decode_fast_supported(const Problem& pr) {
  return (pr.dtype == DT_BF16 || pr.dtype == DT_F16) && (pr.d == 64 || pr.d == 128) &&
         pr.g <= kMaxG && pr.topk <= kMaxK && (int64_t)pr.B * pr.Hkv <= kMaxGroups && pr.L > 0;
}

size_t decode_ws_bytes(const Problem& pr) { return layout(pr).total - kWsHeader; }

void decode_plan_args(const Problem& pr, int64_t pos, void* ws, dplan::Plan* plan, dplan::Geo* geo, bool group) {
  plan_geo(pr, pos, ws, *plan, *geo, group);
}

cudaError_t launch_attend_decode_planned(const Problem& pr, const void* Q, const void* K, const void* V, void* O,
                                         float* lse, const dplan::Plan& plan, const dplan::Geo& geo,
                                         uint32_t* err, cudaStream_t st) {
  if (pr.d == 128) {
    if (pr.dtype == DT_BF16) return attend_16<DT_BF16, 128>(pr, Q, K, V, O, lse, plan, geo, err, st);
    return attend_16<DT_F16, 128>(pr, Q, K, V, O, lse, plan, geo, err, st);
  }
  if (pr.dtype == DT_BF16) return attend_16<DT_BF16, 64>(pr, Q, K, V, O, lse, plan, geo, err, st);
  return attend_16<DT_F16, 64>(pr, Q, K, V, O, lse, plan, geo, err, st);
}

cudaError_t launch_attend_decode_q8_planned(const Problem& pr, const void* Q, const int8_t* Kq, const float* Ks,
                                            const int8_t* Vq, const float* Vs, void* O, float* lse,
                                            const dplan::Plan& plan, const dplan::Geo& geo, uint32_t* err,
                                            cudaStream_t st) {
  if (pr.dtype == DT_BF16) return attend_q8<DT_BF16>(pr, Q, Kq, Ks, Vq, Vs, O, lse, plan, geo, err, st);
  return attend_q8<DT_F16>(pr, Q, Kq, Ks, Vq, Vs, O, lse, plan, geo, err, st);
}

cudaError_t launch_attend_decode(const Problem& pr, const void* Q, int64_t pos, const void* K,
                                 const void* V, const int32_t* sel, void* O, float* lse, void* ws,
                                 cudaStream_t st) {
  Plan plan;
  Geo geo;
  plan_geo(pr, pos, ws, plan, geo);
  uint32_t* err = ws_error(ws);
  cudaError_t e = launch_pdl(decode_plan_kernel, dim3(geo.n_grp), dim3(kPlanThreads), 0, st, sel, plan, geo, err);
  if (e != cudaSuccess) return e;
  return launch_attend_decode_planned(pr, Q, K, V, O, lse, plan, geo, err, st);
}

}  // namespace ssa

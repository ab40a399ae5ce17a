// route_tc.cu -- span scores and top-k selection for a chunk of queries on
// the 5th-generation tensor cores (16-bit queries).
//
// Superlinear release post (geeks.co.kr/post/2077), key-idea section: every
// query scores the candidate spans and keeps the top k; the router is fixed
// by the specification (q . summary in fp32, ties to the lower span).
//
// The fp32 summaries are first split into three 16-bit planes,
// s = s1 + s2 + s3 (each the round-to-nearest of what the previous planes
// left), which carry 24 significant bits; q . s = sum_p q . s_p with the
// products exact and the sums accumulated in fp32 tensor memory.  The score
// of a (query, span) pair is rounded once per 16-element MMA step (3 * d / 16
// times), far below the 1e-3 score margin the selections are checked at.
//
//  split   one pass over the candidate summaries into the workspace
//  route   one CTA per tile of 128 (query, head) rows of one kv-head
//          (128 / g queries x g heads): Q rows gathered into a swizzled
//          K-major tile, 32-span blocks of the three planes stream through
//          a 2-stage TMA ring, one thread issues S = sum_p Q S_p^T into
//          tensor memory (double buffered), and four warps (one row per
//          thread) fold each block into a register list of the row's k best
//          (strictly greater scores only, so among equal scores the earlier,
//          lower span stays).  The list is written in ascending span order.
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace ssa {
namespace {

constexpr int kRows = 128;    // (query, head) rows per tile
constexpr int kBlk = 32;      // candidate spans per block (small, so that two CTAs fit an SM)
constexpr int kRouteThreads = 192;  // warps 0-3 select, 4 TMA, 5 MMA
constexpr int kMaxTopK = 16;  // register list size; larger k uses the fp32 tile router

template <int D>
struct RCfg {
  static constexpr int kRegion = 128 * 128;           // Q: 128 rows x 128 bytes
  static constexpr int kRegionB = kBlk * 128;          // summaries: kBlk rows x 128 bytes
  static constexpr int kQBytes = (D / 64) * kRegion;
  static constexpr int kPlane = (D / 64) * kRegionB;   // one plane of a block
  static constexpr int kStage = 3 * kPlane;
  // per selection warp: its 32 rows' scores of one 32-span chunk, row-major
  // with a padded stride (conflict-free stores, any-column loads)
  static constexpr int kStageStride = 33;
  static constexpr int kPick = 4 * 32 * kStageStride * 4;
  static constexpr size_t kSmem = 1024 + (size_t)kQBytes + 2 * kStage + 256 + kPick;
};

template <int DT>
__device__ __forceinline__ uint16_t to16(float v) {
  if constexpr (DT == DT_BF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    return __half_as_ushort(__float2half_rn(v));
  }
}

template <int DT>
__device__ __forceinline__ float from16(uint16_t u) {
  if constexpr (DT == DT_BF16) {
    return __bfloat162float(__ushort_as_bfloat16(u));
  } else {
    return __half2float(__ushort_as_half(u));
  }
}

// planes [B*Hkv][3][ns_cap][D]: s1 = rn(s), s2 = rn(s - s1), s3 = rn(s - s1 - s2)
template <int DT, int D>
__global__ void __launch_bounds__(256) split_kernel(const float* __restrict__ summ, uint16_t* __restrict__ planes,
                                                    int64_t ns_cap, int64_t n_spans) {
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int64_t bh = blockIdx.y;
  const int64_t total = n_spans * D;
  for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
    const float s = summ[bh * ns_cap * D + e];
    const uint16_t a = to16<DT>(s);
    const float r1 = s - from16<DT>(a);
    const uint16_t b = to16<DT>(r1);
    const float r2 = r1 - from16<DT>(b);
    const uint16_t c = to16<DT>(r2);
    uint16_t* base = planes + (bh * 3) * ns_cap * D;
    base[e] = a;
    base[ns_cap * D + e] = b;
    base[2 * ns_cap * D + e] = c;
  }
}

// A row's 16 best (score, span), sorted by score descending (the first k of
// them are its k best for any k <= 16).  A candidate enters only when
// strictly greater than the 16th, and behind every entry of equal score, so
// among equal scores the earlier (lower) span stays ahead.  All indexing is
// static, so the list lives in registers, and an insertion is one parallel
// shift: since the list is sorted, ge[i] = (v[i] >= s) is true on a prefix,
// and entry i becomes v[i] (inside the prefix), s (first slot after it) or
// v[i - 1] (further down).
struct Top16 {
  float v[16];
  int j[16];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = -INFINITY;
      j[i] = kNoSpan;
    }
  }
  __device__ __forceinline__ float thr() const { return v[15]; }
  __device__ __forceinline__ void push(float s, int span) {
    if (!(s > v[15])) return;
    bool ge[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ge[i] = v[i] >= s;
#pragma unroll
    for (int i = 15; i > 0; --i) {
      v[i] = ge[i] ? v[i] : (ge[i - 1] ? s : v[i - 1]);
      j[i] = ge[i] ? j[i] : (ge[i - 1] ? span : j[i - 1]);
    }
    v[0] = ge[0] ? v[0] : s;
    j[0] = ge[0] ? j[0] : span;
  }
};

template <int DT, int D>
__global__ void __launch_bounds__(kRouteThreads, 2)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmP, const void* __restrict__ Q, int32_t* __restrict__ sel,
                    float* __restrict__ sel_score, int Hq, int Hkv, int64_t n_q, int64_t q_pos0, int S, int topk,
                    uint32_t* __restrict__ err) {
  using C = RCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sB = sQ + C::kQBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + 2 * C::kStage);
  uint64_t* q_full = bar + 0;
  uint64_t* b_full = bar + 1;   // [2]
  uint64_t* b_empty = bar + 3;  // [2]
  uint64_t* s_full = bar + 5;   // [2]
  uint64_t* s_free = bar + 7;   // [2]
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(bar + 9);
  volatile int* abort = reinterpret_cast<volatile int*>(bar + 10);
  float* pick = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bar) + 256);  // [4 warps][32][33]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int g = Hq / Hkv;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int64_t row0 = (int64_t)blockIdx.x * kRows;  // first (query, head) row of the tile
  const int64_t rows_total = n_q * g;
  const int64_t last_row = min(row0 + kRows, rows_total) - 1;
  const int64_t ell_max = (q_pos0 + last_row / g) / S;   // candidates of the tile: [0, ell_max)
  const int nblk = (int)((ell_max + kBlk - 1) / kBlk);

  if (tid == 0) {
    ptx::mbar_init(q_full, 128);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&b_full[s], 1);
      ptx::mbar_init(&b_empty[s], 1);
      ptx::mbar_init(&s_full[s], 1);
      ptx::mbar_init(&s_free[s], 4);
    }
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) tc::alloc(tmem_base, 2 * kBlk);
  if (warp == 4 && lane == 0) ptx::prefetch_tmap(&tmP);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_base;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int bh = b * Hkv + kvh;

  if (warp == 4) {
    if (lane == 0) {
      for (int blk = 0; blk < nblk && !*abort; ++blk) {
        const int st = blk & 1;
        if (blk >= 2 && !ptx::mbar_wait(&b_empty[st], (uint32_t)(((blk - 2) >> 1) & 1))) {
          flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
          *abort = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(&b_full[st], C::kStage);
        uint8_t* dst = sB + st * C::kStage;
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int r = 0; r < D / 64; ++r)
            ptx::tma_load_3d(dst + p * C::kPlane + r * C::kRegionB, &tmP, &b_full[st], r * 64, blk * kBlk,
                             bh * 3 + p);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t id = tc::idesc_f16(kRows, kBlk, DT == DT_BF16 ? 1 : 0, 0, 0);
      const uint32_t aQ = ptx::smem_u32(sQ), aB = ptx::smem_u32(sB);
      bool ok = ptx::mbar_wait(q_full, 0);
      for (int blk = 0; blk < nblk && ok && !*abort; ++blk) {
        const int st = blk & 1;
        ok = ptx::mbar_wait(&b_full[st], (uint32_t)((blk >> 1) & 1));
        if (ok && blk >= 2) ok = ptx::mbar_wait(&s_free[st], (uint32_t)(((blk - 2) >> 1) & 1));
        if (!ok) break;
        tc::fence_after();
        const uint32_t dS = tmem + st * kBlk;
        int step = 0;
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int k = 0; k < D / 16; ++k, ++step) {
            const uint64_t qd = tc::sdesc_sw128(aQ + (k >> 2) * C::kRegion + (k & 3) * 32, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(aB + st * C::kStage + p * C::kPlane + (k >> 2) * C::kRegionB +
                                                    (k & 3) * 32,
                                                16, 1024);
            tc::mma(dS, qd, bd, id, step > 0 ? 1u : 0u);
          }
        tc::commit(&s_full[st]);
        tc::commit(&b_empty[st]);
      }
      if (!ok) {
        flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
        *abort = 1;
      }
    }
  } else {
    // ------------------------------------------------ selection: row r = tid
    const int r = tid;
    const int64_t grow = row0 + r;
    const bool valid = grow < rows_total;
    const int64_t i = valid ? grow / g : 0;
    const int h = kvh * g + (int)(valid ? grow % g : 0);
    const int64_t qrow = (int64_t)(b * Hq + h) * n_q + i;
    const int64_t ell = valid ? (q_pos0 + i) / S : 0;
    // gather the row of Q (zeros beyond the chunk)
    {
      const uint8_t* src = static_cast<const uint8_t*>(Q) + (valid ? qrow : 0) * (int64_t)D * 2;
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        uint8_t* dst = sQ + (ch >> 3) * C::kRegion + r * 128 + ((((uint32_t)ch & 7) ^ ((uint32_t)r & 7)) << 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
                     "l"(src + ch * 16), "r"(valid ? 16u : 0u)
                     : "memory");
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      tc::fence_proxy_async_smem();
      ptx::mbar_arrive(q_full);
    }
    Top16 best;
    best.init();
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float* my_pick = pick + (warp * 32 + lane) * C::kStageStride;
    for (int blk = 0; blk < nblk; ++blk) {
      const int st = blk & 1;
      if (!ptx::mbar_wait(&s_full[st], (uint32_t)((blk >> 1) & 1))) {
        flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
        *abort = 1;
        break;
      }
      tc::fence_after();
      const int jb = blk * kBlk;
#pragma unroll 1
      for (int q = 0; q < kBlk / 32; ++q) {
        uint32_t rr[32];
        tc::ld32(tmem + st * kBlk + lane_off + q * 32, rr);
        if (q == kBlk / 32 - 1) {
          tc::fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s_free[st]);
        }
        const int j0 = jb + q * 32;
        // spans j0 + c with c >= nvalid are no candidates of this row (only
        // its last chunk has any)
        const int64_t nvalid = ell - j0;
        if (nvalid < 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= nvalid) rr[c] = 0xff800000u;  // -inf
        }
        // the chunk's best score first: most chunks of most rows have none
        // above the current 16th best and stop here
        float mx = __uint_as_float(rr[0]);
#pragma unroll
        for (int c = 1; c < 31; c += 2) mx = ptx::max3(mx, __uint_as_float(rr[c]), __uint_as_float(rr[c + 1]));
        mx = fmaxf(mx, __uint_as_float(rr[31]));
        const float t0 = best.thr();
        if (!__any_sync(0xffffffffu, mx > t0)) continue;
        // candidates that beat the current 16th best
        uint32_t pass = 0;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (__uint_as_float(rr[c]) > t0) pass |= 1u << c;
        // the lane's row of scores, so that any column can be read back by
        // index (a load instead of a select tree over the registers)
        if (pass) {
#pragma unroll
          for (int c = 0; c < 32; ++c) my_pick[c] = __uint_as_float(rr[c]);
        }
        // insert them in lockstep across the warp, lowest span first
        while (__any_sync(0xffffffffu, pass != 0u)) {
          if (pass) {
            const int p = __ffs(pass) - 1;
            pass &= pass - 1u;
            best.push(my_pick[p], j0 + p);
          }
        }
      }
    }
    if (valid) {
      // the first topk entries, written in ascending span order
      int32_t* out = sel + qrow * topk;
      float* osc = sel_score ? sel_score + qrow * topk : nullptr;
      int n = 0;
#pragma unroll
      for (int a = 0; a < 16; ++a) {
        if (a >= topk || best.j[a] == kNoSpan) continue;
        ++n;
        int rank = 0;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c < topk && best.j[c] < best.j[a]) ++rank;
        out[rank] = best.j[a];
        if (osc) osc[rank] = best.v[a];
      }
      for (int a = n; a < topk; ++a) {
        out[a] = -1;
        if (osc) osc[a] = __int_as_float(0x7fc00000);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 5) tc::dealloc(tmem, 2 * kBlk);
}

template <int DT, int D>
cudaError_t launch_k(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, int32_t* sel, float* sel_score,
                     const CUtensorMap& tmP, uint32_t* err, cudaStream_t st) {
  using C = RCfg<D>;
  static bool attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_attr(route_tc_kernel<DT, D>, C::kSmem, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (n_q * pr.g + kRows - 1) / kRows;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(route_tc_kernel<DT, D>, dim3((unsigned)tiles, pr.Hkv, pr.B), dim3(kRouteThreads), C::kSmem,
                    st, tmP, Q, sel, sel_score, pr.Hq, pr.Hkv, n_q, q_pos0, pr.S, pr.topk, err);
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                         int32_t* sel, float* sel_score, void* ws, cudaStream_t st) {
  uint16_t* planes = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + kWsHeader);
  uint32_t* err = ws_error(ws);
  const int64_t n_spans = (q_pos0 + n_q - 1) / pr.S;  // candidates of the chunk's last query
  if (n_spans > 0) {
    const int64_t total = n_spans * D;
    const int64_t nb = (total + 255) / 256;
    const unsigned gx = (unsigned)(nb < 1024 ? nb : 1024);
    cudaError_t e = launch_pdl(split_kernel<DT, D>, dim3(gx, pr.B * pr.Hkv), dim3(256), 0, st, summ, planes,
                               pr.ns_cap, n_spans);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tmP;
  const int64_t bh = (int64_t)pr.B * pr.Hkv;
  cudaError_t e = make_kv_tmap(&tmP, planes, pr.dtype, D, pr.ns_cap, pr.ns_cap, bh * 3, kBlk);
  if (e != cudaSuccess) return e;
  return launch_k<DT, D>(pr, Q, n_q, q_pos0, sel, sel_score, tmP, err, st);
}

}  // namespace

bool route_tc_supported(const Problem& pr, int64_t n_q) {
  return n_q > 1 && (pr.dtype == DT_BF16 || pr.dtype == DT_F16) && (pr.d == 64 || pr.d == 128) &&
         pr.g <= 16 && (kRows % pr.g) == 0 && pr.topk <= kMaxTopK;
}

size_t route_tc_ws_bytes(const Problem& pr) {
  return (size_t)pr.B * pr.Hkv * 3 * (size_t)pr.ns_cap * pr.d * 2;
}

cudaError_t launch_route_tc(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                            int32_t* sel, float* sel_score, void* ws, cudaStream_t st) {
  if (pr.d == 128) {
    if (pr.dtype == DT_BF16) return launch_typed<DT_BF16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
    return launch_typed<DT_F16, 128>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
  }
  if (pr.dtype == DT_BF16) return launch_typed<DT_BF16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
  return launch_typed<DT_F16, 64>(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st);
}

}  // namespace ssa

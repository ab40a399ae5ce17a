// prefill.cu -- chunked-prefill attention on the 5th-generation tensor cores.
//
// Superlinear release post (geeks.co.kr/post/2077): chunked prefill against
// the kept cache, and, in its key-idea section, token-level attention inside
// each query's chosen spans; SubQ SSA page (stork.ai): exact attention over
// the content-selected subset.
//
// The queries of a chunk choose different spans, so the work is dispatched
// span-major: the (query, head) rows that chose span j of kv-head h form a
// bucket, and a bucket is cut into tiles of 128 rows that share the span's
// keys and values.  Each query's own span (causal) is a second kind of tile:
// 128 / g consecutive queries times the g heads of a kv-head.
//
//  count    per (b, query head, 128 queries): validates sel rows and counts
//           each bucket's rows (shared-memory histogram, one global atomic
//           per non-empty bucket)
//  scan     one CTA: bucket offsets, the tile table (span tiles, then local
//           tiles)
//  scatter  writes each row's id and its rank in the sel row into its
//           bucket
//  attend   persistent, one CTA per SM, eleven warps.  A loader warp
//           gathers each tile's 128 query rows into one of two Q buffers
//           (128-byte swizzled K-major operand) ahead of use; a TMA warp
//           streams key / value blocks of 128 tokens through their own
//           rings; one thread issues tcgen05.mma: S = Q K^T into tensor
//           memory (double buffered), then O += P V with P read from tensor
//           memory.  Eight softmax warps (two per row quarter, one row per
//           thread, each warp half of the keys) turn S into P = 2^(S c - m)
//           (16-bit, double buffered in tensor memory), rescale O only when
//           the running maximum grows by more than 2^8, and end each tile
//           by writing one partial (m, l, normalised o) per row.
//  merge    per (b, head, query): combines the row's partials (its spans in
//           sel order, then the local span) into O and lse.
#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace ssa {
namespace {

constexpr int kTileRows = 128;
constexpr int kKeyBlk = 128;
constexpr int kMaxK = 64;
constexpr int kMaxG = 16;
constexpr int kHistMax = 12288;  // spans per kv-head the shared histogram covers
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by more than 2^8

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PrefLayout {
  size_t counts, offsets, cursors, tiles, ntiles, rows, pml, po, total;
  int64_t n_buckets, max_entries, max_tiles;
};

// Workspace of a chunk of n_q queries (the bucket index space covers every
// span slot of the cache, so the layout needs no query positions).
PrefLayout pref_layout(const Problem& pr, int64_t n_q) {
  PrefLayout l;
  const int64_t bh = (int64_t)pr.B * pr.Hkv;
  l.n_buckets = bh * pr.ns_cap;
  l.max_entries = (int64_t)pr.B * pr.Hq * n_q * pr.topk;
  const int64_t mq = kTileRows / pr.g;  // queries per local tile
  const int64_t local_tiles = bh * ((n_q + mq - 1) / mq + n_q / pr.S + 2);
  l.max_tiles = l.max_entries / kTileRows + l.n_buckets + local_tiles;
  const int64_t parts = (int64_t)pr.B * pr.Hq * n_q * (pr.topk + 1);
  size_t off = kWsHeader;
  l.counts = off; off = align256(off + l.n_buckets * 4);
  l.offsets = off; off = align256(off + l.n_buckets * 4);
  l.cursors = off; off = align256(off + l.n_buckets * 4);
  l.ntiles = off; off = align256(off + 16);
  l.tiles = off; off = align256(off + l.max_tiles * 16);
  l.rows = off; off = align256(off + l.max_entries * 4);
  l.pml = off; off = align256(off + parts * 8);
  l.po = off; off = align256(off + parts * (size_t)pr.d * 2);
  l.total = off;
  return l;
}

struct PrefArgs {
  int* counts;
  int* offsets;
  int* cursors;
  int* ntiles;     // [0] tiles in the table
  int4* tiles;     // {bucket or -1 - bh, row0 or first query, rows or queries, 0}
  int* rows;       // bucket entries: row id << 6 | rank
  float2* pml;     // [rows of Q][topk + 1] (m base 2, l)
  uint16_t* po;    // [rows of Q][topk + 1][d] normalised partial output (Q's type)
  int B, Hq, Hkv, g, d, S, topk;
  int64_t n_q, q_pos0, ns_cap, n_buckets;
  float scale_log2e;
};

// The used entries of a sel row (the leading strictly ascending run of
// candidate spans; anything else but -1 after it is an error), one thread.
__device__ __forceinline__ int row_used(const int32_t* row, int topk, int64_t ell, int* js, bool* bad) {
  int n = 0;
  int64_t prev = -1;
  bool stop = false;
  *bad = false;
  for (int r = 0; r < topk; ++r) {
    const int j = row[r];
    if (!stop && j >= 0 && j < ell && j > prev) {
      js[n++] = j;
      prev = j;
    } else {
      stop = true;
      if (j != -1) *bad = true;
    }
  }
  return n;
}

// ---------------------------------------------------------------- count
// grid (ceil(n_q / 256), B * Hq), one thread per query of one query head.
__global__ void __launch_bounds__(256) prefill_count_kernel(const int32_t* __restrict__ sel, PrefArgs a,
                                                            uint32_t* __restrict__ err) {
  extern __shared__ int hist[];
  const int bhq = blockIdx.y;
  const int b = bhq / a.Hq, h = bhq - b * a.Hq;
  const int kvh = h / a.g;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t ns = a.ns_cap;
  const bool use_hist = ns <= kHistMax;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  if (use_hist)
    for (int x = threadIdx.x; x < ns; x += 256) hist[x] = 0;
  __syncthreads();
  int* gcount = a.counts + (int64_t)(b * a.Hkv + kvh) * ns;
  if (i < a.n_q) {
    const int64_t row = (int64_t)bhq * a.n_q + i;
    const int64_t ell = (a.q_pos0 + i) / a.S;
    int js[kMaxK];
    bool bad;
    const int n = row_used(sel + row * a.topk, a.topk, ell, js, &bad);
    if (bad) flag_error(err, SSA_DEVERR_BAD_SELECTION);
    for (int r = 0; r < n; ++r) {
      if (use_hist) atomicAdd(&hist[js[r]], 1);
      else atomicAdd(&gcount[js[r]], 1);
    }
  }
  __syncthreads();
  if (use_hist)
    for (int x = threadIdx.x; x < ns; x += 256)
      if (hist[x]) atomicAdd(&gcount[x], hist[x]);
}

// ---------------------------------------------------------------- scan
// One CTA of 1024 threads: exclusive scan of the bucket counts, the span
// tiles, then the local tiles (queries of one local span, 128 / g at a time).
constexpr int kScanThreads = 1024;

__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* tmp, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < (int)(blockDim.x >> 5) ? tmp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    tmp[lane] = w;
  }
  __syncthreads();
  const int64_t before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kScanThreads) prefill_scan_kernel(PrefArgs a) {
  __shared__ int64_t tmp[32];
  __shared__ int64_t carry_e, carry_t;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  if (threadIdx.x == 0) carry_e = carry_t = 0;
  __syncthreads();
  for (int64_t base = 0; base < a.n_buckets; base += kScanThreads) {
    const int64_t bk = base + threadIdx.x;
    const int c = bk < a.n_buckets ? a.counts[bk] : 0;
    const int nt = (c + kTileRows - 1) / kTileRows;
    int64_t tot_e, tot_t;
    const int64_t pe = block_exclusive_scan(c, tmp, &tot_e) + carry_e;
    const int64_t pt = block_exclusive_scan(nt, tmp, &tot_t) + carry_t;
    if (bk < a.n_buckets) {
      a.offsets[bk] = (int)pe;
      a.cursors[bk] = (int)pe;
      for (int t = 0; t < nt; ++t)
        a.tiles[pt + t] = make_int4((int)bk, t * kTileRows, min(kTileRows, c - t * kTileRows), 0);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_e += tot_e;
      carry_t += tot_t;
    }
    __syncthreads();
  }
  // local tiles: for every (b, kv-head) and every span the chunk's queries touch
  const int64_t mq = kTileRows / a.g;
  const int64_t l0 = a.q_pos0 / a.S, l1 = (a.q_pos0 + a.n_q - 1) / a.S;
  const int64_t nspan = l1 - l0 + 1;
  const int64_t bh_n = (int64_t)a.B * a.Hkv;
  for (int64_t base = 0; base < bh_n * nspan; base += kScanThreads) {
    const int64_t e = base + threadIdx.x;
    int64_t qa = 0, qn = 0;
    if (e < bh_n * nspan) {
      const int64_t ell = l0 + e % nspan;
      const int64_t pa = max(a.q_pos0, ell * a.S), pb = min(a.q_pos0 + a.n_q, (ell + 1) * a.S);
      qa = pa - a.q_pos0;
      qn = pb - pa;
    }
    const int64_t nt = qn > 0 ? (qn + mq - 1) / mq : 0;
    int64_t tot;
    const int64_t pt = block_exclusive_scan(nt, tmp, &tot) + carry_t;
    if (e < bh_n * nspan) {
      const int bh = (int)(e / nspan);
      for (int64_t t = 0; t < nt; ++t)
        a.tiles[pt + t] = make_int4(-1 - bh, (int)(qa + t * mq), (int)min(mq, qn - t * mq), 0);
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_t += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) a.ntiles[0] = (int)carry_t;
}

// ---------------------------------------------------------------- scatter
__global__ void __launch_bounds__(256) prefill_scatter_kernel(const int32_t* __restrict__ sel, PrefArgs a) {
  extern __shared__ int sh[];
  const int bhq = blockIdx.y;
  const int b = bhq / a.Hq, h = bhq - b * a.Hq;
  const int kvh = h / a.g;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t ns = a.ns_cap;
  const bool use_hist = ns <= kHistMax;
  int* hist = sh;
  int* base = sh + (use_hist ? ns : 0);
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  if (use_hist)
    for (int x = threadIdx.x; x < ns; x += 256) hist[x] = 0;
  __syncthreads();
  const int64_t bkt0 = (int64_t)(b * a.Hkv + kvh) * ns;
  int js[kMaxK];
  int n = 0;
  const int64_t row = (int64_t)bhq * a.n_q + i;
  if (i < a.n_q) {
    bool bad;
    n = row_used(sel + row * a.topk, a.topk, (a.q_pos0 + i) / a.S, js, &bad);
    if (use_hist)
      for (int r = 0; r < n; ++r) atomicAdd(&hist[js[r]], 1);
  }
  __syncthreads();
  if (use_hist) {
    for (int x = threadIdx.x; x < ns; x += 256) {
      const int c = hist[x];
      base[x] = c ? atomicAdd(&a.cursors[bkt0 + x], c) : 0;
      hist[x] = 0;
    }
  }
  __syncthreads();
  for (int r = 0; r < n; ++r) {
    const int j = js[r];
    const int pos = use_hist ? base[j] + atomicAdd(&hist[j], 1) : atomicAdd(&a.cursors[bkt0 + j], 1);
    a.rows[pos] = (int)((row << 6) | r);
  }
}

// ---------------------------------------------------------------- attend
template <int D>
struct ACfg {
  static constexpr int kRegion = kTileRows * 128;      // 128 rows x 128 bytes
  static constexpr int kQBytes = (D / 64) * kRegion;    // Q tile, D/64 regions
  static constexpr int kKVBytes = (D / 64) * kRegion;   // one K (or V) block of 128 tokens
  // two stages each: a K slot is free once S of its block is done (s_full),
  // a V slot once O += P V of its block is done (p_free); with two stages
  // those barriers can never run two phases ahead of the producer's wait
  static constexpr int kKStages = 2;
  static constexpr int kVStages = 2;
  // small state first (barriers, pair exchange, tile metadata), then the
  // 1024-byte aligned operand buffers: Q[2], K[kKStages], V[kVStages]
  static constexpr int kBarBytes = 256;
  static constexpr int kXchgBytes = 2 * 2 * kTileRows * 4;
  static constexpr int kMetaBytes = 2 * 16 + 2 * kTileRows * 4;
  static constexpr int kSlotBytes = 2 * kTileRows * 8;  // pending tile: partial slot per softmax thread
  static constexpr int kSmallBytes = ((kBarBytes + kXchgBytes + kMetaBytes + kSlotBytes + 1023) / 1024) * 1024;
  static constexpr size_t kSmem =
      1024 + kSmallBytes + 2 * (size_t)kQBytes + (size_t)(kKStages + kVStages) * kKVBytes;
  // tensor memory: S0 [0, 128), S1 [128, 256) (P of a block is written over
  // the S columns it came from), then the two key-half accumulators
  // O0 [256, 256 + D) and O1 [256 + D, 256 + 2 D)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

constexpr int kSoftWarps = 8;      // two warps per tensor-memory lane quarter
constexpr int kTmaWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1, kQWarp = kSoftWarps + 2;
constexpr int kAttThreads = (kSoftWarps + 3) * 32;

struct Tile {
  int kind_bh;  // bucket (>= 0) or -1 - bh
  int row0, nrows;
  int bh;
  int64_t key0, key_end;  // keys [key0, key_end)
  int nkb;
  int64_t i0;              // local tiles: first query index
};

__device__ __forceinline__ Tile decode_tile(const PrefArgs& a, int4 v) {
  Tile x;
  x.kind_bh = v.x;
  if (v.x >= 0) {
    const int64_t bk = v.x;
    x.bh = (int)(bk / a.ns_cap);
    const int64_t j = bk - (int64_t)x.bh * a.ns_cap;
    x.row0 = v.y;
    x.nrows = v.z;
    x.key0 = j * a.S;
    x.key_end = x.key0 + a.S;
    x.i0 = 0;
  } else {
    x.bh = -1 - v.x;
    x.i0 = v.y;
    x.row0 = 0;
    x.nrows = v.z * a.g;
    const int64_t t0 = a.q_pos0 + v.y;
    x.key0 = (t0 / a.S) * a.S;
    x.key_end = t0 + v.z;  // up to the last query's own position
  }
  x.nkb = (int)((x.key_end - x.key0 + kKeyBlk - 1) / kKeyBlk);
  return x;
}

// Row r of a local tile: query i0 + r / g of head kvh * g + r % g.
__device__ __forceinline__ int64_t local_row(const PrefArgs& a, const Tile& x, int r, int64_t* i_out) {
  const int b = x.bh / a.Hkv, kvh = x.bh - b * a.Hkv;
  const int64_t i = x.i0 + r / a.g;
  const int h = kvh * a.g + r % a.g;
  *i_out = i;
  return (int64_t)(b * a.Hq + h) * a.n_q + i;
}

// Warp roles: 0-7 softmax (warps w and w + 4 share the tensor-memory lanes
// of quarter w % 4 and split the key / output columns), 8 TMA producer of
// the K / V blocks, 9 MMA issuer, 10 Q loader.
//
// Block g (a global count of key blocks over this CTA's tiles):
//   S(g) = Q K(g)^T       -> tensor memory S[g % 2]
//   P(g) = 2^(S c - m)    -> tensor memory P[g % 2] (16-bit, written by the softmax warps)
//   O   += P(g) V(g)      A operand read from tensor memory
// The softmax of block g waits only for O += P(g - 2) V (its P buffer), or
// for O += P(g - 1) V when it must rescale O.  The Q loader fills the other
// Q buffer while a tile runs, so the next tile's first S can start while
// the softmax warps write the previous tile's partials.
template <int DT, int D>
__global__ void __launch_bounds__(kAttThreads, 1)
    prefill_attend_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const void* __restrict__ Q, PrefArgs a, uint32_t* __restrict__ err) {
  using C = ACfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(base);
  uint64_t* q_full = bar + 0;    // [2] Q tile and its metadata loaded
  uint64_t* q_empty = bar + 2;   // [2] last S of the tile done + partials written
  uint64_t* k_full = bar + 4;    // [2]
  uint64_t* v_full = bar + 6;    // [2]
  uint64_t* s_full = bar + 8;    // [2] S of the buffer's last block done (its K slot is free)
  uint64_t* p_full = bar + 10;   // [2 buffers][2 halves]
  uint64_t* p_free = bar + 14;   // [2] O += P V of the buffer's last block done (its V slot is free)
  uint64_t* o_free = bar + 24;   // O read out by the epilogue
  uint64_t* drain = bar + 25;    // every MMA issued has completed
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(bar + 26);
  volatile int* abort = reinterpret_cast<volatile int*>(bar + 27);
  float* xchg = reinterpret_cast<float*>(base + C::kBarBytes);   // [2 halves][m, l][128 rows]
  int4* tinfo = reinterpret_cast<int4*>(base + C::kBarBytes + C::kXchgBytes);  // [2] tile entries
  int* meta = reinterpret_cast<int*>(tinfo + 2);                  // [2][128] bucket entries or -1
  int64_t* pslot = reinterpret_cast<int64_t*>(meta + 2 * kTileRows);  // [256] pending partial slot or -1
  uint8_t* sQ = base + C::kSmallBytes;
  uint8_t* sK = sQ + 2 * C::kQBytes;
  uint8_t* sV = sK + C::kKStages * C::kKVBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&q_full[s], 1);
      ptx::mbar_init(&q_empty[s], 1 + kSoftWarps);
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&s_full[s], 1);
      ptx::mbar_init(&p_free[s], 1);
      for (int h = 0; h < 2; ++h) ptx::mbar_init(&p_full[2 * s + h], kSoftWarps / 2);
    }
    ptx::mbar_init(o_free, kSoftWarps);
    ptx::mbar_init(drain, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::alloc(tmem_base, C::kTmemCols);
  if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_base;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int ntiles = a.ntiles[0];

  auto fail = [&](uint32_t bit) {
    flag_error(err, bit);
    *abort = 1;
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------ K / V producer
    // Loads in the order the MMAs consume them: K(g), then V(g - 1).
    if (lane == 0) {
      int64_t g = 0;
      int prev_bh = 0, prev_y = 0;
      bool have_prev = false, ok = true;
      auto load_v = [&](int64_t gv, int bh, int y) -> bool {
        const int st = (int)(gv % C::kVStages);
        if (gv >= 2 && !ptx::mbar_wait(&p_free[(gv - 2) & 1], (uint32_t)(((gv - 2) >> 1) & 1))) return false;
        ptx::mbar_arrive_expect_tx(&v_full[st], C::kKVBytes);
#pragma unroll
        for (int r = 0; r < D / 64; ++r)
          ptx::tma_load_3d(sV + st * C::kKVBytes + r * C::kRegion, &tmV, &v_full[st], r * 64, y, bh);
        return true;
      };
      for (int t = blockIdx.x; t < ntiles && ok && !*abort; t += gridDim.x) {
        const Tile x = decode_tile(a, a.tiles[t]);
        for (int kb = 0; kb < x.nkb && ok; ++kb, ++g) {
          const int st = (int)(g % C::kKStages);
          if (g >= 2 && !ptx::mbar_wait(&s_full[(g - 2) & 1], (uint32_t)(((g - 2) >> 1) & 1))) {
            ok = false;
            break;
          }
          const int y = (int)(x.key0 + (int64_t)kb * kKeyBlk);
          ptx::mbar_arrive_expect_tx(&k_full[st], C::kKVBytes);
#pragma unroll
          for (int r = 0; r < D / 64; ++r)
            ptx::tma_load_3d(sK + st * C::kKVBytes + r * C::kRegion, &tmK, &k_full[st], r * 64, y, x.bh);
          if (have_prev && !load_v(g - 1, prev_bh, prev_y)) {
            ok = false;
            break;
          }
          prev_bh = x.bh;
          prev_y = y;
          have_prev = true;
        }
      }
      if (ok && have_prev) ok = load_v(g - 1, prev_bh, prev_y);
      if (!ok) fail(SSA_DEVERR_WAIT_TIMEOUT);
      // let every load this thread issued land before the CTA can exit
      const int64_t nk = g, nv = have_prev ? g : 0;
      for (int s = 0; s < C::kKStages; ++s) {
        if (nk <= s) break;
        const int64_t last = s + ((nk - 1 - s) / C::kKStages) * C::kKStages;
        if (!ptx::mbar_wait(&k_full[s], (uint32_t)((last / C::kKStages) & 1))) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      }
      for (int s = 0; s < C::kVStages; ++s) {
        if (nv <= s) break;
        const int64_t last = s + ((nv - 1 - s) / C::kVStages) * C::kVStages;
        if (!ptx::mbar_wait(&v_full[s], (uint32_t)((last / C::kVStages) & 1))) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      }
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------ Q loader
    // Gathers the tile's 128 query rows into the swizzled K-major Q buffer
    // and publishes the tile entry and the rows' bucket entries.
    int tcount = 0;
    for (int t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++tcount) {
      const int qb = tcount & 1;
      if (tcount >= 2 && !ptx::mbar_wait(&q_empty[qb], (uint32_t)(((tcount - 2) >> 1) & 1))) {
        fail(SSA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      const int4 v = a.tiles[t];
      const Tile x = decode_tile(a, v);
      if (lane == 0) tinfo[qb] = v;
      const int64_t off0 = x.kind_bh >= 0 ? (int64_t)a.offsets[x.kind_bh] + x.row0 : 0;
      uint8_t* q = sQ + qb * C::kQBytes;
#pragma unroll 1
      for (int rr = 0; rr < kTileRows / 32; ++rr) {
        const int r = rr * 32 + lane;
        int64_t qrow = -1;
        int entry = -1;
        if (r < x.nrows) {
          if (x.kind_bh >= 0) {
            const int e = a.rows[off0 + r];
            const int64_t row = (int64_t)(e >> 6);
            if (e < 0 || row >= (int64_t)a.B * a.Hq * a.n_q || (e & 63) >= a.topk) {
              flag_error(err, SSA_DEVERR_OVERFLOW);
            } else {
              qrow = row;
              entry = e;
            }
          } else {
            int64_t i;
            qrow = local_row(a, x, r, &i);
          }
        }
        meta[qb * kTileRows + r] = entry;
        const uint8_t* src = static_cast<const uint8_t*>(Q) + (qrow < 0 ? 0 : qrow) * (int64_t)D * 2;
        const uint32_t n = qrow < 0 ? 0u : 16u;
        const uint32_t rsw = (uint32_t)(r & 7);
#pragma unroll
        for (int ch = 0; ch < D / 8; ++ch) {
          uint8_t* dst = q + (ch >> 3) * C::kRegion + r * 128 + ((((uint32_t)ch & 7) ^ rsw) << 4);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
                       "l"(src + ch * 16), "r"(n)
                       : "memory");
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&q_full[qb]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int ab16 = DT == DT_BF16 ? 1 : 0;
      const uint32_t id_qk = tc::idesc_f16(128, kKeyBlk, ab16, 0, 0);
      const uint32_t id_pv = tc::idesc_f16(128, D, ab16, 0, 1);
      const uint32_t aQ0 = ptx::smem_u32(sQ), aK = ptx::smem_u32(sK), aV = ptx::smem_u32(sV);
      int64_t g = 0;
      int64_t pend = -1;        // block whose O += P V is still to be issued
      bool pend_first = false;  // ... first block of its tile (overwrites O)
      int pend_tile = 0;
      // O_h += P_h V_h for the two key halves h of block gg: P_h sits in
      // tensor memory over the S columns of its half, V_h is rows
      // [64 h, 64 h + 64) of the block's V tile.
      auto issue_pv = [&](int64_t gg, bool first, int tc_) -> bool {
        if (first && tc_ > 0 && !ptx::mbar_wait(o_free, (uint32_t)((tc_ - 1) & 1))) return false;
        const int pb = (int)(gg & 1), sv = (int)(gg % C::kVStages);
        const uint32_t par = (uint32_t)((gg >> 1) & 1);
        if (!ptx::mbar_wait(&v_full[sv], (uint32_t)((gg / C::kVStages) & 1))) return false;
        const uint32_t vbase = aV + sv * C::kKVBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!ptx::mbar_wait(&p_full[2 * pb + h], par)) return false;
          tc::fence_after();
          const uint32_t tP = tmem + pb * 128 + h * 64;
          const uint32_t tOh = tmem + C::kColO + h * D;
#pragma unroll
          for (int k = 0; k < kKeyBlk / 32; ++k) {
            const uint64_t vd = tc::sdesc_sw128(vbase + (h * (kKeyBlk / 32) + k) * 2048, C::kRegion, 1024);
            tc::mma_ts(tOh, tP + k * 8, vd, id_pv, (first && k == 0) ? 0u : 1u);
          }
        }
        tc::commit(&p_free[pb]);
        return true;
      };
      bool ok = true;
      int tcount = 0;
      for (int t = blockIdx.x; t < ntiles && ok && !*abort; t += gridDim.x, ++tcount) {
        const int qb = tcount & 1;
        if (!ptx::mbar_wait(&q_full[qb], (uint32_t)((tcount >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after();
        const Tile x = decode_tile(a, tinfo[qb]);
        const uint32_t aQ = aQ0 + qb * C::kQBytes;
        for (int kb = 0; kb < x.nkb && ok; ++kb, ++g) {
          const int sb = (int)(g & 1);
          const int sk = (int)(g % C::kKStages);
          // S(g) overwrites S[g % 2], which holds P(g - 2): its O += P V was
          // issued before, and the tensor pipe runs this thread's MMAs in order
          ok = ptx::mbar_wait(&k_full[sk], (uint32_t)((g / C::kKStages) & 1));
          if (!ok) break;
          tc::fence_after();
          const uint32_t kbase = aK + sk * C::kKVBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t qd = tc::sdesc_sw128(aQ + (k >> 2) * C::kRegion + (k & 3) * 32, 16, 1024);
            const uint64_t kd = tc::sdesc_sw128(kbase + (k >> 2) * C::kRegion + (k & 3) * 32, 16, 1024);
            tc::mma(tmem + sb * 128, qd, kd, id_qk, k > 0 ? 1u : 0u);
          }
          tc::commit(&s_full[sb]);
          if (kb == x.nkb - 1) tc::commit(&q_empty[qb]);
          if (pend >= 0) ok = issue_pv(pend, pend_first, pend_tile);
          pend = g;
          pend_first = kb == 0;
          pend_tile = tcount;
        }
      }
      if (ok && pend >= 0 && !*abort) ok = issue_pv(pend, pend_first, pend_tile);
      if (!ok) fail(SSA_DEVERR_WAIT_TIMEOUT);
      // every MMA issued completes before the tensor memory is released
      tc::commit(drain);
      if (!ptx::mbar_wait(drain, 0)) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------ softmax warps
    // Warp (quarter, half) owns tensor-memory lanes 32 quarter .. + 31 (its
    // rows) and the keys of one half of every block.  It keeps its own
    // running max and sum for its half and writes P of its half over the S
    // columns it read; O_half accumulates only that half's keys.  The two
    // halves of a row meet once per tile, in the epilogue: with M = max(m0,
    // m1), O = (2^(m0 - M) O0 + 2^(m1 - M) O1) / (2^(m0 - M) l0 + 2^(m1 - M) l1).
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int pair_bar = 1 + quarter;  // named barrier of the warp pair
    const float c = a.scale_log2e;
    constexpr int KH = kKeyBlk / 2;    // key columns per half
    constexpr int OH = D / 2;          // output columns this warp writes
    const uint32_t tOown = tmem + C::kColO + half * D + lane_off;   // this half's accumulator
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    int64_t gb = 0;
    int tcount = 0;
    // the previous tile's epilogue, still to run
    // (its rows' m and l wait in xchg, its partial slots in pslot: only the
    // flag stays in registers while the next tile runs)
    bool pend = false;
    // Epilogue of the pending tile: combine the halves' accumulators into
    // this warp's output columns [half * D / 2, + D / 2), normalised, to the
    // row's partial slot.  Returns false when a bounded wait gave up.
    auto epilogue = [&]() -> bool {
      pend = false;
      const int64_t glast = gb - 1;  // the pending tile's last block: every call site has gb one past it
      if (!ptx::mbar_wait(&p_free[glast & 1], (uint32_t)((glast >> 1) & 1))) return false;
      tc::fence_after();
      pair_sync();
      const float m0 = xchg[r], l0 = xchg[128 + r];
      const float m1 = xchg[256 + r], l1 = xchg[256 + 128 + r];
      const int64_t slot = pslot[threadIdx.x];
      pair_sync();
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : ptx::ex2(m0 - M);
      const float w1 = m1 == -INFINITY ? 0.f : ptx::ex2(m1 - M);
      const float lt = l0 * w0 + l1 * w1;
      const float inv = 1.f / lt;
      const float s0 = w0 * inv, s1 = w1 * inv;
      const uint32_t tO0 = tmem + C::kColO + lane_off + half * OH;
      const uint32_t tO1 = tO0 + D;
      uint16_t* dst = a.po + slot * D + half * OH;  // 32-byte aligned: the slot is D * 2 bytes
      // 32 columns at a time: read both accumulators, combine, store
#pragma unroll
      for (int q = 0; q < OH / 32; ++q) {
        uint32_t o0[32], o1[32], pk[16];
        tc::ld32x2(tO0 + q * 32, o0, tO1 + q * 32, o1);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = ptx::pack2<DT>(
              __uint_as_float(o0[2 * j]) * s0 + __uint_as_float(o1[2 * j]) * s1,
              __uint_as_float(o0[2 * j + 1]) * s0 + __uint_as_float(o1[2 * j + 1]) * s1);
        if (slot >= 0) {
          ptx::st_global_v8(dst + 32 * q, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          ptx::st_global_v8(dst + 32 * q + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_relaxed(o_free);
      if (slot >= 0 && half == 0) a.pml[slot] = make_float2(M, lt);
      return true;
    };
    // No abort check here: both warps of a pair must walk the same tiles
    // (they meet at a named barrier per tile); they leave only through
    // bounded waits, which time out together.
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tcount) {
      const int qb = tcount & 1;
      if (!ptx::mbar_wait(&q_full[qb], (uint32_t)((tcount >> 1) & 1))) {
        fail(SSA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      const Tile x = decode_tile(a, tinfo[qb]);
      // row identity
      int64_t qrow = -1;  // row of Q / sel / partials
      int rank = a.topk;
      int64_t tpos = 0;   // query position (local tiles)
      if (x.kind_bh >= 0) {
        const int e = meta[qb * kTileRows + r];
        if (e >= 0) {
          qrow = (int64_t)(e >> 6);
          rank = e & 63;
        }
      } else if (r < x.nrows) {
        int64_t i;
        qrow = local_row(a, x, r, &i);
        tpos = a.q_pos0 + i;
      }
      // the tile entry and row entries are in registers now: the loader may
      // reuse them (with the Q buffer, once the tile's last S is done)
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&q_empty[qb]);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int kb = 0; kb < x.nkb && ok; ++kb) {
        const int64_t g = gb + kb;
        const int st = (int)(g & 1);
        // the previous tile's epilogue, once this tile's first P is out
        if (kb == 1 && pend && !epilogue()) {
          ok = false;
          break;
        }
        if (!ptx::mbar_wait(&s_full[st], (uint32_t)((g >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after();
        // valid keys of this block: [0, klim)
        const int64_t kstart = x.key0 + (int64_t)kb * kKeyBlk;
        int64_t klim = x.key_end - kstart;
        if (x.kind_bh < 0) klim = min(klim, tpos - kstart + 1);
        const int64_t hlim = klim - half * KH;  // valid keys of this half
        const bool partial = hlim < KH;
        static_assert(KH == 64, "one 64-column load per half row");
        const uint32_t tS = tmem + st * 128 + lane_off + half * KH;
        uint32_t sr[64];
        tc::ld64(tS, sr);
        float mx = -INFINITY;
        if (partial) {
#pragma unroll
          for (int j = 0; j < KH; ++j)
            if (j < hlim) mx = fmaxf(mx, __uint_as_float(sr[j]));
        } else {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int j = 0; j < KH; j += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              m4[u] = ptx::max3(m4[u], __uint_as_float(sr[j + 2 * u]), __uint_as_float(sr[j + 2 * u + 1]));
          mx = ptx::max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
        }
        mx *= c;
        // rescale O_half only when this half's max grows by more than 2^8
        float m_new = m;
        if (kb == 0) {
          m_new = mx;
        } else if (mx > m + kRescaleLog2) {
          m_new = mx;
        }
        const bool need = kb > 0 && m_new != m;
        if (__any_sync(0xffffffffu, need)) {
          // O_half += P_half(g - 1) V must be complete before it is rescaled
          if (!ptx::mbar_wait(&p_free[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc::fence_after();
          const float f = need ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t rr[32];
            tc::ld32(tOown + q * 32, rr);
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
            tc::st32(tOown + q * 32, rr);
          }
          l *= f;
        }
        m = m_new;
        const float nb = m == -INFINITY ? 0.f : -m;
        // P_half = 2^(s c - m) as 16-bit pairs, over the S columns just read
        uint32_t pk[32];
        if (!partial) {
          // two partial sums keep the adds off one dependency chain
          float la = 0.f, lb = 0.f;
#pragma unroll
          for (int j = 0; j < KH; j += 2) {
            const float p0 = ptx::ex2(fmaf(__uint_as_float(sr[j]), c, nb));
            const float p1 = ptx::ex2(fmaf(__uint_as_float(sr[j + 1]), c, nb));
            la += p0;
            lb += p1;
            pk[j / 2] = ptx::pack2<DT>(p0, p1);
          }
          l += la + lb;
        } else {
#pragma unroll
          for (int j = 0; j < KH; j += 2) {
            const float p0 = j < hlim ? ptx::ex2(fmaf(__uint_as_float(sr[j]), c, nb)) : 0.f;
            const float p1 = j + 1 < hlim ? ptx::ex2(fmaf(__uint_as_float(sr[j + 1]), c, nb)) : 0.f;
            l += p0 + p1;
            pk[j / 2] = ptx::pack2<DT>(p0, p1);
          }
        }
        tc::st32(tS, pk);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_relaxed(&p_full[2 * st + half]);
      }
      if (!ok) {
        fail(SSA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      // a one-block tile has not run the previous epilogue yet
      if (ok && pend && !epilogue()) ok = false;
      if (!ok) {
        fail(SSA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      // this tile's epilogue runs after the next tile's first block (or
      // after the last tile), so that waiting for its last O += P V overlaps
      // the next tile's softmax
      pend = true;
      xchg[half * 256 + r] = m;
      xchg[half * 256 + 128 + r] = l;
      pslot[threadIdx.x] = qrow >= 0 ? qrow * (a.topk + 1) + rank : -1;
      gb += x.nkb;
    }
    if (pend && !epilogue()) fail(SSA_DEVERR_WAIT_TIMEOUT);
  }
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------- merge
// One warp per row of Q: its used spans (sel order) then its local span.
// The partials of a row are read in batches of kMergeBatch slots with all of
// a batch's loads in flight at once (one memory round trip per batch; one
// batch covers topk <= 16).
constexpr int kMergeBatch = 17;

template <int DT, int E>
__device__ __forceinline__ void widen_partial(const uint16_t* src, float (&v)[E]) {
  if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if constexpr (DT == DT_BF16) {
        v[2 * k] = bf16_bits_to_f32(ww[k] & 0xffffu);
        v[2 * k + 1] = __uint_as_float(ww[k] & 0xffff0000u);
      } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[k]));
        v[2 * k] = f.x;
        v[2 * k + 1] = f.y;
      }
    }
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    if constexpr (DT == DT_BF16) {
      v[0] = bf16_bits_to_f32(w & 0xffffu);
      v[1] = __uint_as_float(w & 0xffff0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
      v[0] = f.x;
      v[1] = f.y;
    }
  }
}

template <int DT, int D>
__device__ __forceinline__ void merge_row(const int32_t* __restrict__ sel, const PrefArgs& a, void* __restrict__ O,
                                          float* __restrict__ lse, int64_t row, int lane) {
  constexpr int E = D / 32;
  const int64_t i = row % a.n_q;
  const int64_t ell = (a.q_pos0 + i) / a.S;
  const int32_t* srow = sel + row * a.topk;
  // the sel row and the partials are loaded together: every slot of the row
  // (ranks 0 .. topk, the local span last) is read whether used or not, and
  // only the used ones (the sel row's valid prefix, then the local span) are
  // combined, in rank order
  const int j0 = lane < a.topk ? srow[lane] : -1;
  const int j1 = lane + 32 < a.topk ? srow[lane + 32] : -1;
  const int nslot = a.topk + 1;
  const int64_t base = row * (a.topk + 1);
  float M = -INFINITY, Ls = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  int used = -1;
  for (int s0 = 0; s0 < nslot; s0 += kMergeBatch) {
    float2 ml[kMergeBatch];
    uint2 raw[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int s = s0 + u;
      if (s < nslot) {
        ml[u] = a.pml[base + s];
        const uint16_t* src = a.po + (base + s) * D + lane * E;
        if constexpr (E == 4) {
          raw[u] = *reinterpret_cast<const uint2*>(src);
        } else {
          raw[u] = make_uint2(*reinterpret_cast<const uint32_t*>(src), 0u);
        }
      }
    }
    if (used < 0) {
      bool bad;
      used = warp_sel_prefix(j0, j1, lane, a.topk, ell, &bad);
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int s = s0 + u;
      if (s >= nslot || (s < a.topk && s >= used)) continue;
      float v[E];
      widen_partial<DT, E>(reinterpret_cast<const uint16_t*>(&raw[u]), v);
      const float Mn = fmaxf(M, ml[u].x);
      const float fa = exp2f(M - Mn), fb = exp2f(ml[u].x - Mn) * ml[u].y;
      Ls = Ls * fa + fb;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = acc[e] * fa + v[e] * fb;
      M = Mn;
    }
  }
  const float inv = 1.f / Ls;
#pragma unroll
  for (int e = 0; e < E; ++e) store_elem<DT>(O, row * D + lane * E + e, acc[e] * inv);
  if (lse && lane == 0) lse[row] = M * kLn2 + logf(Ls);
}

template <int DT, int D>
__global__ void __launch_bounds__(256, 2) prefill_merge_kernel(const int32_t* __restrict__ sel, PrefArgs a,
                                                            void* __restrict__ O, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int64_t n_rows = (int64_t)a.B * a.Hq * a.n_q;
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < n_rows; row += (int64_t)gridDim.x * 8)
    merge_row<DT, D>(sel, a, O, lse, row, lane);
}

PrefArgs make_args(const Problem& pr, int64_t n_q, int64_t q_pos0, void* ws, const PrefLayout& lay) {
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  PrefArgs a;
  a.counts = reinterpret_cast<int*>(w8 + lay.counts);
  a.offsets = reinterpret_cast<int*>(w8 + lay.offsets);
  a.cursors = reinterpret_cast<int*>(w8 + lay.cursors);
  a.ntiles = reinterpret_cast<int*>(w8 + lay.ntiles);
  a.tiles = reinterpret_cast<int4*>(w8 + lay.tiles);
  a.rows = reinterpret_cast<int*>(w8 + lay.rows);
  a.pml = reinterpret_cast<float2*>(w8 + lay.pml);
  a.po = reinterpret_cast<uint16_t*>(w8 + lay.po);
  a.B = pr.B;
  a.Hq = pr.Hq;
  a.Hkv = pr.Hkv;
  a.g = pr.g;
  a.d = pr.d;
  a.S = pr.S;
  a.topk = pr.topk;
  a.n_q = n_q;
  a.q_pos0 = q_pos0;
  a.ns_cap = pr.ns_cap;
  a.n_buckets = lay.n_buckets;
  a.scale_log2e = pr.scale * kLog2e;
  return a;
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const void* K,
                         const void* V, const int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st) {
  using C = ACfg<D>;
  const PrefLayout lay = pref_layout(pr, n_q);
  const PrefArgs a = make_args(pr, n_q, q_pos0, ws, lay);
  uint32_t* err = ws_error(ws);
  cudaError_t e = cudaMemsetAsync(a.counts, 0, lay.n_buckets * 4, st);
  if (e != cudaSuccess) return e;
  CUtensorMap tmK, tmV;
  e = make_kv_tmap(&tmK, K, pr.dtype, D, pr.L, pr.L_cap, (int64_t)pr.B * pr.Hkv, kKeyBlk);
  if (e != cudaSuccess) return e;
  e = make_kv_tmap(&tmV, V, pr.dtype, D, pr.L, pr.L_cap, (int64_t)pr.B * pr.Hkv, kKeyBlk);
  if (e != cudaSuccess) return e;
  const size_t hist_bytes = pr.ns_cap <= kHistMax ? (size_t)pr.ns_cap * 4 : 0;
  const dim3 grid_rows((unsigned)((n_q + 255) / 256), (unsigned)(pr.B * pr.Hq));
  e = launch_pdl(prefill_count_kernel, grid_rows, dim3(256), hist_bytes, st, sel, a, err);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_scatter_kernel, grid_rows, dim3(256), 2 * hist_bytes, st, sel, a);
  if (e != cudaSuccess) return e;
  static bool attr_done[kMaxDevices] = {};
  e = ensure_smem_attr(prefill_attend_kernel<DT, D>, C::kSmem, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_attend_kernel<DT, D>, dim3(device_sm_count()), dim3(kAttThreads), C::kSmem, st,
                 tmK, tmV, Q, a, err);
  if (e != cudaSuccess) return e;
  const int64_t n_rows = (int64_t)pr.B * pr.Hq * n_q;
  const int64_t merge_ctas = min((n_rows + 7) / 8, (int64_t)device_sm_count() * 8);
  return launch_pdl(prefill_merge_kernel<DT, D>, dim3((unsigned)merge_ctas), dim3(256), 0, st, sel, a, O, lse);
}

}  // namespace

bool prefill_fast_supported(const Problem& pr) {
  return (pr.dtype == DT_BF16 || pr.dtype == DT_F16) && (pr.d == 64 || pr.d == 128) && pr.g <= kMaxG &&
         (kTileRows % pr.g) == 0 && pr.topk <= kMaxK && pr.L > 0;
}

size_t prefill_ws_bytes(const Problem& pr, int64_t n_q) {
  // row ids are packed with the rank into 32 bits
  if ((int64_t)pr.B * pr.Hq * n_q >= (1ll << 25)) return 0;
  return pref_layout(pr, n_q).total - kWsHeader;
}

cudaError_t launch_attend_prefill(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                                  const void* K, const void* V, const int32_t* sel, void* O, float* lse,
                                  void* ws, cudaStream_t st) {
  if (pr.d == 128) {
    if (pr.dtype == DT_BF16) return launch_typed<DT_BF16, 128>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws, st);
    return launch_typed<DT_F16, 128>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws, st);
  }
  if (pr.dtype == DT_BF16) return launch_typed<DT_BF16, 64>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws, st);
  return launch_typed<DT_F16, 64>(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws, st);
}

}  // namespace ssa

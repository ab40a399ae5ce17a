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
//  scan     one CTA: bucket offsets, the table of tile pairs (span pairs,
//           then local pairs): two tiles of 128 rows that share one key range
//  scatter  writes each row's id and its rank in the sel row into its
//           bucket
//  attend   persistent, one CTA per SM, twelve warps, one pair at a time.
//           Two loader warps gather the pair's query rows into 128-byte
//           swizzled K-major Q buffers ahead of use (tile A's double
//           buffered, tile B's too for spans of 512 tokens or more); a TMA
//           warp streams the shared key / value blocks of 128 tokens
//           through a four-slot ring (three with tile B's two); one thread
//           issues tcgen05.mma, alternating the tiles: S = Q K^T into
//           tensor memory, then O += P V with P read from tensor memory.  Eight
//           softmax warps (four per tile, one row per thread) turn S into
//           P = 2^(S c - m) (16-bit, written over S), rescale O only when
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
// candidate spans; anything else but -1 after it is an error), one thread:
// f(rank, span) for each, in order.  Returns their count; the rank of a used
// entry is its index in the row.
template <class F>
__device__ __forceinline__ int row_used(const int32_t* row, int topk, int64_t ell, bool* bad, F&& f) {
  int n = 0;
  int64_t prev = -1;
  bool stop = false;
  *bad = false;
  for (int r = 0; r < topk; ++r) {
    const int j = row[r];
    if (!stop && j >= 0 && j < ell && j > prev) {
      f(n++, j);
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
    bool bad;
    row_used(sel + row * a.topk, a.topk, ell, &bad, [&](int, int j) {
      if (use_hist) atomicAdd(&hist[j], 1);
      else atomicAdd(&gcount[j], 1);
    });
    if (bad) flag_error(err, SSA_DEVERR_BAD_SELECTION);
  }
  __syncthreads();
  if (use_hist)
    for (int x = threadIdx.x; x < ns; x += 256)
      if (hist[x]) atomicAdd(&gcount[x], hist[x]);
}

// ---------------------------------------------------------------- scan
// One CTA of 1024 threads: exclusive scan of the bucket counts, then the
// table of tile pairs.  A pair is two tiles of 128 rows that share one key
// range: rows [256 p, 256 p + 128) and [256 p + 128, 256 p + 256) of a
// bucket (entry {bucket, 256 p, rows of tile A, rows of tile B}), then, per
// local span, 2 * 128 / g consecutive queries (entry {-1 - bh, first query,
// queries of tile A, queries of tile B}).  Tile B may be empty.
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
    const int nt = (c + 2 * kTileRows - 1) / (2 * kTileRows);
    int64_t tot_e, tot_t;
    const int64_t pe = block_exclusive_scan(c, tmp, &tot_e) + carry_e;
    const int64_t pt = block_exclusive_scan(nt, tmp, &tot_t) + carry_t;
    if (bk < a.n_buckets) {
      a.offsets[bk] = (int)pe;
      a.cursors[bk] = (int)pe;
      for (int t = 0; t < nt; ++t) {
        const int r0 = 2 * t * kTileRows;
        a.tiles[pt + t] = make_int4((int)bk, r0, min(kTileRows, c - r0), max(0, min(kTileRows, c - r0 - kTileRows)));
      }
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
    const int64_t nt = qn > 0 ? (qn + 2 * mq - 1) / (2 * mq) : 0;
    int64_t tot;
    const int64_t pt = block_exclusive_scan(nt, tmp, &tot) + carry_t;
    if (e < bh_n * nspan) {
      const int bh = (int)(e / nspan);
      for (int64_t t = 0; t < nt; ++t) {
        const int64_t q0 = t * 2 * mq;
        a.tiles[pt + t] = make_int4(-1 - bh, (int)(qa + q0), (int)min(mq, qn - q0),
                                    (int)max((int64_t)0, min(mq, qn - q0 - mq)));
      }
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
  int n = 0;
  const int64_t row = (int64_t)bhq * a.n_q + i;
  const int32_t* srow = sel + (i < a.n_q ? row : 0) * a.topk;
  if (i < a.n_q) {
    bool bad;
    n = row_used(srow, a.topk, (a.q_pos0 + i) / a.S, &bad, [&](int, int j) {
      if (use_hist) atomicAdd(&hist[j], 1);
    });
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
  // the used entries are the row's first n
  for (int r = 0; r < n; ++r) {
    const int j = srow[r];
    const int pos = use_hist ? base[j] + atomicAdd(&hist[j], 1) : atomicAdd(&a.cursors[bkt0 + j], 1);
    a.rows[pos] = (int)((row << 6) | r);
  }
}

// ---------------------------------------------------------------- attend
// QB: tile B's Q buffers.  Seven 128-row operand buffers fit in shared
// memory: tile A's two Q buffers, then either one for tile B and a four-slot
// K / V ring (QB = 1), or two for tile B and a three-slot ring (QB = 2).
// Long spans (many key blocks per pair) gain from tile B's next rows loading
// during the pair; short ones from the deeper ring, which reaches into the
// next pair's blocks.
template <int D, int QB>
struct ACfg {
  static constexpr int kRegion = kTileRows * 128;       // 128 rows x 128 bytes
  static constexpr int kQTile = (D / 64) * kRegion;      // one 128-row Q tile
  static constexpr int kKV = (D / 64) * kRegion;         // one K or V block of 128 tokens
  // one ring for both: K(0), V(0), K(1), V(1), ...  A K slot is free once
  // both tiles' S of its block are done, a V slot once both P V are.  Tile
  // A's Q is double buffered; with one buffer, tile B's next rows load once
  // its last S of the pair is done.
  static constexpr int kSlots = QB == 2 ? 3 : 4;
  static constexpr size_t kOperands = (2 + QB) * (size_t)kQTile + (size_t)kSlots * kKV;
  static constexpr int kSmallBytes = 512;                // barriers and the two pair entries
  static constexpr size_t kSmem = 1024 + kOperands + kSmallBytes;
  // tensor memory: S_A [0, 128), S_B [128, 256) (the P of a block is written
  // over the S columns it came from), O_A [256, 256 + D), O_B [256 + D, 256 + 2 D)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

// Every layout fits the 227 KB of shared memory a CTA may use, and the small
// block holds the barriers (words 0-24), the tensor-memory address (25), the
// abort flag (26) and the two pair entries (words 28-31).
static_assert(ACfg<128, 1>::kSmem <= 227 * 1024 && ACfg<128, 2>::kSmem <= 227 * 1024, "attend layout too large");
static_assert(ACfg<64, 1>::kSmem <= 227 * 1024 && ACfg<64, 2>::kSmem <= 227 * 1024, "attend layout too large");
static_assert(32 * 8 <= ACfg<128, 1>::kSmallBytes, "attend barrier block too small");

constexpr int kSoftWarps = 8;      // warps 0-3: tile A, 4-7: tile B (one lane quarter each)
constexpr int kTmaWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1, kQWarp = kSoftWarps + 2;  // Q loaders: 10, 11
constexpr int kAttThreads = (kSoftWarps + 4) * 32;

struct Pair {
  int kind_bh;          // bucket (>= 0) or -1 - bh
  int bh;
  int row0;             // span pairs: bucket row of tile A's first row (tile B: 128 rows on)
  int n0, n1;           // rows of tiles A and B (0: no tile B)
  __device__ __forceinline__ int n(int t) const { return t ? n1 : n0; }
  int64_t i0;           // local pairs: tile A's first query (tile B: 128 / g queries on)
  int64_t key0, key_end;  // keys [key0, key_end)
  int nkb;
};

__device__ __forceinline__ Pair decode_pair(const PrefArgs& a, int4 v) {
  Pair x;
  x.kind_bh = v.x;
  if (v.x >= 0) {
    const int64_t bk = v.x;
    x.bh = (int)(bk / a.ns_cap);
    const int64_t j = bk - (int64_t)x.bh * a.ns_cap;
    x.row0 = v.y;
    x.n0 = v.z;
    x.n1 = v.w;
    x.key0 = j * a.S;
    x.key_end = x.key0 + a.S;
    x.i0 = 0;
  } else {
    x.bh = -1 - v.x;
    x.i0 = v.y;
    x.row0 = 0;
    x.n0 = v.z * a.g;
    x.n1 = v.w * a.g;
    const int64_t t0 = a.q_pos0 + v.y;
    x.key0 = (t0 / a.S) * a.S;
    const int64_t mq = kTileRows / a.g;
    const int64_t last = v.w > 0 ? v.y + mq + v.w - 1 : v.y + v.z - 1;  // last query of the pair
    x.key_end = a.q_pos0 + last + 1;
  }
  x.nkb = (int)((x.key_end - x.key0 + kKeyBlk - 1) / kKeyBlk);
  return x;
}

// Row r of tile t (0 = A, 1 = B) of a pair: its row of Q / sel / partials
// (-1 when the tile has no such row), its rank in the row's sel (topk for the
// local span) and, for local pairs, its query position.
__device__ __forceinline__ int64_t pair_row(const PrefArgs& a, const Pair& x, int t, int r, int* rank,
                                            int64_t* tpos, uint32_t* err) {
  *rank = a.topk;
  *tpos = x.key_end - 1;
  if (r >= x.n(t)) return -1;
  if (x.kind_bh >= 0) {
    const int e = a.rows[(int64_t)a.offsets[x.kind_bh] + x.row0 + t * kTileRows + r];
    const int64_t row = (int64_t)(e >> 6);
    if (e < 0 || row >= (int64_t)a.B * a.Hq * a.n_q || (e & 63) >= a.topk) {
      flag_error(err, SSA_DEVERR_OVERFLOW);
      return -1;
    }
    *rank = e & 63;
    return row;
  }
  const int b = x.bh / a.Hkv, kvh = x.bh - b * a.Hkv;
  const int64_t i = x.i0 + (int64_t)t * (kTileRows / a.g) + r / a.g;
  const int h = kvh * a.g + r % a.g;
  *tpos = a.q_pos0 + i;
  return (int64_t)(b * a.Hq + h) * a.n_q + i;
}

// Warp roles: 0-3 softmax of tile A and 4-7 of tile B (warp w owns tensor-
// memory lanes 32 (w % 4) .. + 31: one row per thread), 8 TMA producer of the
// K / V blocks, 9 MMA issuer, 10 and 11 Q loaders of tiles A and B.
//
// Both tiles of a pair stream the same key blocks.  Per block b the MMA
// thread issues, in this order,
//   O_A += P_A(b-1) V(b-1),  S_A(b) = Q_A K(b)^T,  O_B += P_B(b-1) V(b-1),  S_B(b) = Q_B K(b)^T
// (one S buffer per tile: S_X(b) overwrites P_X(b-1), which the tensor pipe
// has read by then because it runs one thread's MMAs in order).  While one
// tile's warps turn S into P = 2^(S c - m) (16-bit, written over S), the
// tensor pipe works on the other tile.  O_X is rescaled only when the
// running maximum grows by more than 2^8.  A tile's epilogue (one partial
// (m, l, normalised o) per row) runs after the next pair's first P is out,
// so that waiting for its last P V overlaps that softmax.
template <int DT, int D, int QB>
__global__ void __launch_bounds__(kAttThreads, 1)
    prefill_attend_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const void* __restrict__ Q, PrefArgs a, uint32_t* __restrict__ err) {
  using C = ACfg<D, QB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQA = base;                               // [2 buffers] tile A's Q
  uint8_t* sQB = sQA + 2 * C::kQTile;                // [QB] tile B's Q
  uint8_t* sKV = sQB + QB * C::kQTile;               // [kSlots]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sKV + C::kSlots * C::kKV);
  uint64_t* q_full = bar + 0;     // [2] tile A's Q of a pair and the pair entry loaded
  uint64_t* q_empty = bar + 2;    // [2] last S of the pair done + every softmax warp read the entry
  uint64_t* kv_full = bar + 4;    // [4]
  uint64_t* kv_empty = bar + 8;   // [4]
  uint64_t* s_full = bar + 12;    // [2 tiles] S of the tile's block done
  uint64_t* p_full = bar + 14;    // [2 tiles] P of the tile's block written (4 warps)
  uint64_t* pv_done = bar + 16;   // [2 tiles] O += P V of the tile's block done
  uint64_t* o_free = bar + 18;    // [2 tiles] O read out by the tile's epilogue (4 warps)
  uint64_t* drain = bar + 20;     // every MMA issued has completed
  uint64_t* qb_full = bar + 21;   // [QB] tile B's Q of the pair loaded (every pair)
  uint64_t* qb_empty = bar + 23;  // [QB] last S of the pair done: tile B's buffer is free (every pair)
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(bar + 25);
  volatile int* abort = reinterpret_cast<volatile int*>(bar + 26);
  int4* tinfo = reinterpret_cast<int4*>(bar + 28);  // [2] pair entries

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&q_full[s], 1);
      ptx::mbar_init(&q_empty[s], 1 + kSoftWarps);
      ptx::mbar_init(&s_full[s], 1);
      ptx::mbar_init(&p_full[s], kSoftWarps / 2);
      ptx::mbar_init(&pv_done[s], 1);
      ptx::mbar_init(&o_free[s], kSoftWarps / 2);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    ptx::mbar_init(drain, 1);
    for (int s = 0; s < QB; ++s) {
      ptx::mbar_init(&qb_full[s], 1);
      ptx::mbar_init(&qb_empty[s], 1);
    }
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
  const int npairs = a.ntiles[0];

  auto fail = [&](uint32_t bit) {
    flag_error(err, bit);
    *abort = 1;
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------ K / V producer
    // Ring use u: K(b) for u = 2 b, V(b) for u = 2 b + 1, in slot u % 3.
    if (lane == 0) {
      int64_t u = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < npairs && ok && !*abort; t += gridDim.x) {
        const Pair x = decode_pair(a, a.tiles[t]);
        for (int kb = 0; kb < x.nkb && ok; ++kb) {
          const int y = (int)(x.key0 + (int64_t)kb * kKeyBlk);
#pragma unroll 1
          for (int part = 0; part < 2; ++part, ++u) {
            const int sl = (int)(u % C::kSlots);
            if (u >= C::kSlots && !ptx::mbar_wait(&kv_empty[sl], (uint32_t)(((u - C::kSlots) / C::kSlots) & 1))) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(&kv_full[sl], C::kKV);
#pragma unroll
            for (int r = 0; r < D / 64; ++r)
              ptx::tma_load_3d(sKV + sl * C::kKV + r * C::kRegion, part == 0 ? &tmK : &tmV, &kv_full[sl], r * 64, y,
                               x.bh);
          }
        }
      }
      if (!ok) fail(SSA_DEVERR_WAIT_TIMEOUT);
      // let every load this thread issued land before the CTA can exit
      for (int64_t v = u - C::kSlots < 0 ? 0 : u - C::kSlots; v < u; ++v)
        if (!ptx::mbar_wait(&kv_full[v % C::kSlots], (uint32_t)((v / C::kSlots) & 1)))
          flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp >= kQWarp) {
    // ------------------------------------------------ Q loaders
    // Warp kQWarp + t gathers the 128 query rows of tile t of the pair into
    // the swizzled K-major Q buffer; the tile-A warp publishes the pair
    // entry.  Tile A's buffer is double buffered; tile B's has QB buffers
    // (with one, its warp loads the pair's row entries first and starts the
    // copies as soon as the previous pair's last S has read the buffer).
    const int tt = warp - kQWarp;
    int pc = 0;
    for (int t = blockIdx.x; t < npairs && !*abort; t += gridDim.x, ++pc) {
      const int qb = pc & 1;
      const int qbB = QB == 2 ? qb : 0;  // tile B's buffer
      const int4 v = a.tiles[t];
      const Pair x = decode_pair(a, v);
      int64_t qrow[kTileRows / 32];
      if (x.kind_bh >= 0) {
        const int64_t off = (int64_t)__ldg(a.offsets + x.kind_bh) + x.row0 + tt * kTileRows;
        int e[kTileRows / 32];
#pragma unroll
        for (int i = 0; i < kTileRows / 32; ++i) {
          const int r = i * 32 + lane;
          e[i] = r < x.n(tt) ? __ldg(a.rows + off + r) : -1;
        }
#pragma unroll
        for (int i = 0; i < kTileRows / 32; ++i) {
          const int64_t row = (int64_t)(e[i] >> 6);
          qrow[i] = -1;
          if (i * 32 + lane < x.n(tt)) {
            if (e[i] < 0 || row >= (int64_t)a.B * a.Hq * a.n_q || (e[i] & 63) >= a.topk)
              flag_error(err, SSA_DEVERR_OVERFLOW);
            else
              qrow[i] = row;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < kTileRows / 32; ++i) {
          int rank;
          int64_t tpos;
          qrow[i] = pair_row(a, x, tt, i * 32 + lane, &rank, &tpos, err);
        }
      }
      const bool free_buf = tt == 0 ? (pc < 2 || ptx::mbar_wait(&q_empty[qb], (uint32_t)(((pc - 2) >> 1) & 1)))
                                    : (pc < QB || ptx::mbar_wait(&qb_empty[qbB], (uint32_t)(((pc - QB) / QB) & 1)));
      if (!free_buf) {
        fail(SSA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      if (tt == 0 && lane == 0) tinfo[qb] = v;
      if (x.n(tt) > 0) {
        uint8_t* qt = tt == 0 ? sQA + qb * C::kQTile : sQB + qbB * C::kQTile;
#pragma unroll
        for (int i = 0; i < kTileRows / 32; ++i) {
          const int r = i * 32 + lane;
          const uint8_t* src = static_cast<const uint8_t*>(Q) + (qrow[i] < 0 ? 0 : qrow[i]) * (int64_t)D * 2;
          const uint32_t n = qrow[i] < 0 ? 0u : 16u;
          const uint32_t rsw = (uint32_t)(r & 7);
#pragma unroll
          for (int ch = 0; ch < D / 8; ++ch) {
            uint8_t* dst = qt + (ch >> 3) * C::kRegion + r * 128 + ((((uint32_t)ch & 7) ^ rsw) << 4);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
                         "l"(src + ch * 16), "r"(n)
                         : "memory");
          }
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tt == 0 ? &q_full[qb] : &qb_full[qbB]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int ab16 = DT == DT_BF16 ? 1 : 0;
      const uint32_t id_qk = tc::idesc_f16(128, kKeyBlk, ab16, 0, 0);
      const uint32_t id_pv = tc::idesc_f16(128, D, ab16, 0, 1);
      const uint32_t aQA0 = ptx::smem_u32(sQA), aQB = ptx::smem_u32(sQB), aKV = ptx::smem_u32(sKV);
      int64_t u = 0;                   // ring uses consumed
      int64_t npx[2] = {0, 0};         // pairs with tile X so far (o_free phases)
      // the previous block, whose P V follow this block's S
      bool pend = false, pend_b = false, pend_first = false;
      int pend_slot = 0;
      uint32_t pend_par = 0;
      int64_t pend_g[2] = {0, 0};      // block counts of the tiles at the previous block
      int64_t pend_np[2] = {0, 0};     // ... and their pair counts
      int64_t g[2] = {0, 0};           // blocks of tile X issued
      auto issue_pv = [&](int tx) -> bool {
        // O_X += P_X V: P_X sits in tensor memory over S_X, V is the block in
        // pend_slot.  The first block of a pair overwrites O_X, which the
        // tile's previous epilogue must have read out.
        if (pend_first && pend_np[tx] > 1 && !ptx::mbar_wait(&o_free[tx], (uint32_t)((pend_np[tx] - 2) & 1)))
          return false;
        if (!ptx::mbar_wait(&kv_full[pend_slot], pend_par)) return false;
        if (!ptx::mbar_wait(&p_full[tx], (uint32_t)(pend_g[tx] & 1))) return false;
        tc::fence_after();
        const uint32_t tP = tmem + tx * 128;
        const uint32_t tO = tmem + C::kColO + tx * D;
        const uint32_t vbase = aKV + pend_slot * C::kKV;
#pragma unroll
        for (int k = 0; k < kKeyBlk / 16; ++k) {
          const uint64_t vd = tc::sdesc_sw128(vbase + k * 2048, C::kRegion, 1024);
          tc::mma_ts(tO, tP + k * 8, vd, id_pv, (pend_first && k == 0) ? 0u : 1u);
        }
        tc::commit(&pv_done[tx]);
        return true;
      };
      auto issue_s = [&](int tx, uint32_t aQ, int ks) {
        const uint32_t kbase = aKV + ks * C::kKV;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t qd = tc::sdesc_sw128(aQ + (k >> 2) * C::kRegion + (k & 3) * 32, 16, 1024);
          const uint64_t kd = tc::sdesc_sw128(kbase + (k >> 2) * C::kRegion + (k & 3) * 32, 16, 1024);
          tc::mma(tmem + tx * 128, qd, kd, id_qk, k > 0 ? 1u : 0u);
        }
        tc::commit(&s_full[tx]);
      };
      bool ok = true;
      int pc = 0;
      for (int t = blockIdx.x; t < npairs && ok && !*abort; t += gridDim.x, ++pc) {
        const int qb = pc & 1;
        const int qbB = QB == 2 ? qb : 0;  // tile B's buffer
        if (!ptx::mbar_wait(&q_full[qb], (uint32_t)((pc >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after();
        const Pair x = decode_pair(a, tinfo[qb]);
        const bool hb = x.n1 > 0;
        npx[0] += 1;
        npx[1] += hb ? 1 : 0;
        const uint32_t aQA = aQA0 + qb * C::kQTile;
        for (int kb = 0; kb < x.nkb && ok; ++kb) {
          const int ks = (int)(u % C::kSlots);
          // P_A(b-1) V(b-1) before S_A(b) overwrites P_A(b-1)
          if (pend && !(ok = issue_pv(0))) break;
          if (!(ok = ptx::mbar_wait(&kv_full[ks], (uint32_t)((u / C::kSlots) & 1)))) break;
          tc::fence_after();
          issue_s(0, aQA, ks);
          if (pend) {
            if (pend_b && !(ok = issue_pv(1))) break;
            tc::commit(&kv_empty[pend_slot]);  // V(b-1) read by both tiles
          }
          if (hb) {
            // tile B's Q of this pair (its single buffer) must be in
            if (kb == 0 && !(ok = ptx::mbar_wait(&qb_full[qbB], (uint32_t)((pc / QB) & 1)))) break;
            tc::fence_after();
            issue_s(1, aQB + qbB * C::kQTile, ks);
          }
          tc::commit(&kv_empty[ks]);           // K(b) read by both tiles
          if (kb == x.nkb - 1) {
            tc::commit(&q_empty[qb]);
            tc::commit(&qb_empty[qbB]);
          }
          ++u;
          pend = true;
          pend_b = hb;
          pend_first = kb == 0;
          pend_slot = (int)(u % C::kSlots);
          pend_par = (uint32_t)((u / C::kSlots) & 1);
          ++u;
          pend_g[0] = g[0]++;
          pend_np[0] = npx[0];
          if (hb) {
            pend_g[1] = g[1]++;
            pend_np[1] = npx[1];
          }
        }
      }
      if (ok && pend && !*abort) {
        ok = issue_pv(0);
        if (ok && pend_b) ok = issue_pv(1);
        if (ok) tc::commit(&kv_empty[pend_slot]);
      }
      if (!ok) fail(SSA_DEVERR_WAIT_TIMEOUT);
      // every MMA issued completes before the tensor memory is released
      tc::commit(drain);
      if (!ptx::mbar_wait(drain, 0)) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------ softmax warps
    // Warp w handles tile tx = w / 4 and rows r = 32 (w % 4) + lane: one row
    // per thread, all 128 keys of each block.
    const int tx = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + tx * 128 + lane_off;
    const uint32_t tO = tmem + C::kColO + tx * D + lane_off;
    const float c = a.scale_log2e;
    int64_t gx = 0;                    // blocks of this tile processed
    // the previous pair's epilogue, still to run: its row's partial slot,
    // (m, l) and the block whose P V it waits for
    bool pend = false;
    int64_t pslot = -1, pgx = 0;
    float pm = 0.f, pl = 1.f;
    auto epilogue = [&]() -> bool {
      pend = false;
      if (!ptx::mbar_wait(&pv_done[tx], (uint32_t)(pgx & 1))) return false;
      tc::fence_after();
      // read all of O_X under one wait and release it at once (the next
      // pair's first P V may then overwrite it), then normalise and store
      uint32_t o[D];
      if constexpr (D == 128) {
        tc::ld64x2(tO, *reinterpret_cast<uint32_t(*)[64]>(&o[0]), tO + 64, *reinterpret_cast<uint32_t(*)[64]>(&o[64]));
      } else {
        tc::ld64(tO, *reinterpret_cast<uint32_t(*)[64]>(&o[0]));
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_relaxed(&o_free[tx]);
      if (pslot >= 0) {
        const float inv = 1.f / pl;
        const float2 inv2 = make_float2(inv, inv);
        uint16_t* dst = a.po + pslot * D;  // 32-byte aligned: a slot is D * 2 bytes
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 y = __fmul2_rn(
                make_float2(__uint_as_float(o[16 * q + 2 * j]), __uint_as_float(o[16 * q + 2 * j + 1])), inv2);
            pk[j] = ptx::pack2<DT>(y.x, y.y);
          }
          ptx::st_global_v8(dst + 16 * q, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
        }
        a.pml[pslot] = make_float2(pm, pl);
      }
      return true;
    };
    bool ok = true;
    int pc = 0;
    for (int t = blockIdx.x; t < npairs; t += gridDim.x, ++pc) {
      const int qb = pc & 1;
      if (!ptx::mbar_wait(&q_full[qb], (uint32_t)((pc >> 1) & 1))) {
        ok = false;
        break;
      }
      const int4 v = tinfo[qb];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&q_empty[qb]);
      const Pair x = decode_pair(a, v);
      if (x.n(tx) == 0) {
        // no tile B in this pair: the pending epilogue cannot wait for it
        if (pend && !(ok = epilogue())) break;
        continue;
      }
      int rank;
      int64_t tpos;
      const int64_t qrow = pair_row(a, x, tx, r, &rank, &tpos, err);
      float m = -INFINITY, l = 0.f;
      for (int kb = 0; kb < x.nkb && ok; ++kb, ++gx) {
        if (!(ok = ptx::mbar_wait(&s_full[tx], (uint32_t)(gx & 1)))) break;
        tc::fence_after();
        // valid keys of this block for this row: [0, klim)
        const int64_t kstart = x.key0 + (int64_t)kb * kKeyBlk;
        int64_t klim = x.key_end - kstart;
        if (x.kind_bh < 0) klim = min(klim, tpos - kstart + 1);
        const bool partial = klim < kKeyBlk;
        uint32_t sr[128];
        tc::ld64x2(tS, *reinterpret_cast<uint32_t(*)[64]>(&sr[0]), tS + 64, *reinterpret_cast<uint32_t(*)[64]>(&sr[64]));
        if (partial) {
#pragma unroll
          for (int j = 0; j < 128; ++j)
            if (j >= klim) sr[j] = 0xff800000u;  // -inf
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 128; j += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            m4[u] = ptx::max3(m4[u], __uint_as_float(sr[j + 2 * u]), __uint_as_float(sr[j + 2 * u + 1]));
        const float mx = ptx::max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]) * c;
        // rescale O only when this row's max grows by more than 2^8
        float m_new = m;
        if (kb == 0 || mx > m + kRescaleLog2) m_new = mx;
        const bool need = kb > 0 && m_new != m;
        const float nb = m_new == -INFINITY ? 0.f : -m_new;
        // P = 2^(s c - m) as 16-bit pairs over the S columns just read, in two
        // halves of 64 keys (two partial sums keep the adds off one chain);
        // s c - m of two keys in one packed fp32 FMA (each lane rounded as
        // fmaf would)
        float lsum = 0.f;
        const float2 c2 = make_float2(c, c), nb2 = make_float2(nb, nb);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
          float la = 0.f, lb = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float2 e = __ffma2_rn(
                make_float2(__uint_as_float(sr[64 * hf + j]), __uint_as_float(sr[64 * hf + j + 1])), c2, nb2);
            const float p0 = ptx::ex2(e.x);
            const float p1 = ptx::ex2(e.y);
            la += p0;
            lb += p1;
            pk[j / 2] = ptx::pack2<DT>(p0, p1);
          }
          lsum += la + lb;
          if (hf == 0)
            tc::st32_nowait(tS, pk);
          else
            tc::st32(tS + 32, pk);  // its wait covers both stores
        }
        // the rescale runs after P is out (the S values are dead by then) and
        // before P is released to the tensor pipe
        if (__any_sync(0xffffffffu, need)) {
          // O += P V of the previous block must be complete before O is rescaled
          if (!(ok = ptx::mbar_wait(&pv_done[tx], (uint32_t)((gx - 1) & 1)))) break;
          tc::fence_after();
          const float f = need ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t rr[32];
            tc::ld32(tO + q * 32, rr);
            const float2 f2 = make_float2(f, f);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float2 y = __fmul2_rn(make_float2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])), f2);
              rr[j] = __float_as_uint(y.x);
              rr[j + 1] = __float_as_uint(y.y);
            }
            tc::st32(tO + q * 32, rr);
          }
          l *= f;
        }
        m = m_new;
        l += lsum;
        tc::fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_relaxed(&p_full[tx]);
        // the previous pair's epilogue, once this pair's first P is out
        if (kb == 0 && pend && !(ok = epilogue())) break;
      }
      if (!ok) break;
      pend = true;
      pslot = qrow >= 0 ? qrow * (a.topk + 1) + rank : -1;
      pm = m;
      pl = l;
      pgx = gx - 1;
    }
    if (ok && pend) ok = epilogue();
    if (!ok) fail(SSA_DEVERR_WAIT_TIMEOUT);
  }
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------- merge
// One warp per row of Q, rows in a grid-stride loop.  A row's k + 1 partials
// are one contiguous block of (k + 1) * d 16-bit values: a bulk copy brings
// the next row's block into the warp's other shared-memory stage while the
// warp combines the current one, and its (m, l) and sel entries are read one
// row ahead into registers.  The combine is two-pass: M = the max of the
// used slots' m, w_s = 2^(m_s - M) l_s (one exp2 per slot, lane-parallel),
// O = sum_s w_s o_s / sum_s w_s, lse = M ln 2 + ln sum_s w_s.  Slots are the
// sel row's used prefix (ranks 0 .. used - 1) and the local span (rank k).
constexpr int kMergeWarpsMax = 8;
constexpr size_t kMergeSmemBudget = 96 * 1024;

template <int DT, int E>
__device__ __forceinline__ void widen_partial(uint32_t saddr, float (&v)[E]) {
  if constexpr (E == 4) {
    const uint2 w = ptx::lds64(saddr);
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
    const uint32_t w = ptx::lds32(saddr);
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

// A row's per-lane look-ahead: (m, l) of slots lane, lane + 32, lane + 64
// and its sel entries lane, lane + 32.
struct MergeAhead {
  float2 ml[3];
  int j0, j1;
};

__device__ __forceinline__ void merge_ahead(const int32_t* __restrict__ sel, const PrefArgs& a, int64_t row,
                                            int lane, MergeAhead& x) {
  const int nslot = a.topk + 1;
  const int64_t base = row * nslot;
#pragma unroll
  for (int u = 0; u < 3; ++u) {
    const int s = lane + 32 * u;
    x.ml[u] = s < nslot ? a.pml[base + s] : make_float2(-INFINITY, 0.f);
  }
  const int32_t* srow = sel + row * a.topk;
  x.j0 = lane < a.topk ? srow[lane] : -1;
  x.j1 = lane + 32 < a.topk ? srow[lane + 32] : -1;
}

template <int DT, int D>
__global__ void __launch_bounds__(kMergeWarpsMax * 32) prefill_merge_kernel(const int32_t* __restrict__ sel,
                                                                           PrefArgs a, void* __restrict__ O,
                                                                           float* __restrict__ lse,
                                                                           uint32_t* __restrict__ err) {
  constexpr int E = D / 32;
  extern __shared__ __align__(128) uint8_t msm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int nslot = a.topk + 1;
  const uint32_t row_bytes = (uint32_t)nslot * D * 2;   // a multiple of 16
  uint8_t* ring = msm + (size_t)warp * 2 * row_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(msm + (size_t)nw * 2 * row_bytes) + 2 * warp;
  if (lane == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int64_t n_rows = (int64_t)a.B * a.Hq * a.n_q;
  const int64_t stride = (int64_t)gridDim.x * nw;
  int64_t row = (int64_t)blockIdx.x * nw + warp;
  auto issue = [&](int64_t r, int st) {
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ptx::mbar_arrive_expect_tx(&bars[st], row_bytes);
      ptx::bulk_load(ring + (size_t)st * row_bytes, a.po + r * nslot * D, row_bytes, &bars[st]);
    }
  };
  MergeAhead cur, nxt;
  if (row < n_rows) {
    issue(row, 0);
    merge_ahead(sel, a, row, lane, cur);
  }
  int st = 0;
  uint32_t phb = 0u;            // bit st: the phase stage st waits for next
  bool pending_other = false;   // a copy in flight in stage st ^ 1
  for (; row < n_rows; row += stride) {
    const int64_t rn = row + stride;
    pending_other = rn < n_rows;
    if (pending_other) {
      issue(rn, st ^ 1);
      merge_ahead(sel, a, rn, lane, nxt);
    }
    // the used slots and their weights
    const int64_t i = row % a.n_q;
    const int64_t ell = (a.q_pos0 + i) / a.S;
    bool bad;
    const int used = warp_sel_prefix(cur.j0, cur.j1, lane, a.topk, ell, &bad);
    float w[3];
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int s = lane + 32 * u;
      const bool ok = s < nslot && (s < used || s == a.topk);
      w[u] = ok ? cur.ml[u].x : -INFINITY;
      mx = fmaxf(mx, w[u]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float lsum = 0.f;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      w[u] = w[u] == -INFINITY ? 0.f : exp2f(w[u] - mx) * cur.ml[u].y;
      lsum += w[u];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (!ptx::mbar_wait(&bars[st], (phb >> st) & 1u)) {
      if (lane == 0) flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
      break;
    }
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const uint32_t sbase = ptx::smem_u32(ring + (size_t)st * row_bytes) + lane * E * 2;
    for (int s = 0; s < nslot; ++s) {
      if (s >= used && s != a.topk) continue;   // warp-uniform
      const float ws = __shfl_sync(0xffffffffu, s < 32 ? w[0] : s < 64 ? w[1] : w[2], s & 31);
      float v[E];
      widen_partial<DT, E>(sbase + (uint32_t)s * D * 2, v);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(ws, v[e], acc[e]);
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int e = 0; e < E; ++e) store_elem<DT>(O, row * D + lane * E + e, acc[e] * inv);
    if (lse && lane == 0) lse[row] = mx * kLn2 + logf(lsum);
    phb ^= 1u << st;
    st ^= 1;
    cur = nxt;
    pending_other = false;
    __syncwarp();   // every lane is done with this stage before it is refilled
  }
  // after a timeout: let this warp's own copy in flight land before exiting
  if (pending_other && !ptx::mbar_wait(&bars[st ^ 1], (phb >> (st ^ 1)) & 1u) && lane == 0)
    flag_error(err, SSA_DEVERR_WAIT_TIMEOUT);
}

// Warps per merge CTA: as many as two stages of a row's partials fit in the
// per-CTA shared-memory budget, at most 8.
int merge_warps(const Problem& pr) {
  const size_t row_bytes = (size_t)(pr.topk + 1) * pr.d * 2;
  const size_t w = kMergeSmemBudget / (2 * row_bytes + 16);
  return (int)(w < 1 ? 1 : w > (size_t)kMergeWarpsMax ? kMergeWarpsMax : w);
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

// The attend kernel's launch: tile B's Q double buffered for spans of four
// key blocks or more (A/B on one B300: a 1M chunk with S = 1024 3.097 ->
// 3.048 ms, the 128K prefill with S = 256 21.37 -> 22.03 ms).
template <int DT, int D, int QB>
cudaError_t launch_attend(const PrefArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, const void* Q,
                          uint32_t* err, cudaStream_t st) {
  using C = ACfg<D, QB>;
  static bool attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_attr(prefill_attend_kernel<DT, D, QB>, C::kSmem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_attend_kernel<DT, D, QB>, dim3(device_sm_count()), dim3(kAttThreads), C::kSmem, st,
                    tmK, tmV, Q, a, err);
}

template <int DT, int D>
cudaError_t launch_typed(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const void* K,
                         const void* V, const int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st) {
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
  e = pr.S >= 4 * kKeyBlk ? launch_attend<DT, D, 2>(a, tmK, tmV, Q, err, st)
                          : launch_attend<DT, D, 1>(a, tmK, tmV, Q, err, st);
  if (e != cudaSuccess) return e;
  const int64_t n_rows = (int64_t)pr.B * pr.Hq * n_q;
  const int mw = merge_warps(pr);
  const size_t msmem = (size_t)mw * (2 * (size_t)(pr.topk + 1) * D * 2 + 16);
  static bool mattr_done[kMaxDevices] = {};
  e = ensure_smem_attr(prefill_merge_kernel<DT, D>, kMergeSmemBudget + kMergeWarpsMax * 16, mattr_done);
  if (e != cudaSuccess) return e;
  const int64_t merge_ctas = min((n_rows + mw - 1) / mw, (int64_t)device_sm_count() * 3);
  return launch_pdl(prefill_merge_kernel<DT, D>, dim3((unsigned)merge_ctas), dim3(mw * 32), msmem, st, sel, a, O,
                    lse, err);
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

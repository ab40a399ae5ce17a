// quant.cu -- the 8-bit cache: quantised K / V rows and the summaries of
// their spans.
//
// SubQ release post (geeks.co.kr/post/2077), limitations and quantisation
// plan: fp16 only so far (66 GB for a 1M context), 8-bit / 4-bit K / V coming
// so that a full 1M context runs on a 24 GB card.  The pages fix no scheme;
// this library uses symmetric 8-bit rows with one fp32 scale per (b,
// kv-head, token):
//   s = max_i |x_i| / 127,  q_i = clamp(rint(x_i / s), -127, 127)  (0 if s == 0)
// in fp32 (IEEE division, round to nearest even), and the summaries stay
// fp32: the mean over a span of the dequantised keys q_i * s.
//
// Layouts (declared in include/ssa.h):
//   Kq [B, Hkv, L_cap, d]            int8, row-major
//   Vq [B, Hkv, L_cap / 32, d, 32]   int8, each 32-token tile stored d-major;
//        inside a tile's d-row of 32 bytes, byte 8 c + e holds token
//        16 (e / 4) + tok(c, e % 4) with tok(c, 0..3) = 2c, 2c+1, 2c+8, 2c+9
//   Ks, Vs [B, Hkv, L_cap]           fp32 scales
// The V order is the k order of the m16n8k16 A fragment of V^T, so the
// decode kernel reads a thread's two 16-token fragments with one 8-byte load.
#include "internal.h"

namespace ssa {
namespace {

constexpr int kQRows = 8;  // rows (warps) per CTA

// Byte of token tt (0..31) inside its tile's d-row.
__device__ __forceinline__ int vq_byte(int tt) {
  const int h = tt >> 4, w = tt & 15;
  const int c = (w & 7) >> 1;                    // pair index
  const int e = (w & 1) + ((w >> 3) << 1);       // 0, 1 (tokens 2c, 2c+1) or 2, 3 (2c+8, 2c+9)
  return 8 * c + e + 4 * h;
}

// One warp per (tensor, b*kv-head, token) row: K rows in blockIdx.y == 0,
// V rows in blockIdx.y == 1.
template <int DT, int D>
__global__ void __launch_bounds__(kQRows * 32)
    quantize_kernel(const void* __restrict__ K, const void* __restrict__ V, int64_t L_cap, int64_t t0,
                    int64_t nt, int64_t rows, int8_t* __restrict__ Kq, float* __restrict__ Ks,
                    int8_t* __restrict__ Vq, float* __restrict__ Vs) {
  constexpr int E = D / 32;  // elements per lane
  const int64_t row = (int64_t)blockIdx.x * kQRows + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const bool isv = blockIdx.y == 1;
  const int64_t bh = row / nt, t = t0 + row % nt;
  const int64_t src = (bh * L_cap + t) * D + lane * E;
  const void* X = isv ? V : K;
  float x[E];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    x[e] = load_elem<DT>(X, src + e);
    amax = fmaxf(amax, fabsf(x[e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = __fdiv_rn(amax, 127.0f);
  int8_t q[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int v = 0;
    if (s != 0.f) v = min(127, max(-127, __float2int_rn(__fdiv_rn(x[e], s))));
    q[e] = (int8_t)v;
  }
  if (!isv) {
    int8_t* dst = Kq + (bh * L_cap + t) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = q[e];
    if (lane == 0) Ks[bh * L_cap + t] = s;
  } else {
    const int64_t tile = t >> 5;
    const int b8 = vq_byte((int)(t & 31));
    int8_t* base = Vq + ((bh * (L_cap >> 5) + tile) * D) * 32 + b8;
#pragma unroll
    for (int e = 0; e < E; ++e) base[(int64_t)(lane * E + e) * 32] = q[e];
    if (lane == 0) Vs[bh * L_cap + t] = s;
  }
}

// Summaries of the 8-bit keys: one CTA per (b*kv-head, span), the same
// fixed-order reduction as the 16-bit summaries: thread (row group r, column
// slice c) adds rows r, r + RPP, ... of 16 columns, then the RPP partial
// sums are added in order.
template <int D>
__global__ void __launch_bounds__(256) summaries_q8_kernel(const int8_t* __restrict__ Kq,
                                                           const float* __restrict__ Ks,
                                                           float* __restrict__ summ, int64_t L_cap,
                                                           int64_t L, int S, int64_t span_begin,
                                                           int64_t ns_cap) {
  constexpr int VEC = 16;
  constexpr int TPR = D / VEC;
  constexpr int RPP = 256 / TPR;
  __shared__ float red[RPP * D];
  const int64_t bh = blockIdx.y;
  const int64_t j = span_begin + blockIdx.x;
  const int64_t t0 = j * S;
  const int64_t t1 = t0 + S < L ? t0 + S : L;
  const int n = (int)(t1 - t0);
  const int tr = threadIdx.x / TPR, tc = threadIdx.x % TPR;
  const int8_t* base = Kq + (bh * L_cap + t0) * D + tc * VEC;
  const float* sc = Ks + bh * L_cap + t0;
  float acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
  for (int r = tr; r < n; r += RPP) {
    const int4 w = __ldg(reinterpret_cast<const int4*>(base + (int64_t)r * D));
    const float s = __ldg(sc + r);
    const int ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int q = (int)(int8_t)((ws[u] >> (8 * b)) & 0xff);
        acc[4 * u + b] += (float)q * s;
      }
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
cudaError_t launch_q(const Problem& pr, const void* K, const void* V, int64_t t0, int64_t t1, int8_t* Kq,
                     float* Ks, int8_t* Vq, float* Vs, cudaStream_t st) {
  const int64_t nt = t1 - t0;
  const int64_t rows = (int64_t)pr.B * pr.Hkv * nt;
  const int64_t blocks = (rows + kQRows - 1) / kQRows;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  quantize_kernel<DT, D><<<dim3((unsigned)blocks, 2), kQRows * 32, 0, st>>>(K, V, pr.L_cap, t0, nt, rows, Kq,
                                                                           Ks, Vq, Vs);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 4-bit
// The same scheme with 15 levels (SubQ release post, quantisation plan, its
// 4-bit half): s = max_i |x_i| / 7, q_i = clamp(rint(x_i / s), -7, 7), each
// code stored as the nibble q + 8.  d = 128 only.  A 32-token tile of K and
// of V is one 2 KB block of 32-bit words, laid out for the decode kernel's
// fragment loads (each thread of a warp reads one word per row, the warp's
// 32 words consecutive):
//   Kq4 word [J][tok][c]  (J < d / 32, tok < 32, c < 4): token tok's
//        dimensions d = 32 J + 8 c + e, e < 8
//   Vq4 word [d][c]       (c < 4): dimension d of tokens
//        2c + f(e), f = 0, 1, 8, 9, 16, 17, 24, 25 for e = 0..7
// and inside a word element e sits at bit 4 (e / 2) + 16 (e % 2), so that
// (w >> 4 i) & 0x000F000F holds elements 2i and 2i + 1 in the low bits of
// its two halves: one fp16 pair each.
constexpr int kQ4Tile = 32;
constexpr int kQ4Words = 512;   // words per 32-token tile of K or of V (d = 128)

__device__ __forceinline__ uint32_t q4_shift(int e) { return 4u * (uint32_t)(e >> 1) + 16u * (uint32_t)(e & 1); }

// The V element slot of token tok (0..31) of a tile: word column c and e.
__device__ __forceinline__ void q4_vslot(int tok, int& c, int& e) {
  const int w = tok & 15;
  c = (w & 7) >> 1;
  e = (w & 1) + 2 * ((w >> 3) + 2 * (tok >> 4));
}

// One CTA of 256 threads per (b*kv-head, 32-token tile) overlapping
// [t0, t1): warp w quantises the tile's tokens w, w + 8, ...  K words belong
// to one token and are written whole; V words gather eight tokens, so the
// tile's V block is rebuilt in shared memory from its old contents (tokens
// outside [t0, t1) keep theirs) and written back whole.
template <int DT>
__global__ void __launch_bounds__(256) quantize4_kernel(const void* __restrict__ K, const void* __restrict__ V,
                                                         int64_t L_cap, int64_t t0, int64_t t1, int64_t tile0,
                                                         uint32_t* __restrict__ Kq4, float* __restrict__ Ks,
                                                         uint32_t* __restrict__ Vq4, float* __restrict__ Vs) {
  constexpr int D = 128;
  __shared__ uint32_t vw[kQ4Words];
  const int64_t bh = blockIdx.y;
  const int64_t tile = tile0 + blockIdx.x;
  const int64_t tb = tile * kQ4Tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* vg = Vq4 + (bh * (L_cap / kQ4Tile) + tile) * kQ4Words;
  uint32_t* kg = Kq4 + (bh * (L_cap / kQ4Tile) + tile) * kQ4Words;
  for (int x = threadIdx.x; x < kQ4Words; x += 256) vw[x] = vg[x];
  __syncthreads();
  for (int tok = warp; tok < kQ4Tile; tok += 8) {
    const int64_t t = tb + tok;
    if (t < t0 || t >= t1) continue;
    for (int isv = 0; isv < 2; ++isv) {
      const void* X = isv ? V : K;
      const int64_t src = (bh * L_cap + t) * D + lane * 4;
      float x[4];
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = load_elem<DT>(X, src + e);
        amax = fmaxf(amax, fabsf(x[e]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = __fdiv_rn(amax, 7.0f);
      uint32_t nib[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int v = 0;
        if (sc != 0.f) v = min(7, max(-7, __float2int_rn(__fdiv_rn(x[e], sc))));
        nib[e] = (uint32_t)(v + 8);
      }
      if (!isv) {
        // lanes 2m and 2m + 1 hold dimensions 8m .. 8m + 7: one word
        const int half = lane & 1;
        uint32_t part = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) part |= nib[e] << q4_shift(4 * half + e);
        const uint32_t word = part | __shfl_xor_sync(0xffffffffu, part, 1);
        if (half == 0) {
          const int m = lane >> 1, J = m >> 2, c = m & 3;
          kg[(J * kQ4Tile + tok) * 4 + c] = word;
        }
        if (lane == 0) Ks[bh * L_cap + t] = sc;
      } else {
        int c, e;
        q4_vslot(tok, c, e);
        const uint32_t sh = q4_shift(e);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t* wp = &vw[(lane * 4 + k) * 4 + c];
          atomicAnd(wp, ~(0xFu << sh));
          atomicOr(wp, nib[k] << sh);
        }
        if (lane == 0) Vs[bh * L_cap + t] = sc;
      }
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < kQ4Words; x += 256) vg[x] = vw[x];
}

// Summaries of the 4-bit keys: one CTA per (b*kv-head, span), thread = d
// column, the span's tokens added in order.
__global__ void __launch_bounds__(128) summaries_q4_kernel(const uint32_t* __restrict__ Kq4,
                                                           const float* __restrict__ Ks, float* __restrict__ summ,
                                                           int64_t L_cap, int64_t L, int S, int64_t span_begin,
                                                           int64_t ns_cap) {
  constexpr int D = 128;
  const int64_t bh = blockIdx.y;
  const int64_t j = span_begin + blockIdx.x;
  const int64_t t0 = j * S;
  const int64_t t1 = t0 + S < L ? t0 + S : L;
  const int d = threadIdx.x;
  const int J = d >> 5, c = (d & 31) >> 3;
  const uint32_t sh = q4_shift(d & 7);
  const uint32_t* kb = Kq4 + bh * (L_cap / kQ4Tile) * kQ4Words;
  const float* sc = Ks + bh * L_cap;
  float acc = 0.f;
  for (int64_t t = t0; t < t1; ++t) {
    const uint32_t w = __ldg(kb + (t / kQ4Tile) * kQ4Words + (J * kQ4Tile + (t % kQ4Tile)) * 4 + c);
    const int q = (int)((w >> sh) & 0xFu) - 8;
    acc += (float)q * __ldg(sc + t);
  }
  summ[(bh * ns_cap + j) * D + d] = acc / (float)(t1 - t0);
}

}  // namespace

cudaError_t launch_quantize_kv(const Problem& pr, const void* K, const void* V, int64_t t0, int64_t t1,
                               int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, cudaStream_t st) {
  if (t1 <= t0) return cudaSuccess;
  if (pr.d == 128) {
    switch (pr.dtype) {
      case DT_F32: return launch_q<DT_F32, 128>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
      case DT_BF16: return launch_q<DT_BF16, 128>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
      default: return launch_q<DT_F16, 128>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
    }
  }
  switch (pr.dtype) {
    case DT_F32: return launch_q<DT_F32, 64>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
    case DT_BF16: return launch_q<DT_BF16, 64>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
    default: return launch_q<DT_F16, 64>(pr, K, V, t0, t1, Kq, Ks, Vq, Vs, st);
  }
}

cudaError_t launch_summaries_q8(const Problem& pr, const int8_t* Kq, const float* Ks, int64_t j0, int64_t j1,
                                float* summ, cudaStream_t st) {
  if (j1 <= j0) return cudaSuccess;
  if (j1 - j0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)(j1 - j0), (unsigned)(pr.B * pr.Hkv));
  if (pr.d == 128)
    summaries_q8_kernel<128><<<grid, 256, 0, st>>>(Kq, Ks, summ, pr.L_cap, pr.L, pr.S, j0, pr.ns_cap);
  else
    summaries_q8_kernel<64><<<grid, 256, 0, st>>>(Kq, Ks, summ, pr.L_cap, pr.L, pr.S, j0, pr.ns_cap);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv4(const Problem& pr, const void* K, const void* V, int64_t t0, int64_t t1,
                                uint32_t* Kq4, float* Ks, uint32_t* Vq4, float* Vs, cudaStream_t st) {
  if (t1 <= t0) return cudaSuccess;
  const int64_t tile0 = t0 / kQ4Tile, tile1 = (t1 + kQ4Tile - 1) / kQ4Tile;
  if (tile1 - tile0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)(tile1 - tile0), (unsigned)(pr.B * pr.Hkv));
  switch (pr.dtype) {
    case DT_F32:
      quantize4_kernel<DT_F32><<<grid, 256, 0, st>>>(K, V, pr.L_cap, t0, t1, tile0, Kq4, Ks, Vq4, Vs);
      break;
    case DT_BF16:
      quantize4_kernel<DT_BF16><<<grid, 256, 0, st>>>(K, V, pr.L_cap, t0, t1, tile0, Kq4, Ks, Vq4, Vs);
      break;
    default:
      quantize4_kernel<DT_F16><<<grid, 256, 0, st>>>(K, V, pr.L_cap, t0, t1, tile0, Kq4, Ks, Vq4, Vs);
  }
  return cudaGetLastError();
}

cudaError_t launch_summaries_q4(const Problem& pr, const uint32_t* Kq4, const float* Ks, int64_t j0, int64_t j1,
                                float* summ, cudaStream_t st) {
  if (j1 <= j0) return cudaSuccess;
  if (j1 - j0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)(j1 - j0), (unsigned)(pr.B * pr.Hkv));
  summaries_q4_kernel<<<grid, 128, 0, st>>>(Kq4, Ks, summ, pr.L_cap, pr.L, pr.S, j0, pr.ns_cap);
  return cudaGetLastError();
}

}  // namespace ssa

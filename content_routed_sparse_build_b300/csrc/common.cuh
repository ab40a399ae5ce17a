// common.cuh -- element types, vector loads and the device error record.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssa.h"

namespace ssa {

enum : int { DT_F32 = SSA_F32, DT_BF16 = SSA_BF16, DT_F16 = SSA_F16 };

template <int DT>
struct Elem;
template <>
struct Elem<DT_F32> {
  using T = float;
  static constexpr int kBytes = 4;
};
template <>
struct Elem<DT_BF16> {
  using T = __nv_bfloat16;
  static constexpr int kBytes = 2;
};
template <>
struct Elem<DT_F16> {
  using T = __half;
  static constexpr int kBytes = 2;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Widen the 16 bytes at p (4 fp32 or 8 half-precision elements) to float.
template <int DT>
__device__ __forceinline__ void widen16(const uint4& v, float* out) {
  if constexpr (DT == DT_F32) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
  } else if constexpr (DT == DT_BF16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
}

template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (DT == DT_F32) {
    return static_cast<const float*>(base)[i];
  } else if constexpr (DT == DT_BF16) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  } else {
    return __half2float(static_cast<const __half*>(base)[i]);
  }
}

template <int DT>
__device__ __forceinline__ void store_elem(void* base, int64_t i, float v) {
  if constexpr (DT == DT_F32) {
    static_cast<float*>(base)[i] = v;
  } else if constexpr (DT == DT_BF16) {
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(base)[i] = __float2half_rn(v);
  }
}

// The sticky device error record lives in the first word of a workspace.
__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// Order of the selection: higher score first, lower span index on a tie.
__device__ __forceinline__ bool better(float s, int j, float s2, int j2) {
  return s > s2 || (s == s2 && j < j2);
}

constexpr int kNoSpan = 0x7fffffff;

// Which entries of a sel row are used, computed by one warp (topk <= 64;
// lane r holds entries r and r + 32).  The used entries are the row's
// leading run of candidate spans (0 <= j < ell) in strictly ascending
// order; the row is well formed when everything after that run is -1.
// Returns the number of used entries; *bad is set for a malformed row.
__device__ __forceinline__ int warp_sel_prefix(int j0, int j1, int lane, int topk, int64_t ell,
                                               bool* bad) {
  const int p0 = __shfl_up_sync(0xffffffffu, j0, 1);
  const int last0 = __shfl_sync(0xffffffffu, j0, 31);
  const int p1 = __shfl_up_sync(0xffffffffu, j1, 1);
  const bool in0 = lane < topk, in1 = lane + 32 < topk;
  const bool ok0 = in0 && j0 >= 0 && j0 < ell && (lane == 0 || p0 < j0);
  const bool ok1 = in1 && j1 >= 0 && j1 < ell && (lane == 0 ? last0 < j1 : p1 < j1);
  const uint64_t okm = (uint64_t)__ballot_sync(0xffffffffu, ok0) |
                      ((uint64_t)__ballot_sync(0xffffffffu, ok1) << 32);
  const int n = __ffsll((long long)~okm) - 1;  // first entry that is not used
  const int used = n < 0 || n > topk ? topk : n;
  const bool junk0 = in0 && lane >= used && j0 != -1;
  const bool junk1 = in1 && lane + 32 >= used && j1 != -1;
  *bad = __any_sync(0xffffffffu, junk0 || junk1);
  return used;
}

}  // namespace ssa

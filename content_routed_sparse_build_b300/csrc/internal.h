// internal.h -- validated problem description and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace ssa {

// ssa_params after validation, with derived sizes.
struct Problem {
  int B, Hq, Hkv, d, g;  // g = Hq / Hkv
  int64_t L, L_cap;
  int S, topk;
  float scale;           // resolved (never 0)
  int dtype;
  int64_t ns_cap;        // ceil(L_cap / S): span slots per (b, kv-head) in summ
};

// Workspace layout shared by the attention entry points.
constexpr size_t kWsHeader = 256;  // error record + counters, keeps what follows aligned
inline uint32_t* ws_error(void* ws) { return static_cast<uint32_t*>(ws); }

cudaError_t launch_summaries(const Problem& pr, const void* K, int64_t j0, int64_t j1, float* summ,
                             cudaStream_t st);

// Routing.  Decode (n_q == 1) uses a cluster kernel that splits the
// candidates over 8 CTAs per kv-head; prefill uses query tiles.
cudaError_t launch_route(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const float* summ, int32_t* sel, float* sel_score, cudaStream_t st);

// Reference-quality attention: one warp per query row, any dtype.
cudaError_t launch_attend_rows(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                               const void* K, const void* V, const int32_t* sel, void* O,
                               float* lse, uint32_t* err, cudaStream_t st);

// Decode attention fast path (16-bit types): plan, split spans, merge.
size_t decode_ws_bytes(const Problem& pr);
bool decode_fast_supported(const Problem& pr);
cudaError_t launch_attend_decode(const Problem& pr, const void* Q, int64_t pos, const void* K,
                                 const void* V, const int32_t* sel, void* O, float* lse, void* ws,
                                 cudaStream_t st);

// Prefill attention fast path (16-bit types): dispatch, span tiles, merge.
size_t prefill_ws_bytes(const Problem& pr, int64_t n_q);
bool prefill_fast_supported(const Problem& pr);
cudaError_t launch_attend_prefill(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                                  const void* K, const void* V, const int32_t* sel, void* O,
                                  float* lse, void* ws, cudaStream_t st);

}  // namespace ssa

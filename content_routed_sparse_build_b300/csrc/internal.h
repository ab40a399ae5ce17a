// internal.h -- validated problem description and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#include <utility>

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

// Validates the public parameters and resolves them (SSA_OK or a status).
int check_params(const ssa_params* p, Problem* pr);

// Workspace layout shared by the attention entry points.
constexpr size_t kWsHeader = 256;  // error record + counters, keeps what follows aligned
inline uint32_t* ws_error(void* ws) { return static_cast<uint32_t*>(ws); }

// TMA descriptor of a [B, Hkv, L_cap, d] cache as {d, L, B*Hkv}, 64 x box_rows
// boxes with 128-byte swizzling (16-bit types only).
cudaError_t make_kv_tmap(CUtensorMap* map, const void* base, int dtype, int d, int64_t L,
                         int64_t L_cap, int64_t BH, int box_rows);
int device_sm_count();
// TMA descriptor of an 8-bit [B, Hkv, L_cap, d] cache (d = 128: one
// 128-byte box per row, 128-byte swizzling), box_rows rows per box.
cudaError_t make_q8_tmap(CUtensorMap* map, const void* base, int d, int64_t L, int64_t L_cap, int64_t BH,
                         int box_rows);

// Launches a kernel with programmatic dependent launch enabled: it may begin
// before the previous kernel on the stream ends and must call pdl_wait()
// (ptx.cuh) before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit once per device.
constexpr int kMaxDevices = 64;
template <typename F>
cudaError_t ensure_smem_attr(F* func, size_t bytes, bool* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return e;
}

cudaError_t launch_summaries(const Problem& pr, const void* K, int64_t j0, int64_t j1, float* summ,
                             cudaStream_t st);

// Routing.  Decode (n_q == 1) uses a cluster kernel that splits the
// candidates over 8 CTAs per kv-head; a chunk of 16-bit queries uses the
// tensor-core router (its workspace holds split summaries); anything else
// uses fp32 query tiles.
cudaError_t launch_route(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                         const float* summ, int32_t* sel, float* sel_score, cudaStream_t st);
bool route_tc_supported(const Problem& pr, int64_t n_q);
size_t route_tc_ws_bytes(const Problem& pr);
size_t route_group_ws_bytes(const Problem& pr, int64_t n_q);
cudaError_t launch_route_group(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                               int32_t* sel, float* sel_score, void* ws, cudaStream_t st);
cudaError_t launch_route_tc(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                            const float* summ, int32_t* sel, float* sel_score, void* ws,
                            cudaStream_t st);

// Reference-quality attention: one warp per query row, any dtype.
cudaError_t launch_attend_rows(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                               const void* K, const void* V, const int32_t* sel, void* O,
                               float* lse, uint32_t* err, cudaStream_t st);

// The 8-bit cache (quant.cu): quantised rows and their span summaries.
cudaError_t launch_quantize_kv(const Problem& pr, const void* K, const void* V, int64_t t0, int64_t t1,
                               int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, cudaStream_t st);
cudaError_t launch_summaries_q8(const Problem& pr, const int8_t* Kq, const float* Ks, int64_t j0, int64_t j1,
                                float* summ, cudaStream_t st);
// Decode attention over the 8-bit cache (16-bit Q and O, d = 128).
cudaError_t launch_attend_decode_q8(const Problem& pr, const void* Q, int64_t pos, const int8_t* Kq,
                                    const float* Ks, const int8_t* Vq, const float* Vs, const int32_t* sel,
                                    void* O, float* lse, void* ws, cudaStream_t st);

// Decode attention fast path (16-bit types): plan, split spans, merge.
size_t decode_ws_bytes(const Problem& pr);
bool decode_fast_supported(const Problem& pr);
cudaError_t launch_attend_decode(const Problem& pr, const void* Q, int64_t pos, const void* K,
                                 const void* V, const int32_t* sel, void* O, float* lse, void* ws,
                                 cudaStream_t st);

// A whole decode step (16-bit types, the fast decode path): route with the
// plan built in the route kernel's cluster, then the attention and the
// merge -- three launches.  The group variant selects one top-k per kv-head
// group from the summed queries.
cudaError_t launch_decode_step(const Problem& pr, const void* Q, int64_t pos, const float* summ, const void* K,
                               const void* V, int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st);
cudaError_t launch_decode_step_group(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                     const void* K, const void* V, int32_t* sel, void* O, float* lse, void* ws,
                                     cudaStream_t st);
cudaError_t launch_decode_step_q8(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                  const int8_t* Kq, const float* Ks, const int8_t* Vq, const float* Vs,
                                  int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st);
cudaError_t launch_quantize_kv4(const Problem& pr, const void* K, const void* V, int64_t t0, int64_t t1,
                                uint32_t* Kq4, float* Ks, uint32_t* Vq4, float* Vs, cudaStream_t st);
cudaError_t launch_summaries_q4(const Problem& pr, const uint32_t* Kq4, const float* Ks, int64_t j0, int64_t j1,
                                float* summ, cudaStream_t st);
cudaError_t launch_attend_decode_q4(const Problem& pr, const void* Q, int64_t pos, const uint32_t* Kq4,
                                    const float* Ks, const uint32_t* Vq4, const float* Vs, const int32_t* sel,
                                    void* O, float* lse, void* ws, cudaStream_t st);
cudaError_t launch_decode_step_q4(const Problem& pr, const void* Q, int64_t pos, const float* summ,
                                  const uint32_t* Kq4, const float* Ks, const uint32_t* Vq4, const float* Vs,
                                  int32_t* sel, void* O, float* lse, void* ws, cudaStream_t st);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st);

// Prefill attention fast path (16-bit types): dispatch, span tiles, merge.
size_t prefill_ws_bytes(const Problem& pr, int64_t n_q);
bool prefill_fast_supported(const Problem& pr);
cudaError_t launch_attend_prefill(const Problem& pr, const void* Q, int64_t n_q, int64_t q_pos0,
                                  const void* K, const void* V, const int32_t* sel, void* O,
                                  float* lse, void* ws, cudaStream_t st);

}  // namespace ssa

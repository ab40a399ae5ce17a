// ssa_api.cu -- the C ABI declared in include/ssa.h: argument validation,
// workspace sizing and dispatch to the kernels.  Nothing here throws; every
// failure is a status code.
#include <math.h>
#include <stdint.h>

#include "internal.h"

using namespace ssa;

int ssa::check_params(const ssa_params* p, Problem* pr) {
  if (!p) return SSA_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->S < 1 || p->topk < 1 || p->L < 0 || p->L_cap < 0)
    return SSA_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return SSA_ERR_INVALID_ARG;
  if (p->dtype != SSA_F32 && p->dtype != SSA_BF16 && p->dtype != SSA_F16) return SSA_ERR_INVALID_ARG;
  if (!(p->scale >= 0.f) || isinf(p->scale)) return SSA_ERR_INVALID_ARG;  // NaN, negative, inf
  const int64_t L_cap = p->L_cap ? p->L_cap : p->L;
  if (L_cap < p->L) return SSA_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return SSA_ERR_UNSUPPORTED;
  if (p->topk > 64) return SSA_ERR_UNSUPPORTED;
  if (p->Hq / p->Hkv > 16) return SSA_ERR_UNSUPPORTED;
  if (p->B > 65535 || p->Hkv > 65535) return SSA_ERR_UNSUPPORTED;
  // element counts of K/V and summ must fit int64 comfortably
  const double kv = (double)p->B * p->Hkv * (double)L_cap * p->d;
  if (kv > 4.0e18) return SSA_ERR_UNSUPPORTED;
  pr->B = p->B;
  pr->Hq = p->Hq;
  pr->Hkv = p->Hkv;
  pr->d = p->d;
  pr->g = p->Hq / p->Hkv;
  pr->L = p->L;
  pr->L_cap = L_cap;
  pr->S = p->S;
  pr->topk = p->topk;
  pr->scale = p->scale > 0.f ? p->scale : 1.f / sqrtf((float)p->d);
  pr->dtype = p->dtype;
  pr->ns_cap = (L_cap + p->S - 1) / p->S;
  return SSA_OK;
}

namespace {

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A pointer the kernels may dereference: device or managed memory, or
// page-locked host memory mapped into the device's address space at the same
// address (unified addressing).  Null passes (optional arguments).
bool device_accessible(const void* p) {
  if (!p) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SSA_OK : SSA_ERR_CUDA; }

// The tensor-core prefill path takes 16-bit inputs whose row ids fit its
// 32-bit bucket entries; everything else runs the row kernel.
bool prefill_fast(const Problem& pr, int64_t n_q) {
  return prefill_fast_supported(pr) && prefill_ws_bytes(pr, n_q) > 0;
}

size_t ws_need(const Problem& pr, int64_t n_q, int op) {
  if (op == SSA_OP_ROUTE) return route_tc_supported(pr, n_q) ? kWsHeader + route_tc_ws_bytes(pr) : 0;
  if (op == SSA_OP_DECODE)
    return kWsHeader + (decode_fast_supported(pr) ? decode_ws_bytes(pr) : 0);
  if (op == SSA_OP_PREFILL) return kWsHeader + (prefill_fast(pr, n_q) ? prefill_ws_bytes(pr, n_q) : 0);
  if (op == SSA_OP_ROUTE_GROUP) return kWsHeader + route_group_ws_bytes(pr, n_q);
  return 0;
}

int check_ws(const Problem& pr, int64_t n_q, int op, const void* ws, size_t ws_bytes) {
  const size_t need = ws_need(pr, n_q, op);
  if (need == 0) return SSA_OK;
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return SSA_ERR_WORKSPACE;
  return SSA_OK;
}

}  // namespace

extern "C" {

int ssa_version(void) { return kVersion; }

const char* ssa_status_string(int status) {
  switch (status) {
    case SSA_OK: return "ok";
    case SSA_ERR_INVALID_ARG: return "invalid argument";
    case SSA_ERR_UNSUPPORTED: return "unsupported parameters";
    case SSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSA_ERR_CUDA: return "CUDA error";
    case SSA_ERR_DEVICE: return "device-detected error (see the workspace error bits)";
    case SSA_ERR_IO: return "snapshot file error (open, read, write or format)";
    default: return "unknown status";
  }
}

int ssa_attend_path(const ssa_params* p, int64_t n_q, int op) {
  Problem pr;
  if (check_params(p, &pr) != SSA_OK || n_q < 0) return SSA_PATH_INVALID;
  if (op == SSA_OP_DECODE) return decode_fast_supported(pr) ? SSA_PATH_FAST : SSA_PATH_ROWS;
  if (op == SSA_OP_PREFILL) return prefill_fast(pr, n_q) ? SSA_PATH_FAST : SSA_PATH_ROWS;
  return SSA_PATH_INVALID;
}

size_t ssa_workspace_size(const ssa_params* p, int64_t n_q, int op) {
  Problem pr;
  if (check_params(p, &pr) != SSA_OK || n_q < 0) return 0;
  return ws_need(pr, n_q, op);
}

int ssa_build_summaries(const ssa_params* p, const void* K, int64_t span_begin, int64_t span_end,
                        float* summ, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!K || !summ || !aligned16(K) || !aligned16(summ)) return SSA_ERR_INVALID_ARG;
  const int64_t ns_valid = (pr.L + pr.S - 1) / pr.S;
  if (span_begin < 0 || span_end < span_begin || span_end > ns_valid) return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_summaries(pr, K, span_begin, span_end, summ,
                                      static_cast<cudaStream_t>(stream)));
}

int ssa_route(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
              int32_t* sel, float* sel_score, void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (n_q < 0 || q_pos0 < 0 || q_pos0 + n_q > pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !sel || !aligned16(Q) || !aligned16(summ)) return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, n_q, SSA_OP_ROUTE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (route_tc_supported(pr, n_q))
    return cuda_status(launch_route_tc(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws, st));
  return cuda_status(launch_route(pr, Q, n_q, q_pos0, summ, sel, sel_score, st));
}

int ssa_route_group(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0, const float* summ,
                    int32_t* sel, float* sel_score, void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (n_q < 0 || q_pos0 < 0 || q_pos0 + n_q > pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !sel || !aligned16(Q) || !aligned16(summ)) return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, n_q, SSA_OP_ROUTE_GROUP, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  return cuda_status(launch_route_group(pr, Q, n_q, q_pos0, summ, sel, sel_score, ws,
                                        static_cast<cudaStream_t>(stream)));
}

int ssa_attend_decode(const ssa_params* p, const void* Q, int64_t pos, const void* K, const void* V,
                      const int32_t* sel, void* O, float* lse, void* ws, size_t ws_bytes,
                      void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !K || !V || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_fast_supported(pr))
    return cuda_status(launch_attend_decode(pr, Q, pos, K, V, sel, O, lse, ws, st));
  return cuda_status(launch_attend_rows(pr, Q, 1, pos, K, V, sel, O, lse, ws_error(ws), st));
}

int ssa_decode_step(const ssa_params* p, const void* Q, int64_t pos, const float* summ, const void* K,
                    const void* V, int32_t* sel, void* O, float* lse, void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !K || !V || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(summ) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_fast_supported(pr)) {
    // Q, sel, O and lse may live in mapped page-locked host memory
    if (!device_accessible(Q) || !device_accessible(sel) || !device_accessible(O) || !device_accessible(lse))
      return SSA_ERR_INVALID_ARG;
    return cuda_status(launch_decode_step(pr, Q, pos, summ, K, V, sel, O, lse, ws, st));
  }
  // fp32 (or shapes the fast path does not take): the two calls in sequence
  rc = cuda_status(launch_route(pr, Q, 1, pos, summ, sel, nullptr, st));
  if (rc != SSA_OK) return rc;
  return cuda_status(launch_attend_rows(pr, Q, 1, pos, K, V, sel, O, lse, ws_error(ws), st));
}

int ssa_decode_step_group(const ssa_params* p, const void* Q, int64_t pos, const float* summ, const void* K,
                          const void* V, int32_t* sel, void* O, float* lse, void* ws, size_t ws_bytes,
                          void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!decode_fast_supported(pr)) return SSA_ERR_UNSUPPORTED;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !K || !V || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(summ) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  if (!device_accessible(Q) || !device_accessible(sel) || !device_accessible(O) || !device_accessible(lse))
    return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_decode_step_group(pr, Q, pos, summ, K, V, sel, O, lse, ws,
                                              static_cast<cudaStream_t>(stream)));
}

int ssa_attend_prefill(const ssa_params* p, const void* Q, int64_t n_q, int64_t q_pos0,
                       const void* K, const void* V, const int32_t* sel, void* O, float* lse,
                       void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (n_q < 0 || q_pos0 < 0 || q_pos0 + n_q > pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !K || !V || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, n_q, SSA_OP_PREFILL, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  if (n_q == 0) return SSA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (prefill_fast(pr, n_q))
    return cuda_status(launch_attend_prefill(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws, st));
  return cuda_status(launch_attend_rows(pr, Q, n_q, q_pos0, K, V, sel, O, lse, ws_error(ws), st));
}

int ssa_quantize_kv(const ssa_params* p, const void* K, const void* V, int64_t t_begin, int64_t t_end,
                    int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.L_cap % 32 != 0) return SSA_ERR_UNSUPPORTED;
  if (t_begin < 0 || t_end < t_begin || t_end > pr.L) return SSA_ERR_INVALID_ARG;
  if (!K || !V || !Kq || !Ks || !Vq || !Vs) return SSA_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kq) || !aligned16(Ks) || !aligned16(Vq) || !aligned16(Vs))
    return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_kv(pr, K, V, t_begin, t_end, Kq, Ks, Vq, Vs,
                                        static_cast<cudaStream_t>(stream)));
}

int ssa_build_summaries_q8(const ssa_params* p, const int8_t* Kq, const float* Ks, int64_t span_begin,
                           int64_t span_end, float* summ, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.L_cap % 32 != 0) return SSA_ERR_UNSUPPORTED;
  if (!Kq || !Ks || !summ || !aligned16(Kq) || !aligned16(Ks) || !aligned16(summ)) return SSA_ERR_INVALID_ARG;
  const int64_t ns_valid = (pr.L + pr.S - 1) / pr.S;
  if (span_begin < 0 || span_end < span_begin || span_end > ns_valid) return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_summaries_q8(pr, Kq, Ks, span_begin, span_end, summ,
                                         static_cast<cudaStream_t>(stream)));
}

int ssa_attend_decode_q8(const ssa_params* p, const void* Q, int64_t pos, const int8_t* Kq, const float* Ks,
                         const int8_t* Vq, const float* Vs, const int32_t* sel, void* O, float* lse, void* ws,
                         size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.d != 128 || pr.L_cap % 32 != 0 || (pr.dtype != SSA_BF16 && pr.dtype != SSA_F16) ||
      !decode_fast_supported(pr))
    return SSA_ERR_UNSUPPORTED;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !Kq || !Ks || !Vq || !Vs || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(Kq) || !aligned16(Ks) || !aligned16(Vq) || !aligned16(Vs) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  return cuda_status(launch_attend_decode_q8(pr, Q, pos, Kq, Ks, Vq, Vs, sel, O, lse, ws,
                                             static_cast<cudaStream_t>(stream)));
}

int ssa_decode_step_q8(const ssa_params* p, const void* Q, int64_t pos, const float* summ, const int8_t* Kq,
                       const float* Ks, const int8_t* Vq, const float* Vs, int32_t* sel, void* O, float* lse,
                       void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.d != 128 || pr.L_cap % 32 != 0 || (pr.dtype != SSA_BF16 && pr.dtype != SSA_F16) ||
      !decode_fast_supported(pr))
    return SSA_ERR_UNSUPPORTED;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !Kq || !Ks || !Vq || !Vs || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(summ) || !aligned16(Kq) || !aligned16(Ks) || !aligned16(Vq) ||
      !aligned16(Vs) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  if (!device_accessible(Q) || !device_accessible(sel) || !device_accessible(O) || !device_accessible(lse))
    return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_decode_step_q8(pr, Q, pos, summ, Kq, Ks, Vq, Vs, sel, O, lse, ws,
                                           static_cast<cudaStream_t>(stream)));
}

// The 4-bit cache: d = 128, bf16 / fp16 queries, L_cap a multiple of 32.
bool q4_supported(const Problem& pr) {
  return pr.d == 128 && pr.L_cap % 32 == 0 && (pr.dtype == SSA_BF16 || pr.dtype == SSA_F16) &&
         decode_fast_supported(pr);
}

int ssa_quantize_kv4(const ssa_params* p, const void* K, const void* V, int64_t t_begin, int64_t t_end,
                     void* Kq4, float* Ks, void* Vq4, float* Vs, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.d != 128 || pr.L_cap % 32 != 0) return SSA_ERR_UNSUPPORTED;
  if (t_begin < 0 || t_end < t_begin || t_end > pr.L) return SSA_ERR_INVALID_ARG;
  if (!K || !V || !Kq4 || !Ks || !Vq4 || !Vs) return SSA_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kq4) || !aligned16(Ks) || !aligned16(Vq4) || !aligned16(Vs))
    return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_kv4(pr, K, V, t_begin, t_end, static_cast<uint32_t*>(Kq4), Ks,
                                         static_cast<uint32_t*>(Vq4), Vs, static_cast<cudaStream_t>(stream)));
}

int ssa_build_summaries_q4(const ssa_params* p, const void* Kq4, const float* Ks, int64_t span_begin,
                           int64_t span_end, float* summ, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (pr.d != 128 || pr.L_cap % 32 != 0) return SSA_ERR_UNSUPPORTED;
  if (!Kq4 || !Ks || !summ || !aligned16(Kq4) || !aligned16(Ks) || !aligned16(summ)) return SSA_ERR_INVALID_ARG;
  const int64_t ns_valid = (pr.L + pr.S - 1) / pr.S;
  if (span_begin < 0 || span_end < span_begin || span_end > ns_valid) return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_summaries_q4(pr, static_cast<const uint32_t*>(Kq4), Ks, span_begin, span_end, summ,
                                         static_cast<cudaStream_t>(stream)));
}

int ssa_attend_decode_q4(const ssa_params* p, const void* Q, int64_t pos, const void* Kq4, const float* Ks,
                         const void* Vq4, const float* Vs, const int32_t* sel, void* O, float* lse, void* ws,
                         size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!q4_supported(pr)) return SSA_ERR_UNSUPPORTED;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !Kq4 || !Ks || !Vq4 || !Vs || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(Kq4) || !aligned16(Ks) || !aligned16(Vq4) || !aligned16(Vs) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  return cuda_status(launch_attend_decode_q4(pr, Q, pos, static_cast<const uint32_t*>(Kq4), Ks,
                                             static_cast<const uint32_t*>(Vq4), Vs, sel, O, lse, ws,
                                             static_cast<cudaStream_t>(stream)));
}

int ssa_decode_step_q4(const ssa_params* p, const void* Q, int64_t pos, const float* summ, const void* Kq4,
                       const float* Ks, const void* Vq4, const float* Vs, int32_t* sel, void* O, float* lse,
                       void* ws, size_t ws_bytes, void* stream) {
  Problem pr;
  int rc = check_params(p, &pr);
  if (rc != SSA_OK) return rc;
  if (!q4_supported(pr)) return SSA_ERR_UNSUPPORTED;
  if (pos < 0 || pos >= pr.L) return SSA_ERR_INVALID_ARG;
  if (!Q || !summ || !Kq4 || !Ks || !Vq4 || !Vs || !sel || !O) return SSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(summ) || !aligned16(Kq4) || !aligned16(Ks) || !aligned16(Vq4) ||
      !aligned16(Vs) || !aligned16(O))
    return SSA_ERR_INVALID_ARG;
  rc = check_ws(pr, 1, SSA_OP_DECODE, ws, ws_bytes);
  if (rc != SSA_OK) return rc;
  if (!device_accessible(Q) || !device_accessible(sel) || !device_accessible(O) || !device_accessible(lse))
    return SSA_ERR_INVALID_ARG;
  return cuda_status(launch_decode_step_q4(pr, Q, pos, summ, static_cast<const uint32_t*>(Kq4), Ks,
                                           static_cast<const uint32_t*>(Vq4), Vs, sel, O, lse, ws,
                                           static_cast<cudaStream_t>(stream)));
}

int ssa_selftest_wait_timeout(uint64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  if (limit_ns > 1000000000ull) return SSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kWsHeader) return SSA_ERR_WORKSPACE;
  return cuda_status(launch_wait_selftest(ws_error(ws), limit_ns, static_cast<cudaStream_t>(stream)));
}

int ssa_workspace_error(void* ws, uint32_t* bits, void* stream) {
  if (!ws) return SSA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSA_ERR_CUDA;
  if (cudaMemcpy(&host, ws, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess) return SSA_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof host) != cudaSuccess) return SSA_ERR_CUDA;
  if (bits) *bits = host;
  return host ? SSA_ERR_DEVICE : SSA_OK;
}

}  // extern "C"

// synth_dev.cu -- device filler for the seeded synthetic inputs.
//
// Same element definition as the host filler (synth_core.h); the multiply
// and the add use __fmul_rn / __fadd_rn so nvcc cannot contract them into an
// FMA, and the conversions to bf16 / fp16 are the integer round-to-nearest-
// even helpers of synth_core.h.  The result is bit-identical to the host
// filler for every element.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

namespace {

template <int DT>
__global__ void synth_fill_kernel(void* __restrict__ out, int64_t e0, int64_t e1, synth_spec sp) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = e0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < e1; e += stride) {
    float v = synth_value(&sp, (uint64_t)e);
    int64_t i = e - e0;
    if (DT == SYNTH_F32) {
      static_cast<float*>(out)[i] = v;
    } else if (DT == SYNTH_BF16) {
      static_cast<uint16_t*>(out)[i] = synth_f32_to_bf16(v);
    } else {
      static_cast<uint16_t*>(out)[i] = synth_f32_to_f16(v);
    }
  }
}

}  // namespace

// Returns 0 on success, -1 on a bad argument, or the CUDA error code + 1000.
extern "C" int synth_fill_device(int32_t dtype, void* out, int64_t e0, int64_t e1, int64_t d,
                                 int64_t rows_per_head, int64_t S, const float* bias,
                                 const int32_t* attempt, uint32_t seed, uint32_t tid,
                                 void* stream) {
  if (!out || e1 < e0 || d <= 0) return -1;
  if (bias && (rows_per_head <= 0 || S <= 0)) return -1;
  if (e1 == e0) return 0;
  synth_spec sp;
  sp.d = d;
  sp.rows_per_head = rows_per_head > 0 ? rows_per_head : 1;
  sp.S = S > 0 ? S : 1;
  sp.bias = bias;
  sp.attempt = attempt;
  sp.seed = seed;
  sp.tid = tid;
  sp.dtype = dtype;
  int64_t n = e1 - e0;
  int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 148 * 64) blocks = 148 * 64;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case SYNTH_F32: synth_fill_kernel<SYNTH_F32><<<(unsigned)blocks, threads, 0, st>>>(out, e0, e1, sp); break;
    case SYNTH_BF16: synth_fill_kernel<SYNTH_BF16><<<(unsigned)blocks, threads, 0, st>>>(out, e0, e1, sp); break;
    case SYNTH_F16: synth_fill_kernel<SYNTH_F16><<<(unsigned)blocks, threads, 0, st>>>(out, e0, e1, sp); break;
    default: return -1;
  }
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? 0 : 1000 + (int)err;
}

// bench_alu_probe.cu -- throughput probes for the scan's arithmetic units on the local
// GPU (measurement support for bench.py; not part of libvarlen_ssm).
//
//   kind 0: FP32 FMA        (fma.rn.f32, 8 independent chains per thread)
//   kind 1: packed FP32 FMA (fma.rn.f32x2, 8 chains, 2 lanes each)
//   kind 2: MUFU exp2       (ex2.approx.ftz.f32, 8 chains)
//
// vssm_probe_alu returns operations per second (one FMA = one operation, a
// packed FMA = two, one ex2 = one) measured with CUDA events over a launch of
// `blocks` x 256 threads running `iters` iterations.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void __launch_bounds__(256) ffma_probe(float* out, int iters, float a, float b) {
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = threadIdx.x * 1e-3f + k;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = fmaf(x[k], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += x[k];
  if (s == 1234.5f) out[blockIdx.x] = s;  // keeps the chains alive
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}

__global__ void __launch_bounds__(256) ffma2_probe(float* out, int iters, float a, float b) {
  unsigned long long x[8];
  const unsigned long long av = pack2(a, a), bv = pack2(b, b);
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = pack2(threadIdx.x * 1e-3f + k, k * 0.5f);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[k]) : "l"(av), "l"(bv));
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += __uint_as_float((unsigned)x[k]) + __uint_as_float((unsigned)(x[k] >> 32));
  if (s == 1234.5f) out[blockIdx.x] = s;
}

__global__ void __launch_bounds__(256) ex2_probe(float* out, int iters) {
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = threadIdx.x * 1e-4f + k * 0.1f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[k]) : "f"(-x[k]));
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += x[k];
  if (s == 1234.5f) out[blockIdx.x] = s;
}

}  // namespace

extern "C" int vssm_probe_alu(int kind, int blocks, int iters, double* ops_per_s) {
  float* out = nullptr;
  if (cudaMalloc(&out, sizeof(float) * (size_t)blocks) != cudaSuccess) return -1;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  auto launch = [&](int it) {
    if (kind == 0) ffma_probe<<<blocks, 256>>>(out, it, 0.999f, 1e-3f);
    else if (kind == 1) ffma2_probe<<<blocks, 256>>>(out, it, 0.999f, 1e-3f);
    else ex2_probe<<<blocks, 256>>>(out, it);
  };
  launch(iters / 10 + 1);  // warm up
  cudaEventRecord(e0);
  launch(iters);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  float ms = 0.0f;
  cudaEventElapsedTime(&ms, e0, e1);
  const cudaError_t err = cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  if (err != cudaSuccess || ms <= 0.0f) return -2;
  const double per_iter = kind == 1 ? 16.0 : 8.0;
  *ops_per_s = (double)blocks * 256.0 * iters * per_iter / (ms * 1e-3);
  return 0;
}

// probe.cu -- measured throughput ceilings of the instruction paths the GEMM
// kernels use where no measured peak is supplied: warp-level IMMA
// (mma.sync.m16n8k32 s8 -> s32, the INT8 consumer) and FFMA (the FP32 path).
// Each probe runs independent dependency chains of one instruction on every
// SM long enough (tens of ms) to reach steady clocks, for a few warps-per-SM
// settings, and returns the best rate.  Nothing is read from memory.
#include <cstdio>

#include "gp_device.cuh"
#include "gemm_probe.h"

namespace gp {
namespace {

__device__ int32_t g_probe_sink;

template <int CHAINS>
__global__ void probe_imma_kernel(int iters, int32_t seed) {
  int32_t acc[CHAINS][4];
#pragma unroll
  for (int u = 0; u < CHAINS; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = u;
  const uint32_t a[4] = {static_cast<uint32_t>(seed) ^ threadIdx.x, threadIdx.x * 3u, 0x01020304u, 0x7f7f0101u};
  const uint32_t b0 = 0x01fe01feu ^ threadIdx.x, b1 = 0x03050709u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int u = 0; u < CHAINS; ++u) mma_s8_16832(acc[u], a, b0, b1);
  }
  int32_t s = 0;
#pragma unroll
  for (int u = 0; u < CHAINS; ++u) s += acc[u][0] + acc[u][1] + acc[u][2] + acc[u][3];
  if (s == seed) g_probe_sink = s;   // practically never; keeps the chains live
}

template <int CHAINS>
__global__ void probe_ffma_kernel(int iters, float seed) {
  float x[CHAINS];
#pragma unroll
  for (int u = 0; u < CHAINS; ++u) x[u] = seed + threadIdx.x * 1e-3f + u;
  const float m = 0.99999f, c = 1e-6f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int u = 0; u < CHAINS; ++u) x[u] = fmaf(x[u], m, c);
  }
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < CHAINS; ++u) s += x[u];
  if (s == seed) g_probe_sink = 1;
}

template <typename F>
cudaError_t time_launch(F launch, cudaStream_t st, float* ms) {
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return e;
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) { cudaEventDestroy(e0); return e; }
  launch();   // warm-up (clocks, module load)
  cudaEventRecord(e0, st);
  launch();
  cudaEventRecord(e1, st);
  e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return e;
}

}  // namespace
}  // namespace gp

extern "C" int gemm_probe_peak(int kind, double* ops_per_s, void* stream) {
  using namespace gp;
  if (!ops_per_s || (kind != GP_PROBE_IMMA_S8 && kind != GP_PROBE_FFMA_F32)) return GP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GP_ERR_CUDA;
  double best = 0.0;
  const int warps_per_sm[3] = {8, 16, 32};
  for (int w : warps_per_sm) {
    const int threads = 256;
    const int blocks = sms * (w * 32 / threads);
    float ms = 0.f;
    cudaError_t e;
    double ops;
    if (kind == GP_PROBE_IMMA_S8) {
      const int iters = 32768;
      e = time_launch([&] { probe_imma_kernel<8><<<blocks, threads, 0, st>>>(iters, 12345); }, st, &ms);
      ops = static_cast<double>(blocks) * (threads / 32) * iters * 8 * (2.0 * 16 * 8 * 32);
    } else {
      const int iters = 262144;
      e = time_launch([&] { probe_ffma_kernel<8><<<blocks, threads, 0, st>>>(iters, 0.5f); }, st, &ms);
      ops = static_cast<double>(blocks) * threads * iters * 8 * 2.0;
    }
    if (e != cudaSuccess) return GP_ERR_CUDA;
    if (ms > 0.f && ops / (ms * 1e-3) > best) best = ops / (ms * 1e-3);
  }
  *ops_per_s = best;
  return GP_OK;
}

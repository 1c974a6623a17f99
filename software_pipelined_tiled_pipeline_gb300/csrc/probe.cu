// probe.cu -- measured throughput ceilings of the instruction paths the GEMM
// kernels use where no measured peak is supplied: warp-level IMMA
// (mma.sync.m16n8k32 s8 -> s32, the INT8 consumer) and FFMA (the FP32 path).
// Each probe runs independent dependency chains of one instruction on every
// SM long enough (tens of ms) to reach steady clocks, for a few warps-per-SM
// settings, and returns the best rate.  Nothing is read from memory.  The HBM
// probes time plain 16-byte stores, loads and copies over a caller's buffer.
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

// HBM probes: every thread takes 16-byte elements i, i + stride, ... of the
// buffer, four of them in flight per iteration.
__global__ void probe_write_kernel(uint4* __restrict__ p, size_t n, uint32_t seed) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint4 v = make_uint4(seed ^ threadIdx.x, seed + 1u, seed + 2u, blockIdx.x);
  for (; i + 3 * stride < n; i += 4 * stride) {
    p[i] = v;
    p[i + stride] = v;
    p[i + 2 * stride] = v;
    p[i + 3 * stride] = v;
  }
  for (; i < n; i += stride) p[i] = v;
}

__global__ void probe_read_kernel(const uint4* __restrict__ p, size_t n, uint32_t seed) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = p[i], b = p[i + stride], c = p[i + 2 * stride], d = p[i + 3 * stride];
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n; i += stride) {
    const uint4 a = p[i];
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  if (acc == seed) g_probe_sink = static_cast<int32_t>(acc);   // keeps the loads live
}

__global__ void probe_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
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

extern "C" int gemm_probe_hbm(int kind, void* buf, size_t bytes, double* bytes_per_s, void* stream) {
  using namespace gp;
  if (!buf || !bytes_per_s) return GP_ERR_ARG;
  if (kind != GP_PROBE_HBM_WRITE && kind != GP_PROBE_HBM_READ && kind != GP_PROBE_HBM_COPY) return GP_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(buf) & 15u) != 0 || bytes < (size_t(1) << 20) || bytes % 32 != 0) return GP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GP_ERR_CUDA;
  uint4* p = static_cast<uint4*>(buf);
  const size_t n = bytes / 16;   // 16-byte elements
  const size_t half = n / 2;     // the copy moves the first half onto the second
  double best = 0.0;
  const int blocks_per_sm[3] = {2, 4, 8};
  for (int b : blocks_per_sm) {
    const int blocks = sms * b;
    auto launch = [&] {
      if (kind == GP_PROBE_HBM_WRITE)
        probe_write_kernel<<<blocks, 512, 0, st>>>(p, n, 0x9e3779b9u);
      else if (kind == GP_PROBE_HBM_READ)
        probe_read_kernel<<<blocks, 512, 0, st>>>(p, n, 0x9e3779b9u);
      else
        probe_copy_kernel<<<blocks, 512, 0, st>>>(p, p + half, half);
    };
    const double moved = kind == GP_PROBE_HBM_COPY ? 2.0 * static_cast<double>(half) * 16 : static_cast<double>(n) * 16;
    for (int rep = 0; rep < 5; ++rep) {
      float ms = 0.f;
      if (time_launch(launch, st, &ms) != cudaSuccess) return GP_ERR_CUDA;
      if (ms > 0.f && moved / (ms * 1e-3) > best) best = moved / (ms * 1e-3);
    }
  }
  *bytes_per_s = best;
  return GP_OK;
}

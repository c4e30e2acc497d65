// Calibration of the cost-model constants on the running GPU.
//
// The design note "block coalescing" decides grouping and packing with
// calibrated constants ("The crossover decides whether to coalesce": launch
// cost against flop rate; "Interleaved vs contiguous": pack cost against
// launch savings).  Its numbers are not given, so they are measured here:
//   - the FP64 pipe rate with every lane active, and with one lane in four
//     active (whether idle lanes of a warp still cost pipe time decides how
//     tightly tiny groups must be packed onto lanes);
//   - the cost of one kernel launch on a stream;
//   - the bandwidth of a plain device-to-device copy kernel (the gather).
#include <cuda_runtime.h>

#include <chrono>

#include "bs_host.h"

namespace bs {

namespace {

constexpr int kFmaIters = 4096;

// Eight independent FMA chains per thread keep the pipe busy; `active`
// lanes of each warp do the work, the others skip it.
__global__ void dfma_probe(double *out, double seed, int active) {
  const int lane = threadIdx.x & 31;
  if (lane >= active) return;
  double a0 = seed + threadIdx.x, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3, a4 = a0 + 4, a5 = a0 + 5, a6 = a0 + 6,
         a7 = a0 + 7;
  const double m = 0.999999, c = 1e-7;
#pragma unroll 4
  for (int i = 0; i < kFmaIters; ++i) {
    a0 = fma(a0, m, c);
    a1 = fma(a1, m, c);
    a2 = fma(a2, m, c);
    a3 = fma(a3, m, c);
    a4 = fma(a4, m, c);
    a5 = fma(a5, m, c);
    a6 = fma(a6, m, c);
    a7 = fma(a7, m, c);
  }
  const double s = a0 + a1 + a2 + a3 + a4 + a5 + a6 + a7;
  if (s == 12345.678) out[blockIdx.x * blockDim.x + threadIdx.x] = s;   // keeps the loop alive
}

__global__ void empty_kernel() {}

__global__ void copy_probe(const double4_32a *src, double4_32a *dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

}  // namespace bs

extern "C" bs_status bs_calibrate(bs_calibration *out, void *stream) {
  using namespace bs;
  if (!out) return BS_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BS_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return BS_ERR_CUDA;
  double *scratch = nullptr;
  void *bufs = nullptr;
  const size_t copy_bytes = (size_t)1 << 30;
  bs_status st = BS_OK;
  auto timed = [&](auto &&launch, int reps) -> double {
    launch();
    cudaEventRecord(e0, s);
    for (int r = 0; r < reps; ++r) launch();
    cudaEventRecord(e1, s);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    return ms / reps;
  };
  do {
    const int blocks = sms * 8, threads = 256;
    if (cudaMalloc(&scratch, (size_t)blocks * threads * sizeof(double)) != cudaSuccess) {
      st = BS_ERR_OOM;
      break;
    }
    for (int variant = 0; variant < 2; ++variant) {
      const int active = variant == 0 ? 32 : 8;
      const double ms = timed([&] { dfma_probe<<<blocks, threads, 0, s>>>(scratch, 1.0, active); }, 5);
      const double flops = 2.0 * 8 * kFmaIters * (double)blocks * (threads / 32) * active;
      if (variant == 0) out->fp64_gflops = flops / (ms * 1e6);
      else out->fp64_gflops_quarter_warp = flops / (ms * 1e6);
    }
    out->launch_us = 1e3 * timed([&] { empty_kernel<<<1, 32, 0, s>>>(); }, 2000);
    if (cudaMalloc(&bufs, 2 * copy_bytes) != cudaSuccess) {
      st = BS_ERR_OOM;
      break;
    }
    const size_t n4 = copy_bytes / sizeof(double4_32a);
    const double ms = timed([&] {
      copy_probe<<<sms * 8, 256, 0, s>>>((const double4_32a *)bufs, (double4_32a *)((char *)bufs + copy_bytes), n4);
    }, 10);
    out->copy_gbs = 2.0 * copy_bytes / (ms * 1e6);
    out->sm_count = sms;
    if (cudaGetLastError() != cudaSuccess) st = BS_ERR_CUDA;
  } while (false);
  cudaFree(scratch);
  cudaFree(bufs);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return st;
}

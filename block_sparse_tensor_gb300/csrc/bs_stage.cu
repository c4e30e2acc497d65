// Staging of the host-buffer entry point's inputs.
//
// When both operands sit in pinned host memory that the device can address,
// one kernel pulls them into the plan's device buffers: a single launch whose
// loads are spread over every SM, instead of one copy-engine transfer per
// operand, each with its own start-up cost.
#include <cuda_runtime.h>

#include "bs_host.h"

namespace bs {

namespace {

// Two byte ranges in one launch: 16-byte units, four loads in flight per
// thread, then the ragged bytes at the end of each range.
__global__ void stage_in_kernel(const int4 *s0, int4 *d0, int64_t u0, const int4 *s1, int4 *d1, int64_t u1, int r0,
                                int r1) {
  const int64_t n = u0 + u1;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t i = g;
  for (; i + 3 * stride < n; i += 4 * stride) {
    int4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t j = i + u * stride;
      v[u] = j < u0 ? s0[j] : s1[j - u0];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t j = i + u * stride;
      if (j < u0) d0[j] = v[u];
      else d1[j - u0] = v[u];
    }
  }
  for (; i < n; i += stride) {
    if (i < u0) d0[i] = s0[i];
    else d1[i - u0] = s1[i - u0];
  }
  if (g < r0) ((unsigned char *)(d0 + u0))[g] = ((const unsigned char *)(s0 + u0))[g];
  if (g < r1) ((unsigned char *)(d1 + u1))[g] = ((const unsigned char *)(s1 + u1))[g];
}

}  // namespace

cudaError_t launch_stage_in(const void *src0, void *dst0, size_t n0, const void *src1, void *dst1, size_t n1, int sms,
                            cudaStream_t s) {
  const int64_t u0 = (int64_t)(n0 / 16), u1 = (int64_t)(n1 / 16);
  int64_t grid = (u0 + u1 + 255) / 256;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;
  grid = grid < cap ? grid : cap;
  grid = grid > 1 ? grid : 1;
  stage_in_kernel<<<(int)grid, 256, 0, s>>>((const int4 *)src0, (int4 *)dst0, u0, (const int4 *)src1, (int4 *)dst1, u1,
                                            (int)(n0 % 16), (int)(n1 % 16));
  return cudaGetLastError();
}

}  // namespace bs

// Dense index of the SM a CTA runs on.
//
// The persistent FP64 kernel deals its tail work at plan time onto one queue
// per SM, and a CTA serves the queue of the SM it finds itself on.  The
// hardware's SM identifier (%smid) is not a dense 0 .. sm_count-1 range on
// parts with disabled SMs: it can run past sm_count with gaps, so taking it
// modulo the queue count would leave some queues without a home SM and give
// others two.  This file finds, once per device, the identifiers the device
// actually uses, by a short launch whose CTAs each record their %smid and
// stay resident for a few microseconds so that the CTAs spread over every SM;
// the sorted identifiers are then numbered 0 .. n-1.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "bs_host.h"

namespace bs {

namespace {

// CTA b records its SM identifier in out[b]; CTA 0 also records the
// identifier bound %nsmid in out[gridDim.x].  Each CTA then stays resident for
// hold_ns of global time (at most 1 << 20 polls), so that later CTAs of the
// grid land on other SMs.
__global__ void smid_probe_kernel(int32_t *out, uint64_t hold_ns) {
  if (threadIdx.x != 0) return;
  unsigned smid, nsmid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  asm volatile("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
  out[blockIdx.x] = (int32_t)smid;
  if (blockIdx.x == 0) out[gridDim.x] = (int32_t)nsmid;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int it = 0; it < (1 << 20); ++it) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > hold_ns) break;
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
std::vector<int16_t> g_map[kMaxDevices];

}  // namespace

size_t sm_probe_bytes(int sm_count) { return (size_t)(sm_count * 4 + 1) * sizeof(int32_t); }

bs_status sm_index_map(int device, int sm_count, void *dev_buf, cudaStream_t s, std::vector<int16_t> *out) {
  if (device < 0 || device >= kMaxDevices || sm_count <= 0) return BS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_map[device].empty()) {
    const int grid = sm_count * 4;
    const size_t bytes = sm_probe_bytes(sm_count);
    void *buf = dev_buf;
    if (!buf && cudaMalloc(&buf, bytes) != cudaSuccess) return BS_ERR_OOM;
    smid_probe_kernel<<<grid, 32, 0, s>>>((int32_t *)buf, 20000);
    std::vector<int32_t> ids((size_t)grid + 1);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(ids.data(), buf, bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (!dev_buf) cudaFree(buf);
    if (e != cudaSuccess) return BS_ERR_CUDA;
    const int32_t nsmid = std::max<int32_t>(ids[grid], 1);
    std::vector<int32_t> seen(ids.begin(), ids.begin() + grid);
    std::sort(seen.begin(), seen.end());
    seen.erase(std::unique(seen.begin(), seen.end()), seen.end());
    int32_t bound = nsmid;
    for (int32_t v : seen) bound = std::max(bound, v + 1);
    std::vector<int16_t> map((size_t)bound, (int16_t)-1);
    for (size_t t = 0; t < seen.size(); ++t)
      if (seen[t] >= 0) map[(size_t)seen[t]] = (int16_t)t;
    g_map[device] = std::move(map);
  }
  *out = g_map[device];
  return BS_OK;
}

}  // namespace bs

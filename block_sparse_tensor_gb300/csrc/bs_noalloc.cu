// bs_contract_noalloc: the FP64 contraction for callers that must not allocate
// device memory.
//
// Some callers cannot call cudaMalloc: code that runs under a memory manager
// owning all device memory (a framework's caching pool, a fixed per-process
// budget), or a steady-state loop that is not allowed to allocate after
// start-up.  bs_contract needs device memory of its own: the plan's task
// tables, the work counters of the persistent kernel and, for some plans, a
// gather workspace.  This entry point takes all of that from one file-scope
// device array of fixed size instead, so the only device memory it touches
// besides the caller's A, B and C is memory that exists from the moment the
// library is loaded (kNoAllocScratchBytes on every device that loads it, held
// until the process exits).
//
// The array is shared by every call: a call uploads its plan's tables into it,
// zeroes the work counters, and launches.  Calls that overlap on the GPU (two
// streams, or two host threads) race on it; order them on one stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "bs_plan.h"

namespace bs {

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB
static_assert(kNoAllocScratchBytes == (size_t)BS_NOALLOC_SCRATCH_BYTES, "header and file agree");

static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

// Device address of g_scratch per device, looked up on first use.  In host
// code the name g_scratch is only a host-side stand-in, so the address must
// come from the runtime.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

bs_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return BS_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return BS_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

}  // namespace bs

extern "C" bs_status bs_contract_noalloc(const bs_plan *P, const void *A, const void *B, void *C, void *stream) {
  using namespace bs;
  if (!P || !A || !B || !C) return BS_ERR_INVALID_ARG;
  if (P->dtype != BS_F64) return BS_ERR_UNSUPPORTED;
  if (P->C.nelems == 0) return BS_OK;
  cudaStream_t s = (cudaStream_t)stream;

  // carve the array: [counters+status | tables | gather workspaces]
  const size_t n_tasks = P->ts.tasks.size() * sizeof(Task);
  const size_t n_groups = P->gs.groups.size() * sizeof(Group);
  const size_t n_rsegs = P->gs.rsegs.size() * sizeof(RowSeg);
  const size_t n_ksegs = P->gs.ksegs.size() * sizeof(KSeg);
  const size_t n_tail = P->ts.tail_elems.size() * sizeof(int32_t);
  const size_t n_tdesc = P->ts.tdesc.size() * sizeof(TailDesc);
  const int nq = (int)std::max<size_t>(1, P->ts.tq_ptr.size()) - 1;
  const size_t n_ctr = counter_bytes(nq);
  const size_t n_pack = P->pack_copies.size() * sizeof(PackCopy);
  const size_t n_zero = P->zero_blocks.size() * sizeof(ZeroBlock);
  const size_t n_ws_a = P->pack_a ? (size_t)P->A_pk.nelems * sizeof(double) : 0;
  const size_t n_ws_b = P->pack_b ? (size_t)P->B_pk.nelems * sizeof(double) : 0;
  size_t off = n_ctr;
  const size_t o_tasks = off;
  off = align256(off + n_tasks);
  const size_t o_groups = off;
  off = align256(off + n_groups);
  const size_t o_rsegs = off;
  off = align256(off + n_rsegs);
  const size_t o_ksegs = off;
  off = align256(off + n_ksegs);
  const size_t o_tail = off;
  off = align256(off + n_tail);
  const size_t o_tdesc = off;
  off = align256(off + n_tdesc);
  const size_t o_pack = off;
  off = align256(off + n_pack);
  const size_t o_zero = off;
  off = align256(off + n_zero);
  const size_t o_ws_a = off;
  off = align256(off + n_ws_a);
  const size_t o_ws_b = off;
  off = align256(off + n_ws_b);
  if (off > kNoAllocScratchBytes) return BS_ERR_OVERFLOW;   // the plan does not fit the fixed array

  void *base = nullptr;
  bs_status st = scratch_for_current_device(&base);
  if (st != BS_OK) return st;
  char *b = (char *)base;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BS_ERR_CUDA;
  // the grid bs_contract launches for this plan: the plan's CTAs per SM, else the occupancy limit
  per_sm = P->opts.ctas_per_sm > 0 ? P->opts.ctas_per_sm : std::max(1, fp64_max_ctas_per_sm(P->ts.tasks.empty()));

  // the SM numbering of this device, found once (its probe writes into the array's head)
  std::vector<int16_t> sm_map;
  if (P->ts.tq_ptr.size() > 1) {
    if (sm_probe_bytes(sms) > kNoAllocScratchBytes) return BS_ERR_OVERFLOW;
    st = sm_index_map(dev, sms, b, s, &sm_map);
    if (st != BS_OK) return st;
  }

  auto up = [&](size_t o, const void *src, size_t n) -> bool {
    return n == 0 || cudaMemcpyAsync(b + o, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  // status word and both counter sets start at zero; the rest of the array is overwritten
  if (cudaMemsetAsync(b, 0, n_ctr, s) != cudaSuccess) return BS_ERR_CUDA;
  if (!up(o_tasks, P->ts.tasks.data(), n_tasks) || !up(o_groups, P->gs.groups.data(), n_groups) ||
      !up(o_rsegs, P->gs.rsegs.data(), n_rsegs) || !up(o_ksegs, P->gs.ksegs.data(), n_ksegs) ||
      !up(o_tail, P->ts.tail_elems.data(), n_tail) || !up(o_tdesc, P->ts.tdesc.data(), n_tdesc) ||
      !up(o_pack, P->pack_copies.data(), n_pack) ||
      !up(o_zero, P->zero_blocks.data(), n_zero))
    return BS_ERR_CUDA;

  const void *Ause = P->pack_a ? (const void *)(b + o_ws_a) : A;
  const void *Buse = P->pack_b ? (const void *)(b + o_ws_b) : B;
  if (!P->pack_copies.empty()) {
    PackParams pa{};
    pa.src = A;
    pa.dst = b + o_ws_a;
    pa.copies = (const PackCopy *)(b + o_pack);
    pa.ncopies = P->pack_split.total;
    pa.elem_bytes = 8;
    PackParams pb = pa;
    pb.src = B;
    pb.dst = b + o_ws_b;
    if (launch_pack2(pa, pb, P->pack_split, sms, s) != cudaSuccess) return BS_ERR_CUDA;
  }
  if (!P->zero_blocks.empty() &&
      launch_zero(C, 8, (const ZeroBlock *)(b + o_zero), (int)P->zero_blocks.size(), sms * 4, s) != cudaSuccess)
    return BS_ERR_CUDA;
  const int64_t ntail = (int64_t)(P->ts.tail_elems.size() / 2);
  if (P->ts.tasks.empty() && ntail == 0) return BS_OK;
  Fp64Params p{};
  p.A = (const double *)Ause;
  p.B = (const double *)Buse;
  p.C = (double *)C;
  p.tasks = (const Task *)(b + o_tasks);
  p.groups = (const Group *)(b + o_groups);
  p.rsegs = (const RowSeg *)(b + o_rsegs);
  p.ksegs = (const KSeg *)(b + o_ksegs);
  p.tail_elems = (const int2 *)(b + o_tail);
  p.tdesc = (const TailDesc *)(b + o_tdesc);
  p.ntasks = (int32_t)P->ts.tasks.size();
  p.ntail = (int32_t)ntail;
  p.nct = (int32_t)((ntail + kThreads - 1) / kThreads);
  fill_queue_params(&p, P->ts.tq_ptr, sm_map);
  p.counter = (uint32_t *)(b + 256);
  p.counter_next = (uint32_t *)(b + 256 + counter_set_bytes(nq));
  p.status = (int32_t *)(b + 128);
  const int64_t items = (int64_t)P->ts.tasks.size() + (ntail + kThreads - 1) / kThreads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)sms * per_sm));
  if (launch_fp64_grouped(p, grid, s) != cudaSuccess) return BS_ERR_CUDA;
  return BS_OK;
}

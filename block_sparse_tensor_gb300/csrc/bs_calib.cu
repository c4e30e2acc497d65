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

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "bs_plan.h"

namespace bs {

namespace {

constexpr int kFmaIters = 4096;

// Clock record of one CTA: SM cycles and global time at its start and end.
struct ClockRec {
  long long c0, c1;
  unsigned long long t0, t1;
};

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// C independent FMA chains per thread keep the pipe busy; `active` lanes of
// each warp do the work, the others skip it.  Thread 0 records its CTA's SM
// cycles and global time, which give the SM clock during the probe.
template <int C>
__global__ void dfma_probe(double *out, ClockRec *rec, double seed, int active) {
  const long long c0 = clock64();
  const unsigned long long t0 = gtimer();
  const int lane = threadIdx.x & 31;
  if (lane < active) {
    // every chain has its own operand registers: acc += x * y, as in a GEMM
    double a[C], x[C], y[C];
#pragma unroll
    for (int u = 0; u < C; ++u) {
      a[u] = seed + threadIdx.x + u;
      x[u] = 1e-3 * (u + 1);
      y[u] = 1e-3 * (seed + u);
    }
#pragma unroll 2
    for (int i = 0; i < kFmaIters; ++i) {
#pragma unroll
      for (int u = 0; u < C; ++u) a[u] = fma(x[u], y[u], a[u]);
    }
    double s = 0.0;
#pragma unroll
    for (int u = 0; u < C; ++u) s += a[u];
    if (s == 12345.678) out[blockIdx.x * blockDim.x + threadIdx.x] = s;   // keeps the loop alive
  }
  __syncthreads();
  if (threadIdx.x == 0 && rec) rec[blockIdx.x] = {c0, clock64(), t0, gtimer()};
}

// The FP64 matrix instruction (mma.sync m8n8k4, 512 flops per warp
// instruction) with eight independent accumulator pairs per warp.
__global__ void dmma_probe(double *out, ClockRec *rec, double seed) {
  const long long c0 = clock64();
  const unsigned long long t0 = gtimer();
  double a[8], b[8], d[16];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    a[u] = 1e-3 * (u + 1) + seed * 1e-9 * threadIdx.x;
    b[u] = 1e-3 * (8 - u);
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) d[u] = 0.0;
#pragma unroll 1
  for (int i = 0; i < kFmaIters / 4; ++i) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      asm volatile("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0, %1}, {%2}, {%3}, {%0, %1};"
                   : "+d"(d[2 * u]), "+d"(d[2 * u + 1])
                   : "d"(a[u]), "d"(b[u]));
  }
  double s = 0.0;
#pragma unroll
  for (int u = 0; u < 16; ++u) s += d[u];
  if (s == 12345.678) out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0 && rec) rec[blockIdx.x] = {c0, clock64(), t0, gtimer()};
}

__global__ void empty_kernel() {}

__global__ void copy_probe(const double4_32a *src, double4_32a *dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// ---- cost-model constants from the library's own kernels ------------------

// One synthetic structure: three axes of band sectors (rule |dq| <= band on
// both operands), layouts, plan options.
struct CalStruct {
  std::vector<int32_t> q[3], d[3];
  int32_t band = 1;
  uint32_t flags[3] = {BS_LAYOUT_ROWPANEL | BS_LAYOUT_CHARGE_SORTED, BS_LAYOUT_COLPANEL | BS_LAYOUT_CHARGE_SORTED,
                       BS_LAYOUT_BLOCKROW};
  int32_t dtype = BS_F64;
};

CalStruct cube(int32_t n, int32_t dim, int32_t dtype = BS_F64) {
  CalStruct c;
  for (int a = 0; a < 3; ++a) {
    c.q[a].assign(n, 0);
    c.d[a].assign(n, dim);
  }
  c.band = 0;
  c.dtype = dtype;
  if (dtype == BS_BF16_F32)
    for (auto &f : c.flags) f |= BS_LAYOUT_ALIGN16;
  return c;
}

// Charges -h..h with dims max(1, round(peak exp(-q^2 / width))), on all three axes.
CalStruct gaussian(int32_t h, double peak, double width) {
  CalStruct c;
  for (int a = 0; a < 3; ++a)
    for (int32_t q = -h; q <= h; ++q) {
      c.q[a].push_back(q);
      c.d[a].push_back(std::max(1, (int32_t)std::lround(peak * std::exp(-(double)q * q / width))));
    }
  return c;
}

struct CalRun {
  double us = 0;            // median event-to-event time of bs_contract
  double gather_ms = 0, zero_ms = 0;
  double exec_tile = 0, exec_tail = 0, exec_general = 0, slots = 0;
  double mtask = 0, mslots = 0, par = 1;   // costliest tile task: flops, slots; resident CTAs
  double c_bytes = 0;       // populated C bytes
  bs_plan_stats st{};
  int64_t stages_max = 0, tiles_max = 0;   // BF16: the busiest CTA's stages and tiles
};

// Build the structure's layouts and plan, run bs_contract `reps` times with
// L2 emptied before each (a write over `flush`), and report medians.
bs_status cal_run(const CalStruct &cs, bs_plan_options o, void *flush, size_t flush_bytes, cudaStream_t s,
                  cudaEvent_t e0, cudaEvent_t e1, int reps, CalRun *out, bool phases = false) {
  bs_axis_desc ax[3];
  for (int a = 0; a < 3; ++a) ax[a] = {(int32_t)cs.q[a].size(), cs.q[a].data(), nullptr, cs.d[a].data()};
  const bs_rule rule{-cs.band, cs.band, 0};
  const int32_t eb = cs.dtype == BS_F64 ? 8 : 2, ec = cs.dtype == BS_F64 ? 8 : 4;
  bs_layout *A = nullptr, *B = nullptr;
  bs_plan *P = nullptr;
  void *da = nullptr, *db = nullptr, *dc = nullptr;
  bs_status st = bs_layout_create(&ax[0], &ax[1], &rule, cs.flags[0], eb, &A);
  if (st == BS_OK) st = bs_layout_create(&ax[1], &ax[2], &rule, cs.flags[1], eb, &B);
  o.c_layout_flags = cs.flags[2];
  o.host_only = 0;
  o.profile = phases ? 1 : 0;   // phase events cost time of their own: only where a phase is measured
  if (st == BS_OK) st = bs_plan_create(A, B, cs.dtype, &o, &P);
  if (st == BS_OK) {
    const size_t na = (size_t)std::max<int64_t>(A->nelems, 8) * eb, nb = (size_t)std::max<int64_t>(B->nelems, 8) * eb;
    const size_t nc = (size_t)std::max<int64_t>(P->C.nelems, 8) * ec;
    if (cudaMalloc(&da, na) != cudaSuccess || cudaMalloc(&db, nb) != cudaSuccess || cudaMalloc(&dc, nc) != cudaSuccess)
      st = BS_ERR_OOM;
    else if (cudaMemsetAsync(da, 0, na, s) != cudaSuccess || cudaMemsetAsync(db, 0, nb, s) != cudaSuccess)
      st = BS_ERR_CUDA;
  }
  std::vector<double> t, g, z;
  for (int r = 0; st == BS_OK && r < reps + 2; ++r) {
    cudaMemsetAsync(flush, r, flush_bytes, s);
    cudaEventRecord(e0, s);
    st = bs_contract(P, da, db, dc, s);
    cudaEventRecord(e1, s);
    if (st != BS_OK) break;
    if (cudaEventSynchronize(e1) != cudaSuccess) {
      st = BS_ERR_CUDA;
      break;
    }
    float ms = 0;
    cudaEventElapsedTime(&ms, e0, e1);
    bs_phase_times ph{};
    if (phases) bs_plan_profile(P, &ph);
    if (r >= 2) {   // two warm-up runs
      t.push_back(ms * 1e3);
      g.push_back(ph.gather_ms);
      z.push_back(ph.zero_ms);
    }
  }
  if (st == BS_OK) st = bs_plan_last_device_error(P, s);
  auto median = [](std::vector<double> v) {
    if (v.empty()) return 0.0;
    std::nth_element(v.begin(), v.begin() + v.size() / 2, v.end());
    return v[v.size() / 2];
  };
  if (st == BS_OK) {
    out->us = median(t);
    out->gather_ms = median(g);
    out->zero_ms = median(z);
    out->exec_tile = P->ts.exec_tile;
    out->exec_tail = P->ts.exec_tail;
    out->exec_general = P->ts.exec_general;
    out->slots = P->ts.tile_slots;
    out->mtask = P->ts.max_tile_task;
    out->mslots = (double)P->ts.max_tile_slots;
    out->par = std::max(1, P->parallel_ctas);
    for (const auto &b : P->C.blocks) out->c_bytes += (double)b.rows * b.cols * ec;
    out->st = P->stats;
    for (const auto &c : P->bctas) {
      out->stages_max = std::max<int64_t>(out->stages_max, c.stage_count);
      out->tiles_max = std::max<int64_t>(out->tiles_max, c.task_count);
    }
    if (std::getenv("BS_LOG"))
      std::fprintf(stderr,
                   "[bs] calibration run: %d sectors x %d, axis %d, packed %d, groups %lld, tasks %lld: %.2f us "
                   "(gather %.2f us, zero %.2f us), executed tile %.3g tail %.3g general %.3g\n",
                   (int)cs.q[0].size(), cs.d[0].empty() ? 0 : cs.d[0][0], out->st.axis, out->st.packed_a,
                   (long long)out->st.groups, (long long)out->st.tasks, out->us, out->gather_ms * 1e3,
                   out->zero_ms * 1e3, out->exec_tile, out->exec_tail, out->exec_general);
  }
  cudaFree(da);
  cudaFree(db);
  cudaFree(dc);
  bs_plan_destroy(P);
  bs_layout_destroy(A);
  bs_layout_destroy(B);
  return st;
}

// The cost-model constants of the planner, each from the run that isolates it
// (forced axis and gather policies, so each run takes the path it measures).
bs_status calibrate_model(bs_calibration *out, cudaStream_t s) {
  const size_t flush_bytes = (size_t)256 << 20;
  void *flush = nullptr;
  cudaEvent_t e0, e1;
  if (cudaMalloc(&flush, flush_bytes) != cudaSuccess) return BS_ERR_OOM;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  bs_plan_options o;
  bs_plan_options_default(&o);
  bs_plan_options oc = o;   // contraction axis, zero copy
  oc.axis_policy = BS_AXIS_CONTRACTION;
  oc.pack_policy = BS_PACK_NEVER;
  bs_plan_options of = oc;  // free axis, zero copy
  of.axis_policy = BS_AXIS_FREE;
  bs_plan_options op = oc;  // contraction axis, gathered operands
  op.pack_policy = BS_PACK_ALWAYS;
  bs_status st = BS_OK;
  auto run = [&](const CalStruct &cs, const bs_plan_options &opt, int reps, CalRun *r, bool phases = false) {
    return cal_run(cs, opt, flush, flush_bytes, s, e0, e1, reps, r, phases);
  };
  do {
    CalRun one, tile, tile_short, tail, general, tail_free, pack_small, pack_big, zero_big, bone, bdeep, bwide;
    // a contraction with almost no work: launch, first-task chain, exit
    if ((st = run(cube(1, 1), oc, 20, &one)) != BS_OK) break;
    out->t_fixed_us = one.us;
    // tile path at long K: one dense 1536^3 group (its rate; k0 is fitted below)
    if ((st = run(cube(1, 1536), oc, 5, &tile)) != BS_OK) break;
    // tail path, one view per group: the 31-charge tail structure, contraction axis
    CalStruct g31 = gaussian(15, 64.0, 50.0);
    if ((st = run(g31, oc, 20, &tail)) != BS_OK) break;
    out->tail_gflops = (tail.exec_tail + tail.exec_general) / std::max(1e-3, tail.us - one.us) / 1e3;
    // several views per group: the same with block-row operands, contraction axis, no gather
    CalStruct g31b = g31;
    g31b.flags[0] = g31b.flags[1] = BS_LAYOUT_BLOCKROW;
    if ((st = run(g31b, oc, 20, &general)) != BS_OK) break;
    const double t_single = general.exec_tail / (out->tail_gflops * 1e3);
    out->general_gflops = general.exec_general / std::max(1e-3, general.us - one.us - t_single) / 1e3;
    // the zero fill before atomic scatter: the large structure on the free axis
    if ((st = run(gaussian(20, 384.0, 60.0), of, 5, &zero_big, true)) != BS_OK) break;
    out->zero_gbs = zero_big.zero_ms > 0 ? zero_big.c_bytes / (zero_big.zero_ms * 1e-3) / 1e9 : 0.0;
    // atomic stores: 1000 small sectors (charges spread over -30..30, dims
    // 1..8) on the free axis, where every group is a tail group stored with
    // atomics, against the time its flops take at the plain rates
    CalStruct small;
    for (int a = 0; a < 3; ++a)
      for (int32_t t = 0; t < 1000; ++t) {
        small.q[a].push_back((t * 37 + a * 11) % 61 - 30);
        small.d[a].push_back(1 + (t * 7 + a * 3) % 8);
      }
    small.band = 1;
    if ((st = run(small, of, 10, &tail_free)) != BS_OK) break;
    {
      const double plain = tail_free.exec_tail / (out->tail_gflops * 1e3) + tail_free.exec_general / (out->general_gflops * 1e3);
      const double t = tail_free.us - one.us - out->launch_us - tail_free.c_bytes / (out->zero_gbs * 1e3);
      out->atomic_factor = t > 0 ? std::min(1.0, plain / t) : 1.0;
    }
    // short-K tile tasks: the tail structure on the free axis (rows of up to
    // three sectors stacked, K = one inner sector of at most 64), where the
    // per-chunk staging shows; k0 is the extra K a task costs so that the
    // model meets this run, and the long-K rate is refitted with it
    if ((st = run(g31, of, 20, &tile_short)) != BS_OK) break;
    {
      PlanModel pm;
      pm.parallel_ctas = std::max(1, (int)tile.par);
      pm.t_launch_us = out->launch_us;
      pm.zero_gbs = out->zero_gbs;
      pm.tail_gflops = out->tail_gflops;
      pm.general_gflops = out->general_gflops;
      pm.atomic_penalty = out->atomic_factor;
      auto model_tile = [&](const CalRun &r, double rate, double k0) {
        const double rt = rate * 1e3, per_cta = rt / std::max(1, (int)r.par);
        const double work = (r.exec_tile + 2.0 * k0 * r.slots) / rt;
        const double drain = r.mtask > 0 ? (r.mtask + 2.0 * k0 * r.mslots) / per_cta : 0.0;
        const double tail = (r.exec_tail / (pm.tail_gflops * 1e3) + r.exec_general / (pm.general_gflops * 1e3)) /
                            (r.st.axis == BS_AXIS_CONTRACTION ? 1.0 : pm.atomic_penalty);
        return work + std::max(drain, tail);
      };
      double rate = tile.exec_tile / std::max(1e-3, tile.us - one.us) / 1e3, k0 = 0;
      const double t_short = tile_short.us - one.us - out->launch_us - tile_short.c_bytes / (out->zero_gbs * 1e3);
      for (int it = 0; it < 4; ++it) {
        // k0 by bisection on the short-K run (the model grows with k0) ...
        double lo = 0, hi = 1024;
        if (model_tile(tile_short, rate, 0) >= t_short) hi = 0;
        for (int b = 0; b < 40 && hi > 0; ++b) {
          const double mid = 0.5 * (lo + hi);
          if (model_tile(tile_short, rate, mid) < t_short) lo = mid;
          else hi = mid;
        }
        k0 = 0.5 * (lo + hi);
        // ... then the long-K rate with that k0 (the model falls as the rate grows)
        double rl = 10, rh = 1e5;
        for (int b = 0; b < 60; ++b) {
          const double mid = std::sqrt(rl * rh);
          if (model_tile(tile, mid, k0) > tile.us - one.us) rl = mid;
          else rh = mid;
        }
        rate = std::sqrt(rl * rh);
      }
      out->tile_gflops = rate;
      out->tile_k0 = k0;
    }
    // the gather, small (its fixed cost) and large (its bandwidth)
    if ((st = run(g31b, op, 20, &pack_small, true)) != BS_OK) break;
    out->pack_fixed_us = pack_small.gather_ms * 1e3;
    CalStruct g41b = gaussian(20, 384.0, 60.0);
    g41b.flags[0] = g41b.flags[1] = g41b.flags[2] = BS_LAYOUT_BLOCKROW;
    if ((st = run(g41b, op, 5, &pack_big, true)) != BS_OK) break;
    // gather time = fixed + 2 x packed bytes / bandwidth, through both points
    out->pack_gbs = 2.0 * (double)(pack_big.st.packed_bytes - pack_small.st.packed_bytes) /
                    std::max(1e-3, (pack_big.gather_ms - pack_small.gather_ms) * 1e3) / 1e3;
    out->pack_fixed_us = std::max(0.0, pack_small.gather_ms * 1e3 -
                                            2.0 * pack_small.st.packed_bytes / (out->pack_gbs * 1e3));
    // BF16: one 128 x 256 tile with one stage (fixed cost), one deep group
    // (stages), many shallow groups (tiles)
    CalStruct b1 = cube(1, 64, BS_BF16_F32);
    b1.d[2].assign(1, 256);
    b1.d[0].assign(1, 128);
    if ((st = run(b1, o, 20, &bone)) != BS_OK) break;
    CalStruct b2 = cube(1, 256, BS_BF16_F32);
    b2.d[0].assign(1, 128 * 152);
    b2.d[1].assign(1, 4096);   // 64 stages of 64 on every CTA at once
    if ((st = run(b2, o, 10, &bdeep)) != BS_OK) break;
    out->bf16_stage_us = std::max(0.0, bdeep.us - bone.us) / std::max<int64_t>(1, bdeep.stages_max - 1);
    CalStruct b3 = cube(1, 64, BS_BF16_F32);
    b3.d[0].assign(1, 128 * 152 * 8);   // eight 128 x 256 tiles of one stage on every CTA
    b3.d[2].assign(1, 256);
    if ((st = run(b3, o, 10, &bwide)) != BS_OK) break;
    out->bf16_tile_us = std::max(0.0, bwide.us - bone.us - (bwide.stages_max - 1) * out->bf16_stage_us) /
                        std::max<int64_t>(1, bwide.tiles_max - 1);
  } while (false);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(flush);
  return st;
}

}  // namespace

}  // namespace bs

extern "C" bs_status bs_calibrate(bs_calibration *out, void *stream) {
  using namespace bs;
  if (!out) return BS_ERR_INVALID_ARG;
  *out = bs_calibration{};
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BS_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return BS_ERR_CUDA;
  double *scratch = nullptr;
  ClockRec *recs = nullptr;
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
    // Probe shapes: CTAs per SM x threads x chains.  The best one is taken as the
    // FP64 pipe's rate; its SM clock comes from the CTAs' cycle and time stamps.
    const int max_blocks = sms * 8, threads = 256;
    if (cudaMalloc(&scratch, (size_t)max_blocks * 1024 * sizeof(double)) != cudaSuccess ||
        cudaMalloc(&recs, (size_t)max_blocks * sizeof(ClockRec)) != cudaSuccess) {
      st = BS_ERR_OOM;
      break;
    }
    std::vector<ClockRec> host((size_t)max_blocks);
    auto clock_mhz = [&](int blocks) {
      cudaMemcpy(host.data(), recs, (size_t)blocks * sizeof(ClockRec), cudaMemcpyDeviceToHost);
      std::vector<double> f;
      for (int b = 0; b < blocks; ++b)
        if (host[b].t1 > host[b].t0) f.push_back((double)(host[b].c1 - host[b].c0) / (double)(host[b].t1 - host[b].t0) * 1e3);
      if (f.empty()) return 0.0;
      std::nth_element(f.begin(), f.begin() + f.size() / 2, f.end());
      return f[f.size() / 2];
    };
    struct Shape {
      int per_sm, thr, chains;
    };
    const Shape shapes[] = {{8, 256, 8}, {4, 256, 8}, {2, 256, 8}, {4, 256, 16}, {1, 1024, 8}, {2, 512, 4}};
    double best = 0.0, best_mhz = 0.0;
    for (const Shape &sh : shapes) {
      const int blocks = sms * sh.per_sm;
      auto launch = [&] {
        if (sh.chains == 4) dfma_probe<4><<<blocks, sh.thr, 0, s>>>(scratch, recs, 1.0, 32);
        else if (sh.chains == 8) dfma_probe<8><<<blocks, sh.thr, 0, s>>>(scratch, recs, 1.0, 32);
        else dfma_probe<16><<<blocks, sh.thr, 0, s>>>(scratch, recs, 1.0, 32);
      };
      const double ms = timed(launch, 3);
      const double flops = 2.0 * sh.chains * kFmaIters * (double)blocks * sh.thr;
      const double gf = flops / (ms * 1e6);
      if (gf > best) {
        best = gf;
        best_mhz = clock_mhz(blocks);
      }
    }
    out->fp64_gflops = best;
    out->fp64_sm_mhz = best_mhz;
    out->fp64_flop_per_clk_sm = best_mhz > 0 ? best * 1e3 / (sms * best_mhz) : 0.0;
    {
      const int blocks = sms * 8;
      const double ms = timed([&] { dfma_probe<8><<<blocks, threads, 0, s>>>(scratch, nullptr, 1.0, 8); }, 3);
      out->fp64_gflops_quarter_warp = 2.0 * 8 * kFmaIters * (double)blocks * (threads / 32) * 8 / (ms * 1e6);
    }
    {
      double bestm = 0.0, mhz = 0.0;
      for (int per_sm : {4, 8}) {
        const int blocks = sms * per_sm;
        const double ms = timed([&] { dmma_probe<<<blocks, threads, 0, s>>>(scratch, recs, 1.0); }, 3);
        const double gf = 512.0 * 8 * (kFmaIters / 4) * (double)blocks * (threads / 32) / (ms * 1e6);
        if (gf > bestm) {
          bestm = gf;
          mhz = clock_mhz(blocks);
        }
      }
      out->fp64_dmma_gflops = bestm;
      out->dmma_flop_per_clk_sm = mhz > 0 ? bestm * 1e3 / (sms * mhz) : 0.0;
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
    st = calibrate_model(out, s);
    if (st != BS_OK) break;
    {
      std::vector<int16_t> map;
      if (sm_index_map(dev, sms, nullptr, s, &map) == BS_OK) {
        int32_t bound = 0;
        for (size_t t = 0; t < map.size(); ++t)
          if (map[t] >= 0) bound = (int32_t)t + 1;
        out->sm_id_bound = bound;
      }
    }
    if (cudaGetLastError() != cudaSuccess) st = BS_ERR_CUDA;
  } while (false);
  cudaFree(scratch);
  cudaFree(recs);
  cudaFree(bufs);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return st;
}

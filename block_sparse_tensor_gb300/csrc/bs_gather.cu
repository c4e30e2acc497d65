// The FP64 gather into panels by shared-memory segments (uni20 design note
// "block coalescing", "Interleaved vs contiguous": operands that are not one
// strided view are gathered into contiguous panels by one pack kernel).
//
// The source side of a gather is read in order: consecutive blocks of the
// source layout (or a band of one) form a segment of at most 2048 doubles,
// and one thread has the copy engine bring each segment, as a 16-byte-aligned
// window, into shared memory together with its piece records (cp.async.bulk:
// ten segments in flight per SM, no registers held while they are).  Sixteen
// warps then write each piece to its place in the panel (all together on a
// piece of 512 elements or more, else a warp per piece), reading shared
// memory instead of waiting on a global load per element.
// Every wait is bounded by the global timer; on expiry the kernel records
// DS_TIMEOUT, lets the copies in flight land and returns.
#include <cuda_runtime.h>

#include <cstdint>

#include "bs_host.h"

namespace bs {

namespace {

constexpr int kSegThreads = 544;   // warp 0 lane 0 issues the copies; warps 1-16 write the pieces
constexpr int kSegWarps = 16;
constexpr int kSegDataBytes = kSegElems * 8 + 16;                           // a segment and its window's slack
constexpr int kSegStageBytes = kSegDataBytes + kSegPieces * (int)sizeof(PackPiece);
constexpr int kSegCache = 256;                                              // segment records a CTA keeps
constexpr size_t kSegSmem = (size_t)kSegStages * kSegStageBytes + kSegCache * sizeof(PackSeg) + 128;
static_assert(kSegDataBytes % 16 == 0 && kSegStageBytes % 16 == 0, "16-byte aligned stages");

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_expect(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ bool bar_test(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity: false once `limit_ns` has
// passed or another thread has aborted the CTA's work.
__device__ __forceinline__ bool bar_wait(uint32_t a, uint32_t parity, volatile int32_t *abort, uint64_t limit_ns) {
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    if (bar_test(a, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort) return false;
      const uint64_t now = global_ns();
      if (start == 0) start = now;
      else if (now - start > limit_ns) return false;
    }
  }
}

// dst (shared) <- [src, src + bytes) (global); both 16-byte aligned, bytes a
// multiple of 16; completion counted on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// The window of a segment: the 16-byte-aligned range [lo, hi) around its
// source elements, cut at the last 16-byte boundary inside the caller's
// buffer (a buffer of an odd number of doubles keeps its last one out; the
// writers read that one from global memory).  `shift` is the window index of
// the segment's first element.
struct Window {
  uintptr_t lo, hi;
  int shift;
};

__device__ __forceinline__ Window window_of(const SegParams &p, const PackSeg &sg) {
  const uintptr_t base = (uintptr_t)(sg.operand ? p.src[1] : p.src[0]);
  const uintptr_t s = base + (uintptr_t)sg.src * 8u;
  Window w;
  w.lo = s & ~(uintptr_t)15;
  w.hi = (s + (uintptr_t)sg.n * 8u + 15u) & ~(uintptr_t)15;
  const uintptr_t cap = base + ((uintptr_t)(sg.operand ? p.src_nelems[1] : p.src_nelems[0]) * 8u & ~(uintptr_t)15);
  if (w.hi > cap) w.hi = cap > w.lo ? cap : w.lo;
  w.shift = (int)((s - w.lo) >> 3);
  return w;
}

// Element i (counted from the segment's first) of a segment: window index
// shift + i, or global memory past the window's end when kTail.
template <bool kTail>
__device__ __forceinline__ double piece_elem(const double *win, int loaded, int shift, const double *gseg, int i) {
  if constexpr (kTail) return shift + i < loaded ? win[shift + i] : __ldg(gseg + i);
  else return win[shift + i];
}

// Lane `lane` of a warp writes its share of one piece: element (r, c) is
// element src_off + r src_ld + c of the segment and goes to dst[r dst_ld + c].
// Rows of at most 32 elements fix each lane's row offset and column; longer
// rows step each lane 32 columns at a time, wrapping to the next row.
template <bool kTail>
__device__ __forceinline__ void write_piece_warp(const double *win, int loaded, int shift, const double *gseg,
                                                 double *dst, const PackPiece &pc, int lane) {
  const int rows = pc.rows, cols = pc.cols;
  if (cols <= 32) {
    const int rpw = 32 / cols;
    const int lr = lane / cols, lc = lane - lr * cols;
    if (lr >= rpw) return;
    for (int r = lr; r < rows; r += rpw)
      dst[(int64_t)r * pc.dst_ld + lc] = piece_elem<kTail>(win, loaded, shift, gseg, pc.src_off + r * pc.src_ld + lc);
    return;
  }
  int r = 0, c = lane;
  while (r < rows) {
    dst[(int64_t)r * pc.dst_ld + c] = piece_elem<kTail>(win, loaded, shift, gseg, pc.src_off + r * pc.src_ld + c);
    c += 32;
    if (c >= cols) {   // cols > 32: one wrap at most
      c -= cols;
      ++r;
    }
  }
}

// All kSegWarps writer warps together write a piece of at least kCoopElems
// elements: writer t starts at element t and steps kWriters elements at a
// time (a fixed number of rows and columns per step, so no division per
// element), four positions per step.
constexpr int kWriters = 32 * kSegWarps;
constexpr int kCoopElems = 512;

template <bool kTail>
__device__ __forceinline__ void write_piece_all(const double *win, int loaded, int shift, const double *gseg,
                                                double *dst, const PackPiece &pc, int t) {
  const int rows = pc.rows, cols = pc.cols;
  const int dr = kWriters / cols, dc = kWriters - dr * cols;
  int r = t / cols, c = t - r * cols;
  while (r < rows) {
    int rr[4], cc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      rr[q] = r;
      cc[q] = c;
      c += dc;
      r += dr;
      if (c >= cols) {
        c -= cols;
        ++r;
      }
    }
    double v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (rr[q] < rows) v[q] = piece_elem<kTail>(win, loaded, shift, gseg, pc.src_off + rr[q] * pc.src_ld + cc[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (rr[q] < rows) dst[(int64_t)rr[q] * pc.dst_ld + cc[q]] = v[q];
  }
}

// Whether a piece reaches past the loaded window (only at the very end of a
// buffer of an odd number of doubles).
__device__ __forceinline__ bool piece_tail(const PackPiece &pc, int loaded, int shift) {
  return shift + pc.src_off + (pc.rows - 1) * pc.src_ld + pc.cols > loaded;
}

__global__ void __launch_bounds__(kSegThreads, 1) seg_gather_kernel(const SegParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kSegStages], empty[kSegStages];
  __shared__ uint32_t issued[kSegStages];
  __shared__ int32_t abort_flag;
  unsigned char *stages = (unsigned char *)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  PackSeg *cache = (PackSeg *)(stages + (size_t)kSegStages * kSegStageBytes);
  volatile int32_t *abort = &abort_flag;
  // this CTA's segment records (segments blockIdx.x, blockIdx.x + gridDim.x,
  // ...), loaded once by every thread together
  for (int k = threadIdx.x; k < kSegCache; k += kSegThreads) {
    const int64_t g = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
    if (g >= p.nseg) break;
    cache[k] = p.segs[g];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSegStages; ++s) {
      bar_init(smem_addr(&full[s]), 1);
      bar_init(smem_addr(&empty[s]), kSegWarps);
      issued[s] = 0;
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto fail = [&](int32_t code) {
    abort_flag = 1;
    atomicExch(p.status, code);
  };
  auto seg_at = [&](int k, int64_t g) { return k < kSegCache ? cache[k] : p.segs[g]; };

  if (threadIdx.x == 0) {
    // ------------------------------------------------------------ copy issue
    int k = 0;
    for (int64_t g = blockIdx.x; g < p.nseg; g += gridDim.x, ++k) {
      const PackSeg sg = seg_at(k, g);
      const int slot = k % kSegStages;
      const uint32_t ph = (uint32_t)(k / kSegStages) & 1u;
      if (k >= kSegStages && !bar_wait(smem_addr(&empty[slot]), ph ^ 1u, abort, p.timeout_ns)) {
        fail(DS_TIMEOUT);
        break;
      }
      const Window w = window_of(p, sg);
      const uint32_t data = (uint32_t)(w.hi - w.lo), recs = (uint32_t)sg.piece_count * (uint32_t)sizeof(PackPiece);
      if (data > (uint32_t)kSegDataBytes || sg.piece_count < 1 || sg.piece_count > kSegPieces) {   // never planned
        fail(DS_BOUNDS);
        break;
      }
      unsigned char *st = stages + (size_t)slot * kSegStageBytes;
      const uint32_t fb = smem_addr(&full[slot]);
      bar_expect(fb, data + recs);
      if (data) bulk_load(smem_addr(st), (const void *)w.lo, data, fb);
      bulk_load(smem_addr(st + kSegDataBytes), p.pieces + sg.piece_begin, recs, fb);
      issued[slot] = ph + 1u;
    }
    // Every copy issued lands before the CTA exits (on the normal path the
    // writers have consumed them all already).
    for (int s = 0; s < kSegStages; ++s)
      if (issued[s]) {
        const uint64_t t0 = global_ns();
        while (!bar_test(smem_addr(&full[s]), issued[s] - 1u) && global_ns() - t0 < p.timeout_ns) {
        }
      }
  } else if (threadIdx.x >= 32) {
    // ------------------------------------------------------------ writers
    const int wi = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
    int k = 0;
    for (int64_t g = blockIdx.x; g < p.nseg; g += gridDim.x, ++k) {
      const PackSeg sg = seg_at(k, g);
      const int slot = k % kSegStages;
      const uint32_t ph = (uint32_t)(k / kSegStages) & 1u;
      // lane 0 polls (512 threads spinning on one barrier slow its updates);
      // then every lane takes the completed phase's ordering itself
      bool ok = true;
      if (lane == 0) ok = bar_wait(smem_addr(&full[slot]), ph, abort, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) ok = __all_sync(0xffffffffu, bar_wait(smem_addr(&full[slot]), ph, abort, p.timeout_ns));
      if (!ok) {
        if (lane == 0) fail(DS_TIMEOUT);
        break;
      }
      const Window w = window_of(p, sg);
      const unsigned char *st = stages + (size_t)slot * kSegStageBytes;
      const PackPiece *pcs = (const PackPiece *)(st + kSegDataBytes);
      const double *gseg = (sg.operand ? p.src[1] : p.src[0]) + sg.src;
      double *dbase = sg.operand ? p.dst[1] : p.dst[0];
      const int loaded = (int)((w.hi - w.lo) >> 3);
      // pieces of at least kCoopElems elements by every writer together, the
      // others a warp each
      const double *win = (const double *)st;
      for (int q = 0; q < sg.piece_count; ++q) {
        const PackPiece pc = pcs[q];
        if (pc.rows * pc.cols < kCoopElems) continue;
        if (piece_tail(pc, loaded, w.shift))
          write_piece_all<true>(win, loaded, w.shift, gseg, dbase + pc.dst, pc, threadIdx.x - 32);
        else
          write_piece_all<false>(win, loaded, w.shift, gseg, dbase + pc.dst, pc, threadIdx.x - 32);
      }
      for (int q = wi; q < sg.piece_count; q += kSegWarps) {
        const PackPiece pc = pcs[q];
        if (pc.rows * pc.cols >= kCoopElems) continue;
        if (piece_tail(pc, loaded, w.shift))
          write_piece_warp<true>(win, loaded, w.shift, gseg, dbase + pc.dst, pc, lane);
        else
          write_piece_warp<false>(win, loaded, w.shift, gseg, dbase + pc.dst, pc, lane);
      }
      __syncwarp();
      if (lane == 0) bar_arrive(smem_addr(&empty[slot]));
    }
  }
}

}  // namespace

cudaError_t launch_seg_gather(const SegParams &p, int sms, cudaStream_t s) {
  if (p.nseg <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(seg_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSegSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n = sms > 0 ? sms : 1;
  const int grid = p.nseg < n ? p.nseg : n;
  seg_gather_kernel<<<grid, kSegThreads, kSegSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bs

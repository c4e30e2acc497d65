// FP64 persistent grouped GEMM, gather ("pack") kernel, zero fill, and the
// one-launch-per-triple control kernel.
//
// The grouped kernel runs the whole task list of a plan in one launch
// (uni20 design note "block coalescing", Summary: fewer, larger kernels;
// the inferensys glossary "Sparse Operator Fusion": persistent thread blocks
// and warp-level gather-compute-scatter).  Resident CTAs first take tile tasks
// from a global counter in longest-first order, then their warps take tail
// warp-tasks from a queue per SM, dealt longest-first onto the least loaded
// queue at plan time (and steal from other queues once their own is empty):
//   - TILE: the CTA computes a tm x tn tile of one group.  Each K chunk of the
//     group's concatenated inner axis is staged in shared memory through
//     per-row and per-k address tables, so inner blocks of any size and any
//     number of views cost no padding flops.  Outputs are spread one per
//     thread slot, so a tile of any shape keeps the FP64 lanes busy.
//   - TAIL: small groups (at most 4096 outputs each) with one output per
//     thread, outputs of consecutive groups packed lane after lane so that no
//     FMA is issued for an idle lane, accumulating in registers straight from
//     the L1-cached operands.  Idle lanes of a warp cost the FP64 pipe as much
//     as busy ones on this part, which is why outputs, not groups, are spread
//     over the lanes.
// Stores are plain for contraction-axis groups (each C block has one writer)
// and atomic adds for free-axis groups (several k add into one C block).
#include <algorithm>

#include "bs_host.h"

namespace bs {

namespace {

__device__ __forceinline__ int find_rseg(const RowSeg *rs, int n, int r) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rs[mid].r0 <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int find_kseg(const KSeg *ks, int n, int k) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ks[mid].k0 <= k) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Operand loads and C stores.  The checked instance (bs_contract_checked)
// tests every index against the buffer's element count first: an access
// outside is skipped (a load reads zero) and the status word records it.
__device__ __forceinline__ void flag_bounds(const Fp64Params &p) { atomicExch(p.status, (int32_t)DS_BOUNDS); }

template <bool kCheck>
__device__ __forceinline__ double ld_op(const Fp64Params &p, const double *base, int64_t n, const double *ptr) {
  if (kCheck) {
    const int64_t i = ptr - base;
    if (i < 0 || i >= n) {
      flag_bounds(p);
      return 0.0;
    }
  }
  return __ldg(ptr);
}

template <bool kCheck>
__device__ __forceinline__ void st_c(const Fp64Params &p, double *ptr, double v, bool atomic) {
  if (kCheck) {
    const int64_t i = ptr - p.C;
    if (i < 0 || i >= p.nC) {
      flag_bounds(p);
      return;
    }
  }
  if (atomic) atomicAdd(ptr, v);
  else *ptr = v;
}

struct TileSmem {
  double As[kKC][kTileMaxDim + 1];   // A chunk, inner index major: As[kk][row]
  double Bs[kKC][kTileMaxDim + 1];   // B chunk: Bs[kk][col]
  int64_t rowA[kTileMaxDim];
  int64_t rowC[kTileMaxDim];
  int64_t rowL[kTileMaxDim];
  int64_t kA[kKC];
  int64_t kL[kKC];
  int64_t kB[kKC];
  int task;
};

template <bool kCheck>
__device__ void run_tile(const Fp64Params &p, const Task &T, TileSmem &sm) {
  const int tid = threadIdx.x;
  const Group G = p.groups[T.g];
  const RowSeg *rs = p.rsegs + G.rseg_begin;
  const KSeg *ks = p.ksegs + G.kseg_begin;
  const int tm = T.tm, tn = T.tn;
  for (int r = tid; r < tm; r += kThreads) {
    const int gr = T.m0 + r;
    const RowSeg s = rs[find_rseg(rs, G.rseg_count, gr)];
    const int64_t lr = gr - s.r0;
    sm.rowA[r] = s.ra + lr * s.lda;
    sm.rowL[r] = s.rl ? lr : 0;
    sm.rowC[r] = s.rc + lr * s.ldc;
  }
  // this thread's outputs: e = tid + kThreads * u
  const int ne = tm * tn;
  int orow[kElemsPerThread], ocol[kElemsPerThread];
  double acc[kElemsPerThread];
#pragma unroll
  for (int u = 0; u < kElemsPerThread; ++u) {
    const int e = tid + kThreads * u;
    orow[u] = e < ne ? e / tn : -1;
    ocol[u] = e < ne ? e - (e / tn) * tn : 0;
    acc[u] = 0.0;
  }
  const bool active = tid < ne;   // warps past the tile's outputs only help load
  for (int kc0 = 0; kc0 < G.k; kc0 += kKC) {
    const int kn = min(kKC, G.k - kc0);
    if (tid < kn) {
      const int kk = kc0 + tid;
      const KSeg s = ks[find_kseg(ks, G.kseg_count, kk)];
      const int64_t pp = kk - s.k0;
      sm.kA[tid] = s.ka + pp;
      sm.kL[tid] = s.kl;
      sm.kB[tid] = s.kb + pp * s.ldb + T.n0;
    }
    __syncthreads();
    for (int idx = tid; idx < tm * kn; idx += kThreads) {
      const int r = idx / kn, kk = idx - r * kn;
      sm.As[kk][r] = ld_op<kCheck>(p, p.A, p.nA, p.A + sm.rowA[r] + sm.kA[kk] + sm.rowL[r] * sm.kL[kk]);
    }
    for (int idx = tid; idx < kn * tn; idx += kThreads) {
      const int kk = idx / tn, c = idx - kk * tn;
      sm.Bs[kk][c] = ld_op<kCheck>(p, p.B, p.nB, p.B + sm.kB[kk] + c);
    }
    __syncthreads();
    if (active) {
      for (int kk = 0; kk < kn; ++kk) {
#pragma unroll
        for (int u = 0; u < kElemsPerThread; ++u)
          if (orow[u] >= 0) acc[u] = fma(sm.As[kk][orow[u]], sm.Bs[kk][ocol[u]], acc[u]);
      }
    }
    __syncthreads();
  }
  const bool atomic = (G.flags & GF_ATOMIC) != 0;
#pragma unroll
  for (int u = 0; u < kElemsPerThread; ++u) {
    if (orow[u] < 0) continue;
    st_c<kCheck>(p, p.C + sm.rowC[orow[u]] + T.n0 + ocol[u], acc[u], atomic);
  }
}

// One output per lane for 32 consecutive outputs of the tail list.  The loop
// count is the warp's longest K; a lane whose group is shorter stops adding.
// When every lane's group is one view (the usual case with panel layouts) the
// loop is unrolled with six accumulators; otherwise each lane walks its
// group's views, switching view on its own.
template <bool kCheck>
__device__ void run_tail_warp(const Fp64Params &p, int w) {
  const int lane = threadIdx.x & 31;
  const int e = w * 32 + lane;
  int2 el = e < p.ntail ? p.tail_elems[e] : make_int2(p.tail_elems[w * 32].x, kTailPad);
  const bool hi = (el.x & kTailHi) != 0;   // second half of a split output's K
  el.x &= ~kTailHi;
  const bool ok = el.y != kTailPad;   // a padding entry holds no output
  const int r = el.y >> 16, c = el.y & 0xFFFF;
  // single-segment groups: addressing resolved at plan time, one table load
  const TailDesc D = p.tdesc[el.x];
  double acc = 0.0;
  int64_t cofs;
  int flags;
  bool live = ok;   // this lane owns a real output (padded lanes of a bucket do not)
  if (__all_sync(0xFFFFFFFFu, D.k > 0)) {
    live = ok && r < D.m && c < D.n;
    // a split output's lanes sum K steps [0, kh) and [kh, kpad); others [0, kpad)
    const bool split = __any_sync(0xFFFFFFFFu, hi);   // split groups fill whole warps
    const int kh = split ? (D.kpad + 1) >> 1 : 0;
    const int k0 = hi ? kh : 0;
    const int kend = split && !hi ? kh : D.kpad;
    const int kg = live ? max(0, min(D.k, kend) - k0) : 0;   // steps that load data
    const int kmax = __reduce_max_sync(0xFFFFFFFFu, ok ? (unsigned)(kend - k0) : 0u);   // steps run
    const double *ap = p.A + D.a0 + (int64_t)r * D.as + k0;
    const double *bp = p.B + D.b0 + (int64_t)k0 * D.ldb + c;
    const int64_t ldb = D.ldb;
    cofs = D.c0 + (int64_t)r * D.ldc + c;
    flags = D.flags;
    // six independent chains with their loads issued ahead, so that a warp
    // left alone on its SM at the end of the launch still keeps B rows in
    // flight (six measure faster than eight or ten, which need more registers
    // than four resident CTAs leave); steps past this lane's K load nothing
    // and add 0 * 0
    constexpr int U = 6;
    double a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] = 0.0;
    int it = 0;
    for (; it + U <= kmax; it += U) {
      double x[U], y[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        x[u] = it + u < kg ? ld_op<kCheck>(p, p.A, p.nA, ap + it + u) : 0.0;
        y[u] = it + u < kg ? ld_op<kCheck>(p, p.B, p.nB, bp + (it + u) * ldb) : 0.0;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] = fma(x[u], y[u], a[u]);
    }
    for (; it < kmax; ++it)
      if (it < kg) a[0] = fma(ld_op<kCheck>(p, p.A, p.nA, ap + it), ld_op<kCheck>(p, p.B, p.nB, bp + it * ldb), a[0]);
    acc = ((a[0] + a[1]) + (a[2] + a[3])) + (a[4] + a[5]);
    if (split) {   // the second half's partial sum joins its output on the lane 16 below
      acc += __shfl_down_sync(0xFFFFFFFFu, acc, 16);
      live = live && !hi;
    }
  } else {
    // general path: walk the group's row and inner segments
    const Group G = p.groups[el.x];
    const int kg = ok ? G.k : 0;
    const int kmax = __reduce_max_sync(0xFFFFFFFFu, (unsigned)kg);
    const RowSeg *rs = p.rsegs + G.rseg_begin;
    const KSeg *ks = p.ksegs + G.kseg_begin;
    const RowSeg s = rs[find_rseg(rs, G.rseg_count, r)];
    const int64_t lr = r - s.r0;
    const int64_t ra = s.ra + lr * s.lda, rl = s.rl ? lr : 0;
    KSeg k = ks[0];
    const double *ap = p.A + ra + k.ka + rl * k.kl;
    const double *bp = p.B + k.kb + c;
    int64_t ldb = k.ldb;
    cofs = s.rc + lr * s.ldc + c;
    flags = G.flags;
    int si = 0, rem = k.klen;
    for (int it = 0; it < kmax; ++it) {
      if (it < kg) {
        if (rem == 0) {
          k = ks[++si];
          ap = p.A + ra + k.ka + rl * k.kl;
          bp = p.B + k.kb + c;
          ldb = k.ldb;
          rem = k.klen;
        }
        acc = fma(ld_op<kCheck>(p, p.A, p.nA, ap), ld_op<kCheck>(p, p.B, p.nB, bp), acc);
        ++ap;
        bp += ldb;
        --rem;
      }
    }
  }
  if (live) {
    st_c<kCheck>(p, p.C + cofs, acc, (flags & GF_ATOMIC) != 0);
  }
}

// The tail queue of the SM this CTA runs on: the SM's dense index (the
// hardware identifiers may skip values), modulo the queue count.
__device__ __forceinline__ int home_queue(const Fp64Params &p) {
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  int idx = (int)smid;
  if ((int)smid < p.nsm_ids && p.sm_queue[smid] >= 0) idx = p.sm_queue[smid];
  return idx % p.nq;
}

// A counter set as a launch finds it: every count at zero.
__device__ __forceinline__ void init_counter_set(const Fp64Params &p, uint32_t *set) {
  for (int q = threadIdx.x; q < p.nq; q += kThreads) atomicExch(&set[kQueueCounterBase + q], 0u);
  if (threadIdx.x == 0) {
    atomicExch(&set[0], 0u);
    atomicExch(&set[2], 0u);
  }
}

// Two instances: four CTAs per SM (64 registers a thread) for plans with tile
// tasks, whose shared-memory staging wants the most resident warps, and three
// for plans made only of tail tasks, which measure faster with fewer, quicker
// CTAs sharing each SM.
template <int kMinCtas, bool kCheck>
__global__ void __launch_bounds__(kThreads, kMinCtas) fp64_grouped_kernel(Fp64Params p) {
  __shared__ TileSmem sm;
  // CTA 0 prepares the other counter set for the next launch (the set is idle
  // during this one), so this launch's own set needs no reset at exit
  if (blockIdx.x == 0 && p.counter_next) init_counter_set(p, p.counter_next);
  // tile tasks, one CTA each, longest first
  for (; p.ntasks > 0;) {
    if (threadIdx.x == 0) sm.task = (int)atomicAdd(&p.counter[0], 1u);
    __syncthreads();
    const int t = sm.task;
    __syncthreads();
    if (t >= p.ntasks) break;
    run_tile<kCheck>(p, p.tasks[t], sm);
  }
  // Then the tail: CTA-sized tasks (kThreads consecutive outputs of the tail
  // list, so the 8 warps walk the same B rows through L1), dealt at plan time
  // longest first onto one queue per SM, each queue's tasks numbered
  // consecutively.  A CTA serves the queue of the SM it runs on; once that
  // queue is empty it takes tasks from the others (so no output depends on
  // every SM receiving CTAs).  Thread 0 claims; the CTA runs the task, warp w
  // on its w-th 32 outputs.
  if (p.nct > 0) {
    const int warp = threadIdx.x >> 5;
    int q0 = 0, qk = 0;          // thread 0: home queue, queues emptied so far
    unsigned nx = 0;             // thread 0: claim on the home queue made during the last task
    bool have_nx = false;
    if (threadIdx.x == 0) q0 = home_queue(p);
    for (;;) {
      if (threadIdx.x == 0) {
        int got = -1;
        while (qk < p.nq) {
          const int q = q0 + qk < p.nq ? q0 + qk : q0 + qk - p.nq;
          const int beg = p.qptr[q], n = p.qptr[q + 1] - beg;
          unsigned i;
          if (qk == 0 && have_nx) {
            i = nx;
            have_nx = false;
          } else {
            if (qk > 0 && *(volatile uint32_t *)&p.counter[2] >= (uint32_t)p.nct) {   // all taken
              qk = p.nq;
              break;
            }
            i = atomicAdd(&p.counter[kQueueCounterBase + q], 1u);
          }
          if (i < (unsigned)n) {
            atomicAdd(&p.counter[2], 1u);
            got = beg + (int)i;
            break;
          }
          ++qk;
        }
        sm.task = got;
        // In a tail-only plan the next claim travels while this task runs.  In
        // a plan with tile tasks the tail fills the end of the launch, where a
        // task claimed by a CTA that is still busy is what ends it, so there a
        // CTA claims only once it is free (measured: 12.58 against 12.63 ms on
        // the stress workload; the tail workload keeps its 41.0 us with the
        // claim in advance)
        if (kMinCtas < 4 && got >= 0 && qk == 0) {
          nx = atomicAdd(&p.counter[kQueueCounterBase + q0], 1u);
          have_nx = true;
        }
      }
      __syncthreads();
      const int ct = sm.task;
      __syncthreads();
      if (ct < 0) break;
      const int w = ct * (kThreads / 32) + warp;
      if (w * 32 < p.ntail) run_tail_warp<kCheck>(p, w);
    }
  }
  if (p.reset_at_exit) {
    // a replayed launch finds its own set as it found it: the last CTA to
    // leave (every CTA has taken its final work index before it counts
    // itself out) writes the initial values back
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      sm.task = atomicAdd(&p.counter[1], 1u) == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (sm.task) {
      init_counter_set(p, p.counter);
      __syncthreads();
      if (threadIdx.x == 0) atomicExch(&p.counter[1], 0u);
    }
  }
}

// The gather: one warp per block copy, copies listed at plan time (doubles in
// destination order, 2-byte elements largest first) and dealt to the warps
// in turn (each warp fetches its next copy's
// descriptor while it moves the current one); then the small copies (at most
// kPackSmallElems elements), four to a warp, 8 lanes each, so that a warp has
// four of them in flight instead of waiting on each in turn.  A copy is moved
// in 16-byte units when both views allow it (every row start 16-byte aligned
// and whole rows of units), else element by element.  A group of G lanes
// walks the copy's (row, column) positions G at a time with four loads in
// flight per lane and divides no index: rows of at most G units map each lane
// to one fixed (row offset, column) pair, so a step covers floor(G / cols)
// rows; wider rows advance each lane's position by G columns, wrapping to the
// next row.
template <class U, int G, int kU>
__device__ __forceinline__ void copy_2d(const U *__restrict__ src, int64_t sld, U *__restrict__ dst, int64_t dld,
                                        int rows, int cols, int lane) {
  if (cols <= G) {
    const int rpw = G / cols;
    const int lr = lane / cols, lc = lane - lr * cols;
    if (lr >= rpw) return;
    const U *sp = src + lc;
    U *dp = dst + lc;
    int r = lr;
    for (; r + (kU - 1) * rpw < rows; r += kU * rpw) {
      U t[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q) t[q] = __ldg(sp + (int64_t)(r + q * rpw) * sld);
#pragma unroll
      for (int q = 0; q < kU; ++q) dp[(int64_t)(r + q * rpw) * dld] = t[q];
    }
    for (; r < rows; r += rpw) dp[(int64_t)r * dld] = __ldg(sp + (int64_t)r * sld);
    return;
  }
  // cols > G: a step of G positions moves a lane at most into the next row
  int r = 0, c = lane;
  for (;;) {
    int rr[kU], cc[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      rr[q] = r;
      cc[q] = c;
      c += G;
      if (c >= cols) {
        c -= cols;
        ++r;
      }
    }
    U t[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q)
      if (rr[q] < rows) t[q] = __ldg(src + (int64_t)rr[q] * sld + cc[q]);
#pragma unroll
    for (int q = 0; q < kU; ++q)
      if (rr[q] < rows) dst[(int64_t)rr[q] * dld + cc[q]] = t[q];
    if (rr[kU - 1] >= rows || r >= rows) break;
  }
}

// One copy by a group of G lanes (lane = the lane's index inside the group),
// kU loads in flight per lane.
template <class T, int G, int kU>
__device__ __forceinline__ void pack_one(const PackParams &pp, const PackCopy &cur, int lane) {
  constexpr int V = 16 / (int)sizeof(T);
  const T *src = (const T *)pp.src + cur.src;
  T *dst = (T *)pp.dst + cur.dst;
  const bool base16 = (((uintptr_t)pp.src | (uintptr_t)pp.dst) & 15u) == 0;
  int64_t sld = cur.src_ld, dld = cur.dst_ld;
  int rows = cur.rows, cols = cur.cols;
  if (sld == cols && dld == cols) {   // contiguous on both sides: one flat row
    cols = rows * cols;
    rows = 1;
    sld = dld = cols;
  }
  if (base16 && ((cur.src | cur.dst | sld | dld | (int64_t)cols) % V) == 0)
    copy_2d<int4, G, kU>((const int4 *)src, sld / V, (int4 *)dst, dld / V, rows, cols / V, lane);
  else
    copy_2d<T, G, kU>(src, sld, dst, dld, rows, cols, lane);
}

constexpr int kPackGroup = 8, kPackGroupU = 4;   // lanes per small copy, loads in flight per lane

template <class T>
__global__ void __launch_bounds__(256, 4) pack_kernel(PackParams a, PackParams b, PackSplit sp) {
  const int lane = threadIdx.x & 31;
  const int gw = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
  const int nw = (int)(gridDim.x * (blockDim.x >> 5));
  PackCopy cp;
  // whole-warp copies
  int c = gw;
  if (c < sp.big) cp = a.copies[c];
  for (; c < sp.big; c += nw) {
    const PackCopy cur = cp;
    if (c + nw < sp.big) cp = a.copies[c + nw];   // the next descriptor, in flight meanwhile
    pack_one<T, 32, 4>(c < sp.big_a ? a : b, cur, lane);
  }
  // small copies, dealt from the last warp backwards (so that when there are
  // warps to spare, a warp takes whole-warp copies or small ones, not both):
  // lane group g of warp nw-1-r takes copies big + kPerWarp r + g, then every
  // kPerWarp nw-th
  constexpr int kPerWarp = 32 / kPackGroup;
  c = sp.big + kPerWarp * (nw - 1 - gw) + lane / kPackGroup;
  if (c < sp.total) cp = a.copies[c];
  for (; c < sp.total; c += kPerWarp * nw) {
    const PackCopy cur = cp;
    if (c + kPerWarp * nw < sp.total) cp = a.copies[c + kPerWarp * nw];
    pack_one<T, kPackGroup, kPackGroupU>(c < sp.small_a ? a : b, cur, lane % kPackGroup);
  }
}

template <class T>
__global__ void zero_kernel(T *C, const ZeroBlock *blocks, int nblocks) {
  for (int bi = blockIdx.x; bi < nblocks; bi += gridDim.x) {
    const ZeroBlock z = blocks[bi];
    const int n = z.rows * z.cols;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int r = e / z.cols, q = e - r * z.cols;
      C[z.off + (int64_t)r * z.ld + q] = T(0);
    }
  }
}

__global__ void control_fp64_kernel(const double *A, const double *B, double *C, int64_t a_off, int64_t lda,
                                    int64_t b_off, int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= m * n) return;
  const int r = e / n, c = e - r * n;
  double acc = 0.0;
  for (int q = 0; q < k; ++q) acc = fma(A[a_off + r * lda + q], B[b_off + q * ldb + c], acc);
  C[c_off + r * ldc + c] += acc;
}

__global__ void control_bf16_kernel(const uint16_t *A, const uint16_t *B, float *C, int64_t a_off, int64_t lda,
                                    int64_t b_off, int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= m * n) return;
  const int r = e / n, c = e - r * n;
  float acc = 0.f;
  for (int q = 0; q < k; ++q) {
    const float a = __uint_as_float((uint32_t)A[a_off + r * lda + q] << 16);
    const float b = __uint_as_float((uint32_t)B[b_off + q * ldb + c] << 16);
    acc = fmaf(a, b, acc);
  }
  C[c_off + r * ldc + c] += acc;
}

}  // namespace

cudaError_t launch_fp64_grouped(const Fp64Params &p, int grid, cudaStream_t s) {
  if (p.check) {
    if (p.ntasks > 0) fp64_grouped_kernel<4, true><<<grid, kThreads, 0, s>>>(p);
    else fp64_grouped_kernel<3, true><<<grid, kThreads, 0, s>>>(p);
  } else {
    if (p.ntasks > 0) fp64_grouped_kernel<4, false><<<grid, kThreads, 0, s>>>(p);
    else fp64_grouped_kernel<3, false><<<grid, kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

int fp64_max_ctas_per_sm(bool tail_only) {
  int n = 0;
  const cudaError_t e = tail_only
                            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp64_grouped_kernel<3, false>, kThreads, 0)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp64_grouped_kernel<4, false>, kThreads, 0);
  return e == cudaSuccess && n > 0 ? n : 1;
}

cudaError_t launch_pack2(const PackParams &a, const PackParams &b, const PackSplit &split, int sms, cudaStream_t s) {
  if (split.total <= 0) return cudaSuccess;
  // eight CTAs per SM, about two waves at this kernel's occupancy: the copies
  // are dealt to the warps in turn, and the second wave's warps pick up the
  // shares of the first wave's slowest (measured faster than one wave)
  int grid = std::max(1, sms) * 8;
  constexpr int64_t kPerWarp = 32 / kPackGroup;
  const int64_t warps = split.big + ((int64_t)split.total - split.big + kPerWarp - 1) / kPerWarp;
  const int64_t need = (warps + 7) / 8;   // eight warps a CTA
  grid = grid < need ? grid : (int)need;
  if (a.elem_bytes == 8) pack_kernel<double><<<grid, 256, 0, s>>>(a, b, split);
  else pack_kernel<uint16_t><<<grid, 256, 0, s>>>(a, b, split);
  return cudaGetLastError();
}

cudaError_t launch_zero(void *C, int elem_bytes, const ZeroBlock *blocks, int nblocks, int grid, cudaStream_t s) {
  if (nblocks <= 0) return cudaSuccess;
  grid = grid < nblocks ? grid : nblocks;
  if (elem_bytes == 8) zero_kernel<double><<<grid, 256, 0, s>>>((double *)C, blocks, nblocks);
  else zero_kernel<float><<<grid, 256, 0, s>>>((float *)C, blocks, nblocks);
  return cudaGetLastError();
}

cudaError_t launch_control_fp64(const double *A, const double *B, double *C, int64_t a_off, int64_t lda, int64_t b_off,
                                int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k, cudaStream_t s) {
  const int e = m * n;
  control_fp64_kernel<<<(e + 127) / 128, 128, 0, s>>>(A, B, C, a_off, lda, b_off, ldb, c_off, ldc, m, n, k);
  return cudaGetLastError();
}

cudaError_t launch_control_bf16(const uint16_t *A, const uint16_t *B, float *C, int64_t a_off, int64_t lda,
                                int64_t b_off, int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k,
                                cudaStream_t s) {
  const int e = m * n;
  control_bf16_kernel<<<(e + 127) / 128, 128, 0, s>>>(A, B, C, a_off, lda, b_off, ldb, c_off, ldc, m, n, k);
  return cudaGetLastError();
}

}  // namespace bs

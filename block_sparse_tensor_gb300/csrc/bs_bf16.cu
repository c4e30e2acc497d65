// BF16-in / FP32-out persistent grouped GEMM on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// The tensor-core path is taken only where a coalesced group is a genuine
// dense contraction in a type with a tensor-core path (uni20 design note
// "block coalescing", "Two coalescing modes": a single-axis group is one
// zero-waste GEMM).  One task is a 128 x BN tile (BN <= 256) of one
// contraction-axis group; its K loop walks the group's inner segments, each
// with its own tensor maps for the A view (group rows x d_k) and the B view
// (d_k x group columns).  The copy engine fills everything past a view's edge
// with zeros, so ragged d_k needs no padding in memory and adds nothing.
//
// Warp roles (192 threads, one CTA per SM, tasks striped over CTAs):
//   warp 0  TMA producer: A tile 128 x 64 (K-major, 128-byte swizzle) and B
//           tile 64 x BN (N-major, 128-byte swizzle) per stage, 4 stages;
//   warp 1  TMEM owner and MMA issuer (one thread): 4 x (M128, N=BN, K16) per
//           stage into one of two 256-column FP32 accumulators;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, staged through
//           swizzled shared memory, TMA tensor stores clipped at the group edge.
// Every wait is bounded by the global timer; on expiry the kernel records
// a timeout in the status word, drains its copies and MMAs (again bounded),
// frees its tensor memory and returns.
#include <cuda.h>

#include "bs_host.h"

namespace bs {

namespace {

constexpr int kStages = 4;
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;        // 16 KB
constexpr int kBChunkBytes = 64 * kBK * 2;        // one 64-column N chunk: 8 KB
constexpr int kBTileBytes = 4 * kBChunkBytes;     // BN up to 256
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kTmemCols = 512;
constexpr int kThreadsBf16 = 192;

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr int kCtlBytes = 256;                    // Ctl rounded up
constexpr int kEpiBufBytes = 32 * 128;            // 32 rows x 32 FP32 columns
constexpr size_t kSmemBytes =
    1024 /*align slack*/ + (size_t)kStages * kStageBytes + kCtlBytes + 4 * 2 * kEpiBufBytes;
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false on timeout or when another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int32_t *abort_flag, uint64_t limit) {
  uint64_t start = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(a, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort_flag) return false;
      const uint64_t now = gtime();
      if (start == 0) start = now;
      else if (now - start > limit) return false;
    }
  }
}

__device__ __forceinline__ void prefetch_map(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Warm the descriptor cache with every tensor map task `t` will use.
__device__ __forceinline__ void prefetch_task_maps(const Bf16Params &p, const char *maps, int t) {
  if (t >= p.ntasks) return;
  const Bf16Task T = p.tasks[t];
  for (int q = 0; q < T.pair_count; ++q) {
    const Bf16Pair pr = p.pairs[T.pair_begin + q];
    prefetch_map(maps + (size_t)pr.map_a * 128);
    prefetch_map(maps + (size_t)pr.map_b * 128);
  }
  if (T.map_c >= 0) prefetch_map(maps + (size_t)T.map_c * 128);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, uint32_t mbar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(mbar), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start, leading and stride byte
// offsets in 16-byte units, descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D = F32, A = B = BF16, A K-major,
// B N-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t instr_desc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void record_timeout(const Bf16Params &p, Ctl *ctl) {
  ctl->abort_flag = 1;
  atomicExch(p.status, (int32_t)DS_TIMEOUT);
}

__global__ void __launch_bounds__(kThreadsBf16, 1) bf16_grouped_kernel(const Bf16Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // [stages | epilogue staging, 1024-aligned for the 128-byte swizzle | control block]
  Ctl *ctl = (Ctl *)(smem + (size_t)kStages * kStageBytes + 4 * 2 * kEpiBufBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t *abort_flag = &ctl->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), 4);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const char *maps = (const char *)p.maps;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued_phase[kStages];
      bool outstanding[kStages];
      for (int s = 0; s < kStages; ++s) outstanding[s] = false;
      prefetch_task_maps(p, maps, blockIdx.x);
      for (int t = blockIdx.x; ok && t < p.ntasks; t += gridDim.x) {
        const Bf16Task T = p.tasks[t];
        prefetch_task_maps(p, maps, t + gridDim.x);   // the next task's descriptors load while this one streams
        const int nb = (T.bn + 63) / 64;
        const uint32_t bytes = kATileBytes + nb * kBChunkBytes;
        for (int q = 0; ok && q < T.pair_count; ++q) {
          const Bf16Pair pr = p.pairs[T.pair_begin + q];
          const void *ma = maps + (size_t)pr.map_a * 128;
          const void *mb = maps + (size_t)pr.map_b * 128;
          for (int kc = 0; kc < pr.klen; kc += kBK) {
            if (!mbar_wait(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
              record_timeout(p, ctl);
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&ctl->full[stage]);
            if ((p.debug_flags & 1) && blockIdx.x == 0 && t == (int)blockIdx.x && q == 0 && kc == 0) {
              // test hook: this stage is never filled, so the MMA thread's
              // bounded wait on it runs out and the kernel reports a timeout
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            mbar_expect_tx(fb, bytes);
            unsigned char *st = smem + (size_t)stage * kStageBytes;
            tma_load_2d(smem_u32(st), ma, fb, kc, T.m0);
            for (int c = 0; c < nb; ++c)
              tma_load_2d(smem_u32(st + kATileBytes + c * kBChunkBytes), mb, fb, T.n0 + 64 * c, kc);
            outstanding[stage] = true;
            issued_phase[stage] = phase;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: every issued stage completes its transfer before the CTA exits.
      // (On the normal path the MMA thread has consumed them all already.)
      for (int s = 0; s < kStages; ++s)
        if (outstanding[s]) {
          uint64_t t0 = gtime();
          while (!mbar_try(smem_u32(&ctl->full[s]), issued_phase[s]) && gtime() - t0 < p.timeout_ns) {
          }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued_any = false;
      for (int t = blockIdx.x; ok && t < p.ntasks; t += gridDim.x) {
        const Bf16Task T = p.tasks[t];
        const uint32_t idesc = instr_desc(T.bn);
        if (!mbar_wait(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          record_timeout(p, ctl);
          break;
        }
        fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        uint32_t accumulate = 0;
        for (int q = 0; ok && q < T.pair_count; ++q) {
          const int klen = p.pairs[T.pair_begin + q].klen;
          for (int kc = 0; kc < klen; kc += kBK) {
            if (!mbar_wait(smem_u32(&ctl->full[stage]), phase, abort_flag, p.timeout_ns)) {
              record_timeout(p, ctl);
              ok = false;
              break;
            }
            fence_after();
            const uint32_t a0 = smem_u32(smem + (size_t)stage * kStageBytes);
            const uint32_t b0 = a0 + kATileBytes;
            const int ksteps = min(4, (klen - kc + 15) / 16);
            for (int ks = 0; ks < ksteps; ++ks) {
              const uint64_t ad = smem_desc(a0 + ks * 32, 16, 1024);
              const uint64_t bd = smem_desc(b0 + ks * 2048, kBChunkBytes, 1024);
              mma_bf16(d_tmem, ad, bd, idesc, accumulate);
              accumulate = 1;
            }
            mma_commit(smem_u32(&ctl->empty[stage]));
            issued_any = true;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&ctl->tfull[acc]));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: all MMAs issued by this thread finish before tensor memory is freed.
      if (issued_any) {
        mma_commit(smem_u32(&ctl->drain));
        uint64_t t0 = gtime();
        while (!mbar_try(smem_u32(&ctl->drain), 0) && gtime() - t0 < p.timeout_ns) {
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Each warp owns TMEM lanes 32*quarter .. +31 (tile rows) and two 4 KB
    // staging buffers.  A 32 x 32 FP32 chunk goes TMEM -> registers -> shared
    // memory (128-byte swizzle, so the 32 row writes of one column group hit
    // distinct banks) -> one TMA tensor store, which clips rows and columns
    // past the group's edge.  Unaligned C views fall back to direct stores.
    const int quarter = warp & 3;
    unsigned char *stage_buf = smem + (size_t)kStages * kStageBytes + (size_t)quarter * 2 * kEpiBufBytes;
    const char *maps = (const char *)p.maps;
    int acc = 0;
    uint32_t acc_phase = 0;
    int buf = 0;
    for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
      const Bf16Task T = p.tasks[t];
      if (!mbar_wait(smem_u32(&ctl->tfull[acc]), acc_phase, abort_flag, p.timeout_ns)) {
        if (lane == 0) record_timeout(p, ctl);
        break;
      }
      fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256);
      if (T.map_c >= 0 && T.m0 + quarter * 32 < T.m) {   // quarters wholly past the last row store nothing
        const void *mc = maps + (size_t)T.map_c * 128;
        for (int c0 = 0; c0 < T.bn; c0 += 32) {
          float v[32];
          tmem_ld16(trow + c0, v);
          tmem_ld16(trow + c0 + 16, v + 16);
          // the buffer written two chunks ago must have been read by its store
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
          unsigned char *b = stage_buf + buf * kEpiBufBytes + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *(float4 *)(b + ((j ^ (lane & 7)) << 4)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            asm volatile(
                "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(mc),
                "r"(smem_u32(stage_buf + buf * kEpiBufBytes)), "r"(T.n0 + c0), "r"(T.m0 + quarter * 32)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
          buf ^= 1;
        }
      } else if (T.map_c < 0) {
        const int row = T.m0 + quarter * 32 + lane;
        const bool row_ok = row < T.m;
        float *crow = p.C + T.c_off + (int64_t)row * T.ldc + T.n0;
        const int ncols = min(T.bn, T.n - T.n0);
        for (int c0 = 0; c0 < T.bn; c0 += 16) {
          float v[16];
          tmem_ld16(trow + c0, v);
          if (!row_ok) continue;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c0 + i < ncols) crow[c0 + i] = v[i];
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // staged stores finish reading shared memory before the CTA can exit
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

size_t bf16_smem_bytes() { return kSmemBytes; }

cudaError_t launch_bf16_grouped(const Bf16Params &p, int grid, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bf16_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  bf16_grouped_kernel<<<grid, kThreadsBf16, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bs

// BF16-in / FP32-out persistent grouped GEMM on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// The tensor-core path is taken only where a coalesced group is a genuine
// dense contraction in a type with a tensor-core path (uni20 design note
// "block coalescing", "Two coalescing modes": a single-axis group is one
// zero-waste GEMM).  One task is a 128 x BN tile (BN <= 256) of one
// contraction-axis group.  Its K loop walks the group's inner segments, each
// with its own tensor maps for the A view (group rows x d_k) and the B view
// (d_k x group columns).  The copy engine fills everything past a view's edge
// with zeros, so ragged d_k needs no padding in memory and adds nothing.
//
// One CTA per SM.  At plan time each CTA gets its own task list (longest
// first onto the least loaded CTA), unrolled into a flat list of 64-deep K
// stages; the CTA preloads the head of both lists to shared memory and reads
// the rest one stage ahead of its use.
//   warp 0 and the last warp  TMA copies (one thread each, alternate stages:
//           issuing a stage's copies costs a thread about the same time
//           whatever their size, so two issuers keep the copy engine busier):
//           per stage one A box 128 x 64 (K-major, 128-byte swizzle) and the
//           tile's B columns, 64 x 64 chunks (N-major, 128-byte swizzle), its
//           whole chunks in one 3-D box and a ragged last chunk in a 2-D box.
//           Thread 0 fills the first ring of stages straight from the global
//           list while the rest of the CTA is still setting up;
//   warp 1  TMEM owner and MMA issuer (one thread): per stage up to four
//           M128 x N=BN x K16 MMAs (one instruction block when all four reach
//           real K) into 256-column FP32 slots used in rotation, so the
//           epilogue of one tile overlaps the next tile's MMAs;
//   warps 2-9  epilogue, two warps per 32-lane TMEM quarter: tcgen05.ld of 32
//           columns at a time, a swizzled shared-memory transpose, coalesced
//           masked stores (plain stores: no padding byte of C is written).
// Every wait is bounded by the global timer; on expiry the kernel records
// a timeout in the status word, drains its copies and MMAs (again bounded),
// frees its tensor memory and returns.
#include <cuda.h>

#include "bs_host.h"

namespace bs {

namespace {

#ifndef BS_BF16_STAGES
#define BS_BF16_STAGES 4
#endif
#ifndef BS_BF16_EPI_WARPS
#define BS_BF16_EPI_WARPS 8
#endif
constexpr int kStages = BS_BF16_STAGES;
constexpr int kBM = 128;                          // rows of the accumulator (UMMA M)
constexpr int kBK = 64;                           // K per stage (one 128-byte swizzle row of BF16)
constexpr int kATileBytes = kBM * kBK * 2;        // 16 KB: 128 rows of A
constexpr int kBChunkBytes = 64 * kBK * 2;        // one 64-column N chunk of B: 8 KB
constexpr int kBTileBytes = 4 * kBChunkBytes;     // BN up to 256
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kTmemCols = 512;                    // two 256-column FP32 accumulator slots
constexpr int kEpiWarps = BS_BF16_EPI_WARPS;      // epilogue warps, a multiple of 4 (one group per TMEM lane quarter)
static_assert(kEpiWarps % 4 == 0, "epilogue warps per lane quarter");
constexpr int kProducer1Warp = 2 + kEpiWarps;     // the second copy thread's warp, after the epilogue warps
constexpr int kThreadsBf16 = 32 * (kProducer1Warp + 1);
static_assert(kStages % 2 == 0, "each of the two copy threads owns every other stage");
constexpr int kEpiBufBytes = 32 * 128;            // 32 rows x 32 FP32 columns per epilogue warp
constexpr int kTaskCache = 16;                    // head of this CTA's task list, in shared memory
constexpr int kStageCache = 32;                   // head of this CTA's stage list, in shared memory

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t issued[kStages];   // 1 + phase of the last copy issued into the stage, 0 if none
  uint32_t tmem_base;
  int32_t abort_flag;
};

// [control block | task cache | stage cache | pad to 1024 | stages | epilogue staging]
constexpr int kCtlBytes = 256;
constexpr int kHeadBytes = kCtlBytes + kTaskCache * (int)sizeof(Bf16Task) + kStageCache * (int)sizeof(Bf16Stage);
constexpr size_t kSmemBytes = kHeadBytes + 1023 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kEpiBufBytes;
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, uint32_t mbar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(mbar), "r"(x), "r"(y), "r"(z)
      : "memory");
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

// The four K16 steps of a full stage in one instruction block: the shared
// memory descriptors advance by 32 bytes of A (2 units) and 2048 bytes of B
// (128 units) per step, so only the first MMA of a tile starts from zero.
__device__ __forceinline__ void mma_bf16_x4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, 0, 0;\n"
      " add.s64 a1, %1, 2;\n add.s64 a2, %1, 4;\n add.s64 a3, %1, 6;\n"
      " add.s64 b1, %2, 128;\n add.s64 b2, %2, 256;\n add.s64 b3, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive FP32 columns of this thread's TMEM lane, one wait for all.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void record_timeout(const Bf16Params &p, Ctl *ctl) {
  ctl->abort_flag = 1;
  atomicExch(p.status, (int32_t)DS_TIMEOUT);
}

// The ti-th task and the si-th stage of this CTA's lists (the heads come from shared memory).
__device__ __forceinline__ Bf16Task task_at(const Bf16Params &p, const Bf16Task *cache, const Bf16Cta &me, int ti) {
  return ti < kTaskCache ? cache[ti] : p.tasks[me.task_begin + ti];
}
__device__ __forceinline__ Bf16Stage stage_at(const Bf16Params &p, const Bf16Stage *cache, const Bf16Cta &me, int si) {
  return si < kStageCache ? cache[si] : p.stages[me.stage_begin + si];
}

__global__ void __launch_bounds__(kThreadsBf16, 1) bf16_grouped_kernel(const Bf16Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Ctl *ctl = (Ctl *)smem_raw;
  Bf16Task *tcache = (Bf16Task *)(smem_raw + kCtlBytes);
  Bf16Stage *scache = (Bf16Stage *)(smem_raw + kCtlBytes + kTaskCache * sizeof(Bf16Task));
  // stage buffers 1024-aligned for the 128-byte swizzle
  unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + kHeadBytes + 1023) & ~(uintptr_t)1023);
  unsigned char *epi_base = smem + (size_t)kStages * kStageBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t *abort_flag = &ctl->abort_flag;
  const char *maps = (const char *)p.maps;
  const Bf16Cta me = p.ctas[blockIdx.x];

  // Copy issue: stage ps of this CTA's list goes to ring slot ps % kStages.
  // The slot's copies all complete on its full barrier; issued[] remembers
  // the last phase so that a copy thread can wait out its copies on exit.
  auto issue = [&](const Bf16Stage &E, int ps) {
    const int slot = ps % kStages;
    const uint32_t phase = (uint32_t)(ps / kStages) & 1u;
    const uint32_t fb = smem_u32(&ctl->full[slot]);
    // test hook: CTA 0's first stage is never filled, so the MMA thread's
    // bounded wait on it runs out and the kernel reports a timeout
    const bool withhold = (p.debug_flags & 1) && blockIdx.x == 0 && ps == 0;
    if (!withhold) {
      mbar_expect_tx(fb, (uint32_t)(kATileBytes + E.nb * kBChunkBytes));
      unsigned char *st = smem + (size_t)slot * kStageBytes;
      tma_load_2d(smem_u32(st), maps + (size_t)E.map_a * 128, fb, E.k0, E.m0);   // rows past the group read as zero
      // the tile's first nb3 whole B chunks in one 3-D box, the rest chunk by chunk
      const int nb3 = E.flags >> 8;
      if (nb3 > 0) tma_load_3d(smem_u32(st + kATileBytes), maps + (size_t)E.map_b3 * 128, fb, 0, E.k0, E.n0 >> 6);
      const void *mb = maps + (size_t)E.map_b * 128;
      for (int c = nb3; c < E.nb; ++c) tma_load_2d(smem_u32(st + kATileBytes + c * kBChunkBytes), mb, fb, E.n0 + 64 * c, E.k0);
      ctl->issued[slot] = phase + 1u;
    }
  };
  // One copy thread's share after the first ring: stages first, first + 2, ...
  // (slots of one parity), each once its slot is free.  Issuing a stage's
  // copies takes its thread a fixed time whatever their size, so two threads
  // issuing alternate stages keep the copy engine busier than one.
  auto produce = [&](int first) {
    // each stage's record is read one of this thread's stages ahead (past the
    // shared-memory head of the list it comes from global memory)
    Bf16Stage F = first < me.stage_count ? stage_at(p, scache, me, first) : Bf16Stage{};
    for (int ps = first; ps < me.stage_count; ps += 2) {
      const Bf16Stage E = F;
      if (ps + 2 < me.stage_count) F = stage_at(p, scache, me, ps + 2);
      const int slot = ps % kStages;
      const uint32_t phase = (uint32_t)(ps / kStages) & 1u;
      if (!mbar_wait(smem_u32(&ctl->empty[slot]), phase ^ 1u, abort_flag, p.timeout_ns)) {
        record_timeout(p, ctl);
        break;
      }
      issue(E, ps);
      if (ps + 2 < me.stage_count) {   // warm the descriptor cache for this thread's next stage
        prefetch_map(maps + (size_t)F.map_a * 128);
        prefetch_map(maps + (size_t)((F.flags >> 8) ? F.map_b3 : F.map_b) * 128);
      }
    }
    // Drain: every copy issued into this thread's slots completes before the
    // CTA exits.  (On the normal path the MMA thread has consumed them all.)
    for (int s = first % 2; s < kStages; s += 2)
      if (ctl->issued[s]) {
        const uint64_t t0 = gtime();
        while (!mbar_try(smem_u32(&ctl->full[s]), ctl->issued[s] - 1u) && gtime() - t0 < p.timeout_ns) {
        }
      }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), kEpiWarps);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    for (int s = 0; s < kStages; ++s) ctl->issued[s] = 0u;
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // The first ring of stages needs no free slot: fill it from the global
    // list while the other warps allocate tensor memory and load the lists.
    for (int ps = 0; ps < min(kStages, me.stage_count); ++ps) issue(p.stages[me.stage_begin + ps], ps);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x >= 64) {   // the epilogue warps preload the heads of both lists
    const int i = threadIdx.x - 64;
    if (i < kTaskCache && i < me.task_count) tcache[i] = p.tasks[me.task_begin + i];
    const int j = i - 64;
    if (j >= 0 && j < kStageCache && j < me.stage_count) scache[j] = p.stages[me.stage_begin + j];
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) produce(kStages);   // ------------------------------ copies, even stages
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // Tiles take the two accumulator slots in turn; the epilogue walks the
      // same sequence.  Everything the issue loop touches stays in scalar
      // registers (a local array here cost more than half the tensor
      // throughput), and a full stage is one instruction block.
      int stage = 0, slot = 0;
      uint32_t phase = 0, te0 = 0, te1 = 0;   // ring phase; tempty phase per slot
      uint32_t d = tmem_base, idesc = 0, acc = 0;
      bool issued_any = false;
      // each stage's record is read one stage ahead (past the shared-memory
      // head of the list it comes from global memory)
      Bf16Stage En = me.stage_count > 0 ? stage_at(p, scache, me, 0) : Bf16Stage{};
      for (int si = 0; si < me.stage_count; ++si) {
        const Bf16Stage E = En;
        if (si + 1 < me.stage_count) En = stage_at(p, scache, me, si + 1);
        if (E.flags & kStageFirst) {
          if (!mbar_wait(smem_u32(&ctl->tempty[slot]), (slot ? te1 : te0) ^ 1u, abort_flag, p.timeout_ns)) {
            record_timeout(p, ctl);
            break;
          }
          if (slot) te1 ^= 1u;
          else te0 ^= 1u;
          fence_after();
          d = tmem_base + (uint32_t)(slot * 256);
          idesc = instr_desc(E.bn);
          acc = 0;
        }
        if (!mbar_wait(smem_u32(&ctl->full[stage]), phase, abort_flag, p.timeout_ns)) {
          record_timeout(p, ctl);
          break;
        }
        fence_after();
        const uint32_t a0 = smem_u32(smem + (size_t)stage * kStageBytes);
        const uint64_t ad = smem_desc(a0, 16, 1024), bd = smem_desc(a0 + kATileBytes, kBChunkBytes, 1024);
        if (E.ksteps == 4) {
          mma_bf16_x4(d, ad, bd, idesc, acc);
        } else {
          for (int ks = 0; ks < E.ksteps; ++ks) mma_bf16(d, ad + 2 * ks, bd + 128 * ks, idesc, acc | (uint32_t)ks);
        }
        acc = 1;
        mma_commit(smem_u32(&ctl->empty[stage]));
        issued_any = true;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (E.flags & kStageLast) {
          mma_commit(smem_u32(&ctl->tfull[slot]));
          slot ^= 1;
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
  } else if (warp == kProducer1Warp) {
    if (lane == 0) produce(kStages + 1);   // -------------------------- copies, odd stages
  } else {
    // -------------------------------------------------------------- epilogue
    // A warp may read only TMEM lanes 32*(warp%4) .. +31 (tile rows).  Each
    // 32 x 32 FP32 chunk goes TMEM -> registers -> shared memory (row per
    // lane, 16-byte pieces XOR-swizzled by row so both the row writes and
    // the column reads are free of bank conflicts) -> coalesced global stores
    // of four 128-byte row segments per instruction, masked at the group edge.
    const int quarter = warp & 3;
    const int ew = warp - 2;
    const int grp = ew >> 2;                  // which 32-column chunks: grp, grp + kEpiWarps/4, ...
    unsigned char *stg = epi_base + (size_t)ew * kEpiBufBytes;
    int slot = 0;
    uint32_t tf0 = 0, tf1 = 0;   // tfull phase per slot
    for (int ti = 0; ti < me.task_count; ++ti) {
      const Bf16Task T = task_at(p, tcache, me, ti);
      if (!mbar_wait(smem_u32(&ctl->tfull[slot]), slot ? tf1 : tf0, abort_flag, p.timeout_ns)) {
        if (lane == 0) record_timeout(p, ctl);
        break;
      }
      if (slot) tf1 ^= 1u;
      else tf0 ^= 1u;
      fence_after();
      const int row0 = T.m0 + 32 * quarter;
      if (row0 < T.m) {
        const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(slot * 256);
        float *cbase = p.C + T.c_off;
        for (int c0 = 32 * grp; c0 < T.bn; c0 += 32 * (kEpiWarps / 4)) {
          float v[32];
          tmem_ld32(trow + c0, v);
          unsigned char *mine = stg + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *(float4 *)(mine + ((j ^ (lane & 7)) << 4)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          __syncwarp();
          const int j = lane & 7;
          const int gcol = T.n0 + c0 + 4 * j;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const int grow = row0 + r;
            const float4 x = *(const float4 *)(stg + r * 128 + ((j ^ (r & 7)) << 4));
            if (grow < T.m) {
              float *dst = cbase + (int64_t)grow * T.ldc + gcol;
              if (T.c_vec && gcol + 4 <= T.n) {
                *(float4 *)dst = x;
              } else {
                if (gcol + 0 < T.n) dst[0] = x.x;
                if (gcol + 1 < T.n) dst[1] = x.y;
                if (gcol + 2 < T.n) dst[2] = x.z;
                if (gcol + 3 < T.n) dst[3] = x.w;
              }
            }
          }
          __syncwarp();
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[slot]));
      slot ^= 1;
    }
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

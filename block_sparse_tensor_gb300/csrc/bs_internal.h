// Internal structures shared by the host planner and the device kernels.
//
// A coalesced group is one dense GEMM, C_g[M x N] (+)= A_g[M x K] B_g[K x N],
// whose operands are unions of block views ("Expressed as strided views over
// shared storage", uni20 design note "block coalescing").  Every group is
// described by two segment lists and one addressing rule:
//
//   A(r, kk) = A[ RA(r) + KA(kk) + RL(r) * KL(kk) ]
//   B(kk, c) = B[ KB(kk) + c ]
//   C(r, c)  = C[ RC(r) + c ]
//
// Row segment t covers rows r0 .. r0+rows-1 of the group:
//   RA(r) = ra + (r - r0) * lda,  RL(r) = rl ? (r - r0) : 0,  RC(r) = rc + (r - r0) * ldc.
// Inner segment s covers k0 .. k0+klen-1 of the group's concatenated K:
//   KA(kk) = ka + (kk - k0),  KL(kk) = kl,  KB(kk) = kb + (kk - k0) * ldb.
//
// Contraction-axis group (fixed i, j; K concatenated): one row segment
// {ra 0, lda 0, rl 1, rc c_off, ldc} and one inner segment per run of
// adjacent blocks {ka a_off, kl lda, kb b_off, ldb}.
// Free-axis group (fixed k, j; rows stacked): one row segment per run of
// stacked A blocks {ra a_off, lda, rl 0, rc c_off(i, j), ldc} and one inner
// segment {ka 0, kl 0, kb b_off, ldb}; its stores are atomic adds.
#pragma once
#include <stdint.h>
#include <vector_types.h>

namespace bs {

struct RowSeg {
  int64_t ra;
  int64_t lda;
  int64_t rc;
  int64_t ldc;
  int32_t r0;
  int32_t rows;
  int32_t rl;
  int32_t pad_;
};

struct KSeg {
  int64_t ka;
  int64_t kl;
  int64_t kb;
  int64_t ldb;
  int32_t k0;
  int32_t klen;
};

enum GroupFlags : int32_t { GF_ATOMIC = 1 };

struct Group {
  int32_t m, n, k;
  int32_t flags;
  int32_t rseg_begin, rseg_count;
  int32_t kseg_begin, kseg_count;
};

// A tail group with one row segment and one inner segment, resolved at plan
// time: output (r, c) is sum over kk < k of A[a0 + r*as + kk] * B[b0 + kk*ldb + c],
// stored at C[c0 + r*ldc + c].  k = 0 marks a group that takes the general path
// (several segments).  When the plan pads the group to a bucket shape, its
// outputs run kpad steps (loads past k give zero) and its list may carry
// outputs with r >= m or c >= n that load and store nothing.
struct TailDesc {
  int64_t a0, as;
  int64_t b0, ldb;
  int64_t c0, ldc;
  int32_t k;
  int32_t flags;
  int32_t kpad;
  int32_t m, n;
  int32_t pad_;
};

enum TaskKind : int32_t { TK_TILE = 0 };

// TK_TILE: one CTA computes rows m0 .. m0+tm-1, columns n0 .. n0+tn-1 of group `g`.
// Small groups are not tile tasks: their outputs form the tail list
// tail_elems[e] = {group, r << 16 | c}, groups in decreasing K, row-major
// inside a group.  A tail task is kThreads consecutive outputs, one per
// thread, so the lanes of one warp run loops of nearly equal length (every
// FMA instruction carries almost 32 useful lanes) and the warps of one CTA
// walk the same B rows together.
struct Task {
  int32_t kind;
  int32_t g;       // group
  int32_t m0;
  int32_t n0;
  int32_t tm;
  int32_t tn;
};

constexpr int kThreads = 256;          // threads of the FP64 grouped kernel
constexpr int kElemsPerThread = 4;     // tile outputs per thread
constexpr int kTileMaxElems = kThreads * kElemsPerThread;
constexpr int kTileMaxDim = 128;       // bound on tm and tn
constexpr int kKC = 16;                // inner chunk per shared-memory stage
constexpr int kTailMaxElems = 4096;    // groups up to this many outputs take the lane-packed path

// One block copy of the gather ("pack") kernel.
struct PackCopy {
  int64_t src;
  int64_t src_ld;
  int64_t dst;
  int64_t dst_ld;
  int32_t rows;
  int32_t cols;
};

// One C block for the zero fill that precedes atomic scatter.
struct ZeroBlock {
  int64_t off;
  int64_t ld;
  int32_t rows;
  int32_t cols;
};

// Counter block of a plan: a 256-byte status block (the status word at byte
// 128), then two sets of work counters used by alternate launches of the FP64
// kernel (each launch prepares the other set for the next, so no launch has to
// reset its own at exit; a launch captured into a graph resets its own set
// instead).  A set: [0] next tile task, [1] CTAs finished (exit reset only),
// [2] tail tasks taken, [64 + q] next task of tail queue q.
inline size_t counter_set_bytes(int nq) { return (size_t)(256 + 4 * nq + 255) / 256 * 256; }
inline size_t counter_bytes(int nq) { return 256 + 2 * counter_set_bytes(nq); }
constexpr int kQueueCounterBase = 64;   // in uint32 units

// Device status word values (first int of the status buffer).
enum DeviceStatus : int32_t { DS_OK = 0, DS_TIMEOUT = 1, DS_BOUNDS = 2 };

constexpr int kMaxQueues = 160;   // tail queues: one per SM, at most this many
constexpr int kMaxSmIds = 256;    // hardware SM identifiers the parameter map covers
// Tail-list entry that pads a tail task to kThreads outputs: no output.
constexpr int32_t kTailPad = 0x7FFF7FFF;
// Set in a tail entry's group field: the entry sums the second half of K of an
// output whose first half the lane 16 below sums (a split group).
constexpr int32_t kTailHi = 1 << 30;

struct Fp64Params {
  const double *A;
  const double *B;
  double *C;
  const Task *tasks;
  const Group *groups;
  const RowSeg *rsegs;
  const KSeg *ksegs;
  const int2 *tail_elems;  // tail task t covers tail_elems[kThreads t .. kThreads t + kThreads - 1]
  const TailDesc *tdesc;   // per group (used for tail groups)
  int32_t ntasks;
  int32_t ntail;       // entries of the tail list (a multiple of kThreads, padding included)
  int32_t nct;         // tail tasks
  int32_t nq;          // queues (one per SM of the planned device)
  uint32_t *counter;       // this launch's counter set (zeroed by the previous launch or the host)
  uint32_t *counter_next;  // the set the next launch uses: this launch zeroes it
  int32_t reset_at_exit;   // 1 (counter_next null): the last CTA to finish returns this launch's set to
                           // zero, for a launch captured into a graph that replays it
  int32_t *status;
  int64_t nA, nB, nC;  // elements of the buffers read and written (the checked instance tests them)
  int32_t check;       // 1: the checked instance
  int32_t nsm_ids;     // entries of sm_queue in use (0: take %smid modulo nq)
  // Kept in the parameters, so a CTA finds its first task without a memory load:
  int32_t qptr[kMaxQueues + 1];   // queue q holds tail tasks qptr[q] .. qptr[q+1]-1 (consecutive)
  int16_t sm_queue[kMaxSmIds];    // dense SM index per hardware SM identifier, -1 if unknown
};

struct PackParams {
  const void *src;
  void *dst;
  const PackCopy *copies;
  int32_t ncopies;
  int32_t elem_bytes;
};

// The gather's copy list in four runs: [0, big_a) A's copies moved by whole
// warps, [big_a, big) B's; [big, small_a) A's small copies (at most
// kPackSmallElems elements) moved by 8-lane groups, four to a warp, and
// [small_a, total) B's.
constexpr int32_t kPackSmallElems = 64;
struct PackSplit {
  int32_t big_a, big, small_a, total;
  bool of_a(int64_t t) const { return t < big_a || (t >= big && t < small_a); }
};

// The FP64 gather in shared-memory segments: a segment is a source range of
// at most kSegElems elements (consecutive blocks of the source layout, or a
// band or row chunk of one block) that one bulk copy brings into shared
// memory, with the pieces it holds (a block, or a band or row chunk of one)
// and where each goes in the destination.  Segments are listed in source
// order, A's first.
constexpr int32_t kSegElems = 2048;
constexpr int32_t kSegPieces = 128;   // pieces a segment holds at most
constexpr int32_t kSegStages = 10;    // segments in flight per SM
constexpr int32_t kSegMaxPerSm = 2;   // a plan gathers by segments only up to this many per SM
struct PackPiece {
  int64_t dst;       // first destination element
  int32_t src_off;   // first source element, counted from the segment's first
  int32_t rows, cols;
  int32_t src_ld, dst_ld;
  int32_t pad_;
};
static_assert(sizeof(PackPiece) == 32, "piece record");
struct PackSeg {
  int64_t src;   // first source element
  int32_t n;     // elements from src to the end of its last piece
  int32_t piece_begin, piece_count;
  int32_t operand;   // 0: A, 1: B
  int64_t pad_;
};
static_assert(sizeof(PackSeg) == 32, "segment record");
struct SegParams {
  const double *src[2];    // A, B
  double *dst[2];          // their panel workspaces
  int64_t src_nelems[2];   // elements the caller's A and B buffers hold (the layouts' counts)
  const PackSeg *segs;
  const PackPiece *pieces;
  int32_t nseg;
  int32_t *status;
  uint64_t timeout_ns;
};

// ---- BF16 tensor-core path ------------------------------------------------
// One task = a 128 x BN tile of a contraction-axis group; its K loop walks the
// group's block pairs, each with its own tensor maps (zero fill past the block
// edge keeps ragged K exact).  At plan time every CTA's tasks are unrolled into
// a flat list of 64-deep K stages, so the copy and MMA threads only walk a list.

struct Bf16Pair {
  int32_t map_a;   // index of the A tensor map (rows of the group x d_k)
  int32_t map_b;   // index of the B tensor map (d_k x cols of the group)
  int32_t klen;    // d_k
  int32_t map_b3[5];   // 3-D B map whose box takes c whole 64-column chunks at once (c = 2..4), -1 if none
};

struct Bf16Task {
  int32_t pair_begin;
  int32_t pair_count;
  int32_t m0;        // first row of the tile inside the group
  int32_t n0;        // first column of the tile inside the group
  int32_t m;         // rows of the group
  int32_t n;         // columns of the group
  int32_t bn;        // UMMA N of the tile (multiple of 16, <= 256)
  int32_t c_vec;     // 1 when every C row of the group starts 16-byte aligned (vector stores)
  int64_t c_off;     // C offset of the group's (0, 0) element
  int64_t ldc;
};

// One K stage: an A box (128 rows x 64 K) and nb B boxes (64 K x 64 columns).
constexpr int kStageFirst = 1;   // first stage of its tile: the accumulator starts from zero
constexpr int kStageLast = 2;    // last stage of its tile: the accumulator is complete afterwards

struct Bf16Stage {
  int32_t map_a;
  int32_t map_b;
  int32_t k0;       // K coordinate of the stage inside the pair's views
  int32_t m0;       // row coordinate of the A box
  int32_t n0;       // column coordinate of the first B box
  int16_t nb;       // B boxes (64 columns each)
  int16_t ksteps;   // K16 MMA steps that reach real K (1..4)
  int16_t bn;       // UMMA N of the tile
  int16_t flags;    // kStageFirst | kStageLast; bits 8-15: B chunks copied by map_b3 (0: none)
  int32_t map_b3;   // 3-D B map taking the tile's first (flags >> 8) chunks in one box
};
static_assert(sizeof(Bf16Stage) == 32, "stage record");

// This CTA's slice of the task and stage lists (both in execution order).
struct Bf16Cta {
  int32_t task_begin, task_count;
  int32_t stage_begin, stage_count;
};

}  // namespace bs

// Plan objects and planner entry points (host).
#pragma once
#include <array>
#include <vector>

#include "bs_host.h"

struct bs_plan;

namespace bs {

struct GroupSet {
  std::vector<Group> groups;
  std::vector<RowSeg> rsegs;
  std::vector<KSeg> ksegs;
  // (i, k, j) triples of each group's first row sector: tptr[g] .. tptr[g+1]
  std::vector<int64_t> tptr;
  std::vector<int32_t> triples;
  // triples of row sectors merged into an existing group: {group, i, k, j}
  std::vector<std::array<int32_t, 4>> extra_triples;
};

struct TileSet {
  std::vector<Task> tasks;
  std::vector<int32_t> tail_elems;   // pairs: group, r << 16 | c
  std::vector<TailDesc> tdesc;       // per group: resolved addressing of single-segment tail groups
  std::vector<int32_t> tq_ptr;       // per-SM queues of tail tasks (LPT-balanced): queue q holds
                                     // tasks tq_ptr[q] .. tq_ptr[q+1]-1 of the tail list
  double executed_flops = 0;
  // the same split by path: tile tasks, tail groups of one view (the unrolled
  // loop), tail groups of several views (the segment walk)
  double exec_tile = 0, exec_tail = 0, exec_general = 0;
  double max_tail_task = 0;   // executed flops of the costliest tail task
  double max_tile_task = 0;   // executed flops of the costliest tile task
  double tile_slots = 0;      // sum over tile tasks of their output slots (lanes)
  int64_t max_tile_slots = 0; // output slots of the costliest tile task
};

// Cost model of one contraction (microseconds).  The defaults are this
// build's measurements on a GB300; bs_calibrate measures them on the running
// device and bs_calibration_apply hands them to the planner.
struct PlanModel {
  double t_launch_us = 2.0;      // each kernel of a contraction after the first
  double t_task_us = 0.0;        // extra fixed cost per task (none measured beyond the terms below)
  double t_segment_us = 0.0;     // extra cost per view segment (likewise)
  double pack_gbs = 3700.0;
  double pack_fixed_us = 8.0;
  double fp64_gflops = 1190.0;   // tile path at long K, useful = executed
  double tile_k0 = 0.0;          // a tile task costs as if its K were K + tile_k0
  double tail_gflops = 1000.0;   // tail path, one view per group, executed flops
  double general_gflops = 500.0; // tail path, several views per group
  double zero_gbs = 3000.0;
  double t_fixed_us = 10.0;      // a contraction whose kernel has almost no work
  double atomic_penalty = 0.5;   // rate factor of tail groups stored with atomics
  double bf16_stage_us = 0.5;
  double bf16_tile_us = 2.8;
  double task_slots = 4096;   // LPT weight of a task's fixed cost, in lane-flop units
  int parallel_ctas = 456;
  int sms = 152;
  bool bucket_pad = false;    // pad single-segment tail groups to power-of-two shapes
  int tail_split_k = 0;       // single-view tail groups of at least this K run each output on two lanes (0: never)
};

// `cmask` (indexed by C block, may be null): only the triples whose C block it
// marks are grouped (a shard of the contraction); null groups every triple.
GroupSet make_contraction_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C, bool merge_rows,
                                 bool atomic, bool unchecked = false, const std::vector<uint8_t> *cmask = nullptr);
GroupSet make_free_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C,
                          const std::vector<uint8_t> *cmask = nullptr);
GroupSet make_triple_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C,
                            const std::vector<uint8_t> *cmask = nullptr);
// C blocks of shard `rank` out of `world`: every populated C block weighted by
// its flops (sum over its triples of d_i d_k d_j), dealt largest first onto
// the least loaded shard (ties: lowest shard), so every rank computes the same
// partition on its own.  Returns a mask over C blocks.
std::vector<uint8_t> shard_mask(const bs_layout &A, const bs_layout &B, const bs_layout &C, int rank, int world);
void group_triples(const GroupSet &gs, std::vector<int64_t> *ptr, std::vector<int32_t> *out);
// With materialize = false only what the cost model reads is produced: the
// tile tasks (unsorted) and the executed flops; the tail list, its
// descriptors and queues are left empty.  The planner costs every candidate
// that way and materializes the chosen one.
void tile_fp64(GroupSet &gs, const PlanModel &pm, TileSet *ts, bool materialize = true);
double model_fp64_us(const GroupSet &gs, const TileSet &ts, const PlanModel &pm, int64_t pack_bytes, int launches,
                     int64_t zero_bytes);

// Forward: the BF16 model reads the plan's per-CTA lists.
double model_bf16_us(const bs_plan &P, const PlanModel &pm);

// Host description of one TMA tensor map of the BF16 path (encoded per call
// with the caller's base pointer, then cached while the pointers stay the same).
struct MapDesc {
  int32_t operand;      // 0: A, 1: B
  int64_t off;          // element offset of the view's first element
  int64_t inner;        // contiguous extent (elements)
  int64_t outer;        // rows
  int64_t ld;           // elements between rows
  int32_t box_inner;
  int32_t box_outer;
  // 0: a 2-D map of the view (inner x outer).  Otherwise a 3-D map of its first
  // `chunks` whole 64-column chunks (64 x outer x chunks, the chunk stride 128
  // bytes), whose box takes box_chunks chunks at once; the view's footprint
  // (inner = 64 * chunks) stays inside the 2-D view's.
  int32_t chunks = 0;
  int32_t box_chunks = 0;
};

}  // namespace bs

struct bs_plan {
  int32_t dtype = BS_F64;
  int32_t shard_rank = 0, shard_world = 1;   // this plan computes shard shard_rank of shard_world
  std::vector<uint8_t> cmask;                // C blocks of the shard (empty: every block)
  bs_plan_options opts{};
  bs_layout A, B, C;
  bs_layout A_pk, B_pk;
  bool pack_a = false, pack_b = false;
  int32_t axis = BS_AXIS_CONTRACTION;
  bs::GroupSet gs;
  bs::TileSet ts;
  std::vector<bs::PackCopy> pack_copies;   // whole-warp copies of A then B, then small copies of A then B
  std::vector<bs::PackSeg> pack_segs;      // the same gather as shared-memory segments (FP64 plans)
  std::vector<bs::PackPiece> pack_pieces;
  bs::PackSplit pack_split{};
  std::vector<bs::ZeroBlock> zero_blocks;
  // BF16 path
  std::vector<bs::Bf16Task> btasks;   // plan order (longest first)
  std::vector<bs::Bf16Pair> bpairs;
  std::vector<bs::Bf16Cta> bctas;     // one per CTA: its slices of bstasks and bstages
  std::vector<bs::Bf16Task> bstasks;  // tasks in execution order, CTA after CTA
  std::vector<bs::Bf16Stage> bstages; // K stages in execution order, CTA after CTA
  std::vector<bs::MapDesc> maps;
  std::vector<unsigned char> map_bytes;   // encoded maps (128 bytes each)
  std::vector<int16_t> sm_map;            // dense SM index per hardware SM identifier (FP64 tail queues)
  const void *maps_a_ptr = nullptr, *maps_b_ptr = nullptr;
  // device state
  int device = -1;
  int sm_count = 0;
  int parallel_ctas = 0;   // resident CTAs the cost model assumed
  int grid = 0;
  void *d_tables = nullptr;
  size_t tables_bytes = 0;
  bs::Task *d_tasks = nullptr;
  bs::Group *d_groups = nullptr;
  bs::RowSeg *d_rsegs = nullptr;
  bs::KSeg *d_ksegs = nullptr;
  int32_t *d_tail = nullptr;
  bs::TailDesc *d_tdesc = nullptr;
  size_t counter_bytes = 256;
  bs::PackCopy *d_pack = nullptr;
  bs::PackSeg *d_segs = nullptr;
  bs::PackPiece *d_pieces = nullptr;
  bs::ZeroBlock *d_zero = nullptr;
  bs::Bf16Cta *d_bctas = nullptr;
  bs::Bf16Task *d_bstasks = nullptr;
  bs::Bf16Stage *d_bstages = nullptr;
  void *d_maps = nullptr;
  void *d_ws_a = nullptr, *d_ws_b = nullptr;
  uint32_t *d_counter = nullptr;
  int counter_parity = 0;   // which counter set the next FP64 launch uses
  int32_t *d_status = nullptr;
  // phase events of bs_contract when profiling: before the gather, after it,
  // after the zero fill, after the grouped kernel
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  bool ev_recorded = false;
  // staging for bs_contract_host
  void *d_host_a = nullptr, *d_host_b = nullptr, *d_host_c = nullptr;
  bs_plan_stats stats{};
};

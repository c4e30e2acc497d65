/*
 * bs.h — C ABI of the coalesced block-sparse contraction library (libbs.so).
 *
 * The library computes C[i,j] = sum_k A[i,k] B[k,j] for block-sparse tensors
 * over symmetry sectors, as described in the uni20 design note "block
 * coalescing" (uni20-dev.github.io, docs/symmetry/block_coalescing):
 *   - Summary: every populated (row, inner, column) sector triple is one small
 *     dense GEMM; the remedy for the many tiny ones is fewer, larger kernels.
 *   - "Why single-axis coalescing is hole-free": groups are formed along one
 *     axis only (free axis: stack the A blocks sharing an inner index k into a
 *     taller GEMM; contraction axis: concatenate the k blocks of one output
 *     block into a wider-K GEMM), so no group contains a structural zero.
 *   - "Expressed as strided views over shared storage": each block is an
 *     (offset, leading dimension) view into one caller-owned buffer, and a
 *     coalesced operand is a wider view of the same bytes.
 *   - "Interleaved vs contiguous": a group whose blocks are not stride
 *     compatible, or not addressable by the tensor-memory copy engine, is
 *     gathered ("packed") into a workspace; a cost model decides per plan.
 *   - "Coalescing is a plan-time transform": bs_plan_create builds the groups,
 *     the task list and the scatter map once; bs_contract only launches.
 *
 * Conventions shared by every entry point:
 *   - Every function returns a bs_status and never throws or aborts.
 *   - Sizes and offsets are in elements of the buffer's type unless stated.
 *   - Handles (bs_layout, bs_plan) are opaque and owned by the library; free
 *     them with the matching *_destroy call.  Destroying NULL is a no-op.
 *   - Device pointers are CUDA device (or managed) addresses on the device
 *     that was current when the plan was created.  Streams are cudaStream_t
 *     passed as void* (NULL = the legacy default stream).
 */
#ifndef BS_H
#define BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bs_status {
  BS_OK = 0,
  BS_ERR_INVALID_ARG = 1,     /* NULL handle/pointer, negative size, bad flag, bad option */
  BS_ERR_SHAPE_MISMATCH = 2,  /* inner axes differ, or a given C layout is not the product */
  BS_ERR_UNSUPPORTED = 3,     /* dtype or device not supported (needs sm_103 / sm_100 family) */
  BS_ERR_OOM = 4,             /* host or device allocation failed */
  BS_ERR_CUDA = 5,            /* a CUDA runtime or driver call failed */
  BS_ERR_TIMEOUT = 6,         /* a bounded device-side wait ran out (reported by the kernel) */
  BS_ERR_MISALIGNED = 7,      /* a buffer or view breaks the 16-byte rule of the chosen path */
  BS_ERR_DEVICE = 8,          /* a device-side consistency check failed */
  BS_ERR_OVERFLOW = 9,        /* an element count or offset does not fit in int64 / int32 */
  BS_ERR_HOLE = 10            /* a coalesced group is not a hole-free view of its blocks */
} bs_status;

/* One sector axis: n sectors, each with a U(1) charge, an optional Z2 parity
 * (q_z2 may be NULL) and a dimension >= 1.  Sector identity is its index;
 * repeated charges are allowed.  Arrays are read during the call only. */
typedef struct bs_axis_desc {
  int32_t n;
  const int32_t *q_u1;
  const uint8_t *q_z2;
  const int32_t *dim;
} bs_axis_desc;

/* Allowed-charge rule of a two-axis tensor: block (r, c) exists iff
 * dq_min <= q_u1[r] - q_u1[c] <= dq_max and, if z2 != 0, q_z2[r] == q_z2[c]
 * (both axes must then carry parities). */
typedef struct bs_rule {
  int32_t dq_min;
  int32_t dq_max;
  int32_t z2;
} bs_rule;

/* Layout flags.  The arrangement (low two bits) is one of:
 *   BLOCKROW : rows in order, then columns in order; each block row-major with
 *              ld = its (rounded) width, stored one after another.
 *   ROWPANEL : one row-major panel per row sector holding that row's blocks
 *              side by side in column order; ld = panel width.  A row's blocks
 *              then form one strided view (the "interleaved" arrangement for
 *              contraction-axis groups).
 *   COLPANEL : one panel per column sector with that column's blocks stacked in
 *              row order; ld = the column's (rounded) width.
 * CHARGE_SORTED orders sectors by (charge, parity, index) instead of index.
 * ALIGN16 rounds every block width up to a multiple of 16 bytes, so every
 * block start and leading dimension is 16-byte aligned (tensor-map rule).
 * ALIGN64 rounds it up to a multiple of 64 bytes instead (and wins over
 * ALIGN16): every row of every block then starts on a 64-byte boundary, which
 * the BF16 kernel's tensor-map copies move markedly faster than rows that
 * start 16 bytes off one.  (FP64 plans do not gain from it: the padding
 * between narrow blocks splits a group's K into more views.) */
enum {
  BS_LAYOUT_BLOCKROW = 0,
  BS_LAYOUT_ROWPANEL = 1,
  BS_LAYOUT_COLPANEL = 2,
  BS_LAYOUT_CHARGE_SORTED = 4,
  BS_LAYOUT_ALIGN16 = 8,
  BS_LAYOUT_ALIGN64 = 16
};

typedef struct bs_layout bs_layout;
typedef struct bs_plan bs_plan;

typedef struct bs_block_info {
  int32_t row;     /* row sector index */
  int32_t col;     /* column sector index */
  int64_t offset;  /* first element of the block in the buffer */
  int32_t rows;    /* = dim of the row sector */
  int32_t cols;    /* = dim of the column sector */
  int64_t ld;      /* elements between consecutive rows of the block */
} bs_block_info;

/* Build the layout of a tensor over (rows x cols) whose populated blocks are
 * those the rule allows (uni20 design note "block coalescing", "Expressed as
 * strided views over shared storage": every block an (offset, leading
 * dimension) view into one buffer; "Interleaved vs contiguous": the
 * arrangement decides which blocks form one wider view).  elem_bytes (2, 4 or 8) matters only for ALIGN16 and ALIGN64.
 * Errors: INVALID_ARG (NULL, n < 0, dim < 1, z2 rule without parities, bad
 * flags or elem_bytes), OVERFLOW (element count beyond int64, or an axis
 * whose dimensions add up to more than INT32_MAX), OOM. */
bs_status bs_layout_create(const bs_axis_desc *rows, const bs_axis_desc *cols, const bs_rule *rule,
                           uint32_t flags, int32_t elem_bytes, bs_layout **out);

/* Number of populated blocks and buffer length in elements (padding included). */
bs_status bs_layout_query(const bs_layout *layout, int64_t *nblocks, int64_t *nelems);

/* Copy the block table, in storage order, into out[0 .. nblocks-1]. */
bs_status bs_layout_blocks(const bs_layout *layout, bs_block_info *out);

void bs_layout_destroy(bs_layout *layout);

typedef enum bs_dtype {
  BS_F64 = 0,      /* A, B, C double; FP64 pipe */
  BS_BF16_F32 = 1  /* A, B bfloat16; C float; FP32 accumulation on the tensor cores */
} bs_dtype;

typedef enum bs_axis_policy {
  BS_AXIS_AUTO = 0,         /* cost model picks contraction or free axis for the plan */
  BS_AXIS_CONTRACTION = 1,  /* one group per C block, K = concatenated inner blocks */
  BS_AXIS_FREE = 2,         /* one group per (k, j): stacked A rows, atomic scatter into C */
  BS_AXIS_NONE = 3          /* one group per (i, k, j) triple: no coalescing (atomic scatter) */
} bs_axis_policy;

typedef enum bs_pack_policy {
  BS_PACK_AUTO = 0,    /* cost model: pack bytes against saved per-segment work */
  BS_PACK_NEVER = 1,   /* zero-copy views only (BF16 path: MISALIGNED if views break TMA rules) */
  BS_PACK_ALWAYS = 2   /* gather A and B into panel workspaces before every contraction */
} bs_pack_policy;

/* Planner options.  Call bs_plan_options_default first, then override. */
typedef struct bs_plan_options {
  int32_t axis_policy;        /* bs_axis_policy */
  int32_t pack_policy;        /* bs_pack_policy */
  uint32_t c_layout_flags;    /* arrangement flags of C (its elem size follows the dtype) */
  int32_t merge_rows;         /* 1: stack row sectors whose groups share structure and
                                 whose A and C rows are stride compatible (LocalSpace keys) */
  int32_t host_only;          /* 1: build the plan on the host only (inspection; no contract) */
  int32_t ctas_per_sm;        /* 0: choose from occupancy */
  /* cost-model constants (microseconds, GB/s, GFLOP/s); <= 0 keeps the built-in value */
  double t_launch_us;         /* fixed cost of one kernel launch on the stream */
  double t_task_us;           /* fixed cost of one task in the persistent kernel */
  double t_segment_us;        /* extra cost of one zero-copy view segment inside a task */
  double pack_gbs;            /* achieved bandwidth of the gather kernel */
  double fp64_gflops;         /* sustained FP64 pipe rate of the grouped kernel */
  double atomic_penalty;      /* rate factor (0..1] of tail groups stored with atomics (free axis, none) */
  int32_t wait_timeout_ms;    /* limit of every device-side wait (BF16 path); <= 0: 2000 ms */
  int32_t debug_flags;        /* testing only, 0 in normal use: BS_DEBUG_WITHHOLD_COPY makes
                                 the BF16 producer skip its first copy so the consumer's bounded
                                 wait runs out and the kernel reports BS_ERR_TIMEOUT;
                                 BS_DEBUG_MERGE_UNCHECKED lets merge_rows stack row sectors
                                 whose inner blocks differ (groups with holes, for testing
                                 bs_plan_check_groups); such a plan must be host_only */
  int32_t bucket_pad;         /* FP64 tail: 0 (default) computes every small group exactly; 1 pads
                                 each single-segment tail group to power-of-two M, N and K so that
                                 groups of one padded shape run as one batched call (uni20 design
                                 note "block coalescing", Open questions: bucketing near-same
                                 shapes by padding); padded rows, columns and K add only zeros */
  int32_t profile;            /* 1: bs_contract records CUDA events around each of its phases (gather,
                                 zero fill, grouped kernel) on the caller's stream; read them with
                                 bs_plan_profile.  0 (default): no events */
  int32_t tail_split_k;       /* FP64 tail: a group of one view whose K reaches this (> 0) runs
                                 each output on two lanes, each summing half of K (halves the
                                 longest tail tasks; measured no faster on the tail workload and
                                 6% slower on the stress workload, so off by default); <= 0: never */
  int32_t reserved[3];
  /* further cost-model constants, also <= 0 for the built-in value (bs_calibration_apply fills
     them from a measurement on the device) */
  double t_fixed_us;          /* event-timed cost of a bs_contract whose kernel has almost no work */
  double fp64_tail_gflops;    /* executed-flop rate of the lane-packed tail path, one view per group */
  double fp64_general_gflops; /* the same for tail groups of several views (segment walk) */
  double pack_fixed_us;       /* fixed cost of the gather launch */
  double zero_gbs;            /* bandwidth of the zero fill that precedes atomic scatter */
  double bf16_stage_us;       /* BF16 kernel: time per 64-deep K stage of a CTA's list */
  double bf16_tile_us;        /* BF16 kernel: time per 128 x 256 output tile (epilogue) */
  double tile_k0;             /* FP64 tile path: a task costs as if its K were K + tile_k0 */
  double reserved2[3];
} bs_plan_options;

enum { BS_DEBUG_WITHHOLD_COPY = 1, BS_DEBUG_MERGE_UNCHECKED = 2 };

void bs_plan_options_default(bs_plan_options *opts);

typedef struct bs_plan_stats {
  int64_t triples;            /* populated (i, k, j) block GEMMs */
  int64_t c_blocks;           /* populated C blocks */
  int64_t groups;             /* coalesced groups (one GEMM each) */
  int64_t tasks;              /* persistent-kernel work items */
  int64_t tile_tasks;         /* CTA-wide tiles */
  int64_t tail_tasks;         /* CTA-sized pieces (256 outputs, one per thread) of the small-group list */
  int64_t segments;           /* zero-copy view segments over all groups */
  int64_t packed_bytes;       /* bytes gathered per contraction (0: zero-copy) */
  int64_t workspace_bytes;    /* device workspace owned by the plan */
  int32_t axis;               /* bs_axis_policy actually used */
  int32_t packed_a;           /* 1 if A is gathered */
  int32_t packed_b;           /* 1 if B is gathered */
  int32_t launches;           /* kernels one bs_contract enqueues */
  double useful_flops;        /* sum over triples of 2 * d_i * d_k * d_j */
  double useful_bytes;        /* populated A + B elements read once, C written once */
  double executed_flops;      /* flops the kernels issue, idle lanes and bucket padding included */
  double model_us;            /* cost-model estimate of one contraction */
  double model_us_alt;        /* estimate for the other axis / pack choice */
  double plan_ms;             /* host time spent in bs_plan_create */
} bs_plan_stats;

/* Build the contraction plan for C = A B (uni20 design note "block
 * coalescing": Summary, the populated triples; "Why single-axis coalescing is
 * hole-free", the contraction-axis and free-axis groups; "The crossover
 * decides whether to coalesce" and "Interleaved vs contiguous", the cost model
 * that picks the axis and whether to gather; "Coalescing is a plan-time
 * transform", all of it done here once).  A's column axis and B's row axis
 * must be identical (same n, charges, parities, dims) or SHAPE_MISMATCH.
 * dtype fixes the element types; elem_bytes of the layouts must match it
 * (8 for F64; 2 for BF16 inputs).  C's layout is built by the plan over
 * (A rows, B cols) with the structural product as its populated set and
 * opts->c_layout_flags as arrangement; get it with bs_plan_c_layout.
 * The plan copies what it needs: A and B layouts may be destroyed afterwards.
 * Device tables and workspaces are allocated here (cudaMalloc) on the current
 * device, unless opts->host_only.  Errors: INVALID_ARG, SHAPE_MISMATCH,
 * UNSUPPORTED, OOM, CUDA, OVERFLOW (a task, tail, segment or copy table longer
 * than the kernels' 32-bit indices reach). */
bs_status bs_plan_create(const bs_layout *A, const bs_layout *B, int32_t dtype,
                         const bs_plan_options *opts, bs_plan **out);

/* The same plan onto a C layout the caller already has (a tensor to write
 * into, another stage's layout): C's row axis must be A's, its column axis
 * B's, and its populated blocks exactly the structural product, else
 * BS_ERR_SHAPE_MISMATCH; its elem_bytes must be 8 for F64 and 4 for BF16_F32
 * (INVALID_ARG otherwise).  The plan keeps its own copy of C's description
 * (opts->c_layout_flags is not used); C may be destroyed afterwards. */
bs_status bs_plan_create_into(const bs_layout *A, const bs_layout *B, const bs_layout *C, int32_t dtype,
                              const bs_plan_options *opts, bs_plan **out);

/* One shard of the contraction for `world` GPUs (or processes), each running
 * its own plan with no exchange of partial results: every populated C block is
 * an independent unit (its value needs no other C block), so the C blocks are
 * dealt largest first by flops onto the least loaded of `world` shards, and
 * the plan of shard `rank` computes exactly its blocks (uni20 design note
 * "block coalescing", "One mechanism, three payoffs": the same groups that
 * cut launches are the units of distribution).  Every rank computes the same
 * partition on its own.  C's layout is the whole structural product, so the
 * shards agree on every offset; a shard writes only its own C blocks and
 * reads only the A and B blocks their triples use (listed by
 * bs_plan_operand_blocks, so a caller whose operands are distributed can
 * gather just those).  The statistics count the shard only.  world = 1 is
 * bs_plan_create.  INVALID_ARG unless 0 <= rank < world. */
bs_status bs_plan_create_shard(const bs_layout *A, const bs_layout *B, int32_t dtype, const bs_plan_options *opts,
                               int32_t rank, int32_t world, bs_plan **out);

/* Blocks of operand 0 (A), 1 (B) or 2 (C) that the plan reads (A, B) or
 * writes (C), as indices into that layout's block table in storage order
 * (bs_layout_blocks; C's layout is bs_plan_c_layout), ascending.  Call with
 * out = NULL for the count in *n. */
bs_status bs_plan_operand_blocks(const bs_plan *plan, int32_t operand, int64_t *n, int32_t *out);

/* C's layout, owned by the plan (valid until bs_plan_destroy). */
const bs_layout *bs_plan_c_layout(const bs_plan *plan);

bs_status bs_plan_stats_get(const bs_plan *plan, bs_plan_stats *out);

/* Phase times of the plan's last bs_contract, for a plan built with
 * opts->profile = 1: milliseconds between CUDA events recorded on the call's
 * stream before and after the gather, the zero fill and the grouped kernel
 * (0 for a phase the plan does not have), and their sum.  Waits for the last
 * event.  INVALID_ARG when the plan does not profile or has not run. */
typedef struct bs_phase_times {
  double gather_ms;
  double zero_ms;
  double kernel_ms;
  double total_ms;
  int64_t gather_bytes;   /* bytes the gather reads plus writes (2 x packed bytes) */
  int64_t reserved[3];
} bs_phase_times;

bs_status bs_plan_profile(bs_plan *plan, bs_phase_times *out);

/* Group table for inspection: for each group g, out[g*8 + 0..7] =
 * {axis (1 contraction, 2 free, 3 none), M, N, K, m_segments, k_segments,
 *  first C block row sector, first C block column sector}.
 * Call with out = NULL to get the count in *ngroups. */
bs_status bs_plan_groups(const bs_plan *plan, int64_t *ngroups, int64_t *out);

/* The FP64 gather's shared-memory segments, for inspection ("Interleaved vs
 * contiguous" of the uni20 note: the pack that makes fragmented operands
 * contiguous).  A plan that gathers at most two segments per SM keeps them and
 * gathers by them; otherwise *nseg is 0 (it gathers block copy by block copy).
 * For segment s, seg_out[5*s .. 5*s+4] = {first source element, source
 * elements it spans (at most 2048), first piece, pieces (at most 128), operand
 * (0 A, 1 B)}, segments of A first, each operand's in source order; for piece
 * p, piece_out[6*p .. 6*p+5] = {first destination element in the operand's
 * panel workspace, first source element counted from its segment's first,
 * rows, cols, source ld, destination ld}.  Pass NULL arrays to get the counts.
 * Host only, reads no device memory. */
bs_status bs_plan_gather_segments(const bs_plan *plan, int64_t *nseg, int64_t *npieces, int64_t *seg_out,
                                  int64_t *piece_out);

/* Triple coverage for inspection: for each group, the (i, k, j) triples it
 * computes, as out[3*t .. 3*t+2], group by group; group_ptr[g] .. group_ptr[g+1]
 * delimit group g.  Pass NULL arrays to get the sizes. */
bs_status bs_plan_triples(const bs_plan *plan, int64_t *ntriples, int64_t *ngroups, int64_t *group_ptr,
                          int32_t *out);

/* Proof that every group is a hole-free view of its blocks (uni20 design note
 * "block coalescing", "Why single-axis coalescing is hole-free", and its
 * LocalSpace keys stacked as a second coalesced axis).  For each group, with
 * the row sectors and inner sectors of its triples taken in order of first
 * appearance: (1) the triples are exactly every (row sector, inner sector)
 * pair, once each, and the sectors' dimensions add up to the group's M and K
 * (and the column sector's to N), so the blocks tile the M x K rectangle with
 * no hole; (2) the group's row and inner segments address each triple's A, B
 * and C blocks exactly where the operand layouts (after any gather) store them:
 * first element and leading dimension.  Host only, reads no device memory.
 * Returns BS_OK, or BS_ERR_HOLE with the first failing group in *bad_group
 * (may be NULL); -1 there when every group passes. */
bs_status bs_plan_check_groups(const bs_plan *plan, int64_t *bad_group);

/* Enqueue C = A B on `stream` and return at once (uni20 design note "block
 * coalescing", Summary: the plain sum over populated triples, run as few
 * large launches instead of one per triple).  A, B, C are device
 * pointers to buffers laid out per the plan's A, B and C layouts; every
 * populated C element is overwritten; padding and absent blocks are not
 * touched.  A, B and C must not overlap.  Work: an optional gather, an optional
 * zero fill of C, one persistent grouped-GEMM kernel.  BF16 plans need A and B
 * 16-byte aligned (MISALIGNED otherwise).  A plan holds one workspace and two
 * sets of work counters that alternate from call to call: do not run the same
 * plan on two streams at once.  A call made while `stream` is being captured
 * into a CUDA graph is recorded so that every replay of the graph gives the
 * same result (its launch returns its counters to zero at exit); a BF16 plan
 * must first have run once, outside the capture, with the same A and B
 * pointers (a change of operand pointers re-encodes the tensor maps with a
 * host synchronisation, so inside a capture such a call returns UNSUPPORTED
 * before it enqueues anything and the capture stays valid).  Errors found on the device are reported by
 * bs_plan_last_device_error. */
bs_status bs_contract(bs_plan *plan, const void *A, const void *B, void *C, void *stream);

/* bs_contract with every access checked against the caller's buffer sizes
 * (a debugging aid, slower than bs_contract).  nA, nB and nC are the elements
 * the A, B and C buffers hold.  Before anything is enqueued the host checks
 * the views the gather reads, the C blocks the zero fill writes and, for a
 * BF16 plan, every tensor map's view and every output tile against them, and
 * returns BS_ERR_DEVICE on the first that does not fit.  An FP64 plan then
 * runs a checked instance of its kernel: every load of A or B and every store
 * of C is tested against the counts first; an access outside is skipped (a
 * load reads zero) and the kernel records a bounds violation, which
 * bs_plan_last_device_error reports as BS_ERR_DEVICE.  No access ever leaves
 * the buffers, and a plan whose layouts fit its buffers trips nothing.
 * INVALID_ARG for negative counts, otherwise as bs_contract. */
bs_status bs_contract_checked(bs_plan *plan, const void *A, int64_t nA, const void *B, int64_t nB, void *C,
                              int64_t nC, void *stream);

/* The same contraction on HOST buffers: copies A and B to plan-owned device
 * buffers (allocated on first use), contracts into C_host (which must hold the
 * C layout's element count) and synchronizes the stream before returning.
 * When A_host and B_host are both 16-byte aligned pinned host memory the
 * device can address (cudaHostAlloc, cudaHostRegister), one copy kernel pulls
 * them in; otherwise each goes through the copy engine.  When C_host is pinned
 * host memory the device can address, the plan writes each C element once (no
 * zero fill) and C is either at most 4 MiB or written at no more than 50 GB/s
 * over the plan's modelled kernel time (stats.model_us), the kernel stores C
 * straight into C_host: every populated element is written and the rest of
 * C_host is left unchanged.  Otherwise the whole C buffer is copied back and its padding and
 * absent blocks arrive as zeros.  Pinned host memory gives the fastest calls.
 * On a stream that is being captured into a graph the call returns
 * UNSUPPORTED before it enqueues anything (it has to wait for its copies). */
bs_status bs_contract_host(bs_plan *plan, const void *A_host, const void *B_host, void *C_host,
                           void *stream);

/* The uncoalesced control: zero the whole C buffer (padding included), then
 * one kernel launch per populated (i, k, j) triple on `stream`, each adding
 * A[i,k] B[k,j] into C[i,j] with a plain one-output-per-thread kernel.  It is
 * the one-launch-per-block baseline that coalescing is measured against
 * (design note "block coalescing", Summary: tiny GEMMs are launch-bound). */
bs_status bs_contract_uncoalesced(bs_plan *plan, const void *A, const void *B, void *C, void *stream);

/* The FP64 contraction without any device allocation.  The design note has no
 * counterpart to this call; it exists for callers that cannot call cudaMalloc
 * (code running under a memory manager that owns all device memory, or a
 * steady-state loop that must not allocate after start-up).  It does what
 * bs_contract does, but the task tables, work counters and gather workspace
 * live in one fixed device array of BS_NOALLOC_SCRATCH_BYTES inside the
 * library (held on every device that loads the library until the process
 * exits), so the plan may be built with host_only = 1 and nothing is allocated
 * on the device, by this call or by the plan.  Each call copies the plan's
 * tables into the array and zeroes its counters, on `stream`.
 *   - FP64 plans only (UNSUPPORTED otherwise).
 *   - A plan whose tables and workspace exceed the array returns OVERFLOW
 *     before anything is enqueued.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture begins.
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race; order them on one stream.
 *   - The tables are copied from the plan's host memory (ordinary pageable
 *     memory), so a call may wait for earlier work on `stream` before it
 *     returns, and the plan must stay alive until the call's work is done.
 *   - A host_only plan built while a device is current is dealt for that
 *     device's SM count; the grid is the one bs_contract would launch.
 *   - The FP64 kernel has no device waits, so there is no device status to read. */
#define BS_NOALLOC_SCRATCH_BYTES (16u << 20)
bs_status bs_contract_noalloc(const bs_plan *plan, const void *A, const void *B, void *C, void *stream);

/* Synchronize `stream`, read and clear the plan's device status word.
 * Returns BS_OK, or the error a kernel recorded (TIMEOUT, DEVICE, ...). */
bs_status bs_plan_last_device_error(bs_plan *plan, void *stream);

void bs_plan_destroy(bs_plan *plan);

const char *bs_status_string(bs_status status);

/* Cost-model constants measured on the current device.  The design note
 * "block coalescing" ("The crossover decides whether to coalesce") takes its
 * launch cost and flop rate from calibrated constants that the pages do not
 * print; this call measures them with small probe kernels on `stream`
 * (allocating and freeing about 2 GiB of scratch) and synchronizes. */
typedef struct bs_calibration {
  double fp64_gflops;               /* FP64 FMA rate, every lane of every warp active (best probe shape) */
  double fp64_gflops_quarter_warp;  /* the same with 8 of 32 lanes active (useful flops) */
  double launch_us;                 /* back-to-back empty-kernel launch interval */
  double copy_gbs;                  /* device copy bandwidth, read + write bytes */
  int32_t sm_count;
  int32_t sm_id_bound;              /* 1 + the largest hardware SM identifier in use (> sm_count when
                                       the identifiers skip values) */
  double fp64_sm_mhz;               /* SM clock during the best FMA probe (cycle / global-time stamps) */
  double fp64_flop_per_clk_sm;      /* FMA flops per SM clock at that rate */
  double fp64_dmma_gflops;          /* FP64 matrix instruction (mma.sync m8n8k4) rate */
  double dmma_flop_per_clk_sm;      /* its flops per SM clock */
  /* cost-model constants, measured by running the library's own kernels on
   * small synthetic structures (L2 flushed before every run, medians): */
  double t_fixed_us;                /* bs_contract of a one-triple plan, event to event */
  double tile_gflops;               /* tile path at long K (one dense 1536^3 FP64 group) */
  double tail_gflops;               /* tail path, one view per group: executed flops / time */
  double general_gflops;            /* tail path, several views per group */
  double pack_gbs;                  /* gather kernel: 2 x packed bytes / time */
  double pack_fixed_us;             /* gather kernel: time of a small gather */
  double zero_gbs;                  /* zero fill: bytes / time */
  double bf16_stage_us;             /* BF16 kernel: time per K stage, from one long dense group */
  double bf16_tile_us;              /* BF16 kernel: time per output tile, from many short groups */
  double tile_k0;                   /* tile path: extra K steps a task costs (from a short-K group) */
  double atomic_factor;             /* tail path: rate of atomically stored groups relative to plain ones */
  double reserved[5];
} bs_calibration;

/* Copy the cost-model constants of a calibration into planner options. */
void bs_calibration_apply(const bs_calibration *cal, bs_plan_options *opts);

bs_status bs_calibrate(bs_calibration *out, void *stream);

/* Library build identification, e.g. "bs 0.1 sm_103a". */
const char *bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BS_H */

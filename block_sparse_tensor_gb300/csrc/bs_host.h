// Host-side objects behind the opaque handles of bs.h.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/bs.h"
#include "bs_internal.h"

namespace bs {

struct AxisCopy {
  int32_t n = 0;
  std::vector<int32_t> q;
  std::vector<uint8_t> p;   // empty when the axis has no parity
  std::vector<int32_t> d;
  bool same_as(const AxisCopy &o) const { return n == o.n && q == o.q && p == o.p && d == o.d; }
};

// Populated set given as rows of sorted column indices (CSR).
struct Sparsity {
  std::vector<int64_t> ptr;   // n_rows + 1
  std::vector<int32_t> cols;  // ascending within a row
};

}  // namespace bs

struct bs_layout {
  bs::AxisCopy rows, cols;
  uint32_t flags = 0;
  int32_t elem_bytes = 8;
  int64_t nelems = 0;
  std::vector<bs_block_info> blocks;   // storage order
  // CSR by row sector over blocks: row_ptr[r] .. row_ptr[r+1] index row_blk,
  // listing the row's blocks in storage order; csc likewise by column.
  std::vector<int64_t> row_ptr, col_ptr;
  std::vector<int32_t> row_blk, col_blk;
  // dense (row, col) -> block index when the grid is small enough, else empty
  std::vector<int32_t> grid;
  int32_t find(int32_t r, int32_t c) const;
};

namespace bs {

bs_status build_layout(const AxisCopy &rows, const AxisCopy &cols, const Sparsity &sp, uint32_t flags,
                       int32_t elem_bytes, bs_layout *out);
bs_status copy_axis(const bs_axis_desc *d, AxisCopy *out);
Sparsity rule_sparsity(const AxisCopy &r, const AxisCopy &c, const bs_rule &rule);

// Launchers (bs_fp64.cu, bs_bf16.cu, bs_stage.cu).
cudaError_t launch_fp64_grouped(const Fp64Params &p, int grid, cudaStream_t s);
// The gather of both operands in one launch, eight CTAs per SM of `sms`.
cudaError_t launch_pack2(const PackParams &a, const PackParams &b, const PackSplit &split, int sms, cudaStream_t s);
// The FP64 gather by segments (every base pointer 16-byte aligned), one CTA
// per SM of `sms`.
cudaError_t launch_seg_gather(const SegParams &p, int sms, cudaStream_t s);
cudaError_t launch_zero(void *C, int elem_bytes, const ZeroBlock *blocks, int nblocks, int grid,
                        cudaStream_t s);
// Copies n0 bytes src0 -> dst0 and n1 bytes src1 -> dst1 in one launch; every pointer 16-byte aligned.
cudaError_t launch_stage_in(const void *src0, void *dst0, size_t n0, const void *src1, void *dst1, size_t n1, int sms,
                            cudaStream_t s);
cudaError_t launch_control_fp64(const double *A, const double *B, double *C, int64_t a_off, int64_t lda,
                                int64_t b_off, int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k,
                                cudaStream_t s);
cudaError_t launch_control_bf16(const uint16_t *A, const uint16_t *B, float *C, int64_t a_off, int64_t lda,
                                int64_t b_off, int64_t ldb, int64_t c_off, int64_t ldc, int m, int n, int k,
                                cudaStream_t s);
// Dense SM index per hardware SM identifier (-1: not seen), found once per
// device by a short probe launch on `s` (into dev_buf, or a temporary
// allocation when it is NULL; dev_buf needs sm_probe_bytes(sm_count) bytes).
size_t sm_probe_bytes(int sm_count);
bs_status sm_index_map(int device, int sm_count, void *dev_buf, cudaStream_t s, std::vector<int16_t> *out);
// Queue bounds and SM map of the FP64 tail, copied into the kernel parameters.
inline void fill_queue_params(Fp64Params *p, const std::vector<int32_t> &tq_ptr, const std::vector<int16_t> &sm_map) {
  p->nq = tq_ptr.size() > 1 ? (int32_t)tq_ptr.size() - 1 : 0;
  for (int q = 0; q <= kMaxQueues; ++q) p->qptr[q] = q < (int)tq_ptr.size() ? tq_ptr[q] : 0;
  p->nsm_ids = sm_map.size() <= (size_t)kMaxSmIds ? (int32_t)sm_map.size() : 0;
  for (int i = 0; i < kMaxSmIds; ++i) p->sm_queue[i] = i < p->nsm_ids ? sm_map[i] : (int16_t)-1;
}
// Resident CTAs per SM of the FP64 kernel instance a plan with (false) or
// without (true) tile tasks launches.
int fp64_max_ctas_per_sm(bool tail_only);

struct Bf16Params {
  const void *maps;          // CUtensorMap array in device memory (64-byte aligned)
  const Bf16Cta *ctas;       // CTA b runs tasks[ctas[b].task_begin ..] and stages[ctas[b].stage_begin ..]
  const Bf16Task *tasks;     // per-CTA task lists, concatenated in execution order
  const Bf16Stage *stages;   // per-CTA stage lists, concatenated in execution order
  float *C;
  int32_t *status;
  uint32_t *counter;
  uint64_t timeout_ns;
  int32_t debug_flags;
  int32_t pad_;
};
cudaError_t launch_bf16_grouped(const Bf16Params &p, int grid, cudaStream_t s);
size_t bf16_smem_bytes();

}  // namespace bs

// C ABI entry points (include/bs.h): argument checks, plan construction,
// device tables, and the launches that make up one contraction.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <future>
#include <map>
#include <new>
#include <system_error>
#include <tuple>

#include "bs_plan.h"

using namespace bs;

namespace {

bs_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BS_OK;
  if (e == cudaErrorMemoryAllocation) return BS_ERR_OOM;
  return BS_ERR_CUDA;
}

#define BS_CUDA(call)                                        \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_status(e_);           \
  } while (0)

// Host allocation fault injection for tests: with BS_FAULT_INJECT=alloc in the
// environment, the allocations of layout and plan construction fail (as if the
// host were out of memory), so the error path and its clean-up can be
// exercised without exhausting anything.  Nothing on the device is involved.
bool alloc_fault_injected() {
  const char *v = std::getenv("BS_FAULT_INJECT");
  return v && std::strstr(v, "alloc") != nullptr;
}

Sparsity sparsity_of(const bs_layout &L) {
  Sparsity sp;
  sp.ptr.assign(L.rows.n + 1, 0);
  for (int32_t r = 0; r < L.rows.n; ++r) {
    std::vector<int32_t> cs;
    for (int64_t t = L.row_ptr[r]; t < L.row_ptr[r + 1]; ++t) cs.push_back(L.blocks[L.row_blk[t]].col);
    std::sort(cs.begin(), cs.end());
    sp.cols.insert(sp.cols.end(), cs.begin(), cs.end());
    sp.ptr[r + 1] = (int64_t)sp.cols.size();
  }
  return sp;
}

// Populated C blocks: (i, j) with some k holding A[i,k] and B[k,j].
Sparsity product_sparsity(const bs_layout &A, const bs_layout &B) {
  Sparsity sp;
  const int32_t ni = A.rows.n, nj = B.cols.n;
  sp.ptr.assign(ni + 1, 0);
  std::vector<uint8_t> seen(nj, 0);
  std::vector<int32_t> row;
  for (int32_t i = 0; i < ni; ++i) {
    row.clear();
    for (int64_t t = A.row_ptr[i]; t < A.row_ptr[i + 1]; ++t) {
      const int32_t k = A.blocks[A.row_blk[t]].col;
      for (int64_t u = B.row_ptr[k]; u < B.row_ptr[k + 1]; ++u) {
        const int32_t j = B.blocks[B.row_blk[u]].col;
        if (!seen[j]) {
          seen[j] = 1;
          row.push_back(j);
        }
      }
    }
    std::sort(row.begin(), row.end());
    for (int32_t j : row) seen[j] = 0;
    sp.cols.insert(sp.cols.end(), row.begin(), row.end());
    sp.ptr[i + 1] = (int64_t)sp.cols.size();
  }
  return sp;
}

int64_t populated_elems(const bs_layout &L) {
  int64_t s = 0;
  for (const auto &b : L.blocks) s += (int64_t)b.rows * b.cols;
  return s;
}

// Block copies of the gather, split into row bands of at most 2048 elements
// so one huge block does not serialise the launch on a few warps.  Copies of
// doubles are listed in destination order, so that the warps that take them
// in turn write neighbouring pieces of a panel row close together in time
// (their partial sectors meet in L2); copies of 2-byte elements largest
// first, for equal shares.  Copies of at most kPackSmallElems elements go to
// `small` (moved four to a warp).
void pack_list(const bs_layout &src, const bs_layout &dst, int elem_bytes, std::vector<PackCopy> *big,
               std::vector<PackCopy> *small) {
  std::vector<PackCopy> all;
  for (const auto &b : src.blocks) {
    const auto &d = dst.blocks[dst.find(b.row, b.col)];
    const int32_t band = std::max<int32_t>(1, 2048 / b.cols);
    for (int32_t r0 = 0; r0 < b.rows; r0 += band) {
      PackCopy c{};
      c.src = b.offset + (int64_t)r0 * b.ld;
      c.src_ld = b.ld;
      c.dst = d.offset + (int64_t)r0 * d.ld;
      c.dst_ld = d.ld;
      c.rows = std::min(band, b.rows - r0);
      c.cols = b.cols;
      all.push_back(c);
    }
  }
  if (elem_bytes == 8)
    std::stable_sort(all.begin(), all.end(), [](const PackCopy &x, const PackCopy &y) { return x.dst < y.dst; });
  else
    std::stable_sort(all.begin(), all.end(), [](const PackCopy &x, const PackCopy &y) {
      return (int64_t)x.rows * x.cols > (int64_t)y.rows * y.cols;
    });
  for (const auto &c : all) ((int64_t)c.rows * c.cols <= kPackSmallElems ? small : big)->push_back(c);
}

// The same gather as shared-memory segments: every block of the source
// layout becomes pieces (bands of rows spanning at most kSegElems source
// elements, or row chunks of at most kSegElems columns when one row is
// longer), and pieces taken in source order fill segments while the span from
// the segment's first element to the end of its last piece stays within
// kSegElems and it holds at most kSegPieces of them.
void seg_list(const bs_layout &src, const bs_layout &dst, int32_t operand, std::vector<PackSeg> *segs,
              std::vector<PackPiece> *pieces) {
  struct Placed {
    int64_t src;   // first source element
    PackPiece p;
  };
  std::vector<Placed> ps;
  for (const auto &b : src.blocks) {
    const auto &d = dst.blocks[dst.find(b.row, b.col)];
    if (b.cols > kSegElems) {
      for (int32_t r = 0; r < b.rows; ++r)
        for (int32_t c0 = 0; c0 < b.cols; c0 += kSegElems) {
          PackPiece p{};
          p.dst = d.offset + (int64_t)r * d.ld + c0;
          p.rows = 1;
          p.cols = std::min(kSegElems, b.cols - c0);
          p.src_ld = p.dst_ld = p.cols;
          ps.push_back({b.offset + (int64_t)r * b.ld + c0, p});
        }
      continue;
    }
    // h rows span (h - 1) ld + cols <= kSegElems source elements
    const int32_t h = (int32_t)std::max<int64_t>(1, std::min<int64_t>(b.rows, (kSegElems - b.cols) / b.ld + 1));
    for (int32_t r0 = 0; r0 < b.rows; r0 += h) {
      PackPiece p{};
      p.dst = d.offset + (int64_t)r0 * d.ld;
      p.rows = std::min(h, b.rows - r0);
      p.cols = b.cols;
      p.src_ld = (int32_t)b.ld;
      p.dst_ld = (int32_t)d.ld;
      ps.push_back({b.offset + (int64_t)r0 * b.ld, p});
    }
  }
  std::stable_sort(ps.begin(), ps.end(), [](const Placed &x, const Placed &y) { return x.src < y.src; });
  for (size_t i = 0; i < ps.size();) {
    PackSeg s{};
    s.src = ps[i].src;
    s.piece_begin = (int32_t)pieces->size();
    s.operand = operand;
    int64_t end = s.src;
    size_t j = i;
    for (; j < ps.size() && j - i < (size_t)kSegPieces; ++j) {
      const int64_t qend = ps[j].src + (int64_t)(ps[j].p.rows - 1) * ps[j].p.src_ld + ps[j].p.cols;
      if (j > i && qend - s.src > kSegElems) break;
      PackPiece p = ps[j].p;
      p.src_off = (int32_t)(ps[j].src - s.src);
      pieces->push_back(p);
      end = std::max(end, qend);
    }
    s.n = (int32_t)(end - s.src);
    s.piece_count = (int32_t)(j - i);
    segs->push_back(s);
    i = j;
  }
}

void zero_list(const bs_layout &C, const std::vector<uint8_t> *cmask, std::vector<ZeroBlock> *out) {
  for (size_t t = 0; t < C.blocks.size(); ++t) {
    if (cmask && !(*cmask)[t]) continue;   // another shard's C block
    const auto &b = C.blocks[t];
    const int32_t band = std::max<int32_t>(1, 16384 / b.cols);
    for (int32_t r0 = 0; r0 < b.rows; r0 += band)
      out->push_back({b.offset + (int64_t)r0 * b.ld, b.ld, std::min(band, b.rows - r0), b.cols});
  }
}

bool tma_ok(int64_t off, int64_t ld, int eb) { return (off * eb) % 16 == 0 && (ld * eb) % 16 == 0; }

bool groups_tma_ok(const GroupSet &gs) {
  for (const auto &s : gs.ksegs)
    if (!tma_ok(s.ka, s.kl, 2) || !tma_ok(s.kb, s.ldb, 2)) return false;
  return true;
}

template <class T>
size_t append_bytes(std::vector<unsigned char> &buf, const std::vector<T> &v) {
  size_t off = (buf.size() + 255) / 256 * 256;
  buf.resize(off + v.size() * sizeof(T));
  if (!v.empty()) std::memcpy(buf.data() + off, v.data(), v.size() * sizeof(T));
  return off;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

bs_status encode_maps(bs_plan *P, const void *A, const void *B) {
  auto enc = get_encode();
  if (!enc) return BS_ERR_CUDA;
  P->map_bytes.assign(P->maps.size() * sizeof(CUtensorMap), 0);
  for (size_t t = 0; t < P->maps.size(); ++t) {
    const MapDesc &m = P->maps[t];
    const int eb = 2;
    const char *base = (const char *)(m.operand == 0 ? A : B) + m.off * eb;
    const bool three = m.chunks > 0;
    // 3-D: (64 columns of a chunk, rows, chunks 128 bytes apart)
    cuuint64_t dims[3] = {(cuuint64_t)(three ? 64 : m.inner), (cuuint64_t)m.outer, (cuuint64_t)m.chunks};
    cuuint64_t strides[2] = {(cuuint64_t)(m.ld * eb), (cuuint64_t)(64 * eb)};
    cuuint32_t box[3] = {(cuuint32_t)m.box_inner, (cuuint32_t)m.box_outer, (cuuint32_t)m.box_chunks};
    cuuint32_t es[3] = {1, 1, 1};
    CUtensorMap *out = (CUtensorMap *)(P->map_bytes.data() + t * sizeof(CUtensorMap));
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, three ? 3 : 2, (void *)base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return BS_ERR_MISALIGNED;
  }
  return BS_OK;
}

// BF16 tasks: 128-row tiles of each contraction-axis group, one tensor-map
// pair per inner segment.
void build_bf16(bs_plan *P) {
  const GroupSet &gs = P->gs;
  std::map<std::tuple<int, int64_t, int64_t, int64_t, int64_t, int, int, int, int>, int32_t> seen;
  auto map_id = [&](int op, int64_t off, int64_t inner, int64_t outer, int64_t ld, int bi, int bo, int chunks = 0,
                    int box_chunks = 0) {
    // the box is part of a map: the same view with another box is another map
    auto key = std::make_tuple(op, off, inner, outer, ld, bi, bo, chunks, box_chunks);
    auto it = seen.find(key);
    if (it != seen.end()) return it->second;
    MapDesc m{op, off, inner, outer, ld, bi, bo};
    m.chunks = chunks;
    m.box_chunks = box_chunks;
    P->maps.push_back(m);
    int32_t id = (int32_t)P->maps.size() - 1;
    seen[key] = id;
    return id;
  };
  std::vector<std::pair<double, Bf16Task>> costed;
  for (const auto &g : gs.groups) {
    const RowSeg &rs = gs.rsegs[g.rseg_begin];
    const int32_t pb = (int32_t)P->bpairs.size();
    for (int32_t s = 0; s < g.kseg_count; ++s) {
      const KSeg &k = gs.ksegs[g.kseg_begin + s];
      Bf16Pair pr{};
      pr.map_a = map_id(0, k.ka, k.klen, g.m, k.kl, 64, 128);
      pr.map_b = map_id(1, k.kb, g.n, k.klen, k.ldb, 64, 64);
      // a tile's whole 64-column chunks of B go in one 3-D box (one copy
      // instruction instead of one per chunk); a ragged last chunk keeps its
      // 2-D box, which stops at the view's edge
      const int32_t whole = g.n / 64;
      for (int c = 0; c <= 4; ++c) pr.map_b3[c] = -1;
      for (int32_t n0 = 0; n0 < g.n; n0 += 256) {
        const int32_t nfull = std::min<int32_t>(4, std::max<int32_t>(0, (g.n - n0) / 64));
        if (nfull >= 2 && pr.map_b3[nfull] < 0)
          pr.map_b3[nfull] = map_id(1, k.kb, 64 * (int64_t)whole, k.klen, k.ldb, 64, 64, whole, nfull);
      }
      pr.klen = k.klen;
      P->bpairs.push_back(pr);
    }
    // 128-row tiles, up to 256 columns wide
    for (int32_t m0 = 0; m0 < g.m; m0 += 128)
      for (int32_t n0 = 0; n0 < g.n; n0 += 256) {
        Bf16Task t{};
        t.pair_begin = pb;
        t.pair_count = g.kseg_count;
        t.m0 = m0;
        t.n0 = n0;
        t.m = g.m;
        t.n = g.n;
        t.bn = (std::min(256, g.n - n0) + 15) / 16 * 16;
        t.c_off = rs.rc;
        t.ldc = rs.ldc;
        t.c_vec = tma_ok(rs.rc, rs.ldc, 4) ? 1 : 0;   // 16-byte aligned rows: vector stores
        int64_t kch = 0;
        for (int32_t s = 0; s < g.kseg_count; ++s) kch += (gs.ksegs[g.kseg_begin + s].klen + 63) / 64;
        costed.push_back({(double)kch * (t.bn + 64), t});
      }
  }
  std::stable_sort(costed.begin(), costed.end(),
                   [](const std::pair<double, Bf16Task> &a, const std::pair<double, Bf16Task> &b) { return a.first > b.first; });
  for (auto &c : costed) P->btasks.push_back(c.second);
  // One CTA per SM; each task goes, longest first, to the CTA with the least
  // modelled work.  A stage costs a fixed handoff plus MMA time growing with BN.
  const int ncta = std::max(1, std::min<int>((int)P->btasks.size(), P->sm_count > 0 ? P->sm_count : 152));
  std::vector<std::vector<int32_t>> lists(ncta);
  std::vector<std::pair<double, int>> heap;
  for (int c = 0; c < ncta; ++c) heap.push_back({0.0, c});
  auto cmp = [](const std::pair<double, int> &a, const std::pair<double, int> &b) { return a.first > b.first; };
  for (size_t t = 0; t < P->btasks.size(); ++t) {
    const Bf16Task &T = P->btasks[t];
    int64_t st = 0;
    for (int32_t q = 0; q < T.pair_count; ++q) st += (P->bpairs[T.pair_begin + q].klen + 63) / 64;
    std::pop_heap(heap.begin(), heap.end(), cmp);
    heap.back().first += 150.0 + (double)st * (96.0 + T.bn);
    lists[heap.back().second].push_back((int32_t)t);
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  // Unroll every CTA's list into tasks and 64-deep K stages, in execution order.
  P->bctas.assign(ncta, Bf16Cta{});
  for (int c = 0; c < ncta; ++c) {
    Bf16Cta &cd = P->bctas[c];
    cd.task_begin = (int32_t)P->bstasks.size();
    cd.stage_begin = (int32_t)P->bstages.size();
    for (int32_t t : lists[c]) {
      const Bf16Task &T = P->btasks[t];
      P->bstasks.push_back(T);
      const size_t first = P->bstages.size();
      for (int32_t q = 0; q < T.pair_count; ++q) {
        const Bf16Pair &pr = P->bpairs[T.pair_begin + q];
        for (int32_t k0 = 0; k0 < pr.klen; k0 += 64) {
          Bf16Stage e{};
          e.map_a = pr.map_a;
          e.map_b = pr.map_b;
          e.k0 = k0;
          e.m0 = T.m0;
          e.n0 = T.n0;
          e.nb = (int16_t)((T.bn + 63) / 64);
          const int32_t nfull = std::min<int32_t>(e.nb, std::max<int32_t>(0, (T.n - T.n0) / 64));
          if (nfull >= 2 && pr.map_b3[nfull] >= 0) {
            e.map_b3 = pr.map_b3[nfull];
            e.flags = (int16_t)(nfull << 8);
          }
          e.ksteps = (int16_t)std::min(4, (pr.klen - k0 + 15) / 16);
          e.bn = (int16_t)T.bn;
          P->bstages.push_back(e);
        }
      }
      P->bstages[first].flags |= kStageFirst;
      P->bstages.back().flags |= kStageLast;
    }
    cd.task_count = (int32_t)P->bstasks.size() - cd.task_begin;
    cd.stage_count = (int32_t)P->bstages.size() - cd.stage_begin;
  }
}

bs_status upload(bs_plan *P) {
  std::vector<unsigned char> buf;
  size_t o_tasks = append_bytes(buf, P->ts.tasks);
  size_t o_groups = append_bytes(buf, P->gs.groups);
  size_t o_rsegs = append_bytes(buf, P->gs.rsegs);
  size_t o_ksegs = append_bytes(buf, P->gs.ksegs);
  size_t o_tail = append_bytes(buf, P->ts.tail_elems);
  size_t o_tdesc = append_bytes(buf, P->ts.tdesc);
  size_t o_pack = append_bytes(buf, P->pack_copies);
  size_t o_segs = append_bytes(buf, P->pack_segs);
  size_t o_pieces = append_bytes(buf, P->pack_pieces);
  size_t o_zero = append_bytes(buf, P->zero_blocks);
  size_t o_bc = append_bytes(buf, P->bctas);
  size_t o_bt = append_bytes(buf, P->bstasks);
  size_t o_bs = append_bytes(buf, P->bstages);
  std::vector<unsigned char> mapspace(P->maps.size() * sizeof(CUtensorMap), 0);
  size_t o_maps = append_bytes(buf, mapspace);
  size_t total = (buf.size() + 255) / 256 * 256 + 256;
  buf.resize(total, 0);
  BS_CUDA(cudaMalloc(&P->d_tables, total));
  P->tables_bytes = total;
  BS_CUDA(cudaMemcpy(P->d_tables, buf.data(), total, cudaMemcpyHostToDevice));
  char *b = (char *)P->d_tables;
  P->d_tasks = (Task *)(b + o_tasks);
  P->d_groups = (Group *)(b + o_groups);
  P->d_rsegs = (RowSeg *)(b + o_rsegs);
  P->d_ksegs = (KSeg *)(b + o_ksegs);
  P->d_tail = (int32_t *)(b + o_tail);
  P->d_tdesc = (TailDesc *)(b + o_tdesc);
  P->d_pack = (PackCopy *)(b + o_pack);
  P->d_segs = (PackSeg *)(b + o_segs);
  P->d_pieces = (PackPiece *)(b + o_pieces);
  P->d_zero = (ZeroBlock *)(b + o_zero);
  P->d_bctas = (Bf16Cta *)(b + o_bc);
  P->d_bstasks = (Bf16Task *)(b + o_bt);
  P->d_bstages = (Bf16Stage *)(b + o_bs);
  P->d_maps = (void *)(b + o_maps);
  // status word and the two counter sets (initialised once the grid is known)
  void *cs = nullptr;
  P->counter_bytes = counter_bytes((int)std::max<size_t>(1, P->ts.tq_ptr.size()) - 1);
  BS_CUDA(cudaMalloc(&cs, P->counter_bytes));
  BS_CUDA(cudaMemset(cs, 0, P->counter_bytes));
  P->d_counter = (uint32_t *)cs;
  P->d_status = (int32_t *)((char *)cs + 128);
  const int eb = P->dtype == BS_F64 ? 8 : 2;
  if (P->pack_a) BS_CUDA(cudaMalloc(&P->d_ws_a, std::max<int64_t>(P->A_pk.nelems, 1) * eb));
  if (P->pack_b) BS_CUDA(cudaMalloc(&P->d_ws_b, std::max<int64_t>(P->B_pk.nelems, 1) * eb));
  P->stats.workspace_bytes = (int64_t)total + 256 + (P->pack_a ? P->A_pk.nelems * eb : 0) +
                             (P->pack_b ? P->B_pk.nelems * eb : 0);
  return BS_OK;
}

// Both counter sets and the status word of a plan back to zero; the next
// launch uses set 0.
bs_status init_counters(bs_plan *P) {
  if (!P->d_counter) return BS_OK;
  BS_CUDA(cudaMemset(P->d_counter, 0, P->counter_bytes));
  P->counter_parity = 0;
  return BS_OK;
}

void free_device(bs_plan *P) {
  for (auto &e : P->ev)
    if (e) {
      cudaEventDestroy(e);
      e = nullptr;
    }
  cudaFree(P->d_tables);
  cudaFree(P->d_counter);
  cudaFree(P->d_ws_a);
  cudaFree(P->d_ws_b);
  cudaFree(P->d_host_a);
  cudaFree(P->d_host_b);
  cudaFree(P->d_host_c);
  P->d_tables = P->d_ws_a = P->d_ws_b = P->d_host_a = P->d_host_b = P->d_host_c = nullptr;
  P->d_counter = nullptr;
}

struct Candidate {
  int axis;
  bool pack;
  double us;
};

}  // namespace

static bs_status contract_kernel(bs_plan *P, const void *Ause, const void *Buse, void *C, cudaStream_t s,
                                 const int64_t *sizes);
static bs_status contract_impl(bs_plan *P, const void *A, const void *B, void *C, void *stream, const int64_t *sizes);

extern "C" {

const char *bs_status_string(bs_status s) {
  switch (s) {
    case BS_OK: return "ok";
    case BS_ERR_INVALID_ARG: return "invalid argument";
    case BS_ERR_SHAPE_MISMATCH: return "shape mismatch";
    case BS_ERR_UNSUPPORTED: return "unsupported";
    case BS_ERR_OOM: return "out of memory";
    case BS_ERR_CUDA: return "CUDA error";
    case BS_ERR_TIMEOUT: return "device wait timed out";
    case BS_ERR_MISALIGNED: return "misaligned buffer or view";
    case BS_ERR_DEVICE: return "device-side check failed";
    case BS_ERR_OVERFLOW: return "size overflow";
    case BS_ERR_HOLE: return "group is not a hole-free view of its blocks";
  }
  return "unknown status";
}

const char *bs_version(void) { return "bs 0.1 sm_103a"; }

bs_status bs_layout_create(const bs_axis_desc *rows, const bs_axis_desc *cols, const bs_rule *rule, uint32_t flags,
                           int32_t elem_bytes, bs_layout **out) {
  if (!out) return BS_ERR_INVALID_ARG;
  *out = nullptr;
  if (!rows || !cols || !rule) return BS_ERR_INVALID_ARG;
  if (rule->dq_min > rule->dq_max) return BS_ERR_INVALID_ARG;
  bs_layout *L = new (std::nothrow) bs_layout();
  if (!L) return BS_ERR_OOM;
  if (alloc_fault_injected()) {
    delete L;
    return BS_ERR_OOM;
  }
  AxisCopy r, c;
  bs_status st = copy_axis(rows, &r);
  if (st == BS_OK) st = copy_axis(cols, &c);
  if (st == BS_OK && rule->z2 && (r.p.empty() || c.p.empty())) st = BS_ERR_INVALID_ARG;
  if (st == BS_OK) {
    try {
      st = build_layout(r, c, rule_sparsity(r, c, *rule), flags, elem_bytes, L);
    } catch (const std::bad_alloc &) {
      st = BS_ERR_OOM;
    }
  }
  if (st != BS_OK) {
    delete L;
    return st;
  }
  *out = L;
  return BS_OK;
}

bs_status bs_layout_query(const bs_layout *L, int64_t *nblocks, int64_t *nelems) {
  if (!L) return BS_ERR_INVALID_ARG;
  if (nblocks) *nblocks = (int64_t)L->blocks.size();
  if (nelems) *nelems = L->nelems;
  return BS_OK;
}

bs_status bs_layout_blocks(const bs_layout *L, bs_block_info *out) {
  if (!L || (!out && !L->blocks.empty())) return BS_ERR_INVALID_ARG;
  if (!L->blocks.empty()) std::memcpy(out, L->blocks.data(), L->blocks.size() * sizeof(bs_block_info));
  return BS_OK;
}

void bs_layout_destroy(bs_layout *L) { delete L; }

void bs_plan_options_default(bs_plan_options *o) {
  if (!o) return;
  std::memset(o, 0, sizeof *o);
  o->axis_policy = BS_AXIS_AUTO;
  o->pack_policy = BS_PACK_AUTO;
  o->c_layout_flags = BS_LAYOUT_BLOCKROW;
  o->merge_rows = 1;
}

static bs_status plan_create(const bs_layout *A, const bs_layout *B, const bs_layout *Cg, int32_t dtype,
                             const bs_plan_options *opts, bs_plan **out, int32_t rank = 0, int32_t world = 1) {
  if (!out) return BS_ERR_INVALID_ARG;
  *out = nullptr;
  if (!A || !B) return BS_ERR_INVALID_ARG;
  if (world < 1 || rank < 0 || rank >= world) return BS_ERR_INVALID_ARG;
  if (dtype != BS_F64 && dtype != BS_BF16_F32) return BS_ERR_INVALID_ARG;
  bs_plan_options o;
  bs_plan_options_default(&o);
  if (opts) o = *opts;
  if (o.axis_policy < 0 || o.axis_policy > 3 || o.pack_policy < 0 || o.pack_policy > 2) return BS_ERR_INVALID_ARG;
  if ((o.c_layout_flags & ~31u) || (o.c_layout_flags & 3u) == 3u) return BS_ERR_INVALID_ARG;
  const int eb_in = dtype == BS_F64 ? 8 : 2;
  if (A->elem_bytes != eb_in || B->elem_bytes != eb_in) return BS_ERR_INVALID_ARG;
  if (!A->cols.same_as(B->rows)) return BS_ERR_SHAPE_MISMATCH;
  if (dtype == BS_BF16_F32 && (o.axis_policy == BS_AXIS_FREE || o.axis_policy == BS_AXIS_NONE))
    return BS_ERR_UNSUPPORTED;
  // groups with holes are for testing the validator only: such a plan never runs
  const bool unchecked = (o.debug_flags & BS_DEBUG_MERGE_UNCHECKED) != 0;
  if (unchecked && !o.host_only) return BS_ERR_INVALID_ARG;
  const auto t0 = std::chrono::steady_clock::now();
  bs_plan *P = new (std::nothrow) bs_plan();
  if (!P) return BS_ERR_OOM;
  bs_status st = BS_OK;
  try {
    P->dtype = dtype;
    P->opts = o;
    if (alloc_fault_injected()) throw std::bad_alloc();   // taken by the OOM path below
    P->A = *A;
    P->B = *B;
    if (Cg) {
      // a caller's C layout: the same axes, the element size of the dtype's
      // output and exactly the structural product as its populated set
      st = BS_OK;
      if (!Cg->rows.same_as(A->rows) || !Cg->cols.same_as(B->cols)) st = BS_ERR_SHAPE_MISMATCH;
      else if (Cg->elem_bytes != (dtype == BS_F64 ? 8 : 4)) st = BS_ERR_INVALID_ARG;
      else {
        const Sparsity sp = product_sparsity(*A, *B);
        if ((size_t)sp.ptr.back() != Cg->blocks.size()) st = BS_ERR_SHAPE_MISMATCH;
        std::vector<int32_t> cols;
        for (int32_t r = 0; st == BS_OK && r < Cg->rows.n; ++r) {
          cols.clear();
          for (int64_t t = Cg->row_ptr[r]; t < Cg->row_ptr[r + 1]; ++t) cols.push_back(Cg->blocks[Cg->row_blk[t]].col);
          std::sort(cols.begin(), cols.end());
          if (!std::equal(cols.begin(), cols.end(), sp.cols.begin() + sp.ptr[r], sp.cols.begin() + sp.ptr[r + 1]) ||
              (int64_t)cols.size() != sp.ptr[r + 1] - sp.ptr[r])
            st = BS_ERR_SHAPE_MISMATCH;
        }
      }
      if (st == BS_OK) P->C = *Cg;
    } else {
      st = build_layout(A->rows, B->cols, product_sparsity(*A, *B), o.c_layout_flags, dtype == BS_F64 ? 8 : 4, &P->C);
    }
    if (st != BS_OK) {
      delete P;
      return st;
    }
    // a shard computes only its C blocks; C's layout stays the whole product
    if (world > 1) {
      P->cmask = shard_mask(*A, *B, P->C, rank, world);
      P->shard_rank = rank;
      P->shard_world = world;
    }
    const std::vector<uint8_t> *cm = world > 1 ? &P->cmask : nullptr;
    PlanModel pm;
    if (o.t_launch_us > 0) pm.t_launch_us = o.t_launch_us;
    if (o.t_task_us > 0) pm.t_task_us = o.t_task_us;
    if (o.t_segment_us > 0) pm.t_segment_us = o.t_segment_us;
    if (o.pack_gbs > 0) pm.pack_gbs = o.pack_gbs;
    if (o.fp64_gflops > 0) pm.fp64_gflops = o.fp64_gflops;
    if (o.atomic_penalty > 0) pm.atomic_penalty = o.atomic_penalty;
    if (o.t_fixed_us > 0) pm.t_fixed_us = o.t_fixed_us;
    if (o.fp64_tail_gflops > 0) pm.tail_gflops = o.fp64_tail_gflops;
    if (o.fp64_general_gflops > 0) pm.general_gflops = o.fp64_general_gflops;
    if (o.pack_fixed_us > 0) pm.pack_fixed_us = o.pack_fixed_us;
    if (o.zero_gbs > 0) pm.zero_gbs = o.zero_gbs;
    if (o.bf16_stage_us > 0) pm.bf16_stage_us = o.bf16_stage_us;
    if (o.bf16_tile_us > 0) pm.bf16_tile_us = o.bf16_tile_us;
    if (o.tile_k0 > 0) pm.tile_k0 = o.tile_k0;
    if (o.bucket_pad < 0 || o.bucket_pad > 1 || o.profile < 0 || o.profile > 1) {
      delete P;
      return BS_ERR_INVALID_ARG;
    }
    pm.bucket_pad = o.bucket_pad == 1;
    pm.tail_split_k = o.tail_split_k > 0 ? o.tail_split_k : 0;
    if (!o.host_only) {
      int dev = 0, major = 0, minor = 0;
      if (cudaGetDevice(&dev) != cudaSuccess) {
        delete P;
        return BS_ERR_CUDA;
      }
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (major != 10 || minor != 3) {
        delete P;
        return BS_ERR_UNSUPPORTED;
      }
      P->device = dev;
      cudaDeviceGetAttribute(&P->sm_count, cudaDevAttrMultiProcessorCount, dev);
    } else {
      // a host-only plan follows the current device when there is one (so the
      // allocation-free entry point launches the grid the plan was dealt for),
      // else a 152-SM part
      int dev = 0, sms = 0;
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
        P->sm_count = sms;
        P->device = dev;
      } else {
        (void)cudaGetLastError();
        P->sm_count = 152;
      }
    }
    const int cps = o.ctas_per_sm > 0 ? o.ctas_per_sm
                    : (o.host_only && P->device < 0) ? 3
                                                      : std::max(1, fp64_max_ctas_per_sm(false));
    pm.parallel_ctas = P->sm_count * cps;
    P->parallel_ctas = pm.parallel_ctas;
    pm.sms = P->sm_count;

    const bool sorted_pack = true;
    auto packed = [&](const bs_layout &src, uint32_t mode, bs_layout *dst) {
      uint32_t f = mode | (sorted_pack ? BS_LAYOUT_CHARGE_SORTED : 0) | (dtype == BS_BF16_F32 ? BS_LAYOUT_ALIGN64 : 0);
      return build_layout(src.rows, src.cols, sparsity_of(src), f, src.elem_bytes, dst);
    };

    if (dtype == BS_F64) {
      std::vector<int> axes;
      if (o.axis_policy == BS_AXIS_AUTO) axes = {BS_AXIS_CONTRACTION, BS_AXIS_FREE};
      else axes = {o.axis_policy};
      std::vector<bool> packs;
      if (o.pack_policy == BS_PACK_AUTO) packs = {false, true};
      else packs = {o.pack_policy == BS_PACK_ALWAYS};
      std::vector<Candidate> cands;
      double best = 1e300;
      int best_axis = -1;
      bool best_pack = false;
      // Every (axis, pack) candidate is built and costed on its own thread;
      // the cheapest in this order wins, the first of equals.
      struct Built {
        int ax = 0;
        bool pk = false;
        bs_status st = BS_OK;
        bs_layout Apk, Bpk;
        GroupSet gs;
        TileSet ts;
        double us = 0, ms_group = 0, ms_tile = 0;
      };
      std::vector<Built> built;
      for (int ax : axes)
        for (bool pk : packs) {
          if (pk && ax == BS_AXIS_NONE) continue;
          built.emplace_back();
          built.back().ax = ax;
          built.back().pk = pk;
        }
      const bool only = built.size() == 1;   // a single candidate is the plan
      auto build_one = [&](Built &c) {
        const int ax = c.ax;
        const bool pk = c.pk;
        const bs_layout *Ae = &P->A, *Be = &P->B;
        int64_t pbytes = 0;
        if (pk) {
          c.st = packed(P->A, ax == BS_AXIS_FREE ? BS_LAYOUT_COLPANEL : BS_LAYOUT_ROWPANEL, &c.Apk);
          if (c.st != BS_OK) return;
          Ae = &c.Apk;
          pbytes += populated_elems(P->A) * eb_in;
          if (ax == BS_AXIS_CONTRACTION) {
            c.st = packed(P->B, BS_LAYOUT_COLPANEL, &c.Bpk);
            if (c.st != BS_OK) return;
            Be = &c.Bpk;
            pbytes += populated_elems(P->B) * eb_in;
          }
        }
        const auto tg0 = std::chrono::steady_clock::now();
        c.gs = ax == BS_AXIS_CONTRACTION ? make_contraction_groups(*Ae, *Be, P->C, o.merge_rows != 0, false, unchecked, cm)
               : ax == BS_AXIS_FREE      ? make_free_groups(*Ae, *Be, P->C, cm)
                                         : make_triple_groups(*Ae, *Be, P->C, cm);
        const auto tg1 = std::chrono::steady_clock::now();
        tile_fp64(c.gs, pm, &c.ts, only);
        const auto tg2 = std::chrono::steady_clock::now();
        const bool atomic = ax != BS_AXIS_CONTRACTION;
        const int launches = 1 + (pk ? 1 : 0) + (atomic ? 1 : 0);
        int64_t zbytes = 0;   // C blocks of this plan, zero-filled before atomic scatter
        if (atomic)
          for (size_t t = 0; t < P->C.blocks.size(); ++t)
            if (!cm || P->cmask[t]) zbytes += (int64_t)P->C.blocks[t].rows * P->C.blocks[t].cols * 8;
        c.us = model_fp64_us(c.gs, c.ts, pm, pbytes, launches, zbytes);
        c.ms_group = std::chrono::duration<double, std::milli>(tg1 - tg0).count();
        c.ms_tile = std::chrono::duration<double, std::milli>(tg2 - tg1).count();
      };
      if (only) {
        build_one(built[0]);
      } else {
        std::vector<std::future<void>> running;
        size_t started = 0;
        try {
          for (auto &c : built) {
            running.push_back(std::async(std::launch::async, build_one, std::ref(c)));
            ++started;
          }
        } catch (const std::system_error &) {
          // no thread to be had: the remaining candidates are built here
        }
        for (auto &f : running) f.get();
        for (size_t c = started; c < built.size(); ++c) build_one(built[c]);
      }
      for (auto &c : built) {
        if (c.st != BS_OK) {
          st = c.st;
          break;
        }
        if (std::getenv("BS_LOG"))
          std::fprintf(stderr,
                       "[bs] candidate axis=%d pack=%d groups=%zu tasks=%zu model=%.1f us (group %.1f ms, tile %.1f ms) "
                       "executed tile %.4g tail %.4g general %.4g, costliest tile task %.4g tail task %.4g\n",
                       c.ax, (int)c.pk, c.gs.groups.size(), c.ts.tasks.size(), c.us, c.ms_group, c.ms_tile,
                       c.ts.exec_tile, c.ts.exec_tail, c.ts.exec_general, c.ts.max_tile_task, c.ts.max_tail_task);
        cands.push_back({c.ax, c.pk, c.us});
        if (c.us < best) {
          best = c.us;
          best_axis = c.ax;
          best_pack = c.pk;
          P->gs = std::move(c.gs);
          P->ts = std::move(c.ts);
          P->pack_a = c.pk;
          P->pack_b = c.pk && c.ax == BS_AXIS_CONTRACTION;
          if (c.pk) P->A_pk = c.Apk;
          if (P->pack_b) P->B_pk = c.Bpk;
        }
      }
      if (st != BS_OK) {
        delete P;
        return st;
      }
      std::vector<Built>().swap(built);   // the losing candidates go before the winner is listed in full
      if (!only) tile_fp64(P->gs, pm, &P->ts, true);   // the chosen candidate in full
      P->axis = best_axis;
      P->stats.model_us = best;
      double alt = 0;
      for (const auto &c : cands)
        if (!(c.axis == best_axis && c.pack == best_pack)) alt = alt == 0 ? c.us : std::min(alt, c.us);
      P->stats.model_us_alt = alt;
      (void)best_pack;
    } else {
      // BF16: contraction axis; views must satisfy the tensor-map rules, else gather
      GroupSet gs = make_contraction_groups(P->A, P->B, P->C, o.merge_rows != 0, false, unchecked, cm);
      bool need_pack = !groups_tma_ok(gs) || o.pack_policy == BS_PACK_ALWAYS;
      if (need_pack && o.pack_policy == BS_PACK_NEVER) {
        delete P;
        return BS_ERR_MISALIGNED;
      }
      if (need_pack) {
        st = packed(P->A, BS_LAYOUT_ROWPANEL, &P->A_pk);
        if (st == BS_OK) st = packed(P->B, BS_LAYOUT_COLPANEL, &P->B_pk);
        if (st != BS_OK) {
          delete P;
          return st;
        }
        P->pack_a = P->pack_b = true;
        gs = make_contraction_groups(P->A_pk, P->B_pk, P->C, o.merge_rows != 0, false, unchecked, cm);
      }
      P->gs = std::move(gs);
      P->axis = BS_AXIS_CONTRACTION;
      build_bf16(P);
    }
    {
      std::vector<PackCopy> big_a, small_a, big_b, small_b;
      const int eb = P->dtype == BS_F64 ? 8 : 2;
      if (P->pack_a) pack_list(P->A, P->A_pk, eb, &big_a, &small_a);
      if (P->pack_b) pack_list(P->B, P->B_pk, eb, &big_b, &small_b);
      auto &pc = P->pack_copies;
      pc.clear();
      for (const auto *v : {&big_a, &big_b, &small_a, &small_b}) pc.insert(pc.end(), v->begin(), v->end());
      P->pack_split.big_a = (int32_t)std::min<size_t>(big_a.size(), INT32_MAX);
      P->pack_split.big = (int32_t)std::min<size_t>(big_a.size() + big_b.size(), INT32_MAX);
      P->pack_split.small_a = (int32_t)std::min<size_t>(big_a.size() + big_b.size() + small_a.size(), INT32_MAX);
      P->pack_split.total = (int32_t)std::min<size_t>(pc.size(), INT32_MAX);
    }
    if (dtype == BS_F64) {
      if (P->pack_a) seg_list(P->A, P->A_pk, 0, &P->pack_segs, &P->pack_pieces);
      if (P->pack_b) seg_list(P->B, P->B_pk, 1, &P->pack_segs, &P->pack_pieces);
      // only a small gather goes by segments (measured on block-row gathers of
      // stress-like workloads: faster up to 1.2 segments per SM, slower from 3.3)
      if (P->pack_segs.size() > (size_t)std::max(1, P->sm_count) * kSegMaxPerSm) {
        P->pack_segs.clear();
        P->pack_pieces.clear();
      }
    }
    {
      // every table the kernels index with 32 bits
      const size_t lim = (size_t)(INT32_MAX - kThreads);
      if (P->ts.tail_elems.size() / 2 > lim || P->ts.tasks.size() > lim || P->gs.groups.size() > lim ||
          P->gs.rsegs.size() > lim || P->gs.ksegs.size() > lim || P->pack_copies.size() > lim ||
          P->pack_segs.size() > lim || P->pack_pieces.size() > lim ||
          P->btasks.size() > lim || P->bstages.size() > lim) {
        delete P;
        return BS_ERR_OVERFLOW;
      }
    }
    bool any_atomic = false;
    for (const auto &g : P->gs.groups) any_atomic |= (g.flags & GF_ATOMIC) != 0;
    if (any_atomic) zero_list(P->C, cm, &P->zero_blocks);

    // statistics
    bs_plan_stats &S = P->stats;
    std::vector<int64_t> tp;
    std::vector<int32_t> tr;
    group_triples(P->gs, &tp, &tr);
    S.triples = (int64_t)tr.size() / 3;
    double fl = 0;
    for (size_t t = 0; t < tr.size(); t += 3)
      fl += 2.0 * A->rows.d[tr[t]] * A->cols.d[tr[t + 1]] * B->cols.d[tr[t + 2]];
    S.useful_flops = fl;
    S.c_blocks = cm ? (int64_t)std::count(P->cmask.begin(), P->cmask.end(), (uint8_t)1) : (int64_t)P->C.blocks.size();
    S.groups = (int64_t)P->gs.groups.size();
    int64_t nseg = 0;
    for (const auto &g : P->gs.groups) nseg += std::max(g.kseg_count, g.rseg_count);
    S.segments = nseg;
    S.axis = P->axis;
    S.packed_a = P->pack_a;
    S.packed_b = P->pack_b;
    S.packed_bytes = (P->pack_a ? populated_elems(P->A) * eb_in : 0) + (P->pack_b ? populated_elems(P->B) * eb_in : 0);
    const int eb_out = dtype == BS_F64 ? 8 : 4;
    if (!cm) {
      S.useful_bytes = (double)(populated_elems(P->A) + populated_elems(P->B)) * eb_in + (double)populated_elems(P->C) * eb_out;
    } else {   // the blocks this shard reads and writes
      std::vector<uint8_t> ua(P->A.blocks.size(), 0), ub(P->B.blocks.size(), 0);
      double by = 0;
      for (size_t t = 0; t < tr.size(); t += 3) {
        const int32_t a = P->A.find(tr[t], tr[t + 1]), b = P->B.find(tr[t + 1], tr[t + 2]);
        if (!ua[a]) by += (double)P->A.blocks[a].rows * P->A.blocks[a].cols * eb_in;
        if (!ub[b]) by += (double)P->B.blocks[b].rows * P->B.blocks[b].cols * eb_in;
        ua[a] = ub[b] = 1;
      }
      for (size_t t = 0; t < P->C.blocks.size(); ++t)
        if (P->cmask[t]) by += (double)P->C.blocks[t].rows * P->C.blocks[t].cols * eb_out;
      S.useful_bytes = by;
    }
    if (dtype == BS_F64) {
      S.tile_tasks = (int64_t)P->ts.tasks.size();
      S.tail_tasks = (int64_t)(P->ts.tail_elems.size() / 2 + kThreads - 1) / kThreads;   // CTA-sized pieces of the tail list
      S.tasks = S.tile_tasks + S.tail_tasks;
      S.executed_flops = P->ts.executed_flops;
    } else {
      S.tasks = S.tile_tasks = (int64_t)P->btasks.size();
      double ex = 0;
      for (const auto &t : P->btasks) {
        int64_t kk = 0;
        for (int32_t s = 0; s < t.pair_count; ++s) kk += (P->bpairs[t.pair_begin + s].klen + 15) / 16 * 16;
        ex += 2.0 * 128 * t.bn * kk;
      }
      S.executed_flops = ex;
    }
    S.launches = 1 + ((P->pack_a || P->pack_b) ? 1 : 0) + (P->zero_blocks.empty() ? 0 : 1);
    if (dtype == BS_BF16_F32) S.model_us = model_bf16_us(*P, pm);

    if (!o.host_only) {
      if (dtype == BS_F64 && P->ts.tq_ptr.size() > 1) {
        st = sm_index_map(P->device, P->sm_count, nullptr, 0, &P->sm_map);
        if (st != BS_OK) {
          delete P;
          return st;
        }
      }
      st = upload(P);
      if (st != BS_OK) {
        free_device(P);
        delete P;
        return st;
      }
      if (dtype == BS_F64) {
        const int64_t work_items = (int64_t)P->ts.tasks.size() + (int64_t)(P->ts.tail_elems.size() / 2 + kThreads - 1) / kThreads;
        const int launch_cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : fp64_max_ctas_per_sm(P->ts.tasks.empty());
        P->grid = (int)std::max<int64_t>(1, std::min<int64_t>(work_items, (int64_t)P->sm_count * launch_cps));
      }
      else P->grid = std::max(1, (int)P->bctas.size());
      st = init_counters(P);
      if (st != BS_OK) {
        free_device(P);
        delete P;
        return st;
      }
    }
  } catch (const std::bad_alloc &) {
    free_device(P);
    delete P;
    return BS_ERR_OOM;
  }
  P->stats.plan_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  *out = P;
  return BS_OK;
}

bs_status bs_plan_create(const bs_layout *A, const bs_layout *B, int32_t dtype, const bs_plan_options *opts,
                         bs_plan **out) {
  return plan_create(A, B, nullptr, dtype, opts, out);
}

void bs_calibration_apply(const bs_calibration *c, bs_plan_options *o) {
  if (!c || !o) return;
  auto set = [](double v, double *dst) {
    if (v > 0) *dst = v;
  };
  set(c->t_fixed_us, &o->t_fixed_us);
  set(c->launch_us, &o->t_launch_us);
  set(c->tile_gflops, &o->fp64_gflops);
  set(c->tail_gflops, &o->fp64_tail_gflops);
  set(c->general_gflops, &o->fp64_general_gflops);
  set(c->pack_gbs, &o->pack_gbs);
  set(c->pack_fixed_us, &o->pack_fixed_us);
  set(c->zero_gbs, &o->zero_gbs);
  set(c->bf16_stage_us, &o->bf16_stage_us);
  set(c->bf16_tile_us, &o->bf16_tile_us);
  set(c->tile_k0, &o->tile_k0);
  set(c->atomic_factor, &o->atomic_penalty);
}

bs_status bs_plan_create_shard(const bs_layout *A, const bs_layout *B, int32_t dtype, const bs_plan_options *opts,
                               int32_t rank, int32_t world, bs_plan **out) {
  return plan_create(A, B, nullptr, dtype, opts, out, rank, world);
}

bs_status bs_plan_operand_blocks(const bs_plan *P, int32_t operand, int64_t *n, int32_t *out) {
  if (!P || !n || operand < 0 || operand > 2) return BS_ERR_INVALID_ARG;
  const bs_layout &L = operand == 0 ? P->A : operand == 1 ? P->B : P->C;
  std::vector<uint8_t> used(L.blocks.size(), 0);
  std::vector<int64_t> tp;
  std::vector<int32_t> tr;
  group_triples(P->gs, &tp, &tr);
  for (size_t t = 0; t < tr.size(); t += 3) {
    const int32_t r = operand == 1 ? tr[t + 1] : tr[t];
    const int32_t c = operand == 0 ? tr[t + 1] : tr[t + 2];
    used[L.find(r, c)] = 1;
  }
  int64_t cnt = 0;
  for (size_t b = 0; b < used.size(); ++b)
    if (used[b]) {
      if (out) out[cnt] = (int32_t)b;
      ++cnt;
    }
  *n = cnt;
  return BS_OK;
}

bs_status bs_plan_create_into(const bs_layout *A, const bs_layout *B, const bs_layout *C, int32_t dtype,
                              const bs_plan_options *opts, bs_plan **out) {
  if (!C) {
    if (out) *out = nullptr;
    return BS_ERR_INVALID_ARG;
  }
  return plan_create(A, B, C, dtype, opts, out);
}

const bs_layout *bs_plan_c_layout(const bs_plan *P) { return P ? &P->C : nullptr; }

bs_status bs_plan_stats_get(const bs_plan *P, bs_plan_stats *out) {
  if (!P || !out) return BS_ERR_INVALID_ARG;
  *out = P->stats;
  return BS_OK;
}

bs_status bs_plan_groups(const bs_plan *P, int64_t *ngroups, int64_t *out) {
  if (!P || !ngroups) return BS_ERR_INVALID_ARG;
  *ngroups = (int64_t)P->gs.groups.size();
  if (!out) return BS_OK;
  std::vector<int64_t> tp;
  std::vector<int32_t> tr;
  group_triples(P->gs, &tp, &tr);
  for (size_t g = 0; g < P->gs.groups.size(); ++g) {
    const Group &G = P->gs.groups[g];
    int64_t *o = out + 8 * g;
    o[0] = P->axis == BS_AXIS_AUTO ? BS_AXIS_CONTRACTION : P->axis;
    o[1] = G.m;
    o[2] = G.n;
    o[3] = G.k;
    o[4] = G.rseg_count;
    o[5] = G.kseg_count;
    o[6] = tp[g] < tp[g + 1] ? tr[3 * tp[g]] : -1;
    o[7] = tp[g] < tp[g + 1] ? tr[3 * tp[g] + 2] : -1;
  }
  return BS_OK;
}

bs_status bs_plan_gather_segments(const bs_plan *P, int64_t *nseg, int64_t *npieces, int64_t *seg_out,
                                  int64_t *piece_out) {
  if (!P || !nseg || !npieces) return BS_ERR_INVALID_ARG;
  *nseg = (int64_t)P->pack_segs.size();
  *npieces = (int64_t)P->pack_pieces.size();
  if (seg_out)
    for (size_t s = 0; s < P->pack_segs.size(); ++s) {
      const PackSeg &g = P->pack_segs[s];
      int64_t *o = seg_out + 5 * s;
      o[0] = g.src;
      o[1] = g.n;
      o[2] = g.piece_begin;
      o[3] = g.piece_count;
      o[4] = g.operand;
    }
  if (piece_out)
    for (size_t p = 0; p < P->pack_pieces.size(); ++p) {
      const PackPiece &c = P->pack_pieces[p];
      int64_t *o = piece_out + 6 * p;
      o[0] = c.dst;
      o[1] = c.src_off;
      o[2] = c.rows;
      o[3] = c.cols;
      o[4] = c.src_ld;
      o[5] = c.dst_ld;
    }
  return BS_OK;
}

bs_status bs_plan_triples(const bs_plan *P, int64_t *ntriples, int64_t *ngroups, int64_t *group_ptr, int32_t *out) {
  if (!P || !ntriples || !ngroups) return BS_ERR_INVALID_ARG;
  std::vector<int64_t> tp;
  std::vector<int32_t> tr;
  group_triples(P->gs, &tp, &tr);
  *ntriples = (int64_t)tr.size() / 3;
  *ngroups = (int64_t)P->gs.groups.size();
  if (group_ptr) std::memcpy(group_ptr, tp.data(), tp.size() * sizeof(int64_t));
  if (out && !tr.empty()) std::memcpy(out, tr.data(), tr.size() * sizeof(int32_t));
  return BS_OK;
}

bs_status bs_plan_check_groups(const bs_plan *P, int64_t *bad_group) {
  if (!P) return BS_ERR_INVALID_ARG;
  if (bad_group) *bad_group = -1;
  // the layouts the kernels read
  const bs_layout &A = P->pack_a ? P->A_pk : P->A;
  const bs_layout &B = P->pack_b ? P->B_pk : P->B;
  const bs_layout &C = P->C;
  std::vector<int64_t> tp;
  std::vector<int32_t> tr;
  group_triples(P->gs, &tp, &tr);
  std::vector<int32_t> rows, ks;
  std::vector<int64_t> roff, koff;
  for (size_t g = 0; g < P->gs.groups.size(); ++g) {
    const Group &G = P->gs.groups[g];
    bool ok = tp[g + 1] > tp[g];
    // row sectors and inner sectors in order of first appearance, with offsets
    rows.clear();
    ks.clear();
    int32_t jcol = ok ? tr[3 * tp[g] + 2] : -1;
    for (int64_t t = tp[g]; ok && t < tp[g + 1]; ++t) {
      const int32_t i = tr[3 * t], k = tr[3 * t + 1], j = tr[3 * t + 2];
      ok = j == jcol;
      if (std::find(rows.begin(), rows.end(), i) == rows.end()) rows.push_back(i);
      if (std::find(ks.begin(), ks.end(), k) == ks.end()) ks.push_back(k);
    }
    int64_t msum = 0, ksum = 0;
    roff.assign(rows.size(), 0);
    koff.assign(ks.size(), 0);
    for (size_t a = 0; a < rows.size(); ++a) {
      roff[a] = msum;
      msum += A.rows.d[rows[a]];
    }
    for (size_t b = 0; b < ks.size(); ++b) {
      koff[b] = ksum;
      ksum += A.cols.d[ks[b]];
    }
    // (1) the triples tile the M x K rectangle: every pair, once
    ok = ok && msum == G.m && ksum == G.k && B.cols.d[jcol] == G.n &&
         tp[g + 1] - tp[g] == (int64_t)rows.size() * (int64_t)ks.size();
    if (ok) {
      std::vector<char> seen(rows.size() * ks.size(), 0);
      for (int64_t t = tp[g]; ok && t < tp[g + 1]; ++t) {
        const size_t a = std::find(rows.begin(), rows.end(), tr[3 * t]) - rows.begin();
        const size_t b = std::find(ks.begin(), ks.end(), tr[3 * t + 1]) - ks.begin();
        ok = !seen[a * ks.size() + b];
        seen[a * ks.size() + b] = 1;
      }
    }
    // (2) the views address every block where its layout stores it
    const RowSeg *rs = P->gs.rsegs.data() + G.rseg_begin;
    const KSeg *kg = P->gs.ksegs.data() + G.kseg_begin;
    auto rseg_of = [&](int64_t r) -> const RowSeg * {
      for (int32_t q = 0; q < G.rseg_count; ++q)
        if (r >= rs[q].r0 && r < rs[q].r0 + rs[q].rows) return rs + q;
      return nullptr;
    };
    auto kseg_of = [&](int64_t kk) -> const KSeg * {
      for (int32_t q = 0; q < G.kseg_count; ++q)
        if (kk >= kg[q].k0 && kk < kg[q].k0 + kg[q].klen) return kg + q;
      return nullptr;
    };
    // A(r, kk) = A[RA + KA + RL * KL], B(kk, c) = B[KB + c], C(r, c) = C[RC + c]
    auto a_addr = [&](int64_t r, int64_t kk, int64_t *out) {
      const RowSeg *s = rseg_of(r);
      const KSeg *q = kseg_of(kk);
      if (!s || !q) return false;
      const int64_t lr = r - s->r0;
      *out = s->ra + lr * s->lda + q->ka + (kk - q->k0) + (s->rl ? lr : 0) * q->kl;
      return true;
    };
    for (int64_t t = tp[g]; ok && t < tp[g + 1]; ++t) {
      const int32_t i = tr[3 * t], k = tr[3 * t + 1];
      const int64_t r = roff[std::find(rows.begin(), rows.end(), i) - rows.begin()];
      const int64_t kk = koff[std::find(ks.begin(), ks.end(), k) - ks.begin()];
      const int32_t ba = A.find(i, k), bb = B.find(k, jcol), bc = C.find(i, jcol);
      if (ba < 0 || bb < 0 || bc < 0) {
        ok = false;
        break;
      }
      const bs_block_info &ia = A.blocks[ba], &ib = B.blocks[bb], &ic = C.blocks[bc];
      int64_t x0 = 0, x1 = 0;
      ok = a_addr(r, kk, &x0) && x0 == ia.offset;
      if (ok && ia.rows > 1) ok = a_addr(r + 1, kk, &x1) && x1 - x0 == ia.ld;
      if (ok && ia.cols > 1) ok = a_addr(r, kk + ia.cols - 1, &x1) && x1 - x0 == ia.cols - 1;
      const KSeg *q = kseg_of(kk);
      ok = ok && q && q->kb + (kk - q->k0) * q->ldb == ib.offset && (ib.rows == 1 || q->ldb == ib.ld);
      if (ok && ib.rows > 1) {
        const KSeg *q2 = kseg_of(kk + ib.rows - 1);
        ok = q2 == q;
      }
      const RowSeg *s = rseg_of(r);
      ok = ok && s && s->rc + (r - s->r0) * s->ldc == ic.offset && (ic.rows == 1 || s->ldc == ic.ld);
      if (ok && ic.rows > 1) ok = rseg_of(r + ic.rows - 1) == s;
    }
    if (!ok) {
      if (bad_group) *bad_group = (int64_t)g;
      return BS_ERR_HOLE;
    }
  }
  return BS_OK;
}

bs_status bs_contract(bs_plan *P, const void *A, const void *B, void *C, void *stream) {
  return contract_impl(P, A, B, C, stream, nullptr);
}

bs_status bs_contract_checked(bs_plan *P, const void *A, int64_t nA, const void *B, int64_t nB, void *C, int64_t nC,
                              void *stream) {
  if (nA < 0 || nB < 0 || nC < 0) return BS_ERR_INVALID_ARG;
  const int64_t sizes[3] = {nA, nB, nC};
  return contract_impl(P, A, B, C, stream, sizes);
}

}  // extern "C"

// The element range [first, last] a strided view covers, against a buffer of n elements.
static bool view_inside(int64_t off, int64_t rows, int64_t cols, int64_t ld, int64_t n) {
  if (rows <= 0 || cols <= 0) return true;
  return off >= 0 && off + (rows - 1) * ld + cols <= n;
}

static bs_status contract_impl(bs_plan *P, const void *A, const void *B, void *C, void *stream, const int64_t *sizes) {
  if (!P) return BS_ERR_INVALID_ARG;
  if (P->opts.host_only) return BS_ERR_INVALID_ARG;
  if (P->C.nelems == 0) return BS_OK;
  if (!A || !B || !C) return BS_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const void *Ause = P->pack_a ? P->d_ws_a : A;
  const void *Buse = P->pack_b ? P->d_ws_b : B;
  if (sizes) {
    // what the host can check before anything is enqueued: the gather's reads,
    // the zero fill's writes and the BF16 tensor maps' views
    for (size_t t = 0; t < P->pack_copies.size(); ++t) {
      const PackCopy &c = P->pack_copies[t];
      const bool of_a = P->pack_split.of_a((int64_t)t);
      if (!view_inside(c.src, c.rows, c.cols, c.src_ld, sizes[of_a ? 0 : 1])) return BS_ERR_DEVICE;
    }
    for (const auto &z : P->zero_blocks)
      if (!view_inside(z.off, z.rows, z.cols, z.ld, sizes[2])) return BS_ERR_DEVICE;
    for (const auto &m : P->maps) {
      const int64_t n = m.operand == 0 ? (P->pack_a ? P->A_pk.nelems : sizes[0]) : (P->pack_b ? P->B_pk.nelems : sizes[1]);
      if (!view_inside(m.off, m.outer, m.inner, m.ld, n)) return BS_ERR_DEVICE;
    }
    if (P->dtype == BS_BF16_F32)
      for (const auto &t : P->btasks)
        if (!view_inside(t.c_off, t.m, t.n, t.ldc, sizes[2])) return BS_ERR_DEVICE;
  }
  if (P->dtype == BS_BF16_F32 && !P->btasks.empty() && (P->maps_a_ptr != Ause || P->maps_b_ptr != Buse)) {
    // New operand pointers: the tensor maps are re-encoded, uploaded and
    // waited for, which a stream being captured into a graph cannot do;
    // refuse before anything is enqueued, so that the capture stays valid.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    BS_CUDA(cudaStreamIsCapturing(s, &capturing));
    if (capturing != cudaStreamCaptureStatusNone) return BS_ERR_UNSUPPORTED;
  }
  const bool prof = P->opts.profile != 0;
  if (prof) {
    for (auto &e : P->ev)
      if (!e) BS_CUDA(cudaEventCreate(&e));
    BS_CUDA(cudaEventRecord(P->ev[0], s));
  }
  if (!P->pack_copies.empty()) {
    PackParams pp{};
    pp.src = A;
    pp.dst = P->d_ws_a;
    pp.copies = P->d_pack;
    pp.ncopies = P->pack_split.total;
    pp.elem_bytes = P->dtype == BS_F64 ? 8 : 2;
    // one launch gathers both operands: copies [0, n_a) read A, the rest read B
    PackParams pb = pp;
    pb.src = B;
    pb.dst = P->d_ws_b;
    // A small FP64 gather (at most two segments per SM) goes by shared-memory
    // segments: all its copies are issued at once and no load waits on
    // another (the tail workload's block-row gather: 9.9 against 18.0 us).
    // A larger one goes block copy by block copy, where the segment writers
    // fall behind (the stress workload's: 207 against 111 us).  So does any
    // gather whose operand buffers do not start on 16-byte boundaries, and
    // the checked instance, whose reads must stay within the caller's
    // declared sizes.
    uintptr_t bases = 0;
    if (P->pack_a) bases |= (uintptr_t)A;
    if (P->pack_b) bases |= (uintptr_t)B;
    if (!P->pack_segs.empty() && !sizes && (bases & 15u) == 0) {
      SegParams sp{};
      sp.src[0] = (const double *)A;
      sp.src[1] = (const double *)B;
      sp.dst[0] = (double *)P->d_ws_a;
      sp.dst[1] = (double *)P->d_ws_b;
      sp.src_nelems[0] = P->A.nelems;
      sp.src_nelems[1] = P->B.nelems;
      sp.segs = P->d_segs;
      sp.pieces = P->d_pieces;
      sp.nseg = (int32_t)P->pack_segs.size();
      sp.status = P->d_status;
      sp.timeout_ns = (uint64_t)(P->opts.wait_timeout_ms > 0 ? P->opts.wait_timeout_ms : 2000) * 1000000ull;
      BS_CUDA(launch_seg_gather(sp, P->sm_count, s));
    } else {
      BS_CUDA(launch_pack2(pp, pb, P->pack_split, P->sm_count, s));
    }
  }
  if (prof) BS_CUDA(cudaEventRecord(P->ev[1], s));
  if (!P->zero_blocks.empty())
    BS_CUDA(launch_zero(C, P->dtype == BS_F64 ? 8 : 4, P->d_zero, (int)P->zero_blocks.size(), P->sm_count * 4, s));
  if (prof) BS_CUDA(cudaEventRecord(P->ev[2], s));
  bs_status st = contract_kernel(P, Ause, Buse, C, s, sizes);
  if (st == BS_OK && prof) {
    BS_CUDA(cudaEventRecord(P->ev[3], s));
    P->ev_recorded = true;
  }
  return st;
}

static bs_status contract_kernel(bs_plan *P, const void *Ause, const void *Buse, void *C, cudaStream_t s,
                                 const int64_t *sizes) {
  if (P->dtype == BS_F64) {
    if (P->ts.tasks.empty() && P->ts.tail_elems.empty()) return BS_OK;
    Fp64Params p{};
    p.A = (const double *)Ause;
    p.B = (const double *)Buse;
    p.C = (double *)C;
    p.tasks = P->d_tasks;
    p.groups = P->d_groups;
    p.rsegs = P->d_rsegs;
    p.ksegs = P->d_ksegs;
    p.tail_elems = (const int2 *)P->d_tail;
    p.tdesc = P->d_tdesc;
    p.ntasks = (int32_t)P->ts.tasks.size();
    p.ntail = (int32_t)(P->ts.tail_elems.size() / 2);
    p.nct = (int32_t)((p.ntail + kThreads - 1) / kThreads);
    fill_queue_params(&p, P->ts.tq_ptr, P->sm_map);
    if (sizes) {   // the checked instance: every operand load and C store against these counts
      p.check = 1;
      p.nA = P->pack_a ? P->A_pk.nelems : sizes[0];
      p.nB = P->pack_b ? P->B_pk.nelems : sizes[1];
      p.nC = sizes[2];
    }
    // Alternate launches use alternate counter sets, each launch preparing the
    // other; a launch being captured into a graph (replayed with the same
    // pointers) resets its own set at exit instead and leaves the parity.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    BS_CUDA(cudaStreamIsCapturing(s, &capturing));
    const bool captured = capturing != cudaStreamCaptureStatusNone;
    {
      const int nq = (int)std::max<size_t>(1, P->ts.tq_ptr.size()) - 1;   // as counter_bytes was sized
      char *sets = (char *)P->d_counter + 256;
      p.counter = (uint32_t *)(sets + (size_t)P->counter_parity * counter_set_bytes(nq));
      p.counter_next =
          captured ? nullptr : (uint32_t *)(sets + (size_t)(1 - P->counter_parity) * counter_set_bytes(nq));
      p.reset_at_exit = captured ? 1 : 0;
    }
    p.status = P->d_status;
    BS_CUDA(launch_fp64_grouped(p, P->grid, s));
    if (!captured) P->counter_parity ^= 1;
  } else {
    if (((uintptr_t)Ause | (uintptr_t)Buse | (uintptr_t)C) % 16 != 0) return BS_ERR_MISALIGNED;
    if (P->btasks.empty()) return BS_OK;
    if (P->maps_a_ptr != Ause || P->maps_b_ptr != Buse) {
      bs_status st = encode_maps(P, Ause, Buse);
      if (st != BS_OK) return st;
      BS_CUDA(cudaMemcpyAsync(P->d_maps, P->map_bytes.data(), P->map_bytes.size(), cudaMemcpyHostToDevice, s));
      BS_CUDA(cudaStreamSynchronize(s));
      P->maps_a_ptr = Ause;
      P->maps_b_ptr = Buse;
    }
    Bf16Params p{};
    p.maps = P->d_maps;
    p.ctas = P->d_bctas;
    p.tasks = P->d_bstasks;
    p.stages = P->d_bstages;
    p.C = (float *)C;
    p.status = P->d_status;
    p.counter = P->d_counter;
    p.timeout_ns = (uint64_t)(P->opts.wait_timeout_ms > 0 ? P->opts.wait_timeout_ms : 2000) * 1000000ull;
    p.debug_flags = P->opts.debug_flags;
    BS_CUDA(launch_bf16_grouped(p, P->grid, s));
  }
  return BS_OK;
}

extern "C" {

bs_status bs_plan_profile(bs_plan *P, bs_phase_times *out) {
  if (!P || !out || P->opts.host_only || !P->opts.profile || !P->ev_recorded) return BS_ERR_INVALID_ARG;
  *out = bs_phase_times{};
  BS_CUDA(cudaEventSynchronize(P->ev[3]));
  float t[3] = {0, 0, 0};
  for (int i = 0; i < 3; ++i) BS_CUDA(cudaEventElapsedTime(&t[i], P->ev[i], P->ev[i + 1]));
  out->gather_ms = P->pack_copies.empty() ? 0.0 : t[0];
  out->zero_ms = P->zero_blocks.empty() ? 0.0 : t[1];
  out->kernel_ms = t[2];
  out->total_ms = out->gather_ms + out->zero_ms + out->kernel_ms;
  out->gather_bytes = 2 * P->stats.packed_bytes;
  return BS_OK;
}

bs_status bs_contract_host(bs_plan *P, const void *A_host, const void *B_host, void *C_host, void *stream) {
  if (!P || !A_host || !B_host || !C_host || P->opts.host_only) return BS_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  {
    // the call waits for its own copies: not something a graph capture can hold
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    BS_CUDA(cudaStreamIsCapturing(s, &capturing));
    if (capturing != cudaStreamCaptureStatusNone) return BS_ERR_UNSUPPORTED;
  }
  const size_t eb = P->dtype == BS_F64 ? 8 : 2, ec = P->dtype == BS_F64 ? 8 : 4;
  const size_t na = (size_t)P->A.nelems * eb, nb = (size_t)P->B.nelems * eb, nc = (size_t)P->C.nelems * ec;
  if (!P->d_host_c) {
    BS_CUDA(cudaMalloc(&P->d_host_a, std::max<size_t>(na, 16)));
    BS_CUDA(cudaMalloc(&P->d_host_b, std::max<size_t>(nb, 16)));
    BS_CUDA(cudaMalloc(&P->d_host_c, std::max<size_t>(nc, 16)));
    BS_CUDA(cudaMemset(P->d_host_c, 0, std::max<size_t>(nc, 16)));   // padding stays zero
  }
  // A C buffer in pinned host memory that the device can address, under a plan
  // that writes every C element once (no zero fill, no accumulation): the
  // kernel stores C straight into it over the host link and no copy follows.
  // That pays when C is small (the copy's fixed cost is saved) or when the
  // kernel spreads its C stores thinly over a long run (an FP64 contraction
  // bound by its arithmetic, whose stores the link absorbs while the pipe
  // works, so the copy after the kernel disappears).  A kernel that writes C
  // faster than that (the BF16 path) runs slower storing over the link than
  // the copy engine moves C afterwards, and takes the copy.
  constexpr size_t kDirectCBytes = (size_t)4 << 20;
  constexpr double kDirectCBytesPerUs = 50e3;   // 50 GB/s of C over the modelled kernel time
  const double model_us = P->stats.model_us > 0 ? P->stats.model_us : 0.0;
  const bool thin_stores = model_us > 0 && (double)nc <= kDirectCBytesPerUs * model_us;
  void *c_direct = nullptr;
  if (P->zero_blocks.empty() && (nc <= kDirectCBytes || thin_stores)) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, C_host) == cudaSuccess) {
      if (at.type == cudaMemoryTypeHost && at.devicePointer) c_direct = at.devicePointer;
    } else {
      (void)cudaGetLastError();   // not a CUDA allocation: take the copy path
    }
  }
  // Inputs in pinned host memory that the device can address are pulled in by
  // one copy kernel (a single launch, loads spread over the SMs); any other
  // host memory goes through the copy engine, one copy per operand.
  auto device_alias = [](const void *h) -> const void * {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
  };
  const void *a_dev = device_alias(A_host), *b_dev = device_alias(B_host);
  if (a_dev && b_dev && ((uintptr_t)a_dev | (uintptr_t)b_dev) % 16 == 0) {
    BS_CUDA(launch_stage_in(a_dev, P->d_host_a, na, b_dev, P->d_host_b, nb, P->sm_count, s));
  } else {
    BS_CUDA(cudaMemcpyAsync(P->d_host_a, A_host, na, cudaMemcpyHostToDevice, s));
    BS_CUDA(cudaMemcpyAsync(P->d_host_b, B_host, nb, cudaMemcpyHostToDevice, s));
  }
  bs_status st = bs_contract(P, P->d_host_a, P->d_host_b, c_direct ? c_direct : P->d_host_c, stream);
  if (st != BS_OK) return st;
  if (!c_direct) BS_CUDA(cudaMemcpyAsync(C_host, P->d_host_c, nc, cudaMemcpyDeviceToHost, s));
  BS_CUDA(cudaStreamSynchronize(s));
  return BS_OK;
}

bs_status bs_contract_uncoalesced(bs_plan *P, const void *A, const void *B, void *C, void *stream) {
  if (!P || P->opts.host_only) return BS_ERR_INVALID_ARG;
  if (P->C.nelems == 0) return BS_OK;
  if (!A || !B || !C) return BS_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<int64_t> tp;
  std::vector<int32_t> tr;
  group_triples(P->gs, &tp, &tr);
  const size_t ec = P->dtype == BS_F64 ? 8 : 4;
  BS_CUDA(cudaMemsetAsync(C, 0, (size_t)P->C.nelems * ec, s));
  for (size_t t = 0; t < tr.size(); t += 3) {
    const auto &a = P->A.blocks[P->A.find(tr[t], tr[t + 1])];
    const auto &b = P->B.blocks[P->B.find(tr[t + 1], tr[t + 2])];
    const auto &c = P->C.blocks[P->C.find(tr[t], tr[t + 2])];
    cudaError_t e = P->dtype == BS_F64
                        ? launch_control_fp64((const double *)A, (const double *)B, (double *)C, a.offset, a.ld,
                                              b.offset, b.ld, c.offset, c.ld, a.rows, b.cols, a.cols, s)
                        : launch_control_bf16((const uint16_t *)A, (const uint16_t *)B, (float *)C, a.offset, a.ld,
                                              b.offset, b.ld, c.offset, c.ld, a.rows, b.cols, a.cols, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return BS_OK;
}

bs_status bs_plan_last_device_error(bs_plan *P, void *stream) {
  if (!P || P->opts.host_only) return BS_ERR_INVALID_ARG;
  BS_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  int32_t v = 0;
  BS_CUDA(cudaMemcpy(&v, P->d_status, sizeof v, cudaMemcpyDeviceToHost));
  if (v != 0) {
    BS_CUDA(cudaMemset(P->d_status, 0, sizeof v));
    // a kernel that stopped early may leave the work counters set
    bs_status st = init_counters(P);
    if (st != BS_OK) return st;
  }
  if (v == DS_OK) return BS_OK;
  if (v == DS_TIMEOUT) return BS_ERR_TIMEOUT;
  return BS_ERR_DEVICE;
}

void bs_plan_destroy(bs_plan *P) {
  if (!P) return;
  free_device(P);
  delete P;
}

}  // extern "C"

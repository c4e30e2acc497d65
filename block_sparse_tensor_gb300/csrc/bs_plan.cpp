// Structural product, coalescing planner and cost model (host).
//
// Follows the uni20 design note "block coalescing":
//   - "Why single-axis coalescing is hole-free": groups are taken along one
//     axis.  Contraction-axis group = one C block (i, j) with its inner blocks
//     k concatenated into one wider-K GEMM; free-axis group = one (k, j) with
//     the A blocks A[., k] stacked into one taller GEMM.  Either choice lists
//     only populated blocks, so no group holds a structural zero.
//   - "Interleaved vs contiguous": adjacent blocks whose strides agree merge
//     into one wider view (zero copy); otherwise the group walks several views
//     or the operand is gathered into a panel workspace, whichever the cost
//     model prefers ("pack cost vs launch savings").
//   - "Two coalescing modes" / "The crossover decides whether to coalesce": a
//     single-axis group carries no wasted flops, so the only trade is per-task
//     and per-segment overhead against gather bytes.
//   - "Coalescing is a plan-time transform": everything here runs once per plan.
//   - "Interleaved" LocalSpace keys: row sectors whose groups have the same
//     inner blocks and whose A and C rows continue each other with one stride
//     are stacked into one taller group (merge_rows).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <numeric>

#include "bs_plan.h"

namespace bs {

namespace {

struct Builder {
  GroupSet gs;
  void add_triple(int32_t i, int32_t k, int32_t j) {
    gs.triples.push_back(i);
    gs.triples.push_back(k);
    gs.triples.push_back(j);
  }
  void close_group() { gs.tptr.push_back((int64_t)gs.triples.size() / 3); }
};

struct Entry {
  int32_t k, blk_a, blk_b;
};

}  // namespace

// One group per C block: the inner blocks in A's storage order, merged into
// runs where both the A view and the B view continue with the same stride.
GroupSet make_contraction_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C, bool merge_rows,
                                 bool atomic, bool unchecked, const std::vector<uint8_t> *cmask) {
  Builder bd;
  GroupSet &gs = bd.gs;
  gs.tptr.push_back(0);
  const int32_t ni = A.rows.n, nj = B.cols.n;
  std::vector<std::vector<Entry>> bucket(nj);
  std::vector<int32_t> touched;
  // for row merging: the last group per column, its last row sector and entries
  std::vector<int32_t> last_group(nj, -1), last_row(nj, -1);
  std::vector<std::vector<Entry>> last_entries(merge_rows ? nj : 0);
  for (int32_t i = 0; i < ni; ++i) {
    touched.clear();
    for (int64_t t = A.row_ptr[i]; t < A.row_ptr[i + 1]; ++t) {
      const int32_t ba = A.row_blk[t];
      const int32_t k = A.blocks[ba].col;
      for (int64_t u = B.row_ptr[k]; u < B.row_ptr[k + 1]; ++u) {
        const int32_t bb = B.row_blk[u];
        const int32_t j = B.blocks[bb].col;
        if (bucket[j].empty()) touched.push_back(j);
        bucket[j].push_back({k, ba, bb});
      }
    }
    std::sort(touched.begin(), touched.end());
    for (int32_t j : touched) {
      auto &ent = bucket[j];
      const int32_t cb = C.find(i, j);
      if (cmask && !(*cmask)[cb]) {   // another shard's C block
        ent.clear();
        continue;
      }
      const bs_block_info &cbi = C.blocks[cb];
      bool merged = false;
      if (merge_rows && last_group[j] >= 0 && last_row[j] == i - 1 && last_entries[j].size() == ent.size()) {
        Group &g = gs.groups[last_group[j]];
        const RowSeg &rs = gs.rsegs[g.rseg_begin];
        bool ok = g.rseg_count == 1 && (g.flags & GF_ATOMIC) == (atomic ? GF_ATOMIC : 0) && rs.ldc == cbi.ld &&
                  cbi.offset == rs.rc + (int64_t)g.m * rs.ldc;
        for (size_t e = 0; ok && e < ent.size(); ++e) {
          const auto &a0 = A.blocks[last_entries[j][e].blk_a];
          const auto &a1 = A.blocks[ent[e].blk_a];
          // same inner block, same B block, A rows continuing the group's rows
          // (`unchecked`, a testing switch, skips the first two conditions)
          ok = (unchecked || (last_entries[j][e].k == ent[e].k && last_entries[j][e].blk_b == ent[e].blk_b)) &&
               a1.ld == a0.ld && a1.offset == a0.offset + (int64_t)g.m * a0.ld;
        }
        if (ok) {
          // last_entries keeps the group's first row sector, which the offsets are relative to
          g.m += A.rows.d[i];
          gs.rsegs[g.rseg_begin].rows += A.rows.d[i];
          // triples of the merged row: insert before the sentinel of this group
          // (groups are closed in order, so append to the group's range only if it is the last)
          merged = true;
          last_row[j] = i;
          // record the triples of row i for this group
          for (const auto &e : ent) gs.extra_triples.push_back({last_group[j], i, e.k, j});
        }
      }
      if (!merged) {
        Group g{};
        g.n = B.cols.d[j];
        g.m = A.rows.d[i];
        g.flags = atomic ? GF_ATOMIC : 0;
        g.rseg_begin = (int32_t)gs.rsegs.size();
        g.rseg_count = 1;
        RowSeg rs{};
        rs.ra = 0;
        rs.lda = 0;
        rs.rc = cbi.offset;
        rs.ldc = cbi.ld;
        rs.r0 = 0;
        rs.rows = g.m;
        rs.rl = 1;
        gs.rsegs.push_back(rs);
        g.kseg_begin = (int32_t)gs.ksegs.size();
        int32_t kpos = 0;
        for (const auto &e : ent) {
          const auto &a = A.blocks[e.blk_a];
          const auto &b = B.blocks[e.blk_b];
          const int32_t dk = A.cols.d[e.k];
          bool join = false;
          if ((int32_t)gs.ksegs.size() > g.kseg_begin) {
            KSeg &s = gs.ksegs.back();
            join = a.ld == s.kl && a.offset == s.ka + s.klen && b.ld == s.ldb && b.offset == s.kb + (int64_t)s.klen * s.ldb;
            if (join) s.klen += dk;
          }
          if (!join) {
            KSeg s{};
            s.ka = a.offset;
            s.kl = a.ld;
            s.kb = b.offset;
            s.ldb = b.ld;
            s.k0 = kpos;
            s.klen = dk;
            gs.ksegs.push_back(s);
          }
          kpos += dk;
          bd.add_triple(i, e.k, j);
        }
        g.k = kpos;
        g.kseg_count = (int32_t)gs.ksegs.size() - g.kseg_begin;
        gs.groups.push_back(g);
        bd.close_group();
        if (merge_rows) {
          last_group[j] = (int32_t)gs.groups.size() - 1;
          last_row[j] = i;
          last_entries[j] = ent;
        }
      }
      ent.clear();
    }
  }
  return gs;
}

// One group per (k, j): the A blocks of inner sector k stacked in A's storage
// order; runs whose A rows and C rows continue with one stride share a row
// segment.  Several groups add into the same C block, so stores are atomic.
GroupSet make_free_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C,
                          const std::vector<uint8_t> *cmask) {
  Builder bd;
  GroupSet &gs = bd.gs;
  gs.tptr.push_back(0);
  const int32_t nk = A.cols.n;
  int64_t ntr = 0, ngr = 0;
  for (int32_t k = 0; k < nk; ++k) {
    const int64_t nb = B.row_ptr[k + 1] - B.row_ptr[k];
    ntr += (A.col_ptr[k + 1] - A.col_ptr[k]) * nb;
    if (A.col_ptr[k] != A.col_ptr[k + 1]) ngr += nb;
  }
  gs.triples.reserve((size_t)ntr * 3);
  gs.rsegs.reserve((size_t)ntr);
  gs.groups.reserve((size_t)ngr);
  gs.ksegs.reserve((size_t)ngr);
  gs.tptr.reserve((size_t)ngr + 1);
  std::vector<int32_t> cblk;   // C block of (t-th A block of column k, u-th B block of row k)
  for (int32_t k = 0; k < nk; ++k) {
    if (A.col_ptr[k] == A.col_ptr[k + 1]) continue;
    const int64_t na = A.col_ptr[k + 1] - A.col_ptr[k], nb = B.row_ptr[k + 1] - B.row_ptr[k];
    // look the C blocks up row by row (each C row's blocks lie together)
    cblk.resize((size_t)(na * nb));
    for (int64_t t = 0; t < na; ++t) {
      const int32_t i = A.blocks[A.col_blk[A.col_ptr[k] + t]].row;
      for (int64_t u = 0; u < nb; ++u) cblk[t * nb + u] = C.find(i, B.blocks[B.row_blk[B.row_ptr[k] + u]].col);
    }
    for (int64_t u = B.row_ptr[k]; u < B.row_ptr[k + 1]; ++u) {
      const auto &b = B.blocks[B.row_blk[u]];
      const int32_t j = b.col;
      Group g{};
      g.n = B.cols.d[j];
      g.k = A.cols.d[k];
      g.flags = GF_ATOMIC;
      g.rseg_begin = (int32_t)gs.rsegs.size();
      int32_t r = 0;
      for (int64_t t = A.col_ptr[k]; t < A.col_ptr[k + 1]; ++t) {
        const auto &a = A.blocks[A.col_blk[t]];
        const int32_t i = a.row;
        const int32_t cb = cblk[(t - A.col_ptr[k]) * nb + (u - B.row_ptr[k])];
        if (cmask && !(*cmask)[cb]) continue;   // another shard's C block
        const auto &c = C.blocks[cb];
        bool join = false;
        if ((int32_t)gs.rsegs.size() > g.rseg_begin) {
          RowSeg &s = gs.rsegs.back();
          join = a.ld == s.lda && a.offset == s.ra + (int64_t)s.rows * s.lda && c.ld == s.ldc &&
                 c.offset == s.rc + (int64_t)s.rows * s.ldc;
          if (join) s.rows += a.rows;
        }
        if (!join) {
          RowSeg s{};
          s.ra = a.offset;
          s.lda = a.ld;
          s.rc = c.offset;
          s.ldc = c.ld;
          s.r0 = r;
          s.rows = a.rows;
          s.rl = 0;
          gs.rsegs.push_back(s);
        }
        r += a.rows;
        bd.add_triple(i, k, j);
      }
      if (r == 0) continue;   // every row of this (k, j) belongs to other shards
      g.m = r;
      g.rseg_count = (int32_t)gs.rsegs.size() - g.rseg_begin;
      g.kseg_begin = (int32_t)gs.ksegs.size();
      g.kseg_count = 1;
      KSeg s{};
      s.ka = 0;
      s.kl = 0;
      s.kb = b.offset;
      s.ldb = b.ld;
      s.k0 = 0;
      s.klen = g.k;
      gs.ksegs.push_back(s);
      gs.groups.push_back(g);
      bd.close_group();
    }
  }
  return gs;
}

// No coalescing: one group per populated triple, scattered atomically.
GroupSet make_triple_groups(const bs_layout &A, const bs_layout &B, const bs_layout &C,
                            const std::vector<uint8_t> *cmask) {
  Builder bd;
  GroupSet &gs = bd.gs;
  gs.tptr.push_back(0);
  for (int32_t i = 0; i < A.rows.n; ++i)
    for (int64_t t = A.row_ptr[i]; t < A.row_ptr[i + 1]; ++t) {
      const auto &a = A.blocks[A.row_blk[t]];
      const int32_t k = a.col;
      for (int64_t u = B.row_ptr[k]; u < B.row_ptr[k + 1]; ++u) {
        const auto &b = B.blocks[B.row_blk[u]];
        const int32_t cb = C.find(i, b.col);
        if (cmask && !(*cmask)[cb]) continue;   // another shard's C block
        const auto &c = C.blocks[cb];
        Group g{};
        g.m = a.rows;
        g.n = b.cols;
        g.k = a.cols;
        g.flags = GF_ATOMIC;
        g.rseg_begin = (int32_t)gs.rsegs.size();
        g.rseg_count = 1;
        RowSeg rs{};
        rs.rc = c.offset;
        rs.ldc = c.ld;
        rs.rows = g.m;
        rs.rl = 1;
        gs.rsegs.push_back(rs);
        g.kseg_begin = (int32_t)gs.ksegs.size();
        g.kseg_count = 1;
        KSeg s{};
        s.ka = a.offset;
        s.kl = a.ld;
        s.kb = b.offset;
        s.ldb = b.ld;
        s.klen = g.k;
        gs.ksegs.push_back(s);
        gs.groups.push_back(g);
        bd.add_triple(i, k, b.col);
        bd.close_group();
      }
    }
  return gs;
}

std::vector<uint8_t> shard_mask(const bs_layout &A, const bs_layout &B, const bs_layout &C, int rank, int world) {
  const size_t nc = C.blocks.size();
  std::vector<double> cost(nc, 0.0);
  for (int32_t i = 0; i < A.rows.n; ++i)
    for (int64_t t = A.row_ptr[i]; t < A.row_ptr[i + 1]; ++t) {
      const int32_t k = A.blocks[A.row_blk[t]].col;
      const double dik = (double)A.rows.d[i] * A.cols.d[k];
      for (int64_t u = B.row_ptr[k]; u < B.row_ptr[k + 1]; ++u) {
        const int32_t j = B.blocks[B.row_blk[u]].col;
        cost[C.find(i, j)] += dik * B.cols.d[j];
      }
    }
  std::vector<int32_t> order(nc);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
  std::vector<double> load((size_t)world, 0.0);
  std::vector<uint8_t> mask(nc, 0);
  for (int32_t b : order) {
    int best = 0;
    for (int r = 1; r < world; ++r)
      if (load[r] < load[best]) best = r;
    load[best] += cost[b];
    if (best == rank) mask[b] = 1;
  }
  return mask;
}

// Triples of every group, group by group, with merged rows folded in.
void group_triples(const GroupSet &gs, std::vector<int64_t> *ptr, std::vector<int32_t> *out) {
  const size_t ng = gs.groups.size();
  std::vector<std::vector<int32_t>> extra(ng);
  for (const auto &e : gs.extra_triples) {
    extra[e[0]].push_back(e[1]);
    extra[e[0]].push_back(e[2]);
    extra[e[0]].push_back(e[3]);
  }
  ptr->assign(ng + 1, 0);
  out->clear();
  for (size_t g = 0; g < ng; ++g) {
    out->insert(out->end(), gs.triples.begin() + 3 * gs.tptr[g], gs.triples.begin() + 3 * gs.tptr[g + 1]);
    out->insert(out->end(), extra[g].begin(), extra[g].end());
    (*ptr)[g + 1] = (int64_t)out->size() / 3;
  }
}

// ---- FP64 tiling -----------------------------------------------------------

// Outputs are spread one per thread slot, so any tm x tn <= kTileMaxElems keeps
// the lanes busy; the shape follows the group's aspect ratio and its area is
// capped so that no single task outlasts the rest of the launch.
static void tile_shape(int32_t m, int32_t n, int32_t area, int32_t *tm, int32_t *tn) {
  area = std::max(32, std::min(area, kTileMaxElems));
  if (n <= 8) {
    *tn = n;
    *tm = std::min(m, std::min(kTileMaxDim, std::max(1, area / n)));
  } else if (m <= 8) {
    *tm = m;
    *tn = std::min(n, std::min(kTileMaxDim, std::max(1, area / m)));
  } else {
    int32_t side = 8;
    while (side * 2 * side * 2 <= area && side < 32) side *= 2;
    *tn = std::min(n, side);
    *tm = std::min(m, std::min(kTileMaxDim, std::max(1, area / *tn)));
  }
}

static inline int64_t lanes(int64_t e) { return (e + 31) / 32 * 32; }

void tile_fp64(GroupSet &gs, const PlanModel &pm, TileSet *ts, bool materialize) {
  ts->tasks.clear();
  ts->tail_elems.clear();
  ts->tq_ptr.clear();
  ts->tdesc.clear();
  ts->exec_tile = ts->exec_tail = ts->exec_general = ts->max_tail_task = ts->max_tile_task = ts->tile_slots = 0;
  ts->max_tile_slots = 0;
  if (materialize) ts->tdesc.assign(gs.groups.size(), TailDesc{});
  std::vector<std::pair<double, Task>> costed;
  std::vector<int32_t> tails;
  double exec = 0, work = 0;
  for (const auto &G : gs.groups) work += (double)G.m * G.n * G.k;
  // per-task work target: a few tasks per SM, so longest-first scheduling balances
  const double target = std::max(8192.0, work / (std::max(1, pm.sms) * 4.0));
  for (int32_t g = 0; g < (int32_t)gs.groups.size(); ++g) {
    const Group &G = gs.groups[g];
    const int64_t e = (int64_t)G.m * G.n;
    if (e <= kTailMaxElems) {
      tails.push_back(g);
      continue;
    }
    int32_t tm, tn;
    tile_shape(G.m, G.n, (int32_t)std::min<double>(kTileMaxElems, target / std::max(1, G.k)), &tm, &tn);
    for (int32_t m0 = 0; m0 < G.m; m0 += tm)
      for (int32_t n0 = 0; n0 < G.n; n0 += tn) {
        Task t{};
        t.kind = TK_TILE;
        t.g = g;
        t.m0 = m0;
        t.n0 = n0;
        t.tm = std::min(tm, G.m - m0);
        t.tn = std::min(tn, G.n - n0);
        const double slots = (double)lanes((int64_t)t.tm * t.tn);
        exec += 2.0 * slots * G.k;
        ts->exec_tile += 2.0 * slots * G.k;
        ts->tile_slots += slots;
        if (2.0 * slots * G.k > ts->max_tile_task) {
          ts->max_tile_task = 2.0 * slots * G.k;
          ts->max_tile_slots = (int64_t)slots;
        }
        costed.push_back({slots * G.k + pm.task_slots, t});
      }
  }
  // Small groups: every output gets its own lane.  Groups are ordered by
  // decreasing K so that the 32 lanes of a warp run loops of nearly equal
  // length; warps take 32 consecutive outputs at a time.  With bucket_pad a
  // single-segment group is padded to power-of-two M, N and K and groups of
  // one padded shape are listed together: they run as one batched call whose
  // padded lanes and steps add only zeros.
  auto pow2 = [](int32_t x) {
    int32_t p = 1;
    while (p < x) p <<= 1;
    return p;
  };
  auto padded = [&](int32_t g, int32_t *mp, int32_t *np, int32_t *kp) {
    const Group &G = gs.groups[g];
    const bool pad = pm.bucket_pad && G.rseg_count == 1 && G.kseg_count == 1;
    *mp = pad ? pow2(G.m) : G.m;
    *np = pad ? pow2(G.n) : G.n;
    *kp = pad ? pow2(G.k) : G.k;
  };
  // A group of one view whose K reaches tail_split_k runs each output on two
  // lanes of one warp: lanes 0-15 sum the first half of K for 16 outputs,
  // lanes 16-31 the second half for the same outputs, and one shuffle adds
  // them.  Its warps then run half as long, which halves the longest tail
  // tasks (they share an SM's pipe with the other CTAs for their whole life)
  // and lets the plan-time dealing balance the SMs more finely.
  auto split_of = [&](int32_t g, int32_t kp) {
    const Group &G = gs.groups[g];
    return pm.tail_split_k > 0 && G.rseg_count == 1 && G.kseg_count == 1 && kp >= pm.tail_split_k;
  };
  auto lane_k = [&](int32_t g) {
    int32_t mp, np, kp;
    padded(g, &mp, &np, &kp);
    return split_of(g, kp) ? (kp + 1) / 2 : kp;
  };
  std::stable_sort(tails.begin(), tails.end(), [&](int32_t a, int32_t b) {
    const int32_t ka = lane_k(a), kb = lane_k(b);
    if (!pm.bucket_pad) return ka > kb;   // exact: by K per lane only, as listed
    int32_t ma, na, xa, mb, nb, xb;
    padded(a, &ma, &na, &xa);
    padded(b, &mb, &nb, &xb);
    return std::make_tuple(-ka, ma, na) < std::make_tuple(-kb, mb, nb);
  });
  // One walk over the sorted groups lays out the tail list: each warp of 32
  // consecutive entries runs its first lane's K (the list runs longest K
  // first); a split group starts on a warp boundary (the previous warp is
  // padded with entries that hold no output) and takes one warp per 16 of its
  // outputs.  The walk gives the executed flops split by path (groups of one
  // view take the unrolled loop, the others the segment walk) and the cost
  // of the first, costliest task; with `emit` it also writes the list.
  std::vector<int32_t> elem_k;
  auto walk = [&](bool emit) {
    int64_t off = 0;
    auto push = [&](int32_t g, int32_t rc, int32_t k) {
      if (emit) {
        ts->tail_elems.push_back(g);
        ts->tail_elems.push_back(rc);
        elem_k.push_back(k);
      }
    };
    auto count_warps = [&](int64_t from, int64_t to, int32_t k, bool single) {
      const int64_t warps = (to + 31) / 32 - (from + 31) / 32;   // warp starts inside [from, to)
      const double ex = 2.0 * 32.0 * k * (double)warps;
      if (single) ts->exec_tail += ex;
      else ts->exec_general += ex;
      for (int64_t w = (from + 31) / 32 * 32; w < to && w < kThreads; w += 32) ts->max_tail_task += 2.0 * 32.0 * k;
    };
    for (int32_t g : tails) {
      const Group &G = gs.groups[g];
      int32_t mp, np, kp;
      padded(g, &mp, &np, &kp);
      const bool single = G.rseg_count == 1 && G.kseg_count == 1;
      const int64_t nout = (int64_t)mp * np;
      if (split_of(g, kp)) {
        const int32_t lk = (kp + 1) / 2;
        while (off % 32) {   // fill the previous warp
          push(g, kTailPad, 0);
          ++off;
        }
        for (int64_t c0 = 0; c0 < nout; c0 += 16)
          for (int half = 0; half < 2; ++half)
            for (int64_t e = c0; e < c0 + 16; ++e) {
              const int32_t gg = half ? (g | kTailHi) : g;
              if (e < nout) push(gg, (int32_t)(((e / np) << 16) | (e % np)), lk);
              else push(gg, kTailPad, 0);
            }
        const int64_t end = off + (nout + 15) / 16 * 32;
        count_warps(off, end, lk, true);
        off = end;
      } else {
        for (int32_t r = 0; emit && r < mp; ++r)
          for (int32_t c = 0; c < np; ++c) push(g, (r << 16) | c, kp);
        count_warps(off, off + nout, kp, single);
        off += nout;
      }
    }
  };
  walk(!materialize ? false : true);
  if (!materialize) {
    exec += ts->exec_tail + ts->exec_general;
    for (auto &c : costed) ts->tasks.push_back(c.second);
    ts->executed_flops = exec;
    return;
  }
  for (int32_t g : tails) {
    const Group &G = gs.groups[g];
    int32_t mp, np, kp;
    padded(g, &mp, &np, &kp);
    if (G.rseg_count == 1 && G.kseg_count == 1) {   // resolve the addressing once, here
      const RowSeg &rs = gs.rsegs[G.rseg_begin];
      const KSeg &ks = gs.ksegs[G.kseg_begin];
      TailDesc &d = ts->tdesc[g];
      d.a0 = rs.ra + ks.ka;
      d.as = rs.lda + (rs.rl ? ks.kl : 0);
      d.b0 = ks.kb;
      d.ldb = ks.ldb;
      d.c0 = rs.rc;
      d.ldc = rs.ldc;
      d.k = G.k;
      d.flags = G.flags;
      d.kpad = kp;
      d.m = G.m;
      d.n = G.n;
    }
  }
  // Tail tasks of kThreads outputs (one CTA, one output per thread): the 8
  // warps of a task hold consecutive outputs of the same group(s), so they
  // walk the same B rows together and share them through L1.  Tasks are dealt
  // to one queue per SM, longest first onto the least loaded queue, so every
  // SM starts with the same amount of FP64 work whatever order its CTAs
  // arrive in.  Lane 0 of each warp holds that warp's longest K.
  const int nct = (int)((elem_k.size() + kThreads - 1) / kThreads);
  // no more queues than a few tasks each can fill (SMs then share a queue)
  const int nq = std::max(1, std::min(std::min(pm.sms, kMaxQueues), nct / 4));
  std::vector<std::vector<int32_t>> queues(nq);
  std::vector<std::pair<double, int>> heap;   // (load, queue) min-heap
  for (int q = 0; q < nq; ++q) heap.push_back({0.0, q});
  auto cmp = [](const std::pair<double, int> &a, const std::pair<double, int> &b) { return a.first > b.first; };
  std::make_heap(heap.begin(), heap.end(), cmp);
  for (int ct = 0; ct < nct; ++ct) {
    double cost = 64.0;   // fixed cost per task
    for (size_t w = (size_t)ct * kThreads; w < std::min(elem_k.size(), (size_t)(ct + 1) * kThreads); w += 32) {
      exec += 2.0 * 32.0 * elem_k[w];
      cost += elem_k[w];
    }
    std::pop_heap(heap.begin(), heap.end(), cmp);
    heap.back().first += cost;
    queues[heap.back().second].push_back(ct);
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  // Renumber the tasks queue after queue, so queue q holds tasks
  // tq_ptr[q] .. tq_ptr[q+1]-1 and a claim needs no table: the tail list is
  // rewritten in that order, each task's kThreads entries together, the last
  // (partial) task padded with entries that hold no output.
  ts->tq_ptr.assign(nq + 1, 0);
  std::vector<int32_t> listed;
  listed.swap(ts->tail_elems);
  ts->tail_elems.reserve((size_t)nct * kThreads * 2);
  const size_t nel = listed.size() / 2;
  for (int q = 0; q < nq; ++q) {
    for (int32_t ct : queues[q]) {
      for (size_t e = (size_t)ct * kThreads; e < (size_t)(ct + 1) * kThreads; ++e) {
        if (e < nel) {
          ts->tail_elems.push_back(listed[2 * e]);
          ts->tail_elems.push_back(listed[2 * e + 1]);
        } else {
          ts->tail_elems.push_back(listed[2 * (nel - 1)]);   // a real group, so its descriptor can be read
          ts->tail_elems.push_back(kTailPad);
        }
      }
    }
    ts->tq_ptr[q + 1] = ts->tq_ptr[q] + (int32_t)queues[q].size();
  }
  // longest processing time first for the dynamic scheduler
  std::stable_sort(costed.begin(), costed.end(),
                   [](const std::pair<double, Task> &a, const std::pair<double, Task> &b) { return a.first > b.first; });
  for (auto &c : costed) ts->tasks.push_back(c.second);
  ts->executed_flops = exec;
}

double model_fp64_us(const GroupSet &gs, const TileSet &ts, const PlanModel &pm, int64_t pack_bytes, int launches,
                     int64_t zero_bytes) {
  // Tile path: every task costs as if its K were K + tile_k0 (staging and
  // synchronisation per chunk), and the launch cannot end before its
  // costliest task has run at its CTA's share of one SM.
  const double r_tile = pm.fp64_gflops * 1e3;   // flops per microsecond
  const double tile = (ts.exec_tile + 2.0 * pm.tile_k0 * ts.tile_slots) / r_tile;
  const double per_cta = r_tile / std::max(1, pm.parallel_ctas);
  const double drain = ts.max_tile_task > 0 ? (ts.max_tile_task + 2.0 * pm.tile_k0 * ts.max_tile_slots) / per_cta : 0.0;
  // (tile tasks run first, longest first; the last of them overlaps the tail
  // work that the CTAs finishing earlier pick up)
  // Tail path at its measured rates; groups stored with atomics (free axis,
  // no coalescing) run at atomic_penalty of them.
  bool atomic = false;
  int64_t nseg = 0;
  for (const auto &g : gs.groups) {
    nseg += g.kseg_count + g.rseg_count;
    atomic |= (g.flags & GF_ATOMIC) != 0;
  }
  const double f = atomic ? pm.atomic_penalty : 1.0;
  const double tail = ts.exec_tail / (pm.tail_gflops * 1e3 * f) + ts.exec_general / (pm.general_gflops * 1e3 * f);
  const double par = std::max(1, pm.parallel_ctas);
  const double overhead = ((double)ts.tasks.size() * pm.t_task_us + (double)nseg * pm.t_segment_us) / par;
  const double zero = zero_bytes > 0 ? (double)zero_bytes / (pm.zero_gbs * 1e3) : 0.0;
  const double pack = pack_bytes > 0 ? pm.pack_fixed_us + 2.0 * pack_bytes / (pm.pack_gbs * 1e3) : 0.0;
  return pm.t_fixed_us + std::max(0, launches - 1) * pm.t_launch_us + tile + std::max(drain, tail) + overhead + zero +
         pack;
}

double model_bf16_us(const bs_plan &P, const PlanModel &pm) {
  // One CTA per SM walks its own list: per CTA, its K stages and its output
  // tiles (epilogue in proportion to the tile width); the slowest CTA ends it.
  double worst = 0;
  for (const auto &c : P.bctas) {
    double t = c.stage_count * pm.bf16_stage_us;
    for (int32_t i = 0; i < c.task_count; ++i) t += pm.bf16_tile_us * P.bstasks[c.task_begin + i].bn / 256.0;
    worst = std::max(worst, t);
  }
  const double pack = P.stats.packed_bytes > 0 ? pm.pack_fixed_us + 2.0 * P.stats.packed_bytes / (pm.pack_gbs * 1e3)
                                               : 0.0;
  return pm.t_fixed_us + worst + pack;
}

}  // namespace bs
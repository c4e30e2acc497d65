// Sector layouts: which blocks exist and where each one lives in the buffer.
//
// A block is an (offset, leading dimension) view into one shared buffer, as
// in the uni20 design note "block coalescing" ("Expressed as strided views
// over shared storage").  The arrangement is a per-tensor choice made for the
// expected coalescing groups ("Interleaved vs contiguous": interleave the axis
// you will coalesce): ROWPANEL keeps each row sector's blocks side by side so
// one output block's inner blocks form one strided view, COLPANEL stacks each
// column sector's blocks so a free-axis group's rows form one view.
#include <algorithm>
#include <numeric>

#include "bs_host.h"

namespace bs {

bs_status copy_axis(const bs_axis_desc *d, AxisCopy *out) {
  if (!d || d->n < 0) return BS_ERR_INVALID_ARG;
  if (d->n > 0 && (!d->q_u1 || !d->dim)) return BS_ERR_INVALID_ARG;
  out->n = d->n;
  out->q.assign(d->q_u1, d->q_u1 + d->n);
  out->d.assign(d->dim, d->dim + d->n);
  if (d->q_z2) out->p.assign(d->q_z2, d->q_z2 + d->n);
  else out->p.clear();
  for (int32_t t = 0; t < d->n; ++t) {
    if (out->d[t] < 1) return BS_ERR_INVALID_ARG;
    if (!out->p.empty() && out->p[t] > 1) return BS_ERR_INVALID_ARG;
  }
  return BS_OK;
}

Sparsity rule_sparsity(const AxisCopy &r, const AxisCopy &c, const bs_rule &rule) {
  Sparsity sp;
  sp.ptr.assign(r.n + 1, 0);
  // Columns sorted by charge let each row find its allowed charge window by
  // binary search instead of scanning every column.
  std::vector<int32_t> by_q(c.n);
  std::iota(by_q.begin(), by_q.end(), 0);
  std::stable_sort(by_q.begin(), by_q.end(), [&](int32_t a, int32_t b) { return c.q[a] < c.q[b]; });
  std::vector<int32_t> row;
  for (int32_t i = 0; i < r.n; ++i) {
    // allowed: dq_min <= q_r - q_c <= dq_max  <=>  q_r - dq_max <= q_c <= q_r - dq_min
    int64_t lo = (int64_t)r.q[i] - rule.dq_max, hi = (int64_t)r.q[i] - rule.dq_min;
    auto first = std::lower_bound(by_q.begin(), by_q.end(), lo,
                                  [&](int32_t a, int64_t v) { return (int64_t)c.q[a] < v; });
    row.clear();
    for (auto it = first; it != by_q.end() && (int64_t)c.q[*it] <= hi; ++it) {
      if (rule.z2 && r.p[i] != c.p[*it]) continue;
      row.push_back(*it);
    }
    std::sort(row.begin(), row.end());
    sp.cols.insert(sp.cols.end(), row.begin(), row.end());
    sp.ptr[i + 1] = (int64_t)sp.cols.size();
  }
  return sp;
}

static std::vector<int32_t> sector_order(const AxisCopy &a, bool sorted) {
  std::vector<int32_t> o(a.n);
  std::iota(o.begin(), o.end(), 0);
  if (sorted) {
    std::sort(o.begin(), o.end(), [&](int32_t x, int32_t y) {
      int px = a.p.empty() ? 0 : a.p[x], py = a.p.empty() ? 0 : a.p[y];
      if (a.q[x] != a.q[y]) return a.q[x] < a.q[y];
      if (px != py) return px < py;
      return x < y;
    });
  }
  return o;
}

static inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bs_status build_layout(const AxisCopy &rows, const AxisCopy &cols, const Sparsity &sp, uint32_t flags,
                       int32_t elem_bytes, bs_layout *L) {
  if ((flags & ~31u) != 0 || (flags & 3u) == 3u) return BS_ERR_INVALID_ARG;
  if (elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return BS_ERR_INVALID_ARG;
  // a group's M, N and K are sums of one axis's dimensions, held in 32 bits
  for (const AxisCopy *ax : {&rows, &cols}) {
    int64_t total = 0;
    for (int32_t t = 0; t < ax->n; ++t) total += ax->d[t];
    if (total > INT32_MAX) return BS_ERR_OVERFLOW;
  }
  L->rows = rows;
  L->cols = cols;
  L->flags = flags;
  L->elem_bytes = elem_bytes;
  const int64_t al = (flags & BS_LAYOUT_ALIGN64) ? 64 / elem_bytes : (flags & BS_LAYOUT_ALIGN16) ? 16 / elem_bytes : 1;
  const bool sorted = (flags & BS_LAYOUT_CHARGE_SORTED) != 0;
  const std::vector<int32_t> ro = sector_order(rows, sorted), co = sector_order(cols, sorted);
  std::vector<int32_t> col_rank(cols.n);
  for (int32_t t = 0; t < cols.n; ++t) col_rank[co[t]] = t;
  const uint32_t mode = flags & 3u;
  L->blocks.clear();
  L->blocks.reserve(sp.cols.size());
  int64_t pos = 0;
  const int64_t lim = INT64_MAX / 4;
  std::vector<int32_t> rowcols;
  auto width = [&](int32_t c) { return round_up(cols.d[c], al); };
  if (mode == BS_LAYOUT_BLOCKROW || mode == BS_LAYOUT_ROWPANEL) {
    for (int32_t a = 0; a < rows.n; ++a) {
      const int32_t r = ro[a];
      rowcols.assign(sp.cols.begin() + sp.ptr[r], sp.cols.begin() + sp.ptr[r + 1]);
      std::sort(rowcols.begin(), rowcols.end(), [&](int32_t x, int32_t y) { return col_rank[x] < col_rank[y]; });
      int64_t panel = 0;
      for (int32_t c : rowcols) panel += width(c);
      int64_t col = 0;
      for (int32_t c : rowcols) {
        bs_block_info b;
        b.row = r;
        b.col = c;
        b.rows = rows.d[r];
        b.cols = cols.d[c];
        if (mode == BS_LAYOUT_BLOCKROW) {
          b.offset = pos;
          b.ld = width(c);
          pos += (int64_t)rows.d[r] * b.ld;
        } else {
          b.offset = pos + col;
          b.ld = panel;
          col += width(c);
        }
        if (pos > lim) return BS_ERR_OVERFLOW;
        L->blocks.push_back(b);
      }
      if (mode == BS_LAYOUT_ROWPANEL) pos += (int64_t)rows.d[r] * panel;
      if (pos > lim) return BS_ERR_OVERFLOW;
    }
  } else {
    // column panels: gather each column's rows from the CSR
    std::vector<std::vector<int32_t>> by_col(cols.n);
    for (int32_t r = 0; r < rows.n; ++r)
      for (int64_t t = sp.ptr[r]; t < sp.ptr[r + 1]; ++t) by_col[sp.cols[t]].push_back(r);
    std::vector<int32_t> row_rank(rows.n);
    for (int32_t t = 0; t < rows.n; ++t) row_rank[ro[t]] = t;
    for (int32_t b_ = 0; b_ < cols.n; ++b_) {
      const int32_t c = co[b_];
      auto &rs = by_col[c];
      std::sort(rs.begin(), rs.end(), [&](int32_t x, int32_t y) { return row_rank[x] < row_rank[y]; });
      for (int32_t r : rs) {
        bs_block_info b;
        b.row = r;
        b.col = c;
        b.rows = rows.d[r];
        b.cols = cols.d[c];
        b.offset = pos;
        b.ld = width(c);
        pos += (int64_t)rows.d[r] * b.ld;
        if (pos > lim) return BS_ERR_OVERFLOW;
        L->blocks.push_back(b);
      }
    }
  }
  L->nelems = pos;
  // lookup tables
  const int64_t nb = (int64_t)L->blocks.size();
  L->row_ptr.assign(rows.n + 1, 0);
  L->col_ptr.assign(cols.n + 1, 0);
  for (const auto &b : L->blocks) {
    L->row_ptr[b.row + 1]++;
    L->col_ptr[b.col + 1]++;
  }
  for (int32_t t = 0; t < rows.n; ++t) L->row_ptr[t + 1] += L->row_ptr[t];
  for (int32_t t = 0; t < cols.n; ++t) L->col_ptr[t + 1] += L->col_ptr[t];
  L->row_blk.assign(nb, 0);
  L->col_blk.assign(nb, 0);
  std::vector<int64_t> rf(L->row_ptr.begin(), L->row_ptr.end() - 1), cf(L->col_ptr.begin(), L->col_ptr.end() - 1);
  for (int64_t t = 0; t < nb; ++t) {   // storage order is kept inside each row and column list
    L->row_blk[rf[L->blocks[t].row]++] = (int32_t)t;
    L->col_blk[cf[L->blocks[t].col]++] = (int32_t)t;
  }
  L->grid.clear();
  if ((int64_t)rows.n * cols.n <= (int64_t)1 << 24) {
    L->grid.assign((size_t)rows.n * cols.n, -1);
    for (int64_t t = 0; t < nb; ++t) L->grid[(size_t)L->blocks[t].row * cols.n + L->blocks[t].col] = (int32_t)t;
  }
  return BS_OK;
}

}  // namespace bs

int32_t bs_layout::find(int32_t r, int32_t c) const {
  if (!grid.empty()) return grid[(size_t)r * cols.n + c];
  for (int64_t t = row_ptr[r]; t < row_ptr[r + 1]; ++t)
    if (blocks[row_blk[t]].col == c) return row_blk[t];
  return -1;
}

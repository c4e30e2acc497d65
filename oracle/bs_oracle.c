/*
 * Plain CPU oracle for the block-sparse contraction C[i,j] = sum_k A[i,k] B[k,j].
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; the tests, the smoke check and the bench's CPU
 * baseline leg are its only users.  It shares no code, header or table with the
 * CUDA library.
 *
 * What it computes follows the uni20 design note "block coalescing":
 *   - Summary: a block-sparse contraction decomposes into one small dense GEMM
 *     per sector combination, i.e. per populated (row, inner, column) triple;
 *   - "Why single-axis coalescing is hole-free": C[m,n] = sum_k A[m,k] B[k,n]
 *     over block multi-indices;
 *   - "Coalescing is a plan-time transform" and "Decisions made": coalescing is
 *     a lowering that never changes the representation, so the coalesced result
 *     is exactly this plain per-triple sum.
 * The oracle therefore writes that definition out: no grouping, no blocking,
 * no reordering.  Every multiply and add is a separate double operation (the
 * file is compiled with -ffp-contract=off), k ascending, then p ascending.
 *
 * Layouts: the design note expresses every block as a strided view (offset,
 * leading dimension) into one shared buffer ("Expressed as strided views over
 * shared storage") and says the arrangement is chosen per contraction pattern
 * ("Interleaved vs contiguous").  The pages fix no concrete arrangement; the
 * three arrangements below are the library's documented ones, restated here
 * from their written rules.
 *
 * Parity pins (tests/test_oracle.py): dense embedding against a dense matmul,
 * charge conservation, integer-exact brute force, closed forms for all-ones
 * inputs, the one-sector special case, and hand-derived golden fixtures.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BSO_ROWPANEL 1u
#define BSO_COLPANEL 2u
#define BSO_CHARGE_SORTED 4u
#define BSO_ALIGN16 8u
#define BSO_ALIGN64 16u

/* Allowed-charge rule: block (r, c) is populated iff
 * dq_min <= q_r - q_c <= dq_max and, when z2 is set, the parities are equal. */
void bso_rule_mask(int32_t nr, const int32_t *rq, const uint8_t *rp, int32_t nc, const int32_t *cq,
                   const uint8_t *cp, int32_t dq_min, int32_t dq_max, int32_t z2, uint8_t *mask) {
  for (int32_t r = 0; r < nr; ++r) {
    for (int32_t c = 0; c < nc; ++c) {
      int64_t dq = (int64_t)rq[r] - (int64_t)cq[c];
      int ok = dq >= dq_min && dq <= dq_max;
      if (z2 && ok) ok = rp[r] == cp[c];
      mask[(size_t)r * nc + c] = (uint8_t)ok;
    }
  }
}

/* Populated blocks of C: (i, j) such that some k has A[i,k] and B[k,j]. */
void bso_product_mask(int32_t ni, int32_t nk, int32_t nj, const uint8_t *ma, const uint8_t *mb,
                      uint8_t *mc) {
  memset(mc, 0, (size_t)ni * (size_t)nj);
  for (int32_t i = 0; i < ni; ++i)
    for (int32_t k = 0; k < nk; ++k) {
      if (!ma[(size_t)i * nk + k]) continue;
      for (int32_t j = 0; j < nj; ++j)
        if (mb[(size_t)k * nj + j]) mc[(size_t)i * nj + j] = 1;
    }
}

/* Sector order of an axis: by index, or, with CHARGE_SORTED, by
 * (U(1) charge, parity, index) ascending.  Plain insertion sort. */
static void sector_order(int32_t n, const int32_t *q, const uint8_t *p, int sorted, int32_t *order) {
  for (int32_t t = 0; t < n; ++t) order[t] = t;
  if (!sorted) return;
  for (int32_t t = 1; t < n; ++t) {
    int32_t v = order[t];
    int32_t u = t - 1;
    while (u >= 0) {
      int32_t w = order[u];
      int64_t pv = p ? p[v] : 0, pw = p ? p[w] : 0;
      int before = q[v] < q[w] || (q[v] == q[w] && (pv < pw || (pv == pw && v < w)));
      if (!before) break;
      order[u + 1] = w;
      --u;
    }
    order[u + 1] = v;
  }
}

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

/*
 * Offsets and leading dimensions of every populated block, as dense nr x nc
 * tables (off = -1 where the block is absent), in elements.  Rules:
 *   al = 64 / elem_bytes with ALIGN64, else 16 / elem_bytes with ALIGN16,
 *   else 1;  w(c) = d_c rounded up to al.
 *   blockrow : rows in order, then columns in order; each block is row-major
 *              with ld = w(c), placed right after the previous one.
 *   rowpanel : per row sector (in order) one row-major panel of d_r rows whose
 *              columns are the populated blocks in column order, each w(c)
 *              wide; ld = panel width; panels follow each other.
 *   colpanel : per column sector (in order) one row-major panel with ld = w(c)
 *              whose rows are the populated blocks in row order, stacked.
 */
int32_t bso_layout(int32_t nr, const int32_t *rq, const uint8_t *rp, const int32_t *rd, int32_t nc,
                   const int32_t *cq, const uint8_t *cp, const int32_t *cd, const uint8_t *mask,
                   uint32_t flags, int32_t elem_bytes, int64_t *off, int64_t *ld, int64_t *nelems) {
  int64_t al = (flags & BSO_ALIGN64) ? 64 / elem_bytes : (flags & BSO_ALIGN16) ? 16 / elem_bytes : 1;
  int sorted = (flags & BSO_CHARGE_SORTED) != 0;
  int32_t *ro = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nr > 0 ? nr : 1));
  int32_t *co = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nc > 0 ? nc : 1));
  if (!ro || !co) {
    free(ro);
    free(co);
    return -1;
  }
  sector_order(nr, rq, rp, sorted, ro);
  sector_order(nc, cq, cp, sorted, co);
  for (size_t t = 0; t < (size_t)nr * (size_t)nc; ++t) {
    off[t] = -1;
    ld[t] = 0;
  }
  int64_t pos = 0;
  uint32_t mode = flags & 3u;
  if (mode == 0u) {
    for (int32_t a = 0; a < nr; ++a) {
      int32_t r = ro[a];
      for (int32_t b = 0; b < nc; ++b) {
        int32_t c = co[b];
        if (!mask[(size_t)r * nc + c]) continue;
        int64_t w = round_up(cd[c], al);
        off[(size_t)r * nc + c] = pos;
        ld[(size_t)r * nc + c] = w;
        pos += (int64_t)rd[r] * w;
      }
    }
  } else if (mode == BSO_ROWPANEL) {
    for (int32_t a = 0; a < nr; ++a) {
      int32_t r = ro[a];
      int64_t width = 0;
      for (int32_t b = 0; b < nc; ++b) {
        int32_t c = co[b];
        if (mask[(size_t)r * nc + c]) width += round_up(cd[c], al);
      }
      int64_t col = 0;
      for (int32_t b = 0; b < nc; ++b) {
        int32_t c = co[b];
        if (!mask[(size_t)r * nc + c]) continue;
        off[(size_t)r * nc + c] = pos + col;
        ld[(size_t)r * nc + c] = width;
        col += round_up(cd[c], al);
      }
      pos += (int64_t)rd[r] * width;
    }
  } else if (mode == BSO_COLPANEL) {
    for (int32_t b = 0; b < nc; ++b) {
      int32_t c = co[b];
      int64_t w = round_up(cd[c], al);
      for (int32_t a = 0; a < nr; ++a) {
        int32_t r = ro[a];
        if (!mask[(size_t)r * nc + c]) continue;
        off[(size_t)r * nc + c] = pos;
        ld[(size_t)r * nc + c] = w;
        pos += (int64_t)rd[r] * w;
      }
    }
  } else {
    free(ro);
    free(co);
    return -2;
  }
  *nelems = pos;
  free(ro);
  free(co);
  return 0;
}

static double load_value(int32_t dtype, const void *buf, int64_t idx) {
  if (dtype == 0) return ((const double *)buf)[idx];
  /* bfloat16 bits: the upper half of an IEEE single, widened exactly. */
  uint32_t bits = (uint32_t)((const uint16_t *)buf)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/*
 * C[i,j](r,c) = sum over k ascending with A[i,k] and B[k,j] populated, then
 * p = 0 .. d_k-1 ascending, of A[i,k](r,p) * B[k,j](p,c); also
 * S[i,j](r,c) = the same sum of |A| * |B| (the conditioning scale of the sum).
 * A and B are doubles (dtype 0) or bfloat16 bit patterns (dtype 1); C and S
 * are doubles in C's layout.  With nsel > 0 only the listed (i, j) blocks are
 * computed (sel holds i0, j0, i1, j1, ...); otherwise every populated block.
 * Returns the number of blocks computed.
 */
int64_t bso_contract(int32_t ni, int32_t nk, int32_t nj, const int32_t *di, const int32_t *dk,
                     const int32_t *dj, const int64_t *a_off, const int64_t *a_ld,
                     const int64_t *b_off, const int64_t *b_ld, const int64_t *c_off,
                     const int64_t *c_ld, int32_t dtype, const void *A, const void *B, double *C,
                     double *S, int64_t nsel, const int32_t *sel) {
  int64_t done = 0;
  int64_t nblocks = nsel > 0 ? nsel : (int64_t)ni * nj;
  int32_t *klist = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nk > 0 ? nk : 1));
  if (!klist) return -1;
  for (int64_t t = 0; t < nblocks; ++t) {
    int32_t i = nsel > 0 ? sel[2 * t] : (int32_t)(t / nj);
    int32_t j = nsel > 0 ? sel[2 * t + 1] : (int32_t)(t % nj);
    int64_t co = c_off[(size_t)i * nj + j];
    if (co < 0) continue;
    int64_t cl = c_ld[(size_t)i * nj + j];
    /* the inner sectors of this output block, ascending */
    int32_t nkl = 0;
    for (int32_t k = 0; k < nk; ++k)
      if (a_off[(size_t)i * nk + k] >= 0 && b_off[(size_t)k * nj + j] >= 0) klist[nkl++] = k;
    for (int32_t r = 0; r < di[i]; ++r) {
      for (int32_t c = 0; c < dj[j]; ++c) {
        double acc = 0.0;
        double mag = 0.0;
        for (int32_t u = 0; u < nkl; ++u) {
          int32_t k = klist[u];
          int64_t ao = a_off[(size_t)i * nk + k];
          int64_t bo = b_off[(size_t)k * nj + j];
          int64_t al = a_ld[(size_t)i * nk + k];
          int64_t bl = b_ld[(size_t)k * nj + j];
          for (int32_t p = 0; p < dk[k]; ++p) {
            double a = load_value(dtype, A, ao + (int64_t)r * al + p);
            double b = load_value(dtype, B, bo + (int64_t)p * bl + c);
            double prod = a * b;
            acc = acc + prod;
            mag = mag + (prod < 0 ? -prod : prod);
          }
        }
        C[co + (int64_t)r * cl + c] = acc;
        if (S) S[co + (int64_t)r * cl + c] = mag;
      }
    }
    ++done;
  }
  free(klist);
  return done;
}

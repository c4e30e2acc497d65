/*
 * A plain C caller of libbs.so, compiled against include/bs.h only (no CUDA
 * headers): it reads a problem written by tests/test_c_abi.py, builds the
 * layouts and the plan through the C ABI, and either
 *   - (host mode) builds a host-only plan and checks its triple count and C
 *     layout size against the expected ones, or
 *   - (device mode) runs bs_contract_host on the host buffers and checks every
 *     element of C against the oracle's values (integer inputs: exact).
 * Exit status 0 when every check passes.
 *
 * Input file (little-endian): int32 nr, nk, nc; for each of the three axes
 * int32 q[n], int32 d[n]; int32 rule_a[3], rule_b[3]; uint32 flags_a, flags_b,
 * flags_c; int64 triples; int64 na, double A[na]; int64 nb, double B[nb];
 * int64 ncv, double C[ncv].
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "bs.h"

static int read_all(FILE *f, void *dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }

static int32_t *read_i32(FILE *f, int32_t n) {
  int32_t *p = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  if (!p || !read_all(f, p, sizeof(int32_t) * (size_t)n)) exit(3);
  return p;
}

static double *read_f64(FILE *f, int64_t *n) {
  if (!read_all(f, n, sizeof *n)) exit(3);
  double *p = (double *)malloc(sizeof(double) * (size_t)(*n > 0 ? *n : 1));
  if (!p || !read_all(f, p, sizeof(double) * (size_t)*n)) exit(3);
  return p;
}

#define CHECK(call)                                                                   \
  do {                                                                                \
    bs_status s_ = (call);                                                            \
    if (s_ != BS_OK) {                                                                \
      fprintf(stderr, "%s failed: %s (%d)\n", #call, bs_status_string(s_), (int)s_); \
      return 1;                                                                       \
    }                                                                                 \
  } while (0)

int main(int argc, char **argv) {
  if (argc != 3 || (strcmp(argv[1], "host") && strcmp(argv[1], "device"))) {
    fprintf(stderr, "usage: %s host|device problem.bin\n", argv[0]);
    return 2;
  }
  const int device = strcmp(argv[1], "device") == 0;
  FILE *f = fopen(argv[2], "rb");
  if (!f) return 2;
  int32_t n[3];
  if (!read_all(f, n, sizeof n)) return 3;
  int32_t *q[3], *d[3];
  for (int a = 0; a < 3; ++a) {
    q[a] = read_i32(f, n[a]);
    d[a] = read_i32(f, n[a]);
  }
  int32_t ra[3], rb[3];
  uint32_t fl[3];
  int64_t triples = 0;
  if (!read_all(f, ra, sizeof ra) || !read_all(f, rb, sizeof rb) || !read_all(f, fl, sizeof fl) ||
      !read_all(f, &triples, sizeof triples))
    return 3;
  int64_t na = 0, nb = 0, ncv = 0;
  double *A = read_f64(f, &na), *B = read_f64(f, &nb), *Cx = read_f64(f, &ncv);
  fclose(f);

  bs_axis_desc ax[3];
  for (int a = 0; a < 3; ++a) {
    ax[a].n = n[a];
    ax[a].q_u1 = q[a];
    ax[a].q_z2 = NULL;
    ax[a].dim = d[a];
  }
  bs_rule rule_a = {ra[0], ra[1], ra[2]}, rule_b = {rb[0], rb[1], rb[2]};
  bs_layout *LA = NULL, *LB = NULL;
  CHECK(bs_layout_create(&ax[0], &ax[1], &rule_a, fl[0], 8, &LA));
  CHECK(bs_layout_create(&ax[1], &ax[2], &rule_b, fl[1], 8, &LB));
  int64_t nblk = 0, ne_a = 0, ne_b = 0;
  CHECK(bs_layout_query(LA, &nblk, &ne_a));
  CHECK(bs_layout_query(LB, &nblk, &ne_b));
  if (ne_a != na || ne_b != nb) {
    fprintf(stderr, "operand sizes %lld/%lld, expected %lld/%lld\n", (long long)ne_a, (long long)ne_b,
            (long long)na, (long long)nb);
    return 1;
  }
  bs_plan_options o;
  bs_plan_options_default(&o);
  o.c_layout_flags = fl[2];
  o.host_only = device ? 0 : 1;
  bs_plan *P = NULL;
  CHECK(bs_plan_create(LA, LB, BS_F64, &o, &P));
  bs_layout_destroy(LA);   /* the plan keeps its own copies */
  bs_layout_destroy(LB);
  bs_plan_stats st;
  CHECK(bs_plan_stats_get(P, &st));
  int64_t nc_blocks = 0, ne_c = 0;
  CHECK(bs_layout_query(bs_plan_c_layout(P), &nc_blocks, &ne_c));
  if (st.triples != triples || ne_c != ncv) {
    fprintf(stderr, "plan: %lld triples, C of %lld elements; expected %lld and %lld\n", (long long)st.triples,
            (long long)ne_c, (long long)triples, (long long)ncv);
    return 1;
  }
  int64_t bad = 0;
  CHECK(bs_plan_check_groups(P, &bad));
  if (device) {
    double *C = (double *)calloc((size_t)(ncv > 0 ? ncv : 1), sizeof(double));
    if (!C) return 3;
    CHECK(bs_contract_host(P, A, B, C, NULL));
    int64_t wrong = 0;
    for (int64_t e = 0; e < ncv; ++e)
      if (C[e] != Cx[e]) ++wrong;
    if (wrong) {
      fprintf(stderr, "%lld of %lld C elements differ from the oracle\n", (long long)wrong, (long long)ncv);
      return 1;
    }
    free(C);
  }
  bs_plan_destroy(P);
  printf("abi_check %s ok: %lld triples, %lld C blocks, %lld C elements\n", argv[1], (long long)st.triples,
         (long long)nc_blocks, (long long)ncv);
  for (int a = 0; a < 3; ++a) {
    free(q[a]);
    free(d[a]);
  }
  free(A);
  free(B);
  free(Cx);
  return 0;
}

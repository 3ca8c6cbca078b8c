/*
 * threaded.c -- the all-core CPU baseline of the benchmark: the three
 * primitives in fp64 on every host core, fp32 in and fp32 out like the GPU
 * library.  A reported baseline, not the parity reference (that is the
 * single-threaded oracle) and not part of the library.
 *
 * Work split, so that every output keeps a fixed fp64 summation order:
 *   1D sum        contiguous chunks, one per thread, each summed left to
 *                 right; the chunk sums added in chunk order
 *   axis sum      independent outputs: rows (inner == 1) or (o, 256-column
 *                 block) units (inner > 1) split over the threads; each output
 *                 sums its reduce axis in order (r ascending), the columns of
 *                 a block advanced together so x is read row by row
 *   reverse scan  rows split over the threads; a row walked right to left with
 *                 a running fp64 sum.  With fewer rows than threads each row is
 *                 cut into one segment per thread: segment sums, the suffix
 *                 sum of the segment sums in order, then every segment walked
 *                 from its carry
 * The 1D sum follows the "High-Performance Reduction Kernels" README (its
 * benchmark times every backend on one box), the axis sum the POPCORNBENCH
 * trace l1_p47 problem, the scan the POPCORNBENCH trace l1_p91 problem.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef void (*job_fn)(void* ctx, int t, int nt);
typedef struct {
  job_fn fn;
  void* ctx;
  int t, nt;
} worker_arg;

static void* worker(void* p) {
  worker_arg* a = (worker_arg*)p;
  a->fn(a->ctx, a->t, a->nt);
  return NULL;
}

/* Run fn(ctx, t, nt) for t = 0 .. nt-1 on nt threads (t = 0 on the caller). */
static int run_threads(int nt, job_fn fn, void* ctx) {
  if (nt < 1) nt = 1;
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  worker_arg* args = (worker_arg*)calloc((size_t)nt, sizeof(worker_arg));
  if (!th || !args) {
    free(th);
    free(args);
    return -1;
  }
  int started = 1;
  for (int t = 0; t < nt; ++t) args[t] = (worker_arg){fn, ctx, t, nt};
  for (int t = 1; t < nt; ++t) {
    if (pthread_create(&th[t], NULL, worker, &args[t]) != 0) break;
    started = t + 1;
  }
  for (int t = started; t < nt; ++t) args[0].fn(args[0].ctx, t, nt); /* threads that did not start */
  worker(&args[0]);
  for (int t = 1; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  free(args);
  return 0;
}

static int64_t part_lo(int64_t n, int t, int nt) { return n * t / nt; }

/* ---- 1D sum ---------------------------------------------------------------- */
typedef struct {
  const float* x;
  int64_t n;
  double* part;
} sum_ctx;

static void sum_job(void* p, int t, int nt) {
  sum_ctx* c = (sum_ctx*)p;
  const int64_t lo = part_lo(c->n, t, nt), hi = part_lo(c->n, t + 1, nt);
  double s = 0.0;
  for (int64_t i = lo; i < hi; ++i) s += (double)c->x[i];
  c->part[t] = s;
}

int cpub_sum(const float* x, int64_t n, int threads, float* out) {
  double* part = (double*)calloc((size_t)(threads > 0 ? threads : 1), sizeof(double));
  if (!part) return -1;
  sum_ctx c = {x, n, part};
  if (run_threads(threads, sum_job, &c)) {
    free(part);
    return -1;
  }
  double s = 0.0;
  for (int t = 0; t < (threads > 0 ? threads : 1); ++t) s += part[t];
  *out = (float)s;
  free(part);
  return 0;
}

/* ---- axis sum over [outer, reduce, inner] ----------------------------------- */
enum { kColBlock = 256 };
typedef struct {
  const float* x;
  int64_t outer, reduce, inner;
  float* out;
} axis_ctx;

static void axis_job(void* p, int t, int nt) {
  axis_ctx* c = (axis_ctx*)p;
  if (c->inner == 1) {
    const int64_t lo = part_lo(c->outer, t, nt), hi = part_lo(c->outer, t + 1, nt);
    for (int64_t o = lo; o < hi; ++o) {
      const float* row = c->x + o * c->reduce;
      double s = 0.0;
      for (int64_t r = 0; r < c->reduce; ++r) s += (double)row[r];
      c->out[o] = (float)s;
    }
    return;
  }
  const int64_t blocks = (c->inner + kColBlock - 1) / kColBlock;
  const int64_t units = c->outer * blocks;
  const int64_t lo = part_lo(units, t, nt), hi = part_lo(units, t + 1, nt);
  double acc[kColBlock];
  for (int64_t u = lo; u < hi; ++u) {
    const int64_t o = u / blocks, i0 = (u % blocks) * kColBlock;
    const int64_t w = c->inner - i0 < kColBlock ? c->inner - i0 : kColBlock;
    for (int64_t i = 0; i < w; ++i) acc[i] = 0.0;
    for (int64_t r = 0; r < c->reduce; ++r) {
      const float* row = c->x + (o * c->reduce + r) * c->inner + i0;
      for (int64_t i = 0; i < w; ++i) acc[i] += (double)row[i];
    }
    for (int64_t i = 0; i < w; ++i) c->out[o * c->inner + i0 + i] = (float)acc[i];
  }
}

int cpub_axis_sum(const float* x, int64_t outer, int64_t reduce, int64_t inner, int threads, float* out) {
  axis_ctx c = {x, outer, reduce, inner, out};
  return run_threads(threads, axis_job, &c);
}

/* ---- reverse inclusive scan of [rows, N] ------------------------------------ */
typedef struct {
  const float* x;
  int64_t rows, N;
  float* y;
  double* seg; /* one-row form: segment sums, then carries */
} scan_ctx;

static void scan_rows_job(void* p, int t, int nt) {
  scan_ctx* c = (scan_ctx*)p;
  const int64_t lo = part_lo(c->rows, t, nt), hi = part_lo(c->rows, t + 1, nt);
  for (int64_t i = lo; i < hi; ++i) {
    const float* a = c->x + i * c->N;
    float* b = c->y + i * c->N;
    double acc = 0.0;
    for (int64_t j = c->N - 1; j >= 0; --j) {
      acc += (double)a[j];
      b[j] = (float)acc;
    }
  }
}

/* One row in segments: pass 1 sums segment t, pass 2 walks it from its carry. */
static void scan_seg_sum_job(void* p, int t, int nt) {
  scan_ctx* c = (scan_ctx*)p;
  const int64_t lo = part_lo(c->N, t, nt), hi = part_lo(c->N, t + 1, nt);
  double s = 0.0;
  for (int64_t j = hi - 1; j >= lo; --j) s += (double)c->x[j];
  c->seg[t] = s;
}

static void scan_seg_walk_job(void* p, int t, int nt) {
  scan_ctx* c = (scan_ctx*)p;
  const int64_t lo = part_lo(c->N, t, nt), hi = part_lo(c->N, t + 1, nt);
  double acc = c->seg[t]; /* the sum of every segment to the right */
  for (int64_t j = hi - 1; j >= lo; --j) {
    acc += (double)c->x[j];
    c->y[j] = (float)acc;
  }
}

int cpub_reverse_cumsum(const float* x, int64_t rows, int64_t N, int threads, float* y) {
  if (threads < 1) threads = 1;
  if (rows >= threads || threads == 1) {
    scan_ctx c = {x, rows, N, y, NULL};
    return run_threads(threads, scan_rows_job, &c);
  }
  double* seg = (double*)calloc((size_t)threads, sizeof(double));
  if (!seg) return -1;
  for (int64_t i = 0; i < rows; ++i) {
    scan_ctx c = {x + i * N, 1, N, y + i * N, seg};
    if (run_threads(threads, scan_seg_sum_job, &c)) {
      free(seg);
      return -1;
    }
    double carry = 0.0; /* segment t gets the sum of segments t+1 .. threads-1 */
    for (int t = threads - 1; t >= 0; --t) {
      const double s = seg[t];
      seg[t] = carry;
      carry += s;
    }
    if (run_threads(threads, scan_seg_walk_job, &c)) {
      free(seg);
      return -1;
    }
  }
  free(seg);
  return 0;
}

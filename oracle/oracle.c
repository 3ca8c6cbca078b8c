/*
 * oracle.c -- the plain CPU oracle for the three fp32 primitives.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * under reduction_scan_primitives_gb300/csrc and its Python binding) may
 * include, link, load or call this file.  Only the tests, the smoke check and
 * the CPU-baseline leg of the benchmark use it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * Every routine is the written-out definition of what it computes, in fp64,
 * one element at a time, in index order, with no blocking or reordering:
 *
 *   oracle_sum             s = sum_{i<n} x[i]                       (1D sum)
 *   oracle_axis_sum        out[o,i] = sum_r x[o,r,i], r ascending  (axis sum)
 *   oracle_reverse_cumsum  y[i,j] = sum_{k>=j} x[i,k]               (suffix sum)
 *   oracle_cumsum          cumulative sum along the middle axis of [outer, N,
 *                          inner], forward or reverse, inclusive or exclusive
 *   oracle_reduce_op       max, min, mean or Euclidean norm along the middle
 *                          axis of [outer, reduce, inner]
 *
 * Each one also returns the companion sum of |x| over the same terms, which
 * is the scale of the per-element acceptance tolerance
 *     |gpu - ref| <= 1e-5 * sum|x| + 1e-6.
 *
 * Sources, by page:
 *   - "High-Performance Reduction Kernels" (README of a 1D fp32 sum benchmark):
 *     the 1D sum and its synthetic input x[i] = 1/(i+1) ("Layout" section).
 *   - POPCORNBENCH trace l1_p47 (sum over dim=1 of a [128, 4096, 4095] fp32
 *     tensor): the [outer, reduce, inner] view and out[o,i] = sum_r x[o,r,i]
 *     (opening problem statement).
 *   - POPCORNBENCH trace l1_p91 (reverse cumulative sum): y =
 *     cumsum(x.flip(1), 1).flip(1), i.e. y[i,j] = x[i,j] + ... + x[i,N-1]
 *     (opening problem statement); the same trace works an exclusive
 *     (forward) scan of 1..8 by hand, and discusses scanning other dims.
 *   - "Seven-step reduction: 30x from one kernel" (introduction): sum, max,
 *     the softmax denominator, the L2 norm and row sums are all the same
 *     reduction pattern.
 *
 * Build with the host compiler and without -ffast-math, so the sequential
 * fp64 loops are not reassociated (oracle/build.py does this).
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

/* 1D sum: s = x[0] + x[1] + ... + x[n-1], accumulated left to right in fp64. */
void oracle_sum(const float* x, int64_t n, double* sum, double* abs_sum) {
  double s = 0.0;
  double a = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double v = (double)x[i];
    s += v;
    a += fabs(v);
  }
  *sum = s;
  *abs_sum = a;
}

/* Axis sum over the middle axis of a contiguous [outer, reduce, inner] array:
 * out[o*inner + i] = sum over r = 0..reduce-1 of x[(o*reduce + r)*inner + i].
 * An empty reduce axis gives +0.0.  abs_out may be NULL. */
void oracle_axis_sum(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                     double* out, double* abs_out) {
  for (int64_t o = 0; o < outer; ++o) {
    for (int64_t i = 0; i < inner; ++i) {
      double s = 0.0;
      double a = 0.0;
      for (int64_t r = 0; r < reduce; ++r) {
        double v = (double)x[(o * reduce + r) * inner + i];
        s += v;
        a += fabs(v);
      }
      out[o * inner + i] = s;
      if (abs_out) abs_out[o * inner + i] = a;
    }
  }
}

/* Reverse inclusive cumulative sum along each row of a contiguous [rows, N]
 * array: walk a row from its last element to its first, keeping the running
 * sum, and store it at each position, so y[i,j] = x[i,j] + x[i,j+1] + ... +
 * x[i,N-1].  abs_y (may be NULL) gets the running sum of |x| over the same
 * suffix. */
void oracle_reverse_cumsum(const float* x, int64_t rows, int64_t N, double* y,
                           double* abs_y) {
  for (int64_t i = 0; i < rows; ++i) {
    double acc = 0.0;
    double acc_abs = 0.0;
    for (int64_t j = N - 1; j >= 0; --j) {
      double v = (double)x[i * N + j];
      acc += v;
      acc_abs += fabs(v);
      y[i * N + j] = acc;
      if (abs_y) abs_y[i * N + j] = acc_abs;
    }
  }
}

/* Axis sum at a chosen list of flat output positions p = o*inner + i (for
 * checking single outputs of very large inputs).  Same definition as
 * oracle_axis_sum, evaluated only where asked. */
void oracle_axis_sum_at(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                        const int64_t* pos, int64_t m, double* out, double* abs_out) {
  (void)outer;
  for (int64_t k = 0; k < m; ++k) {
    int64_t o = pos[k] / inner;
    int64_t i = pos[k] % inner;
    double s = 0.0;
    double a = 0.0;
    for (int64_t r = 0; r < reduce; ++r) {
      double v = (double)x[(o * reduce + r) * inner + i];
      s += v;
      a += fabs(v);
    }
    out[k] = s;
    if (abs_out) abs_out[k] = a;
  }
}

/* Cumulative sum along the middle axis of a contiguous [outer, N, inner]
 * array, for every (o, i):
 *   forward (reverse == 0):  y[o,j,i] = sum of x[o,k,i] over k <= j
 *   reverse (reverse != 0):  y[o,j,i] = sum of x[o,k,i] over k >= j
 * and with exclusive != 0 the element k == j itself is left out (k < j, or
 * k > j).  Walk the axis in the scan direction with a running fp64 sum; an
 * inclusive result is stored after adding x[o,j,i], an exclusive one before.
 * abs_y (may be NULL) gets the running sum of |x| over the same terms. */
void oracle_cumsum(const float* x, int64_t outer, int64_t N, int64_t inner, int reverse,
                   int exclusive, double* y, double* abs_y) {
  for (int64_t o = 0; o < outer; ++o) {
    for (int64_t i = 0; i < inner; ++i) {
      double acc = 0.0;
      double acc_abs = 0.0;
      for (int64_t step = 0; step < N; ++step) {
        const int64_t j = reverse ? N - 1 - step : step;
        const int64_t idx = (o * N + j) * inner + i;
        const double v = (double)x[idx];
        if (exclusive) {
          y[idx] = acc;
          if (abs_y) abs_y[idx] = acc_abs;
          acc += v;
          acc_abs += fabs(v);
        } else {
          acc += v;
          acc_abs += fabs(v);
          y[idx] = acc;
          if (abs_y) abs_y[idx] = acc_abs;
        }
      }
    }
  }
}

/* Other reductions along the middle axis of a contiguous [outer, reduce,
 * inner] array, one output per (o, i), taken over r = 0..reduce-1 in order:
 *   op 1  mean:  (sum of x) / reduce                  (empty: NaN)
 *   op 2  max:   the largest x, NaN if any x is NaN     (empty: -inf)
 *   op 3  min:   the smallest x, NaN if any x is NaN    (empty: +inf)
 *   op 4  norm:  sqrt(sum of x*x)                     (empty: 0)
 * abs_out (may be NULL) gets the sum of |x| (mean) or of x*x (norm), the
 * scale of the acceptance tolerance; max and min are compared exactly. */
void oracle_reduce_op(const float* x, int64_t outer, int64_t reduce, int64_t inner, int op,
                      double* out, double* abs_out) {
  for (int64_t o = 0; o < outer; ++o) {
    for (int64_t i = 0; i < inner; ++i) {
      double acc = (op == 2) ? -INFINITY : (op == 3) ? INFINITY : 0.0;
      double scale = 0.0;
      for (int64_t r = 0; r < reduce; ++r) {
        const double v = (double)x[(o * reduce + r) * inner + i];
        if (op == 1) {
          acc += v;
          scale += fabs(v);
        } else if (op == 2) {
          if (isnan(v) || isnan(acc)) acc = NAN;
          else if (v > acc) acc = v;
        } else if (op == 3) {
          if (isnan(v) || isnan(acc)) acc = NAN;
          else if (v < acc) acc = v;
        } else {
          acc += v * v;
          scale += v * v;
        }
      }
      double res = acc;
      if (op == 1) res = reduce > 0 ? acc / (double)reduce : NAN;
      if (op == 4) res = sqrt(acc);
      out[o * inner + i] = res;
      if (abs_out) abs_out[o * inner + i] = scale;
    }
  }
}

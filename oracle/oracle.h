/*
 * oracle.h -- declarations of the plain fp64 CPU oracle (test infrastructure
 * only; see oracle.c).  All pointers are host pointers owned by the caller.
 * Arrays are contiguous and row-major.  Sizes are element counts.
 */
#ifndef ORACLE_H_
#define ORACLE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

void oracle_sum(const float* x, int64_t n, double* sum, double* abs_sum);
void oracle_axis_sum(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                     double* out, double* abs_out);
void oracle_reverse_cumsum(const float* x, int64_t rows, int64_t N, double* y,
                           double* abs_y);
void oracle_cumsum(const float* x, int64_t outer, int64_t N, int64_t inner, int reverse,
                   int exclusive, double* y, double* abs_y);
void oracle_reduce_op(const float* x, int64_t outer, int64_t reduce, int64_t inner, int op,
                      double* out, double* abs_out);
void oracle_axis_sum_at(const float* x, int64_t outer, int64_t reduce, int64_t inner,
                        const int64_t* pos, int64_t m, double* out, double* abs_out);

#ifdef __cplusplus
}
#endif

#endif /* ORACLE_H_ */

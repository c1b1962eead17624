/*
 * rra_oracle.c -- CPU oracle for the barrier-free AllReduce.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a separate shared
 * library that only the test-suite, the smoke check and the benchmark's CPU
 * baseline load.  It shares no code, header, table or helper with the CUDA
 * library; the product path never calls it.
 *
 * What it computes (the plain definition of the operation):
 *   "Every Microsecond Matters: Achieving Near Speed-of-Light Latency in GPU
 *   Collectives", Sec. III-A (Low-Latency AllReduce Algorithms): an AllReduce
 *   leaves, in every rank's output, the element-wise reduction of all ranks'
 *   inputs.  The reduction operator here is the sum.
 *
 *       recv[r][i] = round_T( x_0[i] + x_1[i] + ... + x_{N-1}[i] )   for all r
 *
 *   evaluated left to right in rank order p = 0, 1, ..., N-1 (the first term
 *   is taken as is, every later term is added to the running value).  The
 *   running value is binary32 for binary32 and bfloat16 inputs and binary64
 *   for binary64 inputs; for bfloat16 the final binary32 value is rounded to
 *   bfloat16 with round-to-nearest, ties-to-even.  One-shot and two-shot
 *   AllReduce both produce exactly this value when each rank (one-shot) or
 *   each partition owner (two-shot) adds the contributions in rank order.
 *   The LL128-atomic variant adds in an unspecified order; it is compared
 *   against rra_oracle_reference_sum() within an error bound instead.
 *
 * Parity pins (checked by the CPU test-suite, not by re-typing this code):
 *   closed form N(N+1)/2, exact integer sums, an order-sensitive binary32
 *   case, math.fsum error bounds, and torch's bfloat16 conversion.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC -pthread
 * (no FMA contraction, no excess precision).
 */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_FP32 = 0, ORACLE_BF16 = 1, ORACLE_FP64 = 2 };

/* ---- bfloat16 <-> binary32 ------------------------------------------------
 * bfloat16 is the top half of a binary32 bit pattern (1 sign, 8 exponent,
 * 7 fraction bits).  Widening is exact: append 16 zero bits.
 * Narrowing with round-to-nearest, ties-to-even (IEEE 754-2019 Sec. 4.3.1),
 * written from the definition: keep the top 16 bits, then look at the 16
 * discarded bits; more than half an ulp rounds up, less rounds down, exactly
 * half rounds to the candidate whose last kept bit is 0.  Rounding up carries
 * into the exponent naturally, so the largest finite values round to
 * infinity.  NaN stays NaN (made quiet, sign kept).
 */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t rra_oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint32_t exp_bits = u & 0x7F800000u;
    const uint32_t frac_bits = u & 0x007FFFFFu;
    if (exp_bits == 0x7F800000u && frac_bits != 0u) {
        /* NaN: keep sign and the leading fraction bits, force the quiet bit. */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t kept = u >> 16;          /* candidate toward zero */
    uint32_t dropped = u & 0xFFFFu;   /* discarded bits */
    const uint32_t half = 0x8000u;
    if (dropped > half || (dropped == half && (kept & 1u) != 0u)) {
        kept += 1u;                   /* away from zero (magnitude up) */
    }
    return (uint16_t)kept;
}

void rra_oracle_f32_to_bf16_array(const float* in, uint16_t* out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = rra_oracle_f32_to_bf16(in[i]);
}

/* ---- fixed-order sum over ranks, element range [lo, hi) ------------------ */
static void sum_range(int nranks, const void* const* send, void* const* recv,
                      size_t lo, size_t hi, int dtype) {
    if (dtype == ORACLE_FP32) {
        for (size_t i = lo; i < hi; ++i) {
            float acc = ((const float*)send[0])[i];
            for (int p = 1; p < nranks; ++p) acc = acc + ((const float*)send[p])[i];
            for (int r = 0; r < nranks; ++r) ((float*)recv[r])[i] = acc;
        }
    } else if (dtype == ORACLE_BF16) {
        for (size_t i = lo; i < hi; ++i) {
            float acc = bf16_to_f32(((const uint16_t*)send[0])[i]);
            for (int p = 1; p < nranks; ++p)
                acc = acc + bf16_to_f32(((const uint16_t*)send[p])[i]);
            const uint16_t out = rra_oracle_f32_to_bf16(acc);
            for (int r = 0; r < nranks; ++r) ((uint16_t*)recv[r])[i] = out;
        }
    } else {
        for (size_t i = lo; i < hi; ++i) {
            double acc = ((const double*)send[0])[i];
            for (int p = 1; p < nranks; ++p) acc = acc + ((const double*)send[p])[i];
            for (int r = 0; r < nranks; ++r) ((double*)recv[r])[i] = acc;
        }
    }
}

/* Returns 0 on success, -1 on a bad argument.
 * send[p] / recv[r]: host arrays of `count` elements of `dtype`, one per rank.
 * In-place use (recv[r] == send[r]) is allowed: element i of every input is
 * read before element i of any output is written. */
int rra_oracle_allreduce(int nranks, const void* const* send, void* const* recv,
                         size_t count, int dtype) {
    if (nranks < 1 || send == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    if (count == 0) return 0;
    sum_range(nranks, send, recv, 0, count, dtype);
    return 0;
}

/* ---- the same, with the element range split over host threads ----------
 * Each thread owns a contiguous element range and runs the identical
 * per-element loop, so the result does not depend on the thread count.  This
 * is the timed CPU baseline. */
typedef struct {
    int nranks;
    const void* const* send;
    void* const* recv;
    size_t lo, hi;
    int dtype;
} oracle_job;

static void* oracle_worker(void* arg) {
    const oracle_job* j = (const oracle_job*)arg;
    sum_range(j->nranks, j->send, j->recv, j->lo, j->hi, j->dtype);
    return NULL;
}

int rra_oracle_allreduce_mt(int nranks, const void* const* send, void* const* recv,
                            size_t count, int dtype, int nthreads) {
    if (nranks < 1 || send == NULL || recv == NULL || nthreads < 1) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    if (count == 0) return 0;
    if ((size_t)nthreads > count) nthreads = (int)count;
    if (nthreads == 1) {
        sum_range(nranks, send, recv, 0, count, dtype);
        return 0;
    }
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    if (tid == NULL || jobs == NULL) {
        free(tid);
        free(jobs);
        return -1;
    }
    const size_t per = (count + (size_t)nthreads - 1) / (size_t)nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        size_t lo = (size_t)t * per;
        size_t hi = lo + per < count ? lo + per : count;
        if (lo >= hi) break;
        jobs[t] = (oracle_job){nranks, send, recv, lo, hi, dtype};
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) != 0) {
            sum_range(nranks, send, recv, lo, hi, dtype); /* run it here instead */
            tid[t] = (pthread_t)0;
            continue;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (tid[t] != (pthread_t)0) pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
    return 0;
}

/* ---- high-precision reference for error bounds ---------------------------
 * out_sum[i] = x_0[i] + ... + x_{N-1}[i] accumulated in long double (at least
 * binary64; for binary32 and bfloat16 inputs this is far below any binary32
 * rounding error), and out_abs[i] = |x_0[i]| + ... + |x_{N-1}[i]| likewise.
 * Results are returned as double. */
int rra_oracle_reference_sum(int nranks, const void* const* send, size_t count,
                             int dtype, double* out_sum, double* out_abs) {
    if (nranks < 1 || send == NULL || out_sum == NULL || out_abs == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    for (size_t i = 0; i < count; ++i) {
        long double s = 0.0L, a = 0.0L;
        for (int p = 0; p < nranks; ++p) {
            long double x;
            if (dtype == ORACLE_FP32) x = (long double)((const float*)send[p])[i];
            else if (dtype == ORACLE_BF16) x = (long double)bf16_to_f32(((const uint16_t*)send[p])[i]);
            else x = (long double)((const double*)send[p])[i];
            s += x;
            a += x < 0.0L ? -x : x;
        }
        out_sum[i] = (double)s;
        out_abs[i] = (double)a;
    }
    return 0;
}

/* ---- the other collectives ------------------------------------------------
 * "Every Microsecond Matters", Sec. III-A (opening): AllReduce is commonly
 * built as ReduceScatter followed by AllGather, or Reduce followed by
 * Broadcast; the review of the paper (summary) adds that the same
 * barrier-free primitives serve these four collectives.  Their plain
 * definitions, with the sum taken exactly as in sum_range (rank order, the
 * same running type and bfloat16 rounding):
 *
 *   ReduceScatter  send[p] holds N*count elements, recv[r] count:
 *                  recv[r][i] = sum_p send[p][r*count + i]
 *   AllGather      send[p] holds count elements, recv[r] N*count:
 *                  recv[r][p*count + i] = send[p][i]
 *   Broadcast      recv[r][i] = send[root][i]            (every r)
 *   Reduce         recv[root][i] = sum_p send[p][i]      (other outputs untouched)
 *
 * All return 0 on success, -1 on a bad argument.  Outputs must not overlap
 * inputs here (the oracle is not the place to test aliasing). */
static size_t elem_bytes(int dtype) {
    return dtype == ORACLE_FP32 ? 4u : dtype == ORACLE_BF16 ? 2u : 8u;
}

/* Rank-order sum of element i of the N arrays src[p] + off, written to dst. */
static void sum_one(int nranks, const void* const* src, size_t off, size_t i, void* dst, int dtype) {
    if (dtype == ORACLE_FP32) {
        float acc = ((const float*)src[0])[off + i];
        for (int p = 1; p < nranks; ++p) acc = acc + ((const float*)src[p])[off + i];
        ((float*)dst)[i] = acc;
    } else if (dtype == ORACLE_BF16) {
        float acc = bf16_to_f32(((const uint16_t*)src[0])[off + i]);
        for (int p = 1; p < nranks; ++p) acc = acc + bf16_to_f32(((const uint16_t*)src[p])[off + i]);
        ((uint16_t*)dst)[i] = rra_oracle_f32_to_bf16(acc);
    } else {
        double acc = ((const double*)src[0])[off + i];
        for (int p = 1; p < nranks; ++p) acc = acc + ((const double*)src[p])[off + i];
        ((double*)dst)[i] = acc;
    }
}

int rra_oracle_reduce_scatter(int nranks, const void* const* send, void* const* recv,
                              size_t count, int dtype) {
    if (nranks < 1 || send == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    for (int r = 0; r < nranks; ++r)
        for (size_t i = 0; i < count; ++i) sum_one(nranks, send, (size_t)r * count, i, recv[r], dtype);
    return 0;
}

int rra_oracle_all_gather(int nranks, const void* const* send, void* const* recv,
                          size_t count, int dtype) {
    if (nranks < 1 || send == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    const size_t eb = elem_bytes(dtype);
    for (int r = 0; r < nranks; ++r)
        for (int p = 0; p < nranks; ++p)
            memcpy((char*)recv[r] + (size_t)p * count * eb, send[p], count * eb);
    return 0;
}

int rra_oracle_broadcast(int nranks, int root, const void* const* send, void* const* recv,
                         size_t count, int dtype) {
    if (nranks < 1 || root < 0 || root >= nranks || send == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    for (int r = 0; r < nranks; ++r) memcpy(recv[r], send[root], count * elem_bytes(dtype));
    return 0;
}

int rra_oracle_reduce(int nranks, int root, const void* const* send, void* const* recv,
                      size_t count, int dtype) {
    if (nranks < 1 || root < 0 || root >= nranks || send == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    for (size_t i = 0; i < count; ++i) sum_one(nranks, send, 0, i, recv[root], dtype);
    return 0;
}

/* ---- AllReduce with a residual-add epilogue -------------------------------
 * "Every Microsecond Matters" (Abstract; Sec. I, contributions) builds a
 * low-latency device-side API so that custom collective kernels can be
 * written on it.  The custom kernel built here is the AllReduce together
 * with the residual add that follows it in a tensor-parallel transformer
 * layer (the pages' LLM-inference setting): each rank adds its own residual
 * stream to the AllReduce result.  Plain definition used here:
 *
 *   recv[r][i] = round_T( (x_0[i] + x_1[i] + ... + x_{N-1}[i]) + res[r][i] )
 *
 * the rank-order sum in the running type (binary32 for binary32/bfloat16,
 * binary64 for binary64), then the widened residual added to the running
 * value, then one rounding to bfloat16.  Returns 0, or -1 on a bad argument. */
int rra_oracle_allreduce_residual(int nranks, const void* const* send, const void* const* res,
                                  void* const* recv, size_t count, int dtype) {
    if (nranks < 1 || send == NULL || res == NULL || recv == NULL) return -1;
    if (dtype < ORACLE_FP32 || dtype > ORACLE_FP64) return -1;
    for (size_t i = 0; i < count; ++i) {
        for (int r = 0; r < nranks; ++r) {
            if (dtype == ORACLE_FP32) {
                float acc = ((const float*)send[0])[i];
                for (int p = 1; p < nranks; ++p) acc = acc + ((const float*)send[p])[i];
                ((float*)recv[r])[i] = acc + ((const float*)res[r])[i];
            } else if (dtype == ORACLE_BF16) {
                float acc = bf16_to_f32(((const uint16_t*)send[0])[i]);
                for (int p = 1; p < nranks; ++p) acc = acc + bf16_to_f32(((const uint16_t*)send[p])[i]);
                acc = acc + bf16_to_f32(((const uint16_t*)res[r])[i]);
                ((uint16_t*)recv[r])[i] = rra_oracle_f32_to_bf16(acc);
            } else {
                double acc = ((const double*)send[0])[i];
                for (int p = 1; p < nranks; ++p) acc = acc + ((const double*)send[p])[i];
                ((double*)recv[r])[i] = acc + ((const double*)res[r])[i];
            }
        }
    }
    return 0;
}

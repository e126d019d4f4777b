/*
 * tp_peaks.h -- C ABI of libtp_peaks.so: microbenchmarks of the on-chip units that bound the
 * projection kernels of libtp.so, for roofline fractions measured on the same device in the
 * same run.  They compute nothing of the projection method (the pages have no counterpart);
 * the projection kernels' algorithmic work divided by these measured rates gives the
 * "relevant roofline" of each kernel.
 *
 * tp_peak_run enqueues ONE kernel of the given kind on `stream` (a cudaStream_t; NULL = the
 * legacy default stream) with `ctas` CTAs of 256 threads, each running `iters` rounds of its
 * loop, and returns at once; the caller times it with CUDA events on that stream.  `*ops`
 * receives the operations the launch performs (loads, read-modify-writes, reductions or, for
 * TP_PEAK_FMA, floating-point operations) and `*bytes` the bytes those operations move
 * (0 for TP_PEAK_FMA).
 *   scratch        caller-owned device buffer of at least tp_peak_scratch_bytes() bytes,
 *                  256-byte aligned; its contents are overwritten (zero it first so that the
 *                  loads read finite values)
 * Returns 0 on success, 1 for invalid arguments (nothing enqueued), 2 for a launch error.
 * No kernel waits on anything, and every index stays inside the scratch buffer.
 */
#ifndef TP_PEAKS_H
#define TP_PEAKS_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    TP_PEAK_L1_LOAD = 0,         /* coalesced 16-byte loads, L1-resident: data-pipe best case */
    TP_PEAK_L1_GATHER8 = 1,      /* one float2 per lane at random, L1-resident */
    TP_PEAK_L1_GATHER32 = 2,     /* one aligned 32-byte row per lane at random, L1-resident */
    TP_PEAK_SMEM_RMW = 3,        /* shared float2 read-modify-write, 32 consecutive per warp */
    TP_PEAK_SMEM_RMW_RANDOM = 4, /* shared float2 read-modify-write, random per lane */
    TP_PEAK_SMEM_RED = 5,        /* shared red.add.f32, random per lane */
    TP_PEAK_L2_RED = 6,          /* red.global.add.v2.f32, random in an L2-resident 8 MB */
    TP_PEAK_FMA = 7              /* FP32 fused multiply-adds, 8 chains per thread */
};

size_t tp_peak_scratch_bytes(void);

int tp_peak_run(int kind, void* scratch, size_t scratch_bytes, int ctas, int iters,
                void* stream, double* ops, double* bytes);

#ifdef __cplusplus
}
#endif

#endif /* TP_PEAKS_H */

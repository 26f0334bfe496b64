/*
 * tg_probes.h -- peak probes of the two math instruction mixes used by the
 * GEMM, and of the fp16 form of the tensor mix for comparison (measurement
 * helpers; not part of the product path).
 *
 * The roofline discussion of the pages ("PMPP 단권화", roofline card: the
 * knee is peak / bandwidth; "CUDA 성능 최적화", roofline figure) needs the
 * machine's compute ceiling.  These calls launch one kernel each on the
 * current device (compute capability 10.3) and report the floating-point
 * operations it performs; the caller times the launch on `stream` (CUDA
 * events) and divides.  All return TG_ERR_INVALID_VALUE on bad arguments,
 * TG_ERR_UNSUPPORTED_DEVICE on other devices, TG_ERR_CUDA on launch failure.
 */
#ifndef TG_PROBES_H
#define TG_PROBES_H

#include "tg_sgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One CTA per SM; one thread issues iters * 6 tcgen05.mma kind::tf32
 * (M=128, N=256, K=8) on operand tiles resident in shared memory, three per
 * K slice with a commit every six (use_collector != 0: the first two of each
 * three share A through the collector buffer), as the 3xTF32 GEMM does.
 * *tensor_flop receives 2*128*256*8 * 6 * iters * SMs. */
tg_status tg_probe_tf32_mma(int iters, int use_collector, cudaStream_t stream, double* tensor_flop);

/* As tg_probe_tf32_mma without the collector, issuing tcgen05.mma
 * kind::f16 (fp16 A and B, fp32 accumulator, M=128, N=256, K=16: the same
 * 32 bytes of each operand row per MMA as the tf32 form) -- the rate a split
 * of fp32 operands into fp16 halves would be issued at.  Not used by any GEMM
 * path.  *tensor_flop receives 2*128*256*16 * 6 * iters * SMs. */
tg_status tg_probe_f16_mma(int iters, cudaStream_t stream, double* tensor_flop);

/* 8 blocks of 256 threads per SM, each thread running 16 independent fp32
 * FMA chains for `iters` steps.  `sink` is a device float the kernel may write
 * (it never does for finite inputs).  *flop receives 2 * 16 * iters * threads. */
tg_status tg_probe_ffma(int iters, float* sink, cudaStream_t stream, double* flop);

#ifdef __cplusplus
}
#endif

#endif /* TG_PROBES_H */

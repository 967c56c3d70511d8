/*
 * zsynth -- seeded synthetic inputs for the ZeRO step (test and benchmark
 * harness; not part of the optimizer library).
 *
 * Both the host implementation (synth_host.c) and the device implementation
 * (synth_gpu.cu) produce the same values bit for bit.  The generator holds
 * none of the optimizer's arithmetic.
 *
 * Definition (the same on both sides):
 *   Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *   easy as 1, 2, 3", SC'11): multipliers 0xD2511F53 / 0xCD9E8D57, Weyl key
 *   increments 0x9E3779B9 / 0xBB67AE85, ten rounds.
 *   key     = (seed & 0xffffffff, stream)
 *   counter = (q & 0xffffffff, q >> 32, rank, step), q = j >> 1, where j is
 *             the element's index within its tensor (index_offset + local)
 *   element j takes output words 2*(j&1) and 2*(j&1)+1, i.e. four 16-bit
 *   draws u_0..u_3; s = sum_k (2*u_k - 65535) is an Irwin-Hall(4) variate
 *   with mean 0 and standard deviation 65536*sqrt(4/3) (to within 2^-32)
 *   x = (float)s * k, one fp32 rounding; k = (float)(sigma / (65536*sqrt(4/3)))
 *   16-bit outputs are x rounded to nearest-even binary16 or bfloat16.
 *
 * Device functions take device pointers and a cudaStream_t passed as void*;
 * they return 0 or a CUDA error code.
 */
#ifndef ZSYNTH_H
#define ZSYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZSYNTH_FP16 0
#define ZSYNTH_BF16 1

/* host */
void zsynth_host_normal16(uint16_t* dst, int64_t n, int32_t dtype, uint64_t seed, uint32_t stream,
                          uint32_t step, uint32_t rank, int64_t index_offset, float k);
void zsynth_host_normal32(float* dst, int64_t n, uint64_t seed, uint32_t stream, uint32_t step,
                          uint32_t rank, int64_t index_offset, float k);
/* Gather form: values at arbitrary element indices idx[0..n) of one tensor. */
void zsynth_host_normal16_at(uint16_t* dst, int64_t n, const int64_t* idx, int32_t dtype, uint64_t seed,
                             uint32_t stream, uint32_t step, uint32_t rank, float k);
void zsynth_host_normal32_at(float* dst, int64_t n, const int64_t* idx, uint64_t seed, uint32_t stream,
                             uint32_t step, uint32_t rank, float k);
void zsynth_host_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* device */
int zsynth_dev_normal16(void* dst, int64_t n, int32_t dtype, uint64_t seed, uint32_t stream,
                        uint32_t step, uint32_t rank, int64_t index_offset, float k, void* cuda_stream);
int zsynth_dev_normal32(float* dst, int64_t n, uint64_t seed, uint32_t stream, uint32_t step,
                        uint32_t rank, int64_t index_offset, float k, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif

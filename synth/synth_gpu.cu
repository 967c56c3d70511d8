// Device implementation of the zsynth generator (definition in zsynth.h).
// Harness code: fills benchmark and test inputs in HBM; the optimizer library
// does not use it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zsynth.h"

namespace {

__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; round++) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

__device__ __forceinline__ int32_t ih4(uint32_t a, uint32_t b)
{
    return (int32_t)(2 * (a & 0xffffu)) - 65535 + (int32_t)(2 * (a >> 16)) - 65535 +
           (int32_t)(2 * (b & 0xffffu)) - 65535 + (int32_t)(2 * (b >> 16)) - 65535;
}

struct GenArgs {
    void* dst;
    int64_t n;
    int64_t offset;
    uint32_t key0, key1, rank, step;
    float k;
    int32_t kind;   // 0 fp16, 1 bf16, 2 fp32
};

__device__ __forceinline__ uint32_t to_bits(float x, int kind)
{
    if (kind == 1)
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    if (kind == 0)
        return __half_as_ushort(__float2half_rn(x));
    return __float_as_uint(x);
}

// One thread per pair of tensor indices (2q, 2q+1): one Philox call each.
__global__ void gen_kernel(GenArgs a)
{
    const int64_t first_q = a.offset >> 1;
    const int64_t last_q = (a.offset + a.n - 1) >> 1;
    for (int64_t q = first_q + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q <= last_q;
         q += (int64_t)gridDim.x * blockDim.x) {
        uint32_t c[4] = {(uint32_t)q, (uint32_t)((uint64_t)q >> 32), a.rank, a.step};
        philox(c, a.key0, a.key1);
        float x0 = (float)ih4(c[0], c[1]) * a.k;
        float x1 = (float)ih4(c[2], c[3]) * a.k;
        int64_t j0 = 2 * q - a.offset;   // local index of tensor index 2q
        int64_t j1 = j0 + 1;
        if (a.kind == 2) {
            float* d = (float*)a.dst;
            if (j0 >= 0 && j0 < a.n) d[j0] = x0;
            if (j1 >= 0 && j1 < a.n) d[j1] = x1;
        } else {
            uint16_t* d = (uint16_t*)a.dst;
            if (j0 >= 0 && j0 < a.n) d[j0] = (uint16_t)to_bits(x0, a.kind);
            if (j1 >= 0 && j1 < a.n) d[j1] = (uint16_t)to_bits(x1, a.kind);
        }
    }
}

int launch(GenArgs a, void* stream)
{
    if (a.n <= 0)
        return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t pairs = ((a.offset + a.n - 1) >> 1) - (a.offset >> 1) + 1;
    int64_t blocks = (pairs + 255) / 256;
    int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap)
        blocks = cap;
    gen_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace

extern "C" int zsynth_dev_normal16(void* dst, int64_t n, int32_t dtype, uint64_t seed, uint32_t stream,
                                   uint32_t step, uint32_t rank, int64_t index_offset, float k,
                                   void* cuda_stream)
{
    GenArgs a{dst, n, index_offset, (uint32_t)seed, stream, rank, step, k, dtype == ZSYNTH_BF16 ? 1 : 0};
    return launch(a, cuda_stream);
}

extern "C" int zsynth_dev_normal32(float* dst, int64_t n, uint64_t seed, uint32_t stream, uint32_t step,
                                   uint32_t rank, int64_t index_offset, float k, void* cuda_stream)
{
    GenArgs a{dst, n, index_offset, (uint32_t)seed, stream, rank, step, k, 2};
    return launch(a, cuda_stream);
}

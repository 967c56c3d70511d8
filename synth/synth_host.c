/* Host implementation of the zsynth generator (definition in zsynth.h). */
#include <stdint.h>
#include <string.h>

#include "zsynth.h"

void zsynth_host_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

static float draw(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank, int64_t j, float k)
{
    uint64_t q = (uint64_t)j >> 1;
    uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), rank, step};
    uint32_t key[2] = {(uint32_t)seed, stream};
    uint32_t o[4];
    zsynth_host_philox4x32_10(ctr, key, o);
    uint32_t a = o[2 * (j & 1)], b = o[2 * (j & 1) + 1];
    int32_t s = (int32_t)(2 * (a & 0xffff)) - 65535 + (int32_t)(2 * (a >> 16)) - 65535 +
                (int32_t)(2 * (b & 0xffff)) - 65535 + (int32_t)(2 * (b >> 16)) - 65535;
    return (float)s * k;
}

static uint16_t to16(float x, int32_t dtype)
{
    if (dtype == ZSYNTH_BF16) {
        uint32_t u;
        memcpy(&u, &x, 4);
        if ((u & 0x7fffffffu) > 0x7f800000u)
            return (uint16_t)((u >> 16) | 0x40);          /* quiet NaN */
        u += 0x7fffu + ((u >> 16) & 1u);                  /* nearest, ties to even */
        return (uint16_t)(u >> 16);
    }
    _Float16 h = (_Float16)x;                             /* nearest, ties to even */
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

void zsynth_host_normal16(uint16_t* dst, int64_t n, int32_t dtype, uint64_t seed, uint32_t stream,
                          uint32_t step, uint32_t rank, int64_t index_offset, float k)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = to16(draw(seed, stream, step, rank, index_offset + i, k), dtype);
}

void zsynth_host_normal32(float* dst, int64_t n, uint64_t seed, uint32_t stream, uint32_t step,
                          uint32_t rank, int64_t index_offset, float k)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = draw(seed, stream, step, rank, index_offset + i, k);
}

void zsynth_host_normal16_at(uint16_t* dst, int64_t n, const int64_t* idx, int32_t dtype, uint64_t seed,
                             uint32_t stream, uint32_t step, uint32_t rank, float k)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = to16(draw(seed, stream, step, rank, idx[i], k), dtype);
}

void zsynth_host_normal32_at(float* dst, int64_t n, const int64_t* idx, uint64_t seed, uint32_t stream,
                             uint32_t step, uint32_t rank, float k)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = draw(seed, stream, step, rank, idx[i], k);
}

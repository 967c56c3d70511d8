// Device helpers shared by the step kernels: the model-precision formats
// (binary16, bfloat16, and binary32 for fp32 training), vector memory access
// with streaming cache hints, the optimizer element updates and the exact
// sum-of-squares accumulator.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "zero_internal.h"

namespace zg {

enum { kF16 = ZERO_FP16, kBF16 = ZERO_BF16, kF32 = ZERO_FP32 };

// ---- model-precision formats -------------------------------------------------
// Gradients and parameters are binary16 or bfloat16 bit patterns in mixed
// precision, binary32 in fp32 training (where widening and narrowing are the
// identity).
template <int DT>
__device__ __forceinline__ float to_f32(uint32_t bits)
{
    if constexpr (DT == kF32)
        return __uint_as_float(bits);
    else if constexpr (DT == kBF16)
        return __uint_as_float(bits << 16);
    else
        return __half2float(__ushort_as_half((unsigned short)bits));
}

// Round to nearest even.
template <int DT>
__device__ __forceinline__ uint32_t from_f32(float x)
{
    if constexpr (DT == kF32)
        return __float_as_uint(x);
    else if constexpr (DT == kBF16)
        return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else
        return __half_as_ushort(__float2half_rn(x));
}

// Two 16-bit values packed in a word (element 2p in the low half).
template <int DT>
__device__ __forceinline__ float2 to_f32x2(uint32_t w)
{
    if constexpr (DT == kBF16)
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    else
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Round two floats to nearest even and pack them (lo in the low half).
template <int DT>
__device__ __forceinline__ uint32_t from_f32x2(float lo, float hi)
{
    if constexpr (DT == kBF16) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&b);
    } else {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Nonzero if either packed value has an all-ones exponent (inf or NaN):
// adding one exponent LSB to the masked exponent carries into the sign bit
// only then, and never across the two halves.
template <int DT>
__device__ __forceinline__ uint32_t nonfinite_x2(uint32_t w)
{
    if constexpr (DT == kBF16)
        return ((w & 0x7f807f80u) + 0x00800080u) & 0x80008000u;
    else
        return ((w & 0x7c007c00u) + 0x04000400u) & 0x80008000u;
}

// ---- consecutive bucket kernels ---------------------------------------------
// Inside one step the library launches the bucket kernels back to back with
// programmatic dependent launch.  Each bucket kernel lets the next one be
// scheduled once all of its own blocks have started (so the next kernel's
// blocks fill the SMs this one's finished blocks free, hiding its ramp-up
// behind this one's tail), and waits for its predecessor to complete at its
// very end, so kernels still complete in stream order.  Bucket kernels of one
// step touch disjoint elements; the flag and the sums they share are
// atomics.  Without the launch attribute both instructions have no effect.
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prev_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- groups of elements ------------------------------------------------------
// A group is VEC consecutive flat elements starting at a multiple of VEC:
// 8 for 16-bit value types (one 16-byte access per gradient or parameter
// array, two per fp32 state array), 4 for binary32 values (one 16-byte
// access per array).  Measured on GB300, 4-element groups lift the binary32
// steps from 0.91-0.94 to 0.99 of the copy bandwidth (every warp access a
// contiguous 512 bytes) but drop the 16-bit Adam step from 1.01 to 0.90.
// The ragged last group of a bucket uses scalar accesses for its cnt < VEC
// elements.
template <int DT>
constexpr int kVecOf = DT == kF32 ? 4 : 8;

// V 16-bit values, little-endian pairs.
template <int V>
struct H16 {
    uint32_t w[V / 2];
    __device__ __forceinline__ uint32_t get(int j) const { return (w[j >> 1] >> ((j & 1) * 16)) & 0xffffu; }
    __device__ __forceinline__ void set(int j, uint32_t b)
    {
        const int s = (j & 1) * 16;
        w[j >> 1] = (w[j >> 1] & ~(0xffffu << s)) | ((b & 0xffffu) << s);
    }
};

// V binary32 values, as bit patterns.
template <int V>
struct W32 {
    uint32_t w[V];
    __device__ __forceinline__ uint32_t get(int j) const { return w[j]; }
    __device__ __forceinline__ void set(int j, uint32_t b) { w[j] = b; }
};

// A group of model-precision values.
template <int DT>
using Vals = typename std::conditional<DT == kF32, W32<kVecOf<DT>>, H16<kVecOf<DT>>>::type;

template <int V>
__device__ __forceinline__ H16<V> ld_h16(const void* base, int64_t idx, int cnt)
{
    static_assert(V == 8, "16-bit groups are 8 values, one 16-byte access");
    const uint16_t* p = static_cast<const uint16_t*>(base) + idx;
    H16<V> r;
    if (cnt == V) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    } else {
        r.w[0] = r.w[1] = r.w[2] = r.w[3] = 0;
#pragma unroll
        for (int j = 0; j < V; j++)
            if (j < cnt) r.set(j, p[j]);
    }
    return r;
}

template <int V>
__device__ __forceinline__ void st_h16(void* base, int64_t idx, const H16<V>& h, int cnt)
{
    uint16_t* p = static_cast<uint16_t*>(base) + idx;
    if (cnt == V) {
        __stcs(reinterpret_cast<uint4*>(p), make_uint4(h.w[0], h.w[1], h.w[2], h.w[3]));
    } else {
#pragma unroll
        for (int j = 0; j < V; j++)
            if (j < cnt) p[j] = (uint16_t)h.get(j);
    }
}

// V 32-bit words (binary32 values or fp32 state), one 16-byte access per 4.
template <int V>
__device__ __forceinline__ void ld_u32(const void* base, int64_t idx, int cnt, uint32_t x[V])
{
    const uint32_t* p = static_cast<const uint32_t*>(base) + idx;
    if (cnt == V) {
#pragma unroll
        for (int k = 0; k < V / 4; k++) {
            const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p) + k);
            x[4 * k] = a.x; x[4 * k + 1] = a.y; x[4 * k + 2] = a.z; x[4 * k + 3] = a.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; j++)
            x[j] = j < cnt ? p[j] : 0u;
    }
}

template <int V>
__device__ __forceinline__ void st_u32(void* base, int64_t idx, int cnt, const uint32_t x[V])
{
    uint32_t* p = static_cast<uint32_t*>(base) + idx;
    if (cnt == V) {
#pragma unroll
        for (int k = 0; k < V / 4; k++)
            __stcs(reinterpret_cast<uint4*>(p) + k, make_uint4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]));
    } else {
#pragma unroll
        for (int j = 0; j < V; j++)
            if (j < cnt) p[j] = x[j];
    }
}

template <int DT>
__device__ __forceinline__ Vals<DT> ld_vals(const void* base, int64_t idx, int cnt)
{
    if constexpr (DT == kF32) {
        Vals<DT> r;
        ld_u32<kVecOf<DT>>(base, idx, cnt, r.w);
        return r;
    } else {
        return ld_h16<kVecOf<DT>>(base, idx, cnt);
    }
}

template <int DT>
__device__ __forceinline__ void st_vals(void* base, int64_t idx, const Vals<DT>& v, int cnt)
{
    if constexpr (DT == kF32)
        st_u32<kVecOf<DT>>(base, idx, cnt, v.w);
    else
        st_h16<kVecOf<DT>>(base, idx, v, cnt);
}

template <int V>
__device__ __forceinline__ void ld_f(const float* base, int64_t idx, int cnt, float x[V])
{
    uint32_t u[V];
    ld_u32<V>(base, idx, cnt, u);
#pragma unroll
    for (int j = 0; j < V; j++)
        x[j] = __uint_as_float(u[j]);
}

template <int V>
__device__ __forceinline__ void st_f(float* base, int64_t idx, int cnt, const float x[V])
{
    uint32_t u[V];
#pragma unroll
    for (int j = 0; j < V; j++)
        u[j] = __float_as_uint(x[j]);
    st_u32<V>(base, idx, cnt, u);
}

// Nonzero if the binary32 pattern is inf or NaN.
__device__ __forceinline__ uint32_t nonfinite32(uint32_t b) { return (~b & 0x7f800000u) == 0u; }

// h = the fp32 sums s in the model precision (one rounding to nearest even
// for 16-bit types, none for binary32); returns nonzero if any element of h
// is inf or NaN.  Elements past cnt are 0: finite.
template <int DT>
__device__ __forceinline__ uint32_t round_group(const float s[kVecOf<DT>], Vals<DT>& h)
{
    constexpr int V = kVecOf<DT>;
    uint32_t nf = 0;
    if constexpr (DT == kF32) {
#pragma unroll
        for (int j = 0; j < V; j++) {
            h.w[j] = __float_as_uint(s[j]);
            nf |= nonfinite32(h.w[j]);
        }
    } else {
#pragma unroll
        for (int p = 0; p < V / 2; p++) {
            h.w[p] = from_f32x2<DT>(s[2 * p], s[2 * p + 1]);
            nf |= nonfinite_x2<DT>(h.w[p]);
        }
    }
    return nf;
}

// g = float(h) * inv, elementwise.
template <int DT>
__device__ __forceinline__ void unscale_group(const Vals<DT>& h, float inv, float g[kVecOf<DT>])
{
    constexpr int V = kVecOf<DT>;
    if constexpr (DT == kF32) {
#pragma unroll
        for (int j = 0; j < V; j++)
            g[j] = __fmul_rn(__uint_as_float(h.w[j]), inv);
    } else {
#pragma unroll
        for (int p = 0; p < V / 2; p++) {
            const float2 f = to_f32x2<DT>(h.w[p]);
            g[2 * p] = __fmul_rn(f.x, inv);
            g[2 * p + 1] = __fmul_rn(f.y, inv);
        }
    }
}

// Rank-order fp32 sum of the N ranks' gradients for one group:
// s[j] = (((0 + g_0[j]) + g_1[j]) + ...) + g_{N-1}[j].  Loads are issued in
// batches of 8 ranks, i.e. 128 bytes in flight per thread (8 x 16 bytes of
// 16-bit values, or 8 x 16 bytes of binary32 values).
template <int DT>
__device__ __forceinline__ void reduce_group(const StepArgs& a, int64_t gidx, int cnt, float s[kVecOf<DT>])
{
    constexpr int V = kVecOf<DT>;
    constexpr int kB = 8;
#pragma unroll
    for (int j = 0; j < V; j++)
        s[j] = 0.0f;
    for (int r0 = 0; r0 < a.n_ranks; r0 += kB) {
        Vals<DT> q[kB];
#pragma unroll
        for (int k = 0; k < kB; k++)
            if (r0 + k < a.n_ranks)
                q[k] = ld_vals<DT>(a.grads[r0 + k], gidx, cnt);
#pragma unroll
        for (int k = 0; k < kB; k++) {
            if (r0 + k < a.n_ranks) {
                if constexpr (DT == kF32) {
#pragma unroll
                    for (int j = 0; j < V; j++)
                        s[j] = __fadd_rn(s[j], __uint_as_float(q[k].w[j]));
                } else {
#pragma unroll
                    for (int p = 0; p < V / 2; p++) {
                        const float2 f = to_f32x2<DT>(q[k].w[p]);
                        s[2 * p] = __fadd_rn(s[2 * p], f.x);
                        s[2 * p + 1] = __fadd_rn(s[2 * p + 1], f.y);
                    }
                }
            }
        }
    }
}

// Adam (Kingma & Ba, Algorithm 1) on one element, one IEEE rounding per
// operation in this order:
//   m' = b1*m + (1-b1)*g;  v' = b2*v + (1-b2)*(g*g)
//   w' = w - lr * ((m'/bc1) / (sqrt(v'/bc2) + eps))
__device__ __forceinline__ void adam1(float g, float& w, float& m, float& v, const AdamHP& hp)
{
    const float t1 = __fmul_rn(hp.b1, m);
    const float t2 = __fmul_rn(hp.omb1, g);
    const float m1 = __fadd_rn(t1, t2);
    const float t3 = __fmul_rn(g, g);
    const float t4 = __fmul_rn(hp.omb2, t3);
    const float t5 = __fmul_rn(hp.b2, v);
    const float v1 = __fadd_rn(t5, t4);
    const float mh = __fdiv_rn(m1, hp.bc1);
    const float vh = __fdiv_rn(v1, hp.bc2);
    const float d = __fadd_rn(__fsqrt_rn(vh), hp.eps);
    const float u = __fdiv_rn(mh, d);
    const float st = __fmul_rn(hp.lr, u);
    w = __fsub_rn(w, st);
    m = m1;
    v = v1;
}

// SGD with momentum (PyTorch's rule, no dampening): m' = mu*m + g; w' = w - lr*m'.
__device__ __forceinline__ void sgdm1(float g, float& w, float& m, const AdamHP& hp)
{
    const float t1 = __fmul_rn(hp.mu, m);
    const float m1 = __fadd_rn(t1, g);
    const float st = __fmul_rn(hp.lr, m1);
    w = __fsub_rn(w, st);
    m = m1;
}

// Plain SGD: w' = w - lr*g.
__device__ __forceinline__ void sgd1(float g, float& w, const AdamHP& hp)
{
    w = __fsub_rn(w, __fmul_rn(hp.lr, g));
}

// The optimizer update of one group: load the fp32 state the optimizer keeps
// at state index si (w; m; v), update it with the unscaled gradients g,
// store it to the output state and give back the model-precision cast in p.
template <int DT, int OPT>
__device__ __forceinline__ void update_state(const StepArgs& a, const AdamHP& hp, int64_t si, int cnt,
                                             const float g[kVecOf<DT>], Vals<DT>& p)
{
    constexpr int V = kVecOf<DT>;
    float w[V];
    ld_f<V>(a.w_in, si, cnt, w);
    if constexpr (OPT == kAdam) {
        float m[V], v[V];
        ld_f<V>(a.m_in, si, cnt, m);
        ld_f<V>(a.v_in, si, cnt, v);
#pragma unroll
        for (int j = 0; j < V; j++)
            adam1(g[j], w[j], m[j], v[j], hp);
        st_f<V>(a.m_out, si, cnt, m);
        st_f<V>(a.v_out, si, cnt, v);
    } else if constexpr (OPT == kSgdm) {
        float m[V];
        ld_f<V>(a.m_in, si, cnt, m);
#pragma unroll
        for (int j = 0; j < V; j++)
            sgdm1(g[j], w[j], m[j], hp);
        st_f<V>(a.m_out, si, cnt, m);
    } else {
#pragma unroll
        for (int j = 0; j < V; j++)
            sgd1(g[j], w[j], hp);
    }
#pragma unroll
    for (int j = 0; j < V; j++)
        p.set(j, from_f32<DT>(w[j]));
    st_f<V>(a.w_out, si, cnt, w);
}

// ---- exact sum of squares --------------------------------------------------
// A finite 16-bit value is h = M * 2^E with integer M (< 2^11 binary16,
// < 2^8 bfloat16), so h^2 = M^2 * 2^(2E) exactly.  Terms with
// 0 <= 2(E - win_lo) <= 63 are added, shifted, into a 128-bit fixed-point
// accumulator with unit 2^(2 win_lo); the others (rare: a 33-binade window
// covers every binary16 value and the usual bfloat16 gradient range) go to
// per-exponent integer bins in the workspace.  Integer sums are exact and
// independent of order.
struct U128 {
    unsigned long long lo, hi;
};

__device__ __forceinline__ void u128_add(U128& a, unsigned long long lo, unsigned long long hi)
{
    asm("add.cc.u64 %0, %0, %2;\n\taddc.u64 %1, %1, %3;" : "+l"(a.lo), "+l"(a.hi) : "l"(lo), "l"(hi));
}

template <int DT>
__device__ __forceinline__ void sumsq_add(uint32_t bits, int win_lo, U128& acc, unsigned long long* bins)
{
    // Non-finite values are not skipped: they set the step's overflow flag,
    // and an overflowed step discards the norm.
    if constexpr (DT == kBF16) {
        // in the window when 0 <= sh <= 63: the same two shifts as binary16
        // below, with no special case (sh = 64 goes to its bin)
        const uint32_t e = (bits >> 7) & 0xffu;
        const uint32_t M = (bits & 0x7fu) | (e ? 0x80u : 0u);
        const int sh = 2 * ((int)(e ? e : 1u) - 134 - win_lo);
        const unsigned long long m2 = (unsigned long long)(M * M);
        if ((unsigned)sh <= 63u) {
            const unsigned long long lo = m2 << sh;
            const unsigned long long hi = (m2 >> 1) >> (63 - sh);   // 0 when sh == 0
            u128_add(acc, lo, hi);
        } else if (m2) {
            atomicAdd(bins + e, m2);
        }
    } else {
        // binary16: the window starts at the smallest subnormal (win_lo = -24),
        // so every square lands in it at shift sh = 2*(max(e,1) - 1) <= 60.
        const uint32_t e = (bits >> 10) & 0x1fu;
        const uint32_t M = (bits & 0x3ffu) | (e ? 0x400u : 0u);
        const int sh = 2 * (int)((e ? e : 1u) - 1u);
        const unsigned long long m2 = (unsigned long long)(M * M);
        const unsigned long long lo = m2 << sh;
        const unsigned long long hi = (m2 >> 1) >> (63 - sh);   // 0 when sh == 0
        u128_add(acc, lo, hi);
    }
}

// The two binary16 squares of a packed word, as sumsq_add<kF16> for each
// half, with the field extraction done by multiplications (the integer
// multiplier, not the shift and logic unit the rest of this work keeps
// busy): x >> k as the high word of x * 2^(32 - k); the hidden bit as
// (e + 31) >> 5, which is 1 exactly when e > 0; max(e, 1) - 1 as e - hidden.
__device__ __forceinline__ void sumsq_add_f16x2(uint32_t w, U128& acc)
{
    const uint32_t e[2] = {__umulhi(w & 0x00007c00u, 1u << 22), __umulhi(w & 0x7c000000u, 1u << 6)};
    const uint32_t f[2] = {w & 0x000003ffu, __umulhi(w & 0x03ff0000u, 1u << 16)};
#pragma unroll
    for (int k = 0; k < 2; k++) {
        const uint32_t hid = __umulhi(e[k] + 31u, 1u << 27);
        const uint32_t M = f[k] + hid * 0x400u;
        const int sh = 2 * (int)(e[k] - hid);
        const unsigned long long m2 = (unsigned long long)(M * M);
        u128_add(acc, m2 << sh, (m2 >> 1) >> (63 - sh));
    }
}

// Nonzero (in bit 15 or 31) if a binary16 value of the packed pair has an
// exponent field of 20 or more -- |h| >= 32, inf or NaN: adding 12 to the
// masked field carries into the half's top bit exactly then, never across the
// halves.
__device__ __forceinline__ uint32_t f16x2_exp_ge20(uint32_t w)
{
    return ((w & 0x7c007c00u) + 0x30003000u) & 0x80008000u;
}

// The squares of one group of 8 binary16 values, when no exponent field is 20
// or more (f16x2_exp_ge20 of every word is 0; the caller checks).  A value
// with exponent field e and mantissa f is h = X * 2^-24 with X = M << E',
// M = f + 1024 [e > 0], E' = max(e, 1) - 1, so h^2 = X^2 * 2^-48 in the
// accumulator's unit.  With e <= 19, X < 2^29 and X^2 < 2^58: the group's
// eight squares add up in 64 bits, one multiply-add each on the integer
// multiplier, then one 128-bit add.  The same integer as sumsq_add_f16x2.
__device__ __forceinline__ void sumsq_group_f16_small(const H16<8>& h, U128& acc)
{
    unsigned long long s = 0ull;
#pragma unroll
    for (int p = 0; p < 4; p++) {
        const uint32_t w = h.w[p];
        // fields by multiplications, as in sumsq_add_f16x2
        const uint32_t e[2] = {__umulhi(w & 0x00007c00u, 1u << 22), __umulhi(w & 0x7c000000u, 1u << 6)};
        const uint32_t f[2] = {w & 0x000003ffu, __umulhi(w & 0x03ff0000u, 1u << 16)};
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const uint32_t hid = min(e[k], 1u);
            const uint32_t X = (f[k] + hid * 0x400u) << (e[k] - hid);
            asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(s) : "r"(X));
        }
    }
    u128_add(acc, s, 0ull);
}

// The squares of one group of 8 binary16 values into the accumulator; sets
// `bad` if one is inf or NaN.  Groups whose values all lie below 32 in
// magnitude (gradients almost always do) take sumsq_group_f16_small; the
// others the per-value path and the inf/NaN test.
__device__ __forceinline__ void sumsq_group_f16(const H16<8>& h, U128& acc, bool& bad)
{
    uint32_t big = 0;
#pragma unroll
    for (int p = 0; p < 4; p++)
        big |= f16x2_exp_ge20(h.w[p]);
    if (!big) {
        sumsq_group_f16_small(h, acc);
        return;
    }
#pragma unroll
    for (int p = 0; p < 4; p++) {
        bad |= nonfinite_x2<kF16>(h.w[p]) != 0;
        sumsq_add_f16x2(h.w[p], acc);
    }
}

// The squares of one group of 8 bfloat16 values.  Each square is M^2 *
// 2^(2(e - 134)) with M < 2^8 and e = max(exponent field, 1); in units of
// 2^(2(base - 134)), with base = max(e_max - 22, the window's first
// exponent), a square is (M << (e - base))^2 < 2^60, and the group's 8 of
// them add up exactly in 64 bits.  The sum then goes into the 128-bit accumulator
// with one shifted add, at window shift 2(base - first) <= 62.  A group with
// a nonzero value below base, or whose largest value lies above the window,
// takes the per-value path above instead (the same exact integer).  Fewer
// integer instructions per value than the per-value bfloat16 path, whose
// window test and shifted 128-bit adds form one dependent chain: measured on
// GB300, N_d = 2, clipped two-pass step, 0.846 -> 0.864 of the copy
// bandwidth (binary16 groups have their own form, sumsq_group_f16).
__device__ __forceinline__ void sumsq_group_bf16(const H16<8>& h, int win_lo, U128& acc, unsigned long long* bins)
{
    constexpr int kD = 22;                           // binades below the group's largest value
    const int first = win_lo + 134;                  // e of the window's first binade
    {
        // First a fixed window: when every nonzero value of the group has e
        // in [first + 9, first + 31] -- the top 23 binades of the
        // accumulator's window, which is placed by S * N_d so that these
        // hold mean gradients of magnitude about 2^-23 to 1 -- each square
        // is X^2 * 2^18 units with X = M << (e - first - 9) < 2^30: one
        // multiply-add per value, no group maximum, one add at a constant
        // shift.  Subnormals (e = 0, first >= 1) and inf and NaN (e = 255,
        // first <= 222) always lie outside it.
        // Two values per 32-bit word at once: with m = |x|'s 15 bits, bit 15
        // of m + (0x8000 - lim) is set iff m >= lim (no carry between the
        // halves, m < 0x8000), which tests both ends of the window and
        // m != 0; M = f | 0x80 for both halves in one operation (in the
        // window the values are normal), and the shift is PTX shl, whose
        // shift counts of 32 or more give 0, so a zero (e = 0, shift count
        // 0 - fbase, wrapped) adds nothing.  tests/test_bf16_window_bits.py checks
        // this against the value-by-value form for every 16-bit pattern.
        const uint32_t fbase = (uint32_t)(first + 9);                       // 10..231
        const uint32_t k_hi = (0x8000u - ((fbase + 23u) << 7)) * 0x00010001u;
        const uint32_t k_lo = (0x8000u - (fbase << 7)) * 0x00010001u;
        unsigned long long b = 0ull;
        uint32_t outside = 0;
#pragma unroll
        for (int p = 0; p < 4; p++) {
            const uint32_t w = h.w[p];
            const uint32_t mag = w & 0x7fff7fffu;
            outside |= (mag + k_hi) | ((mag + 0x7fff7fffu) & ~(mag + k_lo));
            const uint32_t m2 = (w & 0x007f007fu) | 0x00800080u;
            const uint32_t e2 = (w >> 7) & 0x00ff00ffu;
            uint32_t x0, x1;
            asm("shl.b32 %0, %1, %2;" : "=r"(x0) : "r"(m2 & 0xffffu), "r"((e2 & 0xffu) - fbase));
            asm("shl.b32 %0, %1, %2;" : "=r"(x1) : "r"(m2 >> 16), "r"((e2 >> 16) - fbase));
            asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(b) : "r"(x0));
            asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(b) : "r"(x1));
        }
        if (!(outside & 0x80008000u)) {
            u128_add(acc, b << 18, b >> 46);
            return;
        }
    }
    uint32_t Mv[8];
    int ex[8];
    int emax = 1;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        // fields by multiplications, as in sumsq_add_f16x2: x >> k as the
        // high word of x * 2^(32 - k), the hidden bit as (e + 255) >> 8
        const uint32_t w = h.w[j >> 1];
        const uint32_t e = (j & 1) ? __umulhi(w & 0x7f800000u, 1u << 9) : __umulhi(w & 0x00007f80u, 1u << 25);
        const uint32_t f = (j & 1) ? __umulhi(w & 0x007f0000u, 1u << 16) : (w & 0x0000007fu);
        const uint32_t hid = __umulhi(e + 255u, 1u << 24);
        Mv[j] = f + hid * 0x80u;
        ex[j] = (int)(e + 1u - hid);                 // max(e, 1)
        emax = max(emax, ex[j]);
    }
    const int base = max(emax - kD, first);
    // a square relative to base is X^2 with X = M << (ex - base) < 2^30, so
    // X^2 < 2^60 and the eight add up in 64 bits: one multiply-add each on
    // the integer multiplier.  The sign bit of `below` is set iff some
    // nonzero value lies below base.
    int below = 0;
    unsigned long long b = 0ull;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const int d = ex[j] - base;
        below |= d & -(int)Mv[j];
        const uint32_t X = Mv[j] << max(d, 0);
        asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(b) : "r"(X));
    }
    const int top = 2 * (emax - first);              // window shift of the largest square
    if (below < 0 || top > 62) {
#pragma unroll
        for (int j = 0; j < 8; j++)
            sumsq_add<kBF16>(h.get(j), win_lo, acc, bins);
        return;
    }
    const int t = 2 * (base - first);                // 0..62
    u128_add(acc, b << t, (b >> 1) >> (63 - t));
}

// Block-wide sum of the per-thread accumulators, added to the workspace as
// four 32-bit limbs (each limb sum stays below 2^63 for < 2^31 blocks).
__device__ __forceinline__ void sumsq_flush(U128 acc, unsigned long long* limbs)
{
    __shared__ unsigned long long sh_lo[kThreads / 32], sh_hi[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long lo = __shfl_down_sync(0xffffffffu, acc.lo, off);
        const unsigned long long hi = __shfl_down_sync(0xffffffffu, acc.hi, off);
        u128_add(acc, lo, hi);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sh_lo[warp] = acc.lo;
        sh_hi[warp] = acc.hi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        U128 t{0ull, 0ull};
        for (int w = 0; w < kThreads / 32; w++)
            u128_add(t, sh_lo[w], sh_hi[w]);
        const unsigned long long l[4] = {t.lo & 0xffffffffull, t.lo >> 32, t.hi & 0xffffffffull, t.hi >> 32};
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (l[k]) atomicAdd(limbs + k, l[k]);
    }
}

__device__ __forceinline__ uint32_t* ws_flag(unsigned char* ws) { return reinterpret_cast<uint32_t*>(ws + ws::kFlag); }
__device__ __forceinline__ unsigned long long* ws_acc(unsigned char* ws)
{
    return reinterpret_cast<unsigned long long*>(ws + ws::kAcc);
}
__device__ __forceinline__ unsigned long long* ws_bins(unsigned char* ws)
{
    return reinterpret_cast<unsigned long long*>(ws + ws::kBins);
}

// ---- overflowed steps ----------------------------------------------------------
// An overflowed step is discarded whatever its other buckets hold.  In stages
// 2 and 3 the fused bucket kernels write nothing that outlives a discarded
// step except the 16-bit parameters, so a block that finds the step's flag
// already raised when it starts does nothing at all; a thread raises the flag
// as soon as it meets a non-finite value, so later blocks see it early.  The
// blocks that do run record, in the workspace, their bucket's element window
// (the host then restores parameters only there) and how many elements they
// updated (the bytes the step really moved).
__device__ __forceinline__ bool flag_raised(const unsigned char* ws)
{
    return *reinterpret_cast<const volatile uint32_t*>(ws + ws::kFlag) != 0u;
}

// Raise the step's flag at the first non-finite value this thread meets.
__device__ __forceinline__ void raise_flag(unsigned char* ws, uint32_t nonfinite, bool& raised)
{
    if (nonfinite && !raised) {
        atomicOr(reinterpret_cast<uint32_t*>(ws + ws::kFlag), 1u);
        raised = true;
    }
}

// Elements of the window [lo, hi), cut into groups of V, that this block
// covers when the grid strides over the groups kThreads at a time: block b
// takes groups b*kThreads + t + k*S (t < kThreads, S = gridDim.x*kThreads).
__device__ __forceinline__ int64_t block_elems_grid_stride(int64_t lo, int64_t hi, int V)
{
    const int64_t ng = (hi - lo + V - 1) / V;
    const int64_t base = (int64_t)blockIdx.x * kThreads;
    if (ng <= base) return 0;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t q = (ng - base) / S, r = (ng - base) % S;
    int64_t elems = (q * kThreads + (r < kThreads ? r : (int64_t)kThreads)) * V;
    const int64_t last = (ng - 1) % S;                      // the window's last group, maybe short
    if (last >= base && last < base + kThreads) elems -= ng * V - (hi - lo);
    return elems;
}

// The same for a grid striding over tiles of T elements one per block.
__device__ __forceinline__ int64_t block_elems_tile_stride(int64_t lo, int64_t hi, int64_t T)
{
    const int64_t nt = (hi - lo + T - 1) / T;
    const int64_t b = blockIdx.x;
    if (nt <= b) return 0;
    int64_t elems = ((nt - 1 - b) / gridDim.x + 1) * T;
    if ((nt - 1) % gridDim.x == b) elems -= nt * T - (hi - lo);
    return elems;
}

// One thread per block: this block updated `elems` elements of [lo, hi).
__device__ __forceinline__ void note_updated(unsigned char* ws, int64_t lo, int64_t hi, int64_t elems)
{
    if (elems <= 0) return;
    atomicAdd(reinterpret_cast<unsigned long long*>(ws + ws::kUpdated), (unsigned long long)elems);
    atomicMax(reinterpret_cast<unsigned long long*>(ws + ws::kWroteLoC), ~(unsigned long long)lo);
    atomicMax(reinterpret_cast<unsigned long long*>(ws + ws::kWroteHi), (unsigned long long)hi);
}

// Stage 3: owner rank of a flat index and the index inside its shard.
__device__ __forceinline__ int owner_of(int64_t i, int64_t shard)
{
    return (int)(i / shard);
}

}  // namespace zg

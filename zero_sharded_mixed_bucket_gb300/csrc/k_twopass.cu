// Two-pass step, used with gradient-norm clipping (the update needs the global
// norm first) or when no shadow state is given.
//   pass 1, per bucket  k_reduce:   rank-order reduce, overflow flag, reduced
//                                   gradient materialised (all ranks' grad
//                                   buffers in stages 0/1 -- the all-reduce --,
//                                   the owner's reduced shard in stages 2/3),
//                                   exact integer sum of squares.
//   once                k_finalize: exact sum -> fp64 -> ||g||, clip coefficient.
//   pass 2, per bucket  k_update:   optimizer update in place (k_update.cu).
#include "dev_common.cuh"

namespace zg {

namespace {

// One group's reduced values h (from its fp32 rank-order sums s): the
// overflow test, the exact sum of squares, and the stores.
template <int HDEST, int DT, bool CLIP>
__device__ __forceinline__ void finish_group(const StepArgs& a, int64_t i, int64_t gidx, int cnt,
                                             const float s[kVecOf<DT>], int win_lo, bool& bad, U128& acc,
                                             unsigned long long* bins)
{
    // round to the model precision; elements past cnt are 0 (finite, square 0)
    Vals<DT> h;
    bad |= round_group<DT>(s, h) != 0;
    if constexpr (CLIP) {
        static_assert(DT != kF32, "no exact sum of squares for binary32 values");
        if constexpr (DT == kBF16) {
            sumsq_group_bf16(h, win_lo, acc, bins);
        } else {
#pragma unroll
            for (int p = 0; p < kVecOf<DT> / 2; p++)
                sumsq_add_f16x2(h.w[p], acc);
        }
    }
    if constexpr (HDEST == 0) {
        for (int r = 0; r < a.n_ranks; r++)
            st_vals<DT>(const_cast<void*>(a.grads[r]), gidx, h, cnt);
    } else {
        st_vals<DT>(a.reduced, i, h, cnt);
    }
}

// HDEST 0: write h to every rank's gradient buffer; 1: to the reduced buffer.
// U > 1 (one or two ranks): each thread loads U groups, a grid stride
// apart, before it sums any, so that enough bytes are in flight per thread
// when a group is only one or two 16-byte gradient loads.
// The clipped kernel with four groups in flight is held to 128 registers
// (four blocks per SM instead of three): bf16 0.880 -> 0.884 of the copy
// bandwidth, fp16 0.908 -> 0.910 (clipped N_d = 2 step, A/B; five blocks
// spill and measured 0.857 for bf16).
template <int HDEST, int DT, bool CLIP, int U>
__global__ void __launch_bounds__(kThreads, (CLIP && U > 1) ? 4 : 1) k_reduce(const __grid_constant__ StepArgs a)
{
    if (a.wait_first) wait_prev_grid();   // first bucket of a device-state step (see k_fused)
    allow_next_grid();
    constexpr int V = kVecOf<DT>;
    const int win_lo = a.dyn ? a.dyn->win_lo : a.win_lo;
    const int64_t ngroups = (a.hi - a.lo + V - 1) / V;
    bool bad = false;
    U128 acc{0ull, 0ull};
    unsigned long long* bins = ws_bins(a.ws);
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    if constexpr (U == 1) {
        for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups; gi += stride) {
            const int64_t i = a.lo + gi * V;
            const int cnt = (int)min((int64_t)V, a.hi - i);
            const int64_t gidx = i - a.grad_base;
            float s[V];
            reduce_group<DT>(a, gidx, cnt, s);
            finish_group<HDEST, DT, CLIP>(a, i, gidx, cnt, s, win_lo, bad, acc, bins);
        }
    } else {
        // n_ranks is 1 or 2 here
        for (int64_t g0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; g0 < ngroups; g0 += stride * U) {
            Vals<DT> q[U][2];
#pragma unroll
            for (int k = 0; k < U; k++) {
                const int64_t gi = g0 + k * stride;
                if (gi < ngroups) {
                    const int64_t i = a.lo + gi * V;
                    const int cnt = (int)min((int64_t)V, a.hi - i);
                    q[k][0] = ld_vals<DT>(a.grads[0], i - a.grad_base, cnt);
                    if (a.n_ranks > 1) q[k][1] = ld_vals<DT>(a.grads[1], i - a.grad_base, cnt);
                }
            }
#pragma unroll
            for (int k = 0; k < U; k++) {
                const int64_t gi = g0 + k * stride;
                if (gi < ngroups) {
                    const int64_t i = a.lo + gi * V;
                    const int cnt = (int)min((int64_t)V, a.hi - i);
                    // rank order from 0: s = (0 + g_0) + g_1, as reduce_group
                    float s[V];
#pragma unroll
                    for (int j = 0; j < V; j++) s[j] = __fadd_rn(0.0f, to_f32<DT>(q[k][0].get(j)));
                    if (a.n_ranks > 1) {
#pragma unroll
                        for (int j = 0; j < V; j++) s[j] = __fadd_rn(s[j], to_f32<DT>(q[k][1].get(j)));
                    }
                    finish_group<HDEST, DT, CLIP>(a, i, i - a.grad_base, cnt, s, win_lo, bad, acc, bins);
                }
            }
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        atomicOr(ws_flag(a.ws), 1u);
    if constexpr (CLIP)
        sumsq_flush(acc, ws_acc(a.ws));
    wait_prev_grid();
}

// ---- finalize: exact integer -> nearest fp64 -------------------------------
constexpr int kBigWords = 10;   // 640 bits: covers 2^(2*(-133)) .. 2^(2*127 + 64)

__device__ void big_add(unsigned long long big[kBigWords], unsigned long long val, int shift)
{
    if (!val || shift < 0 || (shift >> 6) >= kBigWords) return;   // callers stay below bit 600
    int w = shift >> 6;
    const int b = shift & 63;
    unsigned long long lo = val << b;
    unsigned long long hi = b ? (val >> (64 - b)) : 0ull;
    unsigned long long s = big[w] + lo;
    unsigned long long carry = s < lo;
    big[w] = s;
    w++;
    while (w < kBigWords && (hi || carry)) {
        const unsigned long long add = hi + carry;   // hi < 2^63, no wrap
        s = big[w] + add;
        carry = s < add;
        big[w] = s;
        hi = 0;
        w++;
    }
}

// The big integer (unit 2^scale_exp) rounded to the nearest double, ties to even.
__device__ double big_to_double(const unsigned long long big[kBigWords], int scale_exp)
{
    int top = kBigWords - 1;
    while (top >= 0 && big[top] == 0) top--;
    if (top < 0) return 0.0;
    const int lz = __clzll(big[top]);
    const int msb = top * 64 + 63 - lz;   // bit index of the leading one
    // 64 bits starting at the leading one
    unsigned long long head = big[top] << lz;
    if (lz && top > 0) head |= big[top - 1] >> (64 - lz);
    bool sticky = false;
    // bits below the 64-bit head
    const int below = msb - 63;   // index of the lowest bit in head
    if (below > 0) {
        const int bw = below >> 6, bb = below & 63;
        if (bb && (big[bw] & ((1ull << bb) - 1ull))) sticky = true;
        for (int k = 0; k < bw && !sticky; k++)
            if (big[k]) sticky = true;
    }
    unsigned long long mant = head >> 11;            // 53 bits
    const unsigned long long rbit = (head >> 10) & 1ull;
    const bool rest = (head & 0x3ffull) != 0 || sticky;
    int exp = msb - 52;
    if (rbit && (rest || (mant & 1ull))) {
        mant++;
        if (mant == (1ull << 53)) {
            mant >>= 1;
            exp++;
        }
    }
    return scalbn((double)mant, exp + scale_exp);
}

__global__ void k_finalize(const FinalArgs a)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(a.ws + ws::kFlag);
    double* norm_out = reinterpret_cast<double*>(a.ws + ws::kNorm);
    float* clip_out = reinterpret_cast<float*>(a.ws + ws::kClip);
    if (flag) {
        *norm_out = __longlong_as_double(0x7ff0000000000000ll);   // +inf
        *clip_out = 1.0f;
        return;
    }
    const int emin = a.dtype == kBF16 ? -133 : -24;   // E of the smallest subnormal
    const int win_lo = a.dyn ? a.dyn->win_lo : a.win_lo;
    const double inv = a.dyn ? a.dyn->inv_d : a.inv;
    unsigned long long big[kBigWords];
    for (int k = 0; k < kBigWords; k++) big[k] = 0ull;
    const unsigned long long* limbs = reinterpret_cast<const unsigned long long*>(a.ws + ws::kAcc);
    for (int k = 0; k < 4; k++)
        big_add(big, limbs[k], 2 * (win_lo - emin) + 32 * k);
    const unsigned long long* bins = reinterpret_cast<const unsigned long long*>(a.ws + ws::kBins);
    for (int e = 0; e < 256; e++) {
        if (!bins[e]) continue;
        const int E = a.dtype == kBF16 ? (e ? e : 1) - 134 : (e ? e : 1) - 25;
        big_add(big, bins[e], 2 * (E - emin));
    }
    const double sumsq = big_to_double(big, 2 * emin);
    const double norm = __dmul_rn(__dsqrt_rn(sumsq), inv);
    const double q = __ddiv_rn(a.max_norm, __dadd_rn(norm, 1e-6));
    *norm_out = norm;
    *clip_out = __double2float_rn(q < 1.0 ? q : 1.0);
}

template <int HDEST, int DT, bool CLIP>
cudaError_t run_reduce(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    if (a.n_ranks <= 2) {
        const int grid = grid_for((const void*)k_reduce<HDEST, DT, CLIP, 4>, groups);
        return launch_step_kernel(k_reduce<HDEST, DT, CLIP, 4>, grid, s, overlap, a);
    }
    const int grid = grid_for((const void*)k_reduce<HDEST, DT, CLIP, 1>, groups);
    return launch_step_kernel(k_reduce<HDEST, DT, CLIP, 1>, grid, s, overlap, a);
}

template <int DT, bool CLIP>
cudaError_t reduce_dt(int stage, const StepArgs& a, cudaStream_t s, bool overlap)
{
    return stage <= 1 ? run_reduce<0, DT, CLIP>(a, s, overlap) : run_reduce<1, DT, CLIP>(a, s, overlap);
}

}  // namespace

cudaError_t launch_reduce(int stage, int dtype, bool clip, const StepArgs& a, cudaStream_t s, bool overlap)
{
    if (dtype == kBF16)
        return clip ? reduce_dt<kBF16, true>(stage, a, s, overlap) : reduce_dt<kBF16, false>(stage, a, s, overlap);
    if (dtype == kF32)   // binary32 steps do not clip (the host refuses the combination)
        return clip ? cudaErrorNotSupported : reduce_dt<kF32, false>(stage, a, s, overlap);
    return clip ? reduce_dt<kF16, true>(stage, a, s, overlap) : reduce_dt<kF16, false>(stage, a, s, overlap);
}

cudaError_t launch_finalize(const FinalArgs& a, cudaStream_t s)
{
    k_finalize<<<1, 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace zg

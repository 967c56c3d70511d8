// Device-state steps (the loss scale and step count live in device memory):
// the per-step scalars derived from the state block, the commit of a step's
// outcome into it, and the restore of an overflowed fused step.  Shared by
// the prepare / commit / restore kernels and by the two-kernel two-pass step
// of a model that is a single bucket (pass 1 derives the scalars, pass 2
// commits).
#pragma once

#include "dev_common.cuh"

namespace zg {

// The step's scalars from the state block: the bias corrections of step t+1
// (beta^t kept as the same sequence of fp64 multiplications as the host
// step), 1/(S*N) in fp64 rounded once to fp32, and the sum-of-squares window
// (binary16: fixed at the smallest subnormal; bfloat16: placed by S*N).
// The sum-of-squares window of a step: binary16 fixed at the smallest
// subnormal; bfloat16 placed by S*N (in [2^(e-1), 2^e): win_lo = e - 40).
__device__ __forceinline__ int window_lo_of(float loss_scale, int n_ranks, int dtype)
{
    if (dtype == kF16) return -24;
    int e = 0;
    frexp(__dmul_rn((double)loss_scale, (double)n_ranks), &e);
    const int lo = -40 + e;
    return lo < -133 ? -133 : (lo > 88 ? 88 : lo);
}

__device__ __forceinline__ Dyn derive_dyn(const DevState* st, float beta1, float beta2, int n_ranks, int dtype)
{
    Dyn d;
    d.beta1_pow_next = __dmul_rn(st->beta1_pow, (double)beta1);
    d.beta2_pow_next = __dmul_rn(st->beta2_pow, (double)beta2);
    d.bc1 = __double2float_rn(__dsub_rn(1.0, d.beta1_pow_next));
    d.bc2 = __double2float_rn(__dsub_rn(1.0, d.beta2_pow_next));
    const double sn = __dmul_rn((double)st->loss_scale, (double)n_ranks);
    d.inv = __double2float_rn(__ddiv_rn(1.0, sn));
    d.inv_d = (double)d.inv;
    d.win_lo = window_lo_of(st->loss_scale, n_ranks, dtype);
    return d;
}

// One thread: the step's outcome into the state block -- t and the beta
// powers advance on a clean step, the loss scaler halves on overflow or
// grows after a run of clean steps -- and the last step's flag, norm and
// clip coefficient.
__device__ inline void commit(const CommitArgs& a)
{
    DevState* st = a.st;
    const uint32_t flag = *reinterpret_cast<const volatile uint32_t*>(a.ws + ws::kFlag);
    if (*reinterpret_cast<const volatile uint32_t*>(a.ws + ws::kErr)) {
        // a kernel gave up a bounded wait (and raised the flag, so nothing was
        // updated): the step is not applied and the scaler keeps its state;
        // bit 1 of last_overflow tells zero_dev_state_read
        st->last_overflow = 3u;
        st->last_skipped = 1;
        st->last_grad_norm = __longlong_as_double(0x7ff8000000000000ll);   // NaN
        st->last_clip_coef = 1.0f;
        return;
    }
    if (flag) {
        if (st->dynamic) {
            const float h = __fmul_rn(st->loss_scale, 0.5f);
            st->loss_scale = h > st->min_loss_scale ? h : st->min_loss_scale;
        }
        st->good_steps = 0;
    } else {
        st->t += 1;
        st->beta1_pow = a.dyn->beta1_pow_next;
        st->beta2_pow = a.dyn->beta2_pow_next;
        st->good_steps += 1;
        if (st->dynamic && st->growth_interval > 0 && st->good_steps >= st->growth_interval) {
            st->loss_scale = __fmul_rn(st->loss_scale, 2.0f);
            st->good_steps = 0;
        }
    }
    st->last_overflow = flag ? 1u : 0u;
    st->last_skipped = flag ? 1 : 0;
    const double norm = *reinterpret_cast<const double*>(a.ws + ws::kNorm);
    const float clip = *reinterpret_cast<const float*>(a.ws + ws::kClip);
    st->last_grad_norm = a.clip ? (flag ? __longlong_as_double(0x7ff0000000000000ll) : norm) : -1.0;
    st->last_clip_coef = a.clip && !flag ? clip : 1.0f;
}

// After an overflowed fused device-state step, for the groups g0, g0 + gs,
// ... of the window [a.lo, a.hi): the unchanged state (w_in, m_in, v_in)
// into the copy the next step reads (w_out, ...), and the parameters back to
// the cast of the master weights.
template <int STAGE, int DT, int OPT>
__device__ __forceinline__ void restore_async_groups(const StepArgs& a, int64_t g0, int64_t gs)
{
    constexpr int V = kVecOf<DT>;
    const int64_t ngroups = (a.hi - a.lo + V - 1) / V;
    const int reps = STAGE == 0 ? a.n_ranks : 1;
    for (int64_t gi = g0; gi < ngroups; gi += gs) {
        const int64_t i = a.lo + gi * V;
        const int cnt = (int)min((int64_t)V, a.hi - i);
        for (int r = 0; r < reps; r++) {
            const int64_t si = (int64_t)r * a.replica_stride + i;
            float w[V];
            ld_f<V>(a.w_in, si, cnt, w);
            st_f<V>(a.w_out, si, cnt, w);
            if constexpr (OPT != kSgd) {
                float m[V];
                ld_f<V>(a.m_in, si, cnt, m);
                st_f<V>(a.m_out, si, cnt, m);
            }
            if constexpr (OPT == kAdam) {
                float v[V];
                ld_f<V>(a.v_in, si, cnt, v);
                st_f<V>(a.v_out, si, cnt, v);
            }
            Vals<DT> p;
#pragma unroll
            for (int j = 0; j < V; j++)
                p.set(j, from_f32<DT>(w[j]));
            if constexpr (STAGE == 0) {
                st_vals<DT>(a.params16[r], i, p, cnt);
            } else if constexpr (STAGE == 3) {
                const int o = owner_of(i, a.shard);
                st_vals<DT>(a.params16[o], i - (int64_t)o * a.shard, p, cnt);
            } else {
                for (int q = 0; q < a.n_ranks; q++)
                    st_vals<DT>(a.params16[q], i, p, cnt);
            }
        }
    }
}

}  // namespace zg

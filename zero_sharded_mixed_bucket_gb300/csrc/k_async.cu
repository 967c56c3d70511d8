// Steps whose loss scale and step count live in device memory, so a step
// needs no host synchronisation and can be captured in a CUDA graph.
//
//   k_prepare        one block: clears the workspace head (flag, sums) and,
//                    in one thread, derives the step's scalars (bias
//                    corrections for step t+1, 1/(S*N), the sum-of-squares
//                    window) from the state block into the workspace, where
//                    the bucket kernels read them;
//   commit           one thread: the step's outcome into the state block --
//                    t and the beta powers advance on a clean step, the loss
//                    scaler halves on overflow or grows after a run of clean
//                    steps -- and the last step's flag, norm and coefficient;
//                    run by k_restore_async on the fused path, by k_commit
//                    after the two-pass path's updates;
//   k_restore_async  fused path: does nothing else unless the step
//                    overflowed; then it puts the unchanged state into the
//                    copy the next step reads (the host alternates the copies
//                    on every call, since it no longer learns the flag) and
//                    restores the parameters to the cast of the master weights.
// The arithmetic matches the host-synchronised step exactly: beta^t is kept
// as the same sequence of fp64 multiplications, 1/(S*N) and the scaler use
// the same fp64 and fp32 operations.
#include "dev_common.cuh"

namespace zg {

namespace {

__global__ void k_prepare(const PrepArgs a)
{
    allow_next_grid();   // the first bucket kernel may launch; it waits for this one
    wait_prev_grid();    // launched early: the previous step's commit must be complete
    // clear the step's flag and sums (the workspace head) ...
    static_assert(ws::kEnd % 16 == 0, "workspace head is cleared in 16-byte words");
    uint4* head = reinterpret_cast<uint4*>(a.ws);
    for (int k = threadIdx.x; k < (int)(ws::kEnd / 16); k += blockDim.x)
        head[k] = make_uint4(0u, 0u, 0u, 0u);
    // ... and derive the step's scalars from the state block
    if (threadIdx.x != 0) return;
    const DevState* st = a.st;
    Dyn d;
    d.beta1_pow_next = __dmul_rn(st->beta1_pow, (double)a.beta1);
    d.beta2_pow_next = __dmul_rn(st->beta2_pow, (double)a.beta2);
    d.bc1 = __double2float_rn(__dsub_rn(1.0, d.beta1_pow_next));
    d.bc2 = __double2float_rn(__dsub_rn(1.0, d.beta2_pow_next));
    const double sn = __dmul_rn((double)st->loss_scale, (double)a.n_ranks);
    d.inv = __double2float_rn(__ddiv_rn(1.0, sn));
    d.inv_d = (double)d.inv;
    if (a.dtype == kF16) {
        d.win_lo = -24;
    } else {
        int e = 0;
        frexp(sn, &e);
        int lo = -40 + e;
        d.win_lo = lo < -133 ? -133 : (lo > 88 ? 88 : lo);
    }
    *a.dyn = d;
}

__device__ void commit(const CommitArgs& a)
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

__global__ void k_commit(const CommitArgs a)
{
    allow_next_grid();
    wait_prev_grid();
    if (threadIdx.x == 0) commit(a);
}

// Also commits the step (block 0, thread 0): the commit writes only the
// state block, which the restore does not touch.
template <int STAGE, int DT, int OPT>
__global__ void __launch_bounds__(kThreads) k_restore_async(const __grid_constant__ StepArgs a,
                                                             const CommitArgs c)
{
    allow_next_grid();
    wait_prev_grid();    // launched early: every bucket kernel of the step must be complete
    if (blockIdx.x == 0 && threadIdx.x == 0) commit(c);
    if (!*reinterpret_cast<const volatile uint32_t*>(ws_flag(a.ws))) return;   // clean step: nothing to do
    const int64_t ngroups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    const int reps = STAGE == 0 ? a.n_ranks : 1;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t i = a.lo + gi * kVecOf<DT>;
        const int cnt = (int)min((int64_t)kVecOf<DT>, a.hi - i);
        for (int r = 0; r < reps; r++) {
            const int64_t si = (int64_t)r * a.replica_stride + i;
            float w[kVecOf<DT>];
            ld_f<kVecOf<DT>>(a.w_in, si, cnt, w);
            st_f<kVecOf<DT>>(a.w_out, si, cnt, w);
            if constexpr (OPT != kSgd) {
                float m[kVecOf<DT>];
                ld_f<kVecOf<DT>>(a.m_in, si, cnt, m);
                st_f<kVecOf<DT>>(a.m_out, si, cnt, m);
            }
            if constexpr (OPT == kAdam) {
                float v[kVecOf<DT>];
                ld_f<kVecOf<DT>>(a.v_in, si, cnt, v);
                st_f<kVecOf<DT>>(a.v_out, si, cnt, v);
            }
            Vals<DT> p;
#pragma unroll
            for (int j = 0; j < kVecOf<DT>; j++)
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

template <int STAGE, int DT, int OPT>
cudaError_t run_restore_async(const StepArgs& a, const CommitArgs& c, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    const int grid = groups > 0 ? grid_for((const void*)k_restore_async<STAGE, DT, OPT>, groups) : 1;
    return launch_kernel(k_restore_async<STAGE, DT, OPT>, grid, kThreads, s, overlap, a, c);
}

template <int STAGE, int DT>
cudaError_t restore_opt(int opt, const StepArgs& a, const CommitArgs& c, cudaStream_t s, bool overlap)
{
    switch (opt) {
    case kSgdm: return run_restore_async<STAGE, DT, kSgdm>(a, c, s, overlap);
    case kSgd: return run_restore_async<STAGE, DT, kSgd>(a, c, s, overlap);
    default: return run_restore_async<STAGE, DT, kAdam>(a, c, s, overlap);
    }
}

template <int DT>
cudaError_t restore_stage(int stage, int opt, const StepArgs& a, const CommitArgs& c, cudaStream_t s, bool overlap)
{
    switch (stage) {
    case 0: return restore_opt<0, DT>(opt, a, c, s, overlap);
    case 1: return restore_opt<1, DT>(opt, a, c, s, overlap);
    case 2: return restore_opt<2, DT>(opt, a, c, s, overlap);
    default: return restore_opt<3, DT>(opt, a, c, s, overlap);
    }
}

}  // namespace

cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s, bool overlap)
{
    return launch_kernel(k_prepare, 1, kThreads, s, overlap, a);
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s, bool overlap)
{
    return launch_kernel(k_commit, 1, 32, s, overlap, a);
}

cudaError_t launch_restore_async(int stage, int dtype, int opt, const StepArgs& a, const CommitArgs& c,
                                 cudaStream_t s, bool overlap)
{
    if (dtype == kF32) return restore_stage<kF32>(stage, opt, a, c, s, overlap);
    return dtype == kBF16 ? restore_stage<kBF16>(stage, opt, a, c, s, overlap)
                          : restore_stage<kF16>(stage, opt, a, c, s, overlap);
}

}  // namespace zg

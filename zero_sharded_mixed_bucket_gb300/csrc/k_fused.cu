// Fused per-bucket step: reduce-scatter + overflow check + unscale + Adam +
// model-precision cast + all-gather, one HBM pass.  New fp32 state goes to the shadow
// copy; the host commits it once the global overflow flag is known.
//
// Stage 0 (plain data parallelism): the reduced gradient is written back to
// every rank (all-reduce) and each of the N replicas updates its own full
// state and parameter copy.
// Stage 1 (P_os): all-reduce write-back; the owner updates its state shard and
// the new parameters go to every rank (step-end all-gather).
// Stage 2 (P_os+g): reduce-scatter to the owner, owner update, all-gather.
// Stage 3 (P_os+g+p): reduce-scatter, owner update, the new parameters stay in
// the owner's shard.
// ("ZeRO：大模型训练的内存优化革命" 3.1.1-3.1.3; ZeRO visual reading, stage list
// and communication accounting.)
#include "dev_common.cuh"

namespace zg {

namespace {

// Stage 0 walks the N replicas' state per group; unconstrained it takes ~107
// registers (4 blocks per SM).  Asking for 5 resident blocks brings it to 96
// without spills and measured 6130 -> 6636 GB/s on GB300.
template <int STAGE, int DT, int OPT>
__global__ void __launch_bounds__(kThreads, STAGE == 0 ? 5 : 1) k_fused(const __grid_constant__ StepArgs a)
{
    // The first bucket kernel of a device-state step is launched early after
    // the prepare kernel: it waits for it before anything else, and lets the
    // next bucket kernel launch only then (that one reads the step scalars
    // without waiting).
    if (a.wait_first) wait_prev_grid();
    allow_next_grid();
    // Step scalars: from the launch, or from the prepare kernel in a
    // device-state step.
    float inv = a.inv;
    AdamHP hp = a.hp;
    if (a.dyn) {
        inv = a.dyn->inv;
        hp.bc1 = a.dyn->bc1;
        hp.bc2 = a.dyn->bc2;
    }
    const int64_t ngroups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    bool bad = false;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t i = a.lo + gi * kVecOf<DT>;
        const int cnt = (int)min((int64_t)kVecOf<DT>, a.hi - i);
        const int64_t gidx = i - a.grad_base;

        float s[kVecOf<DT>];
        reduce_group<DT>(a, gidx, cnt, s);

        // round to the model precision (elements past cnt are 0: finite, no effect)
        Vals<DT> h;
        bad |= round_group<DT>(s, h) != 0;
        float g[kVecOf<DT>];
        unscale_group<DT>(h, inv, g);

        if constexpr (STAGE <= 1) {
            for (int r = 0; r < a.n_ranks; r++)
                st_vals<DT>(const_cast<void*>(a.grads[r]), gidx, h, cnt);
        }

        if constexpr (STAGE == 0) {
            for (int r = 0; r < a.n_ranks; r++) {
                Vals<DT> p;
                update_state<DT, OPT>(a, hp, (int64_t)r * a.replica_stride + i, cnt, g, p);
                st_vals<DT>(a.params16[r], i, p, cnt);
            }
        } else {
            Vals<DT> p;
            update_state<DT, OPT>(a, hp, i, cnt, g, p);
            if constexpr (STAGE == 3) {
                const int o = owner_of(i, a.shard);
                st_vals<DT>(a.params16[o], i - (int64_t)o * a.shard, p, cnt);
            } else {
                for (int r = 0; r < a.n_ranks; r++)
                    st_vals<DT>(a.params16[r], i, p, cnt);
            }
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        atomicOr(ws_flag(a.ws), 1u);
    wait_prev_grid();
}

// After an overflowed fused step: put back the 16-bit parameters the step
// overwrote, as the cast of the unchanged master weights (w_in).
template <int STAGE, int DT>
__global__ void __launch_bounds__(kThreads) k_restore(const __grid_constant__ StepArgs a)
{
    const int64_t ngroups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t i = a.lo + gi * kVecOf<DT>;
        const int cnt = (int)min((int64_t)kVecOf<DT>, a.hi - i);
        const int reps = STAGE == 0 ? a.n_ranks : 1;
        for (int r = 0; r < reps; r++) {
            float w[kVecOf<DT>];
            ld_f<kVecOf<DT>>(a.w_in, (int64_t)r * a.replica_stride + i, cnt, w);
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
cudaError_t run_fused3(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    const int grid = grid_for((const void*)k_fused<STAGE, DT, OPT>, groups);
    return launch_step_kernel(k_fused<STAGE, DT, OPT>, grid, s, overlap, a);
}

template <int STAGE, int DT>
cudaError_t run_fused(int opt, const StepArgs& a, cudaStream_t s, bool overlap)
{
    switch (opt) {
    case kSgdm: return run_fused3<STAGE, DT, kSgdm>(a, s, overlap);
    case kSgd: return run_fused3<STAGE, DT, kSgd>(a, s, overlap);
    default: return run_fused3<STAGE, DT, kAdam>(a, s, overlap);
    }
}

template <int STAGE, int DT>
cudaError_t run_restore(const StepArgs& a, cudaStream_t s)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    const int grid = grid_for((const void*)k_restore<STAGE, DT>, groups);
    k_restore<STAGE, DT><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

#define ZG_DISPATCH_STAGE_DT(fn, stage, dtype, ...)                                   \
    do {                                                                              \
        if ((dtype) == kBF16) {                                                       \
            switch (stage) {                                                          \
            case 0: return fn<0, kBF16>(__VA_ARGS__);                                 \
            case 1: return fn<1, kBF16>(__VA_ARGS__);                                 \
            case 2: return fn<2, kBF16>(__VA_ARGS__);                                 \
            default: return fn<3, kBF16>(__VA_ARGS__);                                \
            }                                                                         \
        } else if ((dtype) == kF32) {                                                 \
            switch (stage) {                                                          \
            case 0: return fn<0, kF32>(__VA_ARGS__);                                  \
            case 1: return fn<1, kF32>(__VA_ARGS__);                                  \
            case 2: return fn<2, kF32>(__VA_ARGS__);                                  \
            default: return fn<3, kF32>(__VA_ARGS__);                                 \
            }                                                                         \
        } else {                                                                      \
            switch (stage) {                                                          \
            case 0: return fn<0, kF16>(__VA_ARGS__);                                  \
            case 1: return fn<1, kF16>(__VA_ARGS__);                                  \
            case 2: return fn<2, kF16>(__VA_ARGS__);                                  \
            default: return fn<3, kF16>(__VA_ARGS__);                                 \
            }                                                                         \
        }                                                                             \
    } while (0)

cudaError_t launch_fused(int stage, int dtype, int opt, const StepArgs& a, cudaStream_t s, bool overlap)
{
    ZG_DISPATCH_STAGE_DT(run_fused, stage, dtype, opt, a, s, overlap);
}

cudaError_t launch_restore(int stage, int dtype, const StepArgs& a, cudaStream_t s)
{
    ZG_DISPATCH_STAGE_DT(run_restore, stage, dtype, a, s);
}

}  // namespace zg

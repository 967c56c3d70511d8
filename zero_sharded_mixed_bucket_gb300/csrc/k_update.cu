// Two-pass step, pass 2 (see k_twopass.cu for pass 1 and the finalize): per
// bucket, the optimizer update in place on the current state, unless the
// step's overflow flag is set, then the model-precision cast and the all-gather.
#include "dev_common.cuh"

namespace zg {

namespace {

template <int STAGE, int DT, bool CLIP, int OPT>
__global__ void __launch_bounds__(kThreads) k_update(const __grid_constant__ StepArgs a)
{
    // The first update kernel of a step is launched in plain stream order after
    // the pass-1 kernels and the finalize, so the flag and the clip
    // coefficient are final before any update kernel starts.
    allow_next_grid();
    if (*reinterpret_cast<volatile uint32_t*>(ws_flag(a.ws))) {
        wait_prev_grid();
        return;   // overflow: the whole step is skipped
    }
    // With clipping on, multiply by c only when c < 1: g * 1 == g for every
    // finite g, so both forms give the same bits.
    const float c = CLIP ? *reinterpret_cast<const float*>(a.ws + ws::kClip) : 1.0f;
    float inv = a.inv;
    AdamHP hp = a.hp;
    if (a.dyn) {
        inv = a.dyn->inv;
        hp.bc1 = a.dyn->bc1;
        hp.bc2 = a.dyn->bc2;
    }
    const int64_t ngroups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t i = a.lo + gi * kVecOf<DT>;
        const int cnt = (int)min((int64_t)kVecOf<DT>, a.hi - i);
        const int reps = STAGE == 0 ? a.n_ranks : 1;
        for (int r = 0; r < reps; r++) {
            Vals<DT> h;
            if constexpr (STAGE == 0)
                h = ld_vals<DT>(a.grads[r], i - a.grad_base, cnt);        // each replica its own all-reduced copy
            else if constexpr (STAGE == 1)
                h = ld_vals<DT>(a.grads[owner_of(i, a.shard)], i - a.grad_base, cnt);
            else
                h = ld_vals<DT>(a.reduced, i, cnt);
            float g[kVecOf<DT>];
            unscale_group<DT>(h, inv, g);
            if (c != 1.0f) {
#pragma unroll
                for (int j = 0; j < kVecOf<DT>; j++)
                    g[j] = __fmul_rn(g[j], c);
            }
            Vals<DT> p;
            update_state<DT, OPT>(a, hp, (int64_t)r * a.replica_stride + i, cnt, g, p);
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
    wait_prev_grid();
}

template <int STAGE, int DT, bool CLIP, int OPT>
cudaError_t run_update(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    const int grid = grid_for((const void*)k_update<STAGE, DT, CLIP, OPT>, groups);
    return launch_step_kernel(k_update<STAGE, DT, CLIP, OPT>, grid, s, overlap, a);
}

template <int DT, bool CLIP, int OPT>
cudaError_t update_stage(int stage, const StepArgs& a, cudaStream_t s, bool overlap)
{
    switch (stage) {
    case 0: return run_update<0, DT, CLIP, OPT>(a, s, overlap);
    case 1: return run_update<1, DT, CLIP, OPT>(a, s, overlap);
    case 2: return run_update<2, DT, CLIP, OPT>(a, s, overlap);
    default: return run_update<3, DT, CLIP, OPT>(a, s, overlap);
    }
}

template <int DT, int OPT>
cudaError_t update_clip(int stage, bool clip, const StepArgs& a, cudaStream_t s, bool overlap)
{
    if constexpr (DT == kF32)   // binary32 steps do not clip (the host refuses the combination)
        return clip ? cudaErrorNotSupported : update_stage<DT, false, OPT>(stage, a, s, overlap);
    else
        return clip ? update_stage<DT, true, OPT>(stage, a, s, overlap)
                    : update_stage<DT, false, OPT>(stage, a, s, overlap);
}

template <int DT>
cudaError_t update_opt(int stage, int opt, bool clip, const StepArgs& a, cudaStream_t s, bool overlap)
{
    switch (opt) {
    case kSgdm: return update_clip<DT, kSgdm>(stage, clip, a, s, overlap);
    case kSgd: return update_clip<DT, kSgd>(stage, clip, a, s, overlap);
    default: return update_clip<DT, kAdam>(stage, clip, a, s, overlap);
    }
}

}  // namespace

cudaError_t launch_update(int stage, int dtype, int opt, bool clip, const StepArgs& a, cudaStream_t s, bool overlap)
{
    if (dtype == kF32) return update_opt<kF32>(stage, opt, clip, a, s, overlap);
    return dtype == kBF16 ? update_opt<kBF16>(stage, opt, clip, a, s, overlap)
                          : update_opt<kF16>(stage, opt, clip, a, s, overlap);
}

}  // namespace zg

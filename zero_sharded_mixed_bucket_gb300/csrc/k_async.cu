// Steps whose loss scale and step count live in device memory, so a step
// needs no host synchronisation and can be captured in a CUDA graph.
//
//   k_prepare        one block: clears the workspace head (flag, sums) and,
//                    in one thread, derives the step's scalars (bias
//                    corrections for step t+1, 1/(S*N), the sum-of-squares
//                    window) from the state block into the workspace, where
//                    the bucket kernels read them;
//   commit           (dev_state.cuh) one thread: the step's outcome into the state block --
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
#include "dev_state.cuh"

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
    if (threadIdx.x == 0) *a.dyn = derive_dyn(a.st, a.beta1, a.beta2, a.n_ranks, a.dtype);
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
    restore_async_groups<STAGE, DT, OPT>(a, (int64_t)blockIdx.x * kThreads + threadIdx.x,
                                         (int64_t)gridDim.x * kThreads);
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

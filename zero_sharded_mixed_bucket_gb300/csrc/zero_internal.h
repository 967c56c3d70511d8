// Internal interface between the host driver (zero_host.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_gb300.h"

namespace zg {

constexpr int kMaxRanks = ZERO_MAX_RANKS;
constexpr int kThreads = 128;   // threads per block of every streaming kernel (measured best for k_fused)

// Workspace layout (caller-provided device memory, zeroed by zero_step_begin).
namespace ws {
constexpr size_t kFlag = 0;     // uint32: 1 once any reduced gradient element is inf/NaN
constexpr size_t kErr = 4;      // uint32: 1 if a kernel gave up a bounded wait (the step is then skipped)
constexpr size_t kNorm = 8;     // double: ||g||_2 (two-pass with clipping)
constexpr size_t kClip = 16;    // float: clip coefficient
constexpr size_t kAcc = 32;     // 4 x uint64: 32-bit limbs of the fixed-point sum of squares
constexpr size_t kBins = 64;    // 256 x uint64: sum of M^2 per exponent field, outside the window
// Fused step, stages 2 and 3: what the bucket kernels that ran wrote (an
// overflowed step restores parameters only there) -- the complement of the
// lowest written flat index (0: nothing written), the end of the highest
// written window, and the number of elements updated.
constexpr size_t kWroteLoC = kBins + 256 * 8;   // uint64: ~lo
constexpr size_t kWroteHi = kWroteLoC + 8;      // uint64: hi
constexpr size_t kUpdated = kWroteHi + 8;       // uint64: elements updated
constexpr size_t kDone = kUpdated + 8;          // 2 x uint32: blocks of a one-bucket step's passes 1, 2 that finished
constexpr size_t kEnd = kDone + 8;              // end of the part cleared before every step (16-byte multiple)
constexpr size_t kDyn = 2176;   // Dyn: per-step scalars of a device-state step (written by the prepare kernel)
constexpr int64_t kBytes = 4096;
static_assert(kEnd % 16 == 0 && kEnd <= kDyn, "workspace head");
}  // namespace ws

// Per-step scalars of a step whose loss scale and step count live on the
// device: written by the prepare kernel, read by the step kernels.
struct Dyn {
    float inv;                      // 1/(S*N)
    float bc1, bc2;                 // 1 - beta^(t+1)
    int32_t win_lo;                 // sum-of-squares window
    double inv_d;                   // the same 1/(S*N) as a double (finalize)
    double beta1_pow_next, beta2_pow_next;
};

enum { kAdam = ZERO_ADAM, kSgdm = ZERO_SGD_MOMENTUM, kSgd = ZERO_SGD };

struct AdamHP {
    float lr, b1, omb1, b2, omb2, eps, bc1, bc2;
    float mu;   // SGD momentum
};

// Arguments of the per-bucket kernels.  Passed by value as a __grid_constant__
// parameter; pointer arrays are indexed with warp-uniform indices.
struct StepArgs {
    const void* grads[kMaxRanks];   // grads[r] + (i - grad_base) addresses flat element i of rank r
    void* params16[kMaxRanks];      // rank r's 16-bit parameters (full vector, or shard in stage 3)
    const float* w_in;
    const float* m_in;
    const float* v_in;
    float* w_out;
    float* m_out;
    float* v_out;
    void* reduced;                  // 16-bit reduced gradient, flat index order
    unsigned char* ws;              // workspace
    int64_t lo, hi;                 // flat element window [lo, hi)
    int64_t grad_base;
    int64_t shard;                  // P
    int64_t replica_stride;         // stage 0: elements between consecutive replicas' state
    int32_t n_ranks;
    float inv;                      // 1/(S*N)
    AdamHP hp;
    int32_t win_lo;                 // lowest exponent E of the sum-of-squares window
    const Dyn* dyn;                 // device-state step: scalars above come from here (else NULL)
    int32_t withhold_tile;          // test hook (environment ZERO_TEST_WITHHOLD_TILE): the staged pass 1's
                                    // block 0 announces its first tile but issues no copy, so its bounded
                                    // waits run out and the step reports ZERO_ETIMEOUT
    int32_t wait_first;             // launched early after a kernel whose results it reads (the prepare kernel
                                    // before a step's first bucket, the finalize or the last pass-1 kernel
                                    // before the first update): wait for it before anything else
};

struct FinalArgs {
    unsigned char* ws;
    int32_t dtype;
    int32_t win_lo;
    double inv;
    double max_norm;
    const Dyn* dyn;                 // device-state step: inv and win_lo from here
};

// Device-resident step state (the C ABI's zero_dev_state_t, same layout).
struct DevState {
    int64_t t;
    double beta1_pow, beta2_pow;    // beta^t, by repeated multiplication
    float loss_scale, min_loss_scale;
    int32_t dynamic, growth_interval, good_steps;
    uint32_t last_overflow;
    double last_grad_norm;
    float last_clip_coef;
    int32_t last_skipped;
};

struct GatherArgs {
    const void* shards[kMaxRanks];
    void* dst[kMaxRanks];
    int64_t start;                  // flat index of the layer's first element
    int64_t len;
    int64_t shard;                  // P
    int32_t n_dst;
};

// Launchers: return the CUDA error of the launch.  `stage` 0..3, `dtype`
// ZERO_FP16 / ZERO_BF16.
// `overlap`: launch with programmatic dependent launch on the previous kernel
// of the stream -- only when that kernel is another bucket kernel of the same
// step pass, launched by the library itself.
cudaError_t launch_fused(int stage, int dtype, int opt, const StepArgs& a, cudaStream_t s, bool overlap);
cudaError_t launch_reduce(int stage, int dtype, bool clip, const StepArgs& a, cudaStream_t s, bool overlap);
cudaError_t launch_finalize(const FinalArgs& a, cudaStream_t s, bool overlap);
cudaError_t launch_update(int stage, int dtype, int opt, bool clip, const StepArgs& a, cudaStream_t s,
                          bool overlap);
cudaError_t launch_restore(int stage, int dtype, const StepArgs& a, cudaStream_t s);
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);

// Device-state steps: per-step scalars from the state block, commit of the
// outcome into it, and (fused path) the restore that also copies the
// unchanged state into the copy the next step reads.
struct PrepArgs {
    DevState* st;
    Dyn* dyn;
    unsigned char* ws;              // its head [0, ws::kEnd) is cleared
    float beta1, beta2;
    int32_t n_ranks;
    int32_t dtype;
};
struct CommitArgs {
    DevState* st;
    const Dyn* dyn;
    const unsigned char* ws;
    int32_t clip;                   // the step clips (norm and coefficient valid)
};
// All three may be launched as programmatic dependents of the kernel before
// them (`overlap`): each waits for it to complete before touching memory.
cudaError_t launch_prepare(const PrepArgs& a, cudaStream_t s, bool overlap);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s, bool overlap);
cudaError_t launch_restore_async(int stage, int dtype, int opt, const StepArgs& a, const CommitArgs& c,
                                 cudaStream_t s, bool overlap);
// The two-pass device-state step of a model that is one bucket (stages 2
// and 3) as two kernels, after the workspace head was cleared: pass 1, whose
// last block to finish derives the step's scalars into p.dyn and, when
// clipping, the norm and clip coefficient; pass 2 (a programmatic dependent
// of pass 1), whose last block commits the step.
cudaError_t launch_reduce_one(int dtype, bool clip, const StepArgs& a, const PrepArgs& p, double max_norm,
                              cudaStream_t s);
cudaError_t launch_update_one(int stage, int dtype, int opt, bool clip, const StepArgs& a, const CommitArgs& c,
                              cudaStream_t s);

// Record the thread-local message that zero_last_error() returns; gives back
// `st`.  For entry points defined outside zero_host.cu.
zero_status_t set_error(zero_status_t st, const char* msg);

// Launch a bucket kernel taking StepArgs, optionally as a programmatic
// dependent of the previous kernel in the stream.
template <typename K, typename... Args>
inline cudaError_t launch_kernel(K kernel, int grid, int threads, cudaStream_t s, bool overlap, const Args&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename K>
inline cudaError_t launch_step_kernel(K kernel, int grid, cudaStream_t s, bool overlap, const StepArgs& a)
{
    return launch_kernel(kernel, grid, kThreads, s, overlap, a);
}

// Grid for a grid-stride kernel over `groups` work items of kThreads-thread
// blocks: at most (SM count x resident blocks per SM), so every block stays
// resident and each SM gets the same share.
int grid_for(const void* kernel, int64_t groups);

}  // namespace zg

// Two-pass step, pass 2 (see k_twopass.cu for pass 1 and the finalize): per
// bucket, the optimizer update in place on the current state, unless the
// step's overflow flag is set, then the model-precision cast and the all-gather.
#include "dev_state.cuh"
#include "host_ptrs.h"

namespace zg {

namespace {

// One group of pass 2 at flat element i: the reduced gradient unscaled
// (and, with clipping, multiplied by c when c < 1: g * 1 == g for every
// finite g, so both forms give the same bits), the update, the cast and the
// stage's parameter writes.
template <int STAGE, int DT, int OPT>
__device__ __forceinline__ void update_group(const StepArgs& a, int64_t i, float c, float inv, const AdamHP& hp)
{
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

template <int STAGE, int DT, bool CLIP, int OPT>
__global__ void __launch_bounds__(kThreads) k_update(const __grid_constant__ StepArgs a)
{
    // The first update kernel of a step is a programmatic dependent of the
    // finalize (or, without clipping, of the last pass-1 kernel): it waits for
    // it before reading the flag and the clip coefficient, and only then lets
    // the next update kernel launch, so those values are final for every
    // update kernel.
    if (a.wait_first) wait_prev_grid();
    allow_next_grid();
    if (*reinterpret_cast<volatile uint32_t*>(ws_flag(a.ws))) {
        wait_prev_grid();
        return;   // overflow: the whole step is skipped
    }
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
         gi += (int64_t)gridDim.x * kThreads)
        update_group<STAGE, DT, OPT>(a, a.lo + gi * kVecOf<DT>, c, inv, hp);
    wait_prev_grid();
}

// Pass 2 of the two-kernel step of a model that is one bucket (k_reduce_one
// is pass 1): as k_update, with the scalars the last pass-1 block wrote, and
// the block that finishes last (the second completion count) commits the
// step.
template <int STAGE, int DT, bool CLIP, int OPT>
__global__ void __launch_bounds__(kThreads) k_update_one(const __grid_constant__ StepArgs a, const CommitArgs cm)
{
    __shared__ int last;
    wait_prev_grid();   // pass 1, its last block's scalars, norm and clip coefficient among it
    if (!*reinterpret_cast<volatile uint32_t*>(ws_flag(a.ws))) {
        const float c = CLIP ? *reinterpret_cast<const float*>(a.ws + ws::kClip) : 1.0f;
        AdamHP hp = a.hp;
        hp.bc1 = a.dyn->bc1;
        hp.bc2 = a.dyn->bc2;
        const float inv = a.dyn->inv;
        const int64_t ngroups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
        for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
             gi += (int64_t)gridDim.x * kThreads)
            update_group<STAGE, DT, OPT>(a, a.lo + gi * kVecOf<DT>, c, inv, hp);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(reinterpret_cast<unsigned int*>(a.ws + ws::kDone) + 1, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (last && threadIdx.x == 0) {
        __threadfence();
        commit(cm);
    }
}

// Stages 1 and 2 with 2 or more ranks: the new parameters for every rank are
// written through shared memory -- a block computes a tile of
// kTileSub x kThreads groups, then the lanes of warp 0 copy it to the ranks'
// parameter buffers, one bulk asynchronous copy per rank (cp.async.bulk
// shared -> global).  Pass 2 is mostly writes (2 N bytes of parameters per 14 bytes
// read); the bulk copies move that replicated stream as the stage-3 gather
// does.  Two tile buffers: a buffer is rewritten after the copies that read
// it two tiles earlier have read it (wait_group.read).  The ragged end of a
// bucket (less than 16 bytes) is stored by the threads.
// Tiles of 4 x 128 groups, two blocks per resident slot (a block's loads and
// arithmetic then overlap another block's copies).  Measured on GB300, the
// clipped stage-2 step at 2^28 parameters: 32 ranks 0.947-0.951 of the copy
// bandwidth with tiles of 2 x 128 groups and one block per slot, 0.985-0.990
// now (8 x 128: 0.982; three blocks per slot: 0.984); fp16 / bf16 with
// per-thread stores against the tiles: 8 ranks 0.933 / 0.910 -> 0.963 /
// 0.954, 4 ranks 0.919 / 0.863 -> 0.945 / 0.886, 2 ranks 0.893 / 0.865 ->
// 0.900 / 0.870.  One rank keeps the per-thread stores (a single copy).
constexpr int kTileSub = 4;
constexpr int kBulkMinRanks = 2;

template <int STAGE, int DT, bool CLIP, int OPT>
__global__ void __launch_bounds__(kThreads) k_update_tiled(const __grid_constant__ StepArgs a)
{
    static_assert(STAGE == 1 || STAGE == 2, "parameters replicated to every rank: stages 1 and 2");
    constexpr int V = kVecOf<DT>;
    constexpr int kEB = DT == kF32 ? 4 : 2;                        // bytes per value
    constexpr int kTileGroups = kThreads * kTileSub;
    constexpr int64_t kTileElems = (int64_t)kTileGroups * V;
    __shared__ __align__(128) Vals<DT> tile[2][kTileGroups];
    if (a.wait_first) wait_prev_grid();   // as k_update
    allow_next_grid();
    if (*reinterpret_cast<volatile uint32_t*>(ws_flag(a.ws))) {
        wait_prev_grid();
        return;   // overflow: the whole step is skipped
    }
    const float c = CLIP ? *reinterpret_cast<const float*>(a.ws + ws::kClip) : 1.0f;
    float inv = a.inv;
    AdamHP hp = a.hp;
    if (a.dyn) {
        inv = a.dyn->inv;
        hp.bc1 = a.dyn->bc1;
        hp.bc2 = a.dyn->bc2;
    }
    const int64_t ntiles = (a.hi - a.lo + kTileElems - 1) / kTileElems;
    int b = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, b ^= 1) {
        // the lanes of warp 0 issue the copies; each waits for its own
        if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const int64_t t0 = a.lo + t * kTileElems;                   // first element of the tile
        const int64_t tel = min(kTileElems, a.hi - t0);              // elements in the tile
        for (int k = 0; k < kTileSub; k++) {
            const int gl = k * kThreads + threadIdx.x;               // group within the tile
            const int64_t i = t0 + (int64_t)gl * V;
            if (i >= a.hi) break;
            const int cnt = (int)min((int64_t)V, a.hi - i);
            Vals<DT> h;
            if constexpr (STAGE == 1)
                h = ld_vals<DT>(a.grads[owner_of(i, a.shard)], i - a.grad_base, cnt);
            else
                h = ld_vals<DT>(a.reduced, i, cnt);
            float g[V];
            unscale_group<DT>(h, inv, g);
            if (c != 1.0f) {
#pragma unroll
                for (int j = 0; j < V; j++)
                    g[j] = __fmul_rn(g[j], c);
            }
            Vals<DT> p;
            update_state<DT, OPT>(a, hp, i, cnt, g, p);
            tile[b][gl] = p;
        }
        // make the tile visible to the bulk-copy (async) proxy, then copy it out
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        const uint32_t bytes = (uint32_t)(tel * kEB) & ~15u;
        if (threadIdx.x < 32) {   // one rank per lane
            if (bytes) {
                const uint32_t sp = (uint32_t)__cvta_generic_to_shared(&tile[b][0]);
                for (int r = threadIdx.x; r < a.n_ranks; r += 32)
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                 :: "l"(static_cast<char*>(a.params16[r]) + t0 * kEB), "r"(sp), "r"(bytes)
                                 : "memory");
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        const int done = (int)(bytes / kEB);
        const int rest = (int)(tel - done);                          // < 16 bytes' worth
        for (int q = threadIdx.x; q < rest * a.n_ranks; q += kThreads) {
            const int r = q / rest, j = done + q % rest;
            const uint32_t pv = tile[b][j / V].get(j % V);
            if constexpr (kEB == 4)
                static_cast<uint32_t*>(a.params16[r])[t0 + j] = pv;
            else
                static_cast<uint16_t*>(a.params16[r])[t0 + j] = (uint16_t)pv;
        }
    }
    // the bulk copies complete before the kernel does
    if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    wait_prev_grid();
}

template <int STAGE, int DT, bool CLIP, int OPT>
cudaError_t run_update(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    if constexpr (STAGE == 1 || STAGE == 2) {
        if (a.n_ranks >= kBulkMinRanks && device_resident(a.params16, a.n_ranks, s)) {
            const int64_t tiles = (groups + kThreads * kTileSub - 1) / (kThreads * kTileSub);
            const int resident = grid_for((const void*)k_update_tiled<STAGE, DT, CLIP, OPT>, tiles * kThreads * 4);
            const int grid = (int)(tiles < 2LL * resident ? tiles : 2LL * resident);
            return launch_step_kernel(k_update_tiled<STAGE, DT, CLIP, OPT>, grid, s, overlap, a);
        }
    }
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

namespace {
template <int STAGE, int DT, bool CLIP, int OPT>
cudaError_t run_update_one(const StepArgs& a, const CommitArgs& c, cudaStream_t s)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaErrorInvalidValue;
    const int grid = grid_for((const void*)k_update_one<STAGE, DT, CLIP, OPT>, groups);
    return launch_kernel(k_update_one<STAGE, DT, CLIP, OPT>, grid, kThreads, s, true, a, c);
}

template <int STAGE, int DT, bool CLIP>
cudaError_t update_one_opt(int opt, const StepArgs& a, const CommitArgs& c, cudaStream_t s)
{
    switch (opt) {
    case kSgdm: return run_update_one<STAGE, DT, CLIP, kSgdm>(a, c, s);
    case kSgd: return run_update_one<STAGE, DT, CLIP, kSgd>(a, c, s);
    default: return run_update_one<STAGE, DT, CLIP, kAdam>(a, c, s);
    }
}

template <int DT, bool CLIP>
cudaError_t update_one_stage(int stage, int opt, const StepArgs& a, const CommitArgs& c, cudaStream_t s)
{
    if (stage == 2) return update_one_opt<2, DT, CLIP>(opt, a, c, s);
    if (stage == 3) return update_one_opt<3, DT, CLIP>(opt, a, c, s);
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_update_one(int stage, int dtype, int opt, bool clip, const StepArgs& a, const CommitArgs& c,
                              cudaStream_t s)
{
    if (dtype == kF32) return clip ? cudaErrorNotSupported : update_one_stage<kF32, false>(stage, opt, a, c, s);
    if (dtype == kBF16) return clip ? update_one_stage<kBF16, true>(stage, opt, a, c, s)
                                    : update_one_stage<kBF16, false>(stage, opt, a, c, s);
    return clip ? update_one_stage<kF16, true>(stage, opt, a, c, s) : update_one_stage<kF16, false>(stage, opt, a, c, s);
}

}  // namespace zg

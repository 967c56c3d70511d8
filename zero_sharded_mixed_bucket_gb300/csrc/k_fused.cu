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
#include "host_ptrs.h"

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
    // Stages 2 and 3: nothing to do once the step has overflowed (the flag
    // was cleared before the step's first bucket kernel started).
    if constexpr (STAGE >= 2) {
        if (flag_raised(a.ws)) {
            wait_prev_grid();
            return;
        }
    }
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
        raise_flag(a.ws, round_group<DT>(s, h), bad);
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
    if constexpr (STAGE >= 2) {
        if (threadIdx.x == 0) note_updated(a.ws, a.lo, a.hi, block_elems_grid_stride(a.lo, a.hi, kVecOf<DT>));
    }
    wait_prev_grid();
}

// Stages 1 and 2 with their replicated outputs -- the new parameters, and in
// stage 1 the all-reduced gradient, each written to every rank -- through
// shared memory: a block computes a tile of kTileSub x kThreads groups, then
// the lanes of warp 0 copy the tile(s) to each rank with bulk asynchronous
// copies (cp.async.bulk shared -> global), one rank per lane.  Two tile
// buffers; a buffer is rewritten after the copies that read it two tiles
// earlier have read it (wait_group.read).  The ragged end of a bucket (less
// than 16 bytes) is stored by the threads.  Two blocks per resident slot:
// one block's loads and arithmetic overlap another's copies.  Measured A/B
// on the 12-layer d=768 list, N_d = 8: stage 1 6352 -> 6595 GB/s, 0.936 ->
// 0.971 of the copy bandwidth with one block per slot, and 1.359-1.362 ->
// 1.329-1.331 ms per step with two (tiles of 4 x 128 groups: the same).
// Stage 2 takes the tiles where the replicated parameters are a large share
// of the traffic: SGD and SGD with momentum (16 of 40 and of 48 bytes per
// parameter; fp16 0.746 -> 0.730 and 0.896 -> 0.873 ms per step, fp32
// 1.331 -> 1.316 and 1.480 -> 1.461) and binary32 Adam (32 of 88; 1.613 ->
// 1.599).  16-bit Adam (16 of 56) keeps per-thread stores: through the
// tiles it measured 1.037-1.042 ms per step against 1.012-1.014.
constexpr int kTileSub = 2;

template <int STAGE, int DT, int OPT>
constexpr bool tiled_step()
{
    return STAGE == 1 || (STAGE == 2 && (OPT != kAdam || DT == kF32));
}

template <int STAGE, int DT, int OPT>
__global__ void __launch_bounds__(kThreads) k_fused_tiled(const __grid_constant__ StepArgs a)
{
    static_assert(STAGE == 1 || STAGE == 2, "outputs replicated to every rank: stages 1 and 2");
    constexpr int V = kVecOf<DT>;
    constexpr int kEB = DT == kF32 ? 4 : 2;                        // bytes per value
    constexpr int kArrays = STAGE == 1 ? 2 : 1;                    // parameters (, gradient)
    constexpr int kTileGroups = kThreads * kTileSub;
    constexpr int64_t kTileElems = (int64_t)kTileGroups * V;
    __shared__ __align__(128) Vals<DT> tile[2][kArrays][kTileGroups];
    if (a.wait_first) wait_prev_grid();
    allow_next_grid();
    if constexpr (STAGE == 2) {   // nothing to do once the step has overflowed (as k_fused)
        if (flag_raised(a.ws)) {
            wait_prev_grid();
            return;
        }
    }
    float inv = a.inv;
    AdamHP hp = a.hp;
    if (a.dyn) {
        inv = a.dyn->inv;
        hp.bc1 = a.dyn->bc1;
        hp.bc2 = a.dyn->bc2;
    }
    const int64_t ntiles = (a.hi - a.lo + kTileElems - 1) / kTileElems;
    bool bad = false;
    int b = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, b ^= 1) {
        if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const int64_t t0 = a.lo + t * kTileElems;                   // first element of the tile
        const int64_t tel = min(kTileElems, a.hi - t0);              // elements in the tile
        for (int k = 0; k < kTileSub; k++) {
            const int gl = k * kThreads + threadIdx.x;               // group within the tile
            const int64_t i = t0 + (int64_t)gl * V;
            if (i >= a.hi) break;
            const int cnt = (int)min((int64_t)V, a.hi - i);
            float s[V];
            reduce_group<DT>(a, i - a.grad_base, cnt, s);
            Vals<DT> h;
            raise_flag(a.ws, round_group<DT>(s, h), bad);
            float g[V];
            unscale_group<DT>(h, inv, g);
            Vals<DT> p;
            update_state<DT, OPT>(a, hp, i, cnt, g, p);
            tile[b][0][gl] = p;
            if constexpr (STAGE == 1) tile[b][kArrays - 1][gl] = h;
        }
        // make the tiles visible to the bulk-copy (async) proxy, then copy them out
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        const uint32_t bytes = (uint32_t)(tel * kEB) & ~15u;
        if (threadIdx.x < 32) {   // one rank per lane
            if (bytes) {
                const uint32_t sp = (uint32_t)__cvta_generic_to_shared(&tile[b][0][0]);
                const uint32_t sg = (uint32_t)__cvta_generic_to_shared(&tile[b][kArrays - 1][0]);
                for (int r = threadIdx.x; r < a.n_ranks; r += 32) {
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                 :: "l"(static_cast<char*>(a.params16[r]) + t0 * kEB), "r"(sp), "r"(bytes)
                                 : "memory");
                    if constexpr (STAGE == 1)
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                     :: "l"(static_cast<char*>(const_cast<void*>(a.grads[r])) +
                                            (t0 - a.grad_base) * kEB),
                                     "r"(sg), "r"(bytes)
                                     : "memory");
                }
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        const int done = (int)(bytes / kEB);
        const int rest = (int)(tel - done);                          // < 16 bytes' worth
        for (int q = threadIdx.x; q < rest * a.n_ranks; q += kThreads) {
            const int r = q / rest, j = done + q % rest;
            const uint32_t pv = tile[b][0][j / V].get(j % V);
            const uint32_t hv = tile[b][kArrays - 1][j / V].get(j % V);
            if constexpr (kEB == 4) {
                static_cast<uint32_t*>(a.params16[r])[t0 + j] = pv;
                if constexpr (STAGE == 1)
                    static_cast<uint32_t*>(const_cast<void*>(a.grads[r]))[t0 - a.grad_base + j] = hv;
            } else {
                static_cast<uint16_t*>(a.params16[r])[t0 + j] = (uint16_t)pv;
                if constexpr (STAGE == 1)
                    static_cast<uint16_t*>(const_cast<void*>(a.grads[r]))[t0 - a.grad_base + j] = (uint16_t)hv;
            }
        }
    }
    if constexpr (STAGE == 2) {
        if (threadIdx.x == 0) note_updated(a.ws, a.lo, a.hi, block_elems_tile_stride(a.lo, a.hi, kTileElems));
    }
    // the bulk copies complete before the kernel does
    if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// The same restore in stages 1 and 2 with two or more ranks, whose output
// is the same tile written to every rank: the cast goes to a shared-memory
// tile of kRestoreTileSub x kThreads groups and the lanes of warp 0 copy it
// to the ranks with bulk asynchronous copies, as the two-pass update does
// (two tile buffers, two blocks per resident slot).
constexpr int kRestoreTileSub = 4;

template <int DT>
__global__ void __launch_bounds__(kThreads) k_restore_tiled(const __grid_constant__ StepArgs a)
{
    constexpr int V = kVecOf<DT>;
    constexpr int kEB = DT == kF32 ? 4 : 2;                        // bytes per value
    constexpr int kTileGroups = kThreads * kRestoreTileSub;
    constexpr int64_t kTileElems = (int64_t)kTileGroups * V;
    __shared__ __align__(128) Vals<DT> tile[2][kTileGroups];
    const int64_t ntiles = (a.hi - a.lo + kTileElems - 1) / kTileElems;
    int b = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, b ^= 1) {
        if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const int64_t t0 = a.lo + t * kTileElems;
        const int64_t tel = min(kTileElems, a.hi - t0);
        for (int k = 0; k < kRestoreTileSub; k++) {
            const int gl = k * kThreads + threadIdx.x;
            const int64_t i = t0 + (int64_t)gl * V;
            if (i >= a.hi) break;
            const int cnt = (int)min((int64_t)V, a.hi - i);
            float w[V];
            ld_f<V>(a.w_in, i, cnt, w);
            Vals<DT> p;
#pragma unroll
            for (int j = 0; j < V; j++)
                p.set(j, from_f32<DT>(w[j]));
            tile[b][gl] = p;
        }
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
    if (threadIdx.x < 32) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int STAGE, int DT, int OPT>
cudaError_t run_fused3(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    if constexpr (tiled_step<STAGE, DT, OPT>()) {
        // device memory only (the bulk copies write the ranks' parameters, and
        // in stage 1 their gradients); stage 2 from two ranks
        if ((STAGE == 1 || a.n_ranks >= 2) && device_resident(const_cast<void* const*>(a.params16), a.n_ranks, s) &&
            (STAGE == 2 || device_resident(const_cast<void* const*>(a.grads), a.n_ranks, s))) {
            const int64_t tiles = (groups + kThreads * kTileSub - 1) / (kThreads * kTileSub);
            const int resident = grid_for((const void*)k_fused_tiled<STAGE, DT, OPT>, tiles * kThreads * 4);
            const int grid = (int)(tiles < 2LL * resident ? tiles : 2LL * resident);
            return launch_step_kernel(k_fused_tiled<STAGE, DT, OPT>, grid, s, overlap, a);
        }
    }
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
    if constexpr (STAGE == 1 || STAGE == 2) {
        if (a.n_ranks >= 2 && device_resident(a.params16, a.n_ranks, s)) {
            const int64_t tiles = (groups + kThreads * kRestoreTileSub - 1) / (kThreads * kRestoreTileSub);
            const int resident = grid_for((const void*)k_restore_tiled<DT>, tiles * kThreads * 4);
            const int grid = (int)(tiles < 2LL * resident ? tiles : 2LL * resident);
            k_restore_tiled<DT><<<grid, kThreads, 0, s>>>(a);
            return cudaGetLastError();
        }
    }
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

// Two-pass step, used with gradient-norm clipping (the update needs the global
// norm first) or when no shadow state is given.
//   pass 1, per bucket  k_reduce:   rank-order reduce, overflow flag, reduced
//                                   gradient materialised (all ranks' grad
//                                   buffers in stages 0/1 -- the all-reduce --,
//                                   the owner's reduced shard in stages 2/3),
//                                   exact integer sum of squares.
//   once                k_finalize: exact sum -> fp64 -> ||g||, clip coefficient.
//   pass 2, per bucket  k_update:   optimizer update in place (k_update.cu).
#include <cstdlib>
#include <mutex>

#include "dev_state.cuh"
#include "host_ptrs.h"

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
        if constexpr (DT == kBF16)
            sumsq_group_bf16(h, win_lo, acc, bins);
        else
            sumsq_group_f16(h, acc, bad);
    }
    if constexpr (HDEST == 0) {
        for (int r = 0; r < a.n_ranks; r++)
            st_vals<DT>(const_cast<void*>(a.grads[r]), gidx, h, cnt);
    } else {
        st_vals<DT>(a.reduced, i, h, cnt);
    }
}

// The reduced values of one group of one or two ranks' 16-bit gradients as
// packed 16-bit additions: h = (g_0 [+ g_1]) + 0, two values per instruction.
// This equals the rank-order fp32 sum (0 + g_0) + g_1 rounded once to 16 bits:
// the fp32 sum of two 16-bit values is exact when their significands (11 bits
// for binary16, 8 for bfloat16) fit together in fp32's 24, and otherwise the
// smaller one lies below a quarter of the larger one's 16-bit ulp, so the
// correctly rounded 16-bit sum and the rounded fp32 sum are both the larger
// value; a single value is rounded exactly.  The trailing + 0 gives -0 + -0 the
// +0 that (0 + -0) + -0 has.  Returns nonzero if any h is inf or NaN.
template <int DT, int NR, bool TEST = true>
__device__ __forceinline__ uint32_t sum16_group(const H16<8> q[NR], H16<8>& h)
{
    static_assert(NR == 1 || NR == 2, "one or two ranks");
    uint32_t nf = 0;
#pragma unroll
    for (int p = 0; p < 4; p++) {
        uint32_t w;
        if constexpr (DT == kBF16) {
            __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&q[0].w[p]);
            if constexpr (NR == 2) x = __hadd2(x, *reinterpret_cast<const __nv_bfloat162*>(&q[1].w[p]));
            x = __hadd2(x, __float2bfloat162_rn(0.0f));
            w = *reinterpret_cast<const uint32_t*>(&x);
        } else {
            __half2 x = *reinterpret_cast<const __half2*>(&q[0].w[p]);
            if constexpr (NR == 2) x = __hadd2(x, *reinterpret_cast<const __half2*>(&q[1].w[p]));
            x = __hadd2(x, __float2half2_rn(0.0f));
            w = *reinterpret_cast<const uint32_t*>(&x);
        }
        h.w[p] = w;
        if constexpr (TEST) nf |= nonfinite_x2<DT>(w);
    }
    return nf;
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

// ---- pass 1 for one or two ranks (stages 2 and 3), staged ---------------------
// With one or two ranks a group of 8 elements is only one or two 16-byte
// gradient loads, while the exact sum of squares costs a dozen integer
// instructions per value: the per-thread kernel above has to keep many
// groups' loads in flight in registers (124 of them, four blocks per SM) and
// then runs out of warps to hide its integer chains (ALU pipe 58 %, DRAM 33 %
// on GB300).  Here the two jobs are split: in each block one lane of a
// producer warp streams every rank's part of a tile into a ring of
// shared-memory stages with bulk asynchronous copies (cp.async.bulk global ->
// shared, completing on the stage's "full" mbarrier), and eight consumer warps
// do the arithmetic from shared memory and release the stage on its "empty"
// mbarrier.  The bytes in flight no longer depend on how many warps are
// resident.  Grid: at most the blocks that fit at once, each striding over
// the bucket's tiles.  Every wait is bounded: past kWaitNs of global time a
// thread records ZERO_ETIMEOUT's cause in the workspace, raises the overflow
// flag (so the update pass skips the step) and stops.
namespace staged {
constexpr int kWarps = 8;                              // consumer warps
constexpr int kConsumers = kWarps * 32;
constexpr int kBlockThreads = kConsumers + 32;         // and one producer warp
constexpr int kGroupsPerThread = 2;
constexpr int kTileElems = kConsumers * kGroupsPerThread * 8;   // 4096 elements: 8 KB per rank
constexpr int kStages = 4;
constexpr uint64_t kWaitNs = 2000000000ull;            // 2 s

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Wait for the completion of the barrier's phase with parity `parity`;
// false once kWaitNs have passed without it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    const uint32_t addr = smem_addr(bar);
    uint64_t t0 = 0;
    for (uint32_t k = 0;; k++) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(addr), "r"(parity) : "memory");
        if (done) return true;
        if ((k & 63) == 0) {
            const uint64_t now = global_ns();
            if (k == 0) t0 = now;
            else if (now - t0 > kWaitNs) return false;
        }
    }
}

// Global -> shared bulk copy of `bytes` (a multiple of 16, both addresses
// 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void report_timeout(unsigned char* ws)
{
    atomicOr(reinterpret_cast<uint32_t*>(ws + ws::kErr), 1u);
    atomicOr(reinterpret_cast<uint32_t*>(ws + ws::kFlag), 1u);
}
}  // namespace staged

template <int DT, bool CLIP, int NR>
__global__ void __launch_bounds__(staged::kBlockThreads, 2) k_reduce_staged(const __grid_constant__ StepArgs a)
{
    using namespace staged;
    static_assert(NR == 1 || NR == 2, "one or two ranks");
    static_assert(DT != kF32, "16-bit values: groups of 8");
    extern __shared__ __align__(128) unsigned char sm[];   // [kStages][NR][kTileElems] 16-bit values
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ unsigned long long red_lo[kWarps], red_hi[kWarps];
    if (a.wait_first) wait_prev_grid();   // first bucket of a device-state step (see k_fused)
    allow_next_grid();
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int st = 0; st < kStages; st++) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t ntiles = (a.hi - a.lo + kTileElems - 1) / kTileElems;
    uint16_t* stage_base = reinterpret_cast<uint16_t*>(sm);
    if (tid >= kConsumers) {
        if (tid == kConsumers) {   // the producer lane
            int k = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, k++) {
                const int st = k % kStages;
                if (!mbar_wait(&empty[st], ((k / kStages) & 1) ^ 1)) {   // released by the consumers
                    ok = false;
                    break;
                }
                const int64_t t0 = a.lo + t * kTileElems;
                const int64_t tel = min((int64_t)kTileElems, a.hi - t0);
                const uint32_t bytes = (uint32_t)(tel * 2) & ~15u;       // whole groups; a short last group is loaded by its thread
                mbar_arrive_expect_tx(&full[st], NR * bytes);
                // test hook: block 0's first tile announced but never copied
                const bool withhold = a.withhold_tile && blockIdx.x == 0 && k == 0;
                if (bytes && !withhold) {
#pragma unroll
                    for (int r = 0; r < NR; r++)
                        bulk_load(stage_base + (size_t)(st * NR + r) * kTileElems,
                                  static_cast<const uint16_t*>(a.grads[r]) + (t0 - a.grad_base), bytes, &full[st]);
                }
            }
            if (!ok) report_timeout(a.ws);
            // the last fill of every stage has landed before the block exits
            // (each wait bounded; one that runs out does not end the others)
            for (int j = k - kStages < 0 ? 0 : k - kStages; j < k; j++)
                if (!mbar_wait(&full[j % kStages], (j / kStages) & 1)) report_timeout(a.ws);
        }
    } else {
        const int win_lo = a.dyn ? a.dyn->win_lo : a.win_lo;
        bool bad = false;
        U128 acc{0ull, 0ull};
        unsigned long long* bins = ws_bins(a.ws);
        int k = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, k++) {
            const int st = k % kStages;
            if (!mbar_wait(&full[st], (k / kStages) & 1)) {
                report_timeout(a.ws);
                break;
            }
            const int64_t t0 = a.lo + t * kTileElems;
#pragma unroll
            for (int g = 0; g < kGroupsPerThread; g++) {
                const int gl = g * kConsumers + tid;                 // group within the tile
                const int64_t i = t0 + (int64_t)gl * 8;
                if (i < a.hi) {
                    const int cnt = (int)min((int64_t)8, a.hi - i);
                    H16<8> q[NR];
#pragma unroll
                    for (int r = 0; r < NR; r++) {
                        if (cnt == 8) {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                stage_base + (size_t)(st * NR + r) * kTileElems + gl * 8);
                            q[r].w[0] = v.x; q[r].w[1] = v.y; q[r].w[2] = v.z; q[r].w[3] = v.w;
                        } else {
                            q[r] = ld_h16<8>(a.grads[r], i - a.grad_base, cnt);
                        }
                    }
                    // h = round16((0 + g_0) + g_1), as packed 16-bit additions;
                    // clipped binary16 tests for inf/NaN inside the sum of squares
                    H16<8> h;
                    constexpr bool kSumsqTests = CLIP && DT == kF16;
                    bad |= sum16_group<DT, NR, !kSumsqTests>(q, h) != 0;
                    if constexpr (CLIP) {
                        if constexpr (DT == kBF16)
                            sumsq_group_bf16(h, win_lo, acc, bins);
                        else
                            sumsq_group_f16(h, acc, bad);
                    }
                    st_h16<8>(a.reduced, i, h, cnt);
                }
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(&empty[st]);
        }
        if (bad) atomicOr(ws_flag(a.ws), 1u);
        if constexpr (CLIP) {
            // consumer warps only (named barrier 1): one 128-bit sum per block
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned long long lo = __shfl_down_sync(0xffffffffu, acc.lo, off);
                const unsigned long long hi = __shfl_down_sync(0xffffffffu, acc.hi, off);
                u128_add(acc, lo, hi);
            }
            if ((tid & 31) == 0) {
                red_lo[tid >> 5] = acc.lo;
                red_hi[tid >> 5] = acc.hi;
            }
            asm volatile("bar.sync 1, %0;" :: "r"(kConsumers) : "memory");
            if (tid == 0) {
                U128 sum{0ull, 0ull};
                for (int w = 0; w < kWarps; w++)
                    u128_add(sum, red_lo[w], red_hi[w]);
                const unsigned long long l[4] = {sum.lo & 0xffffffffull, sum.lo >> 32, sum.hi & 0xffffffffull,
                                                 sum.hi >> 32};
                unsigned long long* limbs = ws_acc(a.ws);
#pragma unroll
                for (int j = 0; j < 4; j++)
                    if (l[j]) atomicAdd(limbs + j, l[j]);
            }
        }
    }
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

// One warp (lanes 0..31 of the calling block): the lanes read the 256
// exponent bins at once (8 each) and mark the non-zero ones by ballot; lane 0
// then folds the sum's limbs and only those bins into the big integer, in
// exponent order, and writes the norm and the clip coefficient.
__device__ void finalize_norm(unsigned char* ws, int dtype, int win_lo, double inv, double max_norm)
{
    __shared__ unsigned long long sbins[256];
    __shared__ uint32_t nonzero[8];
    const int lane = threadIdx.x;
    const unsigned long long* bins = reinterpret_cast<const unsigned long long*>(ws + ws::kBins);
    unsigned long long b[8];
#pragma unroll
    for (int k = 0; k < 8; k++)
        b[k] = bins[k * 32 + lane];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        sbins[k * 32 + lane] = b[k];
        const uint32_t m = __ballot_sync(0xffffffffu, b[k] != 0ull);
        if (lane == 0) nonzero[k] = m;
    }
    __syncwarp();
    if (lane != 0) return;
    const uint32_t flag = *reinterpret_cast<volatile uint32_t*>(ws + ws::kFlag);
    double* norm_out = reinterpret_cast<double*>(ws + ws::kNorm);
    float* clip_out = reinterpret_cast<float*>(ws + ws::kClip);
    if (flag) {
        *norm_out = __longlong_as_double(0x7ff0000000000000ll);   // +inf
        *clip_out = 1.0f;
        return;
    }
    const int emin = dtype == kBF16 ? -133 : -24;   // E of the smallest subnormal
    unsigned long long big[kBigWords];
    for (int k = 0; k < kBigWords; k++) big[k] = 0ull;
    const unsigned long long* limbs = reinterpret_cast<const unsigned long long*>(ws + ws::kAcc);
    for (int k = 0; k < 4; k++)
        big_add(big, limbs[k], 2 * (win_lo - emin) + 32 * k);
    for (int k = 0; k < 8; k++) {
        for (uint32_t m = nonzero[k]; m; m &= m - 1u) {
            const int e = k * 32 + __ffs(m) - 1;
            const int E = dtype == kBF16 ? (e ? e : 1) - 134 : (e ? e : 1) - 25;
            big_add(big, sbins[e], 2 * (E - emin));
        }
    }
    const double sumsq = big_to_double(big, 2 * emin);
    const double norm = __dmul_rn(__dsqrt_rn(sumsq), inv);
    const double q = __ddiv_rn(max_norm, __dadd_rn(norm, 1e-6));
    *norm_out = norm;
    *clip_out = __double2float_rn(q < 1.0 ? q : 1.0);
}

// Launched as a programmatic dependent of the step's last pass-1 kernel: it
// waits for that kernel (hence every pass-1 kernel) to complete first.
__global__ void k_finalize(const FinalArgs a)
{
    allow_next_grid();   // the first update kernel may launch; it waits for this one
    wait_prev_grid();
    if (blockIdx.x != 0) return;
    finalize_norm(a.ws, a.dtype, a.dyn ? a.dyn->win_lo : a.win_lo, a.dyn ? a.dyn->inv_d : a.inv, a.max_norm);
}

// Pass 1 of a device-state two-pass step whose model is one bucket,
// launched right after the workspace head was cleared (no prepare kernel,
// no finalize kernel): each thread takes the sum-of-squares window from the
// state block's loss scale itself, and the block that finishes last (a
// completion count in the workspace) derives the step's scalars into the
// workspace for pass 2 and the commit and, when clipping, folds the exact
// sum of squares into the norm and the clip coefficient (one warp, as
// k_finalize).  A small step is bound by its kernel boundaries: five
// kernels (prepare, pass 1, finalize, pass 2, commit) become two.
template <int DT, bool CLIP>
__global__ void __launch_bounds__(kThreads) k_reduce_one(const __grid_constant__ StepArgs a, const PrepArgs p,
                                                          double max_norm)
{
    __shared__ int last;
    allow_next_grid();   // pass 2 may launch; it waits for this kernel to complete
    constexpr int V = kVecOf<DT>;
    const int win_lo = CLIP ? window_lo_of(p.st->loss_scale, p.n_ranks, DT) : 0;
    const int64_t ngroups = (a.hi - a.lo + V - 1) / V;
    bool bad = false;
    U128 acc{0ull, 0ull};
    unsigned long long* bins = ws_bins(a.ws);
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups; gi += (int64_t)gridDim.x * kThreads) {
        const int64_t i = a.lo + gi * V;
        const int cnt = (int)min((int64_t)V, a.hi - i);
        const int64_t gidx = i - a.grad_base;
        float s[V];
        reduce_group<DT>(a, gidx, cnt, s);
        finish_group<1, DT, CLIP>(a, i, gidx, cnt, s, win_lo, bad, acc, bins);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        atomicOr(ws_flag(a.ws), 1u);
    if constexpr (CLIP)
        sumsq_flush(acc, ws_acc(a.ws));
    // Count the block done.  The barrier orders its threads' writes (the
    // flag, the bins) before thread 0's device-wide fence, so they are
    // visible before the count is.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(reinterpret_cast<unsigned int*>(a.ws + ws::kDone), 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last || threadIdx.x >= 32) return;
    __threadfence();   // every other block's sums and flag are seen from here on
    const Dyn d = derive_dyn(p.st, p.beta1, p.beta2, p.n_ranks, DT);
    if (threadIdx.x == 0) *p.dyn = d;
    if constexpr (CLIP) finalize_norm(a.ws, DT, d.win_lo, d.inv_d, max_norm);
}

// Launch the staged pass 1: dynamic shared memory for the stage ring, grid
// at most the blocks resident at once.
template <int DT, bool CLIP, int NR>
cudaError_t run_reduce_staged(const StepArgs& a, cudaStream_t s, bool overlap)
{
    using namespace staged;
    auto kernel = k_reduce_staged<DT, CLIP, NR>;
    const int smem = kStages * NR * kTileElems * 2;
    struct Entry {
        int dev;
        int resident;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n_cache = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int resident = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int k = 0; k < n_cache; k++)
            if (cache[k].dev == dev) resident = cache[k].resident;
        if (!resident) {
            e = cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            int sms = 0, per_sm = 0;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)kernel, kBlockThreads, smem);
            resident = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
            if (n_cache < 64) cache[n_cache++] = Entry{dev, resident};
        }
    }
    const int64_t tiles = (a.hi - a.lo + kTileElems - 1) / kTileElems;
    const int grid = (int)(tiles < resident ? tiles : resident);
    // the test hook that withholds a tile (see StepArgs::withhold_tile)
    StepArgs args = a;
    args.withhold_tile = std::getenv("ZERO_TEST_WITHHOLD_TILE") ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kBlockThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

template <int HDEST, int DT, bool CLIP>
cudaError_t run_reduce(const StepArgs& a, cudaStream_t s, bool overlap)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaSuccess;
    if constexpr (HDEST == 1 && DT != kF32) {
        // stages 2/3, one or two ranks, gradients in this GPU's memory: staged
        if (a.n_ranks <= 2 && device_resident(const_cast<void* const*>(a.grads), a.n_ranks, s))
            return a.n_ranks == 2 ? run_reduce_staged<DT, CLIP, 2>(a, s, overlap)
                                  : run_reduce_staged<DT, CLIP, 1>(a, s, overlap);
    }
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

cudaError_t launch_finalize(const FinalArgs& a, cudaStream_t s, bool overlap)
{
    return launch_kernel(k_finalize, 1, 32, s, overlap, a);
}

namespace {
template <int DT, bool CLIP>
cudaError_t run_reduce_one(const StepArgs& a, const PrepArgs& p, double max_norm, cudaStream_t s)
{
    const int64_t groups = (a.hi - a.lo + kVecOf<DT> - 1) / kVecOf<DT>;
    if (groups <= 0) return cudaErrorInvalidValue;
    const int grid = grid_for((const void*)k_reduce_one<DT, CLIP>, groups);
    return launch_kernel(k_reduce_one<DT, CLIP>, grid, kThreads, s, false, a, p, max_norm);
}
}  // namespace

cudaError_t launch_reduce_one(int dtype, bool clip, const StepArgs& a, const PrepArgs& p, double max_norm,
                              cudaStream_t s)
{
    if (dtype == kBF16) return clip ? run_reduce_one<kBF16, true>(a, p, max_norm, s)
                                    : run_reduce_one<kBF16, false>(a, p, max_norm, s);
    if (dtype == kF32) return clip ? cudaErrorNotSupported : run_reduce_one<kF32, false>(a, p, max_norm, s);
    return clip ? run_reduce_one<kF16, true>(a, p, max_norm, s) : run_reduce_one<kF16, false>(a, p, max_norm, s);
}

}  // namespace zg

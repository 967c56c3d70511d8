// P_a, partitioned activation checkpoints ("ZeRO：大模型训练的内存优化革命"
// 3.2.1; SC-2020 ZeRO notes, "P_a: Partitioned Activation Checkpointing"):
// the plan, the partition kernel (each model-parallel rank keeps its slice of
// its own replica of a layer checkpoint) and the all-gather that rebuilds the
// checkpoint (the stage-3 layer gather kernel, over the activation slices).
#include <cstdio>
#include <cstring>

#include "dev_common.cuh"
#include "nvtx_ranges.h"

namespace zg {

namespace {

struct PaArgs {
    const void* src[kMaxRanks];   // rank r's replica, offset to its slice
    void* dst[kMaxRanks];         // rank r's slice buffer
    int64_t len[kMaxRanks];       // 16-bit units in rank r's slice
    int32_t n;
};

// blockIdx.y = rank; groups of 8 16-bit units (16 bytes) per thread.
__global__ void __launch_bounds__(kThreads) k_pa_partition(const __grid_constant__ PaArgs a)
{
    const int r = blockIdx.y;
    const int64_t len = a.len[r];
    const uint16_t* src = static_cast<const uint16_t*>(a.src[r]);
    uint16_t* dst = static_cast<uint16_t*>(a.dst[r]);
    const int64_t groups = (len + 7) / 8;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < groups; g += (int64_t)gridDim.x * kThreads) {
        const int64_t j = g * 8;
        if (j + 8 <= len) {
            __stcs(reinterpret_cast<uint4*>(dst + j), __ldcs(reinterpret_cast<const uint4*>(src + j)));
        } else {
            for (int64_t k = j; k < len; k++) dst[k] = src[k];
        }
    }
}

zero_status_t fail_pa(zero_status_t st, const char* msg) { return set_error(st, msg); }

zero_status_t check_pa_plan(const zero_pa_plan_t* p)
{
    if (!p) return fail_pa(ZERO_EINVAL, "P_a plan is NULL");
    zero_pa_plan_t fresh;
    const zero_status_t st = zero_pa_plan(p->act_elems, p->n_mp, p->dtype, p->align_elems, &fresh);
    if (st != ZERO_OK) return st;
    if (std::memcmp(&fresh, p, sizeof fresh) != 0) return fail_pa(ZERO_EINVAL, "P_a plan was not made by zero_pa_plan");
    return ZERO_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace zg

using namespace zg;

extern "C" {

zero_status_t zero_pa_plan(int64_t act_elems, int32_t n_mp, int32_t dtype, int64_t align_elems, zero_pa_plan_t* out)
{
    if (!out) return set_error(ZERO_EINVAL, "zero_pa_plan: out is NULL");
    if (act_elems < 0 || act_elems > (int64_t(1) << 40))
        return set_error(ZERO_EINVAL, "zero_pa_plan: act_elems must be in 0..2^40");
    if (n_mp < 1 || n_mp > kMaxRanks) return set_error(ZERO_EUNSUPPORTED, "zero_pa_plan: n_mp is outside 1..64");
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16 && dtype != ZERO_FP32)
        return set_error(ZERO_EINVAL, "zero_pa_plan: dtype unknown");
    if (align_elems < 0 || align_elems % 8)
        return set_error(ZERO_EINVAL, "zero_pa_plan: align_elems must be 0 or a positive multiple of 8");
    const int64_t A = align_elems ? align_elems : ZERO_DEFAULT_ALIGN;
    const int64_t b = dtype == ZERO_FP32 ? 4 : 2;
    std::memset(out, 0, sizeof *out);
    out->act_elems = act_elems;
    out->align_elems = align_elems;
    out->n_mp = n_mp;
    out->dtype = dtype;
    const int64_t per = (act_elems + n_mp - 1) / n_mp;
    out->shard_elems = (per + A - 1) / A * A;
    out->mem_per_rank_bytes = act_elems * b;
    out->mem_per_rank_pa_bytes = out->shard_elems * b;
    out->gather_bytes = (int64_t)(n_mp - 1) * act_elems * b;   // every rank receives all slices but its own
    return ZERO_OK;
}

zero_status_t zero_pa_partition(const zero_pa_plan_t* plan, const void* const* replicas, void* const* shards,
                                void* stream)
{
    NvtxRange range("zero_pa_partition");
    zero_status_t st = check_pa_plan(plan);
    if (st != ZERO_OK) return st;
    if (!replicas || !shards) return set_error(ZERO_ENOMEM, "zero_pa_partition: pointer arrays must not be NULL");
    const int64_t u = plan->dtype == ZERO_FP32 ? 2 : 1;   // 16-bit units per value
    PaArgs a;
    std::memset(&a, 0, sizeof a);
    a.n = plan->n_mp;
    int64_t most = 0;
    for (int r = 0; r < plan->n_mp; r++) {
        if (!replicas[r] || !shards[r]) return set_error(ZERO_ENOMEM, "zero_pa_partition: a buffer is NULL");
        if (!aligned16(replicas[r]) || !aligned16(shards[r]))
            return set_error(ZERO_EALIGN, "zero_pa_partition: a buffer is not 16-byte aligned");
        const int64_t lo = (int64_t)r * plan->shard_elems;
        const int64_t own = lo < plan->act_elems ? (plan->act_elems - lo < plan->shard_elems ? plan->act_elems - lo
                                                                                           : plan->shard_elems)
                                                 : 0;
        a.src[r] = static_cast<const uint16_t*>(replicas[r]) + lo * u;
        a.dst[r] = shards[r];
        a.len[r] = own * u;
        if (a.len[r] > most) most = a.len[r];
    }
    if (most == 0) return ZERO_OK;
    const int per_rank = grid_for((const void*)k_pa_partition, (most + 7) / 8);
    int gx = (per_rank + plan->n_mp - 1) / plan->n_mp;   // about one wave in total
    if (gx < 1) gx = 1;
    k_pa_partition<<<dim3(gx, plan->n_mp), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "zero_pa_partition: launch failed: %s", cudaGetErrorString(e));
        return set_error(ZERO_ECUDA, msg);
    }
    return ZERO_OK;
}

zero_status_t zero_pa_gather(const zero_pa_plan_t* plan, const void* const* shards, void* const* dst, int32_t n_dst,
                             void* stream)
{
    NvtxRange range("zero_pa_gather");
    zero_status_t st = check_pa_plan(plan);
    if (st != ZERO_OK) return st;
    if (n_dst < 1 || n_dst > kMaxRanks) return set_error(ZERO_EUNSUPPORTED, "zero_pa_gather: n_dst is outside 1..64");
    if (!shards || !dst) return set_error(ZERO_ENOMEM, "zero_pa_gather: pointer arrays must not be NULL");
    GatherArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < plan->n_mp; r++) {
        if (!shards[r]) return set_error(ZERO_ENOMEM, "zero_pa_gather: a slice buffer is NULL");
        if (!aligned16(shards[r])) return set_error(ZERO_EALIGN, "zero_pa_gather: a slice buffer is not 16-byte aligned");
        a.shards[r] = shards[r];
    }
    for (int d = 0; d < n_dst; d++) {
        if (!dst[d]) return set_error(ZERO_ENOMEM, "zero_pa_gather: a destination is NULL");
        if (!aligned16(dst[d])) return set_error(ZERO_EALIGN, "zero_pa_gather: a destination is not 16-byte aligned");
        a.dst[d] = dst[d];
    }
    const int64_t u = plan->dtype == ZERO_FP32 ? 2 : 1;
    a.start = 0;
    a.len = plan->act_elems * u;
    a.shard = plan->shard_elems * u;
    a.n_dst = n_dst;
    const cudaError_t e = launch_gather(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "zero_pa_gather: launch failed: %s", cudaGetErrorString(e));
        return set_error(ZERO_ECUDA, msg);
    }
    return ZERO_OK;
}

}  // extern "C"

// Stage-3 parameter all-gather of one layer into constant-size destination
// buffers, and the grid-size helper shared by every streaming kernel.
//
// In stage 3 each rank keeps only its 1/N_d shard of the 16-bit parameters; a
// layer's parameters are gathered from their owners before the layer runs
// forward and again before it runs backward, then released, so the gather
// buffer only has to hold the largest layer ("ZeRO：大模型训练的内存优化革命"
// 3.1.3; ZeRO visual reading, communication accounting: the second all-gather
// that makes stage 3 cost 3 Psi; SC-2020 ZeRO notes, C_B constant-size
// buffers).
#include <mutex>

#include "dev_common.cuh"

namespace zg {

namespace {

// Groups of 8 16-bit units (16 bytes) per thread.
constexpr int kG = 8;

__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ GatherArgs a)
{
    const int64_t ngroups = (a.len + kG - 1) / kG;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t j0 = gi * kG;
        const int cnt = (int)min((int64_t)kG, a.len - j0);
        const int64_t i = a.start + j0;
        if (cnt == kG && (i & (kG - 1)) == 0) {
            // shards are multiples of 8 units: an aligned group has one owner
            const int o = owner_of(i, a.shard);
            const uint4 v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.shards[o]) +
                                                                  (i - (int64_t)o * a.shard)));
            for (int d = 0; d < a.n_dst; d++)
                __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dst[d]) + j0), v);
        } else {
            uint16_t u[kG];
#pragma unroll
            for (int j = 0; j < kG; j++) {
                u[j] = 0;
                if (j < cnt) {
                    const int o = owner_of(i + j, a.shard);
                    u[j] = static_cast<const uint16_t*>(a.shards[o])[i + j - (int64_t)o * a.shard];
                }
            }
            for (int d = 0; d < a.n_dst; d++) {
                uint16_t* p = static_cast<uint16_t*>(a.dst[d]) + j0;
#pragma unroll
                for (int j = 0; j < kG; j++)
                    if (j < cnt) p[j] = u[j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s)
{
    const int64_t groups = (a.len + kG - 1) / kG;
    if (groups <= 0) return cudaSuccess;
    const int grid = grid_for((const void*)k_gather, groups);
    k_gather<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

int grid_for(const void* kernel, int64_t groups)
{
    struct Entry {
        const void* k;
        int dev;
        int blocks;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int n_cache = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    int resident = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int k = 0; k < n_cache; k++)
            if (cache[k].k == kernel && cache[k].dev == dev) resident = cache[k].blocks;
        if (!resident) {
            int sms = 0, per_sm = 0;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
            resident = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
            if (n_cache < 256) cache[n_cache++] = Entry{kernel, dev, resident};
        }
    }
    const int64_t need = (groups + kThreads - 1) / kThreads;
    return (int)(need < resident ? need : resident);
}

}  // namespace zg

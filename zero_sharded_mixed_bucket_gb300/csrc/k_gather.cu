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
#include <cuda.h>

#include <mutex>

#include "dev_common.cuh"
#include "host_ptrs.h"

namespace zg {

namespace {

constexpr int kG = 8;                 // units per 16-byte group

// Destinations or shards in host memory: each thread reads its 16-byte
// group once and stores it to every destination (each value crosses the
// host link once).
__global__ void __launch_bounds__(kThreads) k_gather_direct(const __grid_constant__ GatherArgs a)
{
    const int64_t ngroups = (a.len + kG - 1) / kG;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups;
         gi += (int64_t)gridDim.x * kThreads) {
        const int64_t j0 = gi * kG;
        const int cnt = (int)min((int64_t)kG, a.len - j0);
        const int64_t i = a.start + j0;
        if (cnt == kG && (i & (kG - 1)) == 0) {
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

// The layer is cut into chunks of kChunk units
// (2 MB) and each chunk into segments of kSeg units (16 KB); a block copies
// one segment of one chunk to one destination -- blockIdx.x the segment,
// blockIdx.y the destination, blockIdx.z the chunk -- with 16-byte loads (L2)
// and stores per thread.  Blocks start in the order of their linear index, x
// fastest, so the device writes the destinations one after another, chunk by
// chunk: each destination's part of a chunk is one sequential sweep, and
// the chunk's source, read from the owners' shards once, stays in L2 for the
// other destinations.  Measured on GB300, 64 destinations (algorithmic
// bytes): 7.53 TB/s on 201 M-unit layers and 7.20 on 2^24-unit ones, against
// 6.77 and 6.43 when each block gathered a tile into shared memory and
// copied it to every destination with bulk copies (many interleaved write
// streams at once), and 6.4-6.5 for per-thread stores without the chunks;
// chunks of 2-4 MB measured the same, 8 MB 2 % less, 16 MB 12 % less.  Eight
// blocks per SM (32 registers): with the owner found by a 64-bit division
// per group, or at 4 blocks per SM, the same order reached only 6.3-6.5.
// Fewer destinations too, against k_gather_direct (201 M / 2^24-unit
// layers, of the copy bandwidth): 1 destination 0.97 / 0.62 against 0.82 /
// 0.56, 2: 0.99 / 0.67 against 0.92 / 0.72, 4: 1.00 / 0.73 against 0.84 /
// 0.67, 7: 1.00 / 0.73 against 0.86 / 0.72.
constexpr int kSegThreads = 256;
constexpr int kPer = 4;                                            // groups per thread
constexpr int64_t kSeg = (int64_t)kSegThreads * kPer * kG;         // 8192 units
constexpr int64_t kChunk = int64_t(1) << 20;                       // 2 MB of 16-bit units
static_assert(kChunk % kSeg == 0, "chunks of whole segments");

// Owner of flat unit i without a 64-bit division: a float estimate of
// i / shard (relative error below 2e-7, and the owner is below 64, so it is
// off by at most one), then one exact integer correction.
__device__ __forceinline__ int owner_fast(int64_t i, int64_t shard, float inv_shard)
{
    int o = (int)((float)i * inv_shard);
    if ((int64_t)(o + 1) * shard <= i)
        o++;
    else if ((int64_t)o * shard > i)
        o--;
    return o;
}

// The cnt units from flat index i, one by one (an unaligned or short group,
// whose units may have different owners).
__device__ __noinline__ uint4 load_units(const GatherArgs& a, int64_t i, int cnt)
{
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < kG; j++) {
        if (j < cnt) {
            const int o = owner_of(i + j, a.shard);
            const uint32_t u = static_cast<const uint16_t*>(a.shards[o])[i + j - (int64_t)o * a.shard];
            w[j >> 1] |= u << ((j & 1) * 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Unit j (constant after unrolling) of a group.
__device__ __forceinline__ uint16_t group_unit(const uint4& v, int j)
{
    const uint32_t w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return (uint16_t)(w >> ((j & 1) * 16));
}

// A thread's groups of a segment that are not all aligned, whole and of
// one owner (a layer that starts off a 16-byte boundary, the layer's ragged
// end, a shard boundary): group by group.
__device__ __noinline__ void gather_groups_slow(const GatherArgs& a, uint16_t* out, int64_t j_first, int nv)
{
    for (int k = 0; k < nv; k++) {
        const int64_t j0 = j_first + (int64_t)k * kSegThreads * kG;
        const int cnt = (int)min((int64_t)kG, a.len - j0);
        const uint4 v = load_units(a, a.start + j0, cnt);
        if (cnt == kG) {
            *reinterpret_cast<uint4*>(out + j0) = v;
        } else {
#pragma unroll
            for (int j = 0; j < kG; j++)
                if (j < cnt) out[j0 + j] = group_unit(v, j);
        }
    }
}

__global__ void __launch_bounds__(kSegThreads, 8) k_gather(const __grid_constant__ GatherArgs a, int64_t chunk,
                                                        float inv_shard)
{
    constexpr int64_t kStride = (int64_t)kSegThreads * kG;          // units between a thread's groups
    const int64_t c_end = min((int64_t)(blockIdx.z + 1) * chunk, a.len);
    const int64_t j_first = (int64_t)blockIdx.z * chunk + (int64_t)blockIdx.x * kSeg + (int64_t)threadIdx.x * kG;
    if (j_first >= c_end) return;
    const int nv = (int)min((int64_t)kPer, (c_end - j_first + kStride - 1) / kStride);   // the thread's groups
    uint16_t* out = static_cast<uint16_t*>(a.dst[blockIdx.y]);
    const int64_t i_first = a.start + j_first;                       // flat unit index
    const int64_t i_last = i_first + (nv - 1) * kStride;             // of the last group
    const int o = owner_fast(i_first, a.shard, inv_shard);
    if ((i_first & (kG - 1)) != 0 || i_last + kG > a.start + a.len || i_last + kG > (int64_t)(o + 1) * a.shard) {
        gather_groups_slow(a, out, j_first, nv);
        return;
    }
    // aligned, whole groups of one owner: 16-byte loads (L2) and stores
    const uint4* sp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.shards[o]) +
                                                     (i_first - (int64_t)o * a.shard));
    uint4* dp = reinterpret_cast<uint4*>(out + j_first);            // destinations are 16-byte aligned
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; k++)
        if (k < nv) v[k] = __ldcg(sp + k * (kStride / kG));
#pragma unroll
    for (int k = 0; k < kPer; k++)
        if (k < nv) dp[k * (kStride / kG)] = v[k];
}

int owner_of_host(int64_t i, int64_t shard) { return (int)(i / shard); }

}  // namespace

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s)
{
    if (a.len <= 0) return cudaSuccess;
    // k_gather reads each chunk's source once per destination (from L2 after
    // the first): only for sources, as well as destinations, in this GPU's
    // memory; a source in host memory would cross the host link n_dst times
    const int o_first = owner_of_host(a.start, a.shard), o_last = owner_of_host(a.start + a.len - 1, a.shard);
    if (!device_resident(const_cast<void* const*>(a.dst), a.n_dst, s) ||
        !device_resident(const_cast<void* const*>(a.shards) + o_first, o_last - o_first + 1, s)) {
        const int grid = grid_for((const void*)k_gather_direct, (a.len + kG - 1) / kG);
        k_gather_direct<<<grid, kThreads, 0, s>>>(a);
        return cudaGetLastError();
    }
    // at most 65535 chunks (the grid's z limit): longer layers take longer
    // chunks, whole segments each
    int64_t chunk = kChunk;
    const int64_t min_chunk = (a.len + 65534) / 65535;
    if (min_chunk > chunk) chunk = (min_chunk + kSeg - 1) / kSeg * kSeg;
    const int64_t first = a.len < chunk ? a.len : chunk;              // units of the first chunk
    const dim3 grid((unsigned)((first + kSeg - 1) / kSeg), (unsigned)a.n_dst, (unsigned)((a.len + chunk - 1) / chunk));
    k_gather<<<grid, kSegThreads, 0, s>>>(a, chunk, 1.0f / (float)a.shard);
    return cudaGetLastError();
}

namespace {

// cuPointerGetAttributes through the runtime's driver entry-point lookup (no
// link against the driver library).  Unlike the one-attribute query it
// succeeds for pointers the driver does not know, reporting them as memory
// type 0.
using PointerAttrsFn = CUresult (*)(unsigned int, CUpointer_attribute*, void**, CUdeviceptr);

PointerAttrsFn pointer_attrs_fn()
{
    static const PointerAttrsFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (PointerAttrsFn) nullptr;
        }
        return reinterpret_cast<PointerAttrsFn>(f);
    }();
    return fn;
}

// Is p plain (not managed) device memory of device `dev`?  Asked of the
// driver each time: an address freed by the caller may later belong to host
// or managed memory.
bool query_device_memory(const void* p, int dev, bool* ok)
{
    *ok = false;
    const PointerAttrsFn fn = pointer_attrs_fn();
    if (!fn) return false;
    unsigned int type = 0;
    unsigned int managed = 0;
    int ordinal = -1;
    CUpointer_attribute attrs[3] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_IS_MANAGED,
                                    CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL};
    void* data[3] = {&type, &managed, &ordinal};
    if (fn(3, attrs, data, (CUdeviceptr) reinterpret_cast<uintptr_t>(p)) != CUDA_SUCCESS) return false;
    *ok = true;
    return type == CU_MEMORYTYPE_DEVICE && !managed && ordinal == dev;
}

}  // namespace

bool device_resident(void* const* ptrs, int n, cudaStream_t stream)
{
    // Outside stream capture every pointer is asked of the driver on every
    // call.  A per-thread table keeps the answers (open addressing; cleared
    // when it fills up) for use while a stream is captured, when no query is
    // made: there a remembered answer stands and an unknown pointer counts
    // as not device memory.
    constexpr int kSlots = 1024;
    struct Entry {
        const void* p;
        int dev;
        bool device;
    };
    thread_local Entry table[kSlots];
    thread_local int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (n < 1) return false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const bool capturing = cs != cudaStreamCaptureStatusNone;
    for (int k = 0; k < n; k++) {
        const void* p = ptrs[k];
        if (!p) return false;
        const uint64_t h = reinterpret_cast<uintptr_t>(p) * 0x9E3779B97F4A7C15ull;
        int slot = (int)(h >> 54);   // 10 bits
        while (table[slot].p && !(table[slot].p == p && table[slot].dev == dev)) slot = (slot + 1) & (kSlots - 1);
        if (capturing) {
            if (!table[slot].p || !table[slot].device) return false;
            continue;
        }
        bool ok = false;
        const bool device = query_device_memory(p, dev, &ok);
        if (!ok) return false;
        if (!table[slot].p) {
            if (used >= kSlots / 2) {   // keep the table sparse
                for (int j = 0; j < kSlots; j++) table[j].p = nullptr;
                used = 0;
                slot = (int)(h >> 54);
            }
            used++;
        }
        table[slot] = Entry{p, dev, device};
        if (!device) return false;
    }
    return true;
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

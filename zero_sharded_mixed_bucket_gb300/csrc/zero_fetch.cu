// Stage 3: layer gathers issued ahead of use under a live-parameter budget.
//
// In stage 3 each layer's parameters are all-gathered before the layer runs
// (forward, then again in reverse for the backward) and released after it
// ("ZeRO：大模型训练的内存优化革命" 3.1.3; ZeRO visual reading, stage-3
// section: the coordinator gathers the next layers ahead of time, and a
// live-parameter cap bounds what is resident at once).  Here the gathered
// copies live in a caller-owned pool of `capacity` elements per destination;
// layers are placed in it as a ring in fetch order and released in the same
// order, so the resident layers never exceed the capacity.  Gathers for up to
// `depth` layers ahead run on a side stream; the caller's stream waits only
// for the layer it asks for, and the side stream waits for a release before
// it reuses the space.
#include <cstdio>
#include <cstring>
#include <new>

#include "nvtx_ranges.h"
#include "zero_internal.h"

namespace zg {
namespace {

constexpr uint32_t kMagic = 0x5a46u;   // 'ZF'
constexpr int kMaxResident = ZERO_FETCH_MAX_RESIDENT;
constexpr int kMaxEvents = 2 * (ZERO_FETCH_MAX_DEPTH + 1);

int64_t round8(int64_t x) { return (x + 7) & ~int64_t(7); }

// FIFO ring allocator over [0, cap): the resident layers in fetch order.
// Plain data (it lives in caller memory, zero-initialised).
struct Ring {
    int64_t cap;
    int32_t first, count;                       // queue of residents (indices into ent)
    struct Ent {
        int32_t pos;
        int64_t off, size;
    } ent[kMaxResident];

    const Ent& oldest() const { return ent[first]; }
    const Ent& newest() const { return ent[(first + count - 1) % kMaxResident]; }

    // Offset for `size` elements, or -1 if it does not fit now.
    int64_t place(int64_t size) const
    {
        if (size > cap || count == kMaxResident) return -1;
        if (count == 0) return 0;
        const int64_t T = oldest().off, H = newest().off + newest().size;
        const bool wrapped = newest().off < T;
        if (!wrapped) {
            if (H + size <= cap) return H;
            if (size <= T) return 0;
            return -1;
        }
        return H + size <= T ? H : -1;
    }
    void push(int32_t pos, int64_t off, int64_t size)
    {
        ent[(first + count) % kMaxResident] = Ent{pos, off, size};
        count++;
    }
    void pop()
    {
        first = (first + 1) % kMaxResident;
        count--;
    }
    int64_t live() const
    {
        int64_t s = 0;
        for (int k = 0; k < count; k++) s += ent[(first + k) % kMaxResident].size;
        return s;
    }
};

struct Fetcher {
    uint32_t magic;
    int32_t n_ranks, n_dst, depth, n_order, n_layers;
    int32_t units;                 // 16-bit units per value: 1, or 2 for binary32
    int64_t shard;
    const int64_t* layer_sizes;    // caller's (config)
    int64_t total;                 // n_params (for a config without layer sizes)
    const int32_t* order;          // caller's
    void* shards[kMaxRanks];
    void* pool[kMaxRanks];
    cudaStream_t side;
    cudaEvent_t ev[kMaxEvents];    // ready[0..depth], released[depth+1..2 depth+1]
    Ring ring;
    int32_t next_issue, next_fetch, next_release, gathers;
    int64_t max_live;
};
static_assert(sizeof(Fetcher) <= sizeof(zero_fetcher_t), "zero_fetcher_t too small");

int64_t layer_len(const int64_t* sizes, int64_t total, int32_t layer)
{
    return sizes ? sizes[layer] : total;
}

int64_t layer_start(const int64_t* sizes, int32_t layer)
{
    int64_t s = 0;
    for (int32_t l = 0; l < layer; l++) s += sizes[l];
    return s;
}

// Issue (in the ring) every position the policy allows before position
// `pos` is used: up to pos + depth, stopping at the first that does not fit.
template <typename OnIssue>
bool issue_for(Ring& ring, int32_t& next_issue, int32_t n, int32_t depth, int32_t pos, const int32_t* order,
               const int64_t* sizes, int64_t total, int64_t& max_live, OnIssue on_issue)
{
    while (next_issue < n && next_issue <= pos + depth) {
        const int64_t size = round8(layer_len(sizes, total, order[next_issue]));
        const int64_t off = ring.place(size);
        if (off < 0) break;
        ring.push(next_issue, off, size);
        const int64_t live = ring.live();
        if (live > max_live) max_live = live;
        if (!on_issue(next_issue, off)) return false;
        next_issue++;
    }
    return next_issue > pos;   // the asked-for position is resident
}

zero_status_t check_order(const zero_config_t* c, const zero_plan_t* p, const int32_t* order, int32_t n_order)
{
    if (!order || n_order <= 0) return set_error(ZERO_EINVAL, "fetch order is empty");
    for (int32_t k = 0; k < n_order; k++)
        if (order[k] < 0 || order[k] >= p->n_layers) return set_error(ZERO_EINVAL, "fetch order names a bad layer");
    (void)c;
    return ZERO_OK;
}

Fetcher* as_fetcher(zero_fetcher_t* f)
{
    Fetcher* F = reinterpret_cast<Fetcher*>(f);
    return (f && F->magic == kMagic) ? F : nullptr;
}

}  // namespace
}  // namespace zg

using namespace zg;

extern "C" {

zero_status_t zero_fetch_schedule(const int64_t* layer_sizes, int32_t n_layers, const int32_t* order, int32_t n_order,
                                  int64_t capacity, int32_t depth, int32_t* issue_at, int64_t* offsets,
                                  int64_t* max_live)
{
    if (!layer_sizes || n_layers <= 0 || !order || n_order <= 0 || !issue_at || !offsets)
        return set_error(ZERO_EINVAL, "zero_fetch_schedule: NULL or empty argument");
    if (depth < 0 || depth > ZERO_FETCH_MAX_DEPTH) return set_error(ZERO_EINVAL, "depth out of range");
    int64_t biggest = 0;
    for (int32_t k = 0; k < n_order; k++) {
        if (order[k] < 0 || order[k] >= n_layers) return set_error(ZERO_EINVAL, "order names a bad layer");
        const int64_t s = round8(layer_sizes[order[k]]);
        if (s <= 0) return set_error(ZERO_EINVAL, "layer size must be positive");
        if (s > biggest) biggest = s;
    }
    if (capacity < biggest) return set_error(ZERO_EINVAL, "capacity is below the largest layer");
    Ring* ring = new (std::nothrow) Ring();
    if (!ring) return set_error(ZERO_ENOMEM, "host allocation failed");
    ring->cap = capacity;
    int32_t next_issue = 0;
    int64_t ml = 0;
    zero_status_t st = ZERO_OK;
    for (int32_t pos = 0; pos < n_order && st == ZERO_OK; pos++) {
        const bool ok = issue_for(*ring, next_issue, n_order, depth, pos, order, layer_sizes, 0, ml,
                                  [&](int32_t q, int64_t off) {
                                      issue_at[q] = pos;
                                      offsets[q] = off;
                                      return true;
                                  });
        if (!ok) st = set_error(ZERO_ENOMEM, "layer does not fit the capacity");
        else ring->pop();   // used, then released (fetch order)
    }
    delete ring;
    if (max_live) *max_live = ml;
    return st;
}

zero_status_t zero_fetcher_init(zero_fetcher_t* f, const zero_config_t* cfg, const zero_plan_t* plan,
                                void* const* param_shards, void* const* pool, int32_t n_dst, int64_t capacity,
                                const int32_t* order, int32_t n_order, int32_t depth, void* side_stream,
                                void* const* events, int32_t n_events)
{
    if (!f) return set_error(ZERO_EINVAL, "fetcher is NULL");
    std::memset(f, 0, sizeof *f);
    zero_plan_t fresh;
    zero_status_t st = zero_plan(cfg, &fresh);
    if (st != ZERO_OK) return st;
    if (!plan || std::memcmp(&fresh, plan, offsetof(zero_plan_t, comm_paper_bytes)) != 0)
        return set_error(ZERO_EINVAL, "plan does not match the config");
    if (cfg->stage != 3) return set_error(ZERO_EINVAL, "layer fetches belong to stage 3");
    if (n_dst < 1 || n_dst > kMaxRanks) return set_error(ZERO_EUNSUPPORTED, "n_dst outside 1..64");
    if (depth < 0 || depth > ZERO_FETCH_MAX_DEPTH) return set_error(ZERO_EINVAL, "depth outside 0..32");
    if (n_events < 2 * (depth + 1) || !events) return set_error(ZERO_EINVAL, "need 2*(depth+1) events");
    st = check_order(cfg, plan, order, n_order);
    if (st != ZERO_OK) return st;
    if (!param_shards || !pool) return set_error(ZERO_ENOMEM, "shard or pool array is NULL");
    int64_t biggest = 0;
    for (int32_t k = 0; k < n_order; k++) {
        const int64_t s = round8(layer_len(cfg->layer_sizes, cfg->n_params, order[k]));
        if (s > biggest) biggest = s;
    }
    if (capacity < biggest) return set_error(ZERO_EINVAL, "capacity is below the largest layer in the order");
    Fetcher* F = reinterpret_cast<Fetcher*>(f);
    for (int r = 0; r < cfg->n_ranks; r++) {
        if (!param_shards[r] || (reinterpret_cast<uintptr_t>(param_shards[r]) & 15))
            return set_error(ZERO_EALIGN, "a parameter shard is NULL or not 16-byte aligned");
        F->shards[r] = param_shards[r];
    }
    for (int d = 0; d < n_dst; d++) {
        if (!pool[d] || (reinterpret_cast<uintptr_t>(pool[d]) & 15))
            return set_error(ZERO_EALIGN, "a pool buffer is NULL or not 16-byte aligned");
        F->pool[d] = pool[d];
    }
    for (int k = 0; k < 2 * (depth + 1); k++) {
        if (!events[k]) return set_error(ZERO_EINVAL, "an event is NULL");
        F->ev[k] = static_cast<cudaEvent_t>(events[k]);
    }
    F->n_ranks = cfg->n_ranks;
    F->n_dst = n_dst;
    F->depth = depth;
    F->n_order = n_order;
    F->n_layers = (int32_t)plan->n_layers;
    F->units = cfg->dtype == ZERO_FP32 ? 2 : 1;
    F->shard = plan->shard_elems;
    F->layer_sizes = cfg->layer_sizes;
    F->total = cfg->n_params;
    F->order = order;
    F->side = static_cast<cudaStream_t>(side_stream);
    F->ring.cap = capacity;
    F->magic = kMagic;
    return ZERO_OK;
}

zero_status_t zero_fetch_layer(zero_fetcher_t* f, int32_t pos, void* stream, int64_t* offset)
{
    zg::NvtxRange range("zero_fetch_layer", pos);
    Fetcher* F = as_fetcher(f);
    if (!F) return set_error(ZERO_EINVAL, "fetcher not initialised");
    if (pos != F->next_fetch) return set_error(ZERO_EINVAL, "layers must be fetched in the order's sequence");
    if (F->next_release != pos) return set_error(ZERO_EINVAL, "release the previous layer before the next fetch");
    cudaError_t err = cudaSuccess;
    const bool ok = issue_for(F->ring, F->next_issue, F->n_order, F->depth, pos, F->order, F->layer_sizes,
                              F->total, F->max_live, [&](int32_t q, int64_t off) {
        const int32_t layer = F->order[q];
        GatherArgs a;
        std::memset(&a, 0, sizeof a);
        for (int r = 0; r < F->n_ranks; r++) a.shards[r] = F->shards[r];
        // the gather copies 16-bit units (two per binary32 value); offsets stay in values
        for (int d = 0; d < F->n_dst; d++) a.dst[d] = static_cast<uint16_t*>(F->pool[d]) + off * F->units;
        a.start = (F->layer_sizes ? layer_start(F->layer_sizes, layer) : 0) * F->units;
        a.len = layer_len(F->layer_sizes, F->total, layer) * F->units;
        a.shard = F->shard * F->units;
        a.n_dst = F->n_dst;
        err = launch_gather(a, F->side);
        if (err == cudaSuccess) err = cudaEventRecord(F->ev[q % (F->depth + 1)], F->side);
        F->gathers++;
        return err == cudaSuccess;
    });
    if (err != cudaSuccess) {
        char msg[160];
        std::snprintf(msg, sizeof msg, "issuing a layer gather: %s", cudaGetErrorString(err));
        return set_error(ZERO_ECUDA, msg);
    }
    if (!ok) return set_error(ZERO_ENOMEM, "the layer does not fit the live-parameter capacity");
    err = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), F->ev[pos % (F->depth + 1)], 0);
    if (err != cudaSuccess) return set_error(ZERO_ECUDA, "waiting for the layer's gather");
    F->next_fetch++;
    if (offset) *offset = F->ring.oldest().off;   // the oldest resident is the one asked for
    return ZERO_OK;
}

zero_status_t zero_release_layer(zero_fetcher_t* f, int32_t pos, void* stream)
{
    Fetcher* F = as_fetcher(f);
    if (!F) return set_error(ZERO_EINVAL, "fetcher not initialised");
    if (pos != F->next_release || pos >= F->next_fetch)
        return set_error(ZERO_EINVAL, "layers must be released in fetch order, after their fetch");
    cudaEvent_t ev = F->ev[F->depth + 1 + pos % (F->depth + 1)];
    cudaError_t err = cudaEventRecord(ev, static_cast<cudaStream_t>(stream));
    if (err == cudaSuccess) err = cudaStreamWaitEvent(F->side, ev, 0);   // reuse of the space waits for the release
    if (err != cudaSuccess) return set_error(ZERO_ECUDA, "recording the layer's release");
    F->ring.pop();
    F->next_release++;
    return ZERO_OK;
}

zero_status_t zero_fetcher_stats(const zero_fetcher_t* f, int64_t* max_live, int32_t* gathers)
{
    const Fetcher* F = reinterpret_cast<const Fetcher*>(f);
    if (!f || F->magic != kMagic) return set_error(ZERO_EINVAL, "fetcher not initialised");
    if (max_live) *max_live = F->max_live;
    if (gathers) *gathers = F->gathers;
    return ZERO_OK;
}

}  // extern "C"

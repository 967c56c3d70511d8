// Host side of the C ABI: planning, argument checks, the step protocol
// (begin / bucket / end), the commit-or-skip decision and the loss scaler;
// and the device-state steps (zero_step_async and the per-bucket async
// protocol), whose commit and scaler run on the GPU (k_async.cu).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "nvtx_ranges.h"
#include "zero_internal.h"

namespace zg {
namespace {

thread_local std::string g_err;
// Caller-created CUDA events recorded around each step's kernels (profiling).
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_end = nullptr;

zero_status_t fail(zero_status_t st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

zero_status_t cuda_fail(cudaError_t e, const char* what)
{
    return fail(ZERO_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// fp32 state bytes per parameter the optimizer keeps (w, m, v / w, m / w).
int64_t state_bytes(int optimizer) { return optimizer == ZERO_SGD ? 4 : (optimizer == ZERO_SGD_MOMENTUM ? 8 : 12); }

// Bytes of one gradient or parameter value: 2 (16-bit types) or 4 (binary32).
int64_t value_bytes(int dtype) { return dtype == ZERO_FP32 ? 4 : 2; }

// Algorithmic HBM bytes per parameter (gradient and parameter values e
// bytes, fp32 state sb bytes, read once and written once).
int64_t bytes_per_param(int stage, int64_t N, bool fused, int64_t sb, int64_t e)
{
    if (fused) {
        switch (stage) {
        case 0: return N * (3 * e + 2 * sb);    // N grads + N write-backs + N x (state r/w + param)
        case 1: return 3 * e * N + 2 * sb;      // N grads + N write-backs + state + N params
        case 2: return 2 * e * N + 2 * sb;      // N grads + state + N params
        default: return e * N + 2 * sb + e;     // N grads + state + owner's param
        }
    }
    switch (stage) {
    case 0: return N * (4 * e + 2 * sb);        // pass 1: 2eN; pass 2: N x (h + state + param)
    case 1: return 3 * e * N + e + 2 * sb;      // pass 1: 2eN; pass 2: h + state + N params
    case 2: return 2 * e * N + 2 * e + 2 * sb;  // pass 1: eN + h; pass 2: h + state + N params
    default: return e * N + 3 * e + 2 * sb;     // pass 1: eN + h; pass 2: h + state + param
    }
}

// Bytes per parameter of the restore after an overflowed fused step: read
// the unchanged master weight, write its cast to each copy (every replica in
// stage 0, every rank in stages 1-2, the owner in stage 3).
int64_t restore_bytes_per_param(int stage, int64_t N, int64_t e)
{
    if (stage == 0) return N * (4 + e);
    if (stage == 3) return 4 + e;
    return 4 + e * N;
}

const int kCollectivePasses[4] = {2, 3, 2, 3};   // RS+AG, AR+AG, RS+AG, RS+2AG

zero_status_t check_config(const zero_config_t* c)
{
    if (!c) return fail(ZERO_EINVAL, "config is NULL");
    if (c->stage < 0 || c->stage > 3) return fail(ZERO_EINVAL, "stage %d is not 0..3", c->stage);
    if (c->n_ranks < 1 || c->n_ranks > kMaxRanks)
        return fail(ZERO_EUNSUPPORTED, "n_ranks %d is outside 1..%d", c->n_ranks, kMaxRanks);
    if (c->n_params < 0) return fail(ZERO_EINVAL, "n_params %lld < 0", (long long)c->n_params);
    if (c->n_params > (int64_t(1) << 40))
        return fail(ZERO_EUNSUPPORTED, "n_params %lld exceeds 2^40", (long long)c->n_params);
    if (c->bucket_elems <= 0 || c->bucket_elems % 8)
        return fail(ZERO_EINVAL, "bucket_elems %lld must be a positive multiple of 8", (long long)c->bucket_elems);
    if (c->align_elems < 0 || c->align_elems % 8)
        return fail(ZERO_EINVAL, "align_elems %lld must be 0 or a positive multiple of 8", (long long)c->align_elems);
    if (c->dtype != ZERO_FP16 && c->dtype != ZERO_BF16 && c->dtype != ZERO_FP32)
        return fail(ZERO_EINVAL, "dtype %d unknown", c->dtype);
    if (c->optimizer < ZERO_ADAM || c->optimizer > ZERO_SGD)
        return fail(ZERO_EINVAL, "optimizer %d unknown", c->optimizer);
    if (c->layer_sizes) {
        if (c->n_layers <= 0) return fail(ZERO_EINVAL, "layer_sizes given with n_layers %d", c->n_layers);
        int64_t sum = 0;
        for (int32_t l = 0; l < c->n_layers; l++) {
            if (c->layer_sizes[l] <= 0)
                return fail(ZERO_EINVAL, "layer %d has size %lld", l, (long long)c->layer_sizes[l]);
            sum += c->layer_sizes[l];
        }
        if (sum != c->n_params)
            return fail(ZERO_EINVAL, "layer sizes add up to %lld, n_params is %lld", (long long)sum,
                        (long long)c->n_params);
    } else if (c->n_layers != 0) {
        return fail(ZERO_EINVAL, "n_layers %d without layer_sizes", c->n_layers);
    }
    return ZERO_OK;
}

void model_state(int64_t psi, int32_t n, int32_t stage, int32_t b, int32_t K, double out[4])
{
    const double P = (double)psi;
    double params = b * P, grads = b * P, optim = K * P;
    if (stage >= 1) optim /= n;
    if (stage >= 2) grads /= n;
    if (stage >= 3) params /= n;
    out[0] = params;
    out[1] = grads;
    out[2] = optim;
    out[3] = params + grads + optim;
}

void make_plan(const zero_config_t* c, zero_plan_t* p)
{
    std::memset(p, 0, sizeof *p);
    const int64_t A = c->align_elems ? c->align_elems : ZERO_DEFAULT_ALIGN;
    const int64_t N = c->n_ranks;
    const int64_t psi = c->n_params;
    p->shard_elems = ceil_div(ceil_div(psi, N), A) * A;
    p->padded_elems = N * p->shard_elems;
    p->n_buckets = ceil_div(psi, c->bucket_elems);
    if (c->layer_sizes) {
        p->n_layers = c->n_layers;
        for (int32_t l = 0; l < c->n_layers; l++)
            if (c->layer_sizes[l] > p->max_layer_elems) p->max_layer_elems = c->layer_sizes[l];
    } else {
        p->n_layers = psi > 0 ? 1 : 0;
        p->max_layer_elems = psi;
    }
    p->state_elems = c->stage == 0 ? N * p->padded_elems : p->padded_elems;
    p->param16_elems = c->stage == 3 ? p->shard_elems : p->padded_elems;
    p->grad16_elems = p->padded_elems;
    p->reduced_elems = c->stage >= 2 ? p->padded_elems : 0;
    p->workspace_bytes = ws::kBytes;
    const int64_t sb = state_bytes(c->optimizer);
    const int64_t e = value_bytes(c->dtype);
    p->hbm_bytes_fused = bytes_per_param(c->stage, N, true, sb, e) * psi;
    p->hbm_bytes_two_pass = bytes_per_param(c->stage, N, false, sb, e) * psi;
    p->comm_counted_bytes = (int64_t)kCollectivePasses[c->stage] * (N - 1) * psi * e;
    p->comm_paper_bytes = (c->stage == 3 ? 3.0 : 2.0) * (double)psi * (double)e;
    double m[4];
    model_state(psi, c->n_ranks, c->stage, (int32_t)e, (int32_t)sb, m);
    p->mem_total_bytes = m[3];
}

// Which path a step takes.
struct Path {
    bool clip;
    bool fused;
};

// A two-pass device-state step of a model that is one bucket (stages 2 and
// 3) runs as two kernels (pass 1 finishing the norm, pass 2 committing)
// when it is small -- its gradients, reduced gradient, state and parameters
// within 64 MiB -- since such a step is bound by its kernel boundaries.
constexpr int64_t kTwoKernelBytes = int64_t(64) << 20;

bool two_kernel_step(const zero_config_t* c, const zero_plan_t* p, const Path& path)
{
    if (path.fused || p->n_buckets != 1 || c->stage < 2) return false;
    const int64_t e = c->dtype == ZERO_FP32 ? 4 : 2;
    return c->n_params * (2 * (int64_t)c->n_ranks * e + 2 * e + 24) <= kTwoKernelBytes;
}

// Number of fp32 state arrays the optimizer uses: w; w, m; w, m, v.
int state_arrays(int optimizer) { return optimizer == ZERO_SGD ? 1 : (optimizer == ZERO_SGD_MOMENTUM ? 2 : 3); }

Path choose_path(const zero_config_t* c, const zero_buffers_t* b, const zero_adam_t* adam)
{
    const int sh = 1 - b->cur;
    const float* shadow[3] = {b->w[sh], b->m[sh], b->v[sh]};
    Path p;
    p.clip = adam->max_grad_norm > 0.0f;
    p.fused = !p.clip;
    for (int k = 0; k < state_arrays(c->optimizer); k++)
        p.fused = p.fused && shadow[k] != nullptr;
    return p;
}

zero_status_t check_plan(const zero_config_t* c, const zero_plan_t* plan)
{
    zero_status_t st = check_config(c);
    if (st != ZERO_OK) return st;
    if (!plan) return fail(ZERO_EINVAL, "plan is NULL");
    zero_plan_t fresh;
    make_plan(c, &fresh);
    if (std::memcmp(&fresh, plan, offsetof(zero_plan_t, comm_paper_bytes)) != 0)
        return fail(ZERO_EINVAL, "plan does not match the config (call zero_plan again)");
    return ZERO_OK;
}

zero_status_t check_step(const zero_config_t* c, const zero_plan_t* plan, const zero_buffers_t* b,
                         const zero_adam_t* adam, const zero_state_t* s)
{
    zero_status_t st = check_plan(c, plan);
    if (st != ZERO_OK) return st;
    if (!b || !adam || !s) return fail(ZERO_EINVAL, "buffers, adam and state must not be NULL");
    if (b->cur != 0 && b->cur != 1) return fail(ZERO_EINVAL, "cur is %d, not 0 or 1", b->cur);
    if (!(std::isfinite(adam->lr) && std::isfinite(adam->max_grad_norm)))
        return fail(ZERO_EINVAL, "learning rate and max_grad_norm must be finite");
    if (c->optimizer == ZERO_ADAM &&
        !(adam->beta1 >= 0.0f && adam->beta1 < 1.0f && adam->beta2 >= 0.0f && adam->beta2 < 1.0f &&
          std::isfinite(adam->eps) && adam->eps >= 0.0f))
        return fail(ZERO_EINVAL, "Adam hyper-parameters out of range");
    if (c->optimizer == ZERO_SGD_MOMENTUM && !(std::isfinite(adam->momentum) && adam->momentum >= 0.0f))
        return fail(ZERO_EINVAL, "momentum must be finite and non-negative");
    if (c->dtype == ZERO_FP32 && adam->max_grad_norm > 0.0f)
        return fail(ZERO_EUNSUPPORTED, "gradient clipping is not available with ZERO_FP32");
    if (!(std::isfinite(s->loss_scale) && s->loss_scale > 0.0f))
        return fail(ZERO_EINVAL, "loss_scale must be positive and finite");
    if (s->dynamic && !(std::isfinite(s->min_loss_scale) && s->min_loss_scale > 0.0f))
        return fail(ZERO_EINVAL, "min_loss_scale must be positive and finite");
    if (s->t < 0 || s->growth_interval < 0 || s->good_steps < 0) return fail(ZERO_EINVAL, "negative step counters");
    const int N = c->n_ranks;
    if (!b->params16) return fail(ZERO_ENOMEM, "params16 array is NULL");
    for (int r = 0; r < N; r++) {
        if (!b->params16[r]) return fail(ZERO_ENOMEM, "params16[%d] is NULL", r);
        if (!aligned16(b->params16[r])) return fail(ZERO_EALIGN, "params16[%d] is not 16-byte aligned", r);
    }
    const int cur = b->cur, sh = 1 - b->cur;
    const float* need[3] = {b->w[cur], b->m[cur], b->v[cur]};
    for (int k = 0; k < state_arrays(c->optimizer); k++) {
        if (!need[k]) return fail(ZERO_ENOMEM, "current fp32 state buffer %d is NULL", k);
        if (!aligned16(need[k])) return fail(ZERO_EALIGN, "current fp32 state buffer %d is not 16-byte aligned", k);
    }
    const float* shadow[3] = {b->w[sh], b->m[sh], b->v[sh]};
    for (int k = 0; k < 3; k++)
        if (shadow[k] && !aligned16(shadow[k]))
            return fail(ZERO_EALIGN, "shadow fp32 state buffer %d is not 16-byte aligned", k);
    if (!b->workspace) return fail(ZERO_ENOMEM, "workspace is NULL");
    if (!aligned16(b->workspace)) return fail(ZERO_EALIGN, "workspace is not 16-byte aligned");
    const Path path = choose_path(c, b, adam);
    if (!path.fused && c->stage >= 2) {
        if (!b->reduced) return fail(ZERO_ENOMEM, "the two-pass path needs the reduced-gradient buffer");
        if (!aligned16(b->reduced)) return fail(ZERO_EALIGN, "reduced is not 16-byte aligned");
    }
    return ZERO_OK;
}

zero_status_t check_grads(const zero_config_t* c, void* const* grads, const char* what)
{
    if (!grads) return fail(ZERO_ENOMEM, "%s array is NULL", what);
    for (int r = 0; r < c->n_ranks; r++) {
        if (!grads[r]) return fail(ZERO_ENOMEM, "%s[%d] is NULL", what, r);
        if (!aligned16(grads[r])) return fail(ZERO_EALIGN, "%s[%d] is not 16-byte aligned", what, r);
    }
    return ZERO_OK;
}

// 1 - beta^t: beta^t by repeated fp64 multiplication, then one rounding to
// fp32.  Once beta^k < 2^-60 every later product is smaller still and
// (float)(1 - beta^t) is 1, so the loop may stop there with the same result.
float bias_correction(float beta, int64_t t)
{
    double p = 1.0;
    for (int64_t k = 0; k < t; k++) {
        p *= (double)beta;
        if (p < 0x1p-60) break;
    }
    return (float)(1.0 - p);
}

// Lowest exponent of the exact sum-of-squares window: every binary16 value
// fits (E >= -24); for bfloat16 the window covers |h| in
// [2^-33, 2^1) * 2^ceil(log2(S*N)) -- the gradient scaled by S and summed
// over N ranks.
int window_lo(int dtype, float scale, int n_ranks)
{
    if (dtype == ZERO_FP16) return -24;
    int e = 0;
    std::frexp((double)scale * (double)n_ranks, &e);   // S*N in [2^(e-1), 2^e)
    int lo = -40 + e;
    if (lo < -133) lo = -133;
    if (lo > 88) lo = 88;
    return lo;
}

StepArgs make_args(const zero_config_t* c, const zero_plan_t* p, const zero_buffers_t* b, const zero_adam_t* adam,
                   const zero_state_t* s, bool fused, void* const* grads, int64_t grad_base)
{
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    const int N = c->n_ranks;
    for (int r = 0; r < N; r++) {
        a.grads[r] = grads ? grads[r] : nullptr;
        a.params16[r] = b->params16[r];
    }
    const int cur = b->cur, out = fused ? 1 - b->cur : b->cur;
    a.w_in = b->w[cur];
    a.m_in = b->m[cur];
    a.v_in = b->v[cur];
    a.w_out = b->w[out];
    a.m_out = b->m[out];
    a.v_out = b->v[out];
    a.reduced = b->reduced;
    a.ws = static_cast<unsigned char*>(b->workspace);
    a.grad_base = grad_base;
    a.shard = p->shard_elems;
    a.replica_stride = p->padded_elems;
    a.n_ranks = N;
    a.inv = (float)(1.0 / ((double)s->loss_scale * (double)N));
    a.hp.lr = adam->lr;
    a.hp.b1 = adam->beta1;
    a.hp.omb1 = 1.0f - adam->beta1;
    a.hp.b2 = adam->beta2;
    a.hp.omb2 = 1.0f - adam->beta2;
    a.hp.eps = adam->eps;
    if (c->optimizer == ZERO_ADAM) {
        a.hp.bc1 = bias_correction(adam->beta1, s->t + 1);
        a.hp.bc2 = bias_correction(adam->beta2, s->t + 1);
    }
    a.hp.mu = adam->momentum;
    a.win_lo = window_lo(c->dtype, s->loss_scale, N);
    return a;
}

zero_status_t begin_impl(const zero_buffers_t* b, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(b->workspace, 0, ws::kEnd, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace");
    if (g_prof_start) {
        e = cudaEventRecord(g_prof_start, st);
        if (e != cudaSuccess) return cuda_fail(e, "recording the profiling start event");
    }
    return ZERO_OK;
}

zero_status_t bucket_impl(const zero_config_t* c, const zero_plan_t* p, const zero_buffers_t* b,
                          const zero_adam_t* adam, const zero_state_t* s, int64_t bucket, void* const* bucket_grads,
                          cudaStream_t st, bool overlap)
{
    NvtxRange range("zero_bucket", bucket);
    const Path path = choose_path(c, b, adam);
    const int64_t lo = bucket * c->bucket_elems;
    const int64_t hi = lo + c->bucket_elems < c->n_params ? lo + c->bucket_elems : c->n_params;
    StepArgs a = bucket_grads ? make_args(c, p, b, adam, s, path.fused, bucket_grads, lo)
                              : make_args(c, p, b, adam, s, path.fused, b->grads, 0);
    a.lo = lo;
    a.hi = hi;
    cudaError_t e = path.fused ? launch_fused(c->stage, c->dtype, c->optimizer, a, st, overlap)
                               : launch_reduce(c->stage, c->dtype, path.clip, a, st, overlap);
    if (e != cudaSuccess) return cuda_fail(e, "launching the bucket kernel");
    return ZERO_OK;
}

zero_status_t end_impl(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b, const zero_adam_t* adam,
                       zero_state_t* s, cudaStream_t st, zero_step_result_t* out)
{
    NvtxRange range("zero_step_end");
    const Path path = choose_path(c, b, adam);
    int launches = (int)p->n_buckets;
    cudaError_t e;
    if (!path.fused) {
        if (path.clip) {
            FinalArgs f;
            f.ws = static_cast<unsigned char*>(b->workspace);
            f.dtype = c->dtype;
            f.win_lo = window_lo(c->dtype, s->loss_scale, c->n_ranks);
            f.inv = (double)(float)(1.0 / ((double)s->loss_scale * (double)c->n_ranks));
            f.max_norm = (double)adam->max_grad_norm;
            f.dyn = nullptr;
            e = launch_finalize(f, st, true);
            if (e != cudaSuccess) return cuda_fail(e, "launching the norm finalize kernel");
            launches++;
        }
        for (int64_t bk = 0; bk < p->n_buckets; bk++) {
            StepArgs a = make_args(c, p, b, adam, s, false, c->stage <= 1 ? b->grads : nullptr, 0);
            a.lo = bk * c->bucket_elems;
            a.hi = a.lo + c->bucket_elems < c->n_params ? a.lo + c->bucket_elems : c->n_params;
            a.wait_first = bk == 0 ? 1 : 0;
            e = launch_update(c->stage, c->dtype, c->optimizer, path.clip, a, st, true);
            if (e != cudaSuccess) return cuda_fail(e, "launching the update kernel");
            launches++;
        }
    }
    if (g_prof_end) {
        e = cudaEventRecord(g_prof_end, st);
        if (e != cudaSuccess) return cuda_fail(e, "recording the profiling end event");
    }
    unsigned char head[ws::kAcc];
    uint64_t wrote[3];   // ~lowest written index, end of the highest written window, elements updated
    e = cudaMemcpyAsync(head, b->workspace, sizeof head, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(wrote, static_cast<unsigned char*>(b->workspace) + ws::kWroteLoC, sizeof wrote,
                            cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the overflow flag");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "synchronising the step");
    uint32_t flag, err;
    double norm;
    float clip;
    std::memcpy(&flag, head + ws::kFlag, 4);
    std::memcpy(&err, head + ws::kErr, 4);
    std::memcpy(&norm, head + ws::kNorm, 8);
    std::memcpy(&clip, head + ws::kClip, 4);
    if (err)   // a kernel gave up a bounded wait; it also raised the flag, so no update ran
        return fail(ZERO_ETIMEOUT, "a bounded wait inside a step kernel ran out; the step was not applied");
    const bool overflow = flag != 0;

    // After an overflowed fused step the 16-bit parameters the bucket kernels
    // wrote are put back.  In stages 2 and 3 the kernels record the window
    // they wrote (kernels that started after the flag was raised wrote
    // nothing); stages 0 and 1 write everywhere.
    const bool skips = path.fused && c->stage >= 2;
    int64_t rlo = 0, rhi = overflow && path.fused ? c->n_params : 0;
    if (overflow && skips) {
        rlo = wrote[0] ? (int64_t)~wrote[0] : 0;
        rhi = wrote[0] ? (int64_t)wrote[1] : 0;
    }
    if (rhi > rlo) {
        StepArgs a = make_args(c, p, b, adam, s, false, nullptr, 0);
        a.lo = rlo;
        a.hi = rhi;
        e = launch_restore(c->stage, c->dtype, a, st);
        if (e != cudaSuccess) return cuda_fail(e, "launching the parameter restore kernel");
        launches++;
    }

    zero_step_result_t r;
    std::memset(&r, 0, sizeof r);
    r.overflow = overflow ? 1u : 0u;
    r.skipped = overflow ? 1 : 0;
    r.loss_scale_used = s->loss_scale;
    r.path = path.fused ? 0 : 1;
    r.grad_norm = path.clip ? (overflow ? INFINITY : norm) : -1.0;
    r.clip_coef = path.clip && !overflow ? clip : 1.0f;
    r.hbm_bytes = path.fused ? p->hbm_bytes_fused : p->hbm_bytes_two_pass;
    r.comm_counted_bytes = p->comm_counted_bytes;
    if (overflow) {
        // the elements the bucket kernels really updated, and the restore
        if (skips)
            r.hbm_bytes = (int64_t)wrote[2] * bytes_per_param(c->stage, c->n_ranks, true, state_bytes(c->optimizer),
                                                               value_bytes(c->dtype));
        r.hbm_bytes += (rhi - rlo) * restore_bytes_per_param(c->stage, c->n_ranks, value_bytes(c->dtype));
        if (s->dynamic) {
            float h = s->loss_scale * 0.5f;
            s->loss_scale = h > s->min_loss_scale ? h : s->min_loss_scale;
        }
        s->good_steps = 0;
    } else {
        if (path.fused) b->cur = 1 - b->cur;
        s->t += 1;
        s->good_steps += 1;
        if (s->dynamic && s->growth_interval > 0 && s->good_steps >= s->growth_interval) {
            s->loss_scale *= 2.0f;
            s->good_steps = 0;
        }
    }
    r.t = s->t;
    r.new_loss_scale = s->loss_scale;
    r.kernel_launches = launches;
    if (out) *out = r;
    return ZERO_OK;
}

zero_status_t step_impl(int want_stage, const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                        const zero_adam_t* adam, zero_state_t* s, void* stream, zero_step_result_t* out)
{
    NvtxRange range("zero_step", c ? c->stage : -1);
    zero_status_t st = check_step(c, p, b, adam, s);
    if (st != ZERO_OK) return st;
    if (want_stage >= 0 && c->stage != want_stage)
        return fail(ZERO_EINVAL, "zero_step_stage%d called with a stage-%d config", want_stage, c->stage);
    st = check_grads(c, b->grads, "grads");
    if (st != ZERO_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    st = begin_impl(b, cs);
    if (st != ZERO_OK) return st;
    // consecutive bucket kernels launched here overlap their edges
    for (int64_t bk = 0; bk < p->n_buckets; bk++) {
        st = bucket_impl(c, p, b, adam, s, bk, nullptr, cs, bk > 0);
        if (st != ZERO_OK) return st;
    }
    return end_impl(c, p, b, adam, s, cs, out);
}

}  // namespace

zero_status_t set_error(zero_status_t st, const char* msg)
{
    g_err = msg;
    return st;
}

// The end of a device-state step after its bucket kernels: the two-pass
// path's norm finalize and update kernels, then the commit (on the fused
// path inside the restore kernel, which also undoes an overflowed step).
// The profiling end event, when set, goes right after the bucket or update
// kernels.
zero_status_t async_tail(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b, const zero_adam_t* adam,
                         const zero_state_t* host_view_p, DevState* dst, Dyn* dyn, unsigned char* ws_ptr,
                         const Path& path, cudaStream_t cs, int* launches_p)
{
    const zero_state_t& host_view = *host_view_p;
    int& launches = *launches_p;
    cudaError_t e;
    if (!path.fused) {
        if (path.clip) {
            FinalArgs f;
            f.ws = ws_ptr;
            f.dtype = c->dtype;
            f.win_lo = 0;
            f.inv = 0.0;
            f.max_norm = (double)adam->max_grad_norm;
            f.dyn = dyn;
            e = launch_finalize(f, cs, true);
            if (e != cudaSuccess) return cuda_fail(e, "launching the norm finalize kernel");
            launches++;
        }
        for (int64_t bk = 0; bk < p->n_buckets; bk++) {
            StepArgs a = make_args(c, p, b, adam, &host_view, false, c->stage <= 1 ? b->grads : nullptr, 0);
            a.dyn = dyn;
            a.lo = bk * c->bucket_elems;
            a.hi = a.lo + c->bucket_elems < c->n_params ? a.lo + c->bucket_elems : c->n_params;
            a.wait_first = bk == 0 ? 1 : 0;
            e = launch_update(c->stage, c->dtype, c->optimizer, path.clip, a, cs, true);
            if (e != cudaSuccess) return cuda_fail(e, "launching an update kernel");
            launches++;
        }
    }
    if (g_prof_end && (e = cudaEventRecord(g_prof_end, cs)) != cudaSuccess)
        return cuda_fail(e, "recording the profiling end event");
    CommitArgs ca{dst, dyn, ws_ptr, path.clip ? 1 : 0};
    if (path.fused) {   // restore on overflow, and the commit, in one kernel
        StepArgs a = make_args(c, p, b, adam, &host_view, true, nullptr, 0);
        a.dyn = dyn;
        a.lo = 0;
        a.hi = c->n_params;
        e = launch_restore_async(c->stage, c->dtype, c->optimizer, a, ca, cs, true);
        if (e != cudaSuccess) return cuda_fail(e, "launching the restore and commit kernel");
    } else {
        e = launch_commit(ca, cs, true);
        if (e != cudaSuccess) return cuda_fail(e, "launching the commit kernel");
    }
    launches++;
    return ZERO_OK;
}

}  // namespace zg

using namespace zg;

extern "C" {

zero_status_t zero_plan(const zero_config_t* cfg, zero_plan_t* out)
{
    zero_status_t st = check_config(cfg);
    if (st != ZERO_OK) return st;
    if (!out) return fail(ZERO_EINVAL, "output plan is NULL");
    make_plan(cfg, out);
    return ZERO_OK;
}

zero_status_t zero_plan_bucket(const zero_config_t* cfg, int64_t bk, int64_t* seg, int32_t* n_seg)
{
    zero_status_t st = check_config(cfg);
    if (st != ZERO_OK) return st;
    if (!seg || !n_seg) return fail(ZERO_EINVAL, "seg and n_seg must not be NULL");
    zero_plan_t p;
    make_plan(cfg, &p);
    if (bk < 0 || bk >= p.n_buckets)
        return fail(ZERO_EINVAL, "bucket %lld is outside 0..%lld", (long long)bk, (long long)p.n_buckets - 1);
    const int64_t lo = bk * cfg->bucket_elems;
    const int64_t hi = lo + cfg->bucket_elems < cfg->n_params ? lo + cfg->bucket_elems : cfg->n_params;
    int32_t n = 0;
    for (int32_t r = 0; r < cfg->n_ranks; r++) {
        const int64_t a = lo > r * p.shard_elems ? lo : r * p.shard_elems;
        const int64_t z = hi < (r + 1) * p.shard_elems ? hi : (r + 1) * p.shard_elems;
        if (a < z) {
            seg[3 * n] = r;
            seg[3 * n + 1] = a - r * p.shard_elems;
            seg[3 * n + 2] = z - a;
            n++;
        }
    }
    *n_seg = n;
    return ZERO_OK;
}

zero_status_t zero_plan_layer(const zero_config_t* cfg, int32_t layer, int64_t* start, int64_t* len)
{
    zero_status_t st = check_config(cfg);
    if (st != ZERO_OK) return st;
    if (!start || !len) return fail(ZERO_EINVAL, "start and len must not be NULL");
    const int32_t nl = cfg->layer_sizes ? cfg->n_layers : (cfg->n_params > 0 ? 1 : 0);
    if (layer < 0 || layer >= nl) return fail(ZERO_EINVAL, "layer %d is outside 0..%d", layer, nl - 1);
    if (!cfg->layer_sizes) {
        *start = 0;
        *len = cfg->n_params;
        return ZERO_OK;
    }
    int64_t s = 0;
    for (int32_t l = 0; l < layer; l++) s += cfg->layer_sizes[l];
    *start = s;
    *len = cfg->layer_sizes[layer];
    return ZERO_OK;
}

zero_status_t zero_model_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t param_bytes,
                                     int32_t optim_K, double out[4])
{
    if (!out) return fail(ZERO_EINVAL, "out is NULL");
    if (n_params < 0 || n_ranks < 1 || stage < 0 || stage > 3 || param_bytes <= 0 || optim_K < 0)
        return fail(ZERO_EINVAL, "bad accounting arguments");
    model_state(n_params, n_ranks, stage, param_bytes, optim_K, out);
    return ZERO_OK;
}

zero_status_t zero_comm_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t param_bytes,
                              double* paper_per_rank, int64_t* counted_all_ranks)
{
    if (!paper_per_rank || !counted_all_ranks) return fail(ZERO_EINVAL, "output pointers are NULL");
    if (n_params < 0 || n_ranks < 1 || stage < 0 || stage > 3 || param_bytes <= 0)
        return fail(ZERO_EINVAL, "bad accounting arguments");
    *paper_per_rank = (stage == 3 ? 3.0 : 2.0) * (double)n_params * param_bytes;
    *counted_all_ranks = (int64_t)kCollectivePasses[stage] * (n_ranks - 1) * n_params * param_bytes;
    return ZERO_OK;
}

zero_status_t zero_step(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b, const zero_adam_t* adam,
                        zero_state_t* s, void* stream, zero_step_result_t* out)
{
    return step_impl(-1, c, p, b, adam, s, stream, out);
}

#define ZG_STAGE_ENTRY(K)                                                                                   \
    zero_status_t zero_step_stage##K(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,       \
                                     const zero_adam_t* adam, zero_state_t* s, void* stream,                \
                                     zero_step_result_t* out)                                               \
    {                                                                                                       \
        return step_impl(K, c, p, b, adam, s, stream, out);                                                 \
    }
ZG_STAGE_ENTRY(0)
ZG_STAGE_ENTRY(1)
ZG_STAGE_ENTRY(2)
ZG_STAGE_ENTRY(3)

zero_status_t zero_step_begin(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                              const zero_adam_t* adam, const zero_state_t* s, void* stream)
{
    zero_status_t st = check_step(c, p, b, adam, s);
    if (st != ZERO_OK) return st;
    return begin_impl(b, static_cast<cudaStream_t>(stream));
}

zero_status_t zero_step_bucket(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                               const zero_adam_t* adam, const zero_state_t* s, int64_t bucket,
                               void* const* bucket_grads, void* stream)
{
    zero_status_t st = check_step(c, p, b, adam, s);
    if (st != ZERO_OK) return st;
    if (bucket < 0 || bucket >= p->n_buckets)
        return fail(ZERO_EINVAL, "bucket %lld is outside 0..%lld", (long long)bucket, (long long)p->n_buckets - 1);
    if (bucket_grads) {
        if (c->stage < 2)
            return fail(ZERO_EINVAL, "per-bucket gradient buffers need stage 2 or 3 (stages 0/1 keep full gradients)");
        st = check_grads(c, bucket_grads, "bucket_grads");
    } else {
        st = check_grads(c, b->grads, "grads");
    }
    if (st != ZERO_OK) return st;
    // The caller may have run work (a staging refill) since the previous bucket
    // kernel: plain stream order.
    return bucket_impl(c, p, b, adam, s, bucket, bucket_grads, static_cast<cudaStream_t>(stream), false);
}

namespace {
// Arguments of a run of buckets: indices in range, gradient pointers valid.
zero_status_t check_run(const zero_config_t* c, const zero_plan_t* p, const zero_buffers_t* b,
                        const int64_t* buckets, int32_t count, void* const* bucket_grads)
{
    if (count < 0) return fail(ZERO_EINVAL, "count %d < 0", count);
    if (count > 0 && !buckets) return fail(ZERO_EINVAL, "buckets is NULL");
    for (int32_t k = 0; k < count; k++)
        if (buckets[k] < 0 || buckets[k] >= p->n_buckets)
            return fail(ZERO_EINVAL, "buckets[%d] = %lld is outside 0..%lld", k, (long long)buckets[k],
                        (long long)p->n_buckets - 1);
    if (!bucket_grads) return count ? check_grads(c, b->grads, "grads") : ZERO_OK;
    if (c->stage < 2)
        return fail(ZERO_EINVAL, "per-bucket gradient buffers need stage 2 or 3 (stages 0/1 keep full gradients)");
    for (int32_t k = 0; k < count; k++) {
        zero_status_t st = check_grads(c, bucket_grads + (size_t)k * c->n_ranks, "bucket_grads");
        if (st != ZERO_OK) return st;
    }
    return ZERO_OK;
}
}  // namespace

zero_status_t zero_step_buckets(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                                const zero_adam_t* adam, const zero_state_t* s, const int64_t* buckets,
                                int32_t count, void* const* bucket_grads, void* stream)
{
    zero_status_t st = check_step(c, p, b, adam, s);
    if (st != ZERO_OK) return st;
    st = check_run(c, p, b, buckets, count, bucket_grads);
    if (st != ZERO_OK) return st;
    // the first kernel in plain stream order after whatever the caller ran;
    // the rest of the run overlap their edges
    for (int32_t k = 0; k < count; k++) {
        st = bucket_impl(c, p, b, adam, s, buckets[k],
                         bucket_grads ? bucket_grads + (size_t)k * c->n_ranks : nullptr,
                         static_cast<cudaStream_t>(stream), k > 0);
        if (st != ZERO_OK) return st;
    }
    return ZERO_OK;
}

zero_status_t zero_step_end(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b, const zero_adam_t* adam,
                            zero_state_t* s, void* stream, zero_step_result_t* out)
{
    zero_status_t st = check_step(c, p, b, adam, s);
    if (st != ZERO_OK) return st;
    if (c->stage <= 1) {
        st = check_grads(c, b->grads, "grads");
        if (st != ZERO_OK) return st;
    }
    return end_impl(c, p, b, adam, s, static_cast<cudaStream_t>(stream), out);
}

zero_status_t zero_gather_layer(const zero_config_t* c, const zero_plan_t* p, int32_t layer,
                                void* const* param_shards, void* const* dst, int32_t n_dst, void* stream)
{
    NvtxRange range("zero_gather_layer", layer);
    zero_status_t st = check_plan(c, p);
    if (st != ZERO_OK) return st;
    if (c->stage != 3) return fail(ZERO_EINVAL, "layer gathers belong to stage 3 (config has stage %d)", c->stage);
    if (n_dst < 1 || n_dst > kMaxRanks) return fail(ZERO_EUNSUPPORTED, "n_dst %d is outside 1..%d", n_dst, kMaxRanks);
    int64_t start = 0, len = 0;
    st = zero_plan_layer(c, layer, &start, &len);
    if (st != ZERO_OK) return st;
    st = check_grads(c, param_shards, "param_shards");
    if (st != ZERO_OK) return st;
    if (!dst) return fail(ZERO_ENOMEM, "dst array is NULL");
    GatherArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < c->n_ranks; r++) a.shards[r] = param_shards[r];
    for (int d = 0; d < n_dst; d++) {
        if (!dst[d]) return fail(ZERO_ENOMEM, "dst[%d] is NULL", d);
        if (!aligned16(dst[d])) return fail(ZERO_EALIGN, "dst[%d] is not 16-byte aligned", d);
        a.dst[d] = dst[d];
    }
    // the gather copies 16-bit units; a binary32 value is two of them
    const int64_t u = value_bytes(c->dtype) / 2;
    a.start = start * u;
    a.len = len * u;
    a.shard = p->shard_elems * u;
    a.n_dst = n_dst;
    cudaError_t e = launch_gather(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching the layer gather kernel");
    return ZERO_OK;
}

// ---- device-state steps -------------------------------------------------------

static_assert(sizeof(DevState) == sizeof(zero_dev_state_t), "device state block size");
static_assert(ws::kDyn + sizeof(Dyn) <= ws::kBytes, "workspace too small for the step scalars");

zero_status_t zero_dev_state_init(void* dev_state, const zero_adam_t* adam, const zero_state_t* s, void* stream)
{
    if (!dev_state || !adam || !s) return fail(ZERO_EINVAL, "dev_state, adam and state must not be NULL");
    if (!aligned16(dev_state)) return fail(ZERO_EALIGN, "dev_state is not 16-byte aligned");
    if (!(std::isfinite(s->loss_scale) && s->loss_scale > 0.0f) || s->t < 0)
        return fail(ZERO_EINVAL, "loss_scale must be positive and finite, t >= 0");
    if (s->dynamic && !(std::isfinite(s->min_loss_scale) && s->min_loss_scale > 0.0f))
        return fail(ZERO_EINVAL, "min_loss_scale must be positive and finite");
    if (s->growth_interval < 0 || s->good_steps < 0) return fail(ZERO_EINVAL, "negative step counters");
    if (!(adam->beta1 >= 0.0f && adam->beta1 < 1.0f && adam->beta2 >= 0.0f && adam->beta2 < 1.0f))
        return fail(ZERO_EINVAL, "beta1 and beta2 must lie in [0, 1)");
    DevState d;
    std::memset(&d, 0, sizeof d);
    d.t = s->t;
    d.beta1_pow = d.beta2_pow = 1.0;
    // beta^t as the same sequence of multiplications; below 2^-60 the bias
    // correction is 1 whatever follows, so the loop may stop there
    for (int64_t k = 0; k < s->t && (d.beta1_pow >= 0x1p-60 || d.beta2_pow >= 0x1p-60); k++) {
        d.beta1_pow *= (double)adam->beta1;
        d.beta2_pow *= (double)adam->beta2;
    }
    d.loss_scale = s->loss_scale;
    d.min_loss_scale = s->min_loss_scale;
    d.dynamic = s->dynamic;
    d.growth_interval = s->growth_interval;
    d.good_steps = s->good_steps;
    d.last_grad_norm = -1.0;
    d.last_clip_coef = 1.0f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dev_state, &d, sizeof d, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "uploading the device step state");
    return ZERO_OK;
}

zero_status_t zero_step_async(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b, const zero_adam_t* adam,
                              void* dev_state, void* stream, int32_t* kernel_launches)
{
    NvtxRange range("zero_step_async");
    zero_state_t host_view;   // the real step state is on the device; this only passes the host checks
    std::memset(&host_view, 0, sizeof host_view);
    host_view.loss_scale = 1.0f;
    host_view.min_loss_scale = 1.0f;
    zero_status_t st = check_step(c, p, b, adam, &host_view);
    if (st != ZERO_OK) return st;
    st = check_grads(c, b->grads, "grads");
    if (st != ZERO_OK) return st;
    if (!dev_state || !aligned16(dev_state)) return fail(ZERO_EALIGN, "dev_state is NULL or not 16-byte aligned");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const Path path = choose_path(c, b, adam);
    unsigned char* ws_ptr = static_cast<unsigned char*>(b->workspace);
    Dyn* dyn = reinterpret_cast<Dyn*>(ws_ptr + ws::kDyn);
    DevState* dst = static_cast<DevState*>(dev_state);
    int launches = 0;
    PrepArgs pa{dst, dyn, ws_ptr, adam->beta1, adam->beta2, c->n_ranks, c->dtype};
    cudaError_t e;
    if (two_kernel_step(c, p, path)) {
        // the workspace head cleared, then pass 1 and pass 2 (the profiling
        // events, when set, around the two)
        e = cudaMemsetAsync(ws_ptr, 0, ws::kEnd, cs);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace");
        if (g_prof_start && (e = cudaEventRecord(g_prof_start, cs)) != cudaSuccess)
            return cuda_fail(e, "recording the profiling start event");
        StepArgs a1 = make_args(c, p, b, adam, &host_view, false, b->grads, 0);
        a1.lo = 0;
        a1.hi = c->n_params;
        e = launch_reduce_one(c->dtype, path.clip, a1, pa, (double)adam->max_grad_norm, cs);
        if (e != cudaSuccess) return cuda_fail(e, "launching the one-bucket pass-1 kernel");
        StepArgs a2 = make_args(c, p, b, adam, &host_view, false, nullptr, 0);
        a2.dyn = dyn;
        a2.lo = 0;
        a2.hi = c->n_params;
        const CommitArgs ca{dst, dyn, ws_ptr, path.clip ? 1 : 0};
        e = launch_update_one(c->stage, c->dtype, c->optimizer, path.clip, a2, ca, cs);
        if (e != cudaSuccess) return cuda_fail(e, "launching the one-bucket pass-2 kernel");
        if (g_prof_end && (e = cudaEventRecord(g_prof_end, cs)) != cudaSuccess)
            return cuda_fail(e, "recording the profiling end event");
        if (kernel_launches) *kernel_launches = 2;
        return ZERO_OK;
    }
    // Every kernel of the step is a programmatic dependent of the one before
    // it: prepare, restore/commit and the first bucket kernel wait for their
    // predecessor at their start, the other bucket kernels at their end.  The
    // profiling events, when set, sit between the prepare kernel and the
    // first bucket kernel and after the last bucket or update kernel, so they
    // time the bucket kernels alone (those two edges then do not overlap).
    e = launch_prepare(pa, cs, true);   // also clears the workspace head
    if (e != cudaSuccess) return cuda_fail(e, "launching the prepare kernel");
    launches++;
    if (g_prof_start && (e = cudaEventRecord(g_prof_start, cs)) != cudaSuccess)
        return cuda_fail(e, "recording the profiling start event");
    for (int64_t bk = 0; bk < p->n_buckets; bk++) {
        NvtxRange bucket_range("zero_bucket", bk);
        StepArgs a = make_args(c, p, b, adam, &host_view, path.fused, b->grads, 0);
        a.dyn = dyn;
        a.wait_first = bk == 0 ? 1 : 0;
        a.lo = bk * c->bucket_elems;
        a.hi = a.lo + c->bucket_elems < c->n_params ? a.lo + c->bucket_elems : c->n_params;
        e = path.fused ? launch_fused(c->stage, c->dtype, c->optimizer, a, cs, true)
                       : launch_reduce(c->stage, c->dtype, path.clip, a, cs, true);
        if (e != cudaSuccess) return cuda_fail(e, "launching a bucket kernel");
        launches++;
    }
    zero_status_t tst = async_tail(c, p, b, adam, &host_view, dst, dyn, ws_ptr, path, cs, &launches);
    if (tst != ZERO_OK) return tst;
    if (path.fused) b->cur = 1 - b->cur;   // alternate on every call: an overflow copies the state across
    if (kernel_launches) *kernel_launches = launches;
    return ZERO_OK;
}

// ---- device-state steps, one bucket at a time ---------------------------------

namespace {
zero_state_t async_host_view()
{
    zero_state_t v;   // the real step state is on the device; this only passes the host checks
    std::memset(&v, 0, sizeof v);
    v.loss_scale = 1.0f;
    v.min_loss_scale = 1.0f;
    return v;
}
}  // namespace

zero_status_t zero_step_begin_async(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                                    const zero_adam_t* adam, void* dev_state, void* stream)
{
    NvtxRange range("zero_step_begin_async");
    const zero_state_t host_view = async_host_view();
    zero_status_t st = check_step(c, p, b, adam, &host_view);
    if (st != ZERO_OK) return st;
    if (!dev_state || !aligned16(dev_state)) return fail(ZERO_EALIGN, "dev_state is NULL or not 16-byte aligned");
    unsigned char* ws_ptr = static_cast<unsigned char*>(b->workspace);
    PrepArgs pa{static_cast<DevState*>(dev_state), reinterpret_cast<Dyn*>(ws_ptr + ws::kDyn), ws_ptr, adam->beta1,
                adam->beta2, c->n_ranks, c->dtype};
    const cudaError_t e = launch_prepare(pa, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess) return cuda_fail(e, "launching the prepare kernel");
    return ZERO_OK;
}

zero_status_t zero_step_bucket_async(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                                     const zero_adam_t* adam, int64_t bucket, void* const* bucket_grads, void* stream)
{
    const zero_state_t host_view = async_host_view();
    zero_status_t st = check_step(c, p, b, adam, &host_view);
    if (st != ZERO_OK) return st;
    if (bucket < 0 || bucket >= p->n_buckets)
        return fail(ZERO_EINVAL, "bucket %lld is outside 0..%lld", (long long)bucket, (long long)p->n_buckets - 1);
    if (bucket_grads) {
        if (c->stage < 2)
            return fail(ZERO_EINVAL, "per-bucket gradient buffers need stage 2 or 3 (stages 0/1 keep full gradients)");
        st = check_grads(c, bucket_grads, "bucket_grads");
    } else {
        st = check_grads(c, b->grads, "grads");
    }
    if (st != ZERO_OK) return st;
    NvtxRange range("zero_bucket", bucket);
    const Path path = choose_path(c, b, adam);
    const int64_t lo = bucket * c->bucket_elems;
    StepArgs a = bucket_grads ? make_args(c, p, b, adam, &host_view, path.fused, bucket_grads, lo)
                              : make_args(c, p, b, adam, &host_view, path.fused, b->grads, 0);
    a.dyn = reinterpret_cast<const Dyn*>(static_cast<unsigned char*>(b->workspace) + ws::kDyn);
    a.lo = lo;
    a.hi = lo + c->bucket_elems < c->n_params ? lo + c->bucket_elems : c->n_params;
    // the caller may have run work (a staging refill) since the previous kernel: plain stream order
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = path.fused ? launch_fused(c->stage, c->dtype, c->optimizer, a, cs, false)
                                     : launch_reduce(c->stage, c->dtype, path.clip, a, cs, false);
    if (e != cudaSuccess) return cuda_fail(e, "launching the bucket kernel");
    return ZERO_OK;
}

zero_status_t zero_step_buckets_async(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                                      const zero_adam_t* adam, const int64_t* buckets, int32_t count,
                                      void* const* bucket_grads, void* stream)
{
    const zero_state_t host_view = async_host_view();
    zero_status_t st = check_step(c, p, b, adam, &host_view);
    if (st != ZERO_OK) return st;
    st = check_run(c, p, b, buckets, count, bucket_grads);
    if (st != ZERO_OK) return st;
    const Path path = choose_path(c, b, adam);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    for (int32_t k = 0; k < count; k++) {
        NvtxRange range("zero_bucket", buckets[k]);
        const int64_t lo = buckets[k] * c->bucket_elems;
        void* const* g = bucket_grads ? bucket_grads + (size_t)k * c->n_ranks : nullptr;
        StepArgs a = g ? make_args(c, p, b, adam, &host_view, path.fused, g, lo)
                       : make_args(c, p, b, adam, &host_view, path.fused, b->grads, 0);
        a.dyn = reinterpret_cast<const Dyn*>(static_cast<unsigned char*>(b->workspace) + ws::kDyn);
        a.lo = lo;
        a.hi = lo + c->bucket_elems < c->n_params ? lo + c->bucket_elems : c->n_params;
        // the first kernel in plain stream order, the rest overlap their edges
        const cudaError_t e = path.fused ? launch_fused(c->stage, c->dtype, c->optimizer, a, cs, k > 0)
                                         : launch_reduce(c->stage, c->dtype, path.clip, a, cs, k > 0);
        if (e != cudaSuccess) return cuda_fail(e, "launching a bucket kernel");
    }
    return ZERO_OK;
}

zero_status_t zero_step_end_async(const zero_config_t* c, const zero_plan_t* p, zero_buffers_t* b,
                                  const zero_adam_t* adam, void* dev_state, void* stream, int32_t* kernel_launches)
{
    NvtxRange range("zero_step_end_async");
    const zero_state_t host_view = async_host_view();
    zero_status_t st = check_step(c, p, b, adam, &host_view);
    if (st != ZERO_OK) return st;
    if (!dev_state || !aligned16(dev_state)) return fail(ZERO_EALIGN, "dev_state is NULL or not 16-byte aligned");
    const Path path = choose_path(c, b, adam);
    unsigned char* ws_ptr = static_cast<unsigned char*>(b->workspace);
    int launches = 0;
    st = async_tail(c, p, b, adam, &host_view, static_cast<DevState*>(dev_state),
                    reinterpret_cast<Dyn*>(ws_ptr + ws::kDyn), ws_ptr, path, static_cast<cudaStream_t>(stream),
                    &launches);
    if (st != ZERO_OK) return st;
    if (path.fused) b->cur = 1 - b->cur;   // alternate on every call: an overflow copies the state across
    if (kernel_launches) *kernel_launches = launches;
    return ZERO_OK;
}

zero_status_t zero_dev_state_read(const void* dev_state, zero_state_t* s, zero_step_result_t* last, void* stream)
{
    if (!dev_state) return fail(ZERO_EINVAL, "dev_state is NULL");
    DevState d;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&d, dev_state, sizeof d, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device step state");
    if (s) {
        s->t = d.t;
        s->loss_scale = d.loss_scale;
        s->min_loss_scale = d.min_loss_scale;
        s->dynamic = d.dynamic;
        s->growth_interval = d.growth_interval;
        s->good_steps = d.good_steps;
    }
    if (last) {
        std::memset(last, 0, sizeof *last);
        last->t = d.t;
        last->overflow = d.last_overflow & 1u;
        last->skipped = d.last_skipped;
        last->grad_norm = d.last_grad_norm;
        last->clip_coef = d.last_clip_coef;
        last->new_loss_scale = d.loss_scale;
        last->path = -1;
    }
    if (d.last_overflow & 2u)
        return fail(ZERO_ETIMEOUT, "a bounded wait inside the last step's kernels ran out; that step was not applied");
    return ZERO_OK;
}

zero_status_t zero_set_profile_events(void* start_event, void* end_event)
{
    if ((start_event == nullptr) != (end_event == nullptr))
        return fail(ZERO_EINVAL, "give both profiling events or neither");
    g_prof_start = static_cast<cudaEvent_t>(start_event);
    g_prof_end = static_cast<cudaEvent_t>(end_event);
    return ZERO_OK;
}

const char* zero_last_error(void) { return g_err.c_str(); }

int32_t zero_version(void) { return ZERO_GB300_VERSION; }

}  // extern "C"

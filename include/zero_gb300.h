/*
 * zero_gb300.h -- C ABI of the ZeRO sharded mixed-precision optimizer step
 * (Adam; also SGD with momentum and SGD) on one GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * ZeRO-DP partitions a data-parallel job's model states -- optimizer state
 * (stage 1, P_os), gradients (stage 2, P_os+g) and parameters (stage 3,
 * P_os+g+p) -- across the N_d data-parallel ranks, each rank keeping 1/N_d
 * ("ZeRO：大模型训练的内存优化革命" 3.1.1-3.1.3; ZeRO visual reading, stage
 * list).  In mixed precision each parameter carries a 16-bit copy, a 16-bit
 * gradient and 12 bytes of fp32 optimizer state (master weight, momentum,
 * variance) ("AI论文陪读·ZeRO" section 01; ZeRO visual reading, 16Ψ account).
 * One optimizer step of a stage-2 rank is: reduce-scatter the gradients of
 * each constant-size bucket to their owners, update the owned fp32 shard with
 * Adam, cast it to 16 bits and all-gather the new parameters to every rank
 * (ZeRO visual reading, communication accounting; SC-2020 ZeRO notes, "Deep
 * Dive into ZeRO-R / C_B" for the fixed-size fusion buffers).
 *
 * Here the N_d ranks are simulated: each rank's buffers are separate regions
 * of one GPU's memory, and each collective is the memory traffic of the fused
 * kernels.  Per bucket, one kernel reads the N_d ranks' 16-bit gradients,
 * sums them in rank order in fp32, rounds once to 16 bits, checks for inf/NaN
 * (loss-scale overflow), unscales by 1/(S*N_d), applies the optimizer --
 * Adam (Kingma & Ba, Algorithm 1: bias correction, eps outside the square
 * root, no weight decay), or SGD with momentum, or SGD -- to the owned fp32
 * state and writes the 16-bit cast to every rank (stages 0-2) or to the
 * owner's shard (stage 3).  The partition does not change the
 * step's result: every stage gives the same numbers as one unpartitioned step.
 *
 * Layout
 * ------
 *   Psi  = n_params; N = n_ranks; A = align_elems (default 2048).
 *   P    = ceil(Psi / N) rounded up to a multiple of A; rank r owns flat
 *          indices [r*P, (r+1)*P).  padded = N*P.
 *   Buckets are consecutive windows of bucket_elems elements over [0, Psi),
 *   in parameter order; the last one may be shorter.  Padding elements
 *   [Psi, padded) are never read or written by a step (keep them zero).
 *   16-bit buffers hold IEEE binary16 or bfloat16 bit patterns (dtype).
 *   With dtype ZERO_FP32 (fp32 training) the gradient, parameter and
 *   reduced buffers hold binary32 values instead -- 4 bytes per element,
 *   the same element counts -- and the "16-bit" cast is the identity.
 *   Per rank r (device memory, caller-owned):
 *     grads[r]    16-bit gradient, grad16_elems = padded elements, flat index
 *                 order (loss-scaled).  Stages 0 and 1 overwrite it with the
 *                 reduced gradient (the all-reduce result).
 *     params16[r] 16-bit parameters: the full vector (padded elements) in
 *                 stages 0-2; only rank r's shard (P elements) in stage 3.
 *   fp32 state w, m, v: state_elems floats each (the arrays the optimizer
 *   uses; see zero_optimizer_t).  Stages 1-3: the N shards
 *   concatenated, i.e. flat index order (padded elements).  Stage 0: N full
 *   replicas, replica r at offset r*padded.  Two copies of each may be given:
 *   [cur] holds the current state; [1-cur] is the shadow that a fused step
 *   writes the new state into (the step is speculative until the global
 *   overflow flag is known; a clean step then flips cur).
 *   reduced: 16-bit reduced gradient, padded elements in flat order (each
 *   owner's shard), needed by the two-pass path in stages 2 and 3.
 *   workspace: workspace_bytes of device memory, 16-byte aligned; contents
 *   are scratch owned by the library during a step.
 *
 * Paths
 * -----
 *   fused     (no clipping and shadow state given): one kernel per bucket,
 *             state read from [cur] and written to [1-cur].  On overflow the
 *             step is discarded and each written 16-bit parameter is restored
 *             to the cast of the unchanged master weights.  In stages 2 and 3
 *             a bucket kernel that starts after the step's flag is raised
 *             writes nothing, and only the window the others wrote is
 *             restored (hbm_bytes counts what really moved); so the 16-bit
 *             parameters must hold the cast of the current master weights
 *             when a step starts, as every step leaves them.
 *   two-pass  (clipping, or no shadow): pass 1 per bucket reduces and checks
 *             the gradient, materialises it (grads[] in stages 0/1, reduced
 *             in stages 2/3) and accumulates the exact sum of squares; a
 *             one-thread kernel forms the global norm and clip coefficient
 *             (16-bit types only);
 *             pass 2 per bucket updates the state in place, or does nothing
 *             when the flag is set.
 *
 *   Inside zero_step / zero_step_stageK (and the update pass of
 *   zero_step_end) consecutive bucket kernels use programmatic dependent
 *   launch: a bucket kernel may start while its predecessor drains; kernels
 *   still complete in stream order.  Kernels launched by zero_step_bucket
 *   follow plain stream order.
 *
 * Conventions
 * -----------
 *   The caller owns all memory; the library allocates nothing and never
 *   throws.  Between calls it keeps only: per process, the resident-block
 *   count of each kernel on each device (behind a lock); per thread, the
 *   error text, the profiling events, and whether each pointer it was given
 *   for a replicated output is device memory of the current device (asked
 *   of the driver on every call outside stream capture, so a freed address
 *   that later holds host or managed memory is seen as such; while a stream
 *   is captured no query is made and the answer last seen on the thread
 *   stands, an unknown pointer counting as not device memory).  A fetcher's state lives in caller memory.  Several threads
 *   may call at once on different jobs and streams.  Every
 *   function returns a zero_status_t; on failure zero_last_error() gives a
 *   message (thread-local).  Kernels run asynchronously on the caller's stream
 *   (a cudaStream_t passed as void*; NULL = legacy default stream).  The
 *   end of a step synchronises that stream once to read the overflow flag
 *   (zero_step_async, below, keeps the step state on the device instead).
 *   Device pointers must be 16-byte aligned (ZERO_EALIGN otherwise).  Any
 *   pointer the GPU can load from and store to is accepted: on GB300 the
 *   gradients or the fp32 optimizer state may live in pinned host memory,
 *   which the kernels then reach over NVLink-C2C.
 *   Pointer arrays (grads, params16, dst) are host arrays of device
 *   pointers, read during the call only.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_GB300_VERSION 1
#define ZERO_MAX_RANKS 64
#define ZERO_DEFAULT_ALIGN 2048

typedef enum {
    ZERO_OK = 0,
    ZERO_EINVAL = 1,         /* bad argument, inconsistent plan or call order */
    ZERO_EALIGN = 2,         /* a device pointer is not 16-byte aligned */
    ZERO_ENOMEM = 3,         /* a caller-provided buffer is missing or too small */
    ZERO_ECUDA = 4,          /* a CUDA runtime call failed (message has the CUDA error) */
    ZERO_ETIMEOUT = 5,       /* a kernel's bounded wait on its own copies ran out (seconds); the step was not applied */
    ZERO_EUNSUPPORTED = 6    /* n_ranks outside 1..64, or another unsupported size */
} zero_status_t;

/* Model precision of gradients and parameters.  ZERO_FP16 / ZERO_BF16:
 * mixed precision (b = 2 bytes, fp32 master state).  ZERO_FP32: fp32
 * training as in the pages' fp32 SGD and SGD-with-momentum examples (b = 4;
 * ZeRO visual reading, worked examples C): the reduced gradient is the fp32
 * rank-order sum itself and the parameters equal the fp32 master weights
 * bit for bit.  The library still keeps the master shard w apart from the
 * parameter copies (a step can then be discarded), so its state holds 4
 * bytes per parameter more than the pages' K; gradient clipping is not
 * available with ZERO_FP32 (ZERO_EUNSUPPORTED).  The no-allocation stage-2
 * entry point takes 16-bit types only. */
typedef enum { ZERO_FP16 = 0, ZERO_BF16 = 1, ZERO_FP32 = 2 } zero_dtype_t;

/* Optimizer on the fp32 master weights ("ZeRO visual reading", accounting
 * with b and K: mixed-precision Adam K = 12, SGD with momentum K = 8, SGD
 * K = 4, each counting the 4-byte fp32 master copy).  State arrays used:
 * Adam w, m, v; SGD with momentum w, m; SGD w (the others may be NULL). */
typedef enum { ZERO_ADAM = 0, ZERO_SGD_MOMENTUM = 1, ZERO_SGD = 2 } zero_optimizer_t;

/* Job description.  56 bytes. */
typedef struct zero_config {
    int64_t n_params;            /* Psi >= 0 */
    int64_t bucket_elems;        /* B > 0, multiple of 8 (gradient bucket, C_B) */
    int64_t align_elems;         /* A: shard alignment in elements; 0 -> 2048; multiple of 8 */
    const int64_t* layer_sizes;  /* stage-3 gather units in parameter order (sum = Psi); NULL -> one */
    int32_t n_layers;            /* entries in layer_sizes (0 when NULL) */
    int32_t stage;               /* ZeRO-DP stage 0..3 */
    int32_t n_ranks;             /* N_d, 1..64 */
    int32_t dtype;               /* zero_dtype_t of parameters and gradients */
    int32_t optimizer;           /* zero_optimizer_t (0: Adam) */
    int32_t reserved;            /* 0 */
} zero_config_t;

/* Partition and sizes derived from a config by zero_plan.  128 bytes. */
typedef struct zero_plan {
    int64_t shard_elems;         /* P */
    int64_t padded_elems;        /* N*P */
    int64_t n_buckets;           /* ceil(Psi / B) */
    int64_t n_layers;
    int64_t max_layer_elems;     /* capacity of a stage-3 gather destination */
    int64_t state_elems;         /* floats in each of w, m, v: N*P, or N*N*P in stage 0 */
    int64_t param16_elems;       /* per rank: N*P in stages 0-2, P in stage 3 */
    int64_t grad16_elems;        /* per rank: N*P */
    int64_t reduced_elems;       /* N*P in stages 2-3 (two-pass path), else 0 */
    int64_t workspace_bytes;
    int64_t hbm_bytes_fused;     /* algorithmic HBM bytes of one fused step (each array access once) */
    int64_t hbm_bytes_two_pass;  /* algorithmic HBM bytes of one two-pass step */
    int64_t comm_counted_bytes;  /* bytes crossing simulated rank boundaries per step, all ranks */
    double comm_paper_bytes;     /* per rank per step: 2*Psi*b (stages 0-2), 3*Psi*b (stage 3) */
    double mem_total_bytes;      /* per rank, paper formula (b = 2, or 4 for ZERO_FP32; K = the fp32
                                    state bytes kept), see zero_model_state_bytes */
    double reserved;
} zero_plan_t;

/* Optimizer hyper-parameters.  Adam (Kingma & Ba, Algorithm 1) uses lr,
 * beta1, beta2, eps; SGD with momentum (PyTorch's rule without dampening:
 * m' = momentum*m + g, w' = w - lr*m') uses lr and momentum; SGD
 * (w' = w - lr*g) uses lr.  24 bytes. */
typedef struct zero_adam {
    float lr, beta1, beta2, eps;
    float max_grad_norm;         /* > 0: clip the global L2 norm of the unscaled gradient; <= 0: off */
    float momentum;              /* SGD with momentum only */
} zero_adam_t;

/* Host-side step state, read and updated by a step.  32 bytes. */
typedef struct zero_state {
    int64_t t;                   /* Adam steps applied so far; a clean step applies t+1 */
    float loss_scale;            /* S: gradients arrive multiplied by S */
    float min_loss_scale;        /* dynamic scaling never halves below this */
    int32_t dynamic;             /* 0 static scale; 1 halve on overflow, double after growth_interval clean steps */
    int32_t growth_interval;     /* 0: never grow */
    int32_t good_steps;          /* consecutive clean steps (dynamic scaling) */
    int32_t reserved;
} zero_state_t;

/* Caller-owned device buffers (layout above).  88 bytes. */
typedef struct zero_buffers {
    void* const* grads;          /* [N] */
    void* const* params16;       /* [N] */
    float* w[2];
    float* m[2];
    float* v[2];
    void* reduced;
    void* workspace;
    int32_t cur;                 /* 0 or 1; the fused path flips it after a clean step */
    int32_t reserved;
} zero_buffers_t;

/* Outcome of one step.  64 bytes. */
typedef struct zero_step_result {
    int64_t t;                   /* step count after the step */
    int64_t hbm_bytes;           /* algorithmic HBM bytes moved */
    int64_t comm_counted_bytes;  /* bytes crossing simulated rank boundaries */
    double grad_norm;            /* clipping on: ||g||_2 (+inf on overflow); off: -1 */
    uint32_t overflow;           /* 1 if any reduced gradient element was inf or NaN */
    int32_t skipped;             /* 1 if the update was discarded (overflow) */
    float clip_coef;             /* min(1, max_grad_norm/(||g||+1e-6)); 1 when off or skipped */
    float loss_scale_used;
    float new_loss_scale;
    int32_t kernel_launches;     /* kernels this step launched */
    int32_t path;                /* 0 fused, 1 two-pass */
    int32_t reserved;
} zero_step_result_t;

/* ---- planning (host only, no CUDA calls) ------------------------------ */

/* Partition, bucket table sizes, buffer sizes and the paper's accounting for
 * cfg.  Source: the shard rule -- each of the N_d ranks keeps one contiguous
 * 1/N_d of the flattened states, per stage (ZeRO visual reading, stage list;
 * "ZeRO：大模型训练的内存优化革命" 3.1.1-3.1.3) -- the constant-size gradient
 * buckets (same page, 3.2.2, C_B; SC-2020 ZeRO notes, "Deep Dive into
 * ZeRO-R") and the per-stage memory and communication formulas (ZeRO visual
 * reading, stage formulas and communication accounting).  The shard is padded
 * to align_elems (a layout choice the pages leave open).  cfg and out are
 * caller memory; nothing is kept.  Errors: ZERO_EINVAL (bad field or NULL),
 * ZERO_EUNSUPPORTED (n_ranks outside 1..64, n_params above 2^40). */
zero_status_t zero_plan(const zero_config_t* cfg, zero_plan_t* out);

/* Segments of bucket b: for each rank owning part of it, in rank order,
 * seg[3k] = rank, seg[3k+1] = offset inside that rank's shard, seg[3k+2] =
 * length -- where the reduce-scatter of one fusion bucket sends its
 * elements ("ZeRO：大模型训练的内存优化革命" 3.1.2 and 3.2.2; ZeRO visual
 * reading, stage list: the owner of a gradient shard reduces it).  seg must
 * hold 3*n_ranks entries; *n_seg receives the count.  Errors: ZERO_EINVAL
 * (b outside 0..n_buckets-1, NULL output), as zero_plan for cfg. */
zero_status_t zero_plan_bucket(const zero_config_t* cfg, int64_t b, int64_t* seg, int32_t* n_seg);

/* Flat start and length of stage-3 layer `layer`: the unit that stage 3
 * gathers before the layer runs and releases after it
 * ("ZeRO：大模型训练的内存优化革命" 3.1.3; ZeRO visual reading, stage-3
 * section).  Errors: ZERO_EINVAL (layer out of range, NULL output). */
zero_status_t zero_plan_layer(const zero_config_t* cfg, int32_t layer, int64_t* start, int64_t* len);

/* Per-rank model-state bytes of the paper's accounting (ZeRO visual reading,
 * stage formulas; Table 1): out[0] parameters, out[1] gradients, out[2]
 * optimizer state, out[3] total.  param_bytes b (2 mixed precision, 4 fp32),
 * optim_K K (12 mixed-precision Adam; the page's calculator also uses 4 for
 * fp32 SGD with momentum, 0 for SGD).  Stage 0: (2b+K)Psi; 1: 2b*Psi +
 * K*Psi/N; 2: b*Psi + (b+K)*Psi/N; 3: (2b+K)*Psi/N. */
zero_status_t zero_model_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage,
                                     int32_t param_bytes, int32_t optim_K, double out[4]);

/* Communication per step.  *paper_per_rank: the paper's volume, 2*Psi*b for
 * stages 0-2 and 3*Psi*b for stage 3 ("AI论文陪读·ZeRO" section 04; ZeRO
 * visual reading, communication accounting).  *counted_all_ranks: bytes that
 * cross simulated rank boundaries, k*(N-1)*Psi*b with k = 2 (stages 0, 2),
 * 3 (stage 1, counting its end-of-step parameter all-gather; stage 3, two
 * parameter all-gathers and one reduce-scatter). */
zero_status_t zero_comm_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t param_bytes,
                              double* paper_per_rank, int64_t* counted_all_ranks);

/* ---- the step (device) --------------------------------------------------- */

/* One complete optimizer step over all buckets: begin, every bucket, end.
 * zero_step dispatches on cfg->stage; zero_step_stageK requires stage K
 * (ZERO_EINVAL otherwise).  Sources, per stage: stage 0 is plain data
 * parallelism (every rank keeps every state, gradients all-reduced); stage 1
 * partitions the optimizer state (P_os), stage 2 also the gradients
 * (P_os+g), stage 3 also the parameters (P_os+g+p)
 * ("ZeRO：大模型训练的内存优化革命" 3.1.1-3.1.3; ZeRO visual reading, stage
 * list and communication accounting: reduce-scatter, update of the owned
 * shard, all-gather).  The update itself is the mixed-precision one: fp32
 * master weights and optimizer state updated from the 16-bit gradient, then
 * cast back to 16 bits (SC-2020 ZeRO notes, "Where Did All the Memory Go? /
 * Model States"; "AI论文陪读·ZeRO" section 01).  Adam is Kingma & Ba,
 * Algorithm 1 (the pages name Adam but do not print it).  The buffers are the
 * caller's (layout above); the call returns after reading the step's
 * overflow flag (one synchronisation of `stream`).  Errors: ZERO_EINVAL,
 * ZERO_EALIGN, ZERO_ENOMEM (missing buffer), ZERO_ECUDA (a launch or the
 * synchronisation failed; the message has the CUDA error), ZERO_EUNSUPPORTED.
 * On any error before the first launch nothing on the device has changed. */
zero_status_t zero_step(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                        const zero_adam_t* adam, zero_state_t* state, void* stream,
                        zero_step_result_t* out);
zero_status_t zero_step_stage0(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                               const zero_adam_t* adam, zero_state_t* state, void* stream,
                               zero_step_result_t* out);
zero_status_t zero_step_stage1(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                               const zero_adam_t* adam, zero_state_t* state, void* stream,
                               zero_step_result_t* out);
zero_status_t zero_step_stage2(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                               const zero_adam_t* adam, zero_state_t* state, void* stream,
                               zero_step_result_t* out);
zero_status_t zero_step_stage3(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                               const zero_adam_t* adam, zero_state_t* state, void* stream,
                               zero_step_result_t* out);

/* The same step, bucket by bucket, for gradients that arrive one bucket at a
 * time (backward hooks filling a constant-size bucket: the fused buffer of
 * "ZeRO：大模型训练的内存优化革命" 3.2.2 and the SC-2020 ZeRO notes, "Deep
 * Dive into ZeRO-R", C_B).  Call begin, then
 * zero_step_bucket exactly once for every bucket b in any order, then end,
 * all on one stream with unchanged arguments.
 * bucket_grads: NULL to read bufs->grads, or (stages 2 and 3 only) a host
 * array of N device pointers, each to this bucket's gradient window (bucket
 * length, element 0 = the bucket's first flat index); it may be reused for
 * the next bucket once this bucket's kernel has run on the stream. */
zero_status_t zero_step_begin(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                              const zero_adam_t* adam, const zero_state_t* state, void* stream);
zero_status_t zero_step_bucket(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                               const zero_adam_t* adam, const zero_state_t* state, int64_t bucket,
                               void* const* bucket_grads, void* stream);
zero_status_t zero_step_end(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                            const zero_adam_t* adam, zero_state_t* state, void* stream,
                            zero_step_result_t* out);
/* Several buckets of the same step in one call: buckets[0..count), in that
 * order, each exactly once in the step as for zero_step_bucket.
 * bucket_grads: NULL, or (stages 2 and 3) count*N device pointers, bucket k's
 * N windows at bucket_grads[k*N .. k*N+N).  The first kernel follows plain
 * stream order; each later one is a programmatic dependent of the one before
 * (it may start while its predecessor drains, as inside zero_step), so every
 * window must hold its gradients before the call's first kernel runs.  Same
 * errors as zero_step_bucket (ZERO_EINVAL for an index out of range). */
zero_status_t zero_step_buckets(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                const zero_adam_t* adam, const zero_state_t* state, const int64_t* buckets,
                                int32_t count, void* const* bucket_grads, void* stream);

/* Stage 3: copy layer `layer`'s 16-bit parameters from the owners' shards
 * (param_shards[r], P elements each) into each of the n_dst destination
 * buffers dst[d] (capacity max_layer_elems; element j = flat index
 * layer_start + j).  The parameter all-gather that runs before a layer's
 * forward and again before its backward (ZeRO visual reading, communication
 * accounting; "ZeRO：大模型训练的内存优化革命" 3.1.3).  n_dst 1..64.  With the
 * destinations and the layer's shards in device memory the layer is written
 * 2 MB chunk by chunk, destination by destination (the chunk's source stays
 * in L2); otherwise each value is read once and stored to every
 * destination. */
zero_status_t zero_gather_layer(const zero_config_t* cfg, const zero_plan_t* plan, int32_t layer,
                                void* const* param_shards, void* const* dst, int32_t n_dst, void* stream);

/* ---- steps without host synchronisation ------------------------------------
 * The step state (t, the beta powers of the bias correction, the loss scale
 * and its scaler) can live in device memory instead: zero_step_async then
 * enqueues the whole step and returns without waiting, so steps pipeline
 * back to back and a step can be captured in a CUDA graph.  A prepare
 * kernel clears the workspace head and derives the step's scalars from the
 * state block; after the bucket kernels a commit writes the outcome back (t
 * and the beta powers advance on a clean step; the scaler halves on
 * overflow and grows after growth_interval clean steps) together with the
 * last step's flag, norm and clip coefficient, which zero_dev_state_read
 * brings to the host.  Results equal the synchronised step's bit for bit.
 * Fused path: the host does not learn the flag, so bufs->cur flips on every
 * call; after an overflow the restore (which also runs the commit) copies
 * the unchanged state into the copy the next step reads and restores the
 * parameters.  A graph captured from one call therefore serves every other
 * step: capture one call per value of bufs->cur and replay them alternately.
 * The step's kernels are launched as one chain of programmatic dependent
 * launches (each small kernel, and the first bucket kernel, waits for its
 * predecessor before it touches memory).  A two-pass step (clipping, or no
 * shadow state) of a model that is one bucket, in stages 2-3, moving at
 * most 64 MiB (n x (2 N e + 2 e + 24) bytes, e the value size) is two
 * kernels after a memset of the workspace head: pass 1, whose last block
 * derives the scalars and finishes the norm, and pass 2, whose last block
 * commits.
 * The device state block is 64 bytes, 16-byte aligned, caller-owned. */
typedef struct zero_dev_state { int64_t opaque[8]; } zero_dev_state_t;   /* 64 bytes */

/* Initialise the block from a host state (synchronises `stream`); `adam`
 * must carry the betas the steps will use (both in [0, 1)). */
zero_status_t zero_dev_state_init(void* dev_state, const zero_adam_t* adam, const zero_state_t* state, void* stream);
/* Enqueue one step (all buckets); never synchronises.  *kernel_launches
 * (may be NULL) receives the kernels it launched. */
zero_status_t zero_step_async(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                              const zero_adam_t* adam, void* dev_state, void* stream, int32_t* kernel_launches);
/* The same step one bucket at a time (for buckets that become ready during
 * the backward pass), with the step state on the device: begin (the prepare
 * kernel), then zero_step_bucket_async for every bucket in any order --
 * bucket_grads as for zero_step_bucket (stages 2/3 only) -- then end (the
 * two-pass path's finalize and update kernels, and the commit; on the fused
 * path bufs->cur flips).  None of them synchronises; the sequence can be
 * captured in a graph. */
zero_status_t zero_step_begin_async(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                    const zero_adam_t* adam, void* dev_state, void* stream);
zero_status_t zero_step_bucket_async(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                     const zero_adam_t* adam, int64_t bucket, void* const* bucket_grads,
                                     void* stream);
/* zero_step_buckets for the device-state protocol (between begin_async and
 * end_async). */
zero_status_t zero_step_buckets_async(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                      const zero_adam_t* adam, const int64_t* buckets, int32_t count,
                                      void* const* bucket_grads, void* stream);
zero_status_t zero_step_end_async(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                  const zero_adam_t* adam, void* dev_state, void* stream, int32_t* kernel_launches);
/* Copy the block to the host (synchronises `stream`): the current step state
 * and the last step's outcome (t, overflow, skipped, grad_norm, clip_coef,
 * new_loss_scale; path -1).  Returns ZERO_ETIMEOUT (outputs still filled) if
 * a bounded wait inside the last step's kernels ran out; that step was not
 * applied and the loss scaler was left as it was. */
zero_status_t zero_dev_state_read(const void* dev_state, zero_state_t* state, zero_step_result_t* last, void* stream);

/* ---- stage 3: gathers ahead of use under a live-parameter budget ---------
 * A fetcher gathers the layers of one pass (an order of layers: forward
 * 0..L-1, backward L-1..0, any sequence) into a caller-owned pool of
 * `capacity` 16-bit elements per destination, placing them as a ring in
 * fetch order, so the layers resident at once never exceed the capacity
 * (DeepSpeed's stage3_max_live_parameters; ZeRO visual reading, stage-3
 * section: gather the next layers ahead of time, release after use).  Up to
 * `depth` layers ahead are gathered on `side_stream`; a fetch makes the
 * caller's stream wait for that layer only; a release makes the side stream
 * wait before reusing the space.  Protocol, per position pos = 0, 1, ...:
 * zero_fetch_layer(pos) -> use the layer at *offset in every pool buffer on
 * `stream` -> zero_release_layer(pos).  The caller keeps `order`, the pool,
 * the shards and the 2*(depth+1) events (cudaEvent_t, created by the caller)
 * alive while the fetcher is used; zero_fetcher_t is caller memory holding
 * the fetcher's state (no allocation).  Layer sizes are rounded up to 8
 * elements in the pool; capacity must hold the largest layer. */
#define ZERO_FETCH_MAX_DEPTH 32
#define ZERO_FETCH_MAX_RESIDENT 128
typedef struct zero_fetcher { int64_t opaque[1024]; } zero_fetcher_t;   /* 8 KB */

zero_status_t zero_fetcher_init(zero_fetcher_t* f, const zero_config_t* cfg, const zero_plan_t* plan,
                                void* const* param_shards, void* const* pool, int32_t n_dst, int64_t capacity,
                                const int32_t* order, int32_t n_order, int32_t depth, void* side_stream,
                                void* const* events, int32_t n_events);
/* Make layer order[pos] resident and ordered before later work on `stream`;
 * *offset receives its element offset in each pool buffer. */
zero_status_t zero_fetch_layer(zero_fetcher_t* f, int32_t pos, void* stream, int64_t* offset);
/* Done with order[pos] (after the work already enqueued on `stream`). */
zero_status_t zero_release_layer(zero_fetcher_t* f, int32_t pos, void* stream);
/* Largest resident element count reached, gathers issued. */
zero_status_t zero_fetcher_stats(const zero_fetcher_t* f, int64_t* max_live, int32_t* gathers);
/* The fetcher's decisions without a GPU: for each position q, issue_at[q] is
 * the position at whose fetch its gather is issued and offsets[q] its pool
 * offset; *max_live the largest resident element count.  ZERO_ENOMEM if a
 * layer cannot fit; ZERO_EINVAL if capacity is below the largest layer. */
zero_status_t zero_fetch_schedule(const int64_t* layer_sizes, int32_t n_layers, const int32_t* order, int32_t n_order,
                                  int64_t capacity, int32_t depth, int32_t* issue_at, int64_t* offsets,
                                  int64_t* max_live);

/* Stage-2 step that allocates nothing and needs no scratch from the caller.
 * The paper has no counterpart: this exists for callers that cannot obtain
 * device memory for the workspace and the reduced-gradient buffer -- code
 * running inside another runtime that owns the device's memory pool, or code
 * that must not allocate after start-up.  The scratch lives in one static
 * device array inside the library (4 KB + 16 MiB, held by every GPU that
 * loads the library until the process exits), so the plan's padded_elems
 * must be at most 8,388,608 (ZERO_EUNSUPPORTED otherwise, with a message).
 * Same arguments and results as zero_step_stage2, except: bufs->workspace,
 * bufs->reduced and the shadow copies bufs->w/m/v[1-cur] are ignored; the
 * step always takes the two-pass path and updates the [cur] state in place
 * (clipping allowed).  The caller still passes the gradients, parameters and
 * fp32 state.  The array used is the current device's, so `stream` must
 * belong to the current device (ZERO_EINVAL otherwise; NULL is the current
 * device's legacy default stream).  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  Each call clears the array's workspace
 * part before use; the rest keeps the last call's contents.  All calls share
 * the array: calls whose kernels overlap on the GPU (other streams or host
 * threads) race on it. */
zero_status_t zero_step_stage2_noalloc(const zero_config_t* cfg, const zero_plan_t* plan, zero_buffers_t* bufs,
                                       const zero_adam_t* adam, zero_state_t* state, void* stream,
                                       zero_step_result_t* out);

/* ---- P_a: partitioned activation checkpoints (ZeRO-R) --------------------
 * Under model parallelism the input of a layer -- the activation checkpoint
 * that backward recomputes the layer from -- is replicated on all N_m
 * model-parallel ranks.  P_a keeps a 1/N_m slice per rank after the forward
 * pass and rebuilds the checkpoint with an all-gather when backward needs
 * it; P_a+cpu keeps the slices in host memory ("ZeRO：大模型训练的内存优化
 * 革命" 3.2.1; SC-2020 ZeRO notes, "P_a: Partitioned Activation
 * Checkpointing").  The N_m ranks are simulated as buffers, like the
 * data-parallel ranks.  Slice of rank r: values [r*P, min((r+1)*P, act_elems)),
 * P = ceil(act_elems / N_m) rounded up to align_elems.  72 bytes. */
typedef struct zero_pa_plan {
    int64_t act_elems;              /* values in one checkpoint, >= 0 */
    int64_t shard_elems;            /* P */
    int64_t align_elems;            /* 0 -> 2048; a multiple of 8 */
    int32_t n_mp;                   /* N_m, 1..64 */
    int32_t dtype;                  /* zero_dtype_t of the activations (2 or 4 bytes) */
    int64_t mem_per_rank_bytes;     /* without P_a: the whole checkpoint on every rank */
    int64_t mem_per_rank_pa_bytes;  /* with P_a: one slice (P_a+cpu: none on the GPU) */
    int64_t gather_bytes;           /* bytes crossing simulated rank boundaries in one all-gather, all ranks */
    int64_t reserved[2];
} zero_pa_plan_t;

zero_status_t zero_pa_plan(int64_t act_elems, int32_t n_mp, int32_t dtype, int64_t align_elems,
                           zero_pa_plan_t* out);
/* After the forward pass: rank r copies its slice of replicas[r] (the
 * checkpoint as rank r holds it: act_elems values) to shards[r] (room for
 * shard_elems values; device or pinned host memory -- P_a+cpu).  Arrays of
 * n_mp pointers, 16-byte aligned.  One kernel launch, asynchronous. */
zero_status_t zero_pa_partition(const zero_pa_plan_t* plan, const void* const* replicas, void* const* shards,
                                void* stream);
/* Before the layer's recomputation: the all-gather -- the checkpoint rebuilt
 * from the n_mp slices into each of dst[0..n_dst) (act_elems values each;
 * n_dst 1..64).  One kernel launch, asynchronous. */
zero_status_t zero_pa_gather(const zero_pa_plan_t* plan, const void* const* shards, void* const* dst, int32_t n_dst,
                             void* stream);

/* Profiling: for the step calls made afterwards on this thread, record
 * start_event (a cudaEvent_t) on the step's stream right after the workspace
 * clear, before the first kernel, and end_event after the step's last kernel,
 * before the overflow flag is read (zero_step_async: after its prepare
 * kernel, and after the last bucket or update kernel, before the restore and
 * commit; those two kernel edges then do not overlap).  The caller creates
 * the events and keeps
 * them valid; (NULL, NULL) turns recording off.  Bucket kernels launched
 * back to back inside one call overlap their edges, so the events give the
 * step's kernel span, not per-kernel durations. */
zero_status_t zero_set_profile_events(void* start_event, void* end_event);

/* Thread-local message of the last failed call ("" if none).  No
 * counterpart on the pages: error reporting of this C ABI.  The string is
 * owned by the library and stays valid until the thread's next failing
 * call. */
const char* zero_last_error(void);
/* ZERO_GB300_VERSION of the loaded library (no counterpart on the pages). */
int32_t zero_version(void);

#ifdef __cplusplus
}
#endif
#endif

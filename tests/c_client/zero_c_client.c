/* A plain C client of libzero_gb300: no Python, no PyTorch.
 *
 * usage: zero_c_client <dir> [graph]
 *   reads  <dir>/in.bin:  int64 n, int32 N, int32 steps, float lr, float S,
 *                         then float w0[n], then for each step N x uint16 g[n]
 *   writes <dir>/out.bin: float w[n], float m[n], float v[n], uint16 p16[N][n],
 *                         int64 t, uint32 overflow of the last step
 * Stage 2, fp16, Adam (beta 0.9/0.999, eps 1e-8), bucket 4096, shadow state.
 * Default: zero_step_stage2 per step.  "graph": the step state in device
 * memory, two CUDA graphs captured from zero_step_async and replayed.
 * Exit status 0 on success; a message on stderr otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "zero_gb300.h"

#define CK(x)                                                                            \
    do {                                                                                 \
        cudaError_t e_ = (x);                                                            \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "CUDA %s at line %d\n", cudaGetErrorString(e_), __LINE__);   \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

#define ZK(x)                                                                            \
    do {                                                                                 \
        zero_status_t s_ = (x);                                                          \
        if (s_ != ZERO_OK) {                                                             \
            fprintf(stderr, "zero status %d: %s\n", (int)s_, zero_last_error());         \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

int main(int argc, char** argv)
{
    if (argc != 2 && argc != 3) return 2;
    char path[4096];
    const int graph_mode = argc > 2 && strcmp(argv[2], "graph") == 0;
    snprintf(path, sizeof path, "%s/in.bin", argv[1]);
    FILE* f = fopen(path, "rb");
    if (!f) return 2;
    int64_t n;
    int32_t N, steps;
    float lr, S;
    if (fread(&n, 8, 1, f) != 1 || fread(&N, 4, 1, f) != 1 || fread(&steps, 4, 1, f) != 1 ||
        fread(&lr, 4, 1, f) != 1 || fread(&S, 4, 1, f) != 1)
        return 2;
    float* w0 = malloc(n * sizeof(float));
    uint16_t* g = malloc((size_t)steps * N * n * sizeof(uint16_t));
    if (fread(w0, 4, n, f) != (size_t)n || fread(g, 2, (size_t)steps * N * n, f) != (size_t)steps * N * n) return 2;
    fclose(f);

    zero_config_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n_params = n;
    cfg.bucket_elems = 4096;
    cfg.stage = 2;
    cfg.n_ranks = N;
    cfg.dtype = ZERO_FP16;
    cfg.optimizer = ZERO_ADAM;
    zero_plan_t plan;
    ZK(zero_plan(&cfg, &plan));

    void* grads[ZERO_MAX_RANKS];
    void* params[ZERO_MAX_RANKS];
    for (int r = 0; r < N; r++) {
        CK(cudaMalloc(&grads[r], plan.grad16_elems * 2));
        CK(cudaMalloc(&params[r], plan.param16_elems * 2));
        CK(cudaMemset(params[r], 0, plan.param16_elems * 2));
    }
    zero_buffers_t b;
    memset(&b, 0, sizeof b);
    b.grads = grads;
    b.params16 = params;
    for (int k = 0; k < 2; k++) {
        CK(cudaMalloc((void**)&b.w[k], plan.state_elems * 4));
        CK(cudaMalloc((void**)&b.m[k], plan.state_elems * 4));
        CK(cudaMalloc((void**)&b.v[k], plan.state_elems * 4));
        CK(cudaMemset(b.w[k], 0, plan.state_elems * 4));
        CK(cudaMemset(b.m[k], 0, plan.state_elems * 4));
        CK(cudaMemset(b.v[k], 0, plan.state_elems * 4));
    }
    CK(cudaMalloc(&b.workspace, plan.workspace_bytes));
    CK(cudaMemcpy(b.w[0], w0, n * 4, cudaMemcpyHostToDevice));

    zero_adam_t adam = {lr, 0.9f, 0.999f, 1e-8f, 0.0f, 0.0f};
    zero_state_t st;
    memset(&st, 0, sizeof st);
    st.loss_scale = S;
    st.min_loss_scale = 1.0f;
    st.dynamic = 1;
    zero_step_result_t res;
    memset(&res, 0, sizeof res);
    cudaStream_t stream;
    CK(cudaStreamCreate(&stream));
    if (!graph_mode) {
        for (int k = 0; k < steps; k++) {
            for (int r = 0; r < N; r++)
                CK(cudaMemcpyAsync(grads[r], g + ((size_t)k * N + r) * n, n * 2, cudaMemcpyHostToDevice, stream));
            ZK(zero_step_stage2(&cfg, &plan, &b, &adam, &st, (void*)stream, &res));
        }
        CK(cudaStreamSynchronize(stream));
    } else {
        /* step state in device memory; one CUDA graph per value of b.cur
         * (the fused path alternates the state copies on every call),
         * replayed alternately with each step's gradients copied in first */
        void* dev_state;
        CK(cudaMalloc(&dev_state, sizeof(zero_dev_state_t)));
        ZK(zero_dev_state_init(dev_state, &adam, &st, (void*)stream));
        cudaGraphExec_t exec[2];
        for (int k = 0; k < 2; k++) {
            cudaGraph_t graph;
            int32_t launches = 0;
            CK(cudaStreamBeginCapture(stream, cudaStreamCaptureModeGlobal));
            ZK(zero_step_async(&cfg, &plan, &b, &adam, dev_state, (void*)stream, &launches));
            CK(cudaStreamEndCapture(stream, &graph));
            CK(cudaGraphInstantiate(&exec[k], graph, 0));
            CK(cudaGraphDestroy(graph));
        }
        for (int k = 0; k < steps; k++) {
            for (int r = 0; r < N; r++)
                CK(cudaMemcpyAsync(grads[r], g + ((size_t)k * N + r) * n, n * 2, cudaMemcpyHostToDevice, stream));
            CK(cudaGraphLaunch(exec[k % 2], stream));
        }
        ZK(zero_dev_state_read(dev_state, &st, &res, (void*)stream));
        b.cur = steps % 2;   /* the copy the last replay wrote */
        for (int k = 0; k < 2; k++) CK(cudaGraphExecDestroy(exec[k]));
        CK(cudaFree(dev_state));
    }

    float* out = malloc(n * 4);
    uint16_t* p = malloc(n * 2);
    snprintf(path, sizeof path, "%s/out.bin", argv[1]);
    FILE* o = fopen(path, "wb");
    if (!o) return 2;
    float* arr[3] = {b.w[b.cur], b.m[b.cur], b.v[b.cur]};
    for (int k = 0; k < 3; k++) {
        CK(cudaMemcpy(out, arr[k], n * 4, cudaMemcpyDeviceToHost));
        fwrite(out, 4, n, o);
    }
    for (int r = 0; r < N; r++) {
        CK(cudaMemcpy(p, params[r], n * 2, cudaMemcpyDeviceToHost));
        fwrite(p, 2, n, o);
    }
    int64_t t = st.t;
    fwrite(&t, 8, 1, o);
    fwrite(&res.overflow, 4, 1, o);
    fclose(o);
    return 0;
}

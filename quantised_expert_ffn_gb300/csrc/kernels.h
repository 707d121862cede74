// kernels.h -- argument blocks and launchers of the kernels (internal to libsmoe.so).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace smoe {

// Launch `kern` on `s`; with `pdl` the launch may begin while the previous
// kernel in the stream is still running (programmatic dependent launch); the
// kernels call griddepcontrol.wait before touching that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct RouteArgs {
    const uint16_t *x;          // [T][D] bf16 residual
    const uint16_t *gain;       // [D] or NULL
    float eps;
    const uint16_t *router_w;   // [E][D]
    int D, E, K, norm_topk_prob;
    float *logits;              // [T][E]
    int32_t *idx;               // [T][K]
    float *w;                   // [T][K]
    uint16_t *xn_out;           // [T][D] bf16 or NULL
    __half *xn16_out;           // [T][D] fp16 or NULL
    int32_t *counters;          // [T], zero on entry and on exit
    int32_t *status;            // device status word
};
cudaError_t launch_route_topk(const RouteArgs &a, int T, cudaStream_t s, bool pdl);

struct UnionArgs {
    const int32_t *idx;         // [T][K]
    const float *w;             // [T][K]
    int T, K, E;
    int32_t *union_ids;         // [E]
    int32_t *n_union;           // [1]
    int32_t *offsets;           // [E+1]
    int32_t *bucket_tok;        // [T*K]
    int32_t *bucket_rank;       // [T*K]
    float *bucket_w;            // [T*K]
    int32_t *status;            // device status word or NULL
    // prefill extras (NULL in the public union call)
    int32_t *slot_of;           // [T*K]: bucket position of entry (t, rank), -1 if skipped
};
cudaError_t launch_expert_union(const UnionArgs &a, cudaStream_t s, bool pdl);

struct DecodeArgs {
    const uint16_t *x;          // [D] residual (bf16)
    const uint16_t *gain;       // RMSNorm gain or NULL
    float eps;
    int D, F, K, E;
    const int32_t *idx;         // [K]
    const float *w;             // [K]
    const uint8_t *gq, *uq, *dq;
    const uint16_t *gs, *gb, *us, *ub, *ds, *db;
    float *h;                   // [K][F] fp32 scratch
    uint16_t *y;                // [D] bf16 out (may alias x)
    float *expert_out;          // [K][D] or NULL
    const smoe_layer *layers;   // stack variant: device table of n_layers layers (NULL: the pointers above)
    int n_layers;               // layers run by one launch (1 unless `layers` is set)
    uint16_t *act0, *act1;      // stack variant: [D] bf16 activations between layers (ping-pong)
    int32_t *status;
};
cudaError_t launch_decode_gateup(const DecodeArgs &a, cudaStream_t s, bool pdl);
cudaError_t launch_decode_down(const DecodeArgs &a, cudaStream_t s, bool pdl);

// One decode layer as one persistent kernel (decode_fused.cu).
struct FusedArgs {
    const uint16_t *x;          // [D] residual in
    uint16_t *y;                // [D] out (may alias x)
    const uint16_t *gain;       // RMSNorm gain or NULL
    float eps;
    int D, F, K, E, norm_topk_prob;
    const uint16_t *router_w;
    const uint8_t *gq, *uq, *dq;
    const uint16_t *gs, *gb, *us, *ub, *ds, *db;
    float *logits;              // [E] scratch
    float *h;                   // [K][F] scratch
    unsigned long long *gctr;   // grid barrier arrival counter (only grows)
    int32_t *status;
    int32_t *idx_out;           // [K] (route variant)
    float *w_out;               // [K]
    const int32_t *idx_in;      // [K] (FFN-only variant)
    const float *w_in;          // [K]
    float *expert_out;          // [K][D] or NULL
    const smoe_layer *layers;   // stack variant: device table of n_layers layers (NULL: the pointers above)
    int n_layers;               // layers run by one launch (1 unless `layers` is set)
    uint16_t *act0, *act1;      // stack variant: [D] bf16 activations between layers (ping-pong)
    int q2;                     // 1: SMOE-Q2 codes (2 bits, 8 bytes per 32 codes), 0: SMOE-Q4
    unsigned long long grid_wait_ns;   // limit of each grid-barrier spin (smoe_set_grid_wait_limit)
    // plan (fused_plan)
    int grid, r_gu, dn_nr, dn_gran, dn_rs, rows_max, slot_bytes, ring_bytes, union_bytes, smem_bytes;
};
bool fused_plan(FusedArgs &a, int num_sms);
size_t fused_h_floats(int F, int K);
// Cooperative launch (every CTA resident before any runs); returns
// cudaErrorCooperativeLaunchTooLarge when the device cannot hold the grid
// (then nothing is enqueued and the caller takes the three-kernel engine).
cudaError_t launch_decode_layer(const FusedArgs &a, cudaStream_t s, bool route);

// Limit of each grid-barrier spin of the persistent decode kernel, ns
// (process-wide; read when a call is enqueued).
unsigned long long grid_wait_limit_ns();

struct PrefillArgs {
    const uint16_t *x;          // [T][D] residual
    int T, D, F, K, E;
    const __half *xn16;         // [T][D] normed input, fp16
    const int32_t *n_union;
    const int32_t *union_ids;   // [E]
    const int32_t *offsets;     // [E+1]
    const int32_t *bucket_tok;  // [T*K]
    const int32_t *bucket_rank; // [T*K]
    const int32_t *slot_of;     // [T*K]
    const float *w;             // [T][K]
    const uint8_t *gq, *uq, *dq;
    const uint16_t *gs, *gb, *us, *ub, *ds, *db;
    __half *xperm;              // [T*K][D] fp16 bucket-ordered inputs
    __half *hbuf;               // [T*K][F] fp16
    float *obuf;                // [T*K][D] fp32 per-(bucket slot) expert outputs
    uint16_t *y;                // [T][D]
    float *expert_out;          // [T][K][D] unweighted o of each (token, rank), or NULL
    int32_t *status;
    int32_t *ready;             // [E] gate/up -> down counters (tensor-core path), or NULL
    int32_t *unit_ctr;          // [2] gate/up and down unit counters (tensor-core path), or NULL
    int num_sms;
    int q2;                     // 1: SMOE-Q2 codes (tensor-core path only)
};
// CUDA-core path: gate/up, down and combine (fp32 h)
cudaError_t launch_prefill_simt(const PrefillArgs &a, const uint16_t *xn, float *h32, cudaStream_t s,
                                bool pdl);
// tensor-core path: bucket gather, gate/up and down grouped GEMMs (fp16 h); combine separately
bool prefill_tc_supported(int D, int F);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_combine(const PrefillArgs &a, cudaStream_t s, bool pdl);

int device_sm_count();

// Bytes at the head of a workspace that must be zero before a call (status
// word, route tickets, grid-barrier counter); the same for every layer shape.
size_t ws_head_bytes();

}  // namespace smoe

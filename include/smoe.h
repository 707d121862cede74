/*
 * smoe.h -- C ABI of libsmoe.so: the routed Mixture-of-Experts layer of the
 * S-MoE engine (exact router gate -> top-k with norm_topk_prob weights ->
 * per-chunk expert union and buckets -> SMOE-Q4 fused dequant expert FFN ->
 * weighted sum into the residual), as CUDA kernels for sm_103a (GB300).
 *
 * Sources of the operations (the S-MoE documentation pages "Optimizations"
 * and "System Overview"):
 *   - exact routing on the true hidden state, top-8, norm_topk_prob mixing
 *     weights: "Optimizations", section "Routing Is Exact -- Prompt and
 *     Generation Alike"; "System Overview", table "What Happens at Each
 *     Generated Token Step" (Heavy pass row);
 *   - per-chunk expert union, chunks of up to 64 tokens: "Optimizations",
 *     section "Prefill Reads Each Expert Once, Not Once Per Token";
 *   - SMOE-Q4 fused dequant FFN, gate+up in one pass, weighted sum into the
 *     residual: "Optimizations", section "Coalesced GPU Kernels -- Expert FFN
 *     and Dense Matvec"; "System Overview", same table, Metal Kernel row;
 *   - RMSNorm before the router (between layers): "Optimizations", section
 *     "The Dense Ceiling -- GPU-Resident Epilogue";
 *   - no allocation in the token loop: "Optimizations", section "Zero
 *     Allocations, Zero Locks in the Token Loop".
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every entry point
 *
 * Memory.  Every pointer is caller-owned DEVICE memory unless a parameter
 * says otherwise.  The library never allocates and never frees; apart from
 * smoe_read_device_status, which synchronises `stream`, all work is enqueued
 * on `stream` (the CUDA stream of the caller, cudaStream_t; NULL = legacy
 * default stream).  The first call of an entry point on a device also sets
 * its kernels' attributes there (a host-side step), so make it outside any
 * stream capture.  This library's benchmark replays smoe_moe_decode_layers,
 * smoe_moe_prefill_chunk and smoe_dense_matvec (and, with its per-layer
 * option, smoe_moe_decode) from CUDA graphs captured after such a first call.
 *
 * Devices.  Every call runs on the caller's current CUDA device, and `stream`
 * must belong to it.  One process may use the library on several devices:
 * its host-side caches (SM count, kernel attributes, the no-workspace decode
 * scratch) are kept per device.
 *
 * Types.  bf16 tensors are passed as smoe_bf16 (the raw 16-bit pattern of a
 * bfloat16).  Shapes are row-major, outermost first.
 *
 * SMOE-Q4 weights (this layout is fixed here; the pages leave it open).  A
 * matrix of `rows` outputs and `cols` inputs stores
 *   codes  uint8 [rows][cols/2]: element 2j is the low nibble of byte j,
 *          element 2j+1 the high nibble; code q in 0..15;
 *   scale  bf16  [rows][cols/64]  and  bias bf16 [rows][cols/64];
 *   weight w[r][c] = scale[r][c/64] * q[r][c] + bias[r][c/64].
 * Within a layer the experts are contiguous: gate and up are [E][F][D]
 * (codes [E][F][D/2], scale/bias [E][F][D/64]); down is [E][D][F]
 * (codes [E][D][F/2], scale/bias [E][D][F/64]); the router is bf16 [E][D].
 *
 * SMOE-Q2 weights ("Optimizations", "Q2 Vaults -- the Next 2x, Twice Over":
 * the 2-bit vault that halves every blob; "System Overview", the "SMOE-Q2/Q4
 * fused dequant + FFN" kernel).  A layer with code_bits = 2 keeps the groups,
 * scales and biases above with 2-bit codes q in 0..3: codes uint8
 * [rows][cols/4], element 4j+k in bits 2k..2k+1 of byte j.  Decode
 * (smoe_moe_decode, smoe_moe_ffn_decode, smoe_moe_decode_layers,
 * smoe_moe_decode_noalloc) takes Q2 layers whose shape fits the one-kernel
 * decode plan (d_model a multiple of 512 up to 4096, ffn_dim a multiple of
 * 128); prefill (smoe_moe_prefill_chunk) takes Q2 layers on its tensor-core
 * path (d_model and ffn_dim multiples of 128).  Other Q2 shapes return
 * SMOE_ERR_UNSUPPORTED before anything is enqueued.
 *
 * Workspace.  Calls that need scratch take `ws`/`ws_bytes`: device memory of
 * at least smoe_workspace_bytes() bytes, 256-byte aligned, that the caller
 * zero-fills once before its first use (smoe_workspace_init() does it on the
 * stream).  Each call leaves its counters zero again.  The first 4 bytes are
 * the int32 DEVICE STATUS WORD: 0, or a negative smoe_status that a kernel
 * found (an expert id out of range, a bounded wait that gave up).  Kernels
 * only ever write a non-zero value there; the caller reads it after a
 * synchronisation (smoe_read_device_status) and clears it with
 * smoe_workspace_init().  Calls that share one workspace must not overlap on
 * the GPU (the same stream, or ordered by events).
 *
 * Errors.  Problems the host can see (NULL pointers, unsupported shapes,
 * misaligned pointers, a workspace that is too small) return a negative
 * smoe_status at once and enqueue nothing.  A failed launch returns
 * SMOE_ERR_CUDA.  Nothing throws across this ABI and no kernel traps.
 *
 * Supported shapes: d_model and ffn_dim multiples of 64 (group_size must be
 * 64), d_model <= 8192, ffn_dim <= 4096, 1 <= top_k <= 16, top_k <= n_experts
 * <= 256, top_k * ffn_dim <= 16384.  Code pointers and the hidden-state
 * pointers must be 16-byte aligned.  Tuned for d_model 2048/4096, 128
 * experts, top-8, ffn_dim 768/1536.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t smoe_bf16;                /* raw bfloat16 bits */
typedef struct CUstream_st *smoe_stream;   /* identical to cudaStream_t */

typedef enum smoe_status {
    SMOE_OK = 0,
    SMOE_ERR_INVALID_ARG = -1,   /* NULL pointer, bad size or alignment */
    SMOE_ERR_UNSUPPORTED = -2,   /* shape outside the supported set */
    SMOE_ERR_WORKSPACE = -3,     /* workspace missing, misaligned or too small */
    SMOE_ERR_CUDA = -4,          /* a CUDA launch or runtime call failed */
    SMOE_ERR_TIMEOUT = -5,       /* device: a bounded wait gave up */
    SMOE_ERR_DEVICE = -6,        /* device: bad data (e.g. expert id out of range) */
    SMOE_ERR_RANGE = -7          /* device: a value beyond fp16's range on the tensor-core prefill */
} smoe_status;

/* One MoE layer: its shape and its device-resident parameters. */
typedef struct smoe_layer {
    int d_model;                 /* D: hidden size */
    int n_experts;               /* E: routed experts */
    int top_k;                   /* k: experts per token */
    int ffn_dim;                 /* F: expert intermediate size */
    int group_size;              /* Q4 group along the input dim; must be 64 */
    int norm_topk_prob;          /* 1: renormalise the top-k probabilities to sum 1 */
    float rms_eps;               /* RMSNorm epsilon (used when rms_gain != NULL) */
    const smoe_bf16 *rms_gain;   /* [D] RMSNorm gain before the router and the FFN; NULL = none */
    const smoe_bf16 *router_w;   /* [E][D] router gate */
    const uint8_t *gate_q;       /* [E][F][D/2] */
    const smoe_bf16 *gate_s;     /* [E][F][D/64] */
    const smoe_bf16 *gate_b;     /* [E][F][D/64] */
    const uint8_t *up_q;         /* [E][F][D/2] */
    const smoe_bf16 *up_s;       /* [E][F][D/64] */
    const smoe_bf16 *up_b;       /* [E][F][D/64] */
    const uint8_t *down_q;       /* [E][D][F/2] */
    const smoe_bf16 *down_s;     /* [E][D][F/64] */
    const smoe_bf16 *down_b;     /* [E][D][F/64] */
    int code_bits;               /* 4 (SMOE-Q4; 0 reads as 4) or 2 (SMOE-Q2, see below) */
} smoe_layer;

/* Bytes of workspace that the calls below need for this layer shape and up
 * to `max_tokens` tokens per call (1 for decode, up to 64 for a prefill
 * chunk).  Host only; returns 0 when the shape is unsupported. */
size_t smoe_workspace_bytes(const smoe_layer *layer, int max_tokens);

/* Zero `ws_bytes` bytes of workspace on `stream` (cudaMemsetAsync). */
int smoe_workspace_init(void *ws, size_t ws_bytes, smoe_stream stream);

/* Copy the device status word of `ws` to *status_host.  This one call
 * synchronises `stream`.  Returns SMOE_OK or SMOE_ERR_CUDA. */
int smoe_read_device_status(const void *ws, int32_t *status_host, smoe_stream stream);

/* Router gate and top-k ("Routing Is Exact"; per-token table, Heavy pass).
 * For each of T tokens x[t] (bf16 [T][D]):
 *   xn = rms_gain ? bf16(x / sqrt(mean(x^2) + eps) * rms_gain) : x
 *   logits[e] = sum_d router_w[e][d] * xn[d]           (fp32 accumulation)
 *   idx[t][0..k)  = the k largest logits, descending; equal logits keep the
 *                   lower expert id
 *   w[t][i] = softmax(logits)[idx_i], renormalised over the k selected when
 *             norm_topk_prob (then equal to a softmax over the k logits)
 * Outputs: idx int32 [T][k], w fp32 [T][k]; logits_opt fp32 [T][E] and
 * xn_opt bf16 [T][D] when non-NULL.  1 <= T <= 64. */
int smoe_route_topk(const smoe_layer *layer, const smoe_bf16 *x, int T, int32_t *idx,
                    float *w, float *logits_opt, smoe_bf16 *xn_opt, void *ws,
                    size_t ws_bytes, smoe_stream stream);

/* Per-chunk expert union and per-expert token buckets ("Prefill Reads Each
 * Expert Once, Not Once Per Token").  idx int32 [T][k], w fp32 [T][k],
 * 1 <= T <= 64, k <= 16, E <= 256.  Outputs (device):
 *   union_ids  int32 [E]: the distinct ids of idx in ascending order, then -1;
 *   n_union    int32 [1]: how many;
 *   offsets    int32 [E+1]: bucket u is [offsets[u], offsets[u+1]); entries
 *              past n_union hold the number of bucketed entries;
 *   bucket_tok, bucket_rank int32 [T*k], bucket_w fp32 [T*k]: for each union
 *              expert in order, its tokens ascending (a token that lists the
 *              expert twice appears once per listing, in rank order), with the
 *              rank i at which the token chose it and w[t][i]; unused tail
 *              entries are -1 / -1 / 0.
 * Ids outside [0, E) are skipped and set *status_dev (device int32, may be
 * NULL) to SMOE_ERR_DEVICE. */
int smoe_expert_union(const int32_t *idx, const float *w, int T, int k, int E,
                      int32_t *union_ids, int32_t *n_union, int32_t *offsets,
                      int32_t *bucket_tok, int32_t *bucket_rank, float *bucket_w,
                      int32_t *status_dev, smoe_stream stream);

/* One decode token through the layer (batch 1):
 *   route x as smoe_route_topk; for each selected expert i (rank order)
 *   h = SiLU(Wgate_e xn) * (Wup_e xn)  [F],   o_i = Wdown_e h  [D]
 *   y = x + sum_i w_i o_i   (fp32, one rounding to bf16)
 * x, y bf16 [D] (y may alias x).  Optional outputs: idx_out int32 [k],
 * w_out fp32 [k], expert_out fp32 [k][D] (the unweighted o_i). */
int smoe_moe_decode(const smoe_layer *layer, const smoe_bf16 *x, smoe_bf16 *y,
                    int32_t *idx_out_opt, float *w_out_opt, float *expert_out_opt, void *ws,
                    size_t ws_bytes, smoe_stream stream);

/* The expert FFN of one decode token for a routing already made (the Metal
 * Kernel row of the per-token table: the SMOE-Q4 fused FFN of each claimed
 * expert, weighted-summed into the residual):
 *   xn = RMSNorm(x) as in smoe_route_topk;  for i in 0..k-1, e = idx[i]:
 *   o_i = Wdown_e (SiLU(Wgate_e xn) * (Wup_e xn));  y = x + sum_i w[i] o_i.
 * idx int32 [k] and w fp32 [k] are device arrays (e.g. smoe_route_topk's
 * outputs); an id outside [0, E) contributes nothing and sets the device
 * status word.  x, y bf16 [D] (y may alias x); expert_out fp32 [k][D] or NULL.
 * smoe_moe_decode is smoe_route_topk followed by this call. */
int smoe_moe_ffn_decode(const smoe_layer *layer, const smoe_bf16 *x, const int32_t *idx,
                        const float *w, smoe_bf16 *y, float *expert_out_opt, void *ws,
                        size_t ws_bytes, smoe_stream stream);

/* One prefill chunk of T tokens (1 <= T <= 64) through the layer: route all
 * tokens, build the expert union and buckets on the device, read each union
 * expert's weights once and apply them to every token of its bucket (grouped
 * GEMM on the tensor cores), then y[t] = x[t] + sum_i w[t][i] o[t][i] in rank
 * order.  x, y bf16 [T][D] (y must not alias x).  Optional outputs:
 * idx_out int32 [T][k], w_out fp32 [T][k].
 * Precision: the tensor cores take fp16 operands -- the normed inputs (bf16,
 * converted exactly when |x| >= 2^-24 or 0), each weight s*q + b (one fp16
 * rounding, exact when b = -8 s), and h = SiLU(g)*u (one fp16 rounding) --
 * with fp32 accumulation.  A value beyond fp16's range (an input above 65504
 * in magnitude, a group whose levels b .. b + 15 s reach past 65504, or an h
 * that rounds to infinity) sets SMOE_ERR_RANGE in the device status word and
 * the outputs of that call are not valid; shapes the tensor-core kernels do
 * not take (d_model or ffn_dim not a multiple of 128) run on CUDA cores in
 * fp32, which have no such bound. */
int smoe_moe_prefill_chunk(const smoe_layer *layer, const smoe_bf16 *x, int T, smoe_bf16 *y,
                           int32_t *idx_out_opt, float *w_out_opt, void *ws, size_t ws_bytes,
                           smoe_stream stream);

/* smoe_moe_prefill_chunk that also returns each token's expert outputs:
 * expert_out fp32 [T][k][D] (16-byte aligned, caller-owned device memory)
 * receives o[t][i] = Wdown_e (SiLU(Wgate_e xn_t) * (Wup_e xn_t)) for the
 * expert e = idx[t][i], unweighted, in rank order -- the values the chunk's
 * grouped GEMMs computed once per union expert and that the residual sum
 * y[t] = x[t] + sum_i w[t][i] o[t][i] consumed.  ("Prefill Reads Each Expert
 * Once, Not Once Per Token": the per-(token, expert) outputs of the union's
 * single read.)  Everything else, including y, is exactly what
 * smoe_moe_prefill_chunk computes.  expert_out must not be NULL. */
int smoe_moe_prefill_chunk_experts(const smoe_layer *layer, const smoe_bf16 *x, int T, smoe_bf16 *y,
                                   int32_t *idx_out_opt, float *w_out_opt, float *expert_out,
                                   void *ws, size_t ws_bytes, smoe_stream stream);

/* One decode token through n_layers routed-MoE layers, each as
 * smoe_moe_decode computes it, in ONE kernel launch ("Optimizations" page,
 * "The Dense Ceiling -- GPU-Resident Epilogue": the per-token work stays on
 * the GPU; here the layers of the token do too, with grid-wide barriers
 * between them instead of kernel boundaries).
 *   layers      HOST array of n_layers layers: checked on the host (shapes,
 *               pointers, alignment); all layers must share d_model,
 *               n_experts, top_k, ffn_dim, norm_topk_prob, rms_eps and the
 *               presence of rms_gain.
 *   layers_dev  DEVICE copy of the same array (caller-owned, same contents,
 *               8-byte aligned); the kernel reads the weight pointers there.
 *   x, y        bf16 [D]; y may alias x.  The activations between layers live
 *               in the workspace (smoe_workspace_bytes(&layers[0], 1)).
 *   idx_out_opt int32 [n_layers][k] and w_out_opt fp32 [n_layers][k]: both or
 *               neither.
 * Results equal n_layers chained smoe_moe_decode calls bit for bit.  Layers
 * whose weights are not 16-byte aligned, or a shape the one-kernel plan does
 * not take, run as one launch sequence per layer with the same results. */
int smoe_moe_decode_layers(const smoe_layer *layers, const smoe_layer *layers_dev, int n_layers,
                           const smoe_bf16 *x, smoe_bf16 *y, int32_t *idx_out_opt,
                           float *w_out_opt, void *ws, size_t ws_bytes, smoe_stream stream);

/* Decode without a workspace.  The pages have no counterpart of this call:
 * it exists for callers that cannot allocate device memory when they run a
 * layer -- real-time loops whose latency budget rules out the device-wide
 * synchronisation an allocation may cause, services that reserve all their
 * device memory at start-up and must not grow afterwards, and plug-ins whose
 * host program owns all device memory through its own pool.
 * Computes exactly what smoe_moe_decode computes (same kernels); the scratch
 * lives in a fixed device array of the library, SMOE_DECODE_NOALLOC_MAX_BYTES
 * bytes, that every GPU which loads the library holds until the process
 * exits.  A layer whose smoe_workspace_bytes(layer, 1) exceeds that size is
 * rejected with SMOE_ERR_WORKSPACE and nothing is enqueued.  The first call on
 * a device looks up the array's device address (once, with that device
 * current); make that first call before any stream capture.  Arguments are
 * checked first (as smoe_moe_decode checks them); then every call zeroes the
 * head of the array -- its status word, route tickets and grid-barrier
 * counter -- with a cudaMemsetAsync on `stream`, and allocates nothing.  All
 * calls share the one array: calls that overlap on the GPU (different
 * streams, no ordering) race and give undefined results.  x, y bf16 [D]
 * (y may alias x); idx_out int32 [k] and w_out fp32 [k] optional.
 * A device-side error of the call (a bounded wait that gave up, an expert
 * id out of range) is left in the array's status word, which
 * smoe_moe_decode_noalloc_status reads; the next call clears it. */
#define SMOE_DECODE_NOALLOC_MAX_BYTES (512u * 1024u)
int smoe_moe_decode_noalloc(const smoe_layer *layer, const smoe_bf16 *x, smoe_bf16 *y,
                            int32_t *idx_out_opt, float *w_out_opt, smoe_stream stream);

/* The status word that the last smoe_moe_decode_noalloc call on the current
 * device left in the fixed scratch (0, or a negative smoe_status found on the
 * device), copied to *status_host.  Synchronises `stream`; call it after the
 * decode call it concerns and before the next one, which clears the word.
 * The pages have no counterpart (see smoe_moe_decode_noalloc).  Returns
 * SMOE_OK, SMOE_ERR_INVALID_ARG or SMOE_ERR_CUDA. */
int smoe_moe_decode_noalloc_status(int32_t *status_host, smoe_stream stream);

/* Dense bf16 matrix-vector product, y[r] = sum_c w[r][c] * x[c], fp32 sums.
 * "Optimizations" page, "Coalesced GPU Kernels -- Expert FFN and Dense
 * Matvec": the bf16 dense matvec twin of the expert kernels, which carries
 * decode's QKV/O projections and the LM head (shapes such as 512 x 4096 and
 * 151,936 x 4096).  w bf16 [rows][cols] row-major and x bf16 [cols], both
 * 16-byte aligned; y fp32 [rows], 4-byte aligned; all caller-owned device
 * memory, read (w, x) or written (y) once.  rows >= 1; cols a multiple of 8
 * and at most 8192 (else SMOE_ERR_UNSUPPORTED).  No workspace; nothing is
 * allocated.  The sums run in fp32 (each lane's chunks in two partial sums,
 * a warp tree, then the 8 warp sums in order).  w is taken as constant
 * weights: the kernel requests its first rows before it waits for the
 * previous kernel in the stream (programmatic dependent launch), so w must
 * not be written by a kernel that may still run when the call starts; x may
 * come from the previous kernel. */
int smoe_dense_matvec(const smoe_bf16 *w, const smoe_bf16 *x, int rows, int cols, float *y,
                      smoe_stream stream);

/* SMOE-Q4 quantiser: bf16 weights -> the Q4 layout above.  The offline step
 * before the path ("System Overview", "The Four-Component Architecture": the
 * Sculptor writes the routed experts as quantised vault blocks); the pages
 * give no formula, this library fixes it as min/max affine per group of 64
 * consecutive weights of a row:
 *   mn, mx = least and greatest weight of the group;
 *   scale  = bf16 (nearest, ties to even) of binary32 ((mx - mn) + 0) / 15;
 *   bias   = mn + 0 (exact in bf16; -0 becomes +0);
 *   q      = the code of the level nearest to w: the integer nearest to the
 *            exact quotient (w - mn) / scale, halves to even (it lies in
 *            [0, 15]); 0 wherever scale is 0.
 * w bf16 [rows][cols] (16-byte aligned); codes uint8 [rows][cols/2]
 * (16-byte aligned), scale and bias bf16 [rows][cols/64]; caller-owned device
 * memory.  cols a multiple of 64 (else SMOE_ERR_UNSUPPORTED), rows >= 1.
 * Weights must be finite.  An expert tensor [E][rows][cols] is one call with
 * rows = E * rows. */
int smoe_quantize_q4(const smoe_bf16 *w, int rows, int cols, uint8_t *codes, smoe_bf16 *scale,
                     smoe_bf16 *bias, smoe_stream stream);

/* SMOE-Q2 quantiser: the same reading with 2-bit codes, 3 levels instead of
 * 15 -- scale = bf16 of binary32 ((mx - mn) + 0) / 3, codes clamped to
 * [0, 3] -- into the Q2 layout above (codes uint8 [rows][cols/4], 16-byte
 * aligned).  Arguments and errors as smoe_quantize_q4. */
int smoe_quantize_q2(const smoe_bf16 *w, int rows, int cols, uint8_t *codes, smoe_bf16 *scale,
                     smoe_bf16 *bias, smoe_stream stream);

/* Limit, in nanoseconds of the GPU's global timer, of each grid-wide barrier
 * wait inside the one-kernel decode (smoe_moe_decode, smoe_moe_ffn_decode,
 * smoe_moe_decode_layers, smoe_moe_decode_noalloc when they take the
 * one-kernel plan).  Those barriers are global-memory polls with no copy or
 * tensor-core work outstanding on their account; a wait that reaches the
 * limit gives up, records SMOE_ERR_TIMEOUT in the device status word and lets
 * the kernel run to its end (results are then not valid).  Every other
 * device wait (copies landing, tensor-core work completing) keeps its own
 * fixed limit of 200 ms.  Process-wide; read when a call is enqueued (a CUDA
 * graph keeps the value it was captured with).  Default 200 ms (200000000);
 * 0 makes every barrier that has to wait at all give up (for tests of the
 * timeout path).  The pages have no counterpart: the bound exists because a
 * GPU kernel must never wait forever.  Always returns SMOE_OK. */
int smoe_set_grid_wait_limit(unsigned long long limit_ns);

/* The current grid-barrier wait limit in nanoseconds. */
unsigned long long smoe_get_grid_wait_limit(void);

/* Name of the last CUDA error behind an SMOE_ERR_CUDA returned on this host
 * thread ("cudaSuccess" if none), for diagnostics. */
const char *smoe_last_cuda_error(void);

/* A static string naming a status code. */
const char *smoe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SMOE_H */

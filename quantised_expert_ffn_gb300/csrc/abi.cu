// abi.cu -- the extern "C" entry points of libsmoe.so (declared in include/smoe.h):
// host-side argument checks, workspace layout and kernel launches.  No entry
// point allocates, frees or synchronises (smoe_read_device_status excepted,
// which exists to synchronise).
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "dense.h"
#include "kernels.h"

namespace smoe {

namespace {

constexpr size_t kAlign = 256;

size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of the workspace sections for a layer shape and a token count.
struct WsLayout {
    size_t status, counters, gbar, idx, w, logits, xn, xn16, h, n_union, union_ids, offsets,
        bucket_tok, bucket_rank, bucket_w, slot_of, ready, unit_ctr, h32, hbuf, xperm, obuf, total;
};

WsLayout ws_layout(const smoe_layer &L, int T) {
    WsLayout o{};
    const size_t D = L.d_model, E = L.n_experts, K = L.top_k, F = L.ffn_dim;
    const size_t TK = (size_t)T * K;
    size_t p = 0;
    o.status = p;      p += kAlign;                       // int32 status word (+ padding)
    o.counters = p;    p = up(p + kMaxChunk * 4);
    o.gbar = p;        p = up(p + 8);                    // grid barrier arrival counter (own line)
    o.idx = p;         p = up(p + TK * 4);
    o.w = p;           p = up(p + TK * 4);
    o.logits = p;      p = up(p + (size_t)T * E * 4);
    o.xn = p;          p = up(p + (size_t)T * D * 2);
    o.xn16 = p;        p = up(p + (size_t)T * D * 2);
    o.h = p;           p = up(p + std::max(K * F, fused_h_floats((int)F, (int)K)) * 4);
    o.n_union = p;     p = up(p + 4);
    o.union_ids = p;   p = up(p + E * 4);
    o.offsets = p;     p = up(p + (E + 1) * 4);
    o.bucket_tok = p;  p = up(p + TK * 4);
    o.bucket_rank = p; p = up(p + TK * 4);
    o.bucket_w = p;    p = up(p + TK * 4);
    o.slot_of = p;     p = up(p + TK * 4);
    o.ready = p;       p = up(p + E * 4);
    o.unit_ctr = p;    p = up(p + 2 * 4);
    o.h32 = p;         p = up(p + TK * F * 4);
    o.hbuf = p;        p = up(p + TK * F * 2);
    o.xperm = p;       p = up(p + TK * D * 2);
    o.obuf = p;        p = up(p + TK * D * 4);
    o.total = p;
    return o;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

// Bytes at the head of every workspace that calls expect to find zeroed: the
// status word, the route tickets and the grid-barrier counter (the same for
// every layer shape and token count).
size_t ws_head_bytes() {
    smoe_layer L{};
    L.d_model = kGroup;
    L.n_experts = 1;
    L.top_k = 1;
    L.ffn_dim = kGroup;
    return ws_layout(L, 1).idx;
}

namespace {

int check_layer(const smoe_layer *L) {
    if (!L) return SMOE_ERR_INVALID_ARG;
    if (!L->router_w || !L->gate_q || !L->gate_s || !L->gate_b || !L->up_q || !L->up_s ||
        !L->up_b || !L->down_q || !L->down_s || !L->down_b)
        return SMOE_ERR_INVALID_ARG;
    if (L->group_size != kGroup) return SMOE_ERR_UNSUPPORTED;
    if (L->code_bits != 0 && L->code_bits != 4 && L->code_bits != 2) return SMOE_ERR_UNSUPPORTED;
    const int D = L->d_model, E = L->n_experts, K = L->top_k, F = L->ffn_dim;
    if (D <= 0 || F <= 0 || E <= 0 || K <= 0) return SMOE_ERR_INVALID_ARG;
    if (D % kGroup || F % kGroup) return SMOE_ERR_UNSUPPORTED;
    if (D > kMaxD || F > kMaxF || E > kMaxExperts || K > kMaxTopK || K > E || K * F > kMaxKF)
        return SMOE_ERR_UNSUPPORTED;
    if (!aligned(L->router_w, 16) || !aligned(L->gate_q, 16) || !aligned(L->up_q, 16) ||
        !aligned(L->down_q, 16))
        return SMOE_ERR_INVALID_ARG;
    if (!aligned(L->gate_s, 2) || !aligned(L->gate_b, 2) || !aligned(L->up_s, 2) ||
        !aligned(L->up_b, 2) || !aligned(L->down_s, 2) || !aligned(L->down_b, 2) ||
        (L->rms_gain && !aligned(L->rms_gain, 2)))
        return SMOE_ERR_INVALID_ARG;
    if (L->rms_gain && !(L->rms_eps >= 0.f)) return SMOE_ERR_INVALID_ARG;
    return SMOE_OK;
}

bool is_q2(const smoe_layer &L) { return L.code_bits == 2; }

int check_ws(const smoe_layer *L, int T, void *ws, size_t ws_bytes) {
    if (!ws || !aligned(ws, kAlign)) return SMOE_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*L, T).total) return SMOE_ERR_WORKSPACE;
    return SMOE_OK;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Limit of each grid-barrier spin of the persistent decode kernel (ns);
// smoe_set_grid_wait_limit changes it for calls enqueued afterwards.
std::atomic<unsigned long long> g_grid_wait_ns{kWaitLimitNs};

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SMOE_OK;
    g_last_cuda_error = e;
    return SMOE_ERR_CUDA;
}

// Decode engine: 1 = fused one-kernel layer, 0 = three kernels (router, gate/up,
// down).  SMOE_DECODE_PATH=split selects the latter (cross-check).
int decode_path() {
    static const int v = [] {
        const char *e = getenv("SMOE_DECODE_PATH");
        return (e && strcmp(e, "split") == 0) ? 0 : 1;
    }();   // read once (thread-safe static initialisation)
    return v;
}

// Prefill FFN engine: 1 = tensor cores (tcgen05), 0 = CUDA cores.  Both are
// hand-written kernels of this library; SMOE_PREFILL_PATH=simt selects the
// CUDA-core one (used to cross-check the two).
int prefill_path() {
    static const int v = [] {
        const char *e = getenv("SMOE_PREFILL_PATH");
        return (e && strcmp(e, "simt") == 0) ? 0 : 1;
    }();
    return v;
}

RouteArgs route_args(const smoe_layer &L, const smoe_bf16 *x, void *ws, const WsLayout &o,
                     int32_t *idx, float *w, float *logits, smoe_bf16 *xn, __half *xn16) {
    RouteArgs r{};
    r.x = x;
    r.gain = L.rms_gain;
    r.eps = L.rms_eps;
    r.router_w = L.router_w;
    r.D = L.d_model;
    r.E = L.n_experts;
    r.K = L.top_k;
    r.norm_topk_prob = L.norm_topk_prob ? 1 : 0;
    r.logits = logits ? logits : at<float>(ws, o.logits);
    r.idx = idx;
    r.w = w;
    r.xn_out = xn;
    r.xn16_out = xn16;
    r.counters = at<int32_t>(ws, o.counters);
    r.status = at<int32_t>(ws, o.status);
    return r;
}

}  // namespace

unsigned long long grid_wait_limit_ns() { return g_grid_wait_ns.load(std::memory_order_relaxed); }

}  // namespace smoe

using namespace smoe;

extern "C" {

size_t smoe_workspace_bytes(const smoe_layer *layer, int max_tokens) {
    if (check_layer(layer) != SMOE_OK || max_tokens < 1 || max_tokens > kMaxChunk) return 0;
    return ws_layout(*layer, max_tokens).total;
}

int smoe_workspace_init(void *ws, size_t ws_bytes, smoe_stream stream) {
    if (!ws || ws_bytes == 0) return SMOE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

int smoe_read_device_status(const void *ws, int32_t *status_host, smoe_stream stream) {
    if (!ws || !status_host) return SMOE_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(status_host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e);
}

int smoe_route_topk(const smoe_layer *layer, const smoe_bf16 *x, int T, int32_t *idx, float *w,
                    float *logits_opt, smoe_bf16 *xn_opt, void *ws, size_t ws_bytes,
                    smoe_stream stream) {
    int st = check_layer(layer);
    if (st != SMOE_OK) return st;
    if (!x || !idx || !w || T < 1 || T > kMaxChunk) return SMOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (xn_opt && !aligned(xn_opt, 2))) return SMOE_ERR_INVALID_ARG;
    if ((st = check_ws(layer, T, ws, ws_bytes)) != SMOE_OK) return st;
    const WsLayout o = ws_layout(*layer, T);
    RouteArgs r = route_args(*layer, x, ws, o, idx, w, logits_opt, xn_opt, nullptr);
    return cuda_status(launch_route_topk(r, T, (cudaStream_t)stream, true));
}

int smoe_expert_union(const int32_t *idx, const float *w, int T, int k, int E, int32_t *union_ids,
                      int32_t *n_union, int32_t *offsets, int32_t *bucket_tok,
                      int32_t *bucket_rank, float *bucket_w, int32_t *status_dev,
                      smoe_stream stream) {
    if (!idx || !w || !union_ids || !n_union || !offsets || !bucket_tok || !bucket_rank ||
        !bucket_w)
        return SMOE_ERR_INVALID_ARG;
    if (T < 1 || T > kMaxChunk || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts)
        return SMOE_ERR_INVALID_ARG;
    UnionArgs u{idx, w, T, k, E, union_ids, n_union, offsets, bucket_tok, bucket_rank,
                bucket_w, status_dev, nullptr};
    return cuda_status(launch_expert_union(u, (cudaStream_t)stream, true));
}

// Decode FFN (and routing when idx_in is NULL): the fused one-kernel layer
// when the shape fits its plan, else the three-kernel path.
static int launch_decode_path(const smoe_layer &L, const smoe_bf16 *x, const int32_t *idx_in,
                              const float *w_in, int32_t *idx_out, float *w_out, smoe_bf16 *y,
                              float *expert_out, void *ws, const WsLayout &o, cudaStream_t s) {
    FusedArgs f{};
    f.x = x;
    f.y = y;
    f.gain = L.rms_gain;
    f.eps = L.rms_eps;
    f.D = L.d_model;
    f.F = L.ffn_dim;
    f.K = L.top_k;
    f.E = L.n_experts;
    f.norm_topk_prob = L.norm_topk_prob ? 1 : 0;
    f.router_w = L.router_w;
    f.gq = L.gate_q; f.gs = L.gate_s; f.gb = L.gate_b;
    f.uq = L.up_q;   f.us = L.up_s;   f.ub = L.up_b;
    f.dq = L.down_q; f.ds = L.down_s; f.db = L.down_b;
    f.logits = at<float>(ws, o.logits);
    f.h = at<float>(ws, o.h);
    f.gctr = at<unsigned long long>(ws, o.gbar);
    f.status = at<int32_t>(ws, o.status);
    f.idx_out = idx_out;
    f.w_out = w_out;
    f.idx_in = idx_in;
    f.w_in = w_in;
    f.expert_out = expert_out;
    f.n_layers = 1;
    f.q2 = is_q2(L) ? 1 : 0;
    f.grid_wait_ns = grid_wait_limit_ns();
    if (decode_path() == 1 && fused_plan(f, device_sm_count())) {
        const cudaError_t e = launch_decode_layer(f, s, idx_in == nullptr);
        if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_status(e);
        (void)cudaGetLastError();                           // refused, nothing enqueued: three kernels
    }
    if (f.q2) return SMOE_ERR_UNSUPPORTED;                    // Q2 runs on the one-kernel plan only
    if (!idx_in) {
        RouteArgs r = route_args(L, x, ws, o, idx_out, w_out, nullptr, nullptr, nullptr);
        const int st = cuda_status(launch_route_topk(r, 1, s, true));
        if (st != SMOE_OK) return st;
        idx_in = idx_out;
        w_in = w_out;
    }
    DecodeArgs d{};
    d.x = x;
    d.gain = L.rms_gain;
    d.eps = L.rms_eps;
    d.D = L.d_model;
    d.F = L.ffn_dim;
    d.K = L.top_k;
    d.E = L.n_experts;
    d.idx = idx_in;
    d.w = w_in;
    d.gq = L.gate_q; d.gs = L.gate_s; d.gb = L.gate_b;
    d.uq = L.up_q;   d.us = L.up_s;   d.ub = L.up_b;
    d.dq = L.down_q; d.ds = L.down_s; d.db = L.down_b;
    d.h = at<float>(ws, o.h);
    d.y = y;
    d.expert_out = expert_out;
    d.status = at<int32_t>(ws, o.status);
    const int st = cuda_status(launch_decode_gateup(d, s, true));
    if (st != SMOE_OK) return st;
    return cuda_status(launch_decode_down(d, s, true));
}

int smoe_moe_ffn_decode(const smoe_layer *layer, const smoe_bf16 *x, const int32_t *idx,
                        const float *w, smoe_bf16 *y, float *expert_out_opt, void *ws,
                        size_t ws_bytes, smoe_stream stream) {
    int st = check_layer(layer);
    if (st != SMOE_OK) return st;
    if (!x || !y || !idx || !w || !aligned(x, 16) || !aligned(y, 16)) return SMOE_ERR_INVALID_ARG;
    if (expert_out_opt && !aligned(expert_out_opt, 4)) return SMOE_ERR_INVALID_ARG;
    if ((st = check_ws(layer, 1, ws, ws_bytes)) != SMOE_OK) return st;
    return launch_decode_path(*layer, x, idx, w, nullptr, nullptr, y, expert_out_opt, ws,
                              ws_layout(*layer, 1), (cudaStream_t)stream);
}

int smoe_moe_decode(const smoe_layer *layer, const smoe_bf16 *x, smoe_bf16 *y,
                    int32_t *idx_out_opt, float *w_out_opt, float *expert_out_opt, void *ws,
                    size_t ws_bytes, smoe_stream stream) {
    int st = check_layer(layer);
    if (st != SMOE_OK) return st;
    if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return SMOE_ERR_INVALID_ARG;
    if (expert_out_opt && !aligned(expert_out_opt, 4)) return SMOE_ERR_INVALID_ARG;
    if ((st = check_ws(layer, 1, ws, ws_bytes)) != SMOE_OK) return st;
    const WsLayout o = ws_layout(*layer, 1);
    int32_t *idx = idx_out_opt ? idx_out_opt : at<int32_t>(ws, o.idx);
    float *w = w_out_opt ? w_out_opt : at<float>(ws, o.w);
    return launch_decode_path(*layer, x, nullptr, nullptr, idx, w, y, expert_out_opt, ws, o,
                              (cudaStream_t)stream);
}

int smoe_moe_decode_layers(const smoe_layer *layers, const smoe_layer *layers_dev, int n_layers,
                           const smoe_bf16 *x, smoe_bf16 *y, int32_t *idx_out_opt, float *w_out_opt,
                           void *ws, size_t ws_bytes, smoe_stream stream) {
    if (!layers || !layers_dev || n_layers < 1 || !aligned(layers_dev, alignof(smoe_layer)))
        return SMOE_ERR_INVALID_ARG;
    if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return SMOE_ERR_INVALID_ARG;
    if ((idx_out_opt == nullptr) != (w_out_opt == nullptr)) return SMOE_ERR_INVALID_ARG;
    const smoe_layer &L0 = layers[0];
    bool stack_ok = true;     // every layer meets the one-kernel plan's alignment
    for (int l = 0; l < n_layers; ++l) {
        const smoe_layer &L = layers[l];
        const int st = check_layer(&L);
        if (st != SMOE_OK) return st;
        if (L.d_model != L0.d_model || L.n_experts != L0.n_experts || L.top_k != L0.top_k ||
            L.ffn_dim != L0.ffn_dim || L.norm_topk_prob != L0.norm_topk_prob ||
            is_q2(L) != is_q2(L0) ||
            (L.rms_gain == nullptr) != (L0.rms_gain == nullptr) || L.rms_eps != L0.rms_eps)
            return SMOE_ERR_INVALID_ARG;
        const void *ptrs[] = {L.router_w, L.gate_q, L.gate_s, L.gate_b, L.up_q, L.up_s, L.up_b,
                              L.down_q, L.down_s, L.down_b};
        for (const void *q : ptrs) stack_ok = stack_ok && aligned(q, 16);
        if (L.rms_gain) stack_ok = stack_ok && aligned(L.rms_gain, 16);
    }
    int st = check_ws(&L0, 1, ws, ws_bytes);
    if (st != SMOE_OK) return st;
    const WsLayout o = ws_layout(L0, 1);
    cudaStream_t s = (cudaStream_t)stream;
    smoe_bf16 *act[2] = {at<smoe_bf16>(ws, o.xn), at<smoe_bf16>(ws, o.xn16)};
    if (stack_ok && decode_path() == 1) {
        FusedArgs f{};
        f.x = x;
        f.y = y;
        f.gain = L0.rms_gain;
        f.eps = L0.rms_eps;
        f.D = L0.d_model;
        f.F = L0.ffn_dim;
        f.K = L0.top_k;
        f.E = L0.n_experts;
        f.norm_topk_prob = L0.norm_topk_prob ? 1 : 0;
        f.router_w = L0.router_w;
        f.gq = L0.gate_q; f.gs = L0.gate_s; f.gb = L0.gate_b;
        f.uq = L0.up_q;   f.us = L0.up_s;   f.ub = L0.up_b;
        f.dq = L0.down_q; f.ds = L0.down_s; f.db = L0.down_b;
        f.logits = at<float>(ws, o.logits);
        f.h = at<float>(ws, o.h);
        f.gctr = at<unsigned long long>(ws, o.gbar);
        f.status = at<int32_t>(ws, o.status);
        f.idx_out = idx_out_opt;
        f.w_out = w_out_opt;
        f.layers = layers_dev;
        f.n_layers = n_layers;
        f.act0 = act[0];
        f.act1 = act[1];
        f.q2 = is_q2(L0) ? 1 : 0;
        f.grid_wait_ns = grid_wait_limit_ns();
        if (fused_plan(f, device_sm_count())) {
            const cudaError_t e = launch_decode_layer(f, s, true);
            if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_status(e);
            (void)cudaGetLastError();                       // refused, nothing enqueued: per layer
        }
    }
    // one launch sequence per layer, activations ping-ponging in the workspace
    for (int l = 0; l < n_layers; ++l) {
        const smoe_bf16 *xin = l == 0 ? x : act[(l - 1) & 1];
        smoe_bf16 *yout = l == n_layers - 1 ? y : act[l & 1];
        int32_t *idx = idx_out_opt ? idx_out_opt + (size_t)l * L0.top_k : at<int32_t>(ws, o.idx);
        float *w = w_out_opt ? w_out_opt + (size_t)l * L0.top_k : at<float>(ws, o.w);
        st = launch_decode_path(layers[l], xin, nullptr, nullptr, idx, w, yout, nullptr, ws, o, s);
        if (st != SMOE_OK) return st;
    }
    return SMOE_OK;
}

static int prefill_chunk(const smoe_layer *layer, const smoe_bf16 *x, int T, smoe_bf16 *y,
                         int32_t *idx_out_opt, float *w_out_opt, float *expert_out, void *ws,
                         size_t ws_bytes, smoe_stream stream) {
    int st = check_layer(layer);
    if (st != SMOE_OK) return st;
    if (!x || !y || T < 1 || T > kMaxChunk || !aligned(x, 16) || !aligned(y, 16) || x == y)
        return SMOE_ERR_INVALID_ARG;
    if (expert_out && !aligned(expert_out, 16)) return SMOE_ERR_INVALID_ARG;
    if ((st = check_ws(layer, T, ws, ws_bytes)) != SMOE_OK) return st;
    const smoe_layer &L = *layer;
    const bool tc = prefill_path() == 1 && prefill_tc_supported(L.d_model, L.ffn_dim);
    if (is_q2(L) && !tc) return SMOE_ERR_UNSUPPORTED;        // Q2 runs on the tensor-core path only
    const WsLayout o = ws_layout(L, T);
    cudaStream_t s = (cudaStream_t)stream;
    int32_t *idx = idx_out_opt ? idx_out_opt : at<int32_t>(ws, o.idx);
    float *w = w_out_opt ? w_out_opt : at<float>(ws, o.w);
    RouteArgs r = route_args(L, x, ws, o, idx, w, nullptr, at<smoe_bf16>(ws, o.xn),
                             at<__half>(ws, o.xn16));
    if ((st = cuda_status(launch_route_topk(r, T, s, true))) != SMOE_OK) return st;
    UnionArgs u{idx, w, T, L.top_k, L.n_experts, at<int32_t>(ws, o.union_ids),
                at<int32_t>(ws, o.n_union), at<int32_t>(ws, o.offsets),
                at<int32_t>(ws, o.bucket_tok), at<int32_t>(ws, o.bucket_rank),
                at<float>(ws, o.bucket_w), at<int32_t>(ws, o.status), at<int32_t>(ws, o.slot_of)};
    if ((st = cuda_status(launch_expert_union(u, s, true))) != SMOE_OK) return st;
    PrefillArgs p{};
    p.x = x;
    p.T = T;
    p.D = L.d_model;
    p.F = L.ffn_dim;
    p.K = L.top_k;
    p.E = L.n_experts;
    p.xn16 = at<__half>(ws, o.xn16);
    p.n_union = u.n_union;
    p.union_ids = u.union_ids;
    p.offsets = u.offsets;
    p.bucket_tok = u.bucket_tok;
    p.bucket_rank = u.bucket_rank;
    p.slot_of = u.slot_of;
    p.w = w;
    p.gq = L.gate_q; p.gs = L.gate_s; p.gb = L.gate_b;
    p.uq = L.up_q;   p.us = L.up_s;   p.ub = L.up_b;
    p.dq = L.down_q; p.ds = L.down_s; p.db = L.down_b;
    p.xperm = at<__half>(ws, o.xperm);
    p.hbuf = at<__half>(ws, o.hbuf);
    p.obuf = at<float>(ws, o.obuf);
    p.y = y;
    p.expert_out = expert_out;
    p.status = at<int32_t>(ws, o.status);
    p.ready = at<int32_t>(ws, o.ready);
    p.unit_ctr = at<int32_t>(ws, o.unit_ctr);
    p.num_sms = device_sm_count();
    p.q2 = is_q2(L) ? 1 : 0;
    if (tc) {
        if ((st = cuda_status(launch_prefill_tc(p, s))) != SMOE_OK) return st;
        return cuda_status(launch_prefill_combine(p, s, true));
    }
    return cuda_status(launch_prefill_simt(p, at<smoe_bf16>(ws, o.xn), at<float>(ws, o.h32), s, true));
}

int smoe_moe_prefill_chunk(const smoe_layer *layer, const smoe_bf16 *x, int T, smoe_bf16 *y,
                           int32_t *idx_out_opt, float *w_out_opt, void *ws, size_t ws_bytes,
                           smoe_stream stream) {
    return prefill_chunk(layer, x, T, y, idx_out_opt, w_out_opt, nullptr, ws, ws_bytes, stream);
}

int smoe_moe_prefill_chunk_experts(const smoe_layer *layer, const smoe_bf16 *x, int T, smoe_bf16 *y,
                                   int32_t *idx_out_opt, float *w_out_opt, float *expert_out,
                                   void *ws, size_t ws_bytes, smoe_stream stream) {
    if (!expert_out) return SMOE_ERR_INVALID_ARG;
    return prefill_chunk(layer, x, T, y, idx_out_opt, w_out_opt, expert_out, ws, ws_bytes, stream);
}

const char *smoe_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

int smoe_set_grid_wait_limit(unsigned long long limit_ns) {
    g_grid_wait_ns.store(limit_ns, std::memory_order_relaxed);
    return SMOE_OK;
}

unsigned long long smoe_get_grid_wait_limit(void) { return g_grid_wait_ns.load(std::memory_order_relaxed); }

int smoe_dense_matvec(const smoe_bf16 *w, const smoe_bf16 *x, int rows, int cols, float *y,
                      smoe_stream stream) {
    if (!w || !x || !y || rows < 1 || cols < 1) return SMOE_ERR_INVALID_ARG;
    if (cols % 8 || cols > kMaxD) return SMOE_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4)) return SMOE_ERR_INVALID_ARG;
    return cuda_status(launch_dense_matvec(w, x, rows, cols, y, (cudaStream_t)stream));
}

int smoe_quantize_q4(const smoe_bf16 *w, int rows, int cols, uint8_t *codes, smoe_bf16 *scale,
                     smoe_bf16 *bias, smoe_stream stream) {
    if (!w || !codes || !scale || !bias || rows < 1 || cols < 1) return SMOE_ERR_INVALID_ARG;
    if (cols % kGroup) return SMOE_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scale, 2) || !aligned(bias, 2))
        return SMOE_ERR_INVALID_ARG;
    const long long n_groups = (long long)rows * (cols / kGroup);
    return cuda_status(launch_quantize(w, n_groups, 4, codes, scale, bias, (cudaStream_t)stream));
}

int smoe_quantize_q2(const smoe_bf16 *w, int rows, int cols, uint8_t *codes, smoe_bf16 *scale,
                     smoe_bf16 *bias, smoe_stream stream) {
    if (!w || !codes || !scale || !bias || rows < 1 || cols < 1) return SMOE_ERR_INVALID_ARG;
    if (cols % kGroup) return SMOE_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(scale, 2) || !aligned(bias, 2))
        return SMOE_ERR_INVALID_ARG;
    const long long n_groups = (long long)rows * (cols / kGroup);
    return cuda_status(launch_quantize(w, n_groups, 2, codes, scale, bias, (cudaStream_t)stream));
}

const char *smoe_status_string(int status) {
    switch (status) {
    case SMOE_OK: return "SMOE_OK";
    case SMOE_ERR_INVALID_ARG: return "SMOE_ERR_INVALID_ARG: NULL pointer, bad size or alignment";
    case SMOE_ERR_UNSUPPORTED: return "SMOE_ERR_UNSUPPORTED: shape outside the supported set";
    case SMOE_ERR_WORKSPACE: return "SMOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SMOE_ERR_CUDA: return "SMOE_ERR_CUDA: a CUDA launch or runtime call failed";
    case SMOE_ERR_TIMEOUT: return "SMOE_ERR_TIMEOUT: a bounded device wait gave up";
    case SMOE_ERR_DEVICE: return "SMOE_ERR_DEVICE: bad data found on the device";
    case SMOE_ERR_RANGE: return "SMOE_ERR_RANGE: a value beyond fp16's range on the tensor-core prefill";
    default: return "unknown smoe status";
    }
}

}  // extern "C"

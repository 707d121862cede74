// route.cu -- RMSNorm + exact router gate + top-k + mixing weights.
//
// "Optimizations" page, "Routing Is Exact -- Prompt and Generation Alike":
// every layer evaluates the real router gate on the true hidden state, with
// top-8 selection and norm_topk_prob mixing weights.  The pages run this
// 128 x d_model matvec on the CPU between GPU command buffers; here it stays
// on the GPU, as the pages' own horizon item ("The Dense Ceiling --
// GPU-Resident Epilogue") proposes, and top-k stays on the GPU too.
//
// Grid (ceil(E / 16), T): a CTA of 16 warps normalises token t's hidden state
// into shared memory, and each warp computes one router row (one expert) as a
// warp-per-row dot product with 16-byte coalesced loads.  The last CTA of a
// token to finish (device-scope ticket, no spinning) ranks the E logits and
// writes the top-k ids and weights (rank = the count of larger unique 64-bit keys).
#include "common.cuh"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kRouteWarps = 16;
constexpr int kRouteThreads = kRouteWarps * 32;

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kRouteWarps; ++i) t += red[i];
    __syncthreads();
    return t;
}

// Total order used by top-k: larger logit first, equal logits keep the lower
// id.  NaN ranks below everything; -0 and +0 are equal.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 0u;
    v = v + 0.0f;
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// At most 32 registers a thread, so 4 CTAs of 512 threads fit an SM and a
// 64-token chunk's 512 CTAs run as one wave (CTAs of 8 warps at the 42
// registers the code would otherwise take left a second wave).
__global__ void __launch_bounds__(kRouteThreads, 4) k_route_topk(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int D = a.D, E = a.E, K = a.K;
    const int t = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);               // [D] normed bf16
    __shared__ float red[kRouteWarps];
    __shared__ __align__(16) unsigned long long keys[kMaxExperts];
    __shared__ float lsel[kMaxTopK];
    __shared__ int isel[kMaxTopK];
    __shared__ int am_last;

    pdl_wait();  // x comes from the previous kernel in the stream
    pdl_launch_dependents();

    const uint16_t *x = a.x + (size_t)t * D;
    // ---- RMSNorm (fp32) into shared memory ----
    if (a.gain) {
        // the reduction order of block_rms_inv (256 threads: stride-256 partials,
        // a warp tree, the 8 warp sums in order), by the first 256 threads
        float ss = 0.f;
        if (tid < 256)
            for (int d = tid; d < D; d += 256) {
                const float v = bf16_to_f32(ld_cg_u16(x + d));
                ss = fmaf(v, v, ss);
            }
        ss = warp_sum(ss);
        if (lane == 0 && warp < 8) red[warp] = ss;
        __syncthreads();
        float tt = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) tt += red[i];
        const float inv = 1.0f / sqrtf(tt / (float)D + a.eps);
        for (int d = tid; d < D; d += kRouteThreads) xs[d] = rms_apply(x[d], inv, a.gain[d]);
    } else {
        for (int d = tid * 8; d < D; d += kRouteThreads * 8)
            *reinterpret_cast<uint4 *>(xs + d) = *reinterpret_cast<const uint4 *>(x + d);
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        if (a.xn_out)
            for (int d = tid; d < D; d += kRouteThreads) a.xn_out[(size_t)t * D + d] = xs[d];
        if (a.xn16_out)   // the tensor-core prefill's fp16 copy: report values past its range
            for (int d = tid; d < D; d += kRouteThreads) {
                const float v = bf16_to_f32(xs[d]);
                if (fabsf(v) > 65504.f) set_status(a.status, SMOE_ERR_RANGE);
                a.xn16_out[(size_t)t * D + d] = __float2half_rn(v);
            }
    }

    // ---- router rows: one warp per expert ----
    const int e = blockIdx.x * kRouteWarps + warp;
    if (e < E) {
        const uint16_t *wr = a.router_w + (size_t)e * D;
        float acc0 = 0.f, acc1 = 0.f;
        for (int d = lane * 8; d < D; d += 256) {
            uint4 wv = ld_stream16(wr + d);
            uint4 xv = *reinterpret_cast<const uint4 *>(xs + d);
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc0 = fmaf(__uint_as_float(ww[q] << 16), __uint_as_float(xx[q] << 16), acc0);
                acc1 = fmaf(__uint_as_float(ww[q] & 0xFFFF0000u), __uint_as_float(xx[q] & 0xFFFF0000u), acc1);
            }
        }
        float l = warp_sum(acc0 + acc1);
        if (lane == 0) a.logits[(size_t)t * E + e] = l;
    }

    // ---- last CTA of this token ranks the logits ----
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int ticket = atomicAdd(&a.counters[t], 1);
        am_last = (ticket == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!am_last) return;
    __threadfence();
    if (tid == 0) a.counters[t] = 0;  // leave the workspace zeroed for the next call

    const float *lg = a.logits + (size_t)t * E;
    float my = -INFINITY;
    unsigned long long k0 = 0;
    if (tid < E) {
        my = __ldcg(lg + tid);
        // unique key: the larger logit first, equal logits keep the lower id
        k0 = ((unsigned long long)order_key(my) << 32) | (0xFFFFFFFFu - (uint32_t)tid);
        keys[tid] = k0;
    }
    __syncthreads();
    if (tid < E) {
        int r0 = 0, r1 = 0;
        const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(keys);
        for (int j = 0; j < E / 2; ++j) {
            const ulonglong2 kk = k2[j];
            r0 += kk.x > k0;
            r1 += kk.y > k0;
        }
        if (E & 1) r0 += keys[E - 1] > k0;
        const int rank = r0 + r1;
        if (rank < K) {
            isel[rank] = tid;
            lsel[rank] = my;
        }
    }
    __syncthreads();
    const float m = lsel[0];
    float denom;
    if (a.norm_topk_prob) {
        float s = 0.f;
        for (int i = 0; i < K; ++i) s += expf(lsel[i] - m);
        denom = s;
    } else {
        float p = (tid < E) ? expf(my - m) : 0.f;
        denom = block_sum(p, red);
    }
    if (tid < K) {
        a.idx[(size_t)t * K + tid] = isel[tid];
        a.w[(size_t)t * K + tid] = expf(lsel[tid] - m) / denom;
    }
}

}  // namespace

cudaError_t launch_route_topk(const RouteArgs &a, int T, cudaStream_t s, bool pdl) {
    dim3 grid((a.E + kRouteWarps - 1) / kRouteWarps, T);
    size_t smem = (size_t)a.D * sizeof(uint16_t);
    return launch_kernel(k_route_topk, grid, dim3(kRouteThreads), smem, s, pdl, a);
}

}  // namespace smoe

// prefill_simt.cu -- prefill chunk FFN on the CUDA cores (bucket by bucket).
//
// "Optimizations" page, "Prefill Reads Each Expert Once, Not Once Per Token":
// each union expert's rows are read once per chunk and applied to every token
// of its bucket.  This path keeps one expert row in registers (warp per row,
// lane per group of 64 inputs, as in the decode kernels) and loops over the
// bucket's tokens, so the row is fetched from HBM once however many tokens
// use it.  It computes exactly what the tensor-core path computes, in fp32
// throughout (h stays fp32), and serves as its cross-check and as the path
// for shapes the tensor-core kernels do not take.
//
// k_prefill_gateup_simt: grid (F/8, E) -- CTA (j-block, union position u);
//   warp -> row j; H[slot][j] = SiLU(gate_e . xn_t) * (up_e . xn_t) for every
//   bucket slot (token t) of u.
// k_prefill_down_simt: grid (D/8, E) -- warp -> row d; O[slot][d] = down_e . H[slot].
// k_prefill_combine: y[t] = x[t] + sum_i w[t][i] O[slot(t, i)], rank order
//   (and, when asked, each token's unweighted O[slot(t, i)] in rank order).
#include "common.cuh"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxNGP = kMaxD / kGroup / 32;   // 4 group passes at D = 8192

__device__ __forceinline__ void load_x64(const uint16_t *xrow, int g, float (&xv)[64]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(xrow + g * 64);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4 v = __ldcg(p + q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            xv[q * 8 + 2 * r] = __uint_as_float(w[r] << 16);
            xv[q * 8 + 2 * r + 1] = __uint_as_float(w[r] & 0xFFFF0000u);
        }
    }
}

// sum over 64 codes of (128 + q) * x (codes in 32 bytes), as two partial sums
__device__ __forceinline__ float dot64(uint4 c0, uint4 c1, const float (&xv)[64]) {
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 8; ++m)
        dot8(cw[m], make_float4(xv[8 * m], xv[8 * m + 1], xv[8 * m + 2], xv[8 * m + 3]),
             make_float4(xv[8 * m + 4], xv[8 * m + 5], xv[8 * m + 6], xv[8 * m + 7]), acc);
    return acc.x + acc.y;
}

struct SimtArgs {
    PrefillArgs p;
    const uint16_t *xn;     // [T][D] bf16 normed inputs
    float *h32;             // [T*K][F]
};

__global__ void __launch_bounds__(kThreads) k_prefill_gateup_simt(SimtArgs sa) {
    const PrefillArgs &a = sa.p;
    pdl_wait();
    pdl_launch_dependents();
    const int u = blockIdx.y;
    if (u >= *a.n_union) return;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (j >= a.F) return;
    const int D = a.D, NG = D / kGroup, NGP = (NG + 31) / 32;
    const int e = a.union_ids[u];
    const int s0 = a.offsets[u], s1 = a.offsets[u + 1];
    const size_t row = (size_t)e * a.F + j;
    uint4 gc[kMaxNGP][2], uc[kMaxNGP][2];
    float gs[kMaxNGP], gb[kMaxNGP], us[kMaxNGP], ub[kMaxNGP];
#pragma unroll
    for (int gp = 0; gp < kMaxNGP; ++gp) {
        const int g = gp * 32 + lane;
        if (gp < NGP && g < NG) {
            const uint8_t *gr = a.gq + row * (D / 2) + g * 32;
            const uint8_t *ur = a.uq + row * (D / 2) + g * 32;
            gc[gp][0] = ld_stream16(gr); gc[gp][1] = ld_stream16(gr + 16);
            uc[gp][0] = ld_stream16(ur); uc[gp][1] = ld_stream16(ur + 16);
            gs[gp] = bf16_to_f32(ld_nc_u16(a.gs + row * NG + g));
            gb[gp] = bf16_to_f32(ld_nc_u16(a.gb + row * NG + g));
            us[gp] = bf16_to_f32(ld_nc_u16(a.us + row * NG + g));
            ub[gp] = bf16_to_f32(ld_nc_u16(a.ub + row * NG + g));
        }
    }
    for (int s = s0; s < s1; ++s) {
        const uint16_t *xrow = sa.xn + (size_t)a.bucket_tok[s] * D;
        float ag = 0.f, au = 0.f;
#pragma unroll
        for (int gp = 0; gp < kMaxNGP; ++gp) {
            const int g = gp * 32 + lane;
            if (gp < NGP && g < NG) {
                float xv[64];
                load_x64(xrow, g, xv);
                float X = 0.f;
#pragma unroll
                for (int k = 0; k < 64; ++k) X += xv[k];
                ag += gs[gp] * dot64(gc[gp][0], gc[gp][1], xv) + (gb[gp] - 128.f * gs[gp]) * X;
                au += us[gp] * dot64(uc[gp][0], uc[gp][1], xv) + (ub[gp] - 128.f * us[gp]) * X;
            }
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) sa.h32[(size_t)s * a.F + j] = silu_mul(ag, au);
    }
}

__global__ void __launch_bounds__(kThreads) k_prefill_down_simt(SimtArgs sa) {
    const PrefillArgs &a = sa.p;
    pdl_wait();
    pdl_launch_dependents();
    const int u = blockIdx.y;
    if (u >= *a.n_union) return;
    const int d = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (d >= a.D) return;
    const int F = a.F, NC = F / 32;        // 16-byte chunks (half groups) per row
    const int e = a.union_ids[u];
    const int s0 = a.offsets[u], s1 = a.offsets[u + 1];
    const size_t row = (size_t)e * a.D + d;
    for (int s = s0; s < s1; ++s) {
        const float *hrow = sa.h32 + (size_t)s * F;
        float acc = 0.f;
        for (int c = lane; c < NC; c += 32) {
            const uint4 cv = ld_stream16(a.dq + row * (F / 2) + c * 16);
            const float sc = bf16_to_f32(ld_nc_u16(a.ds + row * (F / kGroup) + (c >> 1)));
            const float bi = bf16_to_f32(ld_nc_u16(a.db + row * (F / kGroup) + (c >> 1)));
            const float4 *hp = reinterpret_cast<const float4 *>(hrow + c * 32);
            float2 acc2 = make_float2(0.f, 0.f);
            float Hs = 0.f;
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 ha = __ldcg(hp + 2 * m), hb = __ldcg(hp + 2 * m + 1);
                dot8(cw[m], ha, hb, acc2);
                Hs += (ha.x + ha.y) + (ha.z + ha.w) + (hb.x + hb.y) + (hb.z + hb.w);
            }
            acc += sc * (acc2.x + acc2.y) + (bi - 128.f * sc) * Hs;
        }
        acc = warp_sum(acc);
        if (lane == 0) a.obuf[(size_t)s * a.D + d] = acc;
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads) k_prefill_combine(PrefillArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    __shared__ int slot[kMaxTopK];
    __shared__ float wt[kMaxTopK];
    if (threadIdx.x < a.K) {
        slot[threadIdx.x] = a.slot_of[t * a.K + threadIdx.x];
        wt[threadIdx.x] = a.w[t * a.K + threadIdx.x];
    }
    __syncthreads();
    // CTA (t, blockIdx.y) covers elements [1024*by, 1024*by + 1024) of token t,
    // four consecutive ones per thread (D is a multiple of 64).  All K slot
    // rows are requested before the sums, which then run in rank order.
    const int d = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (d >= a.D) return;
    float4 o[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i)
        o[i] = (i < a.K && slot[i] >= 0)
                   ? __ldcg(reinterpret_cast<const float4 *>(a.obuf + (size_t)slot[i] * a.D + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint2 xr = *reinterpret_cast<const uint2 *>(a.x + (size_t)t * a.D + d);
    float y0 = __uint_as_float(xr.x << 16), y1 = __uint_as_float(xr.x & 0xFFFF0000u);
    float y2 = __uint_as_float(xr.y << 16), y3 = __uint_as_float(xr.y & 0xFFFF0000u);
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i)
        if (i < a.K && slot[i] >= 0) {
            y0 = fmaf(wt[i], o[i].x, y0);
            y1 = fmaf(wt[i], o[i].y, y1);
            y2 = fmaf(wt[i], o[i].z, y2);
            y3 = fmaf(wt[i], o[i].w, y3);
        }
    if (a.expert_out) {
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i)
            if (i < a.K)
                *reinterpret_cast<float4 *>(a.expert_out + ((size_t)t * a.K + i) * a.D + d) = o[i];
    }
    uint2 yr;
    yr.x = (uint32_t)f32_to_bf16(y0) | ((uint32_t)f32_to_bf16(y1) << 16);
    yr.y = (uint32_t)f32_to_bf16(y2) | ((uint32_t)f32_to_bf16(y3) << 16);
    *reinterpret_cast<uint2 *>(a.y + (size_t)t * a.D + d) = yr;
}

cudaError_t launch_prefill_combine(const PrefillArgs &a, cudaStream_t s, bool pdl) {
    return launch_kernel(k_prefill_combine, dim3(a.T, (a.D + 1023) / 1024), dim3(kThreads), 0, s, pdl, a);
}

cudaError_t launch_prefill_simt(const PrefillArgs &a, const uint16_t *xn, float *h32,
                                cudaStream_t s, bool pdl) {
    SimtArgs sa{a, xn, h32};
    cudaError_t err = launch_kernel(k_prefill_gateup_simt, dim3((a.F + 7) / 8, a.E), dim3(kThreads), 0,
                                    s, pdl, sa);
    if (err != cudaSuccess) return err;
    err = launch_kernel(k_prefill_down_simt, dim3((a.D + 7) / 8, a.E), dim3(kThreads), 0, s, pdl, sa);
    if (err != cudaSuccess) return err;
    return launch_prefill_combine(a, s, pdl);
}

}  // namespace smoe

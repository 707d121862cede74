// decode.cu -- batch-1 SMOE-Q4 expert FFN: gate+up fused, then down with the
// weighted sum into the residual.  The three-kernel path for shapes outside
// the one-kernel plan of decode_fused.cu (SMOE-Q4 only: SMOE-Q2 layers run on
// that plan or are refused).
//
// "Optimizations" page, "Coalesced GPU Kernels -- Expert FFN and Dense
// Matvec": lanes of one 32-wide group share an output row and read
// consecutive 16-byte chunks; the input vector is staged once per group of
// rows; the inner loop is FMA; the affine dequant is folded into a per-chunk
// epilogue and gate and up are computed in one pass.  "System Overview", per-
// token table, Metal Kernel row: the outputs are weighted-summed into the
// residual.
//
// Arithmetic (exact fp32 dequant): a code q becomes the float 128 + q with one
// byte permute (see dot8 in common.cuh), so a group of 64 inputs gives
//   sum_k w_k x_k = s * sum_k (128 + q_k) x_k + (b - 128 s) * sum_k x_k
// with w_k = s q_k + b; the group sum of x is computed once per CTA.  The
// packed f32x2 FMA halves the FMA issue count.
//
// k_decode_gateup: warp per (expert slot, row j) pair of gate and up rows;
// lane l owns group l (and l+32, ...) of the row: two 16-byte loads per row,
// so a warp reads each 1 KiB row in one coalesced sweep.  The normed input
// sits in shared memory in a lane-interleaved order (conflict-free 16-byte
// reads).  h = SiLU(g) * u goes to an fp32 scratch [k][F].
//
// k_decode_down: CTA per block of output rows d; each 8-lane subgroup owns one
// (expert slot, row) item and reads its row in 128-byte sweeps; per-item
// results land in shared memory and are combined in rank order with the
// residual: y[d] = x[d] + sum_i w_i o_i[d] (fp32, one bf16 rounding).
#include "common.cuh"
#include "host_cache.h"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Normalise x (RMSNorm when gain != NULL) into `xs` (fp32, lane-interleaved:
// element d of group g = 32*gp + l sits at float4 index (gp*16 + m)*32 + l,
// component c, with d % 64 = 4m + c) and its group sums into `xg`.
__device__ void stage_normed_input(const uint16_t *x, const uint16_t *gain, float eps, int D,
                                   float *xs, float *xg, float *red) {
    const int tid = threadIdx.x;
    const float inv = gain ? block_rms_inv(x, D, eps, red) : 1.f;
    for (int d = tid; d < D; d += kThreads) {
        const uint16_t xv = ld_cg_u16(x + d);
        const float v = gain ? bf16_to_f32(rms_apply(xv, inv, gain[d])) : bf16_to_f32(xv);
        const int g = d >> 6, r = d & 63;
        xs[(((g >> 5) * 16 + (r >> 2)) * 32 + (g & 31)) * 4 + (r & 3)] = v;
    }
    // groups past D (when D/64 is not a multiple of 32) read as zeros
    const int NGP0 = (D / kGroup + 31) / 32;
    for (int d = D + tid; d < NGP0 * 2048; d += kThreads) {
        const int g = d >> 6, r = d & 63;
        xs[(((g >> 5) * 16 + (r >> 2)) * 32 + (g & 31)) * 4 + (r & 3)] = 0.f;
    }
    __syncthreads();
    const int NG = D / kGroup;
    const int NGP = (NG + 31) / 32;
    for (int g = tid; g < NGP * 32; g += kThreads) {
        float s = 0.f;
        if (g < NG)
            for (int r = 0; r < kGroup; ++r)
                s += xs[(((g >> 5) * 16 + (r >> 2)) * 32 + (g & 31)) * 4 + (r & 3)];
        xg[g] = s;
    }
    __syncthreads();
}

struct GuUnit {
    uint4 g0, g1, u0, u1;
    float gs, gb, us, ub;
};

__device__ __forceinline__ void gu_load(GuUnit &U, const DecodeArgs &a, const int *eid, int p,
                                        int gp, int lane, int NG) {
    const int i = p / a.F, j = p - i * a.F;
    const int e = eid[i];
    const int g = gp * 32 + lane;
    if (e >= 0 && g < NG) {
        const size_t row = (size_t)e * a.F + j;
        const uint8_t *gr = a.gq + row * (a.D / 2) + (size_t)g * 32;
        const uint8_t *ur = a.uq + row * (a.D / 2) + (size_t)g * 32;
        U.g0 = ld_stream16(gr);
        U.g1 = ld_stream16(gr + 16);
        U.u0 = ld_stream16(ur);
        U.u1 = ld_stream16(ur + 16);
        const size_t si = row * NG + g;
        U.gs = bf16_to_f32(ld_nc_u16(a.gs + si));
        U.gb = bf16_to_f32(ld_nc_u16(a.gb + si));
        U.us = bf16_to_f32(ld_nc_u16(a.us + si));
        U.ub = bf16_to_f32(ld_nc_u16(a.ub + si));
    } else {
        U.g0 = U.g1 = U.u0 = U.u1 = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        U.gs = U.gb = U.us = U.ub = 0.f;
    }
}

__global__ void __launch_bounds__(kThreads) k_decode_gateup(DecodeArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int D = a.D, F = a.F, K = a.K;
    const int NG = D / kGroup, NGP = (NG + 31) / 32;
    float *xs = sm;                         // NGP*16*32*4 floats
    float *xg = sm + NGP * 2048;            // NGP*32 floats
    __shared__ float red[kWarps];
    __shared__ int eid[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // x was written two launches back (before the router ran): safe to read now.
    stage_normed_input(a.x, a.gain, a.eps, D, xs, xg, red);
    pdl_wait();                             // expert ids from the router
    pdl_launch_dependents();
    if (tid < K) {
        int e = a.idx[tid];
        if (e < 0 || e >= a.E) {
            set_status(a.status, SMOE_ERR_DEVICE);
            e = -1;
        }
        eid[tid] = e;
    }
    __syncthreads();

    const int P = K * F;
    const int per = (P + gridDim.x - 1) / gridDim.x;
    const int p0 = blockIdx.x * per, p1 = min(P, p0 + per);
    int p = p0 + warp, gp = 0;
    if (p >= p1) return;
    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);

    GuUnit cur, nxt;
    gu_load(cur, a, eid, p, gp, lane, NG);
    float ag = 0.f, au = 0.f;
    while (true) {
        int np = p, ngp = gp + 1;
        if (ngp == NGP) { ngp = 0; np = p + kWarps; }
        const bool more = np < p1;
        if (more) gu_load(nxt, a, eid, np, ngp, lane, NG);

        const float4 *xv = xs4 + gp * 16 * 32 + lane;
        float2 accg = make_float2(0.f, 0.f), accu = make_float2(0.f, 0.f);
        const uint32_t gw[8] = {cur.g0.x, cur.g0.y, cur.g0.z, cur.g0.w, cur.g1.x, cur.g1.y, cur.g1.z, cur.g1.w};
        const uint32_t uw[8] = {cur.u0.x, cur.u0.y, cur.u0.z, cur.u0.w, cur.u1.x, cur.u1.y, cur.u1.z, cur.u1.w};
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float4 xa = xv[(2 * m) * 32], xb = xv[(2 * m + 1) * 32];
            dot8(gw[m], xa, xb, accg);
            dot8(uw[m], xa, xb, accu);
        }
        const float X = xg[gp * 32 + lane];
        ag += cur.gs * (accg.x + accg.y) + (cur.gb - 128.f * cur.gs) * X;
        au += cur.us * (accu.x + accu.y) + (cur.ub - 128.f * cur.us) * X;
        if (gp == NGP - 1) {
            ag = warp_sum(ag);
            au = warp_sum(au);
            if (lane == 0) a.h[p] = silu_mul(ag, au);
            ag = au = 0.f;
        }
        if (!more) break;
        cur = nxt;
        p = np;
        gp = ngp;
    }
}

// ---------------------------------------------------------------- down + combine

struct DnUnit {
    uint4 c[4];
    float s[4], b[4];
};

// Rows per CTA of the down kernel.
__host__ __device__ inline int down_rows_per_cta(int D) { return D >= 4096 ? 16 : 8; }

__global__ void __launch_bounds__(kThreads) k_decode_down(DecodeArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int D = a.D, F = a.F, K = a.K;
    const int NC = F / 32;                 // 16-byte chunks per row
    const int MC = (NC + 7) / 8;           // chunks per lane
    const int R = down_rows_per_cta(D);
    const int d0 = blockIdx.x * R;
    const int rows = min(R, D - d0);
    float *hs = sm;                        // K*MC*8*8 float4 = K*MC*256 floats
    float *hc = hs + K * MC * 256;         // [K][MC*8] chunk sums
    float *os = hc + K * MC * 8;           // [K][R]
    __shared__ int eid[kMaxTopK];
    __shared__ float wsel[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s8 = lane & 7, sub = lane >> 3;
    const int S = warp * 4 + sub;          // subgroup index 0..31

    pdl_wait();
    pdl_launch_dependents();
    if (tid < K) {
        int e = a.idx[tid];
        if (e < 0 || e >= a.E) e = -1;
        eid[tid] = e;
        wsel[tid] = a.w[tid];
    }
    // stage h (fp32 [K][F]) lane-interleaved: chunk c = s8 + 8m, float4 k of the chunk
    for (int q = tid; q < K * MC * 64; q += kThreads) {
        const int i = q / (MC * 64), rem = q - i * MC * 64;
        const int m = rem / 64, k = (rem / 8) & 7, cs = rem & 7;
        const int c = cs + 8 * m;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < NC) v = __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)i * F + c * 32 + k * 4));
        reinterpret_cast<float4 *>(hs)[q] = v;
    }
    __syncthreads();
    for (int q = tid; q < K * MC * 8; q += kThreads) {
        const int i = q / (MC * 8), c = q - i * MC * 8;
        const int m = c / 8, cs = c & 7;
        float s = 0.f;
        const float4 *hp = reinterpret_cast<const float4 *>(hs) + ((i * MC + m) * 8) * 8 + cs;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = hp[k * 8];
            s += (v.x + v.y) + (v.z + v.w);
        }
        hc[q] = s;
    }
    __syncthreads();

    const int items = K * rows;
    const float4 *hs4 = reinterpret_cast<const float4 *>(hs);
    // warp-uniform trip count: every lane reaches the shuffles below
    for (int base = warp * 4; base < items; base += 32) {
        const int q = base + (S - warp * 4);
        const bool live = q < items;
        const int i = live ? q / rows : 0, dl = live ? q - i * rows : 0;
        const int e = eid[i];
        float acc = 0.f;
        if (live && e >= 0) {
            const size_t row = (size_t)e * D + d0 + dl;
            const uint8_t *rp = a.dq + row * (F / 2);
            for (int mb = 0; mb < MC; mb += 4) {
                DnUnit U;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int c = s8 + 8 * (mb + t);
                    if (mb + t < MC && c < NC) {
                        U.c[t] = ld_stream16(rp + c * 16);
                        const size_t si = row * (F / kGroup) + (c >> 1);
                        U.s[t] = bf16_to_f32(ld_nc_u16(a.ds + si));
                        U.b[t] = bf16_to_f32(ld_nc_u16(a.db + si));
                    } else {
                        U.c[t] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                        U.s[t] = U.b[t] = 0.f;
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int m = mb + t;
                    if (m < MC) {
                        const float4 *hv = hs4 + ((i * MC + m) * 8) * 8 + s8;
                        float2 acc2 = make_float2(0.f, 0.f);
                        const uint32_t cw[4] = {U.c[t].x, U.c[t].y, U.c[t].z, U.c[t].w};
#pragma unroll
                        for (int wq = 0; wq < 4; ++wq) dot8(cw[wq], hv[(2 * wq) * 8], hv[(2 * wq + 1) * 8], acc2);
                        acc += U.s[t] * (acc2.x + acc2.y) + (U.b[t] - 128.f * U.s[t]) * hc[(i * MC + m) * 8 + s8];
                    }
                }
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (live && s8 == 0) {
            os[i * R + dl] = acc;
            if (a.expert_out) a.expert_out[(size_t)i * D + d0 + dl] = acc;
        }
    }
    __syncthreads();
    for (int dl = tid; dl < rows; dl += kThreads) {
        float y = bf16_to_f32(a.x[d0 + dl]);
        for (int i = 0; i < K; ++i) y = fmaf(wsel[i], os[i * R + dl], y);
        a.y[d0 + dl] = f32_to_bf16(y);
    }
}

}  // namespace

// SM count of the current device (cached per device; a failed query is not cached).
int device_sm_count() {
    static std::atomic<int> cached[kMaxCachedDevices];
    const int d = cache_slot();
    if (d >= 0) {
        const int c = cached[d].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 1;
    if (d >= 0) cached[d].store(n, std::memory_order_relaxed);
    return n;
}

size_t decode_gateup_smem(int D) {
    const int NGP = (D / kGroup + 31) / 32;
    return (size_t)NGP * 2048 * sizeof(float) + (size_t)NGP * 32 * sizeof(float);
}

size_t decode_down_smem(int D, int F, int K) {
    const int MC = (F / 32 + 7) / 8;
    return ((size_t)K * MC * 256 + (size_t)K * MC * 8 + (size_t)K * down_rows_per_cta(D)) * sizeof(float);
}

cudaError_t launch_decode_gateup(const DecodeArgs &a, cudaStream_t s, bool pdl) {
    static SmemLimits limits;
    const size_t smem = decode_gateup_smem(a.D);
    const cudaError_t e = allow_dynamic_smem(k_decode_gateup, limits, 64 * 1024);
    if (e != cudaSuccess) return e;
    const int P = a.K * a.F;
    int grid = device_sm_count() * 2;
    if (grid > P) grid = P;
    return launch_kernel(k_decode_gateup, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

cudaError_t launch_decode_down(const DecodeArgs &a, cudaStream_t s, bool pdl) {
    static SmemLimits limits;
    const size_t smem = decode_down_smem(a.D, a.F, a.K);
    const cudaError_t e = allow_dynamic_smem(k_decode_down, limits, 200 * 1024);
    if (e != cudaSuccess) return e;
    const int R = down_rows_per_cta(a.D);
    return launch_kernel(k_decode_down, dim3((a.D + R - 1) / R), dim3(kThreads), smem, s, pdl, a);
}

}  // namespace smoe

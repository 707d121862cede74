// decode_fused.cu -- one batch-1 decode layer as one persistent kernel:
// RMSNorm + router gate + top-k, gate/up, down + weighted residual sum.
//
// "Optimizations" page: "Routing Is Exact" (gate on the true hidden state,
// top-8, norm_topk_prob weights), "Coalesced GPU Kernels -- Expert FFN and
// Dense Matvec" (gate+up in one pass, per-chunk affine dequant, FMA inner
// loop), "The Dense Ceiling -- GPU-Resident Epilogue" (residual, norm and gate
// stay on the GPU); "System Overview", per-token table, Metal Kernel row
// (weighted sum into the residual).
//
// At batch 1 a layer is a chain of three dependent steps (route -> gate/up ->
// down) over ~22 MB (30B shape) to ~86 MB (235B shape) of weights, i.e. a few
// microseconds of HBM time, so the cost is latency.  One CTA per SM runs the
// whole layer with two grid-wide barriers (device-scope counter and
// generation word, bounded spin):
//   phase 0  CTA c < E loads router row c before it waits for the previous
//            kernel (programmatic dependent launch), then normalises x (all
//            CTAs, fp32, the same arithmetic as the stand-alone router) and
//            writes logit c;                                     -- barrier 1
//   phase 1  every CTA ranks the E logits itself (no second launch), and a
//            producer warp streams this CTA's gate/up rows AND its down rows
//            with bulk async copies (cp.async.bulk, the TMA engine) into a
//            ring of shared-memory slots; 8 compute warps turn gate/up rows
//            into h = SiLU(g)*u (fp32, to global);                -- barrier 2
//   phase 2  down rows (already resident in shared memory) times h, combined
//            in rank order with the residual: y = x + sum_i w_i o_i.
// The per-row arithmetic is that of decode.cu: a code q becomes the float
// 128+q by one byte permute; per 32-code chunk s*sum((128+q)x) + (b-128s)*sum(x).
//
// Every wait (mbarrier or grid barrier) is bounded; on timeout the kernel
// records SMOE_ERR_TIMEOUT in the status word and runs to completion.
#include "common.cuh"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kCompute = 256;          // warps 0-7
constexpr int kThreadsF = kCompute + 32;   // + producer warp 8
constexpr int kSlots = 3;

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Named barrier of the 256 compute threads.  The non-aligned form: lanes of a
// warp may arrive from divergent paths (e.g. thread 0 leaving a spin).
__device__ __forceinline__ void bar_compute() { asm volatile("barrier.sync 1, %0;" ::"n"(kCompute) : "memory"); }

__device__ __forceinline__ void mb_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mb_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 s; mbarrier.arrive.shared::cta.b64 s, [%0]; }" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 s; mbarrier.arrive.expect_tx.shared::cta.b64 s, [%0], %1; }" ::"r"(su32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t *b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    return ok;
}
// Wait for the phase of parity `par`, bounded in wall time.
__device__ __forceinline__ bool mb_wait(uint64_t *b, uint32_t par, int32_t *status) {
    if (mb_try(b, par)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mb_try(b, par)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    set_status(status, SMOE_ERR_TIMEOUT);
    return false;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (sizes, addresses: 16-byte multiples)
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier for the compute warps of every CTA (all CTAs resident:
// one per SM).  bar[0] counts arrivals, bar[1] is the generation.
__device__ __forceinline__ void grid_sync(uint32_t *bar, int32_t *status) {
    bar_compute();
    if (threadIdx.x == 0) {
        const uint32_t gen = ld_acquire_u32(bar + 1);
        __threadfence();
        const uint32_t prev = atomicAdd(bar, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u32(bar + 1) == gen) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    set_status(status, SMOE_ERR_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
    }
    __syncwarp();
    bar_compute();
}

__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 0u;
    v = v + 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- work lists

// Gate/up: CTA c owns row pairs [P*c/G, P*(c+1)/G) of the K*F (slot, row) pairs;
// an item is up to R consecutive rows of one expert slot.
struct GuIt {
    int i, j0, n;   // expert slot, first row, rows
};
__device__ __forceinline__ bool gu_item(const FusedArgs &a, int idx, GuIt &it) {
    const long long P = (long long)a.K * a.F;
    int p = (int)(P * blockIdx.x / gridDim.x);
    const int p1 = (int)(P * (blockIdx.x + 1) / gridDim.x);
    for (int k = 0; p < p1; ++k) {
        const int i = p / a.F, j = p - i * a.F;
        int n = min(a.r_gu, min(p1 - p, a.F - j));
        if (k == idx) {
            it = {i, j, n};
            return true;
        }
        p += n;
    }
    return false;
}

// Down: CTA c owns output rows [d0, d1) (multiples of a.dn_gran); an item is
// up to a.e_dn consecutive expert slots of those rows.
__device__ __forceinline__ void dn_rows(const FusedArgs &a, int &d0, int &d1) {
    const int units = a.D / a.dn_gran;
    d0 = (int)((long long)units * blockIdx.x / gridDim.x) * a.dn_gran;
    d1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x) * a.dn_gran;
}

// ---------------------------------------------------------------- kernel

template <bool kRoute>
__global__ void __launch_bounds__(kThreadsF, 1) k_decode_layer(FusedArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    const int D = a.D, F = a.F, K = a.K, E = a.E;
    const int NC = D / 32;                       // 32-code chunks of a gate/up row
    const int NCP = (NC + 63) / 64;              // passes of 64 chunks (2 per lane)
    const int FC = F / 32;                       // chunks of a down row
    const int MC = (FC + 7) / 8;                 // chunks per lane of an 8-lane subgroup
    unsigned char *ring = sm;
    float *u_region = reinterpret_cast<float *>(sm + a.ring_bytes);       // xs+xc | hs+hc
    float *xs = u_region;                        // NCP*64*8 float4 = NCP*2048 floats
    float *xc = xs + NCP * 2048;                 // NCP*64 chunk sums
    float *hs = u_region;                        // K*MC*64 float4 = K*MC*256 floats
    float *hc = hs + K * MC * 256;               // K*MC*8
    uint16_t *xraw = reinterpret_cast<uint16_t *>(sm + a.ring_bytes + a.union_bytes);   // [D]
    float *os = reinterpret_cast<float *>(xraw + D);                                 // [K][rows_max]
    __shared__ uint64_t full[kSlots], empty[kSlots], idx_ready;
    __shared__ float red[8];
    __shared__ uint32_t keys[kMaxExperts];
    __shared__ float lsel[kMaxTopK], wsel[kMaxTopK];
    __shared__ int isel[kMaxTopK], ivalid[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mb_init(&full[s], 1);
            mb_init(&empty[s], 8);      // one arrival per compute warp
        }
        mb_init(&idx_ready, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int d0, d1;
    dn_rows(a, d0, d1);
    const int rows = d1 - d0;

    if (warp == 8) {
        // ================= producer: bulk copies into the ring =================
        if (lane == 0) {
            if (!mb_wait(&idx_ready, 0, a.status)) return;
            uint32_t g = 0;
            auto acquire = [&](uint32_t &s) -> unsigned char * {
                s = g % kSlots;
                mb_wait(&empty[s], ((g / kSlots) & 1) ^ 1, a.status);
                ++g;
                return ring + s * a.slot_bytes;
            };
            const int NG = D / kGroup;
            GuIt it;
            for (int k = 0; gu_item(a, k, it); ++k) {
                uint32_t s;
                unsigned char *dst = acquire(s);
                const int e = isel[it.i];
                const size_t row = (size_t)e * F + it.j0;
                const uint32_t cb = it.n * (D / 2), sb = it.n * NG * 2;
                mb_expect(&full[s], 2 * cb + 4 * sb);
                bulk_g2s(dst, a.gq + row * (D / 2), cb, &full[s]);
                bulk_g2s(dst + cb, a.uq + row * (D / 2), cb, &full[s]);
                bulk_g2s(dst + 2 * cb, a.gs + row * NG, sb, &full[s]);
                bulk_g2s(dst + 2 * cb + sb, a.gb + row * NG, sb, &full[s]);
                bulk_g2s(dst + 2 * cb + 2 * sb, a.us + row * NG, sb, &full[s]);
                bulk_g2s(dst + 2 * cb + 3 * sb, a.ub + row * NG, sb, &full[s]);
            }
            if (rows > 0) {
                const int FG = F / kGroup;
                for (int i0 = 0; i0 < K; i0 += a.e_dn) {
                    const int ne = min(a.e_dn, K - i0);
                    uint32_t s;
                    unsigned char *dst = acquire(s);
                    const uint32_t cb = rows * (F / 2), sb = rows * FG * 2;
                    mb_expect(&full[s], ne * (cb + 2 * sb));
                    for (int q = 0; q < ne; ++q) {
                        const size_t row = (size_t)isel[i0 + q] * D + d0;
                        bulk_g2s(dst + q * cb, a.dq + row * (F / 2), cb, &full[s]);
                        bulk_g2s(dst + ne * cb + q * 2 * sb, a.ds + row * FG, sb, &full[s]);
                        bulk_g2s(dst + ne * cb + q * 2 * sb + sb, a.db + row * FG, sb, &full[s]);
                    }
                }
            }
            // every copy issued has landed before the CTA may exit
            for (uint32_t k = (g > (uint32_t)kSlots ? g - kSlots : 0); k < g; ++k)
                mb_wait(&full[k % kSlots], (k / kSlots) & 1, a.status);
        }
        return;
    }

    // ================= compute warps =================
    // router row of this CTA: load before waiting on the previous kernel
    uint4 rw[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    const bool has_row = kRoute && (int)blockIdx.x < E;
    if (has_row) {
        const uint16_t *wr = a.router_w + (size_t)blockIdx.x * D;
        for (int q = 0; q < 2; ++q) {
            const int d = (tid + q * kCompute) * 8;
            if (d < D) rw[q] = ld_stream16(wr + d);
        }
    }

    pdl_wait();
    pdl_launch_dependents();

    // ---- normalise x: each thread owns 8 consecutive elements per pass ----
    float xv[2][8];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int d = (tid + q * kCompute) * 8;
        if (d < D) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(a.x + d));
            *reinterpret_cast<uint4 *>(xraw + d) = v;
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                xv[q][2 * k] = __uint_as_float(w4[k] << 16);
                xv[q][2 * k + 1] = __uint_as_float(w4[k] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) xv[q][k] = 0.f;
        }
    }
    bar_compute();   // xraw complete before threads read each other's elements
    if (a.gain) {
        // same reduction order as block_rms_inv (stride-256 scalar partials, warp tree, 8 warps in order)
        for (int d = tid; d < D; d += kCompute) {
            const float v = bf16_to_f32(xraw[d]);
            ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        bar_compute();
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += red[i];
        const float inv = 1.0f / sqrtf(t / (float)D + a.eps);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int d = (tid + q * kCompute) * 8;
            if (d < D) {
                const uint4 gv = *reinterpret_cast<const uint4 *>(a.gain + d);
                const uint16_t *gg = reinterpret_cast<const uint16_t *>(&gv);
#pragma unroll
                for (int k = 0; k < 8; ++k) xv[q][k] = bf16_to_f32(rms_apply(xraw[d + k], inv, gg[k]));
            }
        }
    }
    // stage xn (fp32) lane-interleaved for the gate/up sweep: chunk c (32 values)
    // = pass*64 + half*32 + l sits at float4 ((pass*2+half)*8 + k)*32 + l.
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int d = (tid + q * kCompute) * 8;
        if (d < D) {
            const int c = d >> 5, k0 = (d & 31) >> 2;   // chunk, first float4 within it
            const int pass = c >> 6, hl = (c >> 5) & 1, l = c & 31;
            float4 *dst = reinterpret_cast<float4 *>(xs) + ((pass * 2 + hl) * 8 + k0) * 32 + l;
            dst[0] = make_float4(xv[q][0], xv[q][1], xv[q][2], xv[q][3]);
            dst[32] = make_float4(xv[q][4], xv[q][5], xv[q][6], xv[q][7]);
            float s8 = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) s8 += xv[q][k];
            // 4 consecutive threads hold one 32-element chunk
            s8 += __shfl_xor_sync(0xffffffffu, s8, 1);
            s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
            if ((tid & 3) == 0) xc[c] = s8;
        }
    }
    // chunks past D (D not a multiple of 2048) read as zero
    for (int c = NC + tid; c < NCP * 64; c += kCompute) {
        const int pass = c >> 6, hl = (c >> 5) & 1, l = c & 31;
        for (int k = 0; k < 8; ++k)
            reinterpret_cast<float4 *>(xs)[((pass * 2 + hl) * 8 + k) * 32 + l] = make_float4(0.f, 0.f, 0.f, 0.f);
        xc[c] = 0.f;
    }

    // ---- phase 0: router logit of this CTA, then every CTA ranks all of them ----
    if (kRoute) {
        if (has_row) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint32_t w4[4] = {rw[q].x, rw[q].y, rw[q].z, rw[q].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc = fmaf(__uint_as_float(w4[k] << 16), xv[q][2 * k], acc);
                    acc = fmaf(__uint_as_float(w4[k] & 0xFFFF0000u), xv[q][2 * k + 1], acc);
                }
            }
            acc = warp_sum(acc);
            bar_compute();
            if (lane == 0) red[warp] = acc;
            bar_compute();
            if (tid == 0) {
                float t = 0.f;
                for (int i = 0; i < 8; ++i) t += red[i];
                a.logits[blockIdx.x] = t;
            }
        }
        grid_sync(a.bar, a.status);
        float my = -INFINITY;
        if (tid < E) {
            my = __ldcg(a.logits + tid);
            keys[tid] = order_key(my);
        }
        bar_compute();
        if (tid < E) {
            const uint32_t k0 = keys[tid];
            int rank = 0;
            for (int j = 0; j < E; ++j) {
                const uint32_t kj = keys[j];
                rank += (kj > k0) | ((kj == k0) & (j < tid));
            }
            if (rank < K) {
                isel[rank] = tid;
                lsel[rank] = my;
            }
        }
        bar_compute();
        const float m = lsel[0];
        float denom = 0.f;
        if (a.norm_topk_prob) {
            for (int i = 0; i < K; ++i) denom += expf(lsel[i] - m);
        } else {
            float pz = (tid < E) ? expf(my - m) : 0.f;
            pz = warp_sum(pz);
            bar_compute();
            if (lane == 0) red[warp] = pz;
            bar_compute();
            for (int i = 0; i < 8; ++i) denom += red[i];
        }
        if (tid < K) {
            wsel[tid] = expf(lsel[tid] - m) / denom;
            if (blockIdx.x == 0) {
                a.idx_out[tid] = isel[tid];
                a.w_out[tid] = wsel[tid];
            }
        }
    } else {
        if (tid < K) {
            int e = a.idx_in[tid];
            if (e < 0 || e >= E) {
                set_status(a.status, SMOE_ERR_DEVICE);
                e = -1;
            }
            isel[tid] = e;
            wsel[tid] = a.w_in[tid];
        }
    }
    // an id that cannot be used contributes nothing (the ring still streams a
    // harmless copy of expert 0, so producer and consumers stay in step)
    bar_compute();
    if (tid < K) {
        ivalid[tid] = (isel[tid] >= 0 && isel[tid] < E);
        if (!ivalid[tid]) {
            isel[tid] = 0;
            wsel[tid] = 0.f;
        }
    }
    bar_compute();
    if (tid == 0) mb_arrive(&idx_ready);

    // ---- phase 1: gate/up rows -> h ----
    uint32_t g = 0;
    {
        const int NG = D / kGroup;
        const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
        GuIt it;
        for (int k = 0; gu_item(a, k, it); ++k, ++g) {
            const uint32_t s = g % kSlots;
            mb_wait(&full[s], (g / kSlots) & 1, a.status);
            const unsigned char *slot = ring + s * a.slot_bytes;
            const uint32_t cb = it.n * (D / 2), sb = it.n * NG * 2;
            const uint16_t *gsr = reinterpret_cast<const uint16_t *>(slot + 2 * cb);
            const uint16_t *gbr = gsr + it.n * NG, *usr = gbr + it.n * NG, *ubr = usr + it.n * NG;
            for (int r0 = warp; r0 < it.n; r0 += 16) {
                const int r1 = r0 + 8;
                const bool two = r1 < it.n;
                float ag0 = 0.f, au0 = 0.f, ag1 = 0.f, au1 = 0.f;
                for (int pass = 0; pass < NCP; ++pass) {
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl) {
                        const int c = pass * 64 + hl * 32 + lane;
                        if (c >= NC) continue;
                        float4 xq[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) xq[k] = xs4[((pass * 2 + hl) * 8 + k) * 32 + lane];
                        const float X = xc[c];
                        const int gi = c >> 1;
                        {
                            const uint4 cg = *reinterpret_cast<const uint4 *>(slot + r0 * (D / 2) + c * 16);
                            const uint4 cu = *reinterpret_cast<const uint4 *>(slot + cb + r0 * (D / 2) + c * 16);
                            float2 A = make_float2(0.f, 0.f), B = make_float2(0.f, 0.f);
                            dot8(cg.x, xq[0], xq[1], A); dot8(cg.y, xq[2], xq[3], A);
                            dot8(cg.z, xq[4], xq[5], A); dot8(cg.w, xq[6], xq[7], A);
                            dot8(cu.x, xq[0], xq[1], B); dot8(cu.y, xq[2], xq[3], B);
                            dot8(cu.z, xq[4], xq[5], B); dot8(cu.w, xq[6], xq[7], B);
                            const float s0 = bf16_to_f32(gsr[r0 * NG + gi]), b0 = bf16_to_f32(gbr[r0 * NG + gi]);
                            const float s1 = bf16_to_f32(usr[r0 * NG + gi]), b1 = bf16_to_f32(ubr[r0 * NG + gi]);
                            ag0 += s0 * (A.x + A.y) + (b0 - 128.f * s0) * X;
                            au0 += s1 * (B.x + B.y) + (b1 - 128.f * s1) * X;
                        }
                        if (two) {
                            const uint4 cg = *reinterpret_cast<const uint4 *>(slot + r1 * (D / 2) + c * 16);
                            const uint4 cu = *reinterpret_cast<const uint4 *>(slot + cb + r1 * (D / 2) + c * 16);
                            float2 A = make_float2(0.f, 0.f), B = make_float2(0.f, 0.f);
                            dot8(cg.x, xq[0], xq[1], A); dot8(cg.y, xq[2], xq[3], A);
                            dot8(cg.z, xq[4], xq[5], A); dot8(cg.w, xq[6], xq[7], A);
                            dot8(cu.x, xq[0], xq[1], B); dot8(cu.y, xq[2], xq[3], B);
                            dot8(cu.z, xq[4], xq[5], B); dot8(cu.w, xq[6], xq[7], B);
                            const float s0 = bf16_to_f32(gsr[r1 * NG + gi]), b0 = bf16_to_f32(gbr[r1 * NG + gi]);
                            const float s1 = bf16_to_f32(usr[r1 * NG + gi]), b1 = bf16_to_f32(ubr[r1 * NG + gi]);
                            ag1 += s0 * (A.x + A.y) + (b0 - 128.f * s0) * X;
                            au1 += s1 * (B.x + B.y) + (b1 - 128.f * s1) * X;
                        }
                    }
                }
                ag0 = warp_sum(ag0); au0 = warp_sum(au0);
                ag1 = warp_sum(ag1); au1 = warp_sum(au1);
                if (lane == 0) {
                    const bool ok = ivalid[it.i];
                    a.h[(size_t)it.i * F + it.j0 + r0] = ok ? silu_mul(ag0, au0) : 0.f;
                    if (two) a.h[(size_t)it.i * F + it.j0 + r1] = ok ? silu_mul(ag1, au1) : 0.f;
                }
            }
            __syncwarp();
            if (lane == 0) mb_arrive(&empty[s]);
        }
    }

    // ---- barrier 2: all of h written ----
    __threadfence();
    grid_sync(a.bar, a.status);

    // ---- stage h (fp32, lane-interleaved for 8-lane subgroups) and chunk sums ----
    for (int q = tid; q < K * MC * 64; q += kCompute) {
        const int i = q / (MC * 64), rem = q - i * MC * 64;
        const int m = rem / 64, k = (rem / 8) & 7, cs = rem & 7;
        const int c = cs + 8 * m;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < FC) v = __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)i * F + c * 32 + k * 4));
        reinterpret_cast<float4 *>(hs)[q] = v;
    }
    bar_compute();
    for (int q = tid; q < K * MC * 8; q += kCompute) {
        const int i = q / (MC * 8), c = q - i * MC * 8;
        const int m = c / 8, cs = c & 7;
        const float4 *hp = reinterpret_cast<const float4 *>(hs) + ((i * MC + m) * 8) * 8 + cs;
        float sacc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = hp[k * 8];
            sacc += (v.x + v.y) + (v.z + v.w);
        }
        hc[q] = sacc;
    }
    bar_compute();

    // ---- phase 2: down rows of this CTA (8-lane subgroup per (expert, row)) ----
    const int s8 = lane & 7, S = warp * 4 + (lane >> 3);
    const float4 *hs4 = reinterpret_cast<const float4 *>(hs);
    const int FG = F / kGroup;
    if (rows > 0) {
        for (int i0 = 0; i0 < K; i0 += a.e_dn, ++g) {
            const int ne = min(a.e_dn, K - i0);
            const uint32_t s = g % kSlots;
            mb_wait(&full[s], (g / kSlots) & 1, a.status);
            const unsigned char *slot = ring + s * a.slot_bytes;
            const uint32_t cb = rows * (F / 2), sb = rows * FG * 2;
            // warp-uniform trip count: every lane reaches the shuffles below
            for (int base = warp * 4; base < ne * rows; base += 32) {
                const int q = base + (S - warp * 4);
                const bool live = q < ne * rows;
                const int qi = live ? q / rows : 0, r = live ? q - qi * rows : 0, i = i0 + qi;
                const unsigned char *rp = slot + qi * cb + r * (F / 2);
                const uint16_t *sr = reinterpret_cast<const uint16_t *>(slot + ne * cb + qi * 2 * sb) + r * FG;
                const uint16_t *br = sr + rows * FG;
                float acc = 0.f;
                for (int m = 0; m < MC && live; ++m) {
                    const int c = s8 + 8 * m;
                    if (c >= FC) break;
                    const uint4 cv = *reinterpret_cast<const uint4 *>(rp + c * 16);
                    const float4 *hv = hs4 + ((i * MC + m) * 8) * 8 + s8;
                    float2 A = make_float2(0.f, 0.f);
                    dot8(cv.x, hv[0], hv[8], A);
                    dot8(cv.y, hv[16], hv[24], A);
                    dot8(cv.z, hv[32], hv[40], A);
                    dot8(cv.w, hv[48], hv[56], A);
                    const float sc = bf16_to_f32(sr[c >> 1]), bi = bf16_to_f32(br[c >> 1]);
                    acc += sc * (A.x + A.y) + (bi - 128.f * sc) * hc[(i * MC + m) * 8 + s8];
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                if (live && s8 == 0) os[i * a.rows_max + r] = acc;
            }
            __syncwarp();
            if (lane == 0) mb_arrive(&empty[s]);
        }
    }
    bar_compute();
    for (int r = tid; r < rows; r += kCompute) {
        float y = bf16_to_f32(xraw[d0 + r]);
        for (int i = 0; i < K; ++i) {
            const float o = os[i * a.rows_max + r];
            y = fmaf(wsel[i], o, y);
            if (a.expert_out) a.expert_out[(size_t)i * D + d0 + r] = o;
        }
        a.y[d0 + r] = f32_to_bf16(y);
    }
}

}  // namespace

// Host: shape support, work partition and shared-memory plan of the fused layer kernel.
bool fused_plan(FusedArgs &a, int num_sms) {
    const int D = a.D, F = a.F, K = a.K;
    if (D % 512 || F % 128 || D > 4096 || K > kMaxTopK) return false;
    // bulk copies need 16-byte aligned sources
    const void *ptrs[] = {a.gq, a.uq, a.dq, a.gs, a.gb, a.us, a.ub, a.ds, a.db, a.x};
    for (const void *q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) % 16) return false;
    if (a.gain && reinterpret_cast<uintptr_t>(a.gain) % 16) return false;
    a.grid = num_sms;
    if (a.E > a.grid) return false;
    const int NG = D / kGroup, FG = F / kGroup;
    // down rows: units of dn_gran rows whose scale block starts 16-byte aligned
    int gran = 1;
    while ((gran * (F / 32)) % 16) ++gran;
    a.dn_gran = gran;
    const int units = D / gran;
    a.rows_max = ((units + a.grid - 1) / a.grid) * gran;
    const int row_pair_bytes = 2 * (D / 2 + NG * 2 * 2);
    const int dn_bytes_1 = a.rows_max * (F / 2 + FG * 2 * 2);
    // slots: gate/up items of r_gu rows, down items of e_dn experts
    const int target = D >= 4096 ? 36 * 1024 : 20 * 1024;
    a.r_gu = target / row_pair_bytes;
    if (a.r_gu < 1) a.r_gu = 1;
    if (a.r_gu > 16) a.r_gu = 16;
    a.e_dn = (a.r_gu * row_pair_bytes) / dn_bytes_1;
    if (a.e_dn < 1) a.e_dn = 1;
    if (a.e_dn > K) a.e_dn = K;
    a.slot_bytes = max(a.r_gu * row_pair_bytes, a.e_dn * dn_bytes_1);
    a.slot_bytes = (a.slot_bytes + 127) / 128 * 128;
    a.ring_bytes = kSlots * a.slot_bytes;
    const int NCP = (D / 32 + 63) / 64, MC = (F / 32 + 7) / 8;
    const int xs_bytes = (NCP * 2048 + NCP * 64) * 4;
    const int hs_bytes = (K * MC * 256 + K * MC * 8) * 4;
    a.union_bytes = (max(xs_bytes, hs_bytes) + 127) / 128 * 128;
    a.smem_bytes = a.ring_bytes + a.union_bytes + D * 2 + K * a.rows_max * 4;
    return a.smem_bytes <= 200 * 1024;
}

cudaError_t launch_decode_layer(const FusedArgs &a, cudaStream_t s, bool route) {
    static int attr[2] = {0, 0};
    const size_t smem = a.smem_bytes;
    if (route) {
        if (attr[1] < (int)smem) {
            cudaError_t e = cudaFuncSetAttribute(k_decode_layer<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            attr[1] = (int)smem;
        }
        return launch_kernel(k_decode_layer<true>, dim3(a.grid), dim3(kThreadsF), smem, s, true, a);
    }
    if (attr[0] < (int)smem) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_layer<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr[0] = (int)smem;
    }
    return launch_kernel(k_decode_layer<false>, dim3(a.grid), dim3(kThreadsF), smem, s, true, a);
}

}  // namespace smoe

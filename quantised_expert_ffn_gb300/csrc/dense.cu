// dense.cu -- the dense bf16 matrix-vector product and the SMOE-Q4 quantiser.
//
// Matvec: "Optimizations" page, "Coalesced GPU Kernels -- Expert FFN and
// Dense Matvec": the bf16 dense matvec twin of the expert kernels, which
// carries decode's QKV/O projections and the LM head.  y[r] = sum_c W[r][c] x[c]
// with W bf16 [rows][cols], x bf16 [cols], fp32 products and sums.  It reads
// 2 bytes per weight once, so HBM bandwidth bounds it; the design keeps
// enough 16-byte loads in flight on every SM:
//   * CTA = 8 warps; warp w owns the w-th eighth of the 16-byte chunks of
//     every row, lane l the chunks c0 + l + 32 j of that eighth -- a warp's
//     loads of one row are 512 consecutive bytes, and the lane's x values stay
//     in registers for the CTA's whole life (in shared memory for rows of
//     more than 4096, where registers hold the loads instead; cols <= 8192);
//   * four CTAs per SM; CTA b owns the contiguous rows [R b / G, R (b+1) / G)
//     (balanced to one row) and takes RB of them at a time (RB * CPL loads in
//     flight per lane); small row counts use RB = 1 and one row per CTA so
//     that every SM gets rows (the 512-row K/V projection shapes the page
//     names);
//   * per row: packed fp32 FMAs (two partial sums per lane), a warp tree, then
//     the 8 warp sums in warp order from shared memory (double-buffered, one
//     barrier per row block);
//   * launched as a programmatic dependent launch: the first step's weights
//     are requested before the kernel waits for the previous one in the
//     stream (only x can depend on it), so back-to-back calls (decode's
//     projections) overlap a launch and its first DRAM latency with the
//     previous kernel's tail.
//
// Quantiser: the offline step that turns bf16 expert weights into the Q4
// layout ("System Overview", "The Four-Component Architecture": the Sculptor's
// "aggressively quantised" vault blocks).  Per group of 64 consecutive weights
// of a row: mn, mx = least and greatest weight; scale = bf16 nearest-even of
// ((mx - mn) + 0) / 15; bias = mn + 0; q = the integer nearest (halves to
// even) to RN(w - mn) * RN(1 / scale), the product exact (0 where scale is 0).
// Reading 2 bytes and writing 0.5625 per weight, it is HBM-bound once the
// per-weight work is a few instructions: one lane per group, min/max on bf16
// pairs, one packed subtract and one packed fused multiply-add per two
// weights, one shift-add per code.
#include "common.cuh"
#include "dense.h"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kMvWarps = 8;
constexpr int kMvThreads = kMvWarps * 32;
constexpr int kMvCtasPerSm = 4;

// lo/hi bf16 of a 32-bit word as two floats (element 2k, 2k+1)
__device__ __forceinline__ float2 bf16x2_f32(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// XS: x stays in shared memory (bf16) instead of registers, for CPL = 4,
// where registers would not hold both x and every load of a step.
template <int RB, int CPL, bool XS>
__global__ void __launch_bounds__(kMvThreads, kMvCtasPerSm)
    k_dense_matvec(const uint16_t *__restrict__ w, const uint16_t *__restrict__ x, int rows, int cols,
                   float *__restrict__ y) {
    __shared__ float part[2][RB][kMvWarps];
    __shared__ uint4 xsm[XS ? 1024 : 1];                      // x as bf16, cols <= 8192
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int NC = cols >> 3;                                 // 16-byte chunks per row
    const int c0 = NC * warp / kMvWarps, c1 = NC * (warp + 1) / kMvWarps;
    // CTA b owns rows [rows*b/G, rows*(b+1)/G), taken RB at a time
    const int r_beg = (int)((long long)rows * blockIdx.x / gridDim.x);
    const int r_end = (int)((long long)rows * (blockIdx.x + 1) / gridDim.x);
    uint4 wv[RB][CPL];
    auto load_step = [&](int r0) {
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int c = c0 + lane + 32 * j;
                wv[r][j] = (c < c1 && r0 + r < r_end)
                               ? ld_stream16(w + (size_t)(r0 + r) * cols + 8 * (size_t)c)
                               : make_uint4(0, 0, 0, 0);
            }
    };
    // Launched as a programmatic dependent: the weights (constant inputs) of
    // the first step are requested while the previous kernel in the stream may
    // still run; x, which that kernel may produce, and y only after it is done.
    // (Not with x in shared memory: there the early loads would stay live
    // across the staging of x and spill.)
    if (!XS) load_step(r_beg);
    pdl_wait();
    pdl_launch_dependents();
    float2 xr[XS ? 1 : CPL][4];
    if (XS) {
        for (int c = threadIdx.x; c < NC; c += kMvThreads) xsm[c] = __ldg(reinterpret_cast<const uint4 *>(x) + c);
        __syncthreads();
    } else {
#pragma unroll
        for (int j = 0; j < (XS ? 1 : CPL); ++j) {
            const int c = c0 + lane + 32 * j;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (c < c1) v = __ldg(reinterpret_cast<const uint4 *>(x) + c);
            xr[j][0] = bf16x2_f32(v.x);
            xr[j][1] = bf16x2_f32(v.y);
            xr[j][2] = bf16x2_f32(v.z);
            xr[j][3] = bf16x2_f32(v.w);
        }
    }
    int buf = 0;
    for (int r0 = r_beg; r0 < r_end; r0 += RB) {
        if (XS || r0 != r_beg) load_step(r0);
        float acc[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float2 xj[4];
                if (XS) {
                    const int c = c0 + lane + 32 * j;
                    const uint4 v = c < c1 ? xsm[c] : make_uint4(0, 0, 0, 0);
                    xj[0] = bf16x2_f32(v.x);
                    xj[1] = bf16x2_f32(v.y);
                    xj[2] = bf16x2_f32(v.z);
                    xj[3] = bf16x2_f32(v.w);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) xj[k] = xr[XS ? 0 : j][k];
                }
                a2 = ffma2(bf16x2_f32(wv[r][j].x), xj[0], a2);
                a2 = ffma2(bf16x2_f32(wv[r][j].y), xj[1], a2);
                a2 = ffma2(bf16x2_f32(wv[r][j].z), xj[2], a2);
                a2 = ffma2(bf16x2_f32(wv[r][j].w), xj[3], a2);
            }
            acc[r] = warp_sum(a2.x + a2.y);
        }
        if (lane == 0)
#pragma unroll
            for (int r = 0; r < RB; ++r) part[buf][r][warp] = acc[r];
        __syncthreads();
        if (threadIdx.x < RB && r0 + (int)threadIdx.x < r_end) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < kMvWarps; ++i) s += part[buf][threadIdx.x][i];
            y[r0 + threadIdx.x] = s;
        }
        buf ^= 1;
    }
}

template <int RB, int CPL, bool XS = false>
cudaError_t launch_mv(const uint16_t *w, const uint16_t *x, int rows, int cols, float *y, int grid_cap,
                      cudaStream_t s) {
    const int grid = rows < grid_cap ? rows : grid_cap;
    return launch_kernel(k_dense_matvec<RB, CPL, XS>, dim3(grid), dim3(kMvThreads), 0, s, true, w, x, rows, cols,
                         y);
}

template <int RB>
cudaError_t launch_mv_rb(const uint16_t *w, const uint16_t *x, int rows, int cols, float *y, int grid_cap,
                         cudaStream_t s) {
    const int per_warp = ((cols >> 3) + kMvWarps - 1) / kMvWarps;   // chunks of one warp's eighth
    if (per_warp <= 32) return launch_mv<RB, 1>(w, x, rows, cols, y, grid_cap, s);
    if (per_warp <= 64) return launch_mv<RB, 2>(w, x, rows, cols, y, grid_cap, s);
    return launch_mv<(RB > 2 ? 2 : RB), 4, true>(w, x, rows, cols, y, grid_cap, s);
}

// ---------------------------------------------------------------- quantiser

constexpr int kQWarps = 4;
constexpr int kQThreads = kQWarps * 32;
constexpr int kQCtasPerSm = 4;
constexpr int kQStages = 3;                              // 4 KiB stages per warp

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes = 0 fills
// the 16 bytes with zeros without reading.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    unsigned long long ra = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long rb = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long rd;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    return *reinterpret_cast<float2 *>(&rd);
}

// The codes (kBits = 4: SMOE-Q4, 2: SMOE-Q2) of one group of 64 weights (32
// bf16 pairs in u), its scale and bias.  Code q = the integer nearest (halves
// to even) to d * r, d = RN(w - mn), r = RN(1 / scale), the product exact: one
// fused multiply-add d * r + 2^23 rounds it once, onto the integers, leaving
// 0x4B000000 + q as its bits.  The n = 32 / kBits such words e_k of a code
// word combine into sum_k q_k 2^(kBits k) as (sum_k e_k 2^(kBits k)) minus
// 0x4B000000 * sum_k 2^(kBits k) (mod 2^32), one shift-add each.
template <int kBits>
__device__ __forceinline__ void q_group(const uint32_t (&u)[32], uint32_t (&code)[2 * kBits], uint16_t &sb,
                                        uint16_t &bb) {
    constexpr int kWords = 2 * kBits, kPairs = 16 / kBits;  // code words; bf16 pairs per code word
    constexpr uint32_t kPackBias = kBits == 4 ? 0xFB000000u : 0xE7000000u;   // 0x4B000000 * 0x11111111 / 0x55555555
    constexpr float kLevels = (float)((1 << kBits) - 1);
    uint32_t mn2 = u[0], mx2 = u[0];
#pragma unroll
    for (int k = 1; k < 32; ++k) {
        mn2 = bf16x2_min(mn2, u[k]);
        mx2 = bf16x2_max(mx2, u[k]);
    }
    const float mn = fminf(__uint_as_float(mn2 << 16), __uint_as_float(mn2 & 0xFFFF0000u));
    const float mx = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
    sb = f32_to_bf16(__fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), kLevels));
    bb = f32_to_bf16(__fadd_rn(mn, 0.0f));
    const float s = bf16_to_f32(sb);
    if (s == 0.0f) {
#pragma unroll
        for (int k = 0; k < kWords; ++k) code[k] = 0u;
        return;
    }
    if (s >= 0x1p-126f) {
        const float r = __frcp_rn(s);
        const float2 mn_2 = make_float2(mn, mn), r_2 = make_float2(r, r);
        const float2 m23 = make_float2(8388608.0f, 8388608.0f);
#pragma unroll
        for (int k = 0; k < kWords; ++k) {
            uint32_t acc = 0;
#pragma unroll
            for (int j = kPairs - 1; j >= 0; --j) {         // elements 2j+1, 2j of the word, highest first
                const uint32_t p = u[kPairs * k + j];
                const float2 d = fsub2(make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u)), mn_2);
                const float2 c = ffma2(d, r_2, m23);
                acc = (acc << kBits) + __float_as_uint(c.y);
                acc = (acc << kBits) + __float_as_uint(c.x);
            }
            code[k] = acc - kPackBias;
        }
    } else {                                                 // scale below binary32's normal range
#pragma unroll
        for (int k = 0; k < kWords; ++k) {
            uint32_t acc = 0;
#pragma unroll
            for (int e = 2 * kPairs - 1; e >= 0; --e) {
                const uint32_t p = u[kPairs * k + (e >> 1)];
                const float w = __uint_as_float((e & 1) ? (p & 0xFFFF0000u) : (p << 16));
                acc = (acc << kBits) + (uint32_t)rintf(__fdiv_rn(__fsub_rn(w, mn), s));
            }
            code[k] = acc;
        }
    }
}

// Warp steps of 32 groups (4 KiB) are handed out grid-stride; lane l
// quantises group l of a step.  Each warp streams its steps through a ring of
// kQStages stages in shared memory with 16-byte asynchronous copies (lane l
// copies chunks l + 32 j: coalesced), kQStages - 1 steps ahead; chunk c of
// group g sits at g*128 + ((c ^ g) & 7)*16, so the 8 lanes of a read phase
// each take a different 16-byte bank group.
template <int kBits>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    k_quantize(const uint16_t *__restrict__ w, long long n_groups, uint8_t *__restrict__ codes,
               uint16_t *__restrict__ scale, uint16_t *__restrict__ bias) {
    __shared__ __align__(16) unsigned char ring[kQWarps][kQStages][4096];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long warps = (long long)gridDim.x * kQWarps;
    const long long steps = (n_groups + 31) / 32;
    const long long st0 = (long long)blockIdx.x * kQWarps + warp;
    const unsigned char *wb = reinterpret_cast<const unsigned char *>(w);
    auto issue = [&](long long i) {                          // the warp's i-th step into its stage
        const long long g0 = (st0 + i * warps) * 32;
        unsigned char *stage = ring[warp][i % kQStages];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int ch = lane + 32 * j, gl = ch >> 3, c = ch & 7;
            const bool live = g0 + gl < n_groups;
            cp_async16(stage + gl * 128 + ((c ^ gl) & 7) * 16, wb + (live ? (g0 * 128 + ch * 16) : 0),
                       live ? 16u : 0u);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kQStages - 1; ++i) issue(i);
    for (long long i = 0; st0 + i * warps < steps; ++i) {
        issue(i + kQStages - 1);
        cp_async_wait<kQStages - 1>();                       // this lane's copies of step i landed
        __syncwarp();                                        // ... and every other lane's
        const unsigned char *stage = ring[warp][i % kQStages];
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + lane * 128 + ((c ^ lane) & 7) * 16);
            u[4 * c] = v.x;
            u[4 * c + 1] = v.y;
            u[4 * c + 2] = v.z;
            u[4 * c + 3] = v.w;
        }
        __syncwarp();                                        // stage read: free to be refilled
        const long long grp = (st0 + i * warps) * 32 + lane;
        uint32_t code[2 * kBits];
        uint16_t sb, bb;
        q_group<kBits>(u, code, sb, bb);
        if (grp < n_groups) {
            uint4 *cq = reinterpret_cast<uint4 *>(codes + grp * (8 * kBits));
#pragma unroll
            for (int k = 0; k < kBits / 2; ++k)
                cq[k] = make_uint4(code[4 * k], code[4 * k + 1], code[4 * k + 2], code[4 * k + 3]);
            scale[grp] = sb;
            bias[grp] = bb;
        }
    }
    cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_dense_matvec(const uint16_t *w, const uint16_t *x, int rows, int cols, float *y,
                                cudaStream_t s) {
    const int cap = device_sm_count() * kMvCtasPerSm;
    // rows per step: four once every CTA owns at least four rows
    if (rows >= 4 * cap) return launch_mv_rb<4>(w, x, rows, cols, y, cap, s);
    if (rows >= 2 * cap) return launch_mv_rb<2>(w, x, rows, cols, y, cap, s);
    return launch_mv_rb<1>(w, x, rows, cols, y, cap, s);
}

cudaError_t launch_quantize(const uint16_t *w, long long n_groups, int bits, uint8_t *codes, uint16_t *scale,
                            uint16_t *bias, cudaStream_t s) {
    const long long steps = (n_groups + 31) / 32;
    const long long need = (steps + kQWarps - 1) / kQWarps;
    const long long cap = (long long)device_sm_count() * kQCtasPerSm;
    const int grid = (int)(need < cap ? need : cap);
    if (bits == 2)
        k_quantize<2><<<grid, kQThreads, 0, s>>>(w, n_groups, codes, scale, bias);
    else
        k_quantize<4><<<grid, kQThreads, 0, s>>>(w, n_groups, codes, scale, bias);
    return cudaGetLastError();
}

}  // namespace smoe

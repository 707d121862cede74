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
// ((mx - mn) + 0) / 15; bias = mn + 0; q = the integer nearest to the exact
// quotient (w - mn) / scale, halves to even (0 where scale is 0).  Reading 2
// bytes and writing 0.5625 per weight, it is HBM-bound once the per-weight
// work is a few instructions: one lane per group, min/max on bf16 pairs, and
// per two weights a few packed fp32 operations that round RN(w - mn) *
// RN(1 / scale) to a candidate code and measure how far the product sits from
// it.  A weight within 2^-17 of a midpoint between two levels (where the
// candidate could differ from the exact answer) is decided exactly later: its
// byte of the code block goes into a per-warp queue, and whenever 16 or more
// are queued the warp decides up to 32 of them at once, one per lane, and
// overwrites those bytes -- the few such weights cost a share of one warp pass
// instead of a pass of their own for every warp they occur in.
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
constexpr int kQCtasPerSm = 6;                           // 24 warps per SM (registers <= 85)
constexpr int kQStages = 2;                              // 4 KiB stages per warp: 32 KiB per CTA

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

// Sign of (dh + dl) - c, exactly, where dh = RN(d), dl = d - dh and c is a
// binary32 value: rounding is monotonic, so dh > c gives d > c, dh < c gives
// d < c, and dh == c leaves d - c = dl.
__device__ __forceinline__ int cmp_exact(float dh, float dl, float c) {
    if (dh != c) return dh > c ? 1 : -1;
    return dl > 0.f ? 1 : (dl < 0.f ? -1 : 0);
}

// Code q of one weight, decided exactly: q0 is the
// fast path's candidate and e = d r - q0 its residual; the exact quotient is
// within 2^-19 of d r, so it can lie beyond the midpoint on e's side only, and
// that one midpoint s (q0 +- 1/2) -- exact in binary32 -- is compared with the
// exact difference w - mn (Knuth's TwoSum).  Halves go to the even level.
__device__ __forceinline__ uint32_t exact_q1(float w, float kk, float mnk, float sk, float r) {
    const float d = __fmaf_rn(w, kk, -mnk);
    const uint32_t cbits = __float_as_uint(__fmaf_rn(d, r, 8388608.0f));
    const int q0 = (int)(cbits - 0x4B000000u);
    const float e = __fmaf_rn(d, r, -(float)q0);
    const float wk = __fmul_rn(w, kk);
    const float dh = __fsub_rn(wk, mnk);
    const float bb = __fsub_rn(dh, wk);
    const float dl = __fadd_rn(__fsub_rn(wk, __fsub_rn(dh, bb)), __fsub_rn(-mnk, bb));
    const bool up = e >= 0.f;
    const int t = cmp_exact(dh, dl, __fmul_rn(sk, (float)q0 + (up ? 0.5f : -0.5f)));
    int q = q0;
    if (up) {
        if (t > 0 || (t == 0 && (q0 & 1))) q = q0 + 1;
    } else {
        if (t < 0 || (t == 0 && (q0 & 1))) q = q0 - 1;
    }
    return (uint32_t)q;
}

// The codes of a group whose scale is above 2^120 (its reciprocal would be
// near binary32's subnormal range, so no candidate is computed): every weight
// is compared with every midpoint s (k + 1/2), exactly as in exact_q1.
// Such a group needs weights near 2^124 and never occurs in practice; it is
// kept so that every finite input has its exact codes.  `row` is the lane's 64
// weights as they sit in its swizzled shared-memory row.
template <int kBits>
__device__ __noinline__ void q_group_huge(const unsigned char *row, int lane, float mn, float s, uint32_t *out) {
    constexpr int kLevels = (1 << kBits) - 1, kPerWord = 32 / kBits;
#pragma unroll 1
    for (int wd = 0; wd < 2 * kBits; ++wd) {
        uint32_t acc = 0;
#pragma unroll 1
        for (int i = kPerWord - 1; i >= 0; --i) {
            const int el = wd * kPerWord + i, c = el >> 3;
            const float w = bf16_to_f32(*reinterpret_cast<const uint16_t *>(row + ((c ^ lane) & 7) * 16 + (el & 7) * 2));
            const float dh = __fsub_rn(w, mn);
            const float bb = __fsub_rn(dh, w);
            const float dl = __fadd_rn(__fsub_rn(w, __fsub_rn(dh, bb)), __fsub_rn(-mn, bb));
            uint32_t q = 0;
            for (int k = 0; k < kLevels; ++k) {
                const int t = cmp_exact(dh, dl, __fmul_rn(s, (float)k + 0.5f));
                q += (t > 0 || (t == 0 && (k & 1))) ? 1u : 0u;
            }
            acc = (acc << kBits) + q;
        }
        out[wd] = acc;
    }
}

// The codes (kBits = 4: SMOE-Q4, 2: SMOE-Q2) of one group of 64 weights, its
// scale and bias.  `row` is the lane's group in its swizzled shared-memory row
// (chunk c of 8 weights at ((c ^ lane) & 7) * 16); it is read twice, once for
// the least and greatest weight and once for the codes, so that no more than
// one code word's weights are held in registers.  Per pair of weights, in
// packed fp32:
//   d  = RN(w kk - mn kk)              (kk = 1, or 2^64 for a scale below 2^-62:
//                                       a power of two, so every value stays exact)
//   c  = RN(d r + 2^23)                 r = RN(1 / (s kk)): c holds 2^23 + q0,
//                                       q0 = rint(d r), rounded once
//   e  = RN(d r - q0)                   the distance from q0 in scale units
//   t  = RN(e e - (1/4 - 2^-17))        t >= 0 only near a midpoint
// d r is within 2^-19 of the exact (w - mn) / s, so a weight with |e| below
// 1/2 - 2^-17 has q0 as its one nearest level.  The sign of t of both weights
// of each pair goes into a 32-bit mask (one funnel shift a pair), returned as
// `flags`: a set bit marks a pair with an exact tie or a weight within 2^-17
// of a midpoint (about one pair in 300 for the bf16 weights here), whose codes
// the caller has decided exactly (exact_q1) after the words are stored.  The
// n = 32 / kBits words e_k of a code word combine into sum_k q_k 2^(kBits k) as
// (sum_k e_k 2^(kBits k)) minus 0x4B000000 * sum_k 2^(kBits k) (mod 2^32), one
// shift-add each.  A group whose scale is above 2^120 is coded by
// q_group_huge, which writes the codes itself (returns true).
template <int kBits>
__device__ __forceinline__ bool q_group(const unsigned char *row, int lane, uint32_t (&code)[2 * kBits],
                                        uint16_t &sb, uint16_t &bb, uint32_t *out, uint32_t &flags) {
    flags = 0u;
    constexpr int kWords = 2 * kBits, kPairs = 16 / kBits;  // code words; bf16 pairs per code word
    constexpr uint32_t kPackBias = kBits == 4 ? 0xFB000000u : 0xE7000000u;   // 0x4B000000 * 0x11111111 / 0x55555555
    constexpr float kLevels = (float)((1 << kBits) - 1);
    auto chunk = [&](int c) { return *reinterpret_cast<const uint4 *>(row + ((c ^ lane) & 7) * 16); };
    uint32_t mn2, mx2;
    {
        const uint4 v = chunk(0);
        mn2 = bf16x2_min(bf16x2_min(v.x, v.y), bf16x2_min(v.z, v.w));
        mx2 = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
    }
#pragma unroll
    for (int c = 1; c < 8; ++c) {
        const uint4 v = chunk(c);
        mn2 = bf16x2_min(mn2, bf16x2_min(bf16x2_min(v.x, v.y), bf16x2_min(v.z, v.w)));
        mx2 = bf16x2_max(mx2, bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w)));
    }
    const float mn = fminf(__uint_as_float(mn2 << 16), __uint_as_float(mn2 & 0xFFFF0000u));
    const float mx = fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u));
    sb = f32_to_bf16(__fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), kLevels));
    bb = f32_to_bf16(__fadd_rn(mn, 0.0f));
    const float s = bf16_to_f32(sb);
    if (s == 0.0f) {
#pragma unroll
        for (int k = 0; k < kWords; ++k) code[k] = 0u;
        return false;
    }
    if (s > 0x1p120f) {
        if (out) q_group_huge<kBits>(row, lane, mn, s, out);
        return true;
    }
    // Every weight of a group with a scale below 2^-62 is below 2^-49 in
    // magnitude, so scaling by 2^64 is exact and overflows nothing.
    const float kk = s < 0x1p-62f ? 0x1p64f : 1.0f;
    const float sk = __fmul_rn(s, kk), mnk = __fmul_rn(mn, kk);
    const float r = __frcp_rn(sk);
    const float2 k2 = make_float2(kk, kk), nmn2 = make_float2(-mnk, -mnk), r2 = make_float2(r, r);
    const float2 m23 = make_float2(8388608.0f, 8388608.0f);
    const float2 ntie = make_float2(-(0.25f - 0x1p-17f), -(0.25f - 0x1p-17f));
    uint32_t clear = 0;            // bit 31 - n: pair n (in processing order) is clear of every midpoint
#pragma unroll
    for (int k = 0; k < kWords; ++k) {
        uint32_t u[kPairs];
#pragma unroll
        for (int h = 0; h < kPairs / 4; ++h) {
            const uint4 v = chunk(k * (kPairs / 4) + h);
            u[4 * h] = v.x;
            u[4 * h + 1] = v.y;
            u[4 * h + 2] = v.z;
            u[4 * h + 3] = v.w;
        }
        uint32_t acc = 0;
#pragma unroll
        for (int j = kPairs - 1; j >= 0; --j) {             // elements 2j+1, 2j of the word, highest first
            const uint32_t p = u[j];
            const float2 d = ffma2(make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u)), k2, nmn2);
            const float2 c = ffma2(d, r2, m23);
            const float2 e = ffma2(d, r2, fsub2(m23, c));    // m23 - c = -q0 exactly
            const float2 t = ffma2(e, e, ntie);
            clear = __funnelshift_l(__float_as_uint(t.x) & __float_as_uint(t.y), clear, 1);
            acc = (acc << kBits) + __float_as_uint(c.y);
            acc = (acc << kBits) + __float_as_uint(c.x);
        }
        code[k] = acc - kPackBias;
    }
    flags = ~clear;                 // pairs near a midpoint (bit 31 - n: pair n in processing order)
    return false;
}

// A byte of a group's code block whose codes the fast pass could not decide:
// its weights (SMOE-Q4: the pair of the byte; SMOE-Q2: its four weights), the
// group's bf16 scale and minimum, and the byte's index in the code array.
struct FixItem {
    uint2 w;            // bf16 weights, lowest element first
    uint32_t sb_bb;     // scale | minimum << 16 (bf16)
    uint32_t at_lo, at_hi;
};
constexpr int kFixCap = 48;             // queue entries per warp (at most 15 + 32 at a time)

// Decides one queued byte exactly (the scalings as in q_group) and stores it.
template <int kBits>
__device__ __forceinline__ void fix_item(const FixItem &it, uint8_t *codes) {
    const float s = bf16_to_f32((uint16_t)(it.sb_bb & 0xFFFFu)), mn = bf16_to_f32((uint16_t)(it.sb_bb >> 16));
    const float kk = s < 0x1p-62f ? 0x1p64f : 1.0f;
    const float sk = __fmul_rn(s, kk), mnk = __fmul_rn(mn, kk);
    const float r = __frcp_rn(sk);
    uint32_t byte = 0;
    constexpr int kPer = 8 / kBits;     // weights of a byte
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const uint32_t word = i < 2 ? it.w.x : it.w.y;
        const float wi = (i & 1) ? __uint_as_float(word & 0xFFFF0000u) : __uint_as_float(word << 16);
        byte |= exact_q1(wi, kk, mnk, sk, r) << (kBits * i);
    }
    codes[((unsigned long long)it.at_hi << 32) | it.at_lo] = (uint8_t)byte;
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
    __shared__ FixItem fq[kQWarps][kFixCap];
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
    int qn = 0;                                              // queued items (warp-uniform)
    // The first n (<= 32) queued items, one per lane, then the rest moved down.
    auto flush = [&](int n) {
        if (lane < n) fix_item<kBits>(fq[warp][lane], codes);
        FixItem keep{};
        const bool mv = n + lane < qn;
        if (mv) keep = fq[warp][n + lane];
        __syncwarp();
        if (mv) fq[warp][lane] = keep;
        qn -= n;
        __syncwarp();
    };
    for (long long i = 0; st0 + i * warps < steps; ++i) {
        issue(i + kQStages - 1);
        cp_async_wait<kQStages - 1>();                       // this lane's copies of step i landed
        __syncwarp();                                        // ... and every other lane's
        const unsigned char *stage = ring[warp][i % kQStages];
        const long long grp = (st0 + i * warps) * 32 + lane;
        const bool live = grp < n_groups;
        uint32_t code[2 * kBits];
        uint16_t sb, bb;
        uint32_t flags;
        uint32_t *cq = reinterpret_cast<uint32_t *>(codes + (live ? grp : 0) * (8 * kBits));
        const bool exact = q_group<kBits>(stage + lane * 128, lane, code, sb, bb, live ? cq : nullptr, flags);
        if (live) {
            if (!exact) {
#pragma unroll
                for (int k = 0; k < kBits / 2; ++k)
                    reinterpret_cast<uint4 *>(cq)[k] = make_uint4(code[4 * k], code[4 * k + 1], code[4 * k + 2], code[4 * k + 3]);
            }
            scale[grp] = sb;
            bias[grp] = bb;
        }
        // Queue the bytes holding pairs near a midpoint; whenever 16 or more
        // are queued, up to 32 are decided together, one per lane.  A byte
        // written by another lane comes after the owning lane's word store
        // above: the warp barriers between order them.
        {
            constexpr int kPairs = 16 / kBits;
            uint32_t fl = (live && !exact) ? flags : 0u;
            const unsigned char *row = stage + lane * 128;
            while (__any_sync(0xffffffffu, fl != 0u)) {
                int b = -1;
                if (fl) {
                    const int n = __clz(fl);
                    const int k = n / kPairs, j = kPairs - 1 - n % kPairs, pi = kPairs * k + j;
                    if (kBits == 4) {
                        b = pi;
                        fl &= ~(0x80000000u >> n);
                    } else {
                        b = pi >> 1;                                   // pairs 2b, 2b + 1 (same word)
                        const int n0 = kPairs * k + kPairs - 1 - (2 * b - kPairs * k);
                        fl &= ~((0x80000000u >> n0) | (0x80000000u >> (n0 - 1)));
                    }
                }
                const uint32_t m = __ballot_sync(0xffffffffu, b >= 0);
                if (b >= 0) {
                    FixItem it;
                    const int e0 = (8 / kBits) * b;                  // first element of the byte
                    auto wpair = [&](int el) {                       // elements el, el + 1 (el even)
                        const int c = el >> 3;
                        return *reinterpret_cast<const uint32_t *>(row + ((c ^ lane) & 7) * 16 + (el & 7) * 2);
                    };
                    it.w.x = wpair(e0);
                    it.w.y = kBits == 2 ? wpair(e0 + 2) : 0u;
                    it.sb_bb = (uint32_t)sb | ((uint32_t)bb << 16);
                    const unsigned long long at = (unsigned long long)grp * (8 * kBits) + (unsigned long long)b;
                    it.at_lo = (uint32_t)at;
                    it.at_hi = (uint32_t)(at >> 32);
                    fq[warp][qn + __popc(m & ((1u << lane) - 1u))] = it;
                }
                qn += __popc(m);
                __syncwarp();
                if (qn >= 16) flush(qn < 32 ? qn : 32);          // leaves at most 15 queued
            }
        }
        __syncwarp();                                        // stage read by every lane: free to be refilled
    }
    if (qn > 0) flush(qn);
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

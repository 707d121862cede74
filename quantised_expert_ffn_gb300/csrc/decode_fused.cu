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
// down) over ~22 MB (30B shape) to ~86 MB (235B shape) of weights, a few
// microseconds of HBM time, so latency is the cost.  One CTA per SM (14
// compute warps + 1 producer warp) runs the whole layer; grid-wide barriers
// use one 64-bit arrival counter that only grows, on its own cache line, with
// wall-clock-bounded polling:
//   phase 0  CTA c < E loads router row c before it waits for the previous
//            kernel (programmatic dependent launch) or layer, normalises x
//            (fp32, the stand-alone router's arithmetic) and writes logit c;
//                                                                 -- barrier
//   phase 1  every CTA ranks the E logits itself and hands the ranked ids to
//            the producer warp, which streams this CTA's gate/up rows and then
//            its down rows with 1-D bulk async copies (cp.async.bulk, the TMA
//            engine) into a 3-slot shared-memory ring; the compute warps turn
//            gate/up rows into h = SiLU(g)*u and store it, fp32, straight into
//            the layout the down phase reads (while the layer's first item is
//            still in flight they run the row code once on the slot as it
//            stands and discard the result, so that item does not run cold);
//                                                                 -- barrier
//   phase 2  one bulk copy brings all of h into shared memory and each thread
//            keeps its 32 values of h in registers; the down rows (mostly
//            resident already) times h, combined in rank order with the
//            residual: y = x + sum_i w_i o_i.
// The stack variant runs every layer of a token in one launch, a grid barrier
// between layers.  kQ2 selects SMOE-Q2 codes (a 32-code chunk is 8 bytes
// instead of 16); everything else is shared.
// Per-row arithmetic: a code q becomes the float 128+q by one byte permute;
// per 32-code chunk s*sum((128+q)x) + (b-128s)*sum(x).
//
// Every wait (mbarrier or grid barrier) is bounded in wall time; on timeout
// the kernel records SMOE_ERR_TIMEOUT in the status word and runs to the end.
#include "common.cuh"
#include "host_cache.h"
#include "kernels.h"

namespace smoe {

namespace {

// 14 compute warps + 1 producer: 15 warps put at most 4 on each of the SM's
// four schedulers, so each thread may hold 128 registers (the per-scheduler
// register file is 16K), enough to keep a lane's 64 activations resident.
constexpr int kWarpsC = 14;                    // compute warps
constexpr int kCompute = kWarpsC * 32;
constexpr int kThreadsF = kCompute + 32;       // + producer warp
constexpr int kSlots = 3;
constexpr int kSlotMax = 48 * 1024 + 512;     // largest ring slot
constexpr int kMaxGuRows = 128;                // gate/up row pairs per CTA
constexpr int kDnU = 7;                        // down rows per thread per ring item

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Named barrier of the compute threads; the non-aligned form, so lanes of a
// warp may arrive from divergent paths (thread 0 leaving a spin).
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
// Test, without blocking, whether the phase of parity `par` has completed.
__device__ __forceinline__ bool mb_test(uint64_t *b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    return ok;
}
// Wait for the phase of parity `par`, bounded in wall time.  try_wait without
// a suspend hint: each try blocks for the hardware's own short window, and a
// completed phase is seen at once (a long suspend hint wakes threads late).
__device__ __forceinline__ bool mb_wait(uint64_t *b, uint32_t par, int32_t *status) {
    if (mb_try(b, par)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mb_try(b, par)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    set_status(status, SMOE_ERR_TIMEOUT);
    return false;
}
// Compute warps wait on a barrier: one lane polls, then every lane observes the
// completed phase (so each lane's later shared-memory reads are ordered after it).
__device__ __forceinline__ void warp_wait(uint64_t *b, uint32_t par, int32_t *status) {
    if ((threadIdx.x & 31) == 0) mb_wait(b, par, status);
    __syncwarp();
    mb_try(b, par);
}
// 1-D bulk copy global -> shared, completion counted on `bar` (16-byte multiples)
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}

// Grid-wide barrier over the compute warps of all CTAs (one CTA per SM, all
// resident: the kernel is a cooperative launch).  `ctr` only grows: an arrival
// that returns `prev` belongs to the barrier instance that ends at the next
// multiple of gridDim.x.  The spin gives up after `limit_ns` (a kernel
// argument the host sets) and records SMOE_ERR_TIMEOUT; nothing else waits on
// this spin, so giving up early only leaves the results wrong, and every CTA
// still arrives at every barrier, so the counter stays a multiple of the grid
// at the end of the launch.
__device__ __forceinline__ void grid_sync(unsigned long long *ctr, int32_t *status, uint64_t limit_ns) {
    bar_compute();
    if (threadIdx.x == 0) {
        const unsigned long long G = gridDim.x;
        unsigned long long prev, v;
        asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(prev) : "l"(ctr) : "memory");
        const unsigned long long target = (prev / G + 1) * G;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if (v < target) {
            const uint64_t t0 = global_ns();
            while (true) {
                asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
                if (v >= target) break;
                if (global_ns() - t0 > limit_ns) {
                    set_status(status, SMOE_ERR_TIMEOUT);
                    break;
                }
            }
        }
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

// sum_k (128+q_k) x_k over the 32 codes of a 16-byte chunk, two independent chains
__device__ __forceinline__ float dot32(uint4 c, const float4 (&x)[8]) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    dot8(c.x, x[0], x[1], a0);
    dot8(c.y, x[2], x[3], a1);
    dot8(c.z, x[4], x[5], a0);
    dot8(c.w, x[6], x[7], a1);
    return (a0.x + a0.y) + (a1.x + a1.y);
}

// SMOE-Q2: sum_k (128+q_k) x_k over the 32 codes of an 8-byte chunk.  In a
// 32-bit word, element 4j+k sits in bits 2k..2k+1 of byte j: the mask
// (w >> 2k) & 0x03030303 holds elements k, 4+k, 8+k, 12+k one per byte, and
// the byte permute turns each into the float 128 + q exactly.
__device__ __forceinline__ void dot16q2(uint32_t w, const float4 *x, float2 &a0, float2 &a1) {
    const uint32_t t0 = w & 0x03030303u, t1 = (w >> 2) & 0x03030303u;
    const uint32_t t2 = (w >> 4) & 0x03030303u, t3 = (w >> 6) & 0x03030303u;
    a0 = ffma2(make_float2(code_f32<0>(t0), code_f32<0>(t1)), make_float2(x[0].x, x[0].y), a0);
    a1 = ffma2(make_float2(code_f32<0>(t2), code_f32<0>(t3)), make_float2(x[0].z, x[0].w), a1);
    a0 = ffma2(make_float2(code_f32<1>(t0), code_f32<1>(t1)), make_float2(x[1].x, x[1].y), a0);
    a1 = ffma2(make_float2(code_f32<1>(t2), code_f32<1>(t3)), make_float2(x[1].z, x[1].w), a1);
    a0 = ffma2(make_float2(code_f32<2>(t0), code_f32<2>(t1)), make_float2(x[2].x, x[2].y), a0);
    a1 = ffma2(make_float2(code_f32<2>(t2), code_f32<2>(t3)), make_float2(x[2].z, x[2].w), a1);
    a0 = ffma2(make_float2(code_f32<3>(t0), code_f32<3>(t1)), make_float2(x[3].x, x[3].y), a0);
    a1 = ffma2(make_float2(code_f32<3>(t2), code_f32<3>(t3)), make_float2(x[3].z, x[3].w), a1);
}

// The 32-code chunk at p (16 bytes of Q4 codes, or 8 of Q2) against x.
template <bool kQ2>
__device__ __forceinline__ float dot_chunk(const unsigned char *p, const float4 (&x)[8]) {
    if constexpr (kQ2) {
        const uint2 c = *reinterpret_cast<const uint2 *>(p);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        dot16q2(c.x, x, a0, a1);
        dot16q2(c.y, x + 4, a0, a1);
        return (a0.x + a0.y) + (a1.x + a1.y);
    } else {
        return dot32(*reinterpret_cast<const uint4 *>(p), x);
    }
}

// Warp-wide sums of eight values at once (v[j] of every lane): 9 shuffles
// instead of 40.  Each exchange halves the values a lane carries; lane L ends
// with the total of v[4*b4 + 2*b3 + b2] (b = bits of L), held by 4 lanes.
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = (b4 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[j + 4], 16);
    float u[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
        u[j] = (b3 ? w[j + 2] : w[j]) + __shfl_xor_sync(0xffffffffu, b3 ? w[j] : w[j + 2], 8);
    float t = (b2 ? u[1] : u[0]) + __shfl_xor_sync(0xffffffffu, b2 ? u[0] : u[1], 4);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    return t;
}

// ---------------------------------------------------------------- work lists

// Gate/up: CTA c owns row pairs [P*c/G, P*(c+1)/G) of the P = K*F (slot, row)
// pairs; an item is up to r_gu consecutive rows of one expert slot.  All
// products stay below 2^31 (K*F <= 16384, G <= 256).
__device__ __forceinline__ void gu_range(const FusedArgs &a, int &p0, int &p1) {
    const int P = a.K * a.F;
    p0 = P * (int)blockIdx.x / (int)gridDim.x;
    p1 = P * ((int)blockIdx.x + 1) / (int)gridDim.x;
}

// Down: CTA c owns output rows [d0, d1), multiples of a.dn_gran rows (so each
// row block's scale block starts 16-byte aligned); an item is a block of up to
// a.dn_nr of those rows (a multiple of dn_gran) for all K expert slots.
__device__ __forceinline__ void dn_rows(const FusedArgs &a, int &d0, int &d1) {
    const int units = a.D / a.dn_gran;
    d0 = units * (int)blockIdx.x / (int)gridDim.x * a.dn_gran;
    d1 = units * ((int)blockIdx.x + 1) / (int)gridDim.x * a.dn_gran;
}

// Position of h[i][f] in the down phase's layout: chunk c = f/32 of slot i is
// read by the thread that owns (i, c); float4 k = (f%32)/4 of the chunk sits at
// ((i*MC + c/8)*8 + k)*8 + c%8, so the 8 threads of a phase that own
// consecutive chunks read 128 consecutive bytes (no bank conflicts).
__device__ __forceinline__ int h_pos(int i, int f, int MC) {
    const int c = f >> 5, k = (f & 31) >> 2;
    return ((((i * MC + (c >> 3)) * 8 + k) * 8 + (c & 7)) << 2) + (f & 3);
}

// Weights of layer l: the stack variant reads them from the device table.
struct LW {
    const uint16_t *gain, *router_w;
    const uint8_t *gq, *uq, *dq;
    const uint16_t *gs, *gb, *us, *ub, *ds, *db;
};
__device__ __forceinline__ LW layer_w(const FusedArgs &a, int l) {
    if (!a.layers) return {a.gain, a.router_w, a.gq, a.uq, a.dq, a.gs, a.gb, a.us, a.ub, a.ds, a.db};
    const smoe_layer *L = a.layers + l;
    return {L->rms_gain, L->router_w, L->gate_q, L->up_q, L->down_q, L->gate_s, L->gate_b,
            L->up_s, L->up_b, L->down_s, L->down_b};
}

// ---------------------------------------------------------------- kernel

template <bool kRoute, bool kQ2>
__global__ void __launch_bounds__(kThreadsF, 1) k_decode_layer(FusedArgs a) {
    constexpr int kCB = kQ2 ? 8 : 16;            // bytes of a 32-code chunk
    extern __shared__ __align__(128) unsigned char sm[];
    const int D = a.D, F = a.F, K = a.K, E = a.E;
    const int NC = D / 32;                       // 32-code chunks of a gate/up row
    const int NCP = (NC + 63) / 64;              // passes of 64 chunks (2 per lane)
    const int FC = F / 32;                       // 32-code chunks of a down row
    const int FG = F / kGroup;
    const int MC = (FC + 7) / 8;                 // blocks of 8 chunks in the h layout
    const int P = K * FC;                        // (slot, chunk) pairs of the down phase
    unsigned char *ring = sm;
    float *u_region = reinterpret_cast<float *>(sm + a.ring_bytes);       // xs+xc | hs | red
    float *xs = u_region;                        // NCP*64*8 float4
    float *xc = xs + NCP * 2048;                 // NCP*64 chunk sums
    float *hs = u_region;                        // K*MC*256 floats (h, down-phase layout)
    float *red = u_region;                       // [rows][P] down partial sums (after h is in registers)
    uint16_t *xraw = reinterpret_cast<uint16_t *>(sm + a.ring_bytes + a.union_bytes);   // [D]
    float *os = reinterpret_cast<float *>(xraw + D);                                 // [K][rows_max]
    __shared__ uint64_t full[kSlots], empty[kSlots], idx_ready, h_ready;
    __shared__ float red14[kWarpsC];
    __shared__ __align__(16) unsigned long long keys[kMaxExperts];
    __shared__ float lsel[kMaxTopK], wsel[kMaxTopK];
    __shared__ int isel[kMaxTopK], ivalid[kMaxTopK];
    __shared__ float part[kMaxGuRows * 2 * 2];   // gate/up partial sums per (row, pass)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mb_init(&full[s], 1);
            mb_init(&empty[s], kWarpsC);     // one arrival per compute warp
        }
        mb_init(&idx_ready, 1);
        mb_init(&h_ready, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int d0, d1, p0, p1;
    dn_rows(a, d0, d1);
    gu_range(a, p0, p1);
    const int rows = d1 - d0;

    if (warp == kWarpsC) {
        // ================= producer: bulk copies into the ring =================
        // Lane 0 waits for a free slot and posts its byte count; then one lane
        // per copy issues the copies of the item together.  Lane i < K holds
        // the expert of slot i: the ranked id, or -- given ids -- read here as
        // soon as the previous kernel is done, so streaming starts while the
        // compute warps still normalise x (an id that cannot be used streams
        // expert 0, as on the compute side).
        uint32_t g = 0;
        for (int l = 0; l < a.n_layers; ++l) {
        const LW W = layer_w(a, l);
        int my_e = 0;
        if (kRoute) {
            int ok = 1;
            if (lane == 0) ok = mb_wait(&idx_ready, l & 1, a.status);
            if (!__shfl_sync(0xffffffffu, ok, 0)) return;
            mb_try(&idx_ready, l & 1);             // each lane observes the ids
            if (lane < K) my_e = isel[lane];
        } else {
            pdl_wait();
            if (lane < K) {
                const int e = __ldcg(a.idx_in + lane);
                my_e = (e >= 0 && e < E) ? e : 0;
            }
        }
        const int NG = D / kGroup;
        const uint32_t RBg = D / 32 * kCB;
        for (int p = p0; p < p1; ++g) {
            const int i = p / F, j0 = p - i * F, n = min(a.r_gu, min(p1 - p, F - j0));
            const uint32_t s = g % kSlots;
            unsigned char *dst = ring + s * a.slot_bytes;
            const uint32_t cb = n * RBg, sb = n * NG * 2;
            if (lane == 0) {
                mb_wait(&empty[s], ((g / kSlots) & 1) ^ 1, a.status);
                mb_expect(&full[s], 2 * cb + 4 * sb);
            }
            __syncwarp();
            mb_try(&empty[s], ((g / kSlots) & 1) ^ 1);
            const size_t row = (size_t)__shfl_sync(0xffffffffu, my_e, i) * F + j0;
            if (lane < 2) {
                bulk_g2s(dst + lane * cb, (lane ? W.uq : W.gq) + row * RBg, cb, &full[s]);
            } else if (lane < 6) {
                const uint16_t *src = lane == 2 ? W.gs : lane == 3 ? W.gb : lane == 4 ? W.us : W.ub;
                bulk_g2s(dst + 2 * cb + (lane - 2) * sb, src + row * NG, sb, &full[s]);
            }
            p += n;
        }
        for (int r0 = 0; r0 < rows; r0 += a.dn_nr, ++g) {
            const int nr = min(a.dn_nr, rows - r0);
            const uint32_t s = g % kSlots;
            unsigned char *dst = ring + s * a.slot_bytes;
            const uint32_t cb = nr * (F / 32 * kCB), sb = nr * FG * 2;
            if (lane == 0) {
                mb_wait(&empty[s], ((g / kSlots) & 1) ^ 1, a.status);
                mb_expect(&full[s], K * (cb + 2 * sb));
            }
            __syncwarp();
            mb_try(&empty[s], ((g / kSlots) & 1) ^ 1);
            const int e_lo = __shfl_sync(0xffffffffu, my_e, lane % K);
            const int e_hi = __shfl_sync(0xffffffffu, my_e, (lane + 32) % K);
            for (int q = lane; q < 3 * K; q += 32) {
                const int i = q % K, kind = q / K;
                const size_t row = (size_t)(q < 32 ? e_lo : e_hi) * D + d0 + r0;
                if (kind == 0)
                    bulk_g2s(dst + i * cb, W.dq + row * (F / 32 * kCB), cb, &full[s]);
                else
                    bulk_g2s(dst + K * cb + ((kind - 1) * K + i) * sb, (kind == 1 ? W.ds : W.db) + row * FG, sb,
                             &full[s]);
            }
        }
        }   // layers
        // every copy issued has landed before the CTA may exit
        if (lane == 0)
            for (uint32_t k = (g > (uint32_t)kSlots ? g - kSlots : 0); k < g; ++k)
                mb_wait(&full[k % kSlots], (k / kSlots) & 1, a.status);
        __syncwarp();
        return;
    }

    // ================= compute warps =================
    uint32_t g = 0;
    for (int l = 0; l < a.n_layers; ++l) {
    const LW W = layer_w(a, l);
    const uint16_t *xin = l == 0 ? a.x : (((l - 1) & 1) ? a.act1 : a.act0);
    uint16_t *yout = l == a.n_layers - 1 ? a.y : ((l & 1) ? a.act1 : a.act0);
    // Inputs that do not depend on the previous kernel (layer) are requested
    // before waiting for it: this CTA's router row and the RMSNorm gain.
    uint4 rw[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    uint4 gv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    const bool has_row = kRoute && (int)blockIdx.x < E;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int d8 = (tid + q * kCompute) * 8;
        if (d8 < D) {
            if (has_row) rw[q] = ld_stream16(W.router_w + (size_t)blockIdx.x * D + d8);
            if (W.gain) gv[q] = *reinterpret_cast<const uint4 *>(W.gain + d8);
        }
    }

    if (l == 0) {
        pdl_wait();
        pdl_launch_dependents();
    } else {
        grid_sync(a.gctr, a.status, a.grid_wait_ns);     // every CTA's rows of the previous layer's output are written
    }

    // ids and weights given by the caller (FFN-only variant): requested now,
    // consumed after the normalisation
    int e_in = -1;
    float w_in = 0.f;
    if (!kRoute && tid < K) {
        e_in = __ldcg(a.idx_in + tid);
        w_in = __ldcg(a.w_in + tid);
    }

    // ---- normalise x: thread t owns elements [8(t + q*kCompute), +8), q = 0, 1 ----
    float xv[2][8];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int d8 = (tid + q * kCompute) * 8;
        if (d8 < D) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(xin + d8));
            *reinterpret_cast<uint4 *>(xraw + d8) = v;
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
    if (W.gain) {
        // the reduction order of block_rms_inv: stride-256 scalar partials,
        // a warp tree, then the 8 warp sums in order
        float ss = 0.f;
        if (tid < 256)
            for (int d = tid; d < D; d += 256) {
                const float v = bf16_to_f32(xraw[d]);
                ss = fmaf(v, v, ss);
            }
        ss = warp_sum(ss);
        if (lane == 0) red14[warp] = ss;
        bar_compute();
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += red14[i];
        const float inv = 1.0f / sqrtf(t / (float)D + a.eps);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int d8 = (tid + q * kCompute) * 8;
            if (d8 < D) {
                const uint16_t *gg = reinterpret_cast<const uint16_t *>(&gv[q]);
#pragma unroll
                for (int k = 0; k < 8; ++k) xv[q][k] = bf16_to_f32(rms_apply(xraw[d8 + k], inv, gg[k]));
            }
        }
    }
    // stage xn (fp32) lane-interleaved for the gate/up sweep: chunk
    // c = pass*64 + half*32 + l sits at float4 ((pass*2+half)*8 + k)*32 + l.
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int d8 = (tid + q * kCompute) * 8;
        const bool own = d8 < D;
        if (own) {
            const int c = d8 >> 5, k0 = (d8 & 31) >> 2;
            const int pass = c >> 6, hl = (c >> 5) & 1, l = c & 31;
            float4 *dst = reinterpret_cast<float4 *>(xs) + ((pass * 2 + hl) * 8 + k0) * 32 + l;
            dst[0] = make_float4(xv[q][0], xv[q][1], xv[q][2], xv[q][3]);
            dst[32] = make_float4(xv[q][4], xv[q][5], xv[q][6], xv[q][7]);
        }
        float s8 = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) s8 += xv[q][k];
        s8 += __shfl_xor_sync(0xffffffffu, s8, 1);     // 4 consecutive threads = one chunk
        s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
        if (own && (tid & 3) == 0) xc[d8 >> 5] = s8;
    }
    for (int c = NC + tid; c < NCP * 64; c += kCompute) {   // chunks past D read as zero
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
            if (lane == 0) red14[warp] = acc;
            bar_compute();
            if (tid == 0) {
                float t = 0.f;
                for (int i = 0; i < kWarpsC; ++i) t += red14[i];
                a.logits[blockIdx.x] = t;
            }
        }
        grid_sync(a.gctr, a.status, a.grid_wait_ns);
        float my = -INFINITY;
        unsigned long long mykey = 0;
        if (tid < E) {
            my = __ldcg(a.logits + tid);
            // unique key: larger logit first, equal logits keep the lower id
            mykey = ((unsigned long long)order_key(my) << 32) | (0xFFFFFFFFu - (uint32_t)tid);
            keys[tid] = mykey;
        }
        bar_compute();
        if (tid < E) {
            int r0 = 0, r1 = 0;
            const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(keys);
#pragma unroll 8
            for (int j = 0; j < E / 2; ++j) {
                const ulonglong2 kk = k2[j];
                r0 += kk.x > mykey;
                r1 += kk.y > mykey;
            }
            if (E & 1) r0 += keys[E - 1] > mykey;
            const int rank = r0 + r1;
            if (rank < K) {
                isel[rank] = tid;
                lsel[rank] = my;
            }
        }
        bar_compute();
        if (tid == 0) mb_arrive(&idx_ready);   // ranked ids are all the producer needs
        const float m = lsel[0];
        float denom = 0.f;
        if (a.norm_topk_prob) {
            for (int i = 0; i < K; ++i) denom += expf(lsel[i] - m);
        } else {
            float pz = (tid < E) ? expf(my - m) : 0.f;
            pz = warp_sum(pz);
            if (lane == 0) red14[warp] = pz;
            bar_compute();
            for (int i = 0; i < kWarpsC; ++i) denom += red14[i];
        }
        if (tid < K) {
            wsel[tid] = expf(lsel[tid] - m) / denom;
            if (blockIdx.x == 0 && a.idx_out) {
                a.idx_out[l * K + tid] = isel[tid];
                a.w_out[l * K + tid] = wsel[tid];
            }
        }
    } else {
        if (tid < K) {
            if (e_in < 0 || e_in >= E) {
                set_status(a.status, SMOE_ERR_DEVICE);
                e_in = -1;
            }
            isel[tid] = e_in;
            wsel[tid] = w_in;
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
    if (!kRoute && tid == 0) mb_arrive(&idx_ready);

    // ---- phase 1: gate/up rows -> h, the activations in registers ----
    // Warp w takes pass pw = w % NCP (chunks pw*64 + lane and pw*64 + 32 + lane
    // of every row, so its 64 activations stay in registers) and row slot
    // w / NCP of each item; the NCP partial sums of a row meet in shared memory.
    {
        const int NG = D / kGroup;
        const int pw = warp % NCP, rs = warp / NCP, rstep = kWarpsC / NCP;
        const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
        const int ca = pw * 64 + lane, cbk = ca + 32;
        float4 xa[8], xb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            xa[q] = xs4[((pw * 2 + 0) * 8 + q) * 32 + lane];
            xb[q] = xs4[((pw * 2 + 1) * 8 + q) * 32 + lane];
        }
        const float Xa = xc[ca], Xb = xc[cbk];
        // the lane partials of up to four rows wait in registers (newest first)
        // and are summed together by warp_sum8
        float acc8[8];
        uint32_t trow = 0;          // byte k: 1 + row pair index of slot k (0 = empty)
        auto reset = [&]() {
#pragma unroll
            for (int q = 0; q < 8; ++q) acc8[q] = 0.f;
            trow = 0;
        };
        auto flush = [&]() {
            const float tot = warp_sum8(acc8, lane);
            if ((lane & 3) == 0) {
                const int j = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                const int t = (int)((trow >> (8 * (j >> 1))) & 0xFFu) - 1;
                if (t >= 0) part[(t * NCP + pw) * 2 + (j & 1)] = tot;
            }
            reset();
        };
        reset();
        int nacc = 0;
        // Pass 0 runs the row code once over the first item's ring slot as it
        // stands (its copy may still be in flight) and keeps nothing: without
        // it a layer's first item runs these instructions cold, at about 2.5x
        // the time of the items after it.  A warp skips it when that item has
        // already landed.  A warp takes at most one row of an item
        // (r_gu <= rstep), so the pass cannot reach a flush; pass 1 starts
        // from cleared partials.
        const bool dry = p0 < p1 && !__shfl_sync(0xffffffffu, (int)mb_test(&full[g % kSlots], (g / kSlots) & 1), 0);
#pragma unroll 1
        for (int pass = dry ? 0 : 1; pass < 2; ++pass) {
            const bool real = pass == 1;
            if (real) {
                reset();
                nacc = 0;
            }
            for (int p = p0; p < p1; ++g) {
                const int i = p / F, j0 = p - i * F, n = min(a.r_gu, min(p1 - p, F - j0));
                const uint32_t s = g % kSlots;
                if (real) warp_wait(&full[s], (g / kSlots) & 1, a.status);
                const unsigned char *slot = ring + s * a.slot_bytes;
                const uint32_t RBg = D / 32 * kCB, cb = n * RBg;
                const uint16_t *gsr = reinterpret_cast<const uint16_t *>(slot + 2 * cb);
                const uint16_t *gbr = gsr + n * NG, *usr = gbr + n * NG, *ubr = usr + n * NG;
                for (int r = rs; r < n; r += rstep) {
                    float ag = 0.f, au = 0.f;
                    if (ca < NC) {
                        const float A = dot_chunk<kQ2>(slot + r * RBg + ca * kCB, xa);
                        const float B = dot_chunk<kQ2>(slot + cb + r * RBg + ca * kCB, xa);
                        const int gi = r * NG + (ca >> 1);
                        const float s0 = bf16_to_f32(gsr[gi]), b0 = bf16_to_f32(gbr[gi]);
                        const float s1 = bf16_to_f32(usr[gi]), b1 = bf16_to_f32(ubr[gi]);
                        ag = s0 * A + (b0 - 128.f * s0) * Xa;
                        au = s1 * B + (b1 - 128.f * s1) * Xa;
                    }
                    if (cbk < NC) {
                        const float A = dot_chunk<kQ2>(slot + r * RBg + cbk * kCB, xb);
                        const float B = dot_chunk<kQ2>(slot + cb + r * RBg + cbk * kCB, xb);
                        const int gi = r * NG + (cbk >> 1);
                        const float s0 = bf16_to_f32(gsr[gi]), b0 = bf16_to_f32(gbr[gi]);
                        const float s1 = bf16_to_f32(usr[gi]), b1 = bf16_to_f32(ubr[gi]);
                        ag += s0 * A + (b0 - 128.f * s0) * Xb;
                        au += s1 * B + (b1 - 128.f * s1) * Xb;
                    }
#pragma unroll
                    for (int q = 7; q >= 2; --q) acc8[q] = acc8[q - 2];
                    acc8[0] = ag;
                    acc8[1] = au;
                    trow = (trow << 8) | (uint32_t)(p + r - p0 + 1);   // row pair index within this CTA
                    if (++nacc == 4) {
                        flush();
                        nacc = 0;
                    }
                }
                __syncwarp();
                if (!real) break;
                if (lane == 0) mb_arrive(&empty[s]);
                p += n;
            }
        }   // passes
        if (nacc > 0) flush();
    }

    // ---- phase 2 set-up: down rows of this CTA ----
    // Thread t < P*RS owns (slot, chunk) pair pp = t % P -- slot i = pp / FC,
    // chunk c = pp % FC -- and keeps that chunk of h_i in registers; it takes
    // rows s, s+RS, ... (s = t / P) of every item.  Per row it leaves
    // s_ic*sum((128+q)h) + (b_ic-128 s_ic)*sum(h) in red[(row*K + i)*(FC+1) + c]
    // (rows of FC+1 floats: the later per-(row, slot) sums read without bank
    // conflicts).
    const int RS = a.dn_rs;
    const bool dn_live = tid < P * RS;
    const int pp = dn_live ? tid % P : 0, sp = dn_live ? tid / P : 0;
    const int di = pp / FC, dc = pp - di * FC;
    float4 hq[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hq[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float Hc = 0.f;

    // Pass 0 (first layer of a launch) runs the down-row code once on whatever
    // the first ring slot holds and keeps nothing: a warp that is done with
    // gate/up fetches those instructions while it would otherwise wait at the
    // barrier.  Pass 1 is the real one.
#pragma unroll 1
    for (int pass = l == 0 ? 0 : 1; pass < 2; ++pass) {
        const bool real = pass == 1;
        if (real) {
            bar_compute();
            // the passes of each gate/up row, added in pass order: h = SiLU(gate) * up
            for (int t = tid; t < p1 - p0; t += kCompute) {
                float ag = 0.f, au = 0.f;
                for (int q = 0; q < NCP; ++q) {
                    ag += part[(t * NCP + q) * 2];
                    au += part[(t * NCP + q) * 2 + 1];
                }
                const int pq = p0 + t, i = pq / F, j = pq - i * F;
                a.h[h_pos(i, j, MC)] = ivalid[i] ? silu_mul(ag, au) : 0.f;
                asm volatile("fence.proxy.async.global;" ::: "memory");   // h store -> later bulk reads
            }
            // ---- barrier: all of h written; then one bulk copy brings it in ----
            grid_sync(a.gctr, a.status, a.grid_wait_ns);
            const uint32_t hbytes = (uint32_t)(K * MC * 256 * 4);
            if (tid == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mb_expect(&h_ready, hbytes);
                bulk_g2s(hs, a.h, hbytes, &h_ready);
            }
            warp_wait(&h_ready, l & 1, a.status);
            const float4 *hv = reinterpret_cast<const float4 *>(hs) + ((di * MC + (dc >> 3)) * 8) * 8 + (dc & 7);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                hq[k] = hv[k * 8];
                Hc += (hq[k].x + hq[k].y) + (hq[k].z + hq[k].w);
            }
            bar_compute();   // h is in registers: its shared-memory region now holds red
        }
        for (int r0 = 0; r0 < rows; r0 += a.dn_nr) {
            const int nr = min(a.dn_nr, rows - r0);
            const uint32_t s = g % kSlots;
            if (real) warp_wait(&full[s], (g / kSlots) & 1, a.status);
            const unsigned char *slot = ring + (real ? s : 0) * a.slot_bytes;
            if (dn_live && sp < nr) {
                const uint32_t cb = nr * (F / 32 * kCB), sb = nr * FG * 2;
                const unsigned char *cp = slot + di * cb + dc * kCB;
                const uint16_t *sp16 = reinterpret_cast<const uint16_t *>(slot + K * cb + di * sb) + (dc >> 1);
                const uint16_t *bp16 = reinterpret_cast<const uint16_t *>(slot + K * cb + (K + di) * sb) + (dc >> 1);
                float acc[kDnU];
#pragma unroll
                for (int u = 0; u < kDnU; ++u) {
                    const int rr = min(sp + u * RS, nr - 1);          // a row past the item repeats the last
                    const float A = dot_chunk<kQ2>(cp + rr * (F / 32 * kCB), hq);
                    const float sc = bf16_to_f32(sp16[rr * FG]), bi = bf16_to_f32(bp16[rr * FG]);
                    acc[u] = sc * A + (bi - 128.f * sc) * Hc;
                }
#pragma unroll
                for (int u = 0; u < kDnU; ++u)
                    if (real && sp + u * RS < nr) red[((r0 + sp + u * RS) * K + di) * (FC + 1) + dc] = acc[u];
            }
            __syncwarp();
            if (!real) break;
            if (lane == 0) mb_arrive(&empty[s]);
            ++g;
        }
    }
    bar_compute();
    // o_i[r]: the FC chunk partials of slot i, in chunk order
    for (int u = tid; u < rows * K; u += kCompute) {
        const int r = u / K, i = u - r * K;
        const float *rp = red + (r * K + i) * (FC + 1);
        float o = 0.f;
        for (int c = 0; c < FC; ++c) o += rp[c];
        os[i * a.rows_max + r] = o;
    }
    bar_compute();
    for (int r = tid; r < rows; r += kCompute) {
        float y = bf16_to_f32(xraw[d0 + r]);
        for (int i = 0; i < K; ++i) {
            const float o = os[i * a.rows_max + r];
            y = fmaf(wsel[i], o, y);
            if (a.expert_out) a.expert_out[(size_t)i * D + d0 + r] = o;
        }
        yout[d0 + r] = f32_to_bf16(y);
    }
    }   // layers
}

}  // namespace

// Host: shape support, work partition and shared-memory plan of the fused layer kernel.
bool fused_plan(FusedArgs &a, int num_sms) {
    const int D = a.D, F = a.F, K = a.K;
    if (D % 512 || F % 128 || D > 4096 || K > kMaxTopK) return false;
    // bulk copies need 16-byte aligned sources
    const void *ptrs[] = {a.gq, a.uq, a.dq, a.gs, a.gb, a.us, a.ub, a.ds, a.db, a.x, a.h};
    for (const void *q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) % 16) return false;
    if (a.gain && reinterpret_cast<uintptr_t>(a.gain) % 16) return false;
    a.grid = num_sms;
    if (a.E > a.grid || a.grid > 256) return false;
    const int NG = D / kGroup, FG = F / kGroup, FC = F / 32;
    // down: the (slot, chunk) pairs must fit the compute threads (h in registers)
    const int P = K * FC;
    if (P > kCompute) return false;
    a.dn_rs = kCompute / P;
    // row blocks whose scale rows start 16-byte aligned
    int gran = 1;
    while ((gran * FC) % 16) ++gran;
    a.dn_gran = gran;
    const int units = D / gran;
    a.rows_max = ((units + a.grid - 1) / a.grid) * gran;
    const int cb32 = a.q2 ? 8 : 16;                           // bytes of a 32-code chunk
    const int row_pair_bytes = 2 * (D / 32 * cb32 + NG * 2 * 2);
    const int dn_row_bytes = K * (F / 32 * cb32 + FG * 2 * 2);  // one down row, all K slots
    // gate/up: one row pair per (group of NCP warps) per item
    const int NCPh = (D / 32 + 63) / 64;
    a.r_gu = kWarpsC / NCPh;
    while (a.r_gu > 1 && a.r_gu * row_pair_bytes > kSlotMax) --a.r_gu;
    // down: as many rows (multiples of gran) per item as fit in a slot
    a.dn_nr = (kSlotMax / dn_row_bytes) / gran * gran;
    a.dn_nr = min(a.dn_nr, kDnU * a.dn_rs / gran * gran);   // each thread's rows of an item unroll fully
    if (a.dn_nr < gran) return false;
    if (a.dn_nr > a.rows_max) a.dn_nr = a.rows_max;
    a.slot_bytes = max(a.r_gu * row_pair_bytes, a.dn_nr * dn_row_bytes);
    a.slot_bytes = (a.slot_bytes + 127) / 128 * 128;
    a.ring_bytes = kSlots * a.slot_bytes;
    const int NCP = (D / 32 + 63) / 64, MC = (FC + 7) / 8;
    const int xs_bytes = (NCP * 2048 + NCP * 64) * 4;
    const int hs_bytes = K * MC * 256 * 4;
    const int red_bytes = a.rows_max * K * (FC + 1) * 4;
    if ((K * F + a.grid - 1) / a.grid > kMaxGuRows || D / 32 > 128) return false;
    a.union_bytes = (max(xs_bytes, max(hs_bytes, red_bytes)) + 127) / 128 * 128;
    a.smem_bytes = a.ring_bytes + a.union_bytes + D * 2 + K * a.rows_max * 4;
    return a.smem_bytes <= 210 * 1024;
}

// Floats of h scratch the fused kernel needs (its padded down-phase layout).
size_t fused_h_floats(int F, int K) { return (size_t)K * ((F / 32 + 7) / 8) * 256; }

// The grid barriers need every CTA resident at once, so the kernel is a
// cooperative launch: the CTAs start only when all of them fit on the device
// (if other kernels hold SMs, the launch waits for them instead of starting
// part of the grid), and a device that cannot hold the grid at all (fewer
// usable SMs, e.g. a partitioned GPU) refuses the launch with
// cudaErrorCooperativeLaunchTooLarge before anything is enqueued.  It is also
// a programmatic dependent launch: the prologue (router row, gain) runs while
// the previous kernel in the stream finishes, and griddepcontrol.wait orders
// the rest after it.
template <bool kRoute, bool kQ2>
static cudaError_t launch_variant(const FusedArgs &a, cudaStream_t s) {
    static SmemLimits limits;
    const size_t smem = a.smem_bytes;
    const cudaError_t e = allow_dynamic_smem(k_decode_layer<kRoute, kQ2>, limits, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(kThreadsF);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_decode_layer<kRoute, kQ2>, a);
}

cudaError_t launch_decode_layer(const FusedArgs &a, cudaStream_t s, bool route) {
    if (a.q2) return route ? launch_variant<true, true>(a, s) : launch_variant<false, true>(a, s);
    return route ? launch_variant<true, false>(a, s) : launch_variant<false, false>(a, s);
}

}  // namespace smoe

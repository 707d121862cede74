// common.cuh -- device helpers shared by the kernels of libsmoe.so (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/smoe.h"

namespace smoe {

constexpr int kGroup = 64;          // Q4 group along the input dimension
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;
constexpr int kMaxChunk = 64;       // tokens per prefill chunk
constexpr int kMaxD = 8192;
constexpr int kMaxF = 4096;
constexpr int kMaxKF = 16384;       // top_k * ffn_dim

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Streaming 16-byte load of weights that are read once per token: bypass L1.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Load through L2 only (data another kernel may have written while this one was
// already resident under programmatic dependent launch).
__device__ __forceinline__ uint16_t ld_cg_u16(const uint16_t *p) {
    return __ldcg(reinterpret_cast<const unsigned short *>(p));
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t *p) {
    unsigned short r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Four Q4 codes of one byte-lane group to exact floats.
//   lo = w & 0x0F0F0F0F holds codes 0,2,4,6 of the word (one per byte),
//   hi = (w >> 4) & 0x0F0F0F0F holds codes 1,3,5,7.
// prmt places byte k of `lo`/`hi` into bits 16..23 of a float whose upper
// byte is 0x43 and whose low 16 bits are zero: the float 128 + q, exactly.
template <int kByte>
__device__ __forceinline__ float code_f32(uint32_t nib) {
    uint32_t r;
    // selector: byte3 <- b.byte3 (0x43), byte2 <- a.byte kByte, byte1,0 <- b.byte0 (0)
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(nib), "r"(0x43000000u), "n"(0x7044 | (kByte << 8)));
    return __uint_as_float(r);
}

// Packed fp32 FMA on two lanes: (a.x*b.x + c.x, a.y*b.y + c.y).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long rb = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long rc = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long rd;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    return *reinterpret_cast<float2 *>(&rd);
}

// sum_k (128 + q_k) * x_k over the 8 codes of one 32-bit word (codes k of x[k]),
// accumulated into acc (two partial sums).
__device__ __forceinline__ void dot8(uint32_t w, float4 xa, float4 xb, float2 &acc) {
    uint32_t lo = w & 0x0F0F0F0Fu;
    uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
    acc = ffma2(make_float2(code_f32<0>(lo), code_f32<0>(hi)), make_float2(xa.x, xa.y), acc);
    acc = ffma2(make_float2(code_f32<1>(lo), code_f32<1>(hi)), make_float2(xa.z, xa.w), acc);
    acc = ffma2(make_float2(code_f32<2>(lo), code_f32<2>(hi)), make_float2(xb.x, xb.y), acc);
    acc = ffma2(make_float2(code_f32<3>(lo), code_f32<3>(hi)), make_float2(xb.z, xb.w), acc);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void set_status(int32_t *status, int code) {
    if (status) atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inverse RMS 1/sqrt(mean(x^2) + eps) of a bf16 vector, for a CTA of 256
// threads.  Every kernel that normalises a hidden state calls this, so the
// router and the FFN kernels see bit-identical normed inputs.
__device__ __forceinline__ float block_rms_inv(const uint16_t *x, int D, float eps, float *red8) {
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += 256) {
        const float v = bf16_to_f32(ld_cg_u16(x + d));
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red8[threadIdx.x >> 5] = ss;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red8[i];
    __syncthreads();
    return 1.0f / sqrtf(t / (float)D + eps);
}

// One normed element: bf16(x * inv * gain), the value the router sees.
__device__ __forceinline__ uint16_t rms_apply(uint16_t x, float inv, uint16_t gain) {
    return f32_to_bf16(bf16_to_f32(x) * inv * bf16_to_f32(gain));
}

// Nanoseconds of the global timer (bounds every wait of the persistent kernels).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;   // 200 ms: far beyond any legitimate wait

// mbarrier phase test that suspends the calling thread in hardware (up to
// `hint_ns`) until the phase completes, instead of returning at once: waiting
// threads then take no issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_suspend(uint32_t bar_smem, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar_smem), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kSuspendHintNs = 20000;   // 20 us per try; the wall-clock bound still applies

// Programmatic dependent launch controls (no-ops when launched without PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace smoe

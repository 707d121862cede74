// prefill_tc.cu -- prefill chunk FFN as grouped per-expert GEMMs on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA staging).
//
// "Optimizations" page, "Prefill Reads Each Expert Once, Not Once Per Token":
// a chunk's routed experts are deduplicated into a union that is read once;
// here each union expert's Q4 rows are streamed from HBM once and multiplied
// with all the tokens of its bucket.  The pages' token-batch prefill FFN
// kernels keep a thread-per-row layout ("The Dense Ceiling" section); on GB300
// the bucket makes the work a real (if skinny) contraction, so it runs on the
// tensor cores with the weights as the 128-row M side ("swap AB") and the
// bucket's tokens as N (padded to a multiple of 16, at most 64).
//
// One persistent CTA per SM walks a list of units (union expert u and
// its row tiles: a 128-row tile of both gate and up, or two adjacent 128-row
// tiles of down, so that every stage of a unit feeds two MMA threads from one
// set of activation tiles); per unit the K dimension is consumed in stages of
// two Q4 groups (128 codes: a 64-byte slice of each Q4 row, which the memory
// system serves faster than 32-byte slices).  Warp roles:
//   warps 0-7   dequant: read the TMA-staged codes of a stage from shared
//               memory, turn them into fp16 w = s*q + b (one rounding; exact
//               when b = -8 s, since s*(q-8) needs at most 11 bits) group by
//               group and store them straight into tensor memory
//               (tcgen05.st): warp w owns TMEM lanes 32*(w%4).. = tile rows,
//               and the stages of parity w/4, so the two dequant warps of a
//               scheduler work on alternate stages and one's waits overlap the
//               other's arithmetic;
//   warp 12     TMA: code tiles (no swizzle) and the bucket's activation
//               tiles (128-byte swizzle, one per group) into a ring of
//               shared-memory stages;
//   warps 13-14 MMA: one thread of each issues tcgen05.mma with A from tensor
//               memory (M=128 weight rows, K=16) and B from shared memory (N =
//               pad16(bucket) tokens), fp16 x fp16 -> fp32 in TMEM, and commits
//               stages back -- warp 13 the first tile of the unit, warp 14 the
//               second.  A thread blocks on each tcgen05.mma until the tensor
//               pipe takes it, and its later shared-memory accesses (barrier
//               waits included) queue behind the MMAs it issued, so each MMA
//               thread waits only for the stage's A: the dequant warps waited
//               for the stage's tiles before they released it;
//   warps 8-11  epilogue: tcgen05.ld the accumulator (each warp its 32 TMEM
//               lanes = 32 weight rows) and write h = SiLU(g)*u as fp16
//               (gate/up kernel) or the fp32 expert outputs (down kernel).
// Units are handed out in order by a device counter: the TMA thread claims
// the next one while it issues the current unit's last stages and posts it in
// a small shared-memory queue that the other roles read, so a CTA that starts
// late (a down CTA on an SM that gate/up freed late) or runs slow takes fewer.
// The down kernel does not wait for the whole gate/up grid: each gate/up
// epilogue warp counts its stored rows of h per union expert, and the down
// kernel's TMA thread waits, per unit, for its expert's count to be complete,
// so down CTAs start on the SMs that gate/up's last round of units leaves
// idle (a dependent launch: it happens once every gate/up CTA runs, and no
// gate/up CTA waits on down, so the waits always end).
// TMEM: columns 0-255 two accumulator buffers (gate, up: 64 columns each), so
// the epilogue of one unit overlaps the main loop of the next, and columns
// 256-511 two stages of dequantised A (each two groups of both matrices); or,
// for units of many stages (kOneAcc), one accumulator buffer in columns 0-127
// and three A stages in 128-511.  Keeping A out of shared memory leaves
// shared-memory bandwidth to the TMA and to the B operand.  Every wait on an
// mbarrier is bounded: on timeout the CTA records SMOE_ERR_TIMEOUT, all roles
// drain and the TMEM is freed.
//
// The dequant writes the 8 elements of each 32-bit code word as the pairs
// (e0,e4),(e1,e5),(e2,e6),(e3,e7) -- the order the fp16 magic-number unpack
// produces them in.  The activation side (x for gate/up, h for down) is stored
// with the same permutation of each 8-element block, so the contraction is
// unchanged.  kQ2 selects SMOE-Q2 codes (16 per 32-bit word); their dequant
// emits the same element order, so nothing else changes.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "host_cache.h"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kTcThreads = 480;
constexpr int kProdThreads = 256;    // warps 0-7
constexpr int kEpiWarp0 = 8;         // warps 8-11
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kMma2Warp = 14;      // gate/up: the up matrix's MMA thread
constexpr int kTile = 128;
constexpr int kKc = 64;
constexpr int kNmax = 64;
// Two rings.  kStages shared-memory stages hold kGpc groups' codes and
// activation tiles; a stage is refilled once its codes are read and the MMAs
// that read its tiles have completed (the TMA waits on its empty barrier).
// kAStages TMEM stages (columns from kACol0) hold a stage's dequantised A;
// stage g's A overwrites stage g - kAStages's once that stage's MMAs have
// completed, i.e. once its shared-memory stage is empty -- the producers wait
// on that phase, so the TMEM ring needs no barriers of its own and the MMA
// threads one commit per stage.  (The dequant warps release a stage's codes
// only through that same barrier, after the MMAs: a TMA write may not follow
// their reads of the same bytes without a proxy fence, and by then the values
// read have long been consumed.)  Ring depths of 4 to 6 stages measure within
// 3 % of each other; 7 (224 KB) are slower.
constexpr int kGpc = 2;      // Q4 groups (64-code chunks along K) per stage
constexpr int kStages = 6;
constexpr int kAStages = 2;   // with two accumulator buffers; 3 with one (kOneAcc)
constexpr uint32_t kTmemCols = 512;
constexpr int kUQ = 4;       // unit queue entries: how many units the TMA thread may run ahead of the epilogue
constexpr uint32_t kAccStride = 128;                  // two accumulator buffers: columns 0-127, 128-255
constexpr uint32_t kUpCol = 64;                       // up accumulator after gate's (N <= 64 columns each)
constexpr uint32_t kACol0 = 256;                      // A stages: columns 256-511 (128-511 with one buffer)
constexpr uint32_t kACols = 32;                       // one matrix's 128 x 64 fp16 chunk: 32 columns
constexpr uint32_t kAMatCols = kGpc * kACols;         // one matrix's columns of a stage
constexpr int kCodeBytes = kTile * kKc * kGpc / 2;   // 8 KB of codes per matrix per stage
constexpr int kBTileBytes = kNmax * kKc * 2;         // 8 KB fp16 B tile (up to 64 rows)

struct TcParams {
    int n_tiles;            // 128-row tiles per expert
    int n_chunks;           // K / 64
    int rows_per_expert;    // F (gate/up) or D (down)
    int tile_rows;          // weight rows of one unit: 128, or 256 for a pair of down tiles
    int a1_row;             // first row of the second matrix's tile within the unit: 0 (up), 128 (down pair)
    int k_dim;              // K (D or F)
    int out_ld;             // row length of the output (F for h, D for o)
    const int32_t *n_union, *union_ids, *offsets;
    const uint16_t *s0, *b0, *s1, *b1;   // scales/biases of A0 (gate or down) and A1 (up)
    int vec_scales;         // K/64 % 8 == 0 and 16-byte aligned scale arrays: 8 groups per load
    __half *hout;           // gate/up: h [slots][F] fp16, K-permuted
    float *oout;            // down: o [slots][D] fp32
    // Per union slot, the gate/up epilogue warps that have written their rows of
    // h (each warp adds 1 once its 32 rows of a tile are stored).  Gate/up adds to
    // it; down, with it set, waits per unit for ready_target instead of waiting
    // for the whole gate/up grid, so its CTAs start on the SMs that gate/up's
    // last round leaves idle.  NULL: neither.
    int32_t *ready;
    int ready_target;       // down: 4 warps x gate/up tiles per expert
    // Units handed out in order by this counter (zero at launch), so a CTA that
    // starts early or runs fast takes more of them; NULL: the static list
    // blockIdx.x, + gridDim.x, ...
    int32_t *unit_ctr;
    int32_t *status;
};

// ---- PTX wrappers ----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(b))
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                     smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete, bounded in wall time; false on
// timeout (which also raises the CTA's abort flag) or when another role aborted.
// Plain try_wait polling: a long suspend hint wakes the waiter late.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try(b, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    *abort_flag = 1;
    set_status(status, SMOE_ERR_TIMEOUT);
    return false;
}

// Bounded wait until *ctr >= target (gpu-scope acquire), then a proxy fence:
// the bulk tensor reads issued after it see what the counter's writers
// released.  On timeout it records SMOE_ERR_TIMEOUT and raises the CTA's abort
// flag, as mbar_wait does.
__device__ __forceinline__ bool wait_count(const int32_t *ctr, int target, volatile int *abort_flag,
                                           int32_t *status) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v < target) {
        const uint64_t t0 = global_ns();
        while (true) {
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= target) break;
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                set_status(status, SMOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in the 128-byte swizzle: rows of 128 bytes, 8-row groups
// 1024 bytes apart (stride byte offset), leading byte offset unused.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp16 A and B (K-major), fp32 D, M x N.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// A operand from tensor memory: lane m holds row m, two fp16 K elements per
// column.  The MMAs of one K chunk (64 = 4 x 16) for one A matrix in a single block:
// A columns a, a+8, a+16, a+24 of TMEM; B descriptors b0 + 2*kk (32 bytes
// apart); the first MMA accumulates only when `acc` is set.
__device__ __forceinline__ void mma_chunk_ta(uint32_t d, uint32_t a, uint64_t b0, uint32_t idesc,
                                             uint32_t acc) {
    asm volatile(
        "{ .reg .pred p, t; .reg .b64 b1, b2, b3; .reg .b32 a1, a2, a3;"
        " setp.ne.u32 p, %4, 0; setp.eq.u32 t, %4, %4;"
        " add.s64 b1, %2, 2; add.s64 b2, %2, 4; add.s64 b3, %2, 6;"
        " add.s32 a1, %1, 8; add.s32 a2, %1, 16; add.s32 a3, %1, 24;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t; }" ::"r"(d),
        "r"(a), "l"(b0), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[8][4]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0][0]), "r"(r[0][1]), "r"(r[0][2]), "r"(r[0][3]), "r"(r[1][0]), "r"(r[1][1]), "r"(r[1][2]), "r"(r[1][3]),
        "r"(r[2][0]), "r"(r[2][1]), "r"(r[2][2]), "r"(r[2][3]), "r"(r[3][0]), "r"(r[3][1]), "r"(r[3][2]), "r"(r[3][3]),
        "r"(r[4][0]), "r"(r[4][1]), "r"(r[4][2]), "r"(r[4][3]), "r"(r[5][0]), "r"(r[5][1]), "r"(r[5][2]), "r"(r[5][3]),
        "r"(r[6][0]), "r"(r[6][1]), "r"(r[6][2]), "r"(r[6][3]), "r"(r[7][0]), "r"(r[7][1]), "r"(r[7][2]), "r"(r[7][3])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
        " [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- dequant ---------------------------------------------------------------

__device__ __forceinline__ __half2 f2h2(float f) { return __half2half2(__float2half_rn(f)); }

// The levels b .. b + L s of a group (L = 15 for SMOE-Q4, 3 for SMOE-Q2) must
// stay within fp16's range for the dequantised operand to be valid.
__device__ __forceinline__ bool levels_in_fp16(float s, float b, float L) {
    return fabsf(b) <= 65504.f && fabsf(fmaf(s, L, b)) <= 65504.f;
}

__device__ __forceinline__ uint32_t or_masked(uint32_t a, uint32_t mask, uint32_t c) {   // (a & mask) | c
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}

// 8 codes of one word -> 4 half2 (e_i, e_{i+4}), each s*q + b with one rounding.
// A code in bits 0-3 of a half-word under the exponent of 1024 (0x6400) is the
// fp16 1024 + q; one in bits 4-7 under the exponent of 64 (0x5400) is 64 + q
// (the mantissa's unit there is 1/16); a subtraction leaves q exactly.  So the
// lower byte pair needs no shift and the upper one a single shift by 8.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 b2, uint32_t (&o)[4]) {
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    const __half2 k64 = __halves2half2(__ushort_as_half(0x5400), __ushort_as_half(0x5400));
    const uint32_t w8 = w >> 8;
    const uint32_t m[4] = {or_masked(w, 0x000F000Fu, 0x64006400u), or_masked(w, 0x00F000F0u, 0x54005400u),
                           or_masked(w8, 0x000F000Fu, 0x64006400u), or_masked(w8, 0x00F000F0u, 0x54005400u)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 q = __hsub2(*reinterpret_cast<const __half2 *>(&m[i]), (i & 1) ? k64 : k1024);  // exact q
        __half2 v = __hfma2(q, s2, b2);                                                            // s*q + b, one rounding
        o[i] = *reinterpret_cast<uint32_t *>(&v);
    }
}

// SMOE-Q2: the 16 codes of one word (element e in bits 2e) -> 8 half2, in the
// order dequant_word gives a Q4 word's 8 elements -- (e_i, e_{i+4}) of the
// block of elements 0-7 (o0), then of 8-15 (o1) -- so the activation side
// keeps its permutation.  A byte permute puts bytes 0 and 1 (elements 0-3,
// 4-7) into the two half-words of one register, bytes 2 and 3 into another;
// each 2-bit field then becomes the fp16 1024 + q exactly, as for Q4.
__device__ __forceinline__ void dequant_word_q2(uint32_t w, __half2 s2, __half2 b2, uint32_t (&o0)[4],
                                                uint32_t (&o1)[4]) {
    const __half2 k1024 = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(lo) : "r"(w));    // [b0, 0, b1, 0]
    asm("prmt.b32 %0, %1, 0, 0x4342;" : "=r"(hi) : "r"(w));    // [b2, 0, b3, 0]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t m0, m1;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(m0) : "r"(lo >> (2 * i)), "r"(0x00030003u), "r"(0x64006400u));
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(m1) : "r"(hi >> (2 * i)), "r"(0x00030003u), "r"(0x64006400u));
        __half2 v0 = __hfma2(__hsub2(*reinterpret_cast<__half2 *>(&m0), k1024), s2, b2);
        __half2 v1 = __hfma2(__hsub2(*reinterpret_cast<__half2 *>(&m1), k1024), s2, b2);
        o0[i] = *reinterpret_cast<uint32_t *>(&v0);
        o1[i] = *reinterpret_cast<uint32_t *>(&v1);
    }
}

__device__ __forceinline__ int perm8(int f) {   // position of element f in the permuted order
    const int i = f & 7;
    return (f & ~7) | (i < 4 ? 2 * i : 2 * (i - 4) + 1);
}

template <bool kPair>
struct Smem {
    static constexpr int kMats = kPair ? 2 : 1;
    static constexpr int kStageBytes = kMats * kCodeBytes + kGpc * kBTileBytes;
    static constexpr int kStageOff = 0;
    static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
    static constexpr int kBytes = kBarOff + 1024;   // barriers + tmem slot + flags
};

// kPair: two 128-row A tiles per unit share each stage's activation tiles --
// gate and up (kHOut: the epilogue writes h = SiLU(g) * u), or two adjacent
// tiles of the down matrix (the epilogue writes both as fp32 outputs).
template <bool kPair, bool kQ2, bool kHOut, bool kOneAcc>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_prefill_tc(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                 const __grid_constant__ CUtensorMap tm_b16, const __grid_constant__ CUtensorMap tm_b32,
                 const __grid_constant__ CUtensorMap tm_b48, const __grid_constant__ CUtensorMap tm_b64,
                 TcParams p) {
    using S = Smem<kPair>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *st_ring = sm + S::kStageOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::kBarOff);
    uint64_t *full = bars;                    // [kStages] codes + activations landed
    uint64_t *empty = full + kStages;         // [kStages] codes read and the stage's MMAs complete
    // kOneAcc: one accumulator buffer (columns 0-127) and three A stages, so
    // that a stage's A waits for the MMAs of the stage three back, not two;
    // the epilogue of a unit then no longer overlaps the next unit's MMAs
    constexpr int kAS = kOneAcc ? 3 : kAStages;
    constexpr uint32_t kAC0 = kOneAcc ? 128 : kACol0;
    uint64_t *afull = empty + kStages;        // [kAS] dequantised A written
    uint64_t *accfull = afull + 3;            // [2]
    uint64_t *accempty = accfull + 2;         // [2]
    uint64_t *drain = accempty + 2;           // [2] all MMAs issued by MMA thread i complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // the unit queue: the TMA thread claims units from p.unit_ctr and posts
    // them here in order; every consuming warp (or MMA thread) releases an entry
    uint64_t *uq_full = reinterpret_cast<uint64_t *>(tmem_slot + 2);   // [kUQ]
    uint64_t *uq_empty = uq_full + kUQ;                                 // [kUQ]
    volatile int *uq = reinterpret_cast<volatile int *>(uq_empty + kUQ); // [kUQ] unit, -1: none left

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // A stage is dequantised by the 4 warps of its parity (128 threads) and
    // multiplied by one MMA thread per matrix, each committing on its own.
    constexpr uint32_t kIssuers = kPair ? 2 : 1;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kProdThreads / 2 + kIssuers);
        }
        for (int i = 0; i < kAS; ++i) mbar_init(&afull[i], kProdThreads / 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], kIssuers);
            mbar_init(&accempty[i], 128);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        for (int i = 0; i < kUQ; ++i) {
            mbar_init(&uq_full[i], 1);
            mbar_init(&uq_empty[i], kProdThreads / 32 + 4 + kIssuers);   // dequant, epilogue warps, MMA threads
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The down kernel with ready counters waits per unit (see TcParams::ready)
    // and for the previous grid only before it exits.  What else it reads was
    // complete before any gate/up CTA passed its own wait, and its launch, a
    // dependent one, happens only after every gate/up CTA has passed it; it
    // reads the union through L2.
    const bool overlap = !kHOut && p.ready != nullptr;
    if (!overlap) pdl_wait();        // union, buckets and activations of the previous kernels
    pdl_launch_dependents();

    const int nu = __ldcg(p.n_union);
    const int n_units = nu * p.n_tiles;
    const int NC = p.n_chunks;
    const int NSC = NC / kGpc;       // stages per unit (K is a multiple of 128)
    const bool dyn = p.unit_ctr != nullptr;
    // The k-th unit of this CTA for a consuming warp (every lane returns it) or
    // thread (lone = true): the static list, or the queue entry the TMA thread
    // posted, released once read.  -1: no units left, or a wait gave up.
    auto next_unit = [&](uint32_t k, bool lone) -> int {
        if (!dyn) {
            const int u = blockIdx.x + (int)k * (int)gridDim.x;
            return u < n_units ? u : -1;
        }
        const int q = (int)(k % kUQ);
        const bool got = mbar_wait(&uq_full[q], (k / kUQ) & 1, abort_flag, p.status);
        if (lone) {
            if (!got) return -1;
            const int u = uq[q];
            mbar_arrive(&uq_empty[q]);
            return u;
        }
        if (!__all_sync(0xffffffffu, got)) return -1;
        const int u = uq[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&uq_empty[q]);
        return u;
    };

    if (warp == kTmaWarp) {
        if (lane == 0) {
            uint32_t g = 0;
            // dynamic: the next unit is claimed two stages before this unit's
            // last, so the atomic's round trip overlaps the issue of those stages
            int next = dyn ? atomicAdd(p.unit_ctr, 1) : -1;
            const int claim_at = NSC > 2 ? NSC - 2 : 0;
            for (uint32_t k = 0; !*abort_flag; ++k) {
                int unit;
                if (dyn) {
                    unit = next < n_units ? next : -1;
                    const int q = (int)(k % kUQ);
                    if (k >= (uint32_t)kUQ && !mbar_wait(&uq_empty[q], ((k / kUQ) - 1) & 1, abort_flag, p.status)) break;
                    uq[q] = unit;
                    mbar_arrive(&uq_full[q]);
                } else {
                    unit = blockIdx.x + (int)k * (int)gridDim.x;
                    if (unit >= n_units) unit = -1;
                }
                if (unit < 0) break;
                const int u = unit / p.n_tiles, tile = unit - u * p.n_tiles;
                const int e = __ldcg(p.union_ids + u);
                const int off = __ldcg(p.offsets + u);
                int m = __ldcg(p.offsets + u + 1) - off;
                m = m > kNmax ? kNmax : m;
                if (overlap && !wait_count(p.ready + u, p.ready_target, abort_flag, p.status)) break;
                const int nb = (m + 15) >> 4;            // 1..4
                const CUtensorMap *tb = nb <= 1 ? &tm_b16 : nb == 2 ? &tm_b32 : nb == 3 ? &tm_b48 : &tm_b64;
                const uint32_t bbytes = (uint32_t)(nb < 1 ? 1 : nb) * 16 * kKc * 2;  // full box, OOB rows zero-filled
                const int row = e * p.rows_per_expert + tile * p.tile_rows;
                for (int c = 0; c < NSC; ++c, ++g) {
                    if (dyn && c == claim_at) next = atomicAdd(p.unit_ctr, 1);
                    const int s = g % kStages;
                    const uint32_t ph = (g / kStages) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) break;
                    unsigned char *stg = st_ring + s * S::kStageBytes;
                    constexpr int kCodeRow = kGpc * (kQ2 ? kKc / 4 : kKc / 2);   // code bytes of a row's stage
                    mbar_expect_tx(&full[s], S::kMats * kTile * kCodeRow + kGpc * bbytes);
                    tma_load_2d(stg, &tm_a0, c * kCodeRow, row, &full[s]);
                    if (kPair) tma_load_2d(stg + kCodeBytes, &tm_a1, c * kCodeRow, row + p.a1_row, &full[s]);
#pragma unroll
                    for (int h = 0; h < kGpc; ++h)
                        tma_load_2d(stg + S::kMats * kCodeBytes + h * kBTileBytes, tb, (c * kGpc + h) * kKc, off, &full[s]);
                }
            }
            // drain: every stage issued must have landed before the CTA exits
            for (uint32_t k = (g > (uint32_t)kStages ? g - kStages : 0); k < g; ++k)
                mbar_wait(&full[k % kStages], (k / kStages) & 1, abort_flag, p.status);
        }
    } else if (warp == kMmaWarp || warp == kMma2Warp) {
        const int mat = warp - kMmaWarp;          // 0: gate (or down), 1: up
        if (lane == 0 && (mat == 0 || kPair)) {
            uint32_t g = 0, i = 0;
            bool issued = false;
            for (; !*abort_flag; ++i) {
                const int unit = next_unit(i, true);
                if (unit < 0) break;
                const int u = unit / p.n_tiles;
                int m = __ldcg(p.offsets + u + 1) - __ldcg(p.offsets + u);
                m = m > kNmax ? kNmax : m;
                const int npad = ((m + 15) >> 4) << 4;
                const uint32_t idesc = idesc_f16(kTile, npad < 16 ? 16 : npad);
                const uint32_t b = kOneAcc ? 0u : (i & 1);
                if (!mbar_wait(&accempty[b], (kOneAcc ? (i & 1) : ((i >> 1) & 1)) ^ 1, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d0 = tmem + b * kAccStride;
                bool ok = true;
                for (int c = 0; c < NSC; ++c, ++g) {
                    const int s = g % kStages, a = g % kAS;
                    // the stage's tiles have landed: the dequant warps waited for them
                    // before releasing the stage's A (afull orders this thread after them)
                    if (!mbar_wait(&afull[a], (g / kAS) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issued = true;
                    const uint32_t acol = tmem + kAC0 + a * S::kMats * kAMatCols + mat * kAMatCols;
                    const uint32_t bsm = smem_u32(st_ring + s * S::kStageBytes + S::kMats * kCodeBytes);
#pragma unroll
                    for (int h = 0; h < kGpc; ++h)
                        mma_chunk_ta(d0 + mat * kUpCol, acol + h * kACols, smem_desc_sw128(bsm + h * kBTileBytes), idesc,
                                     (c > 0 || h > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&accfull[b]);
            }
            // every issued MMA must be complete before the TMEM is released
            if (issued) {
                mma_commit(&drain[mat]);
                mbar_wait(&drain[mat], 0, abort_flag, p.status);
            }
        }
    } else if (warp < 8) {
        // ---------------- dequant producers ----------------
        // warp w writes TMEM lanes 32*(w%4).. (its quarter of the tile's rows)
        // for the stages of parity w/4, the stage's kGpc groups of each matrix;
        // the two warps of a scheduler thus work on alternate stages, and one's
        // waits overlap the other's arithmetic.
        const int rq = warp & 3, cp = warp >> 2;
        const int r = 32 * rq + lane;
        const uint32_t tlane = (uint32_t)(32 * rq) << 16;
        constexpr float kLv = kQ2 ? 3.f : 15.f;
        uint32_t gbase = 0;     // global index of the current unit's stage 0
        // Scales and biases of a stage's groups, matrix m, group h.
        struct StageSB { float s[2][kGpc], b[2][kGpc]; };
        // Stage c of the unit: wait for its tiles, turn the codes into fp16 s*q + b
        // group by group and store them into the stage's A columns.  false when a
        // wait gave up.
        auto stage = [&](int c, const StageSB &sb) -> bool {
            const uint32_t g = gbase + (uint32_t)c;
            const int s = g % kStages, a = g % kAS;
            __half2 sh[2][kGpc], bh[2][kGpc];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int h = 0; h < kGpc; ++h) {
                    if ((m == 0 || kPair) && !levels_in_fp16(sb.s[m][h], sb.b[m][h], kLv)) set_status(p.status, SMOE_ERR_RANGE);
                    sh[m][h] = f2h2(sb.s[m][h]);
                    bh[m][h] = f2h2(sb.b[m][h]);
                }
            // waits are warp-uniform: the TMEM stores below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (g / kStages) & 1, abort_flag, p.status)))
                return false;
            const unsigned char *stg = st_ring + s * S::kStageBytes;
            constexpr int kRowBytes = kGpc * (kQ2 ? 16 : 32);     // code bytes of a row's stage
            constexpr int kVecs = kRowBytes / 16;
            uint4 cw[2][kVecs];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int v = 0; v < kVecs; ++v)
                    cw[m][v] = (m == 0 || kPair) ? *reinterpret_cast<const uint4 *>(stg + m * kCodeBytes + r * kRowBytes + 16 * v)
                                                 : make_uint4(0, 0, 0, 0);
            mbar_arrive(&empty[s]);                   // codes consumed
            uint32_t q[8][4];
            const uint32_t acol = tmem + tlane + kAC0 + a * S::kMats * kAMatCols;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                if (m == 1 && !kPair) break;
#pragma unroll
                for (int h = 0; h < kGpc; ++h) {
                    if constexpr (kQ2) {              // one 16-byte vector per group
                        const uint4 w = cw[m][h];
                        dequant_word_q2(w.x, sh[m][h], bh[m][h], q[0], q[1]);
                        dequant_word_q2(w.y, sh[m][h], bh[m][h], q[2], q[3]);
                        dequant_word_q2(w.z, sh[m][h], bh[m][h], q[4], q[5]);
                        dequant_word_q2(w.w, sh[m][h], bh[m][h], q[6], q[7]);
                    } else {                          // two per group
                        const uint4 wa = cw[m][2 * h], wb = cw[m][2 * h + 1];
                        dequant_word(wa.x, sh[m][h], bh[m][h], q[0]);
                        dequant_word(wa.y, sh[m][h], bh[m][h], q[1]);
                        dequant_word(wa.z, sh[m][h], bh[m][h], q[2]);
                        dequant_word(wa.w, sh[m][h], bh[m][h], q[3]);
                        dequant_word(wb.x, sh[m][h], bh[m][h], q[4]);
                        dequant_word(wb.y, sh[m][h], bh[m][h], q[5]);
                        dequant_word(wb.z, sh[m][h], bh[m][h], q[6]);
                        dequant_word(wb.w, sh[m][h], bh[m][h], q[7]);
                    }
                    if (m == 0 && h == 0) {
                        // A stage a is free once the MMAs of stage g - kAS completed:
                        // that stage's empty phase (it cannot have moved on since: its
                        // next phase needs the MMAs of stage g - kAS + kStages, which
                        // run after this stage's)
                        if (g >= (uint32_t)kAS) {
                            const uint32_t gp = g - kAS;
                            if (!__all_sync(0xffffffffu, mbar_wait(&empty[gp % kStages], (gp / kStages) & 1, abort_flag, p.status)))
                                return false;
                        }
                        tc_fence_after();
                    }
                    tmem_st32(acol + m * kAMatCols + h * kACols, q);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&afull[a]);
            return true;
        };
        for (uint32_t k = 0; !*abort_flag; ++k, gbase += NSC) {
            const int unit = next_unit(k, false);
            if (unit < 0) break;
            const int u = unit / p.n_tiles, tile = unit - u * p.n_tiles;
            const int e = __ldcg(p.union_ids + u);
            const size_t row = (size_t)e * p.rows_per_expert + tile * p.tile_rows + r;
            const int NG = p.k_dim / kGroup;
            bool ok = true;
            if (p.vec_scales) {
                // Scales and biases of this row, 8 groups (8 / kGpc stages) per 16-byte
                // load, the next 8 requested one block ahead of use; of a block's
                // stages this warp takes those of its parity.
                uint4 vs0{}, vb0{}, vs1{}, vb1{}, ns0{}, nb0{}, ns1{}, nb1{};
                auto load8 = [&](int c8, uint4 &ts0, uint4 &tb0, uint4 &ts1, uint4 &tb1) {
                    const size_t o = row * NG + c8;
                    ts0 = __ldg(reinterpret_cast<const uint4 *>(p.s0 + o));
                    tb0 = __ldg(reinterpret_cast<const uint4 *>(p.b0 + o));
                    if (kPair) {
                        ts1 = __ldg(reinterpret_cast<const uint4 *>(p.s1 + o));
                        tb1 = __ldg(reinterpret_cast<const uint4 *>(p.b1 + o));
                    }
                };
                auto pick = [&](const uint4 &v, int gi) {      // group gi (0..7) of a block
                    const int j2 = gi >> 1;
                    const uint32_t w = j2 == 0 ? v.x : j2 == 1 ? v.y : j2 == 2 ? v.z : v.w;
                    return bf16_to_f32((uint16_t)(w >> (16 * (gi & 1))));
                };
                load8(0, vs0, vb0, vs1, vb1);
                if (NC > 8) load8(8, ns0, nb0, ns1, nb1);
                for (int c8 = 0; c8 < NC && ok; c8 += 8) {
                    if (c8 > 0) {
                        vs0 = ns0; vb0 = nb0; vs1 = ns1; vb1 = nb1;
                        if (c8 + 8 < NC) load8(c8 + 8, ns0, nb0, ns1, nb1);
                    }
#pragma unroll
                    for (int j = 0; j < 8 / kGpc / 2; ++j) {
                        const int l = 2 * j + cp;                  // stage of the block
                        StageSB sb;
#pragma unroll
                        for (int h = 0; h < kGpc; ++h) {
                            sb.s[0][h] = pick(vs0, l * kGpc + h);
                            sb.b[0][h] = pick(vb0, l * kGpc + h);
                            sb.s[1][h] = kPair ? pick(vs1, l * kGpc + h) : sb.s[0][h];
                            sb.b[1][h] = kPair ? pick(vb1, l * kGpc + h) : sb.b[0][h];
                        }
                        if (!stage(c8 / kGpc + l, sb)) {
                            ok = false;
                            break;
                        }
                    }
                }
            } else {
                for (int c = cp; c < NSC; c += 2) {
                    // scales/biases of this row's groups (L1-cached: 16 groups share a sector)
                    StageSB sb;
#pragma unroll
                    for (int h = 0; h < kGpc; ++h) {
                        const size_t o = row * NG + c * kGpc + h;
                        sb.s[0][h] = bf16_to_f32(p.s0[o]);
                        sb.b[0][h] = bf16_to_f32(p.b0[o]);
                        sb.s[1][h] = kPair ? bf16_to_f32(p.s1[o]) : sb.s[0][h];
                        sb.b[1][h] = kPair ? bf16_to_f32(p.b1[o]) : sb.b[0][h];
                    }
                    if (!stage(c, sb)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) break;
        }
    } else {
        // ---------------- epilogue (warps 8-11) ----------------
        const int q = warp - kEpiWarp0;                // TMEM lane quarter
        const int r = q * 32 + lane;                   // weight row in the tile
        for (uint32_t i = 0; !*abort_flag; ++i) {
            const int unit = next_unit(i, false);
            if (unit < 0) break;
            const int u = unit / p.n_tiles, tile = unit - u * p.n_tiles;
            const int off = __ldcg(p.offsets + u);
            int m = __ldcg(p.offsets + u + 1) - off;
            if (m > kNmax) {
                set_status(p.status, SMOE_ERR_DEVICE);
                m = kNmax;
            }
            const uint32_t b = kOneAcc ? 0u : (i & 1);
            const bool got = mbar_wait(&accfull[b], kOneAcc ? (i & 1) : ((i >> 1) & 1), abort_flag, p.status);
            __syncwarp();                               // tcgen05.ld is warp-aligned
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + b * kAccStride;
            const int orow = tile * p.tile_rows + r;
            for (int n0 = 0; n0 < m; n0 += 16) {
                float v0[16];
                tmem_ld16(tbase + n0, v0);
                if (kHOut) {
                    float v1[16];
                    tmem_ld16(tbase + kUpCol + n0, v1);
                    const int pos = perm8(orow);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (n0 + j < m) {
                            const __half hv = __float2half_rn(silu_mul(v0[j], v1[j]));
                            if (__hisinf(hv)) set_status(p.status, SMOE_ERR_RANGE);
                            p.hout[(size_t)(off + n0 + j) * p.out_ld + pos] = hv;
                        }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (n0 + j < m) p.oout[(size_t)(off + n0 + j) * p.out_ld + orow] = v0[j];
                    if (kPair) {                       // the unit's second down tile, 128 rows on
                        float v1[16];
                        tmem_ld16(tbase + kUpCol + n0, v1);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (n0 + j < m) p.oout[(size_t)(off + n0 + j) * p.out_ld + orow + kTile] = v1[j];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&accempty[b]);
            if (kHOut && p.ready) {
                // this warp's 32 rows of h for the unit are stored: count them
                // (the stores ordered before the bulk tensor reads of the down kernel)
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.ready + u) : "memory");
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
    // the previous grid's completion is part of this one's (it has finished all
    // its units by now: every one of them fed some down unit)
    if (overlap) pdl_wait();
}

// Bucket-ordered, 8-block-permuted fp16 copy of the normed inputs:
// xperm[s] = perm(xn16[bucket_tok[s]]) for s < total, zero rows after.
__global__ void __launch_bounds__(256) k_gather_xperm(PrefillArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && a.ready) {  // the gate/up -> down counters and the unit counters start from zero
        for (int i = threadIdx.x; i < a.E; i += blockDim.x) a.ready[i] = 0;
        if (threadIdx.x < 2 && a.unit_ctr) a.unit_ctr[threadIdx.x] = 0;
    }
    const int s = blockIdx.x;
    const int total = a.offsets[*a.n_union];
    const int D = a.D;
    uint4 *dst = reinterpret_cast<uint4 *>(a.xperm + (size_t)s * D);
    if (s >= total) {
        for (int b = threadIdx.x; b < D / 8; b += blockDim.x) dst[b] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(a.xn16 + (size_t)a.bucket_tok[s] * D);
    for (int b = threadIdx.x; b < D / 8; b += blockDim.x) {
        const uint4 v = __ldcg(src + b);   // halves x0..x7 (two per word)
        uint4 o;
        // (x0,x4),(x1,x5),(x2,x6),(x3,x7)
        o.x = __byte_perm(v.x, v.z, 0x5410);
        o.y = __byte_perm(v.x, v.z, 0x7632);
        o.z = __byte_perm(v.y, v.w, 0x5410);
        o.w = __byte_perm(v.y, v.w, 0x7632);
        dst[b] = o;
    }
}

// ---- host side ----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once per process (threads that
// race on the first call store the same pointer).
EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_relaxed);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f, std::memory_order_relaxed);
        }
    }
    return f;
}

// 2-D map over a row-major [rows][cols] array of `esize`-byte elements.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * (cuuint64_t)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kPair, bool kQ2, bool kHOut, bool kOneAcc>
cudaError_t launch_tc(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap (&b)[4],
                      const TcParams &p, cudaStream_t s, int grid) {
    // More than half of an SM's shared memory: one CTA per SM.  Two resident
    // CTAs would each want all 512 TMEM columns, and the second would wait in
    // tcgen05.alloc until the first exits.
    const size_t smem = std::max<size_t>(Smem<kPair>::kBytes + 1024, 120 * 1024);
    static SmemLimits limits;
    const cudaError_t e = allow_dynamic_smem(k_prefill_tc<kPair, kQ2, kHOut, kOneAcc>, limits, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_prefill_tc<kPair, kQ2, kHOut, kOneAcc>, dim3(grid), dim3(kTcThreads), smem, s, true, a0, a1, b[0],
                         b[1], b[2], b[3], p);
}

}  // namespace

bool prefill_tc_supported(int D, int F) { return D % kTile == 0 && F % kTile == 0 && encode_fn() != nullptr; }

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    const int TK = a.T * a.K;
    CUtensorMap mg, mu, md, mx[4], mh[4];
    const int per_byte = a.q2 ? 4 : 2;                    // codes per byte
    bool ok = make_map(&mg, a.gq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.D / per_byte, (uint64_t)a.E * a.F,
                       kGpc * kKc / per_byte, kTile, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&mu, a.uq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.D / per_byte, (uint64_t)a.E * a.F,
                       kGpc * kKc / per_byte, kTile, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&md, a.dq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.F / per_byte, (uint64_t)a.E * a.D,
                       kGpc * kKc / per_byte, kTile, CU_TENSOR_MAP_SWIZZLE_NONE);
    for (int i = 0; i < 4 && ok; ++i)
        ok = make_map(&mx[i], a.xperm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.D, TK, kKc, 16 * (i + 1),
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
             make_map(&mh[i], a.hbuf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.F, TK, kKc, 16 * (i + 1),
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;

    cudaError_t e = launch_kernel(k_gather_xperm, dim3(TK), dim3(256), 0, s, true, a);
    if (e != cudaSuccess) return e;
    const int grid = a.num_sms;
    TcParams gu{};
    gu.n_tiles = a.F / kTile;
    gu.n_chunks = a.D / kKc;
    gu.rows_per_expert = a.F;
    gu.tile_rows = kTile;
    gu.a1_row = 0;
    gu.k_dim = a.D;
    gu.out_ld = a.F;
    gu.n_union = a.n_union;
    gu.union_ids = a.union_ids;
    gu.offsets = a.offsets;
    gu.s0 = a.gs; gu.b0 = a.gb; gu.s1 = a.us; gu.b1 = a.ub;
    auto a16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    gu.vec_scales = (a.D / kGroup) % 8 == 0 && a16(a.gs) && a16(a.gb) && a16(a.us) && a16(a.ub);
    gu.hout = a.hbuf;
    gu.ready = a.ready;
    gu.unit_ctr = a.unit_ctr;
    gu.status = a.status;
    // One accumulator buffer and three A stages pay for units of many stages
    // (235B shape, 4,096 tokens, µs per layer-chunk: gate/up with K = 4096,
    // 32 stages, 247.9 -> 237.8; down with K = 1536, 12 stages, a further ->
    // 235.5).  With units claimed from the counter they pay for the 30B SMOE-Q4
    // gate/up kernel too (K = 2048, 16 stages: 95.4 -> 94.4; under the static
    // unit list the lost epilogue overlap had cost more, 101.4 -> 102.6), but
    // not for its down kernel (K = 768, 6 stages: no change) nor for SMOE-Q2,
    // whose stages carry half the code bytes (30B prefill 19,468 -> 18,961 tok/s).
    const bool one_gu = a.D / (kGpc * kKc) >= (a.q2 ? 20 : 16), one_dn = a.F / (kGpc * kKc) >= 12;
    if (a.q2)
        e = one_gu ? launch_tc<true, true, true, true>(mg, mu, mx, gu, s, grid)
                   : launch_tc<true, true, true, false>(mg, mu, mx, gu, s, grid);
    else
        e = one_gu ? launch_tc<true, false, true, true>(mg, mu, mx, gu, s, grid)
                   : launch_tc<true, false, true, false>(mg, mu, mx, gu, s, grid);
    if (e != cudaSuccess) return e;
    TcParams dn = gu;
    dn.n_tiles = a.D / kTile;
    dn.n_chunks = a.F / kKc;
    dn.rows_per_expert = a.D;
    dn.tile_rows = kTile;
    dn.a1_row = 0;
    dn.k_dim = a.F;
    dn.out_ld = a.D;
    dn.s0 = a.ds; dn.b0 = a.db; dn.s1 = nullptr; dn.b1 = nullptr;
    dn.vec_scales = (a.F / kGroup) % 8 == 0 && a16(a.ds) && a16(a.db);
    dn.hout = nullptr;
    dn.oout = a.obuf;
    dn.ready_target = 4 * gu.n_tiles;
    dn.unit_ctr = a.unit_ctr ? a.unit_ctr + 1 : nullptr;
    if ((a.D / kTile) % 2 == 0) {
        // pairs of adjacent 128-row down tiles: each stage's activation tiles
        // feeds both, as gate and up share theirs
        const size_t tile_groups = (size_t)kTile * (a.F / kGroup);   // scale entries of 128 rows
        dn.n_tiles = a.D / (2 * kTile);
        dn.tile_rows = 2 * kTile;
        dn.a1_row = kTile;
        dn.s1 = a.ds + tile_groups;
        dn.b1 = a.db + tile_groups;
        dn.vec_scales = dn.vec_scales && a16(dn.s1) && a16(dn.b1);
        if (a.q2)
            return one_dn ? launch_tc<true, true, false, true>(md, md, mh, dn, s, grid)
                          : launch_tc<true, true, false, false>(md, md, mh, dn, s, grid);
        return one_dn ? launch_tc<true, false, false, true>(md, md, mh, dn, s, grid)
                      : launch_tc<true, false, false, false>(md, md, mh, dn, s, grid);
    }
    if (a.q2)
        return one_dn ? launch_tc<false, true, false, true>(md, md, mh, dn, s, grid)
                      : launch_tc<false, true, false, false>(md, md, mh, dn, s, grid);
    return one_dn ? launch_tc<false, false, false, true>(md, md, mh, dn, s, grid)
                  : launch_tc<false, false, false, false>(md, md, mh, dn, s, grid);
}

}  // namespace smoe

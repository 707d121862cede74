// union.cu -- per-chunk expert union and per-expert token buckets.
//
// "Optimizations" page, "Prefill Reads Each Expert Once, Not Once Per Token":
// a chunk of up to 64 tokens goes through a layer together and the layer's
// routed experts are deduplicated into a union that is read once per chunk.
// The buckets (which tokens, at which rank, use each union expert) are what
// lets the prefill FFN apply one read of an expert to all of its tokens.
//
// One CTA.  Every routing entry j = t*K + i sets bit j of its expert's
// membership mask (shared memory, 1024 bits per expert); an entry's place in
// its bucket is the number of lower set bits, so the buckets list tokens in
// ascending order, exactly and without sorting, and the result does not
// depend on thread timing.  Expert ids are scanned in ascending order to form
// the union.
#include "common.cuh"
#include "kernels.h"

namespace smoe {

namespace {

constexpr int kUnionThreads = 256;
constexpr int kMaskWords = (kMaxChunk * kMaxTopK) / 64;   // 16 x 64 bits

// Block-wide exclusive scan of two counters (256 threads).
__device__ __forceinline__ void scan2(int a, int b, int &ea, int &eb, int &ta, int &tb,
                                      int (*wt)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) { ia += va; ib += vb; }
    }
    if (lane == 31) { wt[warp][0] = ia; wt[warp][1] = ib; }
    __syncthreads();
    int pa = 0, pb = 0;
    ta = 0; tb = 0;
    for (int w = 0; w < kUnionThreads / 32; ++w) {
        if (w < warp) { pa += wt[w][0]; pb += wt[w][1]; }
        ta += wt[w][0]; tb += wt[w][1];
    }
    ea = pa + ia - a;
    eb = pb + ib - b;
}

__global__ void __launch_bounds__(kUnionThreads) k_expert_union(UnionArgs a) {
    __shared__ unsigned long long mask[kMaxExperts][kMaskWords];
    __shared__ int base[kMaxExperts];
    __shared__ int wt[kUnionThreads / 32][2];
    const int tid = threadIdx.x;
    const int N = a.T * a.K, E = a.E;

    pdl_wait();
    pdl_launch_dependents();

    // entries j = tid + 256 r, read once (N <= kMaxChunk * kMaxTopK = 4 * 256)
    constexpr int kPer = kMaxChunk * kMaxTopK / kUnionThreads;
    int ej[kPer];
    float wj[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int j = tid + kUnionThreads * r;
        ej[r] = j < N ? a.idx[j] : -1;
        wj[r] = j < N ? a.w[j] : 0.f;
    }
    const int words = (N + 63) >> 6;            // mask words in use
    for (int i = tid; i < E * kMaskWords; i += kUnionThreads)
        if ((i % kMaskWords) < words) (&mask[0][0])[i] = 0ull;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int j = tid + kUnionThreads * r;
        if (j >= N) break;
        const int e = ej[r];
        if (e >= 0 && e < E) atomicOr(&mask[e][j >> 6], 1ull << (j & 63));
        else set_status(a.status, SMOE_ERR_DEVICE);
    }
    __syncthreads();

    int cnt = 0;
    if (tid < E)
        for (int q = 0; q < words; ++q) cnt += __popcll(mask[tid][q]);
    int ebase, epos, total, nu;
    scan2(cnt, cnt > 0 ? 1 : 0, ebase, epos, total, nu, wt);
    if (tid < E) base[tid] = ebase;
    if (tid < E && cnt > 0) {
        a.union_ids[epos] = tid;
        a.offsets[epos] = ebase;
    }
    for (int u = nu + tid; u < E; u += kUnionThreads) a.union_ids[u] = -1;
    for (int u = nu + tid; u <= E; u += kUnionThreads) a.offsets[u] = total;
    if (tid == 0) *a.n_union = nu;
    __syncthreads();

#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int j = tid + kUnionThreads * r;
        if (j >= N) break;
        const int e = ej[r];
        int pos = -1;
        if (e >= 0 && e < E) {
            pos = base[e];
            const int wq = j >> 6;
            for (int q = 0; q < wq; ++q) pos += __popcll(mask[e][q]);
            pos += __popcll(mask[e][wq] & ((1ull << (j & 63)) - 1ull));
            a.bucket_tok[pos] = j / a.K;
            a.bucket_rank[pos] = j % a.K;
            a.bucket_w[pos] = wj[r];
        }
        if (a.slot_of) a.slot_of[j] = pos;
    }
    for (int p = total + tid; p < N; p += kUnionThreads) {
        a.bucket_tok[p] = -1;
        a.bucket_rank[p] = -1;
        a.bucket_w[p] = 0.f;
    }
}

}  // namespace

cudaError_t launch_expert_union(const UnionArgs &a, cudaStream_t s, bool pdl) {
    return launch_kernel(k_expert_union, dim3(1), dim3(kUnionThreads), 0, s, pdl, a);
}

}  // namespace smoe

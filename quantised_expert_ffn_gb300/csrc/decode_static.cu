// decode_static.cu -- smoe_moe_decode_noalloc: one decode token through a
// layer, with the scratch memory held in a fixed device array of this
// library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they need to run
// a layer: real-time serving loops whose latency budget rules out the
// device-wide synchronisation an allocation can cause, services that reserve
// all their device memory at start-up and must not grow later, and plug-ins
// loaded into a host program that owns every byte of device memory through
// its own pool.  This entry point lets them decode without a workspace: the
// scratch (status word, route and barrier counters, logits, expert ids and
// weights, the gate/up activations) lives in `g_decode_scratch`, a
// file-scope __device__ array of kStaticScratchBytes that every GPU which
// loads the library holds until the process exits.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 512 * 1024;   // largest layer this entry point takes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch for each device, looked up once with that
// device current.  In host code the array's name is only a host-side stand-in,
// never a device address.  Threads that race on a first call store the same
// value.
std::atomic<void *> g_scratch_ptr[kMaxDevices];

int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMOE_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return SMOE_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_relaxed);
    }
    *out = p;
    return SMOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

static_assert(kStaticScratchBytes == SMOE_DECODE_NOALLOC_MAX_BYTES, "header and library disagree");

extern "C" {

int smoe_moe_decode_noalloc(const smoe_layer *layer, const smoe_bf16 *x, smoe_bf16 *y,
                            int32_t *idx_out_opt, float *w_out_opt, smoe_stream stream) {
    const size_t need = smoe_workspace_bytes(layer, 1);
    if (need == 0) return layer ? SMOE_ERR_UNSUPPORTED : SMOE_ERR_INVALID_ARG;
    if (need > kStaticScratchBytes) return SMOE_ERR_WORKSPACE;   // layer too large for the fixed scratch
    // the arguments smoe_moe_decode would reject, rejected before the scratch is touched
    if (!x || !y || !aligned16(x) || !aligned16(y)) return SMOE_ERR_INVALID_ARG;
    void *ws = nullptr;
    const int st = scratch_for_current_device(&ws);
    if (st != SMOE_OK) return st;
    // the array keeps the previous call's contents: zero the status word and counters
    const size_t clear = smoe::ws_head_bytes();
    if (clear > kStaticScratchBytes) return SMOE_ERR_WORKSPACE;
    if (cudaMemsetAsync(ws, 0, clear, (cudaStream_t)stream) != cudaSuccess) return SMOE_ERR_CUDA;
    return smoe_moe_decode(layer, x, y, idx_out_opt, w_out_opt, nullptr, ws, kStaticScratchBytes, stream);
}

int smoe_moe_decode_noalloc_status(int32_t *status_host, smoe_stream stream) {
    if (!status_host) return SMOE_ERR_INVALID_ARG;
    void *ws = nullptr;
    const int st = scratch_for_current_device(&ws);
    if (st != SMOE_OK) return st;
    return smoe_read_device_status(ws, status_host, stream);
}

}  // extern "C"

// dense.h -- launchers of the dense bf16 matvec and the SMOE-Q4 quantiser
// (dense.cu; internal to libsmoe.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smoe {

// y[r] = sum_c w[r][c] x[c]; w bf16 [rows][cols] and x bf16 [cols] 16-byte
// aligned, cols a multiple of 8 and at most 8192; y fp32 [rows].
cudaError_t launch_dense_matvec(const uint16_t *w, const uint16_t *x, int rows, int cols, float *y,
                                cudaStream_t s);

// SMOE-Q4 (bits 4) or SMOE-Q2 (bits 2) codes, scales and biases of n_groups
// consecutive groups of 64 bf16 weights (w and codes 16-byte aligned, scale
// and bias 2-byte aligned).
cudaError_t launch_quantize(const uint16_t *w, long long n_groups, int bits, uint8_t *codes, uint16_t *scale,
                            uint16_t *bias, cudaStream_t s);

int device_sm_count();

}  // namespace smoe

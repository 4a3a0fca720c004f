// Internal launch interface between the C-ABI layer (convrot_api.cu) and the
// kernels. Arguments here are already validated.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace convrot {

struct PackArgs {
    const float *x;   // [rows, ldx]
    int64_t ldx;
    int64_t rows;
    int32_t k;
    int32_t log4g;    // n with G = 4^n
    void *q;          // [rows, ldq] codes
    int64_t ldq;
    int32_t kpad;     // columns [k, kpad) of q are written as zero
    float *scale;     // [rows]
    int32_t bf16;     // 0: int8 codes, 1: bf16 codes
    int32_t *dev_status;  // receives CONVROT_ERR_TIMEOUT if a bounded wait runs out (may be null)
};

cudaError_t launch_pack(const PackArgs &a, cudaStream_t stream);

struct GemmArgs {
    const void *qx;    // [m, ldqx] codes
    int64_t ldqx;
    const void *qw;    // [n, ldqw] codes
    int64_t ldqw;
    int64_t m, n;
    int32_t kpad;      // K extent read (multiple of 128, zero-padded past k)
    const float *sx;   // [m]
    const float *sw;   // [n]
    const float *bias; // [n] or null
    float *y;          // [m, ldy] (fp32 output) or null
    int32_t *a;        // [m, ldy] (raw int32 output) or null
    int64_t ldy;
    int32_t *dev_status;
};

cudaError_t launch_gemm_imma(const GemmArgs &a, cudaStream_t stream);
cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t stream);

}  // namespace convrot

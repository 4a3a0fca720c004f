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

// Codes and scales of rows whose rotation was applied by the GEMM's epilogue
// (GemmArgs::rot_digits): H_rot [rows, ldh] fp32 (unnormalized, 2^log4g times
// the rotation) and rowmax [rows] (its absmax, fp32 bits) -> q, scale as the
// pack writes them. Columns go from the last to the first, the order in which
// the GEMM left them in L2; each H_rot line is discarded from L2 once read.
cudaError_t launch_requant(const float *h_rot, int64_t ldh, const uint32_t *rowmax, int64_t rows, int32_t k,
                           int32_t log4g, void *q, int64_t ldq, float *scale, int32_t bf16, cudaStream_t stream);

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
    int32_t act;       // convrot_activation applied to Y (not to raw int32 output)
    int32_t i8;        // 1: qx and qw hold int8 codes; 0: bf16 codes
    // > 0: rotate the output in the epilogue along its rot_digits lowest base-4 digits
    // (pair kernel, bf16 codes, n % 256 == 0), fold each row's absmax into rot_rowmax
    // (fp32 bits, atomicMax; zeroed by the caller) and store the rotated values to `a`
    int32_t rot_digits;
    uint32_t *rot_rowmax;
    // LoRA side branch (bf16 codes only): Y += T_ext B_ext^T before the activation
    int32_t lora_r;          // 0: none
    const void *lora_t;      // T_ext bf16 [m, lora_ldt]
    int64_t lora_ldt;
    const void *lora_b;      // B_ext bf16 [n, lora_ldb]
    int64_t lora_ldb;
};

// K extent of the LoRA chunk: 3 r rounded up to 64.
int lora_cols(int r);
cudaError_t launch_lora_prepare(const float *B, int64_t n, int32_t r, int64_t ldb, float scale, void *out,
                                int64_t lde, cudaStream_t stream);
cudaError_t launch_lora_prepare_down(const float *A, int32_t r, int32_t k, int64_t lda, float *out, int64_t ldo,
                                     cudaStream_t stream);
cudaError_t launch_lora_down(const float *X, int64_t m, int32_t k, int64_t ldx, const float *A_ext, int32_t r,
                             int64_t lda, void *t, int64_t ldt, int32_t *dev_status, cudaStream_t stream);

// One CTA waiting on an mbarrier through the kernels' bounded wait (arrive = 0:
// nothing arrives and it reports CONVROT_ERR_TIMEOUT after limit_ns).
cudaError_t launch_wait_check(int32_t *dev_status, uint64_t limit_ns, int arrive, cudaStream_t stream);

// GELU, erf or tanh form (convrot_activation), on the epilogue's fp32 value.
// The tanh form is evaluated through its exact identity
// 0.5 v (1 + tanh(u)) = v / (1 + e^(-2u)), u = sqrt(2/pi) (v + 0.044715 v^3):
// one fast exponential and one fast division. Its relative error, a few 2^-22
// over the range where the result is not negligible, stays inside the
// epilogue's tolerance. (As v -> -inf, e^(-2u) overflows and __fdividef
// returns 0; the result is then -0 or 0, as GELU's value there rounds to.)
// The erf form uses Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (|error in erf| <= 1.5e-7): erf(x) = 1 - t (a1 + t (a2 + t (a3
// + t (a4 + t a5)))) e^(-x^2), t = 1 / (1 + p x), for x >= 0, odd in x. It is
// call-free, so the epilogue can apply it in place.
__device__ __forceinline__ float erf_as7126(float x)
{
    const float ax = fabsf(x);
    const float t = __fdividef(1.0f, fmaf(0.3275911f, ax, 1.0f));
    const float poly =
        t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f),
                 0.254829592f);
    return copysignf(fmaf(-poly, __expf(-ax * ax), 1.0f), x);
}

__device__ __forceinline__ float apply_act(float v, int act)
{
    if (act == 1) return 0.5f * v * (1.0f + erf_as7126(v * 0.70710678118654752f));
    if (act == 2) {
        const float u2 = -1.5957691216057308f * fmaf(0.044715f * v, v * v, v);  // -2u
        return __fdividef(v, 1.0f + __expf(u2));
    }
    return v;
}

template <int kAct>
__device__ __forceinline__ float apply_act_t(float v)
{
    return kAct == 0 ? v : apply_act(v, kAct);
}

cudaError_t launch_gemm_imma(const GemmArgs &a, cudaStream_t stream);
cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t stream);

}  // namespace convrot

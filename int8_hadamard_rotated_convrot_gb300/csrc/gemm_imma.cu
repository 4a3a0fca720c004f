// I8 x I8 -> I32 GEMM on the warp-level integer MMA (mma.sync m16n8k32 s8),
// with the reconstruction fused into the epilogue.
//
// Computes, from "Runtime activation quantization" on the page "INT8 Convrot
// Safetensors" (stable-diffusion.cpp docs):
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]            (exact, int32)
//   Y[r, o] = A[r, o] * s_x[r] * s_w[o] + b[o]        (fp32)
// Both operands are K-major (Y = X W^T), so this is a "TN" GEMM.
//
// sm_103a has no tcgen05 integer MMA kind, so the integer tensor-core path is
// this warp-level instruction. The int32 accumulation makes it bit-exact by
// construction. CTA tile 128 x 128 x 64, 8 warps (2 x 4, 64 x 32 per warp),
// a 4-stage cp.async ring in XOR-swizzled shared memory, ldmatrix fragments.
#include <cstdint>

#include "internal.h"

namespace convrot {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int TILE_BYTES = BM * BK;  // == BN * BK
constexpr int SMEM_BYTES = STAGES * 2 * TILE_BYTES;

// Byte offset of 16-byte chunk `c` (0..3) of row `r` in a 64-byte-row tile;
// the XOR keeps the 8 rows one ldmatrix reads in 8 different bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    return static_cast<uint32_t>(r * BK + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool kRawInt32>
__global__ void __launch_bounds__(THREADS) gemm_imma_kernel(GemmArgs g)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
    const int8_t *qx = static_cast<const int8_t *>(g.qx);
    const int8_t *qw = static_cast<const int8_t *>(g.qw);
    const int ktiles = g.kpad / BK;

    auto load_stage = [&](int stage, int kt) {
        const uint32_t sa = smem_base + stage * 2 * TILE_BYTES;
        const uint32_t sb = sa + TILE_BYTES;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + i * THREADS;  // 0..511: row = idx / 4, chunk = idx % 4
            const int r = idx >> 2, c = idx & 3;
            const int64_t gr = m0 + r, gn = n0 + r;
            const bool va = gr < g.m, vb = gn < g.n;
            const int8_t *pa = qx + (va ? gr : 0) * g.ldqx + kt * BK + c * 16;
            const int8_t *pb = qw + (vb ? gn : 0) * g.ldqw + kt * BK + c * 16;
            cp_async16(sa + swz(r, c), pa, va);
            cp_async16(sb + swz(r, c), pb, vb);
        }
    };

    int32_t acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles) load_stage(s, s);
        asm volatile("cp.async.commit_group;");
    }

    for (int kt = 0; kt < ktiles; ++kt) {
        asm volatile("cp.async.wait_group %0;" ::"n"(STAGES - 2));
        __syncthreads();
        {
            const int nk = kt + STAGES - 1;
            if (nk < ktiles) load_stage(nk % STAGES, nk);
            asm volatile("cp.async.commit_group;");
        }
        const int stage = kt % STAGES;
        const uint32_t sa = smem_base + stage * 2 * TILE_BYTES;
        const uint32_t sb = sa + TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
            uint32_t af[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = wm * 64 + i * 16 + (lane & 15);
                const int c = kk * 2 + (lane >> 4);
                ldsm_x4(sa + swz(r, c), af[i][0], af[i][1], af[i][2], af[i][3]);
            }
            uint32_t bf[4][2];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int r = wn * 32 + jj * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int c = kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(sb + swz(r, c), bf[2 * jj][0], bf[2 * jj][1], bf[2 * jj + 1][0],
                        bf[2 * jj + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
    }
    asm volatile("cp.async.wait_group 0;");

    // epilogue: c0, c1 -> (row g, cols 2t, 2t+1); c2, c3 -> (row g + 8, same cols)
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t r = m0 + wm * 64 + i * 16 + gq + h * 8;
            if (r >= g.m) continue;
            float sxr = 0.f;
            if constexpr (!kRawInt32) sxr = g.sx[r];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t c = n0 + wn * 32 + j * 8 + tq * 2;
                if (c >= g.n) continue;  // n is even-aligned per pair only if c + 1 < n
                const int32_t a0 = acc[i][j][2 * h], a1 = acc[i][j][2 * h + 1];
                if constexpr (kRawInt32) {
                    int32_t *dst = g.a + r * g.ldy + c;
                    if (c + 1 < g.n) {
                        *reinterpret_cast<int2 *>(dst) = make_int2(a0, a1);
                    } else {
                        dst[0] = a0;
                    }
                } else {
                    const float b0 = g.bias ? g.bias[c] : 0.f;
                    const float y0 = apply_act(fmaf(static_cast<float>(a0) * sxr, g.sw[c], b0), g.act);
                    float *dst = g.y + r * g.ldy + c;
                    if (c + 1 < g.n) {
                        const float b1 = g.bias ? g.bias[c + 1] : 0.f;
                        const float y1 = apply_act(fmaf(static_cast<float>(a1) * sxr, g.sw[c + 1], b1), g.act);
                        *reinterpret_cast<float2 *>(dst) = make_float2(y0, y1);
                    } else {
                        dst[0] = y0;
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm_imma(const GemmArgs &g, cudaStream_t stream)
{
    if (g.m == 0 || g.n == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((g.n + BN - 1) / BN),
                    static_cast<unsigned>((g.m + BM - 1) / BM));
    if ((g.m + BM - 1) / BM > 65535) return cudaErrorInvalidConfiguration;
    if (g.a) {
        auto k = gemm_imma_kernel<true>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        k<<<grid, THREADS, SMEM_BYTES, stream>>>(g);
    } else {
        auto k = gemm_imma_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        k<<<grid, THREADS, SMEM_BYTES, stream>>>(g);
    }
    return cudaGetLastError();
}

}  // namespace convrot

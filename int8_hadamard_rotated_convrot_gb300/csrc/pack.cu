// Fused pack kernel: group-wise rotation, row absmax, quantization.
//
// Implements, for each row of X, the steps the page "INT8 Convrot Safetensors"
// (stable-diffusion.cpp docs) gives in "How INT8 convrot works" and
// "Runtime activation quantization" (the offline "Weight quantization" uses
// the same formulas on the rows of W):
//
//   X_rot = X R        R = normalized Kronecker power of H4 per group of G
//   s     = max |X_rot| / 127 over the whole row
//   Q     = clamp(round_half_away(X_rot / s), -127, 127)
//
// HBM-bound: X is read once (4 B/element) and the codes written once (1 or
// 2 B/element). One CTA, or one thread-block cluster for rows longer than a
// CTA holds, owns a row, keeps it in registers, and never stages it through
// memory.
//
// Register layout. The row is split into chunks of 32 lanes x S slots x 4
// floats (128*S floats). Lane l, slot j of a warp holds the float4 with quad
// index q = chunk*32*S + j*32 + l, so every warp-wide load or store touches
// consecutive addresses (512 B per instruction for fp32). The element index
// inside a group, e = 4q + c (c = float4 component), has base-4 digits
//   d0 = c, d1 = lane bits 0-1, d2 = lane bits 2-3,
//   d3 = (lane bit 4, slot bit 0), d4 = slot bits 1-2, d5 = slot bits 3-4,
// so a group of G = 4^n never spans more than one warp: S = 1 for G <= 64,
// 2 for G = 256, 8 for G = 1024, 32 for G = 4096 (then 128 floats a thread).
//
// One radix-4 stage along a digit replaces every 4-tuple (x_0..x_3) that
// differs only in that digit by H4 x, i.e. (H4 rows are the printed matrix
// / 2, a minus sign where row + column = 3)
//   y_D = ((x_D + x_{D^1}) + (x_{D^2} - x_{D^3})) / 2.
// Applying it along every digit of the in-group index is R_G applied to the
// group, by the mixed-product property of the Kronecker product. Partners in
// another lane come from warp shuffles, partners in another slot or
// component are registers.
#include <cuda_bf16.h>

#include "internal.h"

namespace convrot {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// y_D = ((x_D + x_{D^1}) + (x_{D^2} - x_{D^3})) / 2 given the three partners.
__device__ __forceinline__ float h4_out(float x, float p1, float p2, float p3)
{
    return 0.5f * ((x + p1) + (p2 - p3));
}

__device__ __forceinline__ void h4_inplace(float &a, float &b, float &c, float &d)
{
    const float ya = h4_out(a, b, c, d);
    const float yb = h4_out(b, a, d, c);
    const float yc = h4_out(c, d, a, b);
    const float yd = h4_out(d, c, b, a);
    a = ya;
    b = yb;
    c = yc;
    d = yd;
}

// Digit held by two lane bits (masks m1 = low bit, m2 = high bit).
__device__ __forceinline__ float lane_digit(float x, int m1, int m2)
{
    const float p1 = __shfl_xor_sync(kFull, x, m1);
    const float p2 = __shfl_xor_sync(kFull, x, m2);
    const float p3 = __shfl_xor_sync(kFull, x, m1 | m2);
    return h4_out(x, p1, p2, p3);
}

__device__ __forceinline__ float4 lane_digit4(float4 v, int m1, int m2)
{
    return make_float4(lane_digit(v.x, m1, m2), lane_digit(v.y, m1, m2),
                       lane_digit(v.z, m1, m2), lane_digit(v.w, m1, m2));
}

__device__ __forceinline__ float4 f4_h4(float4 x, float4 p1, float4 p2, float4 p3)
{
    return make_float4(h4_out(x.x, p1.x, p2.x, p3.x), h4_out(x.y, p1.y, p2.y, p3.y),
                       h4_out(x.z, p1.z, p2.z, p3.z), h4_out(x.w, p1.w, p2.w, p3.w));
}

__device__ __forceinline__ float4 shfl_xor4(float4 v, int m)
{
    return make_float4(__shfl_xor_sync(kFull, v.x, m), __shfl_xor_sync(kFull, v.y, m),
                       __shfl_xor_sync(kFull, v.z, m), __shfl_xor_sync(kFull, v.w, m));
}

__device__ __forceinline__ float absmax4(float m, float4 v)
{
    return fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
}

// Round half away from zero, clamp to [-127, 127].
__device__ __forceinline__ int code_of(float x, float s)
{
    float v = roundf(__fdiv_rn(x, s));
    v = fminf(fmaxf(v, -127.0f), 127.0f);
    return static_cast<int>(v);
}

__device__ __forceinline__ uint32_t cluster_smem_addr(const void *p, uint32_t rank)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 128 floats a thread (S = 32) need up to 255 registers: at most 8 warps.
template <int S>
constexpr int kPackMaxThreads = S == 32 ? 256 : 1024;

template <int S, int CPT, bool kBf16>
__global__ void __launch_bounds__(kPackMaxThreads<S>) pack_kernel(PackArgs a, int cl, int64_t row0)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int64_t row = row0 + blockIdx.x / cl;
    const int cr = blockIdx.x % cl;  // rank inside the cluster (cluster dims are (cl,1,1))

    const int chunk_quads = 32 * S;
    const int n_chunks = a.kpad / (4 * chunk_quads);  // kpad is a multiple of 128*S
    const int per_cta = (n_chunks + cl - 1) / cl;
    const int kq = a.k >> 2;           // quads that hold data
    const int kpq = a.kpad >> 2;       // quads written (data + zero pad)

    const float4 *xrow = reinterpret_cast<const float4 *>(a.x + row * a.ldx);
    float4 v[CPT][S];
    int chunk[CPT];

#pragma unroll
    for (int t = 0; t < CPT; ++t) {
        const int local = warp + nw * t;
        chunk[t] = (local < per_cta) ? cr * per_cta + local : n_chunks;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const int q = chunk[t] * chunk_quads + j * 32 + lane;
            v[t][j] = (chunk[t] < n_chunks && q < kq) ? __ldcs(xrow + q)
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    const int n = a.log4g;
    // digit 0: the float4 components
#pragma unroll
    for (int t = 0; t < CPT; ++t)
#pragma unroll
        for (int j = 0; j < S; ++j) h4_inplace(v[t][j].x, v[t][j].y, v[t][j].z, v[t][j].w);
    // digits 1 and 2: lane bits 0-1 and 2-3
    if (n > 1) {
#pragma unroll
        for (int t = 0; t < CPT; ++t)
#pragma unroll
            for (int j = 0; j < S; ++j) v[t][j] = lane_digit4(v[t][j], 1, 2);
    }
    if (n > 2) {
#pragma unroll
        for (int t = 0; t < CPT; ++t)
#pragma unroll
            for (int j = 0; j < S; ++j) v[t][j] = lane_digit4(v[t][j], 4, 8);
    }
    // digit 3: lane bit 4 (low) and slot bit 0 (high)
    if constexpr (S >= 2) {
        if (n > 3) {
#pragma unroll
            for (int t = 0; t < CPT; ++t) {
                float4 sh[S];
#pragma unroll
                for (int j = 0; j < S; ++j) sh[j] = shfl_xor4(v[t][j], 16);
                float4 nv[S];
#pragma unroll
                for (int j = 0; j < S; ++j) nv[j] = f4_h4(v[t][j], sh[j], v[t][j ^ 1], sh[j ^ 1]);
#pragma unroll
                for (int j = 0; j < S; ++j) v[t][j] = nv[j];
            }
        }
    }
    // digit 4: slot bits 1-2
    if constexpr (S >= 8) {
        if (n > 4) {
#pragma unroll
            for (int t = 0; t < CPT; ++t) {
                float4 nv[S];
#pragma unroll
                for (int j = 0; j < S; ++j)
                    nv[j] = f4_h4(v[t][j], v[t][j ^ 2], v[t][j ^ 4], v[t][j ^ 6]);
#pragma unroll
                for (int j = 0; j < S; ++j) v[t][j] = nv[j];
            }
        }
    }
    // digit 5: slot bits 3-4
    if constexpr (S >= 32) {
        if (n > 5) {
#pragma unroll
            for (int t = 0; t < CPT; ++t) {
                float4 nv[S];
#pragma unroll
                for (int j = 0; j < S; ++j)
                    nv[j] = f4_h4(v[t][j], v[t][j ^ 8], v[t][j ^ 16], v[t][j ^ 24]);
#pragma unroll
                for (int j = 0; j < S; ++j) v[t][j] = nv[j];
            }
        }
    }

    // absmax over the whole rotated row (padding lanes hold zeros)
    float m = 0.0f;
#pragma unroll
    for (int t = 0; t < CPT; ++t)
#pragma unroll
        for (int j = 0; j < S; ++j) m = absmax4(m, v[t][j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));

    __shared__ float warp_max[32];
    __shared__ float cta_max;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        float mm = (lane < nw) ? warp_max[lane] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, off));
        if (lane == 0) cta_max = mm;
    }
    __syncthreads();
    float amax = cta_max;
    if (cl > 1) {
        cluster_sync_all();  // every CTA's cta_max is written
        for (int r = 0; r < cl; ++r) amax = fmaxf(amax, ld_cluster_f32(cluster_smem_addr(&cta_max, r)));
    }

    const float s = amax / 127.0f;
    const bool zero_row = !(s > 0.0f);
    if (cr == 0 && threadIdx.x == 0) a.scale[row] = s;

#pragma unroll
    for (int t = 0; t < CPT; ++t) {
        if (chunk[t] >= n_chunks) continue;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const int q = chunk[t] * chunk_quads + j * 32 + lane;
            if (q >= kpq) continue;
            int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
            if (!zero_row && q < kq) {
                c0 = code_of(v[t][j].x, s);
                c1 = code_of(v[t][j].y, s);
                c2 = code_of(v[t][j].z, s);
                c3 = code_of(v[t][j].w, s);
            }
            if constexpr (kBf16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(static_cast<float>(c0), static_cast<float>(c1));
                __nv_bfloat162 hi = __floats2bfloat162_rn(static_cast<float>(c2), static_cast<float>(c3));
                uint2 packed;
                packed.x = *reinterpret_cast<uint32_t *>(&lo);
                packed.y = *reinterpret_cast<uint32_t *>(&hi);
                reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.q) + row * a.ldq)[q] = packed;
            } else {
                const uint32_t packed = (static_cast<uint32_t>(c0) & 0xffu) |
                                        ((static_cast<uint32_t>(c1) & 0xffu) << 8) |
                                        ((static_cast<uint32_t>(c2) & 0xffu) << 16) |
                                        (static_cast<uint32_t>(c3) << 24);
                reinterpret_cast<uint32_t *>(static_cast<int8_t *>(a.q) + row * a.ldq)[q] = packed;
            }
        }
    }
    if (cl > 1) cluster_sync_all();  // no CTA leaves while another may still read its cta_max
}

struct PackPlan {
    int S, cpt, warps, cl;
};

// Chooses slots per chunk S from G, then the smallest cluster and the
// fewest floats per thread that keep a CTA at <= 16 warps (<= 32 if needed).
PackPlan plan_pack(int log4g, int kpad)
{
    PackPlan p{};
    p.S = log4g <= 3 ? 1 : (log4g == 4 ? 2 : (log4g == 5 ? 8 : 32));
    static const int opts1[] = {1, 2, 4, 8}, opts2[] = {1, 2, 4}, opts8[] = {1}, opts32[] = {1};
    const int *opts = p.S == 1 ? opts1 : (p.S == 2 ? opts2 : (p.S == 8 ? opts8 : opts32));
    const int n_opts = p.S == 1 ? 4 : (p.S == 2 ? 3 : 1);
    const int pref_warps = p.S == 32 ? 8 : 16;
    const int max_warps = p.S == 32 ? 8 : 32;
    const int n_chunks = kpad / (128 * p.S);
    for (int limit : {pref_warps, max_warps}) {
        for (int cl = 1; cl <= 8; ++cl) {
            const int per_cta = (n_chunks + cl - 1) / cl;
            for (int i = 0; i < n_opts; ++i) {
                const int warps = (per_cta + opts[i] - 1) / opts[i];
                if (warps <= limit) {
                    p.cpt = opts[i];
                    p.warps = warps;
                    p.cl = cl;
                    return p;
                }
            }
        }
    }
    p.cpt = 0;  // no plan (cannot happen for kpad <= 8 CTAs' worth)
    return p;
}

template <int S, int CPT, bool kBf16>
cudaError_t launch_one(const PackArgs &a, const PackPlan &p, cudaStream_t stream)
{
    const int64_t max_rows = (int64_t{1} << 31) / p.cl - 1;
    for (int64_t r0 = 0; r0 < a.rows; r0 += max_rows) {
        const int64_t rows = a.rows - r0 < max_rows ? a.rows - r0 : max_rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(rows * p.cl), 1, 1);
        cfg.blockDim = dim3(static_cast<unsigned>(32 * p.warps), 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.cl);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, pack_kernel<S, CPT, kBf16>, a, p.cl, r0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <bool kBf16>
cudaError_t dispatch(const PackArgs &a, const PackPlan &p, cudaStream_t stream)
{
    switch (p.S * 100 + p.cpt) {
    case 101: return launch_one<1, 1, kBf16>(a, p, stream);
    case 102: return launch_one<1, 2, kBf16>(a, p, stream);
    case 104: return launch_one<1, 4, kBf16>(a, p, stream);
    case 108: return launch_one<1, 8, kBf16>(a, p, stream);
    case 201: return launch_one<2, 1, kBf16>(a, p, stream);
    case 202: return launch_one<2, 2, kBf16>(a, p, stream);
    case 204: return launch_one<2, 4, kBf16>(a, p, stream);
    case 801: return launch_one<8, 1, kBf16>(a, p, stream);
    case 3201: return launch_one<32, 1, kBf16>(a, p, stream);
    default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace

cudaError_t launch_pack(const PackArgs &a, cudaStream_t stream)
{
    if (a.rows == 0) return cudaSuccess;
    const PackPlan p = plan_pack(a.log4g, a.kpad);
    if (p.cpt == 0) return cudaErrorInvalidConfiguration;
    return a.bf16 ? dispatch<true>(a, p, stream) : dispatch<false>(a, p, stream);
}

}  // namespace convrot

// Fused pack kernel: group-wise rotation, row absmax, quantization.
//
// Implements, for each row of X, the steps the page "INT8 Convrot Safetensors"
// (stable-diffusion.cpp docs) gives in "How INT8 convrot works" and
// "Runtime activation quantization" (the offline "Weight quantization" uses
// the same formulas on the rows of W):
//
//   X_rot = X R        R = normalized Kronecker power of H4 per group of G = 4^n
//   s     = max |X_rot| / 127 over the whole row
//   Q     = clamp(round_half_away(X_rot / s), -127, 127)
//
// HBM-bound: X is read once (4 B/element) and the codes written once (1 or
// 2 B/element).
//
// How R_G is applied. The printed H4 is (1/2) D1 P W1 D1 with W1 = [[1,1],
// [1,-1]] (x) [[1,1],[1,-1]], D1 = diag(1,1,1,-1) and P the swap of entries 1
// and 2 (e.g. row 1 of W1 D1 is (1,-1,1,1), which is row 2 of 2*H4). By the
// mixed-product property of the Kronecker product,
//   R_G = H4^(x)n = 2^-n * D * Pi * W * D
// where W is the Walsh-Hadamard matrix of size G (radix-2 butterflies over all
// 2n index bits), D = diag((-1)^(number of base-4 digits of the index equal
// to 3)) and Pi swaps the two bits inside every base-4 digit of the index. So
// the kernel flips input signs by D, runs plain Walsh-Hadamard butterflies
// (adds and subtracts only), applies D again at the output (folded into the
// quantization multiplier; D is invariant under Pi) and writes each value to
// its Pi-permuted position. The factor 2^-n is exact and folded into the scale.
//
// Register layout. A thread holds S float4 "slots". In a tile of 2^LANES
// consecutive threads, thread l, slot j holds the float4 with quad index
//   q = tile * S * 2^LANES + j * 2^LANES + l,
// so a warp-wide access of one slot touches 2^LANES consecutive quads per
// tile. The in-group quad index is q mod G/4; its low bits come from the lane
// (butterflies by warp shuffle) and the rest from the slot (register
// butterflies). The float4 component is digit 0 of the in-group index.
//
// Launch shape. One kernel, loading registers straight from global memory
// with streaming 16-byte loads: a CTA of about 128 threads owns whole rows
// (96 threads per row at K = 3072), and many CTAs per SM overlap their
// load / compute / store phases. Rows longer than 512 threads hold are split
// over a thread-block cluster, whose CTAs exchange their partial row maxima
// through distributed shared memory. (Persistent variants that stream rows
// through a shared-memory ring with bulk copies, with or without a
// shared-memory transpose in place of the lane shuffles, measured no faster
// on any of the DiT shapes, so they were dropped.)
#include <cuda_bf16.h>

#include "../../include/convrot.h"
#include "internal.h"

namespace convrot {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kSign = 0x80000000u;

template <int S>
constexpr int kMaxThreads = S >= 32 ? 256 : 512;

// Pi on an in-group quad index of `bits` bits: swap the two bits of every
// base-4 digit (quad-index bit pairs (0,1), (2,3), ...).
__device__ __forceinline__ uint32_t swap_digit_bits(uint32_t g, int bits)
{
    const uint32_t mask = (1u << bits) - 1u;
    return (((g & 0x55555555u) << 1) | ((g >> 1) & 0x55555555u)) & mask;
}

// Sign of D from the in-group quad index (digits 1..n-1; digit 0 is the component).
__device__ __forceinline__ uint32_t quad_sign(uint32_t g)
{
    return (__popc(g & (g >> 1) & 0x55555555u) & 1) ? kSign : 0u;
}

__device__ __forceinline__ float xor_sign(float x, uint32_t m) { return __uint_as_float(__float_as_uint(x) ^ m); }

// Round half away from zero. For a >= 0, floor(a + 1/2) is the answer; the sum
// rounded toward zero has the same floor (it never drops below an integer the
// exact sum reaches), and it cannot round up across an integer the way a
// round-to-nearest sum can just below 1/2.
__device__ __forceinline__ float round_half_away(float v)
{
    return copysignf(truncf(__fadd_rz(fabsf(v), 0.5f)), v);
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

// Where one thread's slots sit along a row, and everything about them that
// is the same for every row the thread handles: which slots hold data, the
// sign of D at each slot, and how far Pi moves each slot's output.
template <int LANES, int S>
struct Place {
    int l_in;          // lane inside the tile
    int q0;            // quad index of slot 0 along the row
    int lbg, sbg;      // lane / slot bits inside a group
    int qbits;         // in-group quad-index bits (2n - 2)
    uint32_t valid;    // bit j: slot j holds data (quad < k/4)
    uint32_t sgn[S];   // sign of D at slot j (0 or kSign), digit 0 excluded
    int delta[S];      // Pi: output quad = input quad + delta[j]

    __device__ __forceinline__ Place(int t_row, int n, int kq)
    {
        l_in = t_row & ((1 << LANES) - 1);
        q0 = (t_row >> LANES) * (S << LANES) + l_in;
        qbits = 2 * n - 2;
        lbg = qbits < LANES ? qbits : LANES;
        sbg = qbits - lbg;
        const uint32_t gmask = (1u << qbits) - 1u;
        valid = 0;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const int q = quad(j);
            if (q < kq) valid |= 1u << j;
            // a tile is a whole number of groups, so the in-group index depends on (lane, slot) only
            const uint32_t g = static_cast<uint32_t>(q) & gmask;
            sgn[j] = quad_sign(g);
            delta[j] = static_cast<int>(swap_digit_bits(g, qbits)) - static_cast<int>(g);
        }
    }
    __device__ __forceinline__ int quad(int j) const { return q0 + j * (1 << LANES); }
};

// D, then the Walsh-Hadamard butterflies over all 2n in-group bits.
template <int LANES, int S>
__device__ __forceinline__ void rotate(float4 (&v)[S], const Place<LANES, S> &pl)
{
#pragma unroll
    for (int j = 0; j < S; ++j) {
        const uint32_t sg = pl.sgn[j];
        v[j].x = xor_sign(v[j].x, sg);
        v[j].y = xor_sign(v[j].y, sg);
        v[j].z = xor_sign(v[j].z, sg);
        v[j].w = xor_sign(v[j].w, sg ^ kSign);  // component 3: digit 0 equal to 3
        const float s0 = v[j].x + v[j].y, d0 = v[j].x - v[j].y;
        const float s1 = v[j].z + v[j].w, d1 = v[j].z - v[j].w;
        v[j] = make_float4(s0 + s1, d0 + d1, s0 - s1, d0 - d1);
    }
#pragma unroll
    for (int b = 0; b < LANES; ++b) {
        if (b >= pl.lbg) break;
        const float sg = ((pl.l_in >> b) & 1) ? -1.0f : 1.0f;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            v[j].x = fmaf(sg, v[j].x, __shfl_xor_sync(kFull, v[j].x, 1 << b));
            v[j].y = fmaf(sg, v[j].y, __shfl_xor_sync(kFull, v[j].y, 1 << b));
            v[j].z = fmaf(sg, v[j].z, __shfl_xor_sync(kFull, v[j].z, 1 << b));
            v[j].w = fmaf(sg, v[j].w, __shfl_xor_sync(kFull, v[j].w, 1 << b));
        }
    }
#pragma unroll
    for (int b = 0; (1 << b) < S; ++b) {
        if (b >= pl.sbg) break;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            if (j & (1 << b)) continue;
            const int k = j | (1 << b);
            const float4 x = v[j], y = v[k];
            v[j] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
            v[k] = make_float4(x.x - y.x, x.y - y.y, x.z - y.z, x.w - y.w);
        }
    }
}

template <int S>
__device__ __forceinline__ float absmax(const float4 (&v)[S])
{
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < S; ++j)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
    return m;
}

// Codes of one thread's slots, written to their Pi-permuted places (D folded into inv).
template <int LANES, int S, bool kBf16>
__device__ __forceinline__ void quantize_store(const float4 (&v)[S], const Place<LANES, S> &pl, char *qrow,
                                               float inv)
{
#pragma unroll
    for (int j = 0; j < S; ++j) {
        if (!(pl.valid & (1u << j))) continue;
        const int q_out = pl.quad(j) + pl.delta[j];
        const float ip = xor_sign(inv, pl.sgn[j]), in = xor_sign(ip, kSign);
        // Pi on digit 0: components 1 and 2 trade places
        const float r0 = round_half_away(v[j].x * ip);
        const float r1 = round_half_away(v[j].z * ip);
        const float r2 = round_half_away(v[j].y * ip);
        const float r3 = round_half_away(v[j].w * in);
        if constexpr (kBf16) {
            // |r| <= 127: the bf16 of r is the top half of its fp32 bits (a zero code may be -0)
            const uint32_t lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            const uint32_t hi = __byte_perm(__float_as_uint(r2), __float_as_uint(r3), 0x7632);
            reinterpret_cast<uint2 *>(qrow)[q_out] = make_uint2(lo, hi);
        } else {
            // r + 1.5 * 2^23 holds r in its low mantissa bits: the low byte is r as int8
            constexpr float kMagic = 12582912.0f;
            const uint32_t w0 = __float_as_uint(r0 + kMagic), w1 = __float_as_uint(r1 + kMagic);
            const uint32_t w2 = __float_as_uint(r2 + kMagic), w3 = __float_as_uint(r3 + kMagic);
            reinterpret_cast<uint32_t *>(qrow)[q_out] =
                __byte_perm(__byte_perm(w0, w1, 0x0040), __byte_perm(w2, w3, 0x0040), 0x5410);
        }
    }
}

template <bool kBf16>
__device__ __forceinline__ void zero_pad(char *qrow, int kq, int kpq, int t_row, int row_threads)
{
    for (int i = kq + t_row; i < kpq; i += row_threads) {
        if constexpr (kBf16)
            reinterpret_cast<uint2 *>(qrow)[i] = make_uint2(0u, 0u);
        else
            reinterpret_cast<uint32_t *>(qrow)[i] = 0u;
    }
}

// Scale s = max|X_rot| / 127 and the multiplier 2^-n / s applied to the
// unnormalized butterfly output (0 for an all-zero row).
__device__ __forceinline__ float scale_of(float amax_unnorm, int n, float *inv)
{
    const float s = ldexpf(amax_unnorm, -n) / 127.0f;
    *inv = s > 0.0f ? ldexpf(__frcp_rn(s), -n) : 0.0f;
    return s;
}

struct DirectPlan {
    int threads_per_row;  // per CTA
    int rows_per_cta;
    int cl;  // CTAs per row (cluster size); rows_per_cta == 1 when cl > 1
};

template <int LANES, int S, bool kBf16>
__global__ void __launch_bounds__(kMaxThreads<S>) pack_kernel(PackArgs a, DirectPlan L, int64_t row0)
{
    const int lane = threadIdx.x & 31;
    const int cl = L.cl;
    const int cr = cl > 1 ? static_cast<int>(blockIdx.x % cl) : 0;
    const int64_t cta_block = cl > 1 ? blockIdx.x / cl : blockIdx.x;
    const int tpr = L.threads_per_row;
    const int r_local = threadIdx.x / tpr;
    const int t_cta = threadIdx.x - r_local * tpr;
    const int64_t row = row0 + cta_block * L.rows_per_cta + r_local;
    const bool row_ok = row < a.rows;
    const int t_row = cr * tpr + t_cta;
    const int n = a.log4g;
    const int kq = a.k >> 2, kpq = a.kpad >> 2;
    const Place<LANES, S> pl(t_row, n, kq);

    const float4 *src = reinterpret_cast<const float4 *>(a.x + (row_ok ? row : 0) * a.ldx);
    float4 v[S];
#pragma unroll
    for (int j = 0; j < S; ++j)
        v[j] = (row_ok && (pl.valid & (1u << j))) ? __ldcs(src + pl.quad(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    rotate<LANES, S>(v, pl);

    float m = absmax<S>(v);
    const int seg = (tpr & 31) == 0 ? 32 : (tpr & -tpr);
    for (int off = seg >> 1; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    __shared__ float part[kMaxThreads<S>];
    __shared__ float cta_max;
    if ((lane & (seg - 1)) == 0) part[threadIdx.x / seg] = m;
    __syncthreads();
    float amax = 0.0f;
    {
        const int p0 = (r_local * tpr) / seg, np = tpr / seg;
        for (int i = 0; i < np; ++i) amax = fmaxf(amax, part[p0 + i]);
    }
    if (cl > 1) {
        if (threadIdx.x == 0) cta_max = amax;
        cluster_sync_all();  // every CTA's cta_max is written
        amax = 0.0f;
        for (int r = 0; r < cl; ++r) amax = fmaxf(amax, ld_cluster_f32(cluster_smem_addr(&cta_max, r)));
    }
    float inv;
    const float s = scale_of(amax, n, &inv);
    if (row_ok) {
        if (t_row == 0) a.scale[row] = s;
        char *qrow = static_cast<char *>(a.q) + row * a.ldq * (kBf16 ? 2 : 1);
        quantize_store<LANES, S, kBf16>(v, pl, qrow, inv);
        zero_pad<kBf16>(qrow, kq, kpq, t_row, tpr * cl);
    }
    if (cl > 1) cluster_sync_all();  // no CTA leaves while another may still read its cta_max
}

struct Shape {
    int lanes, S;
};

Shape shape_for(int log4g)
{
    if (log4g <= 4) return {3, 8};   // G <= 256
    if (log4g == 5) return {5, 8};   // G = 1024
    return {5, 32};                  // G = 4096
}

int gcd_int(int x, int y)
{
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return x;
}

int threads_per_row(const Shape &sh, int k)
{
    const int tile_q = sh.S << sh.lanes;
    const int tiles = (k / 4 + tile_q - 1) / tile_q;
    return tiles << sh.lanes;
}

DirectPlan direct_plan(const Shape &sh, int k)
{
    const int T = threads_per_row(sh, k);
    const int max_threads = sh.S >= 32 ? 256 : 512;
    DirectPlan L{};
    const int step = 32 / gcd_int(T, 32);
    if (T <= max_threads && step * T <= max_threads) {
        L.cl = 1;
        L.threads_per_row = T;
        int R = step;
        while (R * T < 128 && (R + step) * T <= max_threads) R += step;
        L.rows_per_cta = R;
    } else if (T <= max_threads) {
        L.cl = 1;
        L.threads_per_row = (T + 31) / 32 * 32;  // one row per CTA, trailing threads idle
        L.rows_per_cta = 1;
    } else {
        int cl = (T + max_threads - 1) / max_threads;
        int per = (T + cl - 1) / cl;
        per = (per + 31) / 32 * 32;  // whole warps, a multiple of 2^LANES (<= 32)
        cl = (T + per - 1) / per;
        L.cl = cl;
        L.threads_per_row = per;
        L.rows_per_cta = 1;
    }
    return L;
}

template <int LANES, int S, bool kBf16>
cudaError_t launch_shape(const PackArgs &a, cudaStream_t stream)
{
    const Shape sh{LANES, S};
    const DirectPlan L = direct_plan(sh, a.k);
    if (L.cl > 16) return cudaErrorInvalidConfiguration;
    const int64_t row_blocks = (a.rows + L.rows_per_cta - 1) / L.rows_per_cta;
    const int64_t max_blocks = (int64_t{1} << 31) / L.cl - 1;
    for (int64_t b0 = 0; b0 < row_blocks; b0 += max_blocks) {
        const int64_t blocks = row_blocks - b0 < max_blocks ? row_blocks - b0 : max_blocks;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks * L.cl), 1, 1);
        cfg.blockDim = dim3(static_cast<unsigned>(L.threads_per_row * L.rows_per_cta), 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(L.cl);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        auto kern = pack_kernel<LANES, S, kBf16>;
        if (L.cl > 8) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, L, b0 * L.rows_per_cta);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}


template <bool kBf16>
cudaError_t dispatch(const PackArgs &a, cudaStream_t stream)
{
    if (a.log4g <= 4) return launch_shape<3, 8, kBf16>(a, stream);   // G <= 256
    if (a.log4g == 5) return launch_shape<5, 8, kBf16>(a, stream);   // G = 1024
    if (a.log4g == 6) return launch_shape<5, 32, kBf16>(a, stream);  // G = 4096
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_pack(const PackArgs &a, cudaStream_t stream)
{
    if (a.rows == 0) return cudaSuccess;
    return a.bf16 ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

}  // namespace convrot

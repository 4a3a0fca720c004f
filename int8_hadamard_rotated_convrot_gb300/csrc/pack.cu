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
// Kernels and launch forms.
//  - pack_ring_kernel (G <= 1024, rows short enough for its rings; every DiT
//    shape): persistent CTAs, several per SM, each streaming blocks of whole
//    rows into its own shared-memory ring by bulk copies ahead of the
//    arithmetic; the ring shape (CTAs per SM, rows per stage, stages) is
//    chosen by row length, the grid by the CTAs that are resident at once.
//  - pack_g256_kernel (G <= 1024, longer rows): registers loaded straight
//    from global memory with streaming 16-byte loads; a row longer than one
//    CTA holds is split over a thread-block cluster, whose CTAs exchange
//    their partial row maxima through distributed shared memory.
//  - pack_kernel (G = 4096): the generic layout above (D, Walsh-Hadamard
//    butterflies, Pi at the store), launched like pack_g256_kernel.
// Both G <= 1024 kernels use fixed tile layouts (further down) that apply H4
// along each base-4 digit directly instead of the generic butterflies. The
// ring kernel has three register layouts: 4 lanes x 16 slots per 256-element
// tile (G = 64, 256); 8 lanes x 8 slots (G <= 16: half the registers, twice
// the warps); and at G = 1024 a two-phase rotation that first applies digits
// 0-2 to 64 consecutive elements per thread and writes them back in place,
// so that no digit needs lane shuffles.
#include <cuda_bf16.h>

#include "../../include/convrot.h"
#include "internal.h"
#include "tc_common.cuh"

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

// ---------------------------------------------------------------------------
// Groups of up to 256 (n <= 4, every DiT shape): a fixed layout known at
// compile time.
//
// A tile is 64 consecutive quads (256 elements) of a row, held by 4
// consecutive threads with 16 float4 slots each: lane l of the tile holds quad
// 4 j + l in slot j. Inside the tile the element index is 64 j_hi + 16 j_lo +
// 4 l + c, so base-4 digit 0 is the float4 component c, digit 1 the lane l,
// digit 2 the low two bits of j and digit 3 its high two bits. Digits below n
// lie inside one group; the rest number the groups of the tile.
//
// Digits held in registers use the row structure of 2 H4: every row is all
// ones except a -1 at the mirrored place, so along one digit
// y_i = (x_0 + x_1 + x_2 + x_3) - 2 x_{3-i} (3 adds and 4 fmas, the output
// staying at its own digit value; the signs D are part of the formula).
// The lane digit is 2 H4 = D1 P W1 D1 applied by two shuffle butterflies.
// Rather than flipping input signs, each lane keeps a value that is the true
// one times a known sign and folds the partner's sign into the fma
// coefficient; the last sign and D1 at the output go into the quantization
// multiplier, and P (lanes 1 and 2 trade places) into the store address.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void h4_regs(float &a0, float &a1, float &a2, float &a3)
{
    const float s = (a0 + a1) + (a2 + a3);
    const float y0 = fmaf(-2.0f, a3, s), y1 = fmaf(-2.0f, a2, s);
    const float y2 = fmaf(-2.0f, a1, s), y3 = fmaf(-2.0f, a0, s);
    a0 = y0;
    a1 = y1;
    a2 = y2;
    a3 = y3;
}

// Per lane l of a tile: butterfly coefficients of the two shuffle levels, the
// sign the kept value carries at the end (times D1 at the output), and P(l).
__device__ __forceinline__ float lane_c0(int l) { return (l == 0 || l == 3) ? 1.0f : -1.0f; }
__device__ __forceinline__ float lane_c1(int l) { return (l == 0 || l == 3) ? -1.0f : 1.0f; }
__device__ __forceinline__ int lane_out(int l) { return ((l & 1) << 1) | (l >> 1); }

// One base-4 digit held by lane bits (m0, m1 the xor masks of its two bits).
__device__ __forceinline__ void h4_lanes(float &v, float c0, float c1, int m0, int m1)
{
    v = fmaf(c0, v, __shfl_xor_sync(kFull, v, m0));
    v = fmaf(c1, v, __shfl_xor_sync(kFull, v, m1));
}

// Tile layout of the G <= 1024 kernels: 2^LB lanes x 16 float4 slots, quad
// tile * 16 * 2^LB + 2^LB j + l in slot j. G <= 256 takes LB = 2 (one lane
// digit); G = 1024 takes LB = 4, two lane digits (lane bits 0-1 and 2-3) and
// the slot digits above them. A lane digit's butterfly partners share every
// other digit, so the signs the two lane digits carry simply multiply, and
// each lane digit permutes its own part of the output quad.
template <int N>
struct Tile {
    static constexpr int LB = N == 5 ? 4 : 2;
    static constexpr int LANES = 1 << LB;
    static constexpr int QUADS = 16 << LB;
};

// Round half away from zero of the exact product v * inv: with h = +-1/2
// carrying the product's sign, the fma rounded toward zero never crosses the
// integer that truncation keeps, so trunc(fma_rz(v, inv, h)) is that integer.
// `half_bits` is 1/2 with the sign of inv.
__device__ __forceinline__ float code_of(float v, float inv, uint32_t half_bits)
{
    const float h = __uint_as_float((__float_as_uint(v) & kSign) ^ half_bits);
    return truncf(__fmaf_rz(v, inv, h));
}

// One thread's share of a tile: load, rotate, absmax, quantize and store.

template <int N>
__device__ __forceinline__ void rotate_g256(float4 (&v)[16], int l)
{
    constexpr int LB = Tile<N>::LB;
#pragma unroll
    for (int j = 0; j < 16; ++j) h4_regs(v[j].x, v[j].y, v[j].z, v[j].w);  // digit 0
    if constexpr (N >= 2) {                                                  // digit 1: lane bits 0-1
        const float c0 = lane_c0(l & 3), c1 = lane_c1(l & 3);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            h4_lanes(v[j].x, c0, c1, 1, 2);
            h4_lanes(v[j].y, c0, c1, 1, 2);
            h4_lanes(v[j].z, c0, c1, 1, 2);
            h4_lanes(v[j].w, c0, c1, 1, 2);
        }
    }
    if constexpr (LB == 4) {  // digit 2: lane bits 2-3
        const float c0 = lane_c0((l >> 2) & 3), c1 = lane_c1((l >> 2) & 3);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            h4_lanes(v[j].x, c0, c1, 4, 8);
            h4_lanes(v[j].y, c0, c1, 4, 8);
            h4_lanes(v[j].z, c0, c1, 4, 8);
            h4_lanes(v[j].w, c0, c1, 4, 8);
        }
    }
    if constexpr (N >= LB / 2 + 2) {  // the first slot digit: slots 4 b + (0..3)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float4 &p0 = v[4 * b], &p1 = v[4 * b + 1], &p2 = v[4 * b + 2], &p3 = v[4 * b + 3];
            h4_regs(p0.x, p1.x, p2.x, p3.x);
            h4_regs(p0.y, p1.y, p2.y, p3.y);
            h4_regs(p0.z, p1.z, p2.z, p3.z);
            h4_regs(p0.w, p1.w, p2.w, p3.w);
        }
    }
    if constexpr (N >= LB / 2 + 3) {  // the second slot digit: slots b + 4 (0..3)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float4 &p0 = v[b], &p1 = v[b + 4], &p2 = v[b + 8], &p3 = v[b + 12];
            h4_regs(p0.x, p1.x, p2.x, p3.x);
            h4_regs(p0.y, p1.y, p2.y, p3.y);
            h4_regs(p0.z, p1.z, p2.z, p3.z);
            h4_regs(p0.w, p1.w, p2.w, p3.w);
        }
    }
}

__device__ __forceinline__ float absmax_g256(const float4 (&v)[16])
{
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
    return m;
}

// Codes of slots j < nv. q0 is the thread's slot-0 quad (tile * QUADS + l); inv
// the multiplier from scale_of. Register j holds slot j ^ sw (sw = 0 or 1, see
// the ring kernel); the rotation commutes with that relabeling, because it
// only swaps values along slot digit 2 and y_i = s - 2 x_{3-i} maps i -> i ^ 1
// onto itself.
// kLaneDigits: the lane digits were applied by the sign-carrying shuffle
// butterflies (their last sign, D1 and P are applied here); without it every
// value already sits at its own place with its true sign.
template <int N, bool kBf16, bool kLaneDigits = true>
__device__ __forceinline__ void store_g256(const float4 (&v)[16], int nv, int l, int q0, char *qrow, float inv,
                                           int sw = 0)
{
    constexpr int LB = Tile<N>::LB, LANES = Tile<N>::LANES;
    int lo = l;
    if constexpr (kLaneDigits) {
        // the kept value's sign times D1 at the output, for each lane digit
        if constexpr (N >= 2) inv *= lane_c1(l & 3);
        if constexpr (LB == 4) inv *= lane_c1((l >> 2) & 3);
        // P on each lane digit
        if constexpr (N >= 2) lo = lane_out(l & 3) | (l & ~3);
        if constexpr (LB == 4) lo = lane_out(l & 3) | (lane_out((l >> 2) & 3) << 2);
    }
    const uint32_t half_bits = 0x3f000000u | (__float_as_uint(inv) & kSign);
    const int qo = q0 - l + lo;
    // slot j ^ sw is j + sw for even j and j - sw for odd j
    const int qe = qo + LANES * sw, qd = qo - LANES * sw;
    const int nve = nv - sw, nvd = nv + sw;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (j >= ((j & 1) ? nvd : nve)) continue;
        const int qj = ((j & 1) ? qd : qe) + LANES * j;
        const float r0 = code_of(v[j].x, inv, half_bits), r1 = code_of(v[j].y, inv, half_bits);
        const float r2 = code_of(v[j].z, inv, half_bits), r3 = code_of(v[j].w, inv, half_bits);
        if constexpr (kBf16) {
            // |r| <= 127: the bf16 of r is the top half of its fp32 bits (a zero code may be -0)
            const uint32_t lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            const uint32_t hi = __byte_perm(__float_as_uint(r2), __float_as_uint(r3), 0x7632);
            reinterpret_cast<uint2 *>(qrow)[qj] = make_uint2(lo, hi);
        } else {
            // r + 1.5 * 2^23 holds r in its low mantissa bits: the low byte is r as int8
            constexpr float kMagic = 12582912.0f;
            const uint32_t w0 = __float_as_uint(r0 + kMagic), w1 = __float_as_uint(r1 + kMagic);
            const uint32_t w2 = __float_as_uint(r2 + kMagic), w3 = __float_as_uint(r3 + kMagic);
            reinterpret_cast<uint32_t *>(qrow)[qj] =
                __byte_perm(__byte_perm(w0, w1, 0x0040), __byte_perm(w2, w3, 0x0040), 0x5410);
        }
    }
}

// Slots holding data: quad q0 + 2^LB j < kq. Whole groups are in or out.
template <int LB>
__device__ __forceinline__ int valid_slots(int kq, int q0)
{
    const int nv = (kq - q0 + (1 << LB) - 1) >> LB;
    return nv < 0 ? 0 : (nv > 16 ? 16 : nv);
}

// Row-wide maximum of m over the tpr threads of each row of the CTA: segment
// shuffles, then the segments' partial maxima through shared memory. The
// caller synchronizes between writing `part` and calling row_max_read.
__device__ __forceinline__ void row_max_write(float m, int tpr, float *part)
{
    const int seg = (tpr & 31) == 0 ? 32 : (tpr & -tpr);
    for (int off = seg >> 1; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    if (((threadIdx.x & 31) & (seg - 1)) == 0) part[threadIdx.x / seg] = m;
}

__device__ __forceinline__ float row_max_read(int tpr, int r_local, const float *part)
{
    const int seg = (tpr & 31) == 0 ? 32 : (tpr & -tpr);
    const int p0 = (r_local * tpr) / seg, np = tpr / seg;
    float amax = 0.0f;
    for (int i = 0; i < np; ++i) amax = fmaxf(amax, part[p0 + i]);
    return amax;
}

// Direct form: registers loaded straight from global memory, one pass per CTA;
// rows longer than one CTA holds are split over a cluster.
template <int N, bool kBf16>
__global__ void __launch_bounds__(512) pack_g256_kernel(PackArgs a, DirectPlan L, int64_t row0)
{
    const int cl = L.cl;
    const int cr = cl > 1 ? static_cast<int>(blockIdx.x % cl) : 0;
    const int64_t cta_block = cl > 1 ? blockIdx.x / cl : blockIdx.x;
    const int tpr = L.threads_per_row;
    const int r_local = threadIdx.x / tpr;
    const int t_cta = threadIdx.x - r_local * tpr;
    const int64_t row = row0 + cta_block * L.rows_per_cta + r_local;
    const bool row_ok = row < a.rows;
    const int t_row = cr * tpr + t_cta;
    const int kq = a.k >> 2, kpq = a.kpad >> 2;
    constexpr int LB = Tile<N>::LB;
    const int l = t_row & (Tile<N>::LANES - 1);
    const int q0 = (t_row >> LB) * Tile<N>::QUADS + l;
    const int nv = row_ok ? valid_slots<LB>(kq, q0) : 0;

    const float4 *src = reinterpret_cast<const float4 *>(a.x + (row_ok ? row : 0) * a.ldx) + q0;
    float4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = j < nv ? __ldcs(src + Tile<N>::LANES * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    rotate_g256<N>(v, l);

    __shared__ float part[128];
    __shared__ float cta_max;
    row_max_write(absmax_g256(v), tpr, part);
    __syncthreads();
    float amax = row_max_read(tpr, r_local, part);
    if (cl > 1) {
        if (threadIdx.x == 0) cta_max = amax;
        cluster_sync_all();  // every CTA's cta_max is written
        amax = 0.0f;
        for (int r = 0; r < cl; ++r) amax = fmaxf(amax, ld_cluster_f32(cluster_smem_addr(&cta_max, r)));
    }
    float inv;
    const float s = scale_of(amax, N, &inv);
    if (row_ok) {
        if (t_row == 0) a.scale[row] = s;
        char *qrow = static_cast<char *>(a.q) + row * a.ldq * (kBf16 ? 2 : 1);
        store_g256<N, kBf16>(v, nv, l, q0, qrow, inv);
        zero_pad<kBf16>(qrow, kq, kpq, t_row, tpr * cl);
    }
    if (cl > 1) cluster_sync_all();  // no CTA leaves while another may still read its cta_max
}

// H4 along the slot digit held by slot bits 0-1 (slots 4 b + (0..3)) or by
// slot bits 2-3 (slots b + 4 (0..3)), on every component.
__device__ __forceinline__ void h4_slots_lo(float4 (&v)[16])
{
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float4 &p0 = v[4 * b], &p1 = v[4 * b + 1], &p2 = v[4 * b + 2], &p3 = v[4 * b + 3];
        h4_regs(p0.x, p1.x, p2.x, p3.x);
        h4_regs(p0.y, p1.y, p2.y, p3.y);
        h4_regs(p0.z, p1.z, p2.z, p3.z);
        h4_regs(p0.w, p1.w, p2.w, p3.w);
    }
}

__device__ __forceinline__ void h4_slots_hi(float4 (&v)[16])
{
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float4 &p0 = v[b], &p1 = v[b + 4], &p2 = v[b + 8], &p3 = v[b + 12];
        h4_regs(p0.x, p1.x, p2.x, p3.x);
        h4_regs(p0.y, p1.y, p2.y, p3.y);
        h4_regs(p0.z, p1.z, p2.z, p3.z);
        h4_regs(p0.w, p1.w, p2.w, p3.w);
    }
}

// Two-phase rotation, G >= 64 (n >= 3; used for G = 1024). Phase 1: a thread holds 64
// consecutive elements of its row (16 consecutive quads: digit 0 the
// component, digit 1 slot bits 0-1, digit 2 slot bits 2-3) and applies those
// three digits in registers. Phase 2, after the values are written back in
// place: the tile layout, whose slot digits are digit 3 (G <= 256: slot bits
// 2-3) or digits 3 and 4 (G = 1024: slot bits 0-1 and 2-3). Every digit uses
// the mirror form of 2 H4, so no lane shuffles, signs or output permutation
// are involved, and each output sits at its own place.
template <int N>
__device__ __forceinline__ void rotate_chunk(float4 (&v)[16])
{
#pragma unroll
    for (int j = 0; j < 16; ++j) h4_regs(v[j].x, v[j].y, v[j].z, v[j].w);  // digit 0
    h4_slots_lo(v);                                                          // digit 1
    h4_slots_hi(v);                                                          // digit 2
}

template <int N>
__device__ __forceinline__ void rotate_tile_upper(float4 (&v)[16])
{
    if constexpr (Tile<N>::LB == 4) {
        h4_slots_lo(v);  // digit 3
        h4_slots_hi(v);  // digit 4
    } else if constexpr (N >= 4) {
        h4_slots_hi(v);  // digit 3
    }
}

// Eight-lane tiles for the ring at G <= 256: a 256-element tile is 8 lanes x
// 8 float4 slots, quad q = 8 j + l (slot j, lane l), element 4 q + c. Half the
// registers of the 4-lane tile a thread, so twice the warps fit an SM.
//   digit 0  the component c                        registers
//   digit 1  lane bits 0-1                          sign-carrying shuffle butterflies
//   digit 2  lane bit 2 (low) and slot bit 0 (high) one shuffle and one register butterfly
//   digit 3  slot bits 1-2                          registers
// Digit 2 uses 2 H4 = P D1 W1 D1 with W1 = H2 (x) H2: a radix-2 butterfly on
// each of its two bits, D1 = -1 where both bits are set, P swapping the bits.
// The input D1 folds into the butterfly coefficients (odd slots of lane-bit-0
// threads come out of the shuffle butterfly negated, and the register
// butterfly takes that sign as its coefficient); the output D1 goes into the
// quantization multiplier of odd slots, P into the store address.
template <int N>
__device__ __forceinline__ void rotate_t8(float4 (&v)[8], int l)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) h4_regs(v[j].x, v[j].y, v[j].z, v[j].w);  // digit 0
    if constexpr (N >= 2) {                                                 // digit 1
        const float c0 = lane_c0(l & 3), c1 = lane_c1(l & 3);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            h4_lanes(v[j].x, c0, c1, 1, 2);
            h4_lanes(v[j].y, c0, c1, 1, 2);
            h4_lanes(v[j].z, c0, c1, 1, 2);
            h4_lanes(v[j].w, c0, c1, 1, 2);
        }
    }
    if constexpr (N >= 3) {  // digit 2
        const float ce = (l & 4) ? -1.0f : 1.0f, co = -ce;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float c = (j & 1) ? co : ce;
            v[j].x = fmaf(c, v[j].x, __shfl_xor_sync(kFull, v[j].x, 4));
            v[j].y = fmaf(c, v[j].y, __shfl_xor_sync(kFull, v[j].y, 4));
            v[j].z = fmaf(c, v[j].z, __shfl_xor_sync(kFull, v[j].z, 4));
            v[j].w = fmaf(c, v[j].w, __shfl_xor_sync(kFull, v[j].w, 4));
        }
        // odd slots now carry the sign co: the register butterfly on slot bit 0
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float4 x = v[2 * b], y = v[2 * b + 1];
            v[2 * b] = make_float4(fmaf(co, y.x, x.x), fmaf(co, y.y, x.y), fmaf(co, y.z, x.z), fmaf(co, y.w, x.w));
            v[2 * b + 1] =
                make_float4(fmaf(ce, y.x, x.x), fmaf(ce, y.y, x.y), fmaf(ce, y.z, x.z), fmaf(ce, y.w, x.w));
        }
    }
    if constexpr (N >= 4) {  // digit 3: slots b + 2 (0..3)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float4 &p0 = v[b], &p1 = v[b + 2], &p2 = v[b + 4], &p3 = v[b + 6];
            h4_regs(p0.x, p1.x, p2.x, p3.x);
            h4_regs(p0.y, p1.y, p2.y, p3.y);
            h4_regs(p0.z, p1.z, p2.z, p3.z);
            h4_regs(p0.w, p1.w, p2.w, p3.w);
        }
    }
}

template <int S>
__device__ __forceinline__ float absmax_s(const float4 (&v)[S])
{
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < S; ++j)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
    return m;
}

// Codes of slots j < nv of the eight-lane layout. tq is the tile's first quad.
template <int N, bool kBf16>
__device__ __forceinline__ void store_t8(const float4 (&v)[8], int nv, int l, int tq, char *qrow, float inv)
{
    int lo = l & 3;
    if constexpr (N >= 2) {
        inv *= lane_c1(l & 3);  // digit 1: the kept value's sign times D1
        lo = lane_out(l & 3);   // digit 1: P
    }
    const int lb2 = (l >> 2) & 1;
    float inv_o = inv;
    int off_e = 4 * lb2 + lo, off_o = 8 + 4 * lb2 + lo;  // quad 8 j + l, per slot parity
    if constexpr (N >= 3) {
        if (lb2) inv_o = -inv;                 // digit 2: output D1 at both bits set
        off_e = 8 * lb2 + lo;                  // digit 2: P swaps lane bit 2 (quad bit 2)
        off_o = 8 * lb2 + 4 + lo;              // and slot bit 0 (quad bit 3)
    }
    const uint32_t half_e = 0x3f000000u | (__float_as_uint(inv) & kSign);
    const uint32_t half_o = 0x3f000000u | (__float_as_uint(inv_o) & kSign);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j >= nv) break;
        const float m = (j & 1) ? inv_o : inv;
        const uint32_t h = (j & 1) ? half_o : half_e;
        const int q = tq + 8 * (j & 6) + ((j & 1) ? off_o : off_e);
        const float r0 = code_of(v[j].x, m, h), r1 = code_of(v[j].y, m, h);
        const float r2 = code_of(v[j].z, m, h), r3 = code_of(v[j].w, m, h);
        if constexpr (kBf16) {
            const uint32_t w01 = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            const uint32_t w23 = __byte_perm(__float_as_uint(r2), __float_as_uint(r3), 0x7632);
            reinterpret_cast<uint2 *>(qrow)[q] = make_uint2(w01, w23);
        } else {
            constexpr float kMagic = 12582912.0f;
            const uint32_t w0 = __float_as_uint(r0 + kMagic), w1 = __float_as_uint(r1 + kMagic);
            const uint32_t w2 = __float_as_uint(r2 + kMagic), w3 = __float_as_uint(r3 + kMagic);
            reinterpret_cast<uint32_t *>(qrow)[q] =
                __byte_perm(__byte_perm(w0, w1, 0x0040), __byte_perm(w2, w3, 0x0040), 0x5410);
        }
    }
}

// Ring form: persistent CTAs, several per SM, each streaming blocks of whole
// rows into its own shared-memory ring by bulk copies (cp.async.bulk, one per
// row, completion counted in bytes on the stage's mbarrier). A stage is
// refilled as soon as every thread has its block in registers, so all stages
// are in flight while a block is rotated and stored. CTAs on one SM drift out
// of phase, so the copies of some overlap the arithmetic and stores of others.
//
// Shared-memory banks. With 4 lanes per tile, one slot of a tile is 64
// contiguous bytes and tiles sit 1 KB apart, so the 8 threads that a 16-byte
// load serves at once (two tiles) would hit the same 16 banks. Odd tiles
// therefore keep slot j ^ 1 in register j: the pair then covers all 32 banks.
constexpr int kMaxStages = 8;

struct RingPlan {
    int threads_per_row;  // 4 per 256-element tile
    int rows_per_stage;
    int stages;
    uint32_t row_bytes;    // k * 4
    uint32_t stage_bytes;  // rows_per_stage * row_bytes
};

using tc::mbar_wait;

// Register layouts of the ring kernel.
enum RingLayout { kLanes4 = 0, kTwoPhase4 = 1, kLanes8 = 2 };

template <int N, bool kBf16, int kLayout>
__global__ void __launch_bounds__(512) __maxnreg__(kLayout == 2 ? 80 : 128) pack_ring_kernel(PackArgs a, RingPlan P)
{
    constexpr bool kTwoPhase = kLayout == kTwoPhase4;
    constexpr bool k8 = kLayout == kLanes8;
    static_assert(!kTwoPhase || N >= 3, "the two-phase rotation needs whole 64-element chunks per group");
    static_assert(!k8 || N <= 4, "eight-lane tiles hold groups of up to 256");
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ float part[2][128];

    const int tpr = P.threads_per_row, R = P.rows_per_stage, NS = P.stages;
    const int r_local = threadIdx.x / tpr;
    const int t_row = threadIdx.x - r_local * tpr;
    const int kq = a.k >> 2, kpq = a.kpad >> 2;
    constexpr int LB = k8 ? 3 : Tile<N>::LB;
    constexpr int LANES = 1 << LB;
    constexpr int SLOTS = k8 ? 8 : 16;
    const int l = t_row & (LANES - 1);
    const int tq = (t_row >> LB) * (SLOTS << LB);  // the tile's first quad
    const int q0 = tq + l;
    const int nv = k8 ? min(max((kq - q0 + 7) >> 3, 0), 8) : valid_slots<LB>(kq, q0);
    const int64_t nblocks = (a.rows + R - 1) / R;
    const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const uint32_t bar_base = static_cast<uint32_t>(__cvta_generic_to_shared(full_bar));

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_base + 8u * s) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int stage, int64_t blk) {
        if (blk >= nblocks) return;
        const int64_t r0 = blk * R;
        const int nr = a.rows - r0 < R ? static_cast<int>(a.rows - r0) : R;
        const uint32_t bar = bar_base + 8u * stage;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(static_cast<uint32_t>(nr) * P.row_bytes)
                     : "memory");
        if (NS == 1) {
            // X is read once: its lines go first when L2 needs room, so that what the next
            // kernel reads (the weights and these codes) stays. Measured on the short-row form
            // (one stage, five CTAs an SM; K = 3072): the pack 16.5 -> 16.0 us, G = 4 14.6 ->
            // 14.2, G = 1024 18.1 -> 17.4, the q/k/v step 152-155 -> 149-151 us, MLP up
            // unchanged. On the two-stage form (MLP down, K = 12288) it cost 49.3 -> 51.4 us,
            // so the other forms read X without the hint.
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            for (int i = 0; i < nr; ++i)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
                    "[%3], %4;" ::"r"(ring_base + stage * P.stage_bytes + i * P.row_bytes),
                    "l"(a.x + (r0 + i) * a.ldx), "r"(P.row_bytes), "r"(bar), "l"(policy)
                    : "memory");
        } else {
            for (int i = 0; i < nr; ++i)
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 ring_base + stage * P.stage_bytes + i * P.row_bytes),
                             "l"(a.x + (r0 + i) * a.ldx), "r"(P.row_bytes), "r"(bar)
                             : "memory");
        }
    };

    if (threadIdx.x == 0)
        for (int s = 0; s < NS; ++s) issue(s, blockIdx.x + static_cast<int64_t>(s) * gridDim.x);

    const int sw = LB == 2 ? (t_row >> LB) & 1 : 0;  // odd tiles hold slot j ^ 1 in register j
    const int nve = nv - sw, nvd = nv + sw;
    // phase 1 of the two-phase rotation: register j holds quad j ^ csw of the
    // thread's 16-quad chunk, so the 8 threads of a 16-byte load (chunks 256 B
    // apart) hit 8 different bank groups; the rotation commutes with that
    // relabeling (it xors digit 1 and the low bit of digit 2)
    const int csw = t_row & 7;
    const bool chunk_in = 16 * t_row < kq;  // whole chunks: kq is a multiple of G / 4 >= 16
    int it = 0;
    bool ok = true;
    for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x, ++it) {
        const int stage = it % NS;
        const bool got = mbar_wait(bar_base + 8u * stage, static_cast<uint32_t>(it / NS) & 1u);
        const int64_t row = blk * R + r_local;
        const bool row_ok = got && row < a.rows;
        float4 *rowp = reinterpret_cast<float4 *>(ring + stage * P.stage_bytes + r_local * P.row_bytes);
        float4 v[SLOTS];
        if constexpr (kTwoPhase) {
            float4 *pc = rowp + 16 * t_row;
            if (row_ok && chunk_in) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = pc[j ^ csw];
                rotate_chunk<N>(v);
#pragma unroll
                for (int j = 0; j < 16; ++j) pc[j ^ csw] = v[j];
            }
            __syncthreads();
        }
        const float4 *src = rowp + q0;
        if constexpr (k8) {
            // a quarter-warp is one tile: 8 consecutive quads, no bank conflicts
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (row_ok && j < nv) ? src[8 * j] : make_float4(0.f, 0.f, 0.f, 0.f);
            rotate_t8<N>(v, l);
        } else {
            const float4 *src_e = src + LANES * sw, *src_d = src - LANES * sw;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = (row_ok && j < ((j & 1) ? nvd : nve)) ? ((j & 1) ? src_d : src_e)[LANES * j]
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (kTwoPhase)
                rotate_tile_upper<N>(v);
            else
                rotate_g256<N>(v, l);
        }
        float *pp = part[it & 1];
        row_max_write(absmax_s<SLOTS>(v), tpr, pp);
        // the stage's generic-proxy writes (phase 1) and reads come before the
        // bulk copy that refills it
        if constexpr (kTwoPhase) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // every thread agrees on whether the stage arrived; a failed wait ends the loop everywhere
        if (!__syncthreads_and(got)) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0) {
            // every thread read this stage into registers before the barrier: refill it now
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(stage, blk + static_cast<int64_t>(NS) * gridDim.x);
        }
        float inv;
        const float s = scale_of(row_max_read(tpr, r_local, pp), N, &inv);
        if (row < a.rows) {
            if (t_row == 0) a.scale[row] = s;
            char *qrow = static_cast<char *>(a.q) + row * a.ldq * (kBf16 ? 2 : 1);
            if constexpr (k8)
                store_t8<N, kBf16>(v, nv, l, tq, qrow, inv);
            else
                store_g256<N, kBf16, !kTwoPhase>(v, nv, l, q0, qrow, inv, sw);
            zero_pad<kBf16>(qrow, kq, kpq, t_row, tpr);
        }
    }
    if (!ok && threadIdx.x == 0) {
        if (a.dev_status) atomicExch(a.dev_status, static_cast<int32_t>(CONVROT_ERR_TIMEOUT));
        // let the copies already issued land before the CTA's shared memory goes away
        int64_t blk = blockIdx.x + static_cast<int64_t>(it) * gridDim.x;
        for (int s = 0; s < NS; ++s, blk += gridDim.x)
            if (blk < nblocks) mbar_wait(bar_base + 8u * ((it + s) % NS), static_cast<uint32_t>((it + s) / NS) & 1u);
    }
}

struct Shape {
    int lanes, S;
};

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

template <typename Kernel>
cudaError_t launch_plan(Kernel kern, const Shape sh, const PackArgs &a, cudaStream_t stream)
{
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
        if (L.cl > 8) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, L, b0 * L.rows_per_cta);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}


// Ring form tuning, tried in order: CTAs per SM, ring bytes per CTA and CTA
// size to aim for. Smaller CTAs with one or two rows per stage balance short
// rows better over the SMs (K = 3072: 2048 blocks over 608 CTAs instead of
// 1024 over 304); rows too long for two stages in the first ring take the
// next.
struct RingTuning {
    int ctas_per_sm;
    uint32_t ring_bytes;
    int threads_target;
    int min_stages;
};
constexpr RingTuning kRingTunings[] = {{5, 25 * 1024, 64, 1}, {2, 100 * 1024, 128, 2}, {1, 200 * 1024, 128, 2}};
// Eight-lane layout (half the registers a thread): twice the threads a row, so
// the same rings hold twice the warps.
constexpr RingTuning kRingTunings8[] = {{4, 50 * 1024, 192, 2}, {2, 100 * 1024, 384, 2}, {1, 200 * 1024, 512, 2}};

struct RingLaunch {
    RingPlan P;
    int ctas_per_sm;  // 0: rows too long for a ring
};

template <size_t NT>
RingLaunch ring_plan(int k, int lane_bits, const RingTuning (&tunings)[NT])
{
    const int T = threads_per_row(Shape{lane_bits, lane_bits == 3 ? 8 : 16}, k);
    const int step = 32 / gcd_int(T, 32);  // rows per stage must fill whole warps
    const uint64_t row_bytes = 4ull * static_cast<uint64_t>(k);
    if (step * T > 512) return RingLaunch{};
    for (const RingTuning &tu : tunings) {
        int R = step;
        while (R * T < tu.threads_target && (R + step) * T <= 512) R += step;
        const uint64_t ns_min = static_cast<uint64_t>(tu.min_stages);
        while (R > step && ns_min * R * row_bytes > tu.ring_bytes) R -= step;
        if (ns_min * R * row_bytes > tu.ring_bytes) continue;
        RingLaunch L{};
        L.ctas_per_sm = tu.ctas_per_sm;
        L.P.threads_per_row = T;
        L.P.rows_per_stage = R;
        L.P.row_bytes = static_cast<uint32_t>(row_bytes);
        L.P.stage_bytes = static_cast<uint32_t>(R * row_bytes);
        const int ns = static_cast<int>(tu.ring_bytes / L.P.stage_bytes);
        L.P.stages = ns > kMaxStages ? kMaxStages : ns;
        return L;
    }
    return RingLaunch{};
}

// Launches the ring form; sets *launched = false (and launches nothing) when not
// one CTA of the planned shape fits on an SM, so that the caller can fall back to
// a form that needs no resident grid.
template <typename Kernel>
cudaError_t launch_ring(Kernel kern, const RingLaunch &L, const PackArgs &a, cudaStream_t stream, bool *launched)
{
    *launched = false;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int smem = L.P.stages * static_cast<int>(L.P.stage_bytes);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int threads = L.P.threads_per_row * L.P.rows_per_stage;
    // a persistent grid must be resident at once: never plan more CTAs an SM than fit
    int resident = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (resident <= 0) return cudaSuccess;
    const int per_sm = resident < L.ctas_per_sm ? resident : L.ctas_per_sm;
    const int64_t nblocks = (a.rows + L.P.rows_per_stage - 1) / L.P.rows_per_stage;
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    const int64_t grid = nblocks < slots ? nblocks : slots;
    kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(a, L.P);
    *launched = true;
    return cudaGetLastError();
}

template <int N, bool kBf16>
cudaError_t launch_g256(const PackArgs &a, cudaStream_t stream)
{
    const RingLaunch L = ring_plan(a.k, Tile<N>::LB, kRingTunings);
    // the two-phase rotation replaces two shuffle digits for G = 1024 (19.6 -> 18.1 us
    // at K = 3072); for G = 64 and 256, one shuffle digit, it measured no faster
    bool launched = false;
    if constexpr (N <= 2) {
        const RingLaunch L8 = ring_plan(a.k, 3, kRingTunings8);
        if (L8.ctas_per_sm > 0) {
            const cudaError_t e = launch_ring(pack_ring_kernel<N, kBf16, kLanes8>, L8, a, stream, &launched);
            if (e != cudaSuccess || launched) return e;
        }
    }
    if (L.ctas_per_sm > 0) {
        const cudaError_t e =
            launch_ring(pack_ring_kernel<N, kBf16, N == 5 ? kTwoPhase4 : kLanes4>, L, a, stream, &launched);
        if (e != cudaSuccess || launched) return e;
    }
    return launch_plan(pack_g256_kernel<N, kBf16>, Shape{Tile<N>::LB, 16}, a, stream);
}

// ---------------------------------------------------------------------------
// Groups of 16384 and 65536 (4^7, 4^8; the page admits any power of four that
// divides the row, "Checkpoint format"). R_G = H4^(x)(n-6) (x) R_4096: each
// warp applies R_4096 to one 4096-element block with the generic layout above
// (32 lanes x 32 slots, D, Walsh-Hadamard butterflies, the output D and Pi
// left to the store), then H4 goes along the digits above the block in the
// mirror form of 2 H4 (y_i = s - 2 x_{3-i}): digit 6 across the CTA's four
// warps through shared memory, digit 7 (G = 65536) across four CTAs of the
// cluster through distributed shared memory. The block's output D and Pi act
// the same way in every block, so they commute with those digits.
// A CTA is 128 threads and 16384 elements of a row; the row's CTAs form a
// cluster (k / 16384 <= 8), which also gives the row its absmax.

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Output `idx` of the mirror form of 2 H4 along one digit, componentwise.
__device__ __forceinline__ float4 h4_mirror_out(const float4 &x0, const float4 &x1, const float4 &x2, const float4 &x3,
                                                int idx)
{
    const float4 &m = idx == 0 ? x3 : idx == 1 ? x2 : idx == 2 ? x1 : x0;
    return make_float4(fmaf(-2.0f, m.x, (x0.x + x1.x) + (x2.x + x3.x)), fmaf(-2.0f, m.y, (x0.y + x1.y) + (x2.y + x3.y)),
                       fmaf(-2.0f, m.z, (x0.z + x1.z) + (x2.z + x3.z)), fmaf(-2.0f, m.w, (x0.w + x1.w) + (x2.w + x3.w)));
}

constexpr int kBigThreads = 128;
constexpr int kBigSmem = 4 * 32 * 32 * 16;  // one float4 per (warp, slot, lane): 64 KB

template <bool kBf16, int kHigh>
__global__ void __launch_bounds__(kBigThreads) pack_big_kernel(PackArgs a, int cl)
{
    extern __shared__ float4 xbuf[];
    __shared__ float part[4];
    __shared__ float cta_max;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t crank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    const int64_t row = blockIdx.x / cl;
    const int64_t block = static_cast<int64_t>(crank) * 4 + warp;  // 4096-element block of the row
    const Place<5, 32> pl(lane, 6, 1024);
    const float4 *src = reinterpret_cast<const float4 *>(a.x + row * a.ldx) + block * 1024;
    float4 v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __ldcs(src + pl.quad(j));
    rotate<5, 32>(v, pl);
    // digit 6: the CTA's four blocks
    auto slot = [&](int w, int j) { return (w * 32 + j) * 32 + lane; };
#pragma unroll
    for (int j = 0; j < 32; ++j) xbuf[slot(warp, j)] = v[j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 32; ++j)
        v[j] = h4_mirror_out(xbuf[slot(0, j)], xbuf[slot(1, j)], xbuf[slot(2, j)], xbuf[slot(3, j)], warp);
    if constexpr (kHigh == 2) {
        // digit 7: four CTAs of the cluster (ranks 4 g .. 4 g + 3 hold one group)
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 32; ++j) xbuf[slot(warp, j)] = v[j];
        cluster_sync_all();
        const uint32_t g0 = crank & ~3u, me = crank & 3u;
        const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(xbuf));
        uint32_t rb[4];
#pragma unroll
        for (uint32_t r = 0; r < 4; ++r) {
            uint32_t m;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(m) : "r"(base), "r"(g0 + r));
            rb[r] = m;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t off = static_cast<uint32_t>(slot(warp, j)) * 16u;
            v[j] = h4_mirror_out(ld_cluster_f4(rb[0] + off), ld_cluster_f4(rb[1] + off), ld_cluster_f4(rb[2] + off),
                                 ld_cluster_f4(rb[3] + off), static_cast<int>(me));
        }
        cluster_sync_all();  // no CTA overwrites or leaves its buffer while another reads it
    }
    float m = absmax<32>(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    if (lane == 0) part[warp] = m;
    __syncthreads();
    float amax = fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3]));
    if (cl > 1) {
        if (threadIdx.x == 0) cta_max = amax;
        cluster_sync_all();  // every CTA's cta_max is written
        amax = 0.0f;
        for (int r = 0; r < cl; ++r) amax = fmaxf(amax, ld_cluster_f32(cluster_smem_addr(&cta_max, r)));
    }
    float inv;
    const float s = scale_of(amax, a.log4g, &inv);
    if (crank == 0 && threadIdx.x == 0) a.scale[row] = s;
    char *qblock = static_cast<char *>(a.q) + (row * a.ldq + block * 4096) * (kBf16 ? 2 : 1);
    quantize_store<5, 32, kBf16>(v, pl, qblock, inv);
    if (cl > 1) cluster_sync_all();  // no CTA leaves while another may still read its cta_max
}

template <bool kBf16, int kHigh>
cudaError_t launch_big(const PackArgs &a, cudaStream_t stream)
{
    // a.k is a multiple of G >= 16384 and at most 131072 here
    const int cl = a.k / 16384;
    if (cl < 1 || cl > 8 || a.k % 16384 != 0) return cudaErrorInvalidValue;
    auto kern = pack_big_kernel<kBf16, kHigh>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBigSmem);
    if (e != cudaSuccess) return e;
    const int64_t max_rows = ((int64_t{1} << 31) - 1) / cl;
    for (int64_t r0 = 0; r0 < a.rows; r0 += max_rows) {
        PackArgs b = a;
        b.rows = a.rows - r0 < max_rows ? a.rows - r0 : max_rows;
        b.x = a.x + r0 * a.ldx;
        b.q = static_cast<char *>(a.q) + r0 * a.ldq * (kBf16 ? 2 : 1);
        b.scale = a.scale + r0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(b.rows * cl), 1, 1);
        cfg.blockDim = dim3(kBigThreads, 1, 1);
        cfg.dynamicSmemBytes = kBigSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, b, cl);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <bool kBf16>
cudaError_t dispatch(const PackArgs &a, cudaStream_t stream)
{
    switch (a.log4g) {
    case 1: return launch_g256<1, kBf16>(a, stream);
    case 2: return launch_g256<2, kBf16>(a, stream);
    case 3: return launch_g256<3, kBf16>(a, stream);
    case 4: return launch_g256<4, kBf16>(a, stream);
    case 5: return launch_g256<5, kBf16>(a, stream);                                 // G = 1024
    case 6: return launch_plan(pack_kernel<5, 32, kBf16>, Shape{5, 32}, a, stream);  // G = 4096
    case 7: return launch_big<kBf16, 1>(a, stream);                                  // G = 16384
    case 8: return launch_big<kBf16, 2>(a, stream);                                  // G = 65536
    default: return cudaErrorInvalidValue;
    }
}

// Second half of a pack whose rotation and row absmax a GEMM epilogue already
// applied: per element only the quantization ("Runtime activation
// quantization": Q = round(X_rot / s), s = max |X_rot| / 127, here with the
// unnormalized rotation and the scale's 2^-n as in scale_of). A warp takes one
// row's 256 columns (8 lines of 128 bytes, two coalesced 16-byte loads a
// lane), a CTA eight rows; each line is discarded from L2 once every lane has
// used its values, so that its dirty copy is never written back. Column tiles
// go from the last to the first: the GEMM stored them in that order of
// recency, so the first ones read are still in L2.
template <bool kBf16>
__global__ void __launch_bounds__(256) requant_kernel(const float *__restrict__ h_rot, int64_t ldh,
                                                      const uint32_t *__restrict__ rowmax, int64_t rows, int32_t k,
                                                      int32_t log4g, void *q, int64_t ldq, float *scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t row_blocks = (rows + 7) / 8;
    const int64_t ct = k / 256 - 1 - static_cast<int64_t>(blockIdx.x) / row_blocks;
    const int64_t row = (static_cast<int64_t>(blockIdx.x) % row_blocks) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    float inv;
    const float s = scale_of(__uint_as_float(rowmax[row]), log4g, &inv);
    if (ct == 0 && lane == 0) scale[row] = s;
    const uint32_t half_bits = 0x3f000000u | (__float_as_uint(inv) & kSign);
    const float *src = h_rot + row * ldh + ct * 256;
    const float4 v0 = __ldcs(reinterpret_cast<const float4 *>(src) + lane);        // columns 4 lane ..
    const float4 v1 = __ldcs(reinterpret_cast<const float4 *>(src) + 32 + lane);   // columns 128 + 4 lane ..
    float r[8] = {code_of(v0.x, inv, half_bits), code_of(v0.y, inv, half_bits), code_of(v0.z, inv, half_bits),
                  code_of(v0.w, inv, half_bits), code_of(v1.x, inv, half_bits), code_of(v1.y, inv, half_bits),
                  code_of(v1.z, inv, half_bits), code_of(v1.w, inv, half_bits)};
    const int64_t c0 = ct * 256 + 4 * lane;
    if constexpr (kBf16) {
        __nv_bfloat16 *qrow = static_cast<__nv_bfloat16 *>(q) + row * ldq;
        reinterpret_cast<uint2 *>(qrow + c0)[0] = make_uint2(__byte_perm(__float_as_uint(r[0]), __float_as_uint(r[1]), 0x7632),
                                                             __byte_perm(__float_as_uint(r[2]), __float_as_uint(r[3]), 0x7632));
        reinterpret_cast<uint2 *>(qrow + c0 + 128)[0] = make_uint2(
            __byte_perm(__float_as_uint(r[4]), __float_as_uint(r[5]), 0x7632),
            __byte_perm(__float_as_uint(r[6]), __float_as_uint(r[7]), 0x7632));
    } else {
        int8_t *qrow = static_cast<int8_t *>(q) + row * ldq;
        constexpr float kMagic = 12582912.0f;
        uint32_t b[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) b[e] = __float_as_uint(r[e] + kMagic);
        reinterpret_cast<uint32_t *>(qrow + c0)[0] =
            __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
        reinterpret_cast<uint32_t *>(qrow + c0 + 128)[0] =
            __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
    }
    // every lane has used its loaded values (the codes above depend on them): drop the lines
    __syncwarp();
    if (lane < 8) asm volatile("discard.global.L2 [%0], 128;" ::"l"(src + 32 * lane) : "memory");
}

}  // namespace

cudaError_t launch_requant(const float *h_rot, int64_t ldh, const uint32_t *rowmax, int64_t rows, int32_t k,
                           int32_t log4g, void *q, int64_t ldq, float *scale, int32_t bf16, cudaStream_t stream)
{
    if (rows == 0) return cudaSuccess;
    if (k % 256 != 0) return cudaErrorInvalidValue;
    const int64_t blocks = (rows + 7) / 8 * (k / 256);
    if (blocks >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
    if (bf16)
        requant_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(h_rot, ldh, rowmax, rows, k, log4g, q,
                                                                                ldq, scale);
    else
        requant_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(h_rot, ldh, rowmax, rows, k, log4g, q,
                                                                                 ldq, scale);
    return cudaGetLastError();
}

cudaError_t launch_pack(const PackArgs &a, cudaStream_t stream)
{
    if (a.rows == 0) return cudaSuccess;
    return a.bf16 ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

}  // namespace convrot

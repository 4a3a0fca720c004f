// Runtime LoRA side branch for the convrot linear.
//
// The page "INT8 Convrot Safetensors" (stable-diffusion.cpp docs), section
// "Backend support", paragraph on adapters: they are applied at runtime, the
// INT8 weights stay untouched, the convrot path gives the base output, and
// the adapter computes its correction from the original, unrotated
// activation and adds it to that output. For a LoRA with down matrix A
// [r, K], up matrix B [N, r] and scale s (alpha / r in the usual files):
//
//   Y = base(X) + s * (X A^T) B^T
//
// Two kernels here, and one extra K-chunk in the linear's GEMM:
//
//   lora_prepare_kernel  offline, per adapter: B_ext [N, 3r] bf16 =
//                        [hi(sB) | lo(sB) | hi(sB)], hi/lo the two-term bf16
//                        split (hi = bf16(v), lo = bf16(v - hi)).
//   lora_prepare_down_kernel  offline, per adapter: A_ext [2r, K] fp32 =
//                        [hi(A); lo(A)], hi = A with its low 13 mantissa bits
//                        cleared (exact in TF32), lo = A - hi.
//   lora_down_kernel     per call: T = X A^T on the tensor cores (tcgen05,
//                        kind::tf32) with three-term TF32 splitting
//                        (T = Xh Ah + Xh Al + Xl Ah), so T carries about fp32
//                        accuracy; then T_ext [M, 3r] bf16 =
//                        [hi(T) | hi(T) | lo(T)].
//   the GEMM             T_ext B_ext^T = hi(T) hi(sB) + hi(T) lo(sB) +
//                        lo(T) hi(sB) runs as one more chunk of the
//                        linear's K loop, accumulated in fp32 in tensor
//                        memory and added to the reconstructed output before
//                        any activation.
//
// lora_down_kernel layout: a cluster of CTAs per 128 rows of X, each taking a
// share of K (so that about one CTA runs per SM).
//   warp 0      TMA producer: 32-column fp32 slices of X (128 rows) and of
//               A_ext's hi and lo rows, 128-byte swizzled, into a ring.
//   warp 1      tcgen05.mma, M = 128, K = 8: the A_ext slices from shared
//               memory, fp32 accumulators in tensor memory; lo(X) from a
//               tensor-memory ring, hi(X) from the X slice itself (its TF32
//               view) up to N = 128 an MMA, else from the ring too.
//   warps 2-9   split each X slice, one row a thread: hi = the value with its
//               low 13 mantissa bits cleared, lo = value - hi, written to
//               the tensor-memory ring with tcgen05.st (hi only where the
//               MMAs take it from there).
//   then        each CTA's partial T goes to its shared memory; the cluster
//               adds the partials in rank order (distributed shared memory),
//               each CTA for its share of the rows, and writes T_ext.
// Every wait is bounded; one that runs out writes CONVROT_ERR_TIMEOUT to the
// caller's status word and the CTA winds down.
#include <cuda_bf16.h>

#include "../../include/convrot.h"
#include "internal.h"
#include "tc_common.cuh"

namespace convrot {
namespace {

using namespace tc;

constexpr int LD_BM = 128;  // rows of X per cluster
constexpr int LD_BK = 32;   // fp32 elements per slice: 128 bytes, one swizzle span
constexpr int LD_SPLIT_WARPS = 8;
constexpr int LD_THREADS = 64 + 32 * LD_SPLIT_WARPS;
constexpr int LD_X_BYTES = LD_BM * LD_BK * 4;  // 16 KB
constexpr int LD_SMEM_LIMIT = 227 * 1024;
constexpr int LD_MAX_CLUSTER = 8;
// tensor memory: the accumulators in columns [0, 256), the X ring in [256, 512): a stage is
// lo(X) alone (32 columns) where the MMAs read hi(X) from shared memory, else hi then lo (64)
constexpr int LD_MAX_STAGES = 4;     // hi and lo in the ring
constexpr int LD_MAX_STAGES_LO = 6;  // lo alone (up to eight fit; shared memory holds six)
constexpr uint32_t LD_TMEM_COLS = 512;
constexpr uint32_t LD_XRING_COL = 256;
constexpr uint32_t LD_XRING_STAGE_COLS = 64;

// kind::tf32: D fp32 (bit 4), A and B TF32 (format 2 at bits 7 and 10), both K-major, M = 128, N = n
__host__ __device__ constexpr uint32_t tf32_idesc(int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(LD_BM >> 4) << 24);
}

// The X operand from tensor memory (M = 128 lanes, one TF32 element a column). The
// accumulate flag is an immediate: a predicate computed at run time costs the issuing
// thread about 20 cycles an instruction, and the loop below is bound by that thread.
template <bool kAccumulate>
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc)
{
    if constexpr (kAccumulate)
        asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem),
                     "l"(b), "r"(idesc)
                     : "memory");
    else
        asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem), "r"(a_tmem),
                     "l"(b), "r"(idesc)
                     : "memory");
}

// The X operand from shared memory (the TMA'd slice, K-major, 128-byte swizzle). As a TF32
// operand the tensor core reads an fp32 value's sign, exponent and top 10 mantissa bits, so
// the raw slice serves as hi(X).
template <bool kAccumulate>
__device__ __forceinline__ void mma_tf32_sa(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc)
{
    if constexpr (kAccumulate)
        asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, 1;" ::"r"(d_tmem), "l"(a), "l"(b),
                     "r"(idesc)
                     : "memory");
    else
        asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, 0;" ::"r"(d_tmem), "l"(a), "l"(b),
                     "r"(idesc)
                     : "memory");
}

// hi(X) as the A operand: the raw slice in shared memory (kXhSmem), or the TMEM ring's hi columns
template <bool kXhSmem, bool kAccumulate>
__device__ __forceinline__ void mma_xh(uint32_t d_tmem, uint64_t x_desc, uint32_t x_tmem, uint64_t b, uint32_t idesc)
{
    if constexpr (kXhSmem)
        mma_tf32_sa<kAccumulate>(d_tmem, x_desc, b, idesc);
    else
        mma_tf32_ta<kAccumulate>(d_tmem, x_tmem, b, idesc);
}

// One 32-column slice: four K = 8 steps. kNacc == 3: Xh [Ah; Al] (N = 2 r) into columns
// [0, 2r) and Xl Ah into [2r, 3r); kNacc == 1: the three products into one accumulator.
// lo(X) always comes from the TMEM ring (columns xt + 32 ...); hi(X) from the X slice in shared
// memory (descriptor dx) when kXhSmem, else from the ring (columns xt ...). kFirst: the slice
// that starts the accumulators.
template <int kNacc, bool kXhSmem, bool kFirst>
__device__ __forceinline__ void lora_slice_mma(uint32_t acc, uint32_t xt, uint64_t dx, uint64_t da, uint64_t dal,
                                               int r, uint32_t idesc, uint32_t idesc2)
{
#pragma unroll
    for (int kk = 0; kk < LD_BK / 8; ++kk) {  // K = 8 TF32: 8 columns of X, 32 bytes of X or A a row
        const uint32_t ht = xt + 8u * kk, lt = xt + 32u + 8u * kk;
        const uint64_t hd = dx + 2u * kk, b = da + 2u * kk;
        if constexpr (kNacc == 3) {
            if (kFirst && kk == 0) {
                mma_xh<kXhSmem, false>(acc, hd, ht, b, idesc2);
                mma_tf32_ta<false>(acc + 2 * r, lt, b, idesc);
            } else {
                mma_xh<kXhSmem, true>(acc, hd, ht, b, idesc2);
                mma_tf32_ta<true>(acc + 2 * r, lt, b, idesc);
            }
        } else {
            if (kFirst && kk == 0)
                mma_xh<kXhSmem, false>(acc, hd, ht, b, idesc);
            else
                mma_xh<kXhSmem, true>(acc, hd, ht, b, idesc);
            mma_xh<kXhSmem, true>(acc, hd, ht, dal + 2u * kk, idesc);
            mma_tf32_ta<true>(acc, lt, b, idesc);
        }
    }
}

// 16 consecutive 32-bit columns of this thread's lane (warp-wide, 32 lanes)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// four floats at a 16-byte aligned address of the CTA of the given rank in this cluster
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t local_addr, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

struct DownParams {
    int64_t m;
    int32_t r;
    int32_t kstages;      // ceil(k / 32), split over the cluster's CTAs
    int32_t stages;       // ring depth
    uint32_t a_bytes;     // r * 128: one slice of A (hi or lo)
    uint32_t stage_bytes; // X + A hi + A lo
    __nv_bfloat16 *t;     // T_ext [m, ldt]
    int64_t ldt;
    int32_t t_cols;       // columns of T_ext written: 3r, then zeros up to t_cols
    int32_t *dev_status;
};

__device__ __forceinline__ void split_tf32(float4 &big, float4 &small)
{
    const uint32_t mask = 0xffffe000u;  // keep sign, exponent and the 10 mantissa bits of TF32
    float4 hi;
    hi.x = __uint_as_float(__float_as_uint(big.x) & mask);
    hi.y = __uint_as_float(__float_as_uint(big.y) & mask);
    hi.z = __uint_as_float(__float_as_uint(big.z) & mask);
    hi.w = __uint_as_float(__float_as_uint(big.w) & mask);
    small = make_float4(big.x - hi.x, big.y - hi.y, big.z - hi.z, big.w - hi.w);  // exact
    big = hi;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// One CTA of a cluster: rows [128 * blockIdx.y, +128) of X, its share of the K
// slices. The cluster's CTAs then add their partial T tiles (through
// distributed shared memory, in rank order) and write T_ext.
template <int kNacc, bool kXhSmem>
__global__ void __launch_bounds__(LD_THREADS, 1)
    lora_down_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, DownParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int S = p.stages;
    const uint32_t bars = base + S * p.stage_bytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto conv_bar = [&](int s) { return bars + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    const uint32_t accf_bar = bars + 8u * (3 * S);
    const uint32_t done_bar = bars + 8u * (3 * S + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + S * p.stage_bytes + 8 * (3 * S + 2));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + S * p.stage_bytes + 8 * (3 * S + 2) + 4);
    // stage s: [X | A hi | A lo] in shared memory, [hi(X) | lo(X)] in the tensor-memory ring
    auto x_big = [&](int s) { return base + s * p.stage_bytes; };
    auto a_big = [&](int s) { return x_big(s) + LD_X_BYTES; };
    auto a_small = [&](int s) { return a_big(s) + p.a_bytes; };
    // the column of slice s's hi(X) (lo(X) is 32 further on); with kXhSmem only lo is stored
    auto x_tmem = [&](int s) {
        return kXhSmem ? LD_XRING_COL - 32u + 32u * static_cast<uint32_t>(s)
                       : LD_XRING_COL + LD_XRING_STAGE_COLS * static_cast<uint32_t>(s);
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = static_cast<int>(blockIdx.y) * LD_BM;
    const uint32_t rank = cluster_rank();
    const int csize = static_cast<int>(gridDim.x);
    const int ks_begin = static_cast<int>((static_cast<int64_t>(p.kstages) * rank) / csize);
    const int ks_end = static_cast<int>((static_cast<int64_t>(p.kstages) * (rank + 1)) / csize);
    const int nks = ks_end - ks_begin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(conv_bar(s), LD_SPLIT_WARPS);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(accf_bar, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(tmem_slot))),
                     "r"(LD_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        if (p.dev_status) atomicExch(p.dev_status, static_cast<int32_t>(CONVROT_ERR_TIMEOUT));
    };

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nks; ++i) {
                if (*abort_flag || !mbar_wait(empty_bar(s), ph ^ 1u)) {
                    ok = false;
                    break;
                }
                const int kx = (ks_begin + i) * LD_BK;
                mbar_arrive_expect_tx(full_bar(s), LD_X_BYTES + 2u * p.a_bytes);
                tma_load_2d(x_big(s), &tmX, kx, row0, full_bar(s));
                tma_load_2d(a_big(s), &tmA, kx, 0, full_bar(s));       // rows 0..r-1: hi(A)
                tma_load_2d(a_small(s), &tmA, kx, p.r, full_bar(s));   // rows r..2r-1: lo(A)
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                fail();
                // the copies already issued land before shared memory goes away
                for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
                    mbar_wait(full_bar(i % S), static_cast<uint32_t>(i / S) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tf32_idesc(p.r), idesc2 = tf32_idesc(kNacc == 3 ? 2 * p.r : p.r);
            // This thread bounds the loop: the MMAs of a slice take about 400 cycles, and any
            // shared-memory access this thread makes after issuing them (a barrier wait, a flag
            // read) returns only once they have all entered the tensor pipe, which then runs dry
            // until the next MMAs come. So where the ring holds three slices or more, the thread
            // waits for two at a time and issues both back to back: one such gap every two
            // slices. (With two, the producer could not refill while both are in use.) No
            // division, and one descriptor add a slice.
            const uint64_t da0 = smem_desc(a_big(0));
            const uint64_t dstep = p.stage_bytes >> 4, dlo = p.a_bytes >> 4, dx_off = LD_X_BYTES >> 4;
            uint64_t da = da0;
            bool ok = true;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nks;) {
                const bool pair = S >= 3 && i + 1 < nks;
                const int s1 = s + 1 == S ? 0 : s + 1;
                const uint32_t ph1 = s + 1 == S ? ph ^ 1u : ph;
                if (!mbar_wait(conv_bar(s), ph) || (pair && !mbar_wait(conv_bar(s1), ph1)) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (i == 0)
                    lora_slice_mma<kNacc, kXhSmem, true>(tmem_base, tmem_base + x_tmem(s), da - dx_off, da, da + dlo,
                                                         p.r, idesc, idesc2);
                else
                    lora_slice_mma<kNacc, kXhSmem, false>(tmem_base, tmem_base + x_tmem(s), da - dx_off, da, da + dlo,
                                                          p.r, idesc, idesc2);
                mma_commit(empty_bar(s));
                da = s1 == 0 ? da0 : da + dstep;
                s = s1;
                ph = ph1;
                if (pair) {
                    lora_slice_mma<kNacc, kXhSmem, false>(tmem_base, tmem_base + x_tmem(s), da - dx_off, da, da + dlo,
                                                          p.r, idesc, idesc2);
                    mma_commit(empty_bar(s));
                    const int s2 = s + 1 == S ? 0 : s + 1;
                    if (s2 == 0) ph ^= 1u;
                    da = s2 == 0 ? da0 : da + dstep;
                    s = s2;
                }
                i += pair ? 2 : 1;
            }
            if (!ok) fail();
            mma_commit(accf_bar);  // after every MMA issued above
            mma_commit(done_bar);
            mbar_wait(done_bar, 0);
        }
        __syncwarp();
    } else {
        // a warp reaches only its TMEM lane quadrant (warp % 4): two warps a quadrant, one for
        // columns 0-15 of the slice, one for 16-31; a thread takes one row of X
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        bool ok = true;
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nks; ++i) {
            if (*abort_flag || !mbar_wait(full_bar(s), ph)) {
                ok = false;
                break;
            }
            // the TMEM stage was last read by the MMAs of slice i - S, which completed before the
            // producer refilled this stage
            tc_fence_after();
            // 128-byte swizzle: 16-byte chunk c of a row sits at chunk c ^ (row % 8), so the eight
            // rows of a lane octet read eight distinct bank groups
            const uint8_t *xrow = gbase + (x_big(s) - base) + row * 128;
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = half * 4 + j;
                float4 v = *reinterpret_cast<const float4 *>(xrow + ((c ^ (row & 7)) << 4)), l;
                split_tf32(v, l);
                hi[4 * j] = __float_as_uint(v.x);
                hi[4 * j + 1] = __float_as_uint(v.y);
                hi[4 * j + 2] = __float_as_uint(v.z);
                hi[4 * j + 3] = __float_as_uint(v.w);
                lo[4 * j] = __float_as_uint(l.x);
                lo[4 * j + 1] = __float_as_uint(l.y);
                lo[4 * j + 2] = __float_as_uint(l.z);
                lo[4 * j + 3] = __float_as_uint(l.w);
            }
            const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + x_tmem(s) + 16u * half;
            if constexpr (!kXhSmem) tmem_st16(ta, hi);
            tmem_st16(ta + 32u, lo);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(conv_bar(s));
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) fail();
    }

    // partial T (this CTA's K share) from tensor memory to shared memory, [128][r + 4] fp32
    const int r = p.r;
    // r + 4 with r % 16 == 0: rows start 16-byte aligned, and a lane octet's float4 stores (one
    // row a lane) fall in eight distinct 16-byte bank groups
    const int pitch = r + 4;
    float *part = reinterpret_cast<float *>(gbase);
    const uint32_t part_addr = base;
    bool ok = true;
    if (warp >= 2) {  // eight warps: two a TMEM lane quadrant, alternate 32-column blocks
        ok = mbar_wait(accf_bar, 0) && !*abort_flag;
        if (ok) {
            tc_fence_after();
            const int q = warp & 3, half = (warp - 2) >> 2;
            float *dst = part + (q * 32 + lane) * pitch;
            for (int c0 = 32 * half; c0 < r; c0 += 64) {
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c0;
                uint32_t v[32];
                float t[32];
                tmem_ld32(ta, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) t[j] = __uint_as_float(v[j]);
                if constexpr (kNacc == 3) {  // the accumulators added in a fixed order
#pragma unroll
                    for (int a = 1; a < 3; ++a) {
                        tmem_ld32(ta + a * r, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) t[j] += __uint_as_float(v[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)  // r % 16 == 0: a quad is wholly in or out
                    if (c0 + 4 * j < r)
                        *reinterpret_cast<float4 *>(dst + c0 + 4 * j) =
                            make_float4(t[4 * j], t[4 * j + 1], t[4 * j + 2], t[4 * j + 3]);
            }
        } else {
            fail();
        }
    }
    tc_fence_before();
    cluster_sync();  // every CTA's partial is in its shared memory (all CTAs reach this)
    const int rows_per = (LD_BM + csize - 1) / csize;  // rows [rb, re) are this CTA's to add up and write
    const int rb = static_cast<int>(rank) * rows_per;
    const int re = rb + rows_per < LD_BM ? rb + rows_per : LD_BM;
    // this CTA adds the cluster's partials, in rank order, for its rows: four columns a thread,
    // two such quads in flight so that all their remote loads overlap
    if (!*abort_flag) {
        const int quads = r / 4;
        const int n = re > rb ? (re - rb) * quads : 0;
        for (int i0 = threadIdx.x; i0 < n; i0 += 2 * LD_THREADS) {
            float4 v[2][LD_MAX_CLUSTER];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int idx = i0 + u * LD_THREADS;
                if (idx < n) {
                    const int rr = rb + idx / quads, c = (idx % quads) * 4;
                    const uint32_t a = part_addr + static_cast<uint32_t>((rr * pitch + c) * 4);
#pragma unroll
                    for (int src = 0; src < LD_MAX_CLUSTER; ++src)
                        if (src < csize) v[u][src] = ld_cluster_f32x4(a, static_cast<uint32_t>(src));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int idx = i0 + u * LD_THREADS;
                if (idx >= n) continue;
                const int rr = rb + idx / quads, c = (idx % quads) * 4;
                const int64_t row = static_cast<int64_t>(row0) + rr;
                if (row >= p.m) continue;
                float4 t = v[u][0];
#pragma unroll
                for (int src = 1; src < LD_MAX_CLUSTER; ++src) {
                    if (src < csize) {
                        t.x += v[u][src].x;
                        t.y += v[u][src].y;
                        t.z += v[u][src].z;
                        t.w += v[u][src].w;
                    }
                }
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(t.x, t.y), h23 = __floats2bfloat162_rn(t.z, t.w);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                uint2 hi, lo;
                hi.x = *reinterpret_cast<const uint32_t *>(&h01);
                hi.y = *reinterpret_cast<const uint32_t *>(&h23);
                lo.x = pack_bf16x2(t.x - f01.x, t.y - f01.y);
                lo.y = pack_bf16x2(t.z - f23.x, t.w - f23.y);
                // T_ext is 16-byte aligned with ldt % 8 == 0, and c, r are multiples of 4: 8-byte stores
                __nv_bfloat16 *dst = p.t + row * p.ldt;
                *reinterpret_cast<uint2 *>(dst + c) = hi;
                *reinterpret_cast<uint2 *>(dst + r + c) = hi;
                *reinterpret_cast<uint2 *>(dst + 2 * r + c) = lo;
            }
        }
        // the zero columns past 3 r (a multiple of 16 of them)
        const int zquads = (p.t_cols - 3 * r) / 4;
        for (int idx = threadIdx.x; idx < (re - rb) * zquads; idx += LD_THREADS) {
            const int64_t row = static_cast<int64_t>(row0) + rb + idx / zquads;
            if (row < p.m)
                *reinterpret_cast<uint2 *>(p.t + row * p.ldt + 3 * r + 4 * (idx % zquads)) = make_uint2(0u, 0u);
        }
    }
    cluster_sync();  // no CTA leaves while another may still read its partial
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(LD_TMEM_COLS)
                     : "memory");
}

// A_ext [2r, lda_ext] fp32: rows 0..r-1 = A with the low 13 mantissa bits cleared (exact in TF32),
// rows r..2r-1 = A minus that.
__global__ void lora_prepare_down_kernel(const float *A, int32_t r, int32_t k, int64_t lda, float *out, int64_t ldo)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(r) * k) return;
    const int64_t j = i / k, c = i - j * k;
    const float v = A[j * lda + c];
    const float hi = __uint_as_float(__float_as_uint(v) & 0xffffe000u);
    out[j * ldo + c] = hi;
    out[(j + r) * ldo + c] = v - hi;
}

// B_ext[o] = [hi(s B[o]) | lo(s B[o]) | hi(s B[o]) | 0 ...]: one thread per (o, pair of columns).
__global__ void lora_prepare_kernel(const float *B, int64_t n, int32_t r, int64_t ldb, float scale,
                                    __nv_bfloat16 *out, int64_t lde, int32_t cols)
{
    const int64_t per_row = cols / 2;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n * per_row) return;
    const int64_t o = i / per_row;
    const int c = static_cast<int>(i - o * per_row) * 2;  // even column of the output row
    uint32_t *dst = reinterpret_cast<uint32_t *>(out + o * lde + c);
    if (c >= 3 * r) {
        *dst = 0u;
        return;
    }
    const int part = c / r, j = c - part * r;  // r is even, so a pair never straddles two parts
    const float v0 = scale * B[o * ldb + j], v1 = scale * B[o * ldb + j + 1];
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    if (part == 1) {
        const float2 hf = __bfloat1622float2(h);
        *dst = pack_bf16x2(v0 - hf.x, v1 - hf.y);
    } else {
        *dst = *reinterpret_cast<const uint32_t *>(&h);
    }
}

}  // namespace

int lora_cols(int r) { return (3 * r + 63) / 64 * 64; }

cudaError_t launch_lora_prepare(const float *B, int64_t n, int32_t r, int64_t ldb, float scale, void *out,
                                int64_t lde, cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    const int cols = lora_cols(r);
    const int64_t total = n * (cols / 2);
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    lora_prepare_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        B, n, r, ldb, scale, static_cast<__nv_bfloat16 *>(out), lde, cols);
    return cudaGetLastError();
}

cudaError_t launch_lora_prepare_down(const float *A, int32_t r, int32_t k, int64_t lda, float *out, int64_t ldo,
                                     cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(r) * k;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    lora_prepare_down_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(A, r, k, lda, out, ldo);
    return cudaGetLastError();
}

cudaError_t launch_lora_down(const float *X, int64_t m, int32_t k, int64_t ldx, const float *A_ext, int32_t r,
                             int64_t lda, void *t, int64_t ldt, int32_t *dev_status, cudaStream_t stream)
{
    if (m == 0) return cudaSuccess;
    CUtensorMap mx, ma;
    if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, X, m, k, ldx * 4, LD_BK, LD_BM) ||
        !make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A_ext, 2 * r, k, lda * 4, LD_BK, static_cast<uint32_t>(r)))
        return cudaErrorInvalidValue;
    DownParams p{};
    p.m = m;
    p.r = r;
    p.kstages = (k + LD_BK - 1) / LD_BK;
    p.a_bytes = static_cast<uint32_t>(r) * LD_BK * 4;
    p.stage_bytes = LD_X_BYTES + 2u * p.a_bytes;
    const bool xh_smem = r <= 128;  // hi(X) read from the X slice (see below)
    const int fixed = 1024 + 256;  // alignment slack, barriers, TMEM slot and flag
    int stages = (LD_SMEM_LIMIT - fixed) / static_cast<int>(p.stage_bytes);
    const int max_stages = xh_smem ? LD_MAX_STAGES_LO : LD_MAX_STAGES;  // what the TMEM ring holds
    stages = stages > max_stages ? max_stages : stages;
    if (stages < 2) return cudaErrorInvalidValue;
    // the partial-T tile [128][r + 4] fp32 reuses the ring once the K loop is done
    if (static_cast<int64_t>(LD_BM) * (r + 4) * 4 > static_cast<int64_t>(stages) * p.stage_bytes)
        return cudaErrorInvalidValue;
    p.stages = stages;
    // three accumulators where 3 r columns fit below the X ring, else one; hi(X) read from the X
    // slice in shared memory up to N = 128 an MMA (beyond, those reads bound the loop and the
    // TMEM copy is faster: r = 256 34.6 against 32.9 us, r = 64 17.5 against 18.4)
    auto kernel = 3 * r <= static_cast<int>(LD_XRING_COL) ? lora_down_kernel<3, true>
                  : xh_smem                               ? lora_down_kernel<1, true>
                                                          : lora_down_kernel<1, false>;
    p.t = static_cast<__nv_bfloat16 *>(t);
    p.ldt = ldt;
    p.t_cols = lora_cols(r);
    p.dev_status = dev_status;
    const int smem = fixed + stages * static_cast<int>(p.stage_bytes);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t row_blocks = (m + LD_BM - 1) / LD_BM;
    if (row_blocks > 65535) return cudaErrorInvalidConfiguration;
    // split K over a cluster so that about one CTA runs per SM
    int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    int cs = static_cast<int>(sms / row_blocks);
    cs = cs < 1 ? 1 : (cs > LD_MAX_CLUSTER ? LD_MAX_CLUSTER : cs);
    if (cs > p.kstages) cs = p.kstages;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cs), static_cast<unsigned>(row_blocks), 1);
    cfg.blockDim = dim3(LD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, mx, ma, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace convrot

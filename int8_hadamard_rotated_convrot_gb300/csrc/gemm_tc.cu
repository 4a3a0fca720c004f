// Exact integer GEMM on the 5th-generation tensor cores (tcgen05.mma,
// kind::f16), with the reconstruction fused into the epilogue.
//
// Computes, from "Runtime activation quantization" on the page "INT8 Convrot
// Safetensors" (stable-diffusion.cpp docs):
//   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]            (exact, int32)
//   Y[r, o] = A[r, o] * s_x[r] * s_w[o] + b[o]        (fp32)
//
// sm_103a has no integer kind for tcgen05.mma, so the int8 codes are carried
// as bf16 (every integer in [-127, 127] is exact in bf16) and multiplied with
// fp32 accumulation in tensor memory. Each product is an integer of magnitude
// <= 16129, so any sum of at most 1024 of them stays below 2^24 and is exact
// in fp32. The K loop therefore runs in chunks of 1024: each chunk
// accumulates from zero in a TMEM buffer, and the epilogue warps convert the
// chunk's (exact, integer-valued) fp32 sums to int32 and add them to int32
// register accumulators. The result equals the page's signed 32-bit
// accumulation bit for bit.
//
// Main form, gemm_tc_pair_kernel (m > 128): a CTA pair (cluster of 2,
// tcgen05 cta_group::2), persistent over 256 x 256 output tiles.
//   warp 0      TMA producer of each CTA: 64-wide K slices of its 128 rows of
//               A and 128 rows of B, 128-byte swizzled, into a ring of as many
//               32 KB stages as fit beside the Y staging (6 for 256-wide
//               tiles); both CTAs' copies complete on the even CTA's barrier.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 buffers per
//               CTA); in the even CTA one thread issues tcgen05.mma (M = 256,
//               N = 256, K = 16) over both CTAs' shared memory.
//   warps 4-19  epilogue, sixteen warps (four per TMEM lane quadrant, 32 rows
//               x 64 columns each): drain each finished chunk from TMEM
//               (tcgen05.ld), accumulate in int32, and after the last chunk of
//               a tile write Y (or the raw int32 A) while the MMA warp runs the
//               next chunk into the other TMEM buffer.
// Single-CTA form, gemm_tc_kernel (m <= 128), persistent over 128 x 256
// tiles: warp 0 produces into a 3-stage ring, warp 1 issues M = 128 MMAs,
// warps 2-9 are the epilogue (32 rows x 128 columns each).
// Every mbarrier wait is bounded: a wait that runs out writes
// CONVROT_ERR_TIMEOUT to the caller's status word and the CTA winds down
// (in-flight copies and MMAs are waited for, TMEM is freed).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/convrot.h"
#include "internal.h"
#include "tc_common.cuh"

namespace convrot {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;  // BK bf16 = 128 B = one swizzle span
constexpr int STAGES = 3;
constexpr int UMMA_K = 16;
constexpr int CHUNK_KSTAGES = 1024 / BK;  // K elements per exact fp32 chunk / BK
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
// Y staging for TMA stores: per epilogue warp, two 32 x 32 fp32 boxes (4 KB each).
constexpr int OUT_BOX = 32;
constexpr int OUT_BUF_BYTES = OUT_BOX * OUT_BOX * 4;
constexpr int OUT_WARP_BYTES = 2 * OUT_BUF_BYTES;
constexpr int OUT_BYTES = 8 * OUT_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES;

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M = 128, N = 256
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                            (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// Tile order: bands of kGroupM row blocks, N-fastest inside a band, so that
// the tiles in flight at once (one per CTA or pair) share a few A panels and a
// few B panels that stay in L2. (With M-fastest order on M = 32760 the tiles in
// flight spanned 76 A panels, more than L2, and A streamed from HBM once per
// column of tiles.) For M <= kGroupM row blocks this is the plain M-fastest order.
constexpr int64_t kGroupM = 16;

__device__ __forceinline__ void tile_coords(int64_t t64, int64_t n_mt64, int64_t n_nt64, int64_t &mt, int64_t &nt)
{
    // (tile counts stay far below 2^31: 32-bit arithmetic)
    const uint32_t t = static_cast<uint32_t>(t64), n_mt = static_cast<uint32_t>(n_mt64);
    const uint32_t per_band = static_cast<uint32_t>(kGroupM) * static_cast<uint32_t>(n_nt64);
    const uint32_t band = t / per_band;
    const uint32_t first = band * static_cast<uint32_t>(kGroupM);
    const uint32_t rows = n_mt - first < static_cast<uint32_t>(kGroupM) ? n_mt - first : static_cast<uint32_t>(kGroupM);
    const uint32_t local = t - band * per_band;
    mt = first + local % rows;
    nt = local / rows;
}

struct TcParams {
    int64_t m, n;
    int32_t vec_cols;  // s_w and bias are 16-byte aligned
    int32_t kstages;  // kpad / BK
    const float *sx, *sw, *bias;
    float *y;
    int32_t *a;
    int64_t ldy;
    int32_t *dev_status;
    int32_t act;       // convrot_activation on Y
    int32_t lora_kst;  // 64-wide K slices of the LoRA operands (pair kernel, kLora)
    // pair kernel: tiles [0, full_tiles) run as whole tiles, full_tiles a
    // multiple of the pairs; each tile past them (the last, partial wave) is
    // split along N into tail_split items (1, 2, 4 or 8)
    int64_t full_tiles;
    int32_t tail_split;
    // pair kernel, kRot: the output's rotation (H4 along its rot_digits lowest base-4
    // digits, unnormalized) is applied in the epilogue, and each row's absmax of it is
    // folded into rowmax (fp32 bits, atomicMax); the rotated values go out through y_raw
    uint32_t *rowmax;
    int32_t rot_digits;
};


// One epilogue warp's 32 rows x NACC columns of the tile (lane i holds row
// row0 + i in acc[]): raw int32 A, or Y = float(A) * s_x[row] * s_w[col] +
// b[col]. Each 32 x 32 box is written to one of the warp's NBUF shared-memory
// buffers in the 128-byte-swizzled layout (16-byte chunk c of row r at c ^
// (r & 7): conflict-free for the row-per-lane writes) and stored by TMA, which
// writes whole lines and clips rows >= m. A box that would cross column n is
// written directly with masked stores instead. A buffer is reused only after
// the store issued from it NBUF boxes earlier has read it.
// Activation over the warp's staged 32 x 32 box (lane i owns row i), in a
// loop unrolled only twice so that the accumulators of the boxes still to
// come stay in registers while it runs (fully unrolled, the GELU's
// temporaries pushed all 128 of them to local memory).
// Staged box of 32 rows x BW fp32 columns (BW = 32: 128-byte rows in the
// 128-byte swizzle, 16-byte chunk c of row r at c ^ (r & 7); BW = 16: 64-byte
// rows in the 64-byte swizzle, chunk c at c ^ ((r >> 1) & 3)); either way the
// row-per-lane 16-byte writes are conflict-free.
template <int BW>
__device__ __forceinline__ uint32_t box_addr(uint32_t buf, int lane, int c)
{
    const int phys = BW == 32 ? (c ^ (lane & 7)) : (c ^ ((lane >> 1) & 3));
    return buf + lane * (BW * 4) + (phys << 4);
}

template <int kAct, int BW = 32>
__device__ __forceinline__ void act_box(uint32_t buf, int lane)
{
#pragma unroll 2
    for (int c = 0; c < BW / 4; ++c) {
        const uint32_t addr = box_addr<BW>(buf, lane, c);
        float4 v;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
        v = make_float4(apply_act_t<kAct>(v.x), apply_act_t<kAct>(v.y), apply_act_t<kAct>(v.z), apply_act_t<kAct>(v.w));
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                     : "memory");
    }
}

// With kLora, lora_taddr is the TMEM address of this warp's rows and columns
// of the LoRA chunk (fp32), added to each output before the activation.
// NACC: columns per warp (128 or 64); NBUF: the warp's staging buffers (2 or 1);
// BW: columns per staged box (32 or 16).
template <bool kRawInt32, int kAct, bool kLora = false, int NACC = 128, int NBUF = 2, int BW = 32>
__device__ __forceinline__ void store_tile_rows(const TcParams &p, const CUtensorMap *tmY, uint32_t out_smem,
                                                uint32_t &store_iter, int64_t row0, int64_t col0,
                                                const int32_t (&acc)[NACC], int lane, int ncols = NACC,
                                                uint32_t lora_taddr = 0)
{
    const int64_t row = row0 + lane;
    float sxr = 0.0f;
    if constexpr (!kRawInt32) sxr = row < p.m ? p.sx[row] : 0.0f;
    constexpr uint32_t kBufBytes = 32u * BW * 4u;
#pragma unroll
    for (int cc = 0; cc < NACC / BW; ++cc) {
        if (cc * BW >= ncols) break;
        const int64_t x = col0 + cc * BW;
        if (x >= p.n) break;
        if ((kAct != 0 || kLora) && x + BW > p.n) {
            // ragged last box with an activation or a LoRA term: stage, activate, then masked stores
            const uint32_t buf = out_smem + (NBUF == 2 ? (store_iter & 1u) * kBufBytes : 0u);
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
#pragma unroll
            for (int c = 0; c < BW / 4; ++c) {
                uint32_t w[4], lr[4];
                if constexpr (kLora) tmem_ld4(lora_taddr + cc * BW + c * 4, lr);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t col = x + c * 4 + e;
                    const float swv = col < p.n ? __ldg(p.sw + col) : 0.0f;
                    const float bv = (p.bias && col < p.n) ? __ldg(p.bias + col) : 0.0f;
                    float y = fmaf(static_cast<float>(acc[cc * BW + c * 4 + e]) * sxr, swv, bv);
                    if constexpr (kLora) y += __uint_as_float(lr[e]);
                    w[e] = __float_as_uint(y);
                }
                const uint32_t addr = box_addr<BW>(buf, lane, c);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
            if constexpr (kAct != 0) act_box<kAct, BW>(buf, lane);
            if (row < p.m) {
#pragma unroll 1
                for (int j = 0; j < BW && x + j < p.n; ++j) {
                    const uint32_t addr = box_addr<BW>(buf, lane, j >> 2) | ((j & 3) << 2);
                    float v;
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
                    p.y[row * p.ldy + x + j] = v;
                }
            }
            __syncwarp();
            continue;
        }
        if (x + BW > p.n) {
            // ragged last box: masked stores straight from registers
            if (row < p.m) {
                for (int j = 0; j < BW && x + j < p.n; ++j) {
                    const int64_t col = x + j;
                    if constexpr (kRawInt32) {
                        p.a[row * p.ldy + col] = acc[cc * BW + j];
                    } else {
                        const float b = p.bias ? __ldg(p.bias + col) : 0.0f;
                        p.y[row * p.ldy + col] = fmaf(static_cast<float>(acc[cc * BW + j]) * sxr, __ldg(p.sw + col), b);
                    }
                }
            }
            continue;
        }
        const uint32_t buf = out_smem + (NBUF == 2 ? (store_iter & 1u) * kBufBytes : 0u);
        if (lane == 0) {
            if constexpr (NBUF == 2)
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            else
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < BW / 4; ++c) {
            uint32_t w[4], lr[4];
            if constexpr (kLora) tmem_ld4(lora_taddr + cc * BW + c * 4, lr);
            float4 sw4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (!kRawInt32) {
                const int64_t col = x + c * 4;
                if (p.vec_cols) {  // s_w and bias 16-byte aligned: 4 columns per load
                    sw4 = __ldg(reinterpret_cast<const float4 *>(p.sw + col));
                    if (p.bias) b4 = __ldg(reinterpret_cast<const float4 *>(p.bias + col));
                } else {
                    sw4 = make_float4(__ldg(p.sw + col), __ldg(p.sw + col + 1), __ldg(p.sw + col + 2), __ldg(p.sw + col + 3));
                    if (p.bias)
                        b4 = make_float4(__ldg(p.bias + col), __ldg(p.bias + col + 1), __ldg(p.bias + col + 2),
                                         __ldg(p.bias + col + 3));
                }
            }
            const float swv[4] = {sw4.x, sw4.y, sw4.z, sw4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = cc * BW + c * 4 + e;
                if constexpr (kRawInt32) {
                    w[e] = static_cast<uint32_t>(acc[j]);
                } else {
                    float y = fmaf(static_cast<float>(acc[j]) * sxr, swv[e], bv[e]);
                    if constexpr (kLora) y += __uint_as_float(lr[e]);
                    if constexpr (kAct != 0) y = apply_act_t<kAct>(y);  // short and call-free: applied in place
                    w[e] = __float_as_uint(y);
                }
            }
            const uint32_t addr = box_addr<BW>(buf, lane, c);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            if (row0 < p.m)
                asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                 reinterpret_cast<uint64_t>(tmY)),
                             "r"(static_cast<int>(x)), "r"(static_cast<int>(row0)), "r"(buf)
                             : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        ++store_iter;
    }
}

// The warp's outstanding TMA stores have completed (before the CTA exits).
__device__ __forceinline__ void drain_stores(int lane)
{
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

template <bool kRawInt32, int kAct>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t out_base = base + STAGES * STAGE_BYTES;
    const uint32_t bars = out_base + OUT_BYTES;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + STAGES * STAGE_BYTES + OUT_BYTES + 128);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + STAGES * STAGE_BYTES + OUT_BYTES + 132);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_mt = (p.m + BM - 1) / BM, n_nt = (p.n + BN - 1) / BN;
    const int64_t n_tiles = n_mt * n_nt;
    const int kst = p.kstages;
    const int n_chunks = (kst + CHUNK_KSTAGES - 1) / CHUNK_KSTAGES;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), EPI_WARPS);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmY)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(tmem_slot))),
                     "r"(TMEM_COLS)
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
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                int64_t mt64, nt64;
                tile_coords(t, n_mt, n_nt, mt64, nt64);
                const int mt = static_cast<int>(mt64), nt = static_cast<int>(nt64);
                for (int ks = 0; ks < kst; ++ks) {
                    if (*abort_flag || !mbar_wait(empty_bar(stage), phase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
                    tma_load_2d(sa, &tmA, ks * BK, mt * BM, full_bar(stage));
                    tma_load_2d(sa + A_BYTES, &tmB, ks * BK, nt * BN, full_bar(stage));
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                fail();
                // let the copies already issued land before the CTA's shared memory goes away
                for (int i = 0; i < STAGES && i < issued; ++i) {
                    if (--stage < 0) {
                        stage = STAGES - 1;
                        phase ^= 1u;
                    }
                    mbar_wait(full_bar(stage), phase);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t chunk_iter = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int c = 0; c < n_chunks && ok; ++c, ++chunk_iter) {
                    const uint32_t buf = chunk_iter & 1u;
                    if (*abort_flag || !mbar_wait(acce_bar(buf), ((chunk_iter >> 1) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    const int ks0 = c * CHUNK_KSTAGES;
                    const int ks1 = ks0 + CHUNK_KSTAGES < kst ? ks0 + CHUNK_KSTAGES : kst;
                    for (int ks = ks0; ks < ks1; ++ks) {
                        if (*abort_flag || !mbar_wait(full_bar(stage), phase)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = base + stage * STAGE_BYTES;
                        const uint64_t da = smem_desc(sa), db = smem_desc(sa + A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            // +32 bytes along K inside the swizzle span per K = 16 step
                            mma_bf16(d_tmem, da + 2u * kk, db + 2u * kk, (ks > ks0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(accf_bar(buf));  // chunk finished: epilogue may drain it
                }
            }
            if (!ok) fail();
            // every MMA this thread issued has completed before TMEM is released
            mma_commit(done_bar);
            mbar_wait(done_bar, 0);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;              // TMEM lane quadrant this warp may access
        const int h = (warp - 2) >> 2;       // column half of the 256-wide tile
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t out_smem = out_base + (warp - 2) * OUT_WARP_BYTES;
        uint32_t store_iter = 0;
        uint32_t chunk_iter = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            int64_t mt, nt;
            tile_coords(t, n_mt, n_nt, mt, nt);
            int32_t acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0;
            for (int c = 0; c < n_chunks; ++c, ++chunk_iter) {
                const uint32_t buf = chunk_iter & 1u;
                if (*abort_flag || !mbar_wait(accf_bar(buf), (chunk_iter >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + lane_off + buf * BN + h * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tmem_ld32(taddr + j * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[j * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar(buf));
            }
            if (!ok) break;
            store_tile_rows<kRawInt32, kAct>(p, &tmY, out_smem, store_iter, mt * BM + q * 32, nt * BN + h * 128, acc, lane);
        }
        drain_stores(lane);
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}


// ---------------------------------------------------------------------------
// Rotation in the epilogue (the next linear's pack fused into this one's
// output, "Runtime activation quantization" of the page applied to H). A
// 256-column tile row is one group of G <= 256; its in-group index is
// 64 part + 16 a + 4 b + c for the warp's 64-column slice `part`. H4 along a
// base-4 digit in the mirror form of 2 H4 (every row all ones but a -1 at the
// mirrored place): y_i = (x_0 + x_1 + x_2 + x_3) - 2 x_{3-i}, each output at
// its own index, unnormalized (2^n times the rotation; the scale takes 2^-n).

__device__ __forceinline__ void h4_mirror(float &a0, float &a1, float &a2, float &a3)
{
    const float s = (a0 + a1) + (a2 + a3);
    const float y0 = fmaf(-2.0f, a3, s), y1 = fmaf(-2.0f, a2, s);
    const float y2 = fmaf(-2.0f, a1, s), y3 = fmaf(-2.0f, a0, s);
    a0 = y0;
    a1 = y1;
    a2 = y2;
    a3 = y3;
}

// Digits 0, 1 and 2 (those below nd) of the thread's 64 consecutive values.
__device__ __forceinline__ void rot_slice_digits(float (&h)[64], int nd)
{
    if (nd >= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) h4_mirror(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    if (nd >= 2) {
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) h4_mirror(h[16 * a + c], h[16 * a + 4 + c], h[16 * a + 8 + c], h[16 * a + 12 + c]);
    }
    if (nd >= 3) {
#pragma unroll
        for (int j = 0; j < 16; ++j) h4_mirror(h[j], h[16 + j], h[32 + j], h[48 + j]);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2): two CTAs of a cluster compute a
// 256 x 256 tile. Each CTA loads its own 128 rows of A and its own 128 rows
// of B (half of the tile's N) into a 6-stage ring of 32 KB stages; the even
// CTA of the pair issues M = 256, N = 256 MMAs that read both CTAs' shared
// memory and write each CTA's 128 accumulator rows into that CTA's TMEM.
// Per flop this moves two thirds of the single-CTA kernel's L2 traffic and
// keeps six K slices in flight instead of three. The exact-chunk integer
// accumulation is the same as above; the epilogue has sixteen warps (below).
namespace pair {

constexpr int BMC = 128;  // rows of A and D per CTA (256 per pair)

// Y staging of the pair kernel's sixteen epilogue warps: PAIR_NBUF buffers of
// one 32 x PAIR_BW fp32 box each per warp.
constexpr int PAIR_BW = 16, PAIR_NBUF = 1;
constexpr int PAIR_BUF_BYTES = 32 * PAIR_BW * 4;
constexpr int PAIR_OUT_BYTES = 16 * PAIR_NBUF * PAIR_BUF_BYTES;

// Tile width of a pair: BN columns of D (BN / 2 rows of B in each CTA).
template <int BN>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "pair tile width");
    static constexpr int BNP = BN;
    static constexpr int BNC = BN / 2;
    static constexpr int A_BYTES = BMC * BK * 2;
    static constexpr int B_BYTES = BNC * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (232448 - 1024 - PAIR_OUT_BYTES - BAR_BYTES) / STAGE_BYTES < 6
                                      ? (232448 - 1024 - PAIR_OUT_BYTES - BAR_BYTES) / STAGE_BYTES
                                      : 6;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + PAIR_OUT_BYTES + BAR_BYTES;
    // kind::f16: D fp32, A and B bf16, K-major, M = 256 (both CTAs), N = BN
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                                       (uint32_t(256 >> 4) << 24);
    // I8 codes: the TMA brings 64-wide K slices of int8 rows into a raw ring
    // (8 KB of A and 8 KB of B a stage), and the converter warps widen them to
    // f16 in the usual 32 KB stages, which the MMA reads as kind::f16 with f16
    // operands (A and B of one type; every integer in [-127, 127] is exact).
    static constexpr int RAW_A = BMC * BK, RAW_B = BNC * BK, RAW_STAGE = RAW_A + RAW_B;
    static constexpr int STAGES_I8 = 5, RAW_STAGES = 2;
    static constexpr int SMEM_BYTES_I8 =
        1024 + STAGES_I8 * STAGE_BYTES + RAW_STAGES * RAW_STAGE + PAIR_OUT_BYTES + BAR_BYTES;
    static constexpr uint32_t kIdescF16 = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);
    static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(SMEM_BYTES_I8 <= 232448, "I8 rings fit the shared memory of one CTA");
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tile load into this CTA's shared memory, completion counted on the even CTA's mbarrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t leader_bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(leader_bar)
        : "memory");
}

__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Bounded wait with acquire at cluster scope: the phase completes by arrivals
// (release, cluster scope) of threads in either CTA of the pair.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity)
{
    auto try_once = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (try_once()) return true;
        if (globaltimer() - t0 > kTimeoutNs) return false;
    }
}

// 16 int8 codes (one 16-byte chunk of a raw row) to 16 f16 values in two
// 16-byte chunks. Per 32-bit word: flip the sign bits (byte b + 128, in
// [1, 255]), place each byte in the low mantissa byte of the f16 1024.0
// (0x64nn = 1024 + b + 128), and subtract 1152 = 1024 + 128: exact, since every
// value involved is an integer below 2048.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140), b = __byte_perm(u, 0x64646464u, 0x4342);
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0xE480E480u));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0xE480E480u));
}

// Widens rows [0, rows) of a raw int8 tile (64 bytes a row, unswizzled, as the
// TMA wrote it) into a K-major f16 tile in the 128-byte swizzle the MMA reads
// (16-byte chunk c of row r at c ^ (r & 7)). Thread t of the nt converter
// threads takes raw chunks t, t + nt, ...: eight consecutive threads read 128
// contiguous bytes and write eight distinct chunks of two rows, so neither side
// has bank conflicts.
// Chunks go in batches of eight a thread, all eight loads issued before any
// conversion, so that the shared-memory latency overlaps.
__device__ __forceinline__ void widen_rows(uint32_t src, uint32_t dst, int rows, int t, int nt)
{
    constexpr int kBatch = 4;
    const int n = rows * 4;
#pragma unroll 1
    for (int i0 = t; i0 < n; i0 += kBatch * nt) {
        uint32_t w[kBatch][4];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * nt;
            if (i < n)
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[j][0]), "=r"(w[j][1]), "=r"(w[j][2]), "=r"(w[j][3])
                             : "r"(src + static_cast<uint32_t>(i) * 16u));
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * nt;
            if (i >= n) break;
            const int r = i >> 2, c = i & 3;
            uint32_t h[8];
            i8x4_to_f16x4(w[j][0], h[0], h[1]);
            i8x4_to_f16x4(w[j][1], h[2], h[3]);
            i8x4_to_f16x4(w[j][2], h[4], h[5]);
            i8x4_to_f16x4(w[j][3], h[6], h[7]);
            const uint32_t row = dst + static_cast<uint32_t>(r) * 128u, x = static_cast<uint32_t>(r & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((2u * c) ^ x) << 4)), "r"(h[0]),
                         "r"(h[1]), "r"(h[2]), "r"(h[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((2u * c + 1u) ^ x) << 4)),
                         "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                         : "memory");
        }
    }
}

// Arrive (once the issuing thread's MMAs complete) on the barrier at this offset in both CTAs.
__device__ __forceinline__ void commit_both(uint32_t bar)
{
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void commit_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Warp roles of the pair kernel: warpgroup 0 holds the TMA producer (warp 0),
// the MMA issuer (warp 1) and two idle warps; warpgroups 1-4 are sixteen
// epilogue warps, four per TMEM lane quadrant, each draining 32 rows x 64
// columns. Launched at 96 registers a thread (five warps on some SM
// sub-partitions: 16 K registers / (5 x 32) = 102, rounded down to 8s),
// warpgroup 0 gives registers back and the epilogue warps take them:
// 4 x 32 x 40 + 16 x 32 x 104 = 58368 <= 640 x 96 = 61440.
constexpr int PAIR_EPI_WARPS = 16;
constexpr int PAIR_THREADS = 128 + PAIR_EPI_WARPS * 32;
constexpr int PAIR_COLS = 64;  // columns per epilogue warp
constexpr int kRegsWg0 = 40, kRegsEpi = 104;
static_assert(4 * 32 * kRegsWg0 + PAIR_EPI_WARPS * 32 * kRegsEpi <= PAIR_THREADS * 96, "register split");
// With int8 operands a second warpgroup of converter warps joins (warps 4-7,
// beside warps 2 and 3 of warpgroup 0): 768 threads, launched at 80 registers
// a thread; warpgroups 0 and 1 keep 48 and the epilogue takes 96:
// 2 x 128 x 48 + 16 x 32 x 96 = 61440 = 768 x 80.
constexpr int PAIR_THREADS_I8 = 256 + PAIR_EPI_WARPS * 32;
constexpr int kRegsConvI8 = 48, kRegsEpiI8 = 96;
static_assert(2 * 128 * kRegsConvI8 + PAIR_EPI_WARPS * 32 * kRegsEpiI8 <= PAIR_THREADS_I8 * 80, "register split (I8)");
static_assert(PAIR_EPI_WARPS * PAIR_NBUF * PAIR_BUF_BYTES == PAIR_OUT_BYTES, "staging per epilogue warp");

// kLora: after each tile's K slices, the producer streams lora_kst more slices
// from tmLa (T_ext rows) and tmLb (B_ext rows); the MMA runs them as one extra
// chunk whose fp32 sums are not promoted to int32 but added to the output.
// kI8: the operands are int8 codes. The producer loads them into the raw ring
// (tmA, tmB, tmBt are int8 maps, unswizzled), warps 2 and 3 of each CTA widen
// each raw stage into an f16 stage and arrive on the even CTA's full barrier,
// and the MMA runs kind::f16 on f16 operands.
constexpr int kConvWarps = 6;

// kRot: the output is the next linear's input; each tile row (one group) is
// rotated in the epilogue, its absmax folded into rowmax, and the rotated
// values stored through y_raw (tmY then maps them as 32-bit words). Whole
// tiles only: the last wave is not split along N.
template <int BN, bool kRawInt32, int kAct, bool kLora, bool kI8 = false, bool kRot = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kI8 ? PAIR_THREADS_I8 : PAIR_THREADS, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmLa,
                        const __grid_constant__ CUtensorMap tmLb, const __grid_constant__ CUtensorMap tmBt,
                        const __grid_constant__ CUtensorMap tmLbt, TcParams p)
{
    using C = Cfg<BN>;
    static_assert(!(kI8 && kLora), "the LoRA chunk is bf16: it runs with bf16 codes only");
    static_assert(!kRot || (!kRawInt32 && !kLora && BN == 256), "the rotation epilogue stores whole 256-column rows");
    constexpr int STAGES = kI8 ? C::STAGES_I8 : C::STAGES, RSTAGES = kI8 ? C::RAW_STAGES : 0;
    constexpr int STAGE_BYTES = C::STAGE_BYTES, A_BYTES = C::A_BYTES, BNP = C::BNP, BNC = C::BNC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t raw_base = base + STAGES * STAGE_BYTES;  // kI8: the int8 ring
    const uint32_t out_base = raw_base + RSTAGES * C::RAW_STAGE;
    const uint32_t bars = out_base + PAIR_OUT_BYTES;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    auto raw_full = [&](int r) { return bars + 8u * (2 * STAGES + 5 + r); };
    auto raw_empty = [&](int r) { return bars + 8u * (2 * STAGES + 5 + RSTAGES + r); };
    // kI8, odd CTA: its converter warps arrive here; one thread forwards each phase to the even CTA
    auto conv_done = [&](int s) { return bars + 8u * (2 * STAGES + 5 + 2 * RSTAGES + s); };
    // kRot: the four epilogue warps of TMEM lane quadrant q exchange their slices through these
    constexpr int kXch0 = 2 * STAGES + 5 + (kI8 ? STAGES + 2 * RSTAGES : 0);
    auto xch_bar = [&](int q) { return bars + 8u * (kXch0 + q); };
    constexpr int kSlotOff = (kI8 || kRot) ? 8 * (kXch0 + (kRot ? 4 : 0)) + 8 : 160;
    static_assert(kSlotOff + 8 <= BAR_BYTES, "barriers, TMEM slot and abort flag fit their region");
    uint8_t *const slots = gbase + (out_base - base) + PAIR_OUT_BYTES + kSlotOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(slots);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(slots + 4);

    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_mt = (p.m + 2 * BMC - 1) / (2 * BMC), n_nt = (p.n + BNP - 1) / BNP;
    const int64_t n_tiles = n_mt * n_nt;
    const int64_t pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int kst = p.kstages;
    const int n_chunks = (kst + CHUNK_KSTAGES - 1) / CHUNK_KSTAGES;
    const int lkst = kLora ? p.lora_kst : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // kI8: a converted stage is complete when the even CTA's converter warps and the
            // odd CTA's forwarding thread arrived
            mbar_init(full_bar(s), kI8 ? kConvWarps + 1 : 1);
            mbar_init(empty_bar(s), 1);
            if constexpr (kI8) mbar_init(conv_done(s), kConvWarps);
        }
        for (int r = 0; r < RSTAGES; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), kConvWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * PAIR_EPI_WARPS);
        }
        if constexpr (kRot)
            for (int q = 0; q < 4; ++q) mbar_init(xch_bar(q), 4);
        if constexpr (kLora) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmLa)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmLb)) : "memory");
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmY)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(tmem_slot))),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialized and TMEM is allocated before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        if (p.dev_status) atomicExch(p.dev_status, static_cast<int32_t>(CONVROT_ERR_TIMEOUT));
    };

    // kI8: converter thread ct of kConvWarps * 32 widens each raw int8 stage of
    // this CTA into the next f16 stage, then the stage is released to the
    // producer and announced to the even CTA's MMA thread
    auto run_converter = [&](int ct) {
        int rs = 0, stage = 0;
        uint32_t rph = 0, phase = 0;
        bool ok = true;
        auto convert = [&](int b_rows) {
            for (int ks = 0; ks < kst; ++ks) {
                // every lane waits; the warp goes on only if all of them saw both phases
                const bool got = !*abort_flag && mbar_wait(raw_full(rs), rph) && mbar_wait(empty_bar(stage), phase ^ 1u);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    return;
                }
                const uint32_t ra = raw_base + rs * C::RAW_STAGE, sa = base + stage * STAGE_BYTES;
                widen_rows(ra, sa, BMC, ct, kConvWarps * 32);
                widen_rows(ra + C::RAW_A, sa + A_BYTES, b_rows, ct, kConvWarps * 32);
                // the generic-proxy writes are made visible to the tensor cores' reads
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(raw_empty(rs));
                    // a local arrive; a release at cluster scope from every converter warp
                    // stalled each of them ~900 cycles a stage
                    mbar_arrive(leader ? full_bar(stage) : conv_done(stage));
                }
                if (++rs == RSTAGES) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        };
        for (int64_t t = pair_id; t < p.full_tiles && ok; t += n_pairs) convert(BNC);
        {
            const int sp = p.tail_split, wd = BNP / sp;
            const int64_t n_items = (n_tiles - p.full_tiles) * sp;
            for (int64_t u = pair_id; u < n_items && ok; u += n_pairs) convert(wd / 2);
        }
        if (!ok) fail();
    };
    constexpr int kEpi0 = kI8 ? 8 : 4;  // first epilogue warp

    if (warp < 4) {
      // warpgroup 0: every warp runs this one instruction, then the roles split
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kI8 ? kRegsConvI8 : kRegsWg0));
      if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            // one tile or item: every K slice of its A rows and of this CTA's brow.. B rows
            auto produce = [&](int mt, int brow, uint32_t tx, const CUtensorMap *bmap, const CUtensorMap *lbmap) {
                const int arow = mt * 2 * BMC + static_cast<int>(rank) * BMC;
                for (int ks = 0; ks < kst + lkst; ++ks) {
                    if (*abort_flag || !mbar_wait(empty_bar(stage), phase ^ 1u)) {
                        ok = false;
                        return;
                    }
                    const uint32_t sa = base + stage * STAGE_BYTES;
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), tx);
                    const uint32_t lbar = map_to_rank(full_bar(stage), 0);
                    const bool lo = kLora && ks >= kst;
                    const int kx = (lo ? ks - kst : ks) * BK;
                    tma_load_2d_pair(sa, lo ? &tmLa : &tmA, kx, arow, lbar);
                    tma_load_2d_pair(sa + A_BYTES, lo ? lbmap : bmap, kx, brow, lbar);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            };
            // kI8: every K slice into this CTA's raw ring, completion on its own barrier
            int rs = 0;
            uint32_t rph = 0;
            auto produce8 = [&](int mt, int brow, uint32_t tx, const CUtensorMap *bmap) {
                const int arow = mt * 2 * BMC + static_cast<int>(rank) * BMC;
                for (int ks = 0; ks < kst; ++ks) {
                    if (*abort_flag || !mbar_wait(raw_empty(rs), rph ^ 1u)) {
                        ok = false;
                        return;
                    }
                    const uint32_t ra = raw_base + rs * C::RAW_STAGE;
                    mbar_arrive_expect_tx(raw_full(rs), tx);
                    tma_load_2d(ra, &tmA, ks * BK, arow, raw_full(rs));
                    tma_load_2d(ra + C::RAW_A, bmap, ks * BK, brow, raw_full(rs));
                    ++issued;
                    if (++rs == RSTAGES) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
            };
            for (int64_t t = pair_id; t < p.full_tiles && ok; t += n_pairs) {
                int64_t mt64, nt64;
                tile_coords(t, n_mt, n_nt, mt64, nt64);
                const int brow = static_cast<int>(nt64) * BNP + static_cast<int>(rank) * BNC;
                if constexpr (kI8)
                    produce8(static_cast<int>(mt64), brow, C::RAW_STAGE, &tmB);
                else
                    produce(static_cast<int>(mt64), brow, 2u * STAGE_BYTES, &tmB, &tmLb);
            }
            {  // the last, partial wave: its tiles split along N into items
                const int sp = p.tail_split, wd = BNP / sp;
                const int64_t n_items = (n_tiles - p.full_tiles) * sp;
                for (int64_t u = pair_id; u < n_items && ok; u += n_pairs) {
                    int64_t mt64, nt64;
                    tile_coords(p.full_tiles + u / sp, n_mt, n_nt, mt64, nt64);
                    const int brow = static_cast<int>(nt64) * BNP + static_cast<int>(u % sp) * wd +
                                     static_cast<int>(rank) * (wd / 2);
                    if constexpr (kI8)
                        produce8(static_cast<int>(mt64), brow, static_cast<uint32_t>(C::RAW_A + (wd / 2) * BK),
                                 sp > 1 ? &tmBt : &tmB);
                    else
                        produce(static_cast<int>(mt64), brow, 2u * static_cast<uint32_t>(A_BYTES + (wd / 2) * BK * 2),
                                sp > 1 ? &tmBt : &tmB, sp > 1 ? &tmLbt : &tmLb);
                }
            }
            if (!ok && kI8) {
                fail();
                // this CTA's copies in flight land before its shared memory goes away
                for (int i = 0; i < RSTAGES && i < issued; ++i) {
                    if (--rs < 0) {
                        rs = RSTAGES - 1;
                        rph ^= 1u;
                    }
                    mbar_wait(raw_full(rs), rph);
                }
            } else if (!ok) {
                fail();
                if (leader) {
                    // both CTAs' copies for the stages armed here land before shared memory goes away
                    for (int i = 0; i < STAGES && i < issued; ++i) {
                        if (--stage < 0) {
                            stage = STAGES - 1;
                            phase ^= 1u;
                        }
                        mbar_wait(full_bar(stage), phase);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t chunk_iter = 0;
            bool ok = true;
            // one tile or item; idesc carries its width as the instruction's N
            auto mma_tile = [&](uint32_t idesc) {
                for (int c = 0; c < n_chunks + (kLora ? 1 : 0) && ok; ++c, ++chunk_iter) {
                    const uint32_t buf = chunk_iter & 1u;
                    if (*abort_flag || !mbar_wait(acce_bar(buf), ((chunk_iter >> 1) & 1u) ^ 1u)) {
                        ok = false;
                        return;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BNP;
                    // integer chunks of up to 1024 K, then (kLora) the LoRA slices as one chunk
                    const int ks0 = c < n_chunks ? c * CHUNK_KSTAGES : kst;
                    const int ks1 = c < n_chunks ? (ks0 + CHUNK_KSTAGES < kst ? ks0 + CHUNK_KSTAGES : kst) : kst + lkst;
                    for (int ks = ks0; ks < ks1; ++ks) {
                        const bool got = kI8 ? mbar_wait_cluster(full_bar(stage), phase) : mbar_wait(full_bar(stage), phase);
                        if (*abort_flag || !got) {
                            ok = false;
                            return;
                        }
                        tc_fence_after();
                        const uint32_t sa = base + stage * STAGE_BYTES;
                        const uint64_t da = smem_desc(sa), db = smem_desc(sa + A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            mma_pair(d_tmem, da + 2u * kk, db + 2u * kk, idesc, (ks > ks0 || kk > 0) ? 1u : 0u);
                        commit_both(empty_bar(stage));  // frees this stage in both CTAs once the MMAs finish
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    commit_both(accf_bar(buf));
                }
            };
            constexpr uint32_t kId = kI8 ? C::kIdescF16 : C::kIdesc;
            for (int64_t t = pair_id; t < p.full_tiles && ok; t += n_pairs) mma_tile(kId);
            {
                const int sp = p.tail_split;
                const int64_t n_items = (n_tiles - p.full_tiles) * sp;
                const uint32_t idesc = (kId & ~(0x3Fu << 17)) | (static_cast<uint32_t>((BNP / sp) >> 3) << 17);
                for (int64_t u = pair_id; u < n_items && ok; u += n_pairs) mma_tile(idesc);
            }
            if (!ok) fail();
            commit_local(done_bar);
            mbar_wait(done_bar, 0);
        } else if (kI8 && !leader && lane == 0) {
            // odd CTA: forward converted stages to the even CTA's full barriers. A fence at
            // cluster scope orders the converter warps' writes (acquired from conv_done)
            // before relaxed arrivals; it costs ~1200 cycles however little this thread
            // wrote, so one fence covers every stage already converted when it runs.
            int64_t n_stages = 0;
            for (int64_t t = pair_id; t < p.full_tiles; t += n_pairs) n_stages += kst;
            for (int64_t u = pair_id; u < (n_tiles - p.full_tiles) * p.tail_split; u += n_pairs) n_stages += kst;
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t i = 0; i < n_stages;) {
                if (*abort_flag || !mbar_wait(conv_done(stage), phase)) {
                    fail();
                    break;
                }
                int n = 1, s1 = stage;
                uint32_t ph1 = phase;
                for (;;) {  // the stages after it that are already converted
                    if (++s1 == STAGES) {
                        s1 = 0;
                        ph1 ^= 1u;
                    }
                    if (n == STAGES - 1 || i + n >= n_stages || !mbar_try_wait(conv_done(s1), ph1)) break;
                    ++n;
                }
                asm volatile("fence.acq_rel.cluster;" ::: "memory");
                for (int j = 0; j < n; ++j, ++i) {
                    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                                     map_to_rank(full_bar(stage), 0))
                                 : "memory");
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
      } else if (kI8) {
        run_converter((warp - 2) * 32 + lane);  // warps 2 and 3
      }
    } else if (kI8 && warp < 8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsConvI8));
      run_converter((warp - 2) * 32 + lane);  // warps 4-7
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kI8 ? kRegsEpiI8 : kRegsEpi));
        const int q = warp & 3;                 // TMEM lane quadrant (warp % 4)
        const int part = (warp - kEpi0) >> 2;  // 64-column slice of the tile or item
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t out_smem = out_base + (warp - kEpi0) * PAIR_NBUF * PAIR_BUF_BYTES;
        uint32_t store_iter = 0;
        uint32_t chunk_iter = 0;
        bool ok = true;
        uint32_t xch_phase = 0;
        // kRot: y = act(A s_x s_w + b) for the warp's 32 rows x 64 columns, rotated
        // (digits 0-2 in registers, digit 3 across the quadrant's four slices through
        // the staging buffers), absmax into rowmax, then the rotated values stored.
        // False if a partner warp's exchange did not come within the bounded wait.
        auto rot_store = [&](int64_t row0, int64_t col0, int32_t (&acc)[PAIR_COLS]) -> bool {
            const int64_t row = row0 + lane;
            const float sxr = row < p.m ? p.sx[row] : 0.0f;
            float h[PAIR_COLS];
#pragma unroll
            for (int c = 0; c < PAIR_COLS / 4; ++c) {
                const int64_t col = col0 + 4 * c;  // n is a multiple of 256 in this form
                float4 sw4, b4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.vec_cols) {
                    sw4 = __ldg(reinterpret_cast<const float4 *>(p.sw + col));
                    if (p.bias) b4 = __ldg(reinterpret_cast<const float4 *>(p.bias + col));
                } else {
                    sw4 = make_float4(__ldg(p.sw + col), __ldg(p.sw + col + 1), __ldg(p.sw + col + 2), __ldg(p.sw + col + 3));
                    if (p.bias)
                        b4 = make_float4(__ldg(p.bias + col), __ldg(p.bias + col + 1), __ldg(p.bias + col + 2),
                                         __ldg(p.bias + col + 3));
                }
                h[4 * c] = apply_act_t<kAct>(fmaf(static_cast<float>(acc[4 * c]) * sxr, sw4.x, b4.x));
                h[4 * c + 1] = apply_act_t<kAct>(fmaf(static_cast<float>(acc[4 * c + 1]) * sxr, sw4.y, b4.y));
                h[4 * c + 2] = apply_act_t<kAct>(fmaf(static_cast<float>(acc[4 * c + 2]) * sxr, sw4.z, b4.z));
                h[4 * c + 3] = apply_act_t<kAct>(fmaf(static_cast<float>(acc[4 * c + 3]) * sxr, sw4.w, b4.w));
            }
            rot_slice_digits(h, p.rot_digits);
            if (p.rot_digits >= 4) {
                const uint32_t xb = xch_bar(q);
                auto sync4 = [&]() {  // the quadrant's four warps reach the same point (bounded)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xb);
                    const bool got = mbar_wait(xb, xch_phase);
                    xch_phase ^= 1u;
                    return __all_sync(0xffffffffu, got);
                };
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    __syncwarp();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(box_addr<16>(out_smem, lane, c4)),
                                     "f"(h[16 * r + 4 * c4]), "f"(h[16 * r + 4 * c4 + 1]), "f"(h[16 * r + 4 * c4 + 2]),
                                     "f"(h[16 * r + 4 * c4 + 3])
                                     : "memory");
                    if (!sync4()) return false;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float x[4][4];
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) {
                            if (pp == part) {
#pragma unroll
                                for (int e = 0; e < 4; ++e) x[pp][e] = h[16 * r + 4 * c4 + e];
                            } else {
                                const uint32_t pb = out_base + (4 * pp + q) * PAIR_NBUF * PAIR_BUF_BYTES;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(x[pp][0]), "=f"(x[pp][1]), "=f"(x[pp][2]), "=f"(x[pp][3])
                                             : "r"(box_addr<16>(pb, lane, c4)));
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float sum = (x[0][e] + x[1][e]) + (x[2][e] + x[3][e]);
                            // x_{3 - part}, selected without indexing by a runtime value
                            const float mirror = part == 0 ? x[3][e] : part == 1 ? x[2][e] : part == 2 ? x[1][e] : x[0][e];
                            h[16 * r + 4 * c4 + e] = fmaf(-2.0f, mirror, sum);
                        }
                    }
                    if (!sync4()) return false;
                }
            }
            float mx = 0.0f;
#pragma unroll
            for (int j = 0; j < PAIR_COLS; ++j) mx = fmaxf(mx, fabsf(h[j]));
            if (row < p.m) atomicMax(p.rowmax + row, __float_as_uint(mx));
#pragma unroll
            for (int j = 0; j < PAIR_COLS; ++j) acc[j] = __float_as_int(h[j]);
            store_tile_rows<true, 0, false, PAIR_COLS, PAIR_NBUF, PAIR_BW>(p, &tmY, out_smem, store_iter, row0, col0,
                                                                           acc, lane);
            return true;
        };
        const int ncols = BNP - part * PAIR_COLS < PAIR_COLS ? (BNP - part * PAIR_COLS > 0 ? BNP - part * PAIR_COLS : 0)
                                                             : PAIR_COLS;
        for (int64_t t = pair_id; t < p.full_tiles && ok; t += n_pairs) {
            int64_t mt, nt;
            tile_coords(t, n_mt, n_nt, mt, nt);
            int32_t acc[PAIR_COLS];
#pragma unroll
            for (int i = 0; i < PAIR_COLS; ++i) acc[i] = 0;
            for (int c = 0; c < n_chunks; ++c, ++chunk_iter) {
                const uint32_t buf = chunk_iter & 1u;
                if (*abort_flag || !mbar_wait(accf_bar(buf), (chunk_iter >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + lane_off + buf * BNP + part * PAIR_COLS;
#pragma unroll
                for (int j = 0; j < PAIR_COLS / 32; ++j) {
                    if (j * 32 >= ncols) break;  // the last slice is narrower when BN is not a multiple of 64
                    uint32_t r[32];
                    tmem_ld32(taddr + j * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[j * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_remote(map_to_rank(acce_bar(buf), 0));
            }
            if (!ok) break;
            if constexpr (kLora) {
                const uint32_t buf = chunk_iter & 1u;
                if (*abort_flag || !mbar_wait(accf_bar(buf), (chunk_iter >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the LoRA chunk stays in tensor memory until the store reads it box by box
                store_tile_rows<kRawInt32, kAct, true, PAIR_COLS, PAIR_NBUF, PAIR_BW>(
                    p, &tmY, out_smem, store_iter, mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32,
                    nt * BNP + part * PAIR_COLS, acc, lane, ncols, tmem_base + lane_off + buf * BNP + part * PAIR_COLS);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_remote(map_to_rank(acce_bar(buf), 0));
                ++chunk_iter;
            } else if constexpr (kRot) {
                if (!rot_store(mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32, nt * BNP + part * PAIR_COLS,
                               acc)) {
                    ok = false;
                    break;
                }
            } else {
                store_tile_rows<kRawInt32, kAct, false, PAIR_COLS, PAIR_NBUF, PAIR_BW>(
                    p, &tmY, out_smem, store_iter, mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32,
                    nt * BNP + part * PAIR_COLS, acc, lane, ncols);
            }
        }
        {  // the last, partial wave: its tiles split along N into items (the same steps)
            const int sp = p.tail_split, wd = BNP / sp;
            const int64_t n_items = (n_tiles - p.full_tiles) * sp;
            const int rest = wd - part * PAIR_COLS;
            const int ncols = rest < PAIR_COLS ? (rest > 0 ? rest : 0) : PAIR_COLS;
            for (int64_t u = pair_id; u < n_items && ok; u += n_pairs) {  // (16-column drains: fewer live registers)
                int64_t mt, nt;
                tile_coords(p.full_tiles + u / sp, n_mt, n_nt, mt, nt);
                const int coff = static_cast<int>(u % sp) * wd;
                int32_t acc[PAIR_COLS];
#pragma unroll
                for (int i = 0; i < PAIR_COLS; ++i) acc[i] = 0;
                for (int c = 0; c < n_chunks; ++c, ++chunk_iter) {
                    const uint32_t buf = chunk_iter & 1u;
                    if (*abort_flag || !mbar_wait(accf_bar(buf), (chunk_iter >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + lane_off + buf * BNP + part * PAIR_COLS;
#pragma unroll
                    for (int j = 0; j < PAIR_COLS / 16; ++j) {
                        if (j * 16 >= ncols) break;  // an item narrower than this slice
                        uint32_t r[16];
                        tmem_ld16(taddr + j * 16, r);
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[j * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_remote(map_to_rank(acce_bar(buf), 0));
                }
                if (!ok) break;
                if constexpr (kLora) {
                    const uint32_t buf = chunk_iter & 1u;
                    if (*abort_flag || !mbar_wait(accf_bar(buf), (chunk_iter >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the LoRA chunk stays in tensor memory until the store reads it box by box
                    store_tile_rows<kRawInt32, kAct, true, PAIR_COLS, PAIR_NBUF, PAIR_BW>(
                        p, &tmY, out_smem, store_iter, mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32,
                        nt * BNP + coff + part * PAIR_COLS, acc, lane, ncols,
                        tmem_base + lane_off + buf * BNP + part * PAIR_COLS);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_remote(map_to_rank(acce_bar(buf), 0));
                    ++chunk_iter;
                } else if constexpr (kRot) {  // (whole tiles: tail_split is 1 in this form)
                    if (!rot_store(mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32,
                                   nt * BNP + part * PAIR_COLS, acc)) {
                        ok = false;
                        break;
                    }
                } else {
                    store_tile_rows<kRawInt32, kAct, false, PAIR_COLS, PAIR_NBUF, PAIR_BW>(
                        p, &tmY, out_smem, store_iter, mt * 2 * BMC + static_cast<int64_t>(rank) * BMC + q * 32,
                        nt * BNP + coff + part * PAIR_COLS, acc, lane, ncols);
                }
            }
        }
        drain_stores(lane);
        if (!ok) fail();
    }

    tc_fence_before();
    cluster_sync();  // the pair's MMAs, drains and remote arrivals are all done
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace pair

// 2-D map over a [rows, ld] bf16 matrix, box = box_rows x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t kpad, int64_t ld, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kpad), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a [rows, ld] int8 matrix, box = box_rows x 64 elements, unswizzled
// (the converter warps read it row by row and write the swizzled f16 stage).
bool make_map8(CUtensorMap *map, const void *base, int64_t rows, int64_t kpad, int64_t ld, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kpad), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the [m, ld] output (fp32 Y or int32 A): 32 rows x box_cols boxes,
// 128-byte swizzle for 32 columns, 64-byte swizzle for 16.
bool make_out_map(CUtensorMap *map, void *base, int64_t m, int64_t n, int64_t ld, bool int32_out, int box_cols = OUT_BOX)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(OUT_BOX)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, int32_out ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_pair(const GemmArgs &g, TcParams p, int sms, cudaStream_t stream)
{
    using C = pair::Cfg<BN>;
    CUtensorMap pa, pb, la, lb, ty;
    if (!make_out_map(&ty, g.a ? static_cast<void *>(g.a) : static_cast<void *>(g.y), g.m, g.n, g.ldy, g.a != nullptr,
                      pair::PAIR_BW))
        return cudaErrorInvalidValue;
    auto operand_map = [&](CUtensorMap *m, const void *q, int64_t rows, int64_t ld, uint32_t box_rows) {
        return g.i8 ? make_map8(m, q, rows, g.kpad, ld, box_rows) : make_map(m, q, rows, g.kpad, ld, box_rows);
    };
    if (!operand_map(&pa, g.qx, g.m, g.ldqx, pair::BMC) || !operand_map(&pb, g.qw, g.n, g.ldqw, C::BNC))
        return cudaErrorInvalidValue;
    la = pa;
    lb = pb;
    if (g.lora_r > 0) {
        const int lcols = lora_cols(g.lora_r);
        if (!make_map(&la, g.lora_t, g.m, lcols, g.lora_ldt, pair::BMC) ||
            !make_map(&lb, g.lora_b, g.n, lcols, g.lora_ldb, C::BNC))
            return cudaErrorInvalidValue;
        p.lora_kst = lcols / BK;
    }
    const int64_t tiles = ((g.m + 2 * pair::BMC - 1) / (2 * pair::BMC)) * ((g.n + BN - 1) / BN);
    const int64_t pairs = tiles < sms / 2 ? tiles : sms / 2;
    const unsigned grid = static_cast<unsigned>(2 * pairs);
    // The last, partial wave: when all of its tiles fit split along N (into up
    // to eight items of 32 columns or more), the items spread over that many
    // more pairs. B (and the LoRA chunk's B_ext) then come in narrower boxes.
    const int64_t full = tiles / pairs * pairs, tail = tiles - full;
    int split = 1;
    if (BN == 256 && tail > 0 && g.rot_digits == 0)  // (the rotation epilogue needs whole tiles)
        while (split < 8 && tail * split * 2 <= pairs) split *= 2;
    p.full_tiles = full;
    p.tail_split = split;
    CUtensorMap pbt = pb, lbt = lb;
    if (split > 1) {
        const uint32_t rows = static_cast<uint32_t>(C::BNC / split);
        if (!operand_map(&pbt, g.qw, g.n, g.ldqw, rows)) return cudaErrorInvalidValue;
        if (g.lora_r > 0 && !make_map(&lbt, g.lora_b, g.n, lora_cols(g.lora_r), g.lora_ldb, rows))
            return cudaErrorInvalidValue;
    }
    const int smem = g.i8 ? C::SMEM_BYTES_I8 : C::SMEM_BYTES;
    auto run = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, g.i8 ? pair::PAIR_THREADS_I8 : pair::PAIR_THREADS, smem, stream>>>(pa, pb, ty, la, lb, pbt,
                                                                                          lbt, p);
        return cudaGetLastError();
    };
    if (g.rot_digits > 0) {
        if (g.i8 || g.lora_r > 0 || !g.a || g.n % 256 != 0) return cudaErrorNotSupported;
        p.rowmax = g.rot_rowmax;
        p.rot_digits = g.rot_digits;
        if (p.act == 1) return run(pair::gemm_tc_pair_kernel<BN, false, 1, false, false, true>);
        if (p.act == 2) return run(pair::gemm_tc_pair_kernel<BN, false, 2, false, false, true>);
        return run(pair::gemm_tc_pair_kernel<BN, false, 0, false, false, true>);
    }
    if (g.i8) {
        if (g.lora_r > 0) return cudaErrorNotSupported;
        if (g.a) return run(pair::gemm_tc_pair_kernel<BN, true, 0, false, true>);
        if (p.act == 1) return run(pair::gemm_tc_pair_kernel<BN, false, 1, false, true>);
        if (p.act == 2) return run(pair::gemm_tc_pair_kernel<BN, false, 2, false, true>);
        return run(pair::gemm_tc_pair_kernel<BN, false, 0, false, true>);
    }
    if (g.a) return run(pair::gemm_tc_pair_kernel<BN, true, 0, false>);
    if (g.lora_r > 0) {
        if (p.act == 1) return run(pair::gemm_tc_pair_kernel<BN, false, 1, true>);
        if (p.act == 2) return run(pair::gemm_tc_pair_kernel<BN, false, 2, true>);
        return run(pair::gemm_tc_pair_kernel<BN, false, 0, true>);
    }
    if (p.act == 1) return run(pair::gemm_tc_pair_kernel<BN, false, 1, false>);
    if (p.act == 2) return run(pair::gemm_tc_pair_kernel<BN, false, 2, false>);
    return run(pair::gemm_tc_pair_kernel<BN, false, 0, false>);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs &g, cudaStream_t stream)
{
    if (g.m == 0 || g.n == 0) return cudaSuccess;
    // int8 codes: the CTA-pair kernel widens them on chip; at most 128 rows take the
    // legacy int8 MMA kernel
    if (g.i8 && g.m <= BM) return launch_gemm_imma(g, stream);
    CUtensorMap ta, tb;
    if (!make_map(&ta, g.qx, g.m, g.kpad, g.ldqx, BM) || !make_map(&tb, g.qw, g.n, g.kpad, g.ldqw, BN))
        return cudaErrorInvalidValue;
    CUtensorMap ty;
    if (!make_out_map(&ty, g.a ? static_cast<void *>(g.a) : static_cast<void *>(g.y), g.m, g.n, g.ldy, g.a != nullptr))
        return cudaErrorInvalidValue;
    TcParams p{};
    p.m = g.m;
    p.n = g.n;
    p.kstages = g.kpad / BK;
    p.sx = g.sx;
    p.sw = g.sw;
    p.bias = g.bias;
    p.y = g.y;
    p.a = g.a;
    p.ldy = g.ldy;
    p.dev_status = g.dev_status;
    p.act = g.act;
    p.vec_cols = (reinterpret_cast<uintptr_t>(g.sw) % 16 == 0) && (reinterpret_cast<uintptr_t>(g.bias) % 16 == 0);
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (g.m > BM || g.lora_r > 0 || g.i8 || g.rot_digits > 0) {  // (LoRA, int8 operands, rotation: pair kernel only)
        // CTA pairs on 256 x 256 tiles. (224-wide tiles fill the last wave better on
        // paper but measured no faster on the DiT shapes: each chunk already runs at
        // close to the tensor peak and per-tile costs do not shrink with the width.)
        return launch_pair<256>(g, p, sms, stream);
    }
    const int64_t tiles = ((g.m + BM - 1) / BM) * ((g.n + BN - 1) / BN);
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
    auto run = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kern<<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, ty, p);
        return cudaGetLastError();
    };
    if (g.a) return run(gemm_tc_kernel<true, 0>);
    if (p.act == 1) return run(gemm_tc_kernel<false, 1>);
    if (p.act == 2) return run(gemm_tc_kernel<false, 2>);
    return run(gemm_tc_kernel<false, 0>);
}

}  // namespace convrot

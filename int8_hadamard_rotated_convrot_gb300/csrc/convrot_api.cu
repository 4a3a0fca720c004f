// C-ABI entry points of libconvrot: host-side validation, then launches.
// The operations are those of the page "INT8 Convrot Safetensors"
// (stable-diffusion.cpp docs); see include/convrot.h for the contract.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "../../include/convrot.h"
#include "internal.h"

namespace {

// Scratch of convrot_linear_lora_noalloc: T_ext, one array per device. Every
// GPU that loads the library holds it until the process exits. In host code
// the name is a host-side stand-in: kernels get the device address that
// noalloc_scratch_address looks up.
static __device__ __align__(256) uint8_t g_noalloc_scratch[CONVROT_NOALLOC_SCRATCH_BYTES];

// Unique id of the calling thread's current context (driver entry points
// fetched through the runtime, so the library needs no libcuda at link time).
bool current_context_id(unsigned long long *id)
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch on the current device, or nullptr if
// the lookup fails. It is looked up once per device (with that device
// current), on the first call there, and kept with the id of the context it
// belongs to, so that a new context after a cudaDeviceReset looks it up again.
void *noalloc_scratch_address()
{
    constexpr int kMaxDevices = 64;
    struct Entry {
        unsigned long long ctx_id;
        void *addr;
    };
    static Entry cache[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (have_id && cacheable) {
        std::lock_guard<std::mutex> g(mu);
        if (cache[dev].addr && cache[dev].ctx_id == id) return cache[dev].addr;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    if (!have_id) have_id = current_context_id(&id);  // the lookup made the device's context current
    if (have_id && cacheable) {
        std::lock_guard<std::mutex> g(mu);
        cache[dev] = Entry{id, p};
    }
    return p;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Returns n for G = 4^n (n >= 1, G <= CONVROT_MAX_GROUP), else -1.
int log4_group(int64_t G)
{
    if (G < 4 || G > CONVROT_MAX_GROUP) return -1;
    int n = 0;
    while (G > 1) {
        if (G & 3) return -1;
        G >>= 2;
        ++n;
    }
    return n;
}

convrot_status check_k_g(int64_t k, int32_t G, int *log4g)
{
    if (k < 1 || k > CONVROT_MAX_K) return CONVROT_ERR_K_RANGE;
    const int n = log4_group(G);
    // the group size must be a power of four dividing the input features ("Checkpoint format")
    if (n < 0 || k % G != 0) return CONVROT_ERR_GROUP_SIZE;
    *log4g = n;
    return CONVROT_OK;
}

convrot_status check_packed_buffers(const convrot_packed *p, int64_t rows, int64_t k)
{
    if (!p) return CONVROT_ERR_INVALID_ARG;
    if (p->codes != CONVROT_CODES_I8 && p->codes != CONVROT_CODES_BF16) return CONVROT_ERR_INVALID_ARG;
    if (p->ldq < convrot_ldq(k)) return CONVROT_ERR_INVALID_ARG;
    if (p->ldq % 16 != 0) return CONVROT_ERR_ALIGNMENT;
    if (rows > 0) {
        if (!p->q || !p->scale) return CONVROT_ERR_INVALID_ARG;
        if (!aligned(p->q, 16) || !aligned(p->scale, 4)) return CONVROT_ERR_ALIGNMENT;
    }
    return CONVROT_OK;
}

convrot_status pack_rows(const float *X, int64_t rows, int64_t k, int64_t ld, int32_t G,
                         convrot_packed *out, int32_t *dev_status, cudaStream_t stream)
{
    int log4g = 0;
    if (rows < 0 || !out) return CONVROT_ERR_INVALID_ARG;
    convrot_status st = check_k_g(k, G, &log4g);
    if (st != CONVROT_OK) return st;
    if (ld < k) return CONVROT_ERR_INVALID_ARG;
    st = check_packed_buffers(out, rows, k);
    if (st != CONVROT_OK) return st;
    if (rows > 0) {
        if (!X) return CONVROT_ERR_INVALID_ARG;
        if (!aligned(X, 16) || ld % 4 != 0) return CONVROT_ERR_ALIGNMENT;
        if (dev_status && !aligned(dev_status, 4)) return CONVROT_ERR_ALIGNMENT;
    }
    out->rows = rows;
    out->k = k;
    out->group_size = G;
    if (rows == 0) return CONVROT_OK;
    convrot::PackArgs a{};
    a.x = X;
    a.ldx = ld;
    a.rows = rows;
    a.k = static_cast<int32_t>(k);
    a.log4g = log4g;
    a.q = out->q;
    a.ldq = out->ldq;
    a.kpad = static_cast<int32_t>(convrot_ldq(k));
    a.scale = out->scale;
    a.bf16 = out->codes == CONVROT_CODES_BF16;
    a.dev_status = dev_status;
    return convrot::launch_pack(a, stream) == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}

convrot_status check_pair(const convrot_packed *x, const convrot_packed *w)
{
    if (!x || !w) return CONVROT_ERR_INVALID_ARG;
    if (x->rows < 0 || w->rows < 0) return CONVROT_ERR_INVALID_ARG;
    if (x->k != w->k) return CONVROT_ERR_INVALID_ARG;
    // packed activations are reused only by linears with the same group size ("Runtime activation quantization")
    if (x->group_size != w->group_size) return CONVROT_ERR_GROUP_SIZE;
    if (x->codes != w->codes) return CONVROT_ERR_INVALID_ARG;
    int log4g = 0;
    convrot_status st = check_k_g(x->k, x->group_size, &log4g);
    if (st != CONVROT_OK) return st;
    st = check_packed_buffers(x, x->rows, x->k);
    if (st != CONVROT_OK) return st;
    return check_packed_buffers(w, w->rows, w->k);
}

struct LoraArgs {
    int32_t r = 0;
    const void *t = nullptr;
    int64_t ldt = 0;
    const void *b = nullptr;
    int64_t ldb = 0;
    bool t_is_scratch = false;  // T_ext is the library's static scratch (non-null, 256-byte aligned)
};

bool lora_rank_ok(int32_t r) { return r >= 16 && r <= 256 && r % 16 == 0; }

// Host-side checks of a GEMM request; CONVROT_OK means run_gemm launches.
convrot_status check_gemm(const convrot_packed *x, const convrot_packed *w, const float *bias, float *Y,
                          int32_t *A, int64_t ld, int32_t act, int32_t *dev_status,
                          const LoraArgs &lora = LoraArgs{})
{
    if (act < CONVROT_ACT_NONE || act > CONVROT_ACT_GELU_TANH) return CONVROT_ERR_INVALID_ARG;
    convrot_status st = check_pair(x, w);
    if (st != CONVROT_OK) return st;
    const int64_t m = x->rows, n = w->rows;
    if (ld < n) return CONVROT_ERR_INVALID_ARG;
    if (lora.r != 0) {
        if (!lora_rank_ok(lora.r)) return CONVROT_ERR_INVALID_ARG;
        if (x->codes != CONVROT_CODES_BF16) return CONVROT_ERR_UNSUPPORTED;
        const int64_t cols = (3 * int64_t{lora.r} + 63) / 64 * 64;
        if (lora.ldt < cols || lora.ldb < cols) return CONVROT_ERR_INVALID_ARG;
        if (m > 0 && n > 0) {
            if (!lora.b || (!lora.t_is_scratch && !lora.t)) return CONVROT_ERR_INVALID_ARG;
            if ((!lora.t_is_scratch && !aligned(lora.t, 16)) || !aligned(lora.b, 16) || lora.ldt % 8 ||
                lora.ldb % 8)
                return CONVROT_ERR_ALIGNMENT;
        }
    }
    if (m > 0 && n > 0) {
        void *out = Y ? static_cast<void *>(Y) : static_cast<void *>(A);
        if (!out) return CONVROT_ERR_INVALID_ARG;
        if (!aligned(out, 16) || ld % 4 != 0) return CONVROT_ERR_ALIGNMENT;
        if (bias && !aligned(bias, 4)) return CONVROT_ERR_ALIGNMENT;
        if (dev_status && !aligned(dev_status, 4)) return CONVROT_ERR_ALIGNMENT;
    }
    return CONVROT_OK;
}

convrot_status run_gemm(const convrot_packed *x, const convrot_packed *w, const float *bias, float *Y,
                        int32_t *A, int64_t ld, int32_t act, int32_t *dev_status, cudaStream_t stream,
                        const LoraArgs &lora = LoraArgs{})
{
    const convrot_status st = check_gemm(x, w, bias, Y, A, ld, act, dev_status, lora);
    if (st != CONVROT_OK) return st;
    const int64_t m = x->rows, n = w->rows;
    if (m == 0 || n == 0) return CONVROT_OK;
    convrot::GemmArgs g{};
    g.qx = x->q;
    g.ldqx = x->ldq;
    g.qw = w->q;
    g.ldqw = w->ldq;
    g.m = m;
    g.n = n;
    g.kpad = static_cast<int32_t>(convrot_ldq(x->k));
    g.sx = x->scale;
    g.sw = w->scale;
    g.bias = bias;
    g.y = Y;
    g.a = A;
    g.ldy = ld;
    g.dev_status = dev_status;
    g.act = act;
    g.lora_r = lora.r;
    g.lora_t = lora.t;
    g.lora_ldt = lora.ldt;
    g.lora_b = lora.b;
    g.lora_ldb = lora.ldb;
    g.i8 = x->codes == CONVROT_CODES_I8 ? 1 : 0;
    cudaError_t e = convrot::launch_gemm_tc(g, stream);
    if (e == cudaErrorNotSupported) return CONVROT_ERR_UNSUPPORTED;
    return e == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}

// Work layout of convrot_linear_act_pack: H [m, ldh] fp32 (ldh = n rounded up to
// 64) at offset 0, then the row maxima [m] (32-bit words), each part 256-byte aligned.
int64_t pack_work_ldh(int64_t n) { return (n + 63) / 64 * 64; }
int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }
int64_t pack_work_h_bytes(int64_t m, int64_t n) { return round256(m * pack_work_ldh(n) * 4); }

}  // namespace

extern "C" {

int64_t convrot_linear_pack_work_bytes(int64_t m, int64_t n)
{
    if (m < 0 || n < 1 || n > CONVROT_MAX_K) return 0;
    return pack_work_h_bytes(m, n) + round256(m * 4);
}

convrot_status convrot_linear_act_pack(const convrot_packed *x, const convrot_packed *w, const float *bias,
                                       int32_t act, int32_t G, void *work, int64_t work_bytes, convrot_packed *out_h,
                                       int32_t *dev_status, cudaStream_t stream)
{
    if (!x || !w || !out_h) return CONVROT_ERR_INVALID_ARG;
    const int64_t m = x->rows, n = w->rows;
    if (m < 0 || n < 0) return CONVROT_ERR_INVALID_ARG;
    int log4g = 0;
    // the output is the next linear's input: n is that linear's k
    convrot_status st = check_k_g(n, G, &log4g);
    if (st != CONVROT_OK) return st;
    st = check_packed_buffers(out_h, m, n);
    if (st != CONVROT_OK) return st;
    const int64_t ldh = pack_work_ldh(n);
    if (m > 0) {
        if (!work || work_bytes < convrot_linear_pack_work_bytes(m, n)) return CONVROT_ERR_INVALID_ARG;
        if (!aligned(work, 256)) return CONVROT_ERR_ALIGNMENT;
    }
    float *H = static_cast<float *>(work);
    st = check_gemm(x, w, bias, m > 0 ? H : nullptr, nullptr, ldh, act, dev_status);
    if (st != CONVROT_OK) return st;
    if (m == 0) {
        out_h->rows = 0;
        out_h->k = n;
        out_h->group_size = G;
        return CONVROT_OK;
    }
    const bool fused = x->codes == CONVROT_CODES_BF16 && n % 256 == 0 && G <= 256;
    if (!fused) {  // the same result in two launches: the linear into the work buffer, then the pack
        st = run_gemm(x, w, bias, H, nullptr, ldh, act, dev_status, stream);
        if (st != CONVROT_OK) return st;
        return pack_rows(H, m, n, ldh, G, out_h, dev_status, stream);
    }
    uint32_t *rowmax = reinterpret_cast<uint32_t *>(static_cast<char *>(work) + pack_work_h_bytes(m, n));
    if (cudaMemsetAsync(rowmax, 0, static_cast<size_t>(m) * 4, stream) != cudaSuccess) return CONVROT_ERR_CUDA;
    convrot::GemmArgs g{};
    g.qx = x->q;
    g.ldqx = x->ldq;
    g.qw = w->q;
    g.ldqw = w->ldq;
    g.m = m;
    g.n = n;
    g.kpad = static_cast<int32_t>(convrot_ldq(x->k));
    g.sx = x->scale;
    g.sw = w->scale;
    g.bias = bias;
    g.a = reinterpret_cast<int32_t *>(H);  // the rotated values, stored as 32-bit words
    g.ldy = ldh;
    g.dev_status = dev_status;
    g.act = act;
    g.rot_digits = log4g;
    g.rot_rowmax = rowmax;
    if (convrot::launch_gemm_tc(g, stream) != cudaSuccess) return CONVROT_ERR_CUDA;
    out_h->rows = m;
    out_h->k = n;
    out_h->group_size = G;
    return convrot::launch_requant(H, ldh, rowmax, m, static_cast<int32_t>(n), log4g, out_h->q, out_h->ldq,
                                   out_h->scale, out_h->codes == CONVROT_CODES_BF16, stream) == cudaSuccess
               ? CONVROT_OK
               : CONVROT_ERR_CUDA;
}

int64_t convrot_ldq(int64_t k) { return k <= 0 ? 0 : ((k + 127) / 128) * 128; }

convrot_status convrot_quantize_weights(const float *W, int64_t n, int64_t k, int64_t ldw, int32_t G,
                                        convrot_packed *out_w, int32_t *dev_status, cudaStream_t stream)
{
    return pack_rows(W, n, k, ldw, G, out_w, dev_status, stream);
}

convrot_status convrot_pack_activations(const float *X, int64_t m, int64_t k, int64_t ldx, int32_t G,
                                        convrot_packed *out_x, int32_t *dev_status, cudaStream_t stream)
{
    return pack_rows(X, m, k, ldx, G, out_x, dev_status, stream);
}

convrot_status convrot_linear(const convrot_packed *x, const convrot_packed *w, const float *bias,
                              float *Y, int64_t ldy, int32_t *dev_status, cudaStream_t stream)
{
    if (!Y && x && w && x->rows > 0 && w->rows > 0) return CONVROT_ERR_INVALID_ARG;
    return run_gemm(x, w, bias, Y, nullptr, ldy, CONVROT_ACT_NONE, dev_status, stream);
}

convrot_status convrot_linear_act(const convrot_packed *x, const convrot_packed *w, const float *bias, int32_t act,
                                  float *Y, int64_t ldy, int32_t *dev_status, cudaStream_t stream)
{
    if (!Y && x && w && x->rows > 0 && w->rows > 0) return CONVROT_ERR_INVALID_ARG;
    return run_gemm(x, w, bias, Y, nullptr, ldy, act, dev_status, stream);
}

int64_t convrot_lora_cols(int32_t r) { return lora_rank_ok(r) ? (3 * int64_t{r} + 63) / 64 * 64 : 0; }

convrot_status convrot_lora_prepare(const float *B, int64_t n, int32_t r, int64_t ldb, float scale, void *B_ext,
                                    int64_t lde, cudaStream_t stream)
{
    if (!lora_rank_ok(r) || n < 0 || ldb < r || lde < convrot_lora_cols(r)) return CONVROT_ERR_INVALID_ARG;
    if (n == 0) return CONVROT_OK;
    if (!B || !B_ext) return CONVROT_ERR_INVALID_ARG;
    if (!aligned(B, 4) || !aligned(B_ext, 16) || lde % 8 != 0) return CONVROT_ERR_ALIGNMENT;
    return convrot::launch_lora_prepare(B, n, r, ldb, scale, B_ext, lde, stream) == cudaSuccess ? CONVROT_OK
                                                                                               : CONVROT_ERR_CUDA;
}

convrot_status convrot_lora_prepare_down(const float *A, int32_t r, int64_t k, int64_t lda, float *A_ext,
                                         int64_t lde, cudaStream_t stream)
{
    if (!lora_rank_ok(r)) return CONVROT_ERR_INVALID_ARG;
    if (k < 1 || k > CONVROT_MAX_K) return CONVROT_ERR_K_RANGE;
    if (lda < k || lde < k) return CONVROT_ERR_INVALID_ARG;
    if (!A || !A_ext) return CONVROT_ERR_INVALID_ARG;
    if (!aligned(A, 4) || !aligned(A_ext, 16) || lde % 4 != 0) return CONVROT_ERR_ALIGNMENT;
    return convrot::launch_lora_prepare_down(A, r, static_cast<int32_t>(k), lda, A_ext, lde, stream) == cudaSuccess
               ? CONVROT_OK
               : CONVROT_ERR_CUDA;
}

convrot_status convrot_lora_down(const float *X, int64_t m, int64_t k, int64_t ldx, const float *A, int32_t r,
                                 int64_t lda, void *T_ext, int64_t ldt, int32_t *dev_status, cudaStream_t stream)
{
    if (!lora_rank_ok(r) || m < 0 || ldt < convrot_lora_cols(r)) return CONVROT_ERR_INVALID_ARG;
    if (k < 1 || k > CONVROT_MAX_K) return CONVROT_ERR_K_RANGE;
    if (ldx < k || lda < k || ldx % 4 != 0 || lda % 4 != 0) return CONVROT_ERR_INVALID_ARG;
    if (m == 0) return CONVROT_OK;
    if (!X || !A || !T_ext) return CONVROT_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(A, 16) || !aligned(T_ext, 16) || ldt % 8 != 0) return CONVROT_ERR_ALIGNMENT;
    if (dev_status && !aligned(dev_status, 4)) return CONVROT_ERR_ALIGNMENT;
    return convrot::launch_lora_down(X, m, static_cast<int32_t>(k), ldx, A, r, lda, T_ext, ldt, dev_status, stream) ==
                   cudaSuccess
               ? CONVROT_OK
               : CONVROT_ERR_CUDA;
}

convrot_status convrot_linear_lora(const convrot_packed *x, const convrot_packed *w, const float *bias, int32_t act,
                                   const void *T_ext, int64_t ldt, const void *B_ext, int64_t lde, int32_t r,
                                   float *Y, int64_t ldy, int32_t *dev_status, cudaStream_t stream)
{
    if (!Y && x && w && x->rows > 0 && w->rows > 0) return CONVROT_ERR_INVALID_ARG;
    if (r == 0) return CONVROT_ERR_INVALID_ARG;
    LoraArgs lora;
    lora.r = r;
    lora.t = T_ext;
    lora.ldt = ldt;
    lora.b = B_ext;
    lora.ldb = lde;
    return run_gemm(x, w, bias, Y, nullptr, ldy, act, dev_status, stream, lora);
}

convrot_status convrot_linear_lora_noalloc(const convrot_packed *x, const convrot_packed *w, const float *bias,
                                           int32_t act, const float *X, int64_t ldx, const float *A_ext, int64_t lda,
                                           const void *B_ext, int64_t lde, int32_t r, float *Y, int64_t ldy,
                                           int32_t *dev_status, cudaStream_t stream)
{
    if (!x || !w) return CONVROT_ERR_INVALID_ARG;
    if (!lora_rank_ok(r)) return CONVROT_ERR_INVALID_ARG;
    const int64_t cols = convrot_lora_cols(r);
    if (x->rows < 0) return CONVROT_ERR_INVALID_ARG;
    if (x->rows > CONVROT_NOALLOC_SCRATCH_BYTES / (cols * 2)) return CONVROT_ERR_SCRATCH;
    if (x->rows == 0 || w->rows == 0) return convrot_linear_lora(x, w, bias, act, nullptr, cols, B_ext, lde, r, Y, ldy,
                                                                 dev_status, stream);
    // every check of the linear comes before the first launch, as for the other entry points
    LoraArgs lora;
    lora.r = r;
    lora.ldt = cols;
    lora.b = B_ext;
    lora.ldb = lde;
    lora.t_is_scratch = true;
    convrot_status st = check_gemm(x, w, bias, Y, nullptr, ldy, act, dev_status, lora);
    if (st != CONVROT_OK) return st;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return CONVROT_ERR_CUDA;
    st = convrot_lora_down(X, x->rows, x->k, ldx, A_ext, r, lda, scratch, cols, dev_status, stream);
    if (st != CONVROT_OK) return st;
    return convrot_linear_lora(x, w, bias, act, scratch, cols, B_ext, lde, r, Y, ldy, dev_status, stream);
}

convrot_status convrot_gemm_i32(const convrot_packed *x, const convrot_packed *w, int32_t *A,
                                int64_t lda, int32_t *dev_status, cudaStream_t stream)
{
    if (!A && x && w && x->rows > 0 && w->rows > 0) return CONVROT_ERR_INVALID_ARG;
    return run_gemm(x, w, nullptr, nullptr, A, lda, CONVROT_ACT_NONE, dev_status, stream);
}

convrot_status convrot_wait_check(int32_t *dev_status, uint64_t limit_ns, int32_t arrive, cudaStream_t stream)
{
    if (!dev_status || limit_ns == 0 || limit_ns > CONVROT_WAIT_LIMIT_NS) return CONVROT_ERR_INVALID_ARG;
    return convrot::launch_wait_check(dev_status, limit_ns, arrive, stream) == cudaSuccess ? CONVROT_OK
                                                                                           : CONVROT_ERR_CUDA;
}

const char *convrot_status_string(convrot_status s)
{
    switch (s) {
    case CONVROT_OK: return "ok";
    case CONVROT_ERR_INVALID_ARG: return "invalid argument";
    case CONVROT_ERR_GROUP_SIZE: return "group size must be 4^n (n >= 1, at most 65536) and divide k";
    case CONVROT_ERR_ALIGNMENT: return "pointer or leading dimension is not suitably aligned";
    case CONVROT_ERR_K_RANGE: return "k must be in [1, 133144]";
    case CONVROT_ERR_CUDA: return "CUDA launch failed";
    case CONVROT_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case CONVROT_ERR_UNSUPPORTED: return "valid request that no kernel of the library supports (e.g. LoRA with I8 codes)";
    case CONVROT_ERR_SCRATCH: return "request larger than the static scratch of the no-allocation entry point";
    default: return "unknown status";
    }
}

}  // extern "C"

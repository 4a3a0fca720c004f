/*
 * convrot.h -- C ABI of libconvrot, the GB300 (sm_103a) INT8 convrot linear.
 *
 * The layer is the one defined on the page "INT8 Convrot Safetensors"
 * (stable-diffusion.cpp docs, int8_convrot.md):
 *
 *   X_rot = X R            R = block-diagonal normalized Kronecker power of
 *                          H4, one block per contiguous group of G = 4^n
 *                          input features ("How INT8 convrot works")
 *   s_x[r] = max_i |X_rot[r, i]| / 127
 *   Q_x[r, i] = clamp(round(X_rot[r, i] / s_x[r]), -127, 127)
 *                          ("Runtime activation quantization"; weights use the
 *                          same formulas offline, "Weight quantization")
 *   A[r, o] = sum_i Q_x[r, i] * Q_w[o, i]      (signed 32-bit)
 *   Y[r, o] = A[r, o] * s_x[r] * s_w[o] + b[o]
 *
 * "round" is round half away from zero. A row whose rotated values are all
 * zero gets scale 0 and codes 0 (so its outputs are the bias).
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers unless stated otherwise, in
 *     row-major layout with the given leading dimension (in elements).
 *   - The caller owns every buffer. The library never allocates, frees or
 *     synchronizes; all work is enqueued on `stream` (0 = legacy default).
 *   - Arguments are validated on the host before anything is enqueued; a
 *     non-OK status means nothing was launched.
 *   - CONVROT_ERR_CUDA means a launch failed; the CUDA error is left for the
 *     caller to query (cudaGetLastError / cudaPeekAtLastError).
 *   - Inputs must not alias outputs. Results are deterministic.
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef CONVROT_H_
#define CONVROT_H_

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONVROT_OK = 0,
    CONVROT_ERR_INVALID_ARG = 1, /* null pointer, negative size, ld too small, mismatched operands */
    CONVROT_ERR_GROUP_SIZE = 2,  /* G not 4^n (n >= 1), G does not divide k, or G > 65536 */
    CONVROT_ERR_ALIGNMENT = 3,   /* a pointer or leading dimension breaks the alignment rules */
    CONVROT_ERR_K_RANGE = 4,     /* k < 1 or k > CONVROT_MAX_K */
    CONVROT_ERR_CUDA = 5,        /* a kernel launch failed */
    CONVROT_ERR_TIMEOUT = 6,     /* written to *dev_status by a kernel whose bounded wait ran out */
    CONVROT_ERR_UNSUPPORTED = 7, /* valid request that no kernel of the library supports */
    CONVROT_ERR_SCRATCH = 8      /* larger than the static scratch of convrot_linear_lora_noalloc */
} convrot_status;

/* Largest k: 127 * 127 * k must fit in a signed 32-bit accumulator ("Runtime
 * activation quantization" accumulates in signed 32-bit integers). */
#define CONVROT_MAX_K 133144

/* Largest group size: 4^8, the largest power of four that can divide a k
 * within CONVROT_MAX_K (the page admits any power of four dividing the input
 * features, "Checkpoint format"). */
#define CONVROT_MAX_GROUP 65536

/* Element type of the stored codes. Both hold the same integers in
 * [-127, 127]; BF16 represents every one of them exactly and is the operand
 * type the tensor-core GEMM reads directly. I8 (the page's storage) is read
 * by the same tensor-core GEMM, which widens it to f16 in shared memory
 * (m <= 128: a warp-level int8 MMA kernel); both give the same integers. */
typedef enum {
    CONVROT_CODES_I8 = 0,
    CONVROT_CODES_BF16 = 1
} convrot_codes;

/*
 * Activation applied to Y inside the linear's epilogue. The page's layer is a
 * plain linear; a DiT MLP applies GELU to its up projection's output before
 * the down projection packs it, and fusing it here saves a separate pass over
 * that output. GELU(v) = v * Phi(v) with Phi the standard normal CDF:
 *   CONVROT_ACT_GELU_ERF   0.5 v (1 + erf(v / sqrt(2)))
 *   CONVROT_ACT_GELU_TANH  0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
 */
typedef enum {
    CONVROT_ACT_NONE = 0,
    CONVROT_ACT_GELU_ERF = 1,
    CONVROT_ACT_GELU_TANH = 2
} convrot_activation;

/*
 * A packed, rotated and quantized row block: the page's "packed runtime
 * activation tensor" (I8 rows plus one floating-point scale per row,
 * "Runtime activation quantization"), and equally a quantized weight (Q_w,
 * s_w; "Weight quantization" stores one scale per output row, 1-D).
 * Linears that share an input and G reuse one packed activation.
 *
 *   q          device, [rows, ldq] codes of type `codes`; columns k..kpad-1
 *              (kpad = convrot_ldq(k)) are zero, columns past kpad are
 *              neither read nor written. 16-byte aligned.
 *   scale      device, [rows] fp32, 4-byte aligned.
 *   rows, k    logical shape.
 *   ldq        row pitch in elements; ldq >= convrot_ldq(k) and ldq % 16 == 0.
 *   group_size G it was rotated with.
 *   codes      a convrot_codes value.
 *
 * The pack functions read ldq, codes, q and scale from *out and fill rows,
 * k and group_size.
 */
typedef struct {
    void *q;
    float *scale;
    int64_t rows;
    int64_t k;
    int64_t ldq;
    int32_t group_size;
    int32_t codes;
} convrot_packed;

/* Padded code row length the GEMM reads: k rounded up to a multiple of 128. */
int64_t convrot_ldq(int64_t k);

/*
 * Offline weight quantization ("Weight quantization"): W_rot = W R,
 * s_w[o] = max_i |W_rot[o, i]| / 127, Q_w = clamp(round(W_rot / s_w), +-127).
 *   W      device fp32 [n, ldw], 16-byte aligned, ldw >= k, ldw % 4 == 0.
 *   n      output features (rows of W), n >= 0 (0: nothing is launched).
 *   k      input features, 1 <= k <= CONVROT_MAX_K.
 *   G      4^m with m >= 1, G | k, G <= CONVROT_MAX_GROUP.
 *   out_w  caller-filled q/scale/ldq/codes; receives rows = n, k, G.
 *   dev_status  as for convrot_linear.
 * Same kernel as convrot_pack_activations.
 */
convrot_status convrot_quantize_weights(const float *W, int64_t n, int64_t k, int64_t ldw,
                                        int32_t G, convrot_packed *out_w, int32_t *dev_status,
                                        cudaStream_t stream);

/*
 * Runtime activation pack ("Runtime activation quantization"): rotate each
 * row of X group-wise, take one absmax scale over the whole rotated row, and
 * write the codes and the scale. One fused kernel: X is read once.
 *   X      device fp32 [m, ldx], 16-byte aligned, ldx >= k, ldx % 4 == 0.
 *   m      rows (tokens), m >= 0 (0: nothing is launched).
 *   k, G   as for convrot_quantize_weights.
 *   out_x  caller-filled q/scale/ldq/codes; receives rows = m, k, G.
 *   dev_status  device int32 or NULL; see convrot_linear. (For G <= 1024 the
 *               pack streams rows into shared memory with bulk copies and
 *               waits for them with a 4 s bound; the other forms never wait.)
 */
convrot_status convrot_pack_activations(const float *X, int64_t m, int64_t k, int64_t ldx,
                                        int32_t G, convrot_packed *out_x, int32_t *dev_status,
                                        cudaStream_t stream);

/*
 * The linear: A = Q_x Q_w^T in exact integer arithmetic, then
 * Y[r, o] = A[r, o] * s_x[r] * s_w[o] + b[o] in fp32 ("Runtime activation
 * quantization"), fused into the GEMM's epilogue.
 *   x          packed activations (m = x->rows).
 *   w          packed weights (n = w->rows); same k, group_size and codes as x.
 *   bias       device fp32 [n], or NULL for no bias.
 *   Y          device fp32 [m, ldy], 16-byte aligned, ldy >= n, ldy % 4 == 0.
 *   dev_status device int32 or NULL. A kernel that gives up a bounded wait
 *              writes CONVROT_ERR_TIMEOUT there (read it after synchronizing);
 *              it is never written otherwise, so the caller zeroes it first.
 * m == 0 or n == 0 launches nothing.
 */
convrot_status convrot_linear(const convrot_packed *x, const convrot_packed *w, const float *bias,
                              float *Y, int64_t ldy, int32_t *dev_status, cudaStream_t stream);

/*
 * The linear followed by an activation in the same epilogue:
 * Y[r, o] = act(A[r, o] * s_x[r] * s_w[o] + b[o]). No counterpart on the page
 * (it defines the linear alone); see convrot_activation.
 *   act  a convrot_activation value; anything else is CONVROT_ERR_INVALID_ARG.
 * Everything else as for convrot_linear (which is act = CONVROT_ACT_NONE).
 */
convrot_status convrot_linear_act(const convrot_packed *x, const convrot_packed *w, const float *bias,
                                  int32_t act, float *Y, int64_t ldy, int32_t *dev_status,
                                  cudaStream_t stream);

/*
 * The linear with an activation, followed by the pack of its output for the
 * next linear ("Runtime activation quantization" applied to H): out_h receives
 * the codes and row scales of H = act(x w^T linear) rotated with group size G,
 * exactly what convrot_linear_act into an [m, n] buffer followed by
 * convrot_pack_activations(H, G) gives (H is the same; codes may differ only
 * at exact-tie ulps of the rotation's fp32 summation order). No counterpart
 * on the page as one call: it is the page's pack of the next layer's input,
 * moved into this layer's epilogue (a DiT MLP's up projection feeding its
 * down projection).
 *   act, bias        as for convrot_linear_act.
 *   G                the next linear's group size: 4^n, G | n (n = w->rows).
 *   work, work_bytes device workspace, 256-byte aligned, at least
 *                    convrot_linear_pack_work_bytes(m, n) bytes; it holds the
 *                    rotated H and its row maxima; its contents are undefined
 *                    afterwards and need no initialization.
 *   out_h            caller-filled q/scale/ldq/codes as for
 *                    convrot_pack_activations (ldq >= convrot_ldq(n));
 *                    receives rows = m, k = n, group_size = G.
 * Fused form (bf16 codes, n % 256 == 0, G <= 256): the GEMM's epilogue applies
 * the activation, the rotation (a 256-column output tile row is whole groups)
 * and an atomic row absmax, and stores the rotated values to work; a second
 * launch quantizes them (reading the most recently stored columns first, while
 * they are still in L2). Other requests run the linear into work and then the
 * pack. Errors as for convrot_linear_act and convrot_pack_activations;
 * CONVROT_ERR_INVALID_ARG for a missing or short work buffer.
 */
int64_t convrot_linear_pack_work_bytes(int64_t m, int64_t n);
convrot_status convrot_linear_act_pack(const convrot_packed *x, const convrot_packed *w, const float *bias,
                                       int32_t act, int32_t G, void *work, int64_t work_bytes, convrot_packed *out_h,
                                       int32_t *dev_status, cudaStream_t stream);

/*
 * Runtime LoRA side branch (page "INT8 Convrot Safetensors", "Backend
 * support", paragraph on adapters): the INT8 weights stay as they are, and
 * the adapter's correction is computed from the original, unrotated
 * activation and added to the linear's output:
 *   Y = act(A s_x s_w + b + scale * (X A_lora^T) B_lora^T)
 * with A_lora [r, k] (down) and B_lora [n, r] (up). The correction runs on the
 * tensor cores in split precision (T = X A_lora^T with three-term TF32, then
 * T B^T with two-term bf16 on both sides), close to an fp32 computation.
 *
 * convrot_lora_cols(r): the K extent of the extended operands, 3 r rounded up
 * to 64 (0 for an r that is not accepted). r must be a multiple of 16 in
 * [16, 256].
 */
int64_t convrot_lora_cols(int32_t r);

/*
 * Offline, once per adapter: B_ext [n, lde] bf16 =
 * [hi(scale B) | lo(scale B) | hi(scale B) | 0 ...], hi = bf16(v),
 * lo = bf16(v - hi).
 *   B       device fp32 [n, ldb], 4-byte aligned, ldb >= r.
 *   scale   the adapter's scale (alpha / r in the usual files).
 *   B_ext   device, 16-byte aligned, lde >= convrot_lora_cols(r), lde % 8 == 0.
 */
convrot_status convrot_lora_prepare(const float *B, int64_t n, int32_t r, int64_t ldb, float scale,
                                    void *B_ext, int64_t lde, cudaStream_t stream);

/*
 * Offline, once per adapter: A_ext [2r, lde] fp32 = [hi(A); lo(A)], hi = A with
 * its low 13 mantissa bits cleared (exact in TF32), lo = A - hi.
 *   A       device fp32 [r, lda], 4-byte aligned, lda >= k, 1 <= k <= CONVROT_MAX_K.
 *   A_ext   device, 16-byte aligned, lde >= k, lde % 4 == 0.
 */
convrot_status convrot_lora_prepare_down(const float *A, int32_t r, int64_t k, int64_t lda, float *A_ext,
                                         int64_t lde, cudaStream_t stream);

/*
 * Per call: T = X A_lora^T from the unrotated X, written as
 * T_ext [m, ldt] bf16 = [hi(T) | hi(T) | lo(T) | 0 ...].
 *   X       device fp32 [m, ldx] (the same X the pack reads), 16-byte aligned,
 *           ldx >= k, ldx % 4 == 0; 1 <= k <= CONVROT_MAX_K.
 *   A_ext   from convrot_lora_prepare_down: device fp32 [2r, lda], 16-byte
 *           aligned, lda >= k, lda % 4 == 0.
 *   T_ext   device, 16-byte aligned, ldt >= convrot_lora_cols(r), ldt % 8 == 0.
 *   dev_status  as for convrot_linear (the kernel waits on its copies with a
 *               4 s bound).
 */
convrot_status convrot_lora_down(const float *X, int64_t m, int64_t k, int64_t ldx, const float *A_ext, int32_t r,
                                 int64_t lda, void *T_ext, int64_t ldt, int32_t *dev_status, cudaStream_t stream);

/*
 * The linear with the LoRA correction added in its epilogue (bf16 codes only;
 * I8 codes give CONVROT_ERR_UNSUPPORTED): Y = act(base + T_ext B_ext^T).
 *   T_ext, ldt  from convrot_lora_down on this x's activations (x->rows rows).
 *   B_ext, lde  from convrot_lora_prepare (w->rows rows).
 *   r           the adapter's rank, as given to both.
 * Everything else as for convrot_linear_act.
 */
convrot_status convrot_linear_lora(const convrot_packed *x, const convrot_packed *w, const float *bias, int32_t act,
                                   const void *T_ext, int64_t ldt, const void *B_ext, int64_t lde, int32_t r,
                                   float *Y, int64_t ldy, int32_t *dev_status, cudaStream_t stream);

/*
 * No counterpart on the page (an entry point of this library only): the LoRA
 * linear in one call that allocates nothing, not even the T_ext that
 * convrot_lora_down / convrot_linear_lora ask the caller for.
 *
 * Who needs it: callers that must not call cudaMalloc. A plug-in running
 * inside a host application whose device memory belongs to that
 * application's own pool (a framework's caching allocator, an arena sized
 * once at start-up) cannot take memory behind the pool's back; a real-time
 * or latency-bound loop cannot afford cudaMalloc's cost or the device-wide
 * synchronization that an allocation or free may bring; and code with a
 * fixed device-memory budget set at load time cannot grow it per call.
 *
 * It runs convrot_lora_down into a file-scope device array of the library
 * (CONVROT_NOALLOC_SCRATCH_BYTES = 32 MiB, 256-byte aligned), then
 * convrot_linear_lora reading it. Results equal those of the two calls with
 * a caller's T_ext.
 *   X, ldx  the activations x was packed from: device fp32 [x->rows, ldx],
 *           ldx >= x->k (k = x->k), 16-byte aligned, ldx % 4 == 0.
 *   A_ext, lda  convrot_lora_prepare_down's output for this same r:
 *           device fp32 [2 r, lda], lda >= x->k.
 *   B_ext, lde, r, bias, act, Y, ldy, dev_status   as for convrot_linear_lora.
 * The library takes the row count of X from x->rows and the rows of A_ext
 * from r; it cannot see either buffer's size, so an X with fewer rows or
 * columns, or an A_ext prepared for another rank, makes the kernels read
 * past those buffers. (The Python binding checks both shapes before the call.)
 * Limits and errors: a request whose T_ext (x->rows * convrot_lora_cols(r)
 * bf16 values; e.g. up to 87381 rows at r = 64, 21845 at r = 256) exceeds
 * the array returns CONVROT_ERR_SCRATCH and launches nothing; a failed
 * address lookup returns CONVROT_ERR_CUDA.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress and keeps it for that
 * device's context; make that first call before any stream capture.
 * Sharing: every GPU that loads the library holds the array until the
 * process exits, and every call on a device shares that device's array,
 * which keeps the last call's contents. Nothing in it must start at zero
 * (the down kernel writes every column the GEMM reads, padding included), so
 * nothing is cleared. Calls that overlap on the GPU (on different streams,
 * or from different host threads) race on it; serialize them, e.g. on one
 * stream.
 */
#define CONVROT_NOALLOC_SCRATCH_BYTES (32ll << 20)
convrot_status convrot_linear_lora_noalloc(const convrot_packed *x, const convrot_packed *w, const float *bias,
                                           int32_t act, const float *X, int64_t ldx, const float *A_ext, int64_t lda,
                                           const void *B_ext, int64_t lde, int32_t r, float *Y, int64_t ldy,
                                           int32_t *dev_status, cudaStream_t stream);

/*
 * The integer GEMM alone: A[r, o] = sum_i Q_x[r, i] * Q_w[o, i] as int32, for
 * checking the accumulation bit for bit. Same operand rules as
 * convrot_linear.
 *   A      device int32 [m, lda], 16-byte aligned, lda >= n, lda % 4 == 0.
 */
convrot_status convrot_gemm_i32(const convrot_packed *x, const convrot_packed *w, int32_t *A,
                                int64_t lda, int32_t *dev_status, cudaStream_t stream);

/*
 * No counterpart on the page (an entry point of this library only): checks
 * failure detection without a fault. One CTA waits on an mbarrier through
 * the same bounded wait that the GEMM, LoRA and ring-pack kernels use on
 * their copies and MMAs (those use the limit CONVROT_WAIT_LIMIT_NS).
 *   dev_status  device int32, non-NULL. With arrive == 0 nothing arrives:
 *               the wait gives up after limit_ns and the kernel writes
 *               CONVROT_ERR_TIMEOUT there, as those kernels do on a stall.
 *               With arrive != 0 the wait ends at once and it is untouched.
 *   limit_ns    in (0, CONVROT_WAIT_LIMIT_NS]; anything else is
 *               CONVROT_ERR_INVALID_ARG and launches nothing.
 * The kernel returns normally either way; the context stays usable.
 */
#define CONVROT_WAIT_LIMIT_NS 4000000000ull
convrot_status convrot_wait_check(int32_t *dev_status, uint64_t limit_ns, int32_t arrive, cudaStream_t stream);

/* Static, NUL-terminated description of a status. Never NULL. */
const char *convrot_status_string(convrot_status status);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H_ */

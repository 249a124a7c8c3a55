/*
 * lora_gb300.h -- C ABI of the fused low-rank-adapted linear layer for GB300 (sm_103a).
 *
 * The layer:  y = X W0^T + s (X A^T) B^T (+ bias)   forward and backward, computed
 * without ever forming the dense update dW = B A or its gradient; the DoRA row-scale and
 * column-scale variants with their closed-form norms; a gated (SwiGLU / GeGLU) MLP built from
 * three such projections; a fused query/key/value projection with one adapter per leaf; and an
 * int8 (W8A8) base weight with a per-row dequant scale and a LoRA epilogue.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or retains them.  Tensors are row-major and contiguous:
 *      X [M, d_in], W0 [d_out, d_in], A [r, d_in] (down), B [d_out, r] (up),
 *      bias [d_out], m [d_out], Y / dY [M, d_out], Z = X A^T [M, r].
 *  - dtype LORA_BF16: bf16 storage, fp32 accumulation, bf16 outputs/gradients.
 *    dtype LORA_F32: fp32 storage, fp32 FMA accumulation (no TF32), fp32 outputs.
 *  - s is the complete scale strength * alpha / r (the caller folds strength in).
 *  - Every pointer must be 16-byte aligned; d_in, d_out must be multiples of 8,
 *    r a multiple of 8 with 8 <= r <= 128 (LORA_BF16) or 1 <= r <= 128 (LORA_F32).
 *    M >= 0 (M == 0 is a no-op).  Violations return an error before anything is
 *    launched and leave every output untouched.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  A returned LORA_OK means "validated and launched", not "finished".
 *  - `ws` is caller-allocated device scratch of at least *_workspace_bytes() bytes,
 *    256-byte aligned.  Its first 256 bytes hold a device error word that kernels set
 *    (never clear) when a bounded wait runs out; clear it once with
 *    lora_clear_device_error() before first use and read it with
 *    lora_check_device_error().  Two calls that share one workspace must not overlap
 *    on the GPU (same stream, or ordered by events).
 *  - Where the pages leave a step open, the plain reading is taken: eps is a floor on
 *    the DoRA row norm, n = max(sqrt(max(q, 0)), eps); strength 0 returns the frozen
 *    base layer X W0^T + bias (also for DoRA).
 *
 * Citations name the source page by its title and the section of it that defines the
 * operation.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,     /* null required pointer, bad shape, bad dtype, non-finite s */
    LORA_ERR_UNSUPPORTED = 2,     /* valid request this library does not implement (e.g. r > 128) */
    LORA_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned (ws: 256-byte) */
    LORA_ERR_WORKSPACE = 4,       /* ws is NULL or ws_bytes is below the required size */
    LORA_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed (launch, tensor map) */
    LORA_ERR_DEVICE_TIMEOUT = 6   /* a kernel's bounded wait ran out (read from the error word) */
} lora_status;

typedef enum { LORA_F32 = 0, LORA_BF16 = 1 } lora_dtype;

/* Operation ids for lora_workspace_bytes(). */
typedef enum {
    LORA_OP_LINEAR_FWD = 0, LORA_OP_LINEAR_BWD = 1,
    LORA_OP_DORA_FWD = 2, LORA_OP_DORA_BWD = 3,
    LORA_OP_MLP_FWD = 4, LORA_OP_MLP_BWD = 5,
    LORA_OP_QKV_FWD = 6, LORA_OP_QKV_BWD = 7,
    LORA_OP_DORA_COLS_FWD = 8, LORA_OP_DORA_COLS_BWD = 9,
    LORA_OP_DROPOUT_FWD = 10, LORA_OP_DROPOUT_BWD = 11
} lora_op;

typedef struct {
    int64_t M, d_in, d_out, r;
    int32_t dtype;                /* lora_dtype */
} lora_shape;

/* Gated MLP activation applied to the gate projection e (h = act(e) * u). */
typedef enum {
    LORA_ACT_SWIGLU = 0,          /* silu(e) = e * sigmoid(e) */
    LORA_ACT_GEGLU = 1            /* gelu(e) = e * Phi(e), Phi the normal CDF (erf form) */
} lora_act;

/* Gated MLP: X [M, H]; gate/up project H -> I, down projects I -> H; each projection has its
 * own rank (r_g, r_u, r_d: multiples of 8 in 8..128). */
typedef struct {
    int64_t M, H, I;
    int64_t r_g, r_u, r_d;
    int32_t dtype;                /* LORA_BF16 only */
    int32_t act;                  /* lora_act */
} lora_mlp_shape;

/* One adapted projection of the MLP: W [n_out, n_in], A [r, n_in], B [n_out, r], scale s. */
typedef struct {
    const void* W;
    const void* A;
    const void* B;
    float s;
} lora_proj;

/* Fused projection whose N = n[0] + .. + n[L-1] output columns split into L leaves (the
 * query / key / value heads of an attention block), each leaf with its own rank-r adapter.
 * L in 1..3; r a multiple of 8, at most 128 (the rank-r passes take at most 64 adapter columns at
 * a time: when L * r > 64 the leaves go in groups of at most 64 columns, or one leaf of more than
 * 64 columns, one extra pass over X per extra group or chunk); every n[l] a positive multiple of 8
 * (entries past L ignored); d_in a multiple of 8. */
typedef struct {
    int64_t M, d_in;
    int64_t n[3];
    int32_t L;
    int32_t r;
    int32_t dtype;                /* LORA_BF16 only */
} lora_qkv_shape;

/* One leaf's adapter: A [r, d_in] (down), B [n_l, r] (up), scale s. */
typedef struct {
    const void* A;
    const void* B;
    float s;
} lora_adapter;

/* Human-readable name of a status code (static storage, never NULL). */
const char* lora_status_string(int status);

/* Library ABI version (increments on any signature change). */
int lora_abi_version(void);

/* Bytes of workspace `op` needs for `sh` (LORA_OP_LINEAR_*, LORA_OP_DORA_*, LORA_OP_DORA_COLS_*
 * and LORA_OP_DROPOUT_*). 0 on bad input. */
size_t lora_workspace_bytes(int op, const lora_shape* sh);

/* Bytes of workspace the MLP entry points need (op = LORA_OP_MLP_FWD / LORA_OP_MLP_BWD). */
size_t lora_mlp_workspace_bytes(int op, const lora_mlp_shape* sh);

/* Bytes of workspace the fused-leaf entry points need (op = LORA_OP_QKV_FWD / LORA_OP_QKV_BWD). */
size_t lora_qkv_workspace_bytes(int op, const lora_qkv_shape* sh);

/* Zero the device error word at the head of `ws` (asynchronous on `stream`). */
lora_status lora_clear_device_error(void* ws, void* stream);

/* Synchronise `stream`, then read the device error word of `ws`:
 * LORA_OK if clear, LORA_ERR_DEVICE_TIMEOUT if a kernel recorded a timed-out wait. */
lora_status lora_check_device_error(const void* ws, void* stream);

/* ---------------------------------------------------------------- LoRA linear
 * Forward:  Y = X W0^T + s (X A^T) B^T (+ bias).
 * "LoRA/DoRA fast forward: no weight materialization" (stable-audio-3 #69), What
 * section: the low-rank update is folded into the data GEMMs; "How Unsloth's FastLoRA
 * Kernel Differs from Standard LoRA Implementations", Fused Forward Pass Architecture.
 *   bias:   [d_out] or NULL.
 *   Y:      [M, d_out] output.
 *   Z_save: [M, r] output or NULL; receives X A^T (unscaled) for the backward.
 */
lora_status lora_linear_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                            const void* B, const void* bias, float s, void* Y, void* Z_save,
                            void* ws, size_t ws_bytes, void* stream);

/* Size of the fixed device scratch used by lora_linear_fwd_noalloc (4 MiB). */
#define LORA_NOALLOC_SCRATCH_BYTES (4u << 20)

/* lora_linear_fwd without a workspace argument, for callers that cannot allocate device
 * memory: runtimes that plan all device memory before they start, plugin hosts that forbid
 * allocation once running, or hot paths that must not enter an allocator.  The source pages
 * have no counterpart to this entry point.
 *   Same arguments, layouts and results as lora_linear_fwd, minus ws / ws_bytes.  It
 *   allocates nothing (no cudaMalloc, no cudaFree, no allocating library call): its scratch
 *   is one fixed array of LORA_NOALLOC_SCRATCH_BYTES inside this library's device image,
 *   held by every GPU that loads the library until the process exits.
 *   Limit: the problem must fit that scratch, i.e. lora_workspace_bytes(LORA_OP_LINEAR_FWD,
 *   sh) <= LORA_NOALLOC_SCRATCH_BYTES (about M * r <= 2,097,000 for bf16, half that for
 *   fp32); larger problems return LORA_ERR_WORKSPACE and launch nothing.
 *   The first call on each device looks up the scratch's device address (with that device
 *   current); make that first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents (each call clears
 *   the part that must start at zero): two calls that overlap on the GPU, e.g. on two
 *   streams without ordering, race and corrupt each other.  A timed-out device wait is
 *   recorded only in that shared array and is not reported by this entry point. */
lora_status lora_linear_fwd_noalloc(const lora_shape* sh, const void* X, const void* W0, const void* A,
                                    const void* B, const void* bias, float s, void* Y, void* Z_save,
                                    void* stream);

/* Backward of lora_linear_fwd with W0 frozen:
 *   dX = dY W0 + s (dY B) A,  dA = s (dY B)^T X,  dB = s dY^T Z,  dbias = colsum(dY).
 * "How Unsloth's FastLoRA Kernel Differs ...", Custom Backward Pass Implementation (the
 * scale is folded into the gradient products); "nunchaku-style kernel fusion" (OneTrainer
 * #1680), commit reworking the 8-bit matmuls: the LoRA dgrad folds into the backward and
 * neither direction builds an (M, d_out) intermediate.
 *   Z_saved: [M, r] (X A^T from the forward) or NULL to recompute it.
 *   dX [M, d_in] or NULL (skipped); dA [r, d_in]; dB [d_out, r]; dbias [d_out] or NULL.
 */
lora_status lora_linear_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                            const void* B, const void* Z_saved, const void* dY, float s,
                            void* dX, void* dA, void* dB, void* dbias,
                            void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- LoRA with input dropout
 * The adapter branch sees a dropped-out copy of the input, the base does not:
 *   Xd = X o mask * keep_scale,  Y = X W0^T + s (Xd A^T) B^T (+ bias),
 * mask [M, d_in] uint8 (0 = dropped, 1 = kept; drawn by the caller, the same bytes for the
 * forward and the backward), keep_scale = 1 / (1 - p).  The mask sits between X and A, so this
 * call takes the unfused path: in the backward, the adapter's share of dX is a separate masked
 * rank-r pass instead of the dX GEMM's tail.
 * "Fused Kernels (experimental)" (LyCORIS docs), the note that a call whose mask sits between
 * two factors takes the unfused path; "How Unsloth's FastLoRA Kernel Differs ...", Optimized
 * Dropout and Scaling.  LORA_BF16 only (else LORA_ERR_UNSUPPORTED); other arguments as
 * lora_linear_fwd / _bwd.  mask must be 16-byte aligned and non-NULL when M > 0, keep_scale finite
 * and >= 0 (else LORA_ERR_INVALID_ARG).  With d_in a multiple of 16 no Xd is written: the rank-r
 * passes over X read the mask beside it and form Xd in registers, and the workspace is the plain
 * layer's; otherwise Xd is written once and the workspace adds M * d_in * 2 bytes
 * (lora_workspace_bytes with LORA_OP_DROPOUT_FWD / _BWD gives either).
 *   Backward: G = s dY B;  dX = dY W0 + (G A) o mask * keep_scale;  dA = G^T Xd;
 *             dB = s dY^T Z (Z = Xd A^T, saved by the forward or NULL to recompute);
 *             dbias = colsum(dY).
 */
lora_status lora_linear_dropout_fwd(const lora_shape* sh, const void* X, const uint8_t* mask, float keep_scale,
                                    const void* W0, const void* A, const void* B, const void* bias, float s,
                                    void* Y, void* Z_save, void* ws, size_t ws_bytes, void* stream);
lora_status lora_linear_dropout_bwd(const lora_shape* sh, const void* X, const uint8_t* mask, float keep_scale,
                                    const void* W0, const void* A, const void* B, const void* Z_saved,
                                    const void* dY, float s, void* dX, void* dA, void* dB, void* dbias,
                                    void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- DoRA (rows)
 * r0[o] = sum_k W0[o,k]^2 in fp32: the cached per-layer constant of the closed-form norm.
 * "LoRA/DoRA fast forward ...", commit message (cached rowsum(W0^2) constant) and What
 * section (the cached norm constant is a per-layer vector).  r0: [d_out] fp32 output.
 */
lora_status dora_rownorm2(const lora_shape* sh, const void* W0, float* r0, void* stream);

/* Forward:  n = max(sqrt(q), eps) with the closed form
 *   q = r0 + 2s rowsum((W0 A^T) o B) + s^2 rowsum((B (A A^T)) o B),
 *   Y = (m / n)[o] * (X W0^T + s (X A^T) B^T) + bias   (bias added after the row scale).
 * "LoRA/DoRA fast forward ...", What section (dora-rows is a row scale of the base +
 * low-rank output; norm in closed form) and Fidelity section (1e-12 eps, un-scaled bias).
 *   m [d_out], bias [d_out] or NULL, r0 [d_out] fp32 from dora_rownorm2.
 *   Y [M, d_out]; Z_save [M, r] or NULL; n_save [d_out] fp32 (required, for the backward);
 *   V_save [d_out, r] fp32 (required): W0 A^T, reused by the backward's norm gradient.
 */
lora_status dora_linear_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                            const void* B, const void* m, const void* bias, const float* r0,
                            float s, float eps, void* Y, void* Z_save, float* n_save, float* V_save,
                            void* ws, size_t ws_bytes, void* stream);

/* Backward of dora_linear_fwd, the norm kept in the graph (no detach):
 *   dc = colsum(dY o P) with P = (Y - bias) / c recovered from the saved output, c = m/n;
 *   dm = dc / n;  g = -m dc / (2 n^3) (0 where n was clamped at eps);
 *   dX = (dY o c) W0 + s ((dY o c) B) A;
 *   dA = s ((dY o c) B)^T X + 2s (g o B)^T W0 + 2s^2 (B^T diag(g) B) A;
 *   dB = s c o (dY^T Z) + 2s g o V + 2s^2 g o (B (A A^T)).
 * "LoRA/DoRA fast forward ...", Fidelity section (norm stays in the autograd graph;
 * gradients for A, B and the magnitude).
 *   Y, Z_saved (or NULL to recompute), n_saved and V_saved from the forward.
 *   dX [M, d_in] or NULL; dA [r, d_in]; dB [d_out, r]; dm [d_out]; dbias [d_out] or NULL.
 * bf16: dY o c is formed one slab of rows at a time (at most 64 MiB of the workspace, a multiple
 * of 128 rows chosen so that the slabs' dX GEMMs fill whole waves); the workspace never holds an
 * [M, d_out] copy of it.  The environment variable LORA_GB300_DORA_KSCALE=1 forms it inside the
 * dX GEMM instead (same bits, no copy at all, slower).
 */
lora_status dora_linear_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                            const void* B, const void* m, const void* bias, const void* Y,
                            const void* Z_saved, const float* n_saved, const float* V_saved,
                            const void* dY, float s, float eps,
                            void* dX, void* dA, void* dB, void* dm, void* dbias,
                            void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- DoRA (cols)
 * The column variant: the norm is taken per INPUT column of the adapted weight W' = W0 + s B A,
 * n[k] = max(||W'[:, k]||, eps), and the decomposed weight is W' diag(m / n) with m [d_in].
 * "LoRA/DoRA fast forward ...", What section (lora / dora-rows / dora-cols need no materialised
 * weight) and commit message (the row/col norm from the closed-form norm^2 expansion).
 *
 * c0[k] = sum_o W0[o,k]^2 in fp32: the cached per-layer constant.  c0: [d_in] fp32 output.
 * LORA_BF16 only.
 */
lora_status dora_colnorm2(const lora_shape* sh, const void* W0, float* c0, void* stream);

/* Forward:  q[k] = c0[k] + 2s colsum(A o (B^T W0))[k] + s^2 colsum(A o ((B^T B) A))[k],
 *   n = max(sqrt(max(q, 0)), eps),  c = m / n  (an input-column scale),
 *   Y = (X diag(c)) W0^T + s ((X diag(c)) A^T) B^T + bias.
 * Same pages and sections as dora_colnorm2; strength 0 returns X W0^T + bias.
 *   m [d_in] (bf16, nonzero), bias [d_out] or NULL, c0 [d_in] fp32 from dora_colnorm2.
 *   Y [M, d_out]; Z_save [M, r] = (X diag(c)) A^T or NULL; n_save [d_in] fp32 (required);
 *   U_save [d_in, r] fp32 (required): (B^T W0)^T, reused by the backward's norm gradient.
 */
lora_status dora_cols_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                          const void* B, const void* m, const void* bias, const float* c0,
                          float s, float eps, void* Y, void* Z_save, float* n_save, float* U_save,
                          void* ws, size_t ws_bytes, void* stream);

/* Backward of dora_cols_fwd, the norm kept in the graph:
 *   G = s dY B;  dXt = dY W0 + G A (the gradient of X diag(c));  dX = dXt diag(c);
 *   dc = colsum(X o dXt);  dm = dc / n;  g = -m dc / (2 n^3) (0 where n was clamped at eps);
 *   dA = (G^T X) diag(c) + 2s U^T diag(g) + 2s^2 (B^T B) A diag(g);
 *   dB = s dY^T Z + 2s W0 diag(g) A^T + 2s^2 B (A diag(g) A^T);  dbias = colsum(dY).
 * Same pages as dora_colnorm2 and the Fidelity section of "LoRA/DoRA fast forward ..." (norm in
 * the autograd graph).  Z_saved, n_saved, U_saved from the forward (Z_saved may be NULL).
 *   dX [M, d_in] or NULL; dA [r, d_in]; dB [d_out, r]; dm [d_in]; dbias [d_out] or NULL.
 */
lora_status dora_cols_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A,
                          const void* B, const void* m, const void* Z_saved, const float* n_saved,
                          const float* U_saved, const void* dY, float s, float eps,
                          void* dX, void* dA, void* dB, void* dm, void* dbias,
                          void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- LoRA gated MLP (SwiGLU / GeGLU)
 * e = X Wg^T + sg (X Ag^T) Bg^T,  u = X Wu^T + su (X Au^T) Bu^T,  h = act(e) * u,
 * Y = h Wd^T + sd (h Ad^T) Bd^T,  act = silu (sh->act = LORA_ACT_SWIGLU) or gelu (LORA_ACT_GEGLU).
 * "How Unsloth's FastLoRA Kernel Differs ...", Fused Forward Pass Architecture (LoRA_MLP)
 * and Activation Function Fusion (SwiGLU and GeGLU computed with the LoRA outputs).
 *   gate: W [I, H], A [r_g, H], B [I, r_g];  up: W [I, H], A [r_u, H], B [I, r_u];
 *   down: W [H, I], A [r_d, I], B [H, r_d].
 *   Y [M, H]; e_save, u_save, h_save [M, I] (required: the backward reads them);
 *   Zgu_save [M, r_g + r_u] = [X Ag^T | X Au^T] and Zd_save [M, r_d] = h Ad^T (required).
 */
lora_status lora_mlp_swiglu_fwd(const lora_mlp_shape* sh, const void* X, const lora_proj* gate,
                                const lora_proj* up, const lora_proj* down, void* Y,
                                void* e_save, void* u_save, void* h_save, void* Zgu_save,
                                void* Zd_save, void* ws, size_t ws_bytes, void* stream);

/* Backward of lora_mlp_swiglu_fwd (base weights frozen):
 *   dh = dY Wd + sd (dY Bd) Ad,  de = dh u act'(e),  du = dh act(e),
 *   dX = de Wg + du Wu + sg (de Bg) Ag + su (du Bu) Au,
 *   dA* = s* (d* B*)^T (input),  dB* = s* (d*)^T Z*.
 * "How Unsloth's FastLoRA Kernel Differs ...", Custom Backward Pass Implementation.
 *   dX [M, H] or NULL; dAg [r_g, H], dBg [I, r_g]; dAu [r_u, H], dBu [I, r_u];
 *   dAd [r_d, I], dBd [H, r_d].
 */
lora_status lora_mlp_swiglu_bwd(const lora_mlp_shape* sh, const void* X, const lora_proj* gate,
                                const lora_proj* up, const lora_proj* down,
                                const void* e_saved, const void* u_saved, const void* h_saved,
                                const void* Zgu_saved, const void* Zd_saved, const void* dY,
                                void* dX, void* dAg, void* dBg, void* dAu, void* dBu,
                                void* dAd, void* dBd, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- fused-leaf (QKV) LoRA linear
 * One X stream against the fused base weight, each leaf's low-rank term added to its own
 * output columns:
 *   Y[:, leaf l] = X W0[leaf l]^T + s_l (X A_l^T) B_l^T  (+ bias),
 * i.e. Y = X W0^T + Z blockdiag(s_0 B_0, .., s_{L-1} B_{L-1})^T with Z = X [A_0; ..]^T.
 * "How Unsloth's FastLoRA Kernel Differs ...", Fused Forward Pass Architecture (LoRA_QKV:
 * the attention query/key/value projections) and "nunchaku-style kernel fusion" (OneTrainer
 * #1680, the fused-leaf forward: each leaf's up-projection narrowed to that leaf's rows).
 *   X [M, d_in]; W0 [N, d_in] (leaf l owns rows n[0] + .. + n[l-1] onward); leaves[L];
 *   bias [N] or NULL; Y [M, N]; Z_save [M, L r] = [X A_0^T | X A_1^T | ..] or NULL (all bf16).
 *   A leaf with s == 0 adds exactly nothing to its columns.
 */
lora_status lora_qkv_fwd(const lora_qkv_shape* sh, const void* X, const void* W0, const lora_adapter* leaves,
                         const void* bias, void* Y, void* Z_save, void* ws, size_t ws_bytes, void* stream);

/* Backward of lora_qkv_fwd (W0 frozen), with dY_l the columns of dY that belong to leaf l:
 *   dX = dY W0 + sum_l s_l (dY_l B_l) A_l,  dA_l = s_l (dY_l B_l)^T X,  dB_l = s_l dY_l^T Z_l,
 *   dbias = colsum(dY).
 * Same pages and sections as lora_qkv_fwd (custom backward of the fused projection).
 *   Z_saved [M, L r] from the forward, or NULL (recomputed); dY [M, N];
 *   dX [M, d_in] or NULL; dA[l] [r, d_in] and dB[l] [n_l, r] (arrays of L device pointers,
 *   all required); dbias [N] or NULL.
 */
lora_status lora_qkv_bwd(const lora_qkv_shape* sh, const void* X, const void* W0, const lora_adapter* leaves,
                         const void* Z_saved, const void* dY, void* dX, void* const* dA, void* const* dB,
                         void* dbias, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- W8A8 + LoRA epilogue
 * Per-row symmetric int8 quantisation of a bf16 matrix, decided in fp32:
 *   scale[i] = absmax(X[i, :]) / 127,  Xq = clamp(rint_half_even(X / scale), -127, 127),
 *   an all-zero row gives scale 0 and codes 0.  Optionally also Z = X A^T (bf16) from the
 *   unquantised X in the same call.
 * "nunchaku-style kernel fusion" (OneTrainer #1680), commit reworking the 8-bit matmuls
 * (axis-wise quantisation for the 8-bit matmul; the autograd Function owns the
 * down-projection).
 *   X [rows, cols] bf16; Xq [rows, cols] int8; sx [rows] fp32;
 *   A [r, cols] bf16 and Z [rows, r] bf16, both NULL or both non-NULL (then r in 8..128).
 */
lora_status w8a8_quantize_rows(int64_t rows, int64_t cols, const void* X, int8_t* Xq, float* sx,
                               const void* A, int64_t r, void* Z, void* stream);

/* Step W-1 for the prepacked product: the same quantisation, with the codes written as bf16
 * values (the same integers, exact in bf16) instead of int8, ready to be the A operand of
 * w8a8_lora_fwd_packed (no re-layout in the forward).  Xcodes [rows, cols] bf16; the rest as
 * w8a8_quantize_rows.  Same page and passage as w8a8_quantize_rows. */
lora_status w8a8_quantize_rows_bf16(int64_t rows, int64_t cols, const void* X, void* Xcodes, float* sx,
                                    const void* A, int64_t r, void* Z, void* stream);

/* One-time preparation of the frozen int8 weight Wq [d_out, d_in] (sw [d_out] fp32):
 *   Wb [d_out, d_in] bf16: the weight codes as bf16 values (the same integers, exact in bf16), the
 *   B operand of the tensor-core product (NULL to skip);  Wd [d_out, d_in] bf16 = sw[o] * Wq[o, k],
 *   the dequantised weight of the backward (NULL to skip).  The backward through the int8 base
 *   given Wd is lora_linear_bwd with W0 = Wd (what w8a8_lora_bwd does after dequantising per call).
 * "nunchaku-style kernel fusion" (OneTrainer #1680), commit reworking the 8-bit matmuls (the
 * frozen 8-bit weight, re-laid out for the product once).  d_in a multiple of 32. */
lora_status w8a8_prepack_weight(int64_t d_out, int64_t d_in, const int8_t* Wq, const float* sw, void* Wb,
                                void* Wd, void* stream);

/* Workspace of w8a8_lora_fwd_packed: the error word (256 bytes).  0 on bad input. */
size_t w8a8_packed_workspace_bytes(int64_t M, int64_t d_out);

/* w8a8_lora_fwd on prepacked operands: Xcodes [M, d_in] bf16 from w8a8_quantize_rows_bf16 and
 * Wb [d_out, d_in] bf16 from w8a8_prepack_weight; every other argument, the result and its
 * exactness as w8a8_lora_fwd.  Same pages and passages as w8a8_lora_fwd. */
lora_status w8a8_lora_fwd_packed(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const void* Xcodes,
                                 const float* sx, const void* Wb, const float* sw, const void* Z, const void* B,
                                 float s, const void* bias, void* Y, int32_t* acc_out, void* ws, size_t ws_bytes,
                                 void* stream);

/* Bytes of workspace w8a8_lora_fwd needs: the error word and the int8 codes re-laid out as bf16
 * tensor-core operands (X: M x d_in, W: d_out x d_in).  0 on bad input. */
size_t w8a8_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out);

/* Y = float(acc) * sx[i] * sw[o] + s * (Z B^T)[i, o] (+ bias), acc = Xq Wq^T exact in int32.
 * "nunchaku-style kernel fusion" (OneTrainer #1680): commit reworking the 8-bit matmuls
 * (epilogues: raw product, per-row dequant, dequant plus rank-tiled low-rank update; no
 * int32 (M, d_out) materialisation) and commit unifying the five entry points
 * (mm_8bit(a, b, out_dtype, scale_m, scale_n, lora_xd, lora_up)).
 *   Xq [M, d_in] int8, sx [M] fp32, Wq [d_out, d_in] int8, sw [d_out] fp32,
 *   Z [M, r] bf16 ("lora_xd") and B [d_out, r] bf16 ("lora_up"): both NULL (no LoRA) or both set
 *   (r a multiple of 8 in 8..128),
 *   bias [d_out] bf16 or NULL, Y [M, d_out] bf16 (or NULL when only acc_out is wanted),
 *   acc_out [M, d_out] int32 or NULL: the raw-product epilogue.  d_in multiple of 32.
 *   ws: workspace of at least w8a8_workspace_bytes(M, d_in, d_out) bytes (256-byte aligned).
 *   The product runs on the bf16 tensor cores (sm_103a has no tcgen05 integer kind) with the codes
 *   as bf16 values, the K range in chunks of 1024: every fp32 partial sum of a chunk is an integer
 *   of magnitude at most 127 * 127 * 1024 < 2^24, so each chunk is exact, and the chunks are added
 *   as int32; acc is bit-identical to an integer GEMM for any d_in.  The rank-r term Z B^T is a
 *   separate fp32 accumulator.  LORA_GB300_W8A8_IMMA=1 runs the warp-level integer MMA instead.
 */
lora_status w8a8_lora_fwd(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const int8_t* Xq,
                          const float* sx, const int8_t* Wq, const float* sw, const void* Z,
                          const void* B, float s, const void* bias, void* Y, int32_t* acc_out,
                          void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- tracing
 * Number of kernels this library has launched since it was loaded (host-side count of
 * launch calls; memsets issued through the CUDA runtime are not counted). */
uint64_t lora_launch_count(void);

/* Enable (on != 0) or disable CUDA-event timing of the tcgen05 GEMM launches.  While enabled,
 * each GEMM launch is bracketed by two events recorded on its stream (a few microseconds of
 * host overhead per launch; the device work is unchanged). */
lora_status lora_prof_enable(int on);

/* Summed device time (ms), number of launches and algorithmic flops (base contraction plus
 * rank-r tail, 2*M*N*K) of the GEMM launches recorded since the last reset; waits for the
 * recorded events.  Any output pointer may be NULL.  reset != 0 clears the record. */
lora_status lora_prof_gemm(double* ms, int64_t* launches, double* flops, int reset);

/* The same for the rank-r passes (the skinny HBM-bound kernels: down-projections, column
 * reductions): total event time, launches, and their algorithmic HBM bytes (each input read
 * once, outputs written once).  No counterpart on the pages (tracing). */
lora_status lora_prof_rank(double* ms, int64_t* launches, double* bytes, int reset);

/* Bytes of workspace w8a8_lora_bwd needs (0 on bad input). */
size_t w8a8_bwd_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int64_t r);

/* Backward of the W8A8 + LoRA layer with the int8 base weight frozen.  The activation quantiser
 * is taken as straight-through (its gradient passes unchanged; the pages do not say otherwise),
 * so with W_deq = diag(sw) Wq:
 *   dX = dY W_deq + s (dY B) A,  dA = s (dY B)^T X,  dB = s dY^T Z,  dbias = colsum(dY).
 * "nunchaku-style kernel fusion" (OneTrainer #1680), commit reworking the 8-bit matmuls (the
 * backward's B operand is re-laid out for the tensor cores; the LoRA dgrad folds into the
 * backward; the autograd Function owns the down-projection).
 *   X [M, d_in] bf16 (the unquantised input), Wq [d_out, d_in] int8, sw [d_out] fp32,
 *   A [r, d_in], B [d_out, r], Z_saved [M, r] (X A^T) or NULL, dY [M, d_out] (all bf16);
 *   dX [M, d_in] or NULL, dA [r, d_in], dB [d_out, r], dbias [d_out] or NULL.
 *   d_in multiple of 16; ws of at least w8a8_bwd_workspace_bytes() bytes: the weight is
 *   dequantised into it once per call (a bf16 [d_out, d_in] copy), then the bf16 LoRA backward
 *   runs over it. */
lora_status w8a8_lora_bwd(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const void* X, const int8_t* Wq,
                          const float* sw, const void* A, const void* B, const void* Z_saved, const void* dY,
                          float s, void* dX, void* dA, void* dB, void* dbias, void* ws, size_t ws_bytes,
                          void* stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on an mbarrier
 * that nothing ever arrives on, with a limit of `timeout_us` microseconds; the kernel then
 * records LORA_ERR_DEVICE_TIMEOUT in the error word of `ws` and returns.  It faults and
 * hangs nothing.  Read the result with lora_check_device_error(). */
lora_status lora_debug_wait_timeout(void* ws, uint32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_H */

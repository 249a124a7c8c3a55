// Host-side declarations shared by the translation units of the library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace lg {

typedef __nv_bfloat16 bf16;

int num_sms_current();
// Fills *a with the programmatic-stream-serialization launch attribute and returns 1, or returns 0
// when LORA_GB300_PDL=0.  Only kernels that call pdl_wait() before touching global memory use it.
int pdl_attr(cudaLaunchAttribute* a);
// 2-D bf16 tensor map over `outer` rows of `inner` contiguous elements (row stride `ld` elements),
// box {box_inner, box_outer}, swizzle of 0 / 32 / 64 / 128 bytes; out-of-bounds elements read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                    uint32_t box_inner, uint32_t box_outer, int swizzle_bytes);
// A 2-D uint8 tensor map (no swizzle; ld in bytes, a multiple of 16) for the dropout masks.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                  uint32_t box_outer);

// tracing (prof.cu)
void count_launch(int n = 1);
// Launch with programmatic stream serialization (when enabled) and count it: the kernel may be
// scheduled while its predecessor in the stream finishes, so it must call pdl_wait() before it
// touches global memory (every kernel launched this way does so first).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}
uint64_t launch_count();
bool prof_enabled();
void prof_set(bool on);
// kind 0: tcgen05 GEMM launches (work = algorithmic flops); kind 1: rank-r passes (work =
// algorithmic HBM bytes)
void prof_mark(cudaStream_t st, bool start, double work, int kind = 0);
cudaError_t prof_collect(int kind, double* ms, int64_t* launches, double* work, bool reset);

// ------------------------------------------------------------------ tcgen05 GEMM engine
enum EpiKind { EPI_SCALE_BIAS = 0, EPI_SWIGLU = 1, EPI_SWIGLU_BWD = 2, EPI_W8A8K = 3 };
enum TcMode {
  TC_FWD = 0,          // A0 [M,K0] x B0 [N,K0]^T (+ A1 [M,K1] x B1 [N,K1]^T), epilogue scale/bias
  TC_BWD_DX = 1,       // A0 [M,K0] x B0 [K0,N] (MN-major) (+ A1 x B1 [K1,N]), optional A-scale along K
  TC_SWIGLU_FWD = 2,   // stacked gate/up weights, SwiGLU epilogue writing e, u, h
  TC_SWIGLU_BWD = 3,   // MN-major B, epilogue forms de, du from saved e, u
  TC_W8A8K = 4         // int8 codes held as bf16 (B0 [N,K0] K-major, the full codes): the exact int32
                       // product from K chunks of kc_steps x 64, each summed exactly in fp32 in its
                       // own TMEM accumulator (the two alternate) and added as int32 in the epilogue;
                       // the rank-r term A1 x B1^T (fp32) as one more accumulator; y and/or int32 out
};

struct TcGemmDesc {
  int mode = TC_FWD;
  int M = 0, N = 0, K0 = 0, K1 = 0;
  bool b0_mn = false, b1_mn = false, has_tail = false;
  const void* A0 = nullptr;
  int64_t lda0 = 0;
  const void* B0 = nullptr;
  const void* B0b = nullptr;  // K-major: second stacked half; MN-major: rows of K past k0_split
  int64_t ldb0 = 0;
  int b0_rows = 0, b0b_rows = 0, k0_split = 0;
  const void* A1 = nullptr;
  int64_t lda1 = 0;
  int K1_a = 0;                // columns of the A1 tensor
  const void* B1 = nullptr;
  const void* B1b = nullptr;
  int64_t ldb1 = 0;
  int K1_b = 0;                // columns of a K-major B1 tensor
  int64_t ldb1b = 0;           // stacked tail: row stride and columns of the second half's tensor
  int K1_bb = 0;               //   (0: those of the first half)
  int b1b_x = 0;
  int b1_x = 0;                // stacked tail: x coordinate of the first half (past the tensor = zeros)
  void* out[3] = {nullptr, nullptr, nullptr};
  int64_t ldo = 0;
  const float* col_scale = nullptr;
  const bf16* bias = nullptr;
  const float* a_kscale = nullptr;   // [ceil(K0 / 64) * 64] fp32, zero past K0, 16-byte aligned
  const bf16* e_in = nullptr;
  const bf16* u_in = nullptr;
  int64_t ld_eu = 0;
  // W8A8 epilogue: per-row / per-column dequant scales, scale of the rank-r term (A1 B1^T), raw
  // int32 output
  const float* sx = nullptr;
  const float* sw = nullptr;
  float ls = 0.f;
  int32_t* acc_out = nullptr;
  uint32_t* err = nullptr;
  uint64_t timeout_ns = 2000000000ull;
  int max_ctas = 0;            // cap on the persistent grid in CTAs (0: one per SM)
  int kc_steps = 16;           // TC_W8A8K: K-steps of 64 per exactly summed chunk
  // forward with the down-projection in the GEMM (TC_FWD, has_tail, K1 = dn_r in 8 .. 32): Z =
  // A0 dn_a^T is formed from the staged A0 tiles (dn_a [dn_r, K0], row stride dn_lda), the tail's
  // A operand is bf16(dn_s Z) written on chip (A1 unused), and bf16(Z) goes to dn_z [M, dn_r] when set
  const bf16* dn_a = nullptr;
  int64_t dn_lda = 0;
  float dn_s = 0.f;
  int dn_r = 0;
  bf16* dn_z = nullptr;
  int act = 0;                 // gated MLP activation: 0 SwiGLU, 1 GeGLU
};
cudaError_t tc_gemm(const TcGemmDesc& d, cudaStream_t st);

// ------------------------------------------------------------------ skinny (rank-r) kernels, bf16
// T = S U^T : S [rows, K] (ld lds), U either [R, K] (u_kr = false) or [K, R] (u_kr = true).
// Outputs (each optional): out_a = bf16(scale_a * T), out_b = bf16(scale_b * T), out_f = T (fp32),
// all with leading dimension R.  R multiple of 8, 8 <= R <= 512; above 64 the columns go in
// chunks of 64, one pass over S each (the scaled copy of S is written by the first).
struct RowProjDesc {
  int64_t rows = 0, K = 0;
  int R = 0;
  const bf16* S = nullptr;
  int64_t lds = 0;
  const bf16* U = nullptr;
  bool u_kr = false;
  int64_t ldu = 0;
  bf16* out_a = nullptr;
  float scale_a = 1.f;
  bf16* out_b = nullptr;
  float scale_b = 1.f;
  float* out_f = nullptr;
  int64_t ldo = 0;              // leading dimension of the outputs (0 -> R)
  int split_col = 1 << 30;      // columns >= split_col of out_b use scale_b_hi
  float scale_b_hi = 1.f;
  // optional column-scaled copy of S written on the way: s_out[row, k] = bf16(S[row, k] * s_scale[k])
  const float* s_scale = nullptr;
  bf16* s_out = nullptr;        // [rows, K], leading dimension K
  // optional keep mask on S (uint8 [rows, K], row stride K bytes, a multiple of 16): the pass reads
  // S[row, k] as bf16(S[row, k] mask_scale) where mask[row, k] != 0 and as 0 elsewhere
  const uint8_t* mask = nullptr;
  float mask_scale = 1.f;
  uint32_t* err = nullptr;      // device error word for bounded waits
  uint64_t timeout_ns = 2000000000ull;
};
cudaError_t rowproj(const RowProjDesc& d, cudaStream_t st);

// Column reduction over rows: part[(split K + k) ldp + j0 + j] = sum_{rows of split} S[row, k] T[row, j]
// (S [rows, K] ld lds, T [rows, R] ld ldt; ldp defaults to R, j0 to 0), plus optional per-column
// sums colsum[split][k] = sum S[row,k] and coldot[split][k] = sum S[row,k] * Y[row,k].  R multiple
// of 8 up to 512; above 64 the columns of T go in chunks of 64, one pass over S each (the column
// sums come with the first).
struct ColReduceDesc {
  int64_t rows = 0, K = 0;
  int R = 0;
  const bf16* S = nullptr;
  int64_t lds = 0;
  const bf16* T = nullptr;
  int64_t ldt = 0;
  const bf16* Y = nullptr;     // optional second [rows, K] input for coldot
  int64_t ldy = 0;
  float* part = nullptr;       // [splits, K, ldp]
  int ldp = 0;                 // leading dimension of part (0 -> R)
  int j0 = 0;                  // first column of part written
  float* colsum = nullptr;     // [splits, K] or null
  float* coldot = nullptr;     // [splits, K] or null
  const float* sc = nullptr;   // with sc_out (and Y): column scales [K]
  bf16* sc_out = nullptr;      // optional column-scaled copy of S: sc_out[row K + k] = bf16(S[row, k] sc[k])
  // optional keep mask on S (as RowProjDesc::mask; no Y, no column sums, no copy with it)
  const uint8_t* mask = nullptr;
  float mask_scale = 1.f;
  int splits = 1;
  uint32_t* err = nullptr;     // device error word for bounded waits
  uint64_t timeout_ns = 2000000000ull;
};
// Row splits of a colreduce pass over [rows, K] at rank R (with or without the second input Y, or
// the keep mask):
// the split count whose waves of resident CTAs finish the pass soonest.
int colreduce_splits(int64_t rows, int64_t K, int R = 16, bool has_y = false, bool mask = false);
cudaError_t colreduce(const ColReduceDesc& d, cudaStream_t st);

// One pass over S [rows, K] for both rank-r products that read it:
//   gpart[bn][row][j] = sum_{k in column group bn} S[row, k] U[k, j]   (U [K, R], ld ldu; when U is set)
//   part[(bm K + k) ldp + j0 + j] = sum_{row in row group bm} S[row, k] T[row, j]   (T [rows, R], ld ldt)
//   colsum[bm][k] = sum_{row in row group bm} S[row, k]                 (when colsum is set)
// R in {8, 16, 24, 32}.  The grid is pm row groups of nb 128-row blocks x pn column groups of 512
// columns, from rowcol_plan; gpart is [pn, rows, R] fp32 (summed by gpart_sum), part and colsum
// have the colreduce layout with splits = pm.
struct RowColPlan {
  int pm = 0, pn = 0, nb = 0;
};
RowColPlan rowcol_plan(int64_t rows, int64_t K, int R);
struct RowColDesc {
  int64_t rows = 0, K = 0;
  int R = 0;
  const bf16* S = nullptr;
  int64_t lds = 0;
  const bf16* U = nullptr;
  int64_t ldu = 0;
  const bf16* T = nullptr;
  int64_t ldt = 0;
  float* gpart = nullptr;
  float* part = nullptr;
  int ldp = 0;
  int j0 = 0;
  float* colsum = nullptr;
  int pm = 0, pn = 0, nb = 0;
  uint32_t* err = nullptr;
  uint64_t timeout_ns = 2000000000ull;
};
cudaError_t rowcol(const RowColDesc& d, cudaStream_t st);
// out [rows, R] (row stride ldo) = bf16(scale * sum over the pn partials of gpart)
cudaError_t gpart_sum(const float* gpart, int pn, int64_t rows, int R, float scale, bf16* out, int64_t ldo,
                      cudaStream_t st);

// ------------------------------------------------------------------ small kernels (templated on T)
template <typename T>
cudaError_t rownorm2(const T* W, int64_t rows, int64_t cols, float* r0, cudaStream_t st);
// K = A A^T (fp32 [r, r]) for A [r, cols]
template <typename T>
cudaError_t gram_rows(const T* A, int r, int64_t cols, float* K, cudaStream_t st);
// DoRA norm: q = r0 + 2s sum_j V[o,j] B[o,j] + s^2 sum_j (B Kr)[o,j] B[o,j]; n = max(sqrt(max(q,0)), eps);
// c = m / n.  Writes n (n_out) and c.
template <typename T>
cudaError_t dora_norm(int64_t out, int r, const float* r0, const float* V, const T* B, const float* Kr,
                      const T* m, float s, float eps, float* n_out, float* c, cudaStream_t st);
// sum over splits of column partials: dst[k] = sum_s src[s][k]  (fp32 and, optionally, as T)
template <typename T>
cudaError_t sum_splits(const float* src, int splits, int64_t n, float* dst_f, T* dst_t, cudaStream_t st);
// c = m / n for o < out, and c = 0 for out <= o < padded (a zero tail for readers that fetch whole
// 64-entry blocks)
template <typename T>
cudaError_t dora_c(int64_t out, const T* m, const float* n, float* c, cudaStream_t st, int64_t padded = 0);
// DoRA backward small step: dc = (dot - bias*colsum)/c ; dm = dc/n ; g = -m dc/(2 n^3) (0 if n<=eps);
// dot and csum are [splits, out] partials (csum read only with a bias or dbias).
template <typename T>
cudaError_t dora_dc(int64_t out, const float* dot, const float* csum, int splits, const T* bias, const float* c,
                    const float* n, const T* m, float eps, float* g, T* dm, T* dbias, cudaStream_t st);
// out[o, j] = scale[o] * B[o, j] (bf16 / T out), scale may be null (=1), with extra factor f.
template <typename T>
cudaError_t scale_rows(const T* B, int64_t rows, int r, const float* scale, float f, T* out, cudaStream_t st);
// Final LoRA/DoRA gradient assembly from fp32 partials:
//   dA[j, k] = sA * sum_s PA[s][k][j] + sW * sum_s PW[s][k][j] + s2 * sum_l Kg[j,l] A[l,k]
//   dB[o, j] = sB * rs[o] * sum_s PB[s][o][j] + 2 s g[o] V[o,j] + 2 s^2 g[o] (B Kr)[o,j]
//   (rs null: 1; V null: no norm terms; g null with V: g = 1)
// Partials are laid out [splits][n][ldp] and read at columns j0 .. j0 + r - 1.
struct Partial {
  const float* p = nullptr;
  int splits = 0;
  int ldp = 0;
  int j0 = 0;
};
template <typename T>
cudaError_t finalize_dA(int r, int64_t in, Partial PA, float sA, Partial PW, float sW, const float* Kg, float s2,
                        const T* A, T* dA, cudaStream_t st);
template <typename T>
cudaError_t finalize_dB(int64_t out, int r, Partial PB, float sB, const float* rs, const float* g, const float* V,
                        const T* B, const float* Kr, float s, bool accumulate, T* dB, cudaStream_t st);
// One bf16 gradient assembly of a batch (finalize_batch runs up to kMaxFinJobs in one launch):
//   is_dB == 0: dA [r, rows] as finalize_dA(r, rows, P, sP, PW, sW, Kx (= Kg), s2, M (= A), out)
//   is_dB == 1: dB [rows, r] as finalize_dB(rows, r, P, sP, rs, g, V, M (= B), Kx (= Kr), s, false, out)
constexpr int kMaxFinJobs = 8;
struct FinJob {
  int is_dB = 0;
  int r = 0;
  int64_t rows = 0;
  Partial P{};
  float sP = 0.f;
  Partial PW{};
  float sW = 0.f;
  const float* Kx = nullptr;
  float s2 = 0.f;
  const float* rs = nullptr;
  const float* g = nullptr;
  const float* V = nullptr;
  float s = 0.f;
  const bf16* M = nullptr;
  bf16* out = nullptr;
};
cudaError_t finalize_batch(const FinJob* jobs, int n, cudaStream_t st);
inline FinJob fin_dA(int r, int64_t in, Partial PA, float sA, const void* A, void* dA) {
  FinJob f;
  f.r = r;
  f.rows = in;
  f.P = PA;
  f.sP = sA;
  f.M = static_cast<const bf16*>(A);
  f.out = static_cast<bf16*>(dA);
  return f;
}
inline FinJob fin_dB(int64_t out, int r, Partial PB, float sB, const void* B, void* dB) {
  FinJob f;
  f.is_dB = 1;
  f.r = r;
  f.rows = out;
  f.P = PB;
  f.sP = sB;
  f.M = static_cast<const bf16*>(B);
  f.out = static_cast<bf16*>(dB);
  return f;
}
// Kg = B^T diag(g) B  (fp32 [r, r]; g null = all ones), r <= 128; `work` holds at least
// gram_work_floats(r) floats of chunk partials
size_t gram_work_floats(int r);
template <typename T>
cudaError_t gram_weighted(const T* B, int64_t out, int r, const float* g, float* Kg, float* work, cudaStream_t st);
// rows of two matrices stacked: dst = [X1 ; X2] (rows1 + rows2, cols), same dtype
cudaError_t concat_rows_bf16(const bf16* X1, int64_t rows1, const bf16* X2, int64_t rows2, int64_t cols, bf16* dst,
                             cudaStream_t st);
cudaError_t fill_zero(void* p, size_t bytes, cudaStream_t st);
// Input dropout on the unfused path: out = bf16(X o mask * scale); dX += (G A) o mask * scale
// (mask uint8 0/1 [rows, cols], cols a multiple of 8)
cudaError_t apply_mask_bf16(const bf16* X, const uint8_t* mask, float scale, int64_t rows, int64_t cols, bf16* out,
                            cudaStream_t st);
cudaError_t add_masked_rank_bf16(bf16* dX, const bf16* G, const bf16* A, const uint8_t* mask, float scale,
                                 int64_t rows, int64_t cols, int r, cudaStream_t st);
// DoRA column variant (bf16): c0 = colsum(W^2); the closed-form column norm n, c = m / n and
// A_c = A diag(c); out = A diag(w); K = A diag(w) A^T; and the dA assembly
//   dA[j, k] = c[k] sum_s PA[s][k][j] + 2 s g[k] U[k, j] + 2 s^2 g[k] (Kb A)[j, k].
cudaError_t colnorm2_bf16(const bf16* W, int64_t rows, int64_t cols, float* c0, cudaStream_t st);
cudaError_t dora_colnorm(int64_t in, int r, const float* c0, const float* U, const bf16* A, const float* Kb,
                         const bf16* m, float s, float eps, float* n_out, float* c, bf16* A_c, cudaStream_t st);
cudaError_t scale_cols_bf16(const bf16* A, int r, int64_t in, const float* w, bf16* out, cudaStream_t st);
cudaError_t gram_rows_weighted(const bf16* A, int r, int64_t cols, const float* w, float* K, cudaStream_t st);
cudaError_t finalize_dA_cols(int r, int64_t in, Partial PA, const float* c, const float* g, const float* U,
                             const float* Kb, const bf16* A, float s, bf16* dA, cudaStream_t st);
// Operands of the fused-leaf (QKV) layer: A_stack = [A_0; ..; A_{L-1}] and B_blk = blockdiag(s_l B_l)
// (row0[l] = first row of leaf l in the fused output, row0[0] = 0; in multiple of 8).
constexpr int kMaxLeaves = 3;
struct LeafPack {
  int L = 0, r = 0;
  int64_t in = 0, N = 0;
  int64_t row0[kMaxLeaves] = {0, 0, 0};
  const bf16* A[kMaxLeaves] = {nullptr, nullptr, nullptr};
  const bf16* B[kMaxLeaves] = {nullptr, nullptr, nullptr};
  float s[kMaxLeaves] = {0.f, 0.f, 0.f};
  bf16* A_stack = nullptr;
  bf16* B_blk = nullptr;
};
cudaError_t pack_leaves(const LeafPack& p, cudaStream_t st);

// ------------------------------------------------------------------ fp32 SIMT path
// C[M,N] = alpha * op(A) op(B) (op(A) [M,K], op(B) [K,N]) + beta * C, with optional per-K scale of
// op(A) columns (kscale[K]), per-row output scale (rscale[M]), per-column bias[N] and column scale cs[N]
// applied as C = cs*acc*alpha + bias (+ beta C).
struct SgemmDesc {
  int64_t M = 0, N = 0, K = 0;
  bool ta = false, tb = false;
  const float* A = nullptr;
  int64_t lda = 0;
  const float* B = nullptr;
  int64_t ldb = 0;
  float* C = nullptr;
  int64_t ldc = 0;
  float alpha = 1.f, beta = 0.f;
  const float* kscale = nullptr;
  const float* rscale = nullptr;
  const float* cs = nullptr;
  const float* bias = nullptr;
};
cudaError_t sgemm_f32(const SgemmDesc& d, cudaStream_t st);
// per-column partial sums for fp32 path: colsum[k] = sum_i S[i,k], coldot[k] = sum_i S[i,k]*Y[i,k]
cudaError_t coldot_f32(const float* S, const float* Y, int64_t rows, int64_t K, float* colsum, float* coldot,
                       cudaStream_t st);

// ------------------------------------------------------------------ W8A8
// per-row absmax quantisation: codes as int8 (Xq) and/or as bf16 values (Xb), either may be null
cudaError_t quantize_rows_bf16(const bf16* X, int64_t rows, int64_t cols, int8_t* Xq, float* sx, cudaStream_t st,
                               bf16* Xb = nullptr);
// int8 -> bf16 (exact; n multiple of 16)
cudaError_t i8_to_bf16(const int8_t* q, int64_t n, bf16* out, cudaStream_t st);
// out[o, k] = bf16(sw[o] * q[o, k]) (cols multiple of 16)
cudaError_t i8_dequant_rows_bf16(const int8_t* q, const float* sw, int64_t rows, int64_t cols, bf16* out,
                                 cudaStream_t st);
cudaError_t w8a8_gemm(int64_t M, int64_t K, int64_t N, int r, const int8_t* Xq, const float* sx, const int8_t* Wq,
                      const float* sw, const bf16* Z, const bf16* B, float s, const bf16* bias, bf16* Y,
                      int32_t* acc_out, cudaStream_t st);

// ------------------------------------------------------------------ debug
cudaError_t debug_wait_timeout(uint32_t* err, uint64_t timeout_ns, cudaStream_t st);

}  // namespace lg

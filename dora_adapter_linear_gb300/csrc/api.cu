// C-ABI entry points: argument validation, workspace carving and the launch sequence of each
// operation.  Nothing here computes; every step runs in the kernels of this library.
#include <math.h>
#include <stdlib.h>

#include "../../include/lora_gb300.h"
#include "internal.h"

using namespace lg;

namespace {

constexpr size_t kErrBytes = 256;
inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Dry-run-able bump allocator over the caller's workspace: with base == nullptr it only sums sizes.
struct Carve {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    char* p = base ? base + off : nullptr;
    off += al256(count * sizeof(T));
    return reinterpret_cast<T*>(p);
  }
};

uint64_t wait_timeout_ns() {
  static uint64_t v = 0;
  if (v == 0) {
    const char* e = getenv("LORA_GB300_WAIT_TIMEOUT_MS");
    double ms = e ? atof(e) : 2000.0;
    if (!(ms > 0)) ms = 2000.0;
    v = (uint64_t)(ms * 1e6);
  }
  return v;
}

bool env_flag(const char* name) {
  const char* e = getenv(name);
  return e && atoi(e) != 0;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
#define CK(x)                                  \
  do {                                         \
    if ((x) != cudaSuccess) return LORA_ERR_CUDA; \
  } while (0)
#define REQ(p)                                   \
  do {                                           \
    if ((p) == nullptr) return LORA_ERR_INVALID_ARG; \
  } while (0)
// tensors whose leading extent is the token count may be NULL when there are no tokens
#define REQM(M, p)                                                \
  do {                                                            \
    if ((M) > 0 && (p) == nullptr) return LORA_ERR_INVALID_ARG;   \
  } while (0)
#define ALN(p)                                   \
  do {                                           \
    if ((p) != nullptr && !al16(p)) return LORA_ERR_MISALIGNED; \
  } while (0)

lora_status check_shape(const lora_shape* sh) {
  if (!sh) return LORA_ERR_INVALID_ARG;
  if (sh->M < 0 || sh->d_in <= 0 || sh->d_out <= 0 || sh->r <= 0) return LORA_ERR_INVALID_ARG;
  if (sh->dtype != LORA_F32 && sh->dtype != LORA_BF16) return LORA_ERR_INVALID_ARG;
  if (sh->d_in % 8 || sh->d_out % 8) return LORA_ERR_UNSUPPORTED;
  if (sh->r > 128) return LORA_ERR_UNSUPPORTED;
  if (sh->dtype == LORA_BF16 && sh->r % 8) return LORA_ERR_UNSUPPORTED;
  if (sh->M > (1LL << 31) - 1 || sh->d_in > (1LL << 31) - 1 || sh->d_out > (1LL << 31) - 1)
    return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

// LORA_GB300_DORA_KSCALE=1 makes the DoRA-rows dX product scale each staged dY tile by c inside the
// GEMM instead of reading the slab copy of dY o c (same bits; 1.46 against 1.22 ms per DoRA step).
bool kscale_dx() {
  const char* e = getenv("LORA_GB300_DORA_KSCALE");
  return e && atoi(e) == 1;
}

// LORA_GB300_FUSED_Z=1 makes the bf16 LoRA forward form Z inside the GEMM (ranks 8 .. 32; the one-CTA
// kernel with four down-projection warps).  Measured on the 8192 x 4096 x 4096 forward it takes
// 0.396 ms against 0.184 ms for the separate pass plus the CTA-pair GEMM: the warps that read every
// staged X tile a second time and hold its stage until they are done halve the tensor pipe's rate.
// So the separate pass stays the default.
bool fused_down_projection(int r) {
  if (r < 8 || r > 32 || r % 8) return false;
  const char* e = getenv("LORA_GB300_FUSED_Z");
  return e && atoi(e) == 1;
}

lora_status check_ws(void* ws, size_t have, size_t need) {
  if (ws == nullptr || have < need) return LORA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255) return LORA_ERR_MISALIGNED;
  return LORA_OK;
}

// ------------------------------------------------------------------ workspace plans
struct LinFwdWs {
  uint32_t* err;
  void* Zs;   // bf16: s*Z ; f32: Z when no Z_save
};
size_t plan_lin_fwd(const lora_shape& sh, char* base, LinFwdWs* w) {
  Carve c{base};
  w->err = c.take<uint32_t>(kErrBytes / 4);
  const size_t es = sh.dtype == LORA_BF16 ? 2 : 4;
  w->Zs = c.take<char>((size_t)sh.M * sh.r * es);
  return c.off;
}

struct LinBwdWs {
  uint32_t* err;
  void* Gs;      // [M, r] bf16 s*G (f32: G)
  void* Zrec;    // [M, r] recomputed Z
  float* PB;     // [splitsB, out, r]
  float* PA;     // [splitsA, in, r]
  float* csum;   // [splitsB, out]
  float* Gp;     // [rc.pn, M, r] row partials of G (one pass over dY for G and the dB partials)
  RowColPlan rc; // pm == 0: G and the dB partials take a pass over dY each
  int splitsB, splitsA;
};
// Plan of the one pass over S [M, K] that gives both rank-r products of a backward's dY side (G and
// the dB partials), or an empty plan (pm == 0: a pass each) for other ranks, M == 0, or with
// LORA_GB300_ROWCOL=0.
RowColPlan dy_plan(int64_t M, int64_t K, int64_t r) {
  const char* rc_env = getenv("LORA_GB300_ROWCOL");
  if (!(r == 8 || r == 16 || r == 24 || r == 32) || M <= 0 || (rc_env && atoi(rc_env) == 0)) return RowColPlan{};
  return rowcol_plan(M, K, (int)r);
}
size_t plan_lin_bwd(const lora_shape& sh, char* base, LinBwdWs* w) {
  Carve c{base};
  const size_t es = sh.dtype == LORA_BF16 ? 2 : 4;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->Gs = c.take<char>((size_t)sh.M * sh.r * es);
  w->Zrec = c.take<char>((size_t)sh.M * sh.r * es);
  w->rc = RowColPlan{};
  w->Gp = nullptr;
  if (sh.dtype == LORA_BF16) {
    w->rc = dy_plan(sh.M, sh.d_out, sh.r);
    w->splitsB = w->rc.pm > 0 ? w->rc.pm : colreduce_splits(sh.M, sh.d_out, (int)sh.r);
    w->splitsA = colreduce_splits(sh.M, sh.d_in, (int)sh.r);
    w->PB = c.take<float>((size_t)w->splitsB * sh.d_out * sh.r);
    w->PA = c.take<float>((size_t)w->splitsA * sh.d_in * sh.r);
    w->csum = c.take<float>((size_t)w->splitsB * sh.d_out);
    if (w->rc.pm > 0) w->Gp = c.take<float>((size_t)w->rc.pn * sh.M * sh.r);
  } else {
    w->splitsB = w->splitsA = 1;
    w->PB = w->PA = nullptr;
    w->csum = c.take<float>((size_t)sh.d_out);
  }
  return c.off;
}

struct DoraFwdWs {
  uint32_t* err;
  void* Zs;
  float* Kr;   // [r, r]
  float* c;    // [out]
};
size_t plan_dora_fwd(const lora_shape& sh, char* base, DoraFwdWs* w) {
  Carve c{base};
  const size_t es = sh.dtype == LORA_BF16 ? 2 : 4;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->Zs = c.take<char>((size_t)sh.M * sh.r * es);
  w->Kr = c.take<float>((size_t)sh.r * sh.r);
  w->c = c.take<float>((size_t)sh.d_out);
  return c.off;
}

// Row slabs of the DoRA-rows backward (bf16): the column pass writes dY o c for one slab of rows
// into a buffer of at most kDoraSlabBytes and the dX GEMM of that slab reads it back right away
// (part of it still in L2), before the next slab overwrites it; the buffer's size does not grow
// with M.  The slab height (a multiple of 128 rows) is the one whose GEMMs finish the whole dX
// product in the fewest waves of 128 x 256 tiles over the SMs, the tallest among equals.
constexpr int64_t kDoraSlabBytes = 64ll << 20;
struct DoraSlabs {
  int64_t rows = 0, count = 0;
  int splits = 1, splits_last = 1;   // column-pass row splits of a full slab and of the last one
};
DoraSlabs dora_slabs(int64_t M, int64_t in, int64_t out, int64_t r) {
  DoraSlabs s;
  if (M <= 0) return s;
  const int64_t mt = (M + 127) / 128, nt = (in + 255) / 256, sms = num_sms_current();
  int64_t cap = kDoraSlabBytes / (out * 2) / 128;
  if (cap < 1) cap = 1;
  const char* e = getenv("LORA_GB300_DORA_SLAB_ROWS");   // a fixed slab height (rounded up to 128 rows)
  const int64_t forced = e ? (atoll(e) + 127) / 128 : 0;
  if (forced > 0) {
    s.rows = forced >= mt ? M : forced * 128;
  } else if (cap >= mt) {
    s.rows = M;
  } else {
    int64_t best_h = cap, best_w = (int64_t)1 << 62;
    for (int64_t h = cap; h >= 1; --h) {
      const int64_t n = mt / h, rem = mt - n * h;
      const int64_t w = n * ((h * nt + sms - 1) / sms) + (rem ? (rem * nt + sms - 1) / sms : 0);
      if (w < best_w) {
        best_w = w;
        best_h = h;
      }
    }
    s.rows = best_h * 128;
  }
  s.count = (M + s.rows - 1) / s.rows;
  s.splits = colreduce_splits(s.rows, out, (int)r, true);
  s.splits_last = colreduce_splits(M - (s.count - 1) * s.rows, out, (int)r, true);
  return s;
}

struct DoraBwdWs {
  uint32_t* err;
  float *c, *g, *dot, *csum, *dotp, *csump, *Kr, *Kg, *Gw;
  void *Bc, *gB, *Gs, *Zrec;
  bf16* slab;        // [slab rows, out] dY o c of one slab (bf16)
  DoraSlabs sl;
  float *PB, *PA, *PW;
  int splitsB, splitsA, splitsW;
};
size_t plan_dora_bwd(const lora_shape& sh, char* base, DoraBwdWs* w) {
  Carve c{base};
  const size_t es = sh.dtype == LORA_BF16 ? 2 : 4;
  const int64_t out = sh.d_out, in = sh.d_in, r = sh.r, M = sh.M;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->c = c.take<float>((out + 63) / 64 * 64);   // zero past out: the dX GEMM fetches 64 scales per k-step
  w->g = c.take<float>(out);
  w->dot = c.take<float>(out);
  w->csum = c.take<float>(out);
  w->Kr = c.take<float>(r * r);
  w->Kg = c.take<float>(r * r);
  w->Gw = c.take<float>(gram_work_floats((int)r));
  w->Bc = c.take<char>(out * r * es);
  w->gB = c.take<char>(out * r * es);
  w->Gs = c.take<char>(M * r * es);
  w->Zrec = c.take<char>(M * r * es);
  w->slab = nullptr;
  if (sh.dtype == LORA_BF16) {
    w->sl = dora_slabs(M, in, out, r);
    w->slab = c.take<bf16>(w->sl.rows * out);
    w->splitsB = w->sl.count > 0 ? (int)((w->sl.count - 1) * w->sl.splits + w->sl.splits_last) : 1;   // the slabs' in turn
    w->splitsA = colreduce_splits(M, in, (int)r);
    w->splitsW = colreduce_splits(out, in, (int)r);
    w->PB = c.take<float>(w->splitsB * out * r);
    w->PA = c.take<float>(w->splitsA * in * r);
    w->PW = c.take<float>(w->splitsW * in * r);
    w->dotp = c.take<float>(w->splitsB * out);
    w->csump = c.take<float>(w->splitsB * out);
  } else {
    w->splitsB = w->splitsA = w->splitsW = 1;
    w->PB = w->PA = w->PW = nullptr;
    w->dotp = w->csump = nullptr;
  }
  return c.off;
}

// DoRA column variant (bf16 only)
struct DoraColsFwdWs {
  uint32_t* err;
  float* PU;     // [splitsW, in, r] partials of W0^T B
  float* Kb;     // [r, r] B^T B
  float* Gw;     // gram partials
  float* c;      // [in]
  bf16* Ac;      // [r, in] A diag(c)
  bf16* Zs;      // [M, r] s Z
  bf16* Xc;      // [M, in] X diag(c)
  int splitsW;
};
size_t plan_dora_cols_fwd(const lora_shape& sh, char* base, DoraColsFwdWs* w) {
  Carve c{base};
  const int64_t out = sh.d_out, in = sh.d_in, r = sh.r, M = sh.M;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->splitsW = colreduce_splits(out, in, (int)r);
  w->PU = c.take<float>(w->splitsW * in * r);
  w->Kb = c.take<float>(r * r);
  w->Gw = c.take<float>(gram_work_floats((int)r));
  w->c = c.take<float>(in);
  w->Ac = c.take<bf16>(r * in);
  w->Zs = c.take<bf16>(M * r);
  w->Xc = c.take<bf16>(M * in);
  return c.off;
}

struct DoraColsBwdWs {
  uint32_t* err;
  float *c, *g, *dot, *dotp, *Kb, *Kga, *Vg, *PA, *PB, *csump, *Gw;
  float* Gp;       // row partials of the one pass over dY (rowcol)
  RowColPlan rc;   // pm 0: two passes over dY
  bf16 *Ac, *Ag, *Gs, *Zrec, *dXt;
  int splitsA, splitsB;
};
size_t plan_dora_cols_bwd(const lora_shape& sh, char* base, DoraColsBwdWs* w) {
  Carve c{base};
  const int64_t out = sh.d_out, in = sh.d_in, r = sh.r, M = sh.M;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->splitsA = colreduce_splits(M, in, (int)r, true);   // with dX as the second input
  w->rc = dy_plan(M, out, r);
  w->splitsB = w->rc.pm > 0 ? w->rc.pm : colreduce_splits(M, out, (int)r);
  w->Gp = w->rc.pm > 0 ? c.take<float>((size_t)w->rc.pn * M * r) : nullptr;
  w->c = c.take<float>(in);
  w->g = c.take<float>(in);
  w->dot = c.take<float>(in);
  w->dotp = c.take<float>(w->splitsA * in);
  w->Kb = c.take<float>(r * r);
  w->Kga = c.take<float>(r * r);
  w->Gw = c.take<float>(gram_work_floats((int)r));
  w->Vg = c.take<float>(out * r);
  w->PA = c.take<float>(w->splitsA * in * r);
  w->PB = c.take<float>(w->splitsB * out * r);
  w->csump = c.take<float>(w->splitsB * out);
  w->Ac = c.take<bf16>(r * in);
  w->Ag = c.take<bf16>(r * in);
  w->Gs = c.take<bf16>(M * r);
  w->Zrec = c.take<bf16>(M * r);
  w->dXt = c.take<bf16>(M * in);
  return c.off;
}

struct MlpFwdWs {
  uint32_t* err;
  bf16 *Agu, *Zgus, *Zds;
};
size_t plan_mlp_fwd(const lora_mlp_shape& sh, char* base, MlpFwdWs* w) {
  Carve c{base};
  const int64_t rgu = sh.r_g + sh.r_u;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->Agu = c.take<bf16>(rgu * sh.H);
  w->Zgus = c.take<bf16>(sh.M * rgu);
  w->Zds = c.take<bf16>(sh.M * sh.r_d);
  return c.off;
}

inline int64_t mlp_ipad(const lora_mlp_shape& sh) { return (sh.I + 63) / 64 * 64; }

struct MlpBwdWs {
  uint32_t* err;
  bf16 *dedu, *Gds, *Ggus, *Agu;
  float *PBd, *PAd, *PBg, *PBu, *PAgu;
  float *Gpd, *Gpg, *Gpu;      // row partials of the one-pass dY sides (null: two passes)
  RowColPlan rcd, rcg, rcu;    // one pass over dY, de, du
  int sBd, sAd, sBg, sBu, sAgu;
};
size_t plan_mlp_bwd(const lora_mlp_shape& sh, char* base, MlpBwdWs* w) {
  Carve c{base};
  const int64_t M = sh.M, H = sh.H, I = sh.I, Ip = mlp_ipad(sh);
  const int64_t rg = sh.r_g, ru = sh.r_u, rd = sh.r_d, rgu = rg + ru;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->dedu = c.take<bf16>(M * 2 * Ip);
  w->Gds = c.take<bf16>(M * rd);
  w->Ggus = c.take<bf16>(M * rgu);
  w->Agu = c.take<bf16>(rgu * H);
  w->rcd = dy_plan(M, H, rd);
  w->rcg = dy_plan(M, I, rg);
  w->rcu = dy_plan(M, I, ru);
  w->sBd = w->rcd.pm > 0 ? w->rcd.pm : colreduce_splits(M, H, (int)rd);
  w->sAd = colreduce_splits(M, I, (int)rd);
  w->sBg = w->rcg.pm > 0 ? w->rcg.pm : colreduce_splits(M, I, (int)rg);
  w->sBu = w->rcu.pm > 0 ? w->rcu.pm : colreduce_splits(M, I, (int)ru);
  w->sAgu = colreduce_splits(M, H, (int)rgu);
  w->PBd = c.take<float>(w->sBd * H * rd);
  w->PAd = c.take<float>(w->sAd * I * rd);
  w->PBg = c.take<float>(w->sBg * I * rg);
  w->PBu = c.take<float>(w->sBu * I * ru);
  w->PAgu = c.take<float>(w->sAgu * H * rgu);
  w->Gpd = w->rcd.pm > 0 ? c.take<float>((int64_t)w->rcd.pn * M * rd) : nullptr;
  w->Gpg = w->rcg.pm > 0 ? c.take<float>((int64_t)w->rcg.pn * M * rg) : nullptr;
  w->Gpu = w->rcu.pm > 0 ? c.take<float>((int64_t)w->rcu.pn * M * ru) : nullptr;
  return c.off;
}

// fused-leaf (QKV) plans: packed operands A_stack [L r, in], B_blk [N, L r]
int64_t qkv_N(const lora_qkv_shape& sh) {
  int64_t n = 0;
  for (int l = 0; l < sh.L; ++l) n += sh.n[l];
  return n;
}
struct QkvFwdWs {
  uint32_t* err;
  bf16* A_stack;
  bf16* B_blk;
  bf16* Z;       // when no Z_save
};
size_t plan_qkv_fwd(const lora_qkv_shape& sh, char* base, QkvFwdWs* w) {
  Carve c{base};
  const int64_t R = (int64_t)sh.L * sh.r;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->A_stack = c.take<bf16>(R * sh.d_in);
  w->B_blk = c.take<bf16>(qkv_N(sh) * R);
  w->Z = c.take<bf16>(sh.M * R);
  return c.off;
}
struct QkvBwdWs {
  uint32_t* err;
  bf16* A_stack;
  bf16* Gs;      // [M, L r] = [s_l dY_l B_l]
  bf16* Zrec;    // [M, L r] when no Z_saved
  float* PA;     // [splitsA, in, L r]
  float* PB[kMaxLeaves];    // [splitsB[l], n_l, r]
  float* csum[kMaxLeaves];  // [splitsB[l], n_l]
  RowColPlan rc[kMaxLeaves];  // one pass over each leaf's columns of dY (pm 0: two passes)
  float* Gp;                  // row partials of that pass, reused leaf after leaf
  int splitsA, splitsB[kMaxLeaves];
};
size_t plan_qkv_bwd(const lora_qkv_shape& sh, char* base, QkvBwdWs* w) {
  Carve c{base};
  const int64_t R = (int64_t)sh.L * sh.r;
  w->err = c.take<uint32_t>(kErrBytes / 4);
  w->A_stack = c.take<bf16>(R * sh.d_in);
  w->Gs = c.take<bf16>(sh.M * R);
  w->Zrec = c.take<bf16>(sh.M * R);
  w->splitsA = colreduce_splits(sh.M, sh.d_in, (int)R);
  w->PA = c.take<float>((size_t)w->splitsA * sh.d_in * R);
  size_t gp = 0;
  for (int l = 0; l < kMaxLeaves; ++l) {
    const bool live = l < sh.L;
    w->rc[l] = live ? dy_plan(sh.M, sh.n[l], sh.r) : RowColPlan{};
    w->splitsB[l] = !live ? 0 : w->rc[l].pm > 0 ? w->rc[l].pm : colreduce_splits(sh.M, sh.n[l], sh.r);
    w->PB[l] = live ? c.take<float>((size_t)w->splitsB[l] * sh.n[l] * sh.r) : nullptr;
    w->csum[l] = live ? c.take<float>((size_t)w->splitsB[l] * sh.n[l]) : nullptr;
    if (w->rc[l].pm > 0 && (size_t)w->rc[l].pn * sh.M * sh.r > gp) gp = (size_t)w->rc[l].pn * sh.M * sh.r;
  }
  w->Gp = gp ? c.take<float>(gp) : nullptr;
  return c.off;
}

// ------------------------------------------------------------------ bf16 helpers
TcGemmDesc fwd_desc(int64_t M, int64_t N, int64_t K, const void* X, const void* W, const void* Zs, const void* B,
                    int r, void* Y, const bf16* bias, const float* cs, uint32_t* err) {
  TcGemmDesc d;
  d.mode = TC_FWD;
  d.M = (int)M;
  d.N = (int)N;
  d.K0 = (int)K;
  d.A0 = X;
  d.lda0 = K;
  d.B0 = W;
  d.ldb0 = K;
  d.has_tail = Zs != nullptr;
  d.A1 = Zs;
  d.lda1 = r;
  d.K1 = r;
  d.K1_a = r;
  d.B1 = B;
  d.ldb1 = r;
  d.K1_b = r;
  d.out[0] = Y;
  d.ldo = N;
  d.bias = bias;
  d.col_scale = cs;
  d.err = err;
  d.timeout_ns = wait_timeout_ns();
  return d;
}

TcGemmDesc dx_desc(int64_t M, int64_t N /*in*/, int64_t K /*out*/, const void* dY, const void* W0, const void* Gs,
                   const void* A, int r, void* dX, const float* kscale, uint32_t* err) {
  TcGemmDesc d;
  d.mode = TC_BWD_DX;
  d.M = (int)M;
  d.N = (int)N;
  d.K0 = (int)K;
  d.A0 = dY;
  d.lda0 = K;
  d.B0 = W0;
  d.ldb0 = N;
  d.b0_mn = true;
  d.b0_rows = (int)K;
  d.has_tail = Gs != nullptr;
  d.b1_mn = true;
  d.A1 = Gs;
  d.lda1 = r;
  d.K1 = r;
  d.K1_a = r;
  d.B1 = A;
  d.ldb1 = N;
  d.out[0] = dX;
  d.ldo = N;
  d.a_kscale = kscale;
  d.err = err;
  d.timeout_ns = wait_timeout_ns();
  return d;
}

RowProjDesc rp_desc(int64_t rows, int64_t K, int R, const void* S, const void* U, bool kr, uint32_t* err) {
  RowProjDesc d;
  d.rows = rows;
  d.K = K;
  d.R = R;
  d.S = static_cast<const bf16*>(S);
  d.lds = K;
  d.U = static_cast<const bf16*>(U);
  d.u_kr = kr;
  d.ldu = kr ? R : K;
  d.err = err;
  d.timeout_ns = wait_timeout_ns();
  return d;
}

ColReduceDesc cr_desc(int64_t rows, int64_t K, int R, const void* S, const void* T, int64_t ldt, float* part,
                      int splits, uint32_t* err) {
  ColReduceDesc d;
  d.rows = rows;
  d.K = K;
  d.R = R;
  d.S = static_cast<const bf16*>(S);
  d.lds = K;
  d.T = static_cast<const bf16*>(T);
  d.ldt = ldt;
  d.part = part;
  d.splits = splits;
  d.err = err;
  d.timeout_ns = wait_timeout_ns();
  return d;
}

// The two rank-r products of one projection's backward that read the same S [M, K] (row stride
// lds): the dB partials part[split][K][R] = S^T T per row split and gout [M, R] (row stride ldg) =
// bf16(s S U) with U [K, R], and (when colsum is set) the column sums of S per split.  One rowcol
// pass (plan pl, row partials in gp) when pl.pm > 0, else a colreduce pass and a rowproj pass.
cudaError_t dy_side(const RowColPlan& pl, int64_t M, int64_t K, int R, const void* S, int64_t lds, const void* U,
                    const void* T, int64_t ldt, float* part, int splits, float* gp, float s, bf16* gout, int64_t ldg,
                    uint32_t* err, cudaStream_t st, float* colsum = nullptr) {
  cudaError_t e;
  if (pl.pm > 0) {
    RowColDesc d;
    d.rows = M;
    d.K = K;
    d.R = R;
    d.S = static_cast<const bf16*>(S);
    d.lds = lds;
    d.U = static_cast<const bf16*>(U);
    d.ldu = R;
    d.T = static_cast<const bf16*>(T);
    d.ldt = ldt;
    d.gpart = gp;
    d.part = part;
    d.colsum = colsum;
    d.pm = pl.pm;
    d.pn = pl.pn;
    d.nb = pl.nb;
    d.err = err;
    d.timeout_ns = wait_timeout_ns();
    if ((e = rowcol(d, st)) != cudaSuccess) return e;
    return gpart_sum(gp, pl.pn, M, R, s, gout, ldg, st);
  }
  ColReduceDesc c = cr_desc(M, K, R, S, T, ldt, part, splits, err);
  c.lds = lds;
  c.colsum = colsum;
  if ((e = colreduce(c, st)) != cudaSuccess) return e;
  RowProjDesc d = rp_desc(M, K, R, S, U, true, err);
  d.lds = lds;
  d.out_b = gout;
  d.scale_b = s;
  d.ldo = ldg;
  return rowproj(d, st);
}

// K = B^T T (fp32 [r, r]) for bf16 B, T [rows, r]: a column reduction of B against T on the warp
// MMAs (T = B gives B^T B, T = g o B gives B^T diag(g) B), then the split partials summed in
// order.  `work` holds gram_work_floats(r) floats.
cudaError_t gram_bf16(const void* B, const void* T, int64_t rows, int r, float* K, float* work, uint32_t* err,
                      cudaStream_t st) {
  const int splits = colreduce_splits(rows, r, r);
  cudaError_t e = colreduce(cr_desc(rows, r, r, B, T, r, work, splits, err), st);
  if (e != cudaSuccess) return e;
  return sum_splits<float>(work, splits, (int64_t)r * r, K, nullptr, st);
}

SgemmDesc sg(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, bool ta, const void* B, int64_t ldb, bool tb,
             void* C, int64_t ldc, float alpha = 1.f, float beta = 0.f) {
  SgemmDesc d;
  d.M = M;
  d.N = N;
  d.K = K;
  d.A = static_cast<const float*>(A);
  d.lda = lda;
  d.ta = ta;
  d.B = static_cast<const float*>(B);
  d.ldb = ldb;
  d.tb = tb;
  d.C = static_cast<float*>(C);
  d.ldc = ldc;
  d.alpha = alpha;
  d.beta = beta;
  return d;
}

}  // namespace

// ============================================================================ ABI
extern "C" {

const char* lora_status_string(int status) {
  switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID_ARG: return "invalid argument";
    case LORA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LORA_ERR_MISALIGNED: return "misaligned pointer";
    case LORA_ERR_WORKSPACE: return "workspace missing or too small";
    case LORA_ERR_CUDA: return "CUDA error";
    case LORA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int lora_abi_version(void) { return 8; }

// Input dropout: with rows of d_in bytes a multiple of 16 the mask is read by TMA next to X in the
// rank-r passes (Z = Xd A^T, the dA partials Xd^T (s G)), which form Xd = X o mask k in registers;
// otherwise Xd [M, d_in] is written once into the workspace and those passes read it.
static bool dropout_fused(const lora_shape& sh) {
  const char* e = getenv("LORA_GB300_DROPOUT_XD");   // =1: write Xd even when the mask could be fused
  return sh.d_in % 16 == 0 && !(e && atoi(e) == 1);
}
static size_t dropout_xd_bytes(const lora_shape& sh) {
  return dropout_fused(sh) ? 0 : al256((size_t)sh.M * sh.d_in * 2);
}

size_t lora_workspace_bytes(int op, const lora_shape* sh) {
  if (check_shape(sh) != LORA_OK) return 0;
  switch (op) {
    case LORA_OP_LINEAR_FWD: { LinFwdWs w; return plan_lin_fwd(*sh, nullptr, &w); }
    case LORA_OP_LINEAR_BWD: { LinBwdWs w; return plan_lin_bwd(*sh, nullptr, &w); }
    case LORA_OP_DORA_FWD: { DoraFwdWs w; return plan_dora_fwd(*sh, nullptr, &w); }
    case LORA_OP_DORA_BWD: { DoraBwdWs w; return plan_dora_bwd(*sh, nullptr, &w); }
    case LORA_OP_DROPOUT_FWD:
      if (sh->dtype != LORA_BF16) return 0;
      { LinFwdWs w; return plan_lin_fwd(*sh, nullptr, &w) + dropout_xd_bytes(*sh); }
    case LORA_OP_DROPOUT_BWD:
      if (sh->dtype != LORA_BF16) return 0;
      { LinBwdWs w; return plan_lin_bwd(*sh, nullptr, &w) + dropout_xd_bytes(*sh); }
    case LORA_OP_DORA_COLS_FWD:
      if (sh->dtype != LORA_BF16) return 0;
      { DoraColsFwdWs w; return plan_dora_cols_fwd(*sh, nullptr, &w); }
    case LORA_OP_DORA_COLS_BWD:
      if (sh->dtype != LORA_BF16) return 0;
      { DoraColsBwdWs w; return plan_dora_cols_bwd(*sh, nullptr, &w); }
  }
  return 0;
}

static lora_status check_mlp_shape(const lora_mlp_shape* sh) {
  if (!sh) return LORA_ERR_INVALID_ARG;
  if (sh->M < 0 || sh->H <= 0 || sh->I <= 0 || sh->r_g <= 0 || sh->r_u <= 0 || sh->r_d <= 0)
    return LORA_ERR_INVALID_ARG;
  if (sh->dtype != LORA_BF16) return sh->dtype == LORA_F32 ? LORA_ERR_UNSUPPORTED : LORA_ERR_INVALID_ARG;
  if (sh->act != LORA_ACT_SWIGLU && sh->act != LORA_ACT_GEGLU) return LORA_ERR_INVALID_ARG;
  if (sh->H % 8 || sh->I % 8) return LORA_ERR_UNSUPPORTED;
  for (const int64_t r : {sh->r_g, sh->r_u, sh->r_d})
    if (r % 8 || r > 128) return LORA_ERR_UNSUPPORTED;
  if (sh->M > (1LL << 31) - 1 || 2 * mlp_ipad(*sh) > (1LL << 31) - 1) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

size_t lora_mlp_workspace_bytes(int op, const lora_mlp_shape* sh) {
  if (check_mlp_shape(sh) != LORA_OK) return 0;
  if (op == LORA_OP_MLP_FWD) { MlpFwdWs w; return plan_mlp_fwd(*sh, nullptr, &w); }
  if (op == LORA_OP_MLP_BWD) { MlpBwdWs w; return plan_mlp_bwd(*sh, nullptr, &w); }
  return 0;
}

static lora_status check_qkv_shape(const lora_qkv_shape* sh) {
  if (!sh) return LORA_ERR_INVALID_ARG;
  if (sh->M < 0 || sh->d_in <= 0 || sh->r <= 0 || sh->L < 1 || sh->L > kMaxLeaves) return LORA_ERR_INVALID_ARG;
  if (sh->dtype != LORA_BF16) return sh->dtype == LORA_F32 ? LORA_ERR_UNSUPPORTED : LORA_ERR_INVALID_ARG;
  for (int l = 0; l < sh->L; ++l) {
    if (sh->n[l] <= 0) return LORA_ERR_INVALID_ARG;
    if (sh->n[l] % 8) return LORA_ERR_UNSUPPORTED;
  }
  if (sh->d_in % 8 || sh->r % 8 || sh->r > 128) return LORA_ERR_UNSUPPORTED;
  if (sh->M > (1LL << 31) - 1 || sh->d_in > (1LL << 31) - 1 || qkv_N(*sh) > (1LL << 31) - 1)
    return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

size_t lora_qkv_workspace_bytes(int op, const lora_qkv_shape* sh) {
  if (check_qkv_shape(sh) != LORA_OK) return 0;
  if (op == LORA_OP_QKV_FWD) { QkvFwdWs w; return plan_qkv_fwd(*sh, nullptr, &w); }
  if (op == LORA_OP_QKV_BWD) { QkvBwdWs w; return plan_qkv_bwd(*sh, nullptr, &w); }
  return 0;
}

lora_status lora_clear_device_error(void* ws, void* stream) {
  REQ(ws);
  if (reinterpret_cast<uintptr_t>(ws) & 255) return LORA_ERR_MISALIGNED;
  CK(cudaMemsetAsync(ws, 0, kErrBytes, (cudaStream_t)stream));
  return LORA_OK;
}

lora_status lora_check_device_error(const void* ws, void* stream) {
  REQ(ws);
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  uint32_t h[2] = {0, 0};
  CK(cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  return (h[0] & 1u) ? LORA_ERR_DEVICE_TIMEOUT : LORA_OK;  // bit 0: a bounded wait ran out
}

uint64_t lora_launch_count(void) { return launch_count(); }

lora_status lora_prof_enable(int on) {
  prof_set(on != 0);
  return LORA_OK;
}

lora_status lora_prof_gemm(double* ms, int64_t* launches, double* flops, int reset) {
  CK(prof_collect(0, ms, launches, flops, reset != 0));
  return LORA_OK;
}

lora_status lora_prof_rank(double* ms, int64_t* launches, double* bytes, int reset) {
  CK(prof_collect(1, ms, launches, bytes, reset != 0));
  return LORA_OK;
}

lora_status lora_debug_wait_timeout(void* ws, uint32_t timeout_us, void* stream) {
  REQ(ws);
  if (reinterpret_cast<uintptr_t>(ws) & 255) return LORA_ERR_MISALIGNED;
  CK(debug_wait_timeout(static_cast<uint32_t*>(ws), (uint64_t)timeout_us * 1000ull, (cudaStream_t)stream));
  return LORA_OK;
}

// ------------------------------------------------------------------ LoRA linear
lora_status lora_linear_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                            const void* bias, float s, void* Y, void* Z_save, void* ws, size_t ws_bytes,
                            void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQM(sh->M, Y);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(bias); ALN(Y); ALN(Z_save);
  if (!isfinite(s)) return LORA_ERR_INVALID_ARG;
  LinFwdWs w;
  const size_t need = plan_lin_fwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_lin_fwd(*sh, static_cast<char*>(ws), &w);
  if (sh->M == 0) return LORA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  if (sh->dtype == LORA_BF16) {
    if (s != 0.f && fused_down_projection(r)) {
      // Z = X A^T formed inside the GEMM from the X tiles it stages anyway: no second pass over X
      // and no Z round trip through memory before the tail (bf16(Z) still goes to Z_save)
      TcGemmDesc d = fwd_desc(M, out, in, X, W0, nullptr, B, r, Y, static_cast<const bf16*>(bias), nullptr, w.err);
      d.has_tail = true;
      d.dn_a = static_cast<const bf16*>(A);
      d.dn_lda = in;
      d.dn_s = s;
      d.dn_r = r;
      d.dn_z = static_cast<bf16*>(Z_save);
      CK(tc_gemm(d, st));
      return LORA_OK;
    }
    if (s != 0.f || Z_save) {
      RowProjDesc d = rp_desc(M, in, r, X, A, false, w.err);
      d.out_a = static_cast<bf16*>(Z_save);
      d.out_b = s != 0.f ? static_cast<bf16*>(w.Zs) : nullptr;
      d.scale_b = s;
      CK(rowproj(d, st));
    }
    // strength 0: the frozen base alone (no tail term at all)
    CK(tc_gemm(fwd_desc(M, out, in, X, W0, s != 0.f ? w.Zs : nullptr, B, r, Y, static_cast<const bf16*>(bias),
                        nullptr, w.err),
               st));
  } else {
    void* Z = Z_save ? Z_save : w.Zs;
    if (s != 0.f || Z_save) CK(sgemm_f32(sg(M, r, in, X, in, false, A, in, true, Z, r), st));
    SgemmDesc d = sg(M, out, in, X, in, false, W0, in, true, Y, out);
    d.bias = static_cast<const float*>(bias);
    CK(sgemm_f32(d, st));
    if (s != 0.f) CK(sgemm_f32(sg(M, out, r, Z, r, false, B, r, true, Y, out, s, 1.f), st));
  }
  return LORA_OK;
}

lora_status lora_linear_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                            const void* Z_saved, const void* dY, float s, void* dX, void* dA, void* dB, void* dbias,
                            void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQM(sh->M, dY); REQ(dA); REQ(dB);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(Z_saved); ALN(dY); ALN(dX); ALN(dA); ALN(dB); ALN(dbias);
  if (!isfinite(s)) return LORA_ERR_INVALID_ARG;
  LinBwdWs w;
  const size_t need = plan_lin_bwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_lin_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const size_t es = sh->dtype == LORA_BF16 ? 2 : 4;
  if (M == 0 || s == 0.f) {
    // no tokens, or strength 0: adapter gradients vanish; dX is the frozen base's
    CK(cudaMemsetAsync(dA, 0, (size_t)r * in * es, st));
    CK(cudaMemsetAsync(dB, 0, (size_t)out * r * es, st));
    if (dbias && M == 0) CK(cudaMemsetAsync(dbias, 0, (size_t)out * es, st));
    if (M == 0) return LORA_OK;
  }
  if (sh->dtype == LORA_BF16) {
    if (s == 0.f) {
      if (dX) CK(tc_gemm(dx_desc(M, in, out, dY, W0, nullptr, A, r, dX, nullptr, w.err), st));
      if (dbias) {
        ColReduceDesc d = cr_desc(M, out, 8, dY, dY, out, w.PB, w.splitsB, w.err);  // T unused beyond 8 cols
        d.colsum = w.csum;
        CK(colreduce(d, st));
        CK(sum_splits<bf16>(w.csum, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
      }
      return LORA_OK;
    }
    const void* Z = Z_saved;
    if (!Z) {
      RowProjDesc d = rp_desc(M, in, r, X, A, false, w.err);
      d.out_a = static_cast<bf16*>(w.Zrec);
      CK(rowproj(d, st));
      Z = w.Zrec;
    }
    // s G = s dY B, the dB partials dY^T Z and the column sums of dY: one rowcol pass over dY
    CK(dy_side(w.rc, M, out, r, dY, out, B, Z, r, w.PB, w.splitsB, w.Gp, s, static_cast<bf16*>(w.Gs), r, w.err, st,
               dbias ? w.csum : nullptr));
    if (dX) CK(tc_gemm(dx_desc(M, in, out, dY, W0, w.Gs, A, r, dX, nullptr, w.err), st));
    CK(colreduce(cr_desc(M, in, r, X, w.Gs, r, w.PA, w.splitsA, w.err), st));
    const FinJob fin[2] = {fin_dA(r, in, Partial{w.PA, w.splitsA, r, 0}, 1.f, A, dA),
                           fin_dB(out, r, Partial{w.PB, w.splitsB, r, 0}, s, B, dB)};
    CK(finalize_batch(fin, 2, st));
    if (dbias) CK(sum_splits<bf16>(w.csum, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
  } else {
    if (dX) CK(sgemm_f32(sg(M, in, out, dY, out, false, W0, in, false, dX, in), st));
    if (dbias) {
      CK(coldot_f32(static_cast<const float*>(dY), nullptr, M, out, w.csum, nullptr, st));
      CK(sum_splits<float>(w.csum, 1, out, static_cast<float*>(dbias), nullptr, st));
    }
    if (s == 0.f) return LORA_OK;
    const void* Z = Z_saved;
    if (!Z) {
      CK(sgemm_f32(sg(M, r, in, X, in, false, A, in, true, w.Zrec, r), st));
      Z = w.Zrec;
    }
    CK(sgemm_f32(sg(M, r, out, dY, out, false, B, r, false, w.Gs, r), st));            // G = dY B
    if (dX) CK(sgemm_f32(sg(M, in, r, w.Gs, r, false, A, in, false, dX, in, s, 1.f), st));  // dX += s G A
    CK(sgemm_f32(sg(r, in, M, w.Gs, r, true, X, in, false, dA, in, s), st));            // dA = s G^T X
    CK(sgemm_f32(sg(out, r, M, dY, out, true, Z, r, false, dB, r, s), st));             // dB = s dY^T Z
  }
  return LORA_OK;
}

// ------------------------------------------------------------------ LoRA with input dropout
// The workspace is the plain layer's followed by Xd = X o mask * keep_scale [M, d_in].
lora_status lora_linear_dropout_fwd(const lora_shape* sh, const void* X, const uint8_t* mask, float keep_scale,
                                    const void* W0, const void* A, const void* B, const void* bias, float s,
                                    void* Y, void* Z_save, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  if (sh->dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  REQM(sh->M, mask);
  ALN(mask);
  if (!isfinite(keep_scale) || keep_scale < 0.f) return LORA_ERR_INVALID_ARG;
  LinFwdWs w;
  const size_t lin = plan_lin_fwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, lin + dropout_xd_bytes(*sh))) != LORA_OK) return e;
  if (s == 0.f && Z_save == nullptr)  // nothing of the adapter branch reaches Y: the plain layer
    return lora_linear_fwd(sh, X, W0, A, B, bias, s, Y, nullptr, ws, lin, stream);
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQM(sh->M, Y);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(bias); ALN(Y); ALN(Z_save);
  if (!isfinite(s)) return LORA_ERR_INVALID_ARG;
  plan_lin_fwd(*sh, static_cast<char*>(ws), &w);
  if (sh->M == 0) return LORA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const bool fused = dropout_fused(*sh);
  const bf16* Xa = static_cast<const bf16*>(X);
  if (!fused) {
    bf16* Xd = reinterpret_cast<bf16*>(static_cast<char*>(ws) + lin);
    CK(apply_mask_bf16(static_cast<const bf16*>(X), mask, keep_scale, M, in, Xd, st));
    Xa = Xd;
  }
  {  // Z = Xd A^T (saved unscaled) and s Z for the GEMM tail
    RowProjDesc d = rp_desc(M, in, r, Xa, A, false, w.err);
    if (fused) {
      d.mask = mask;
      d.mask_scale = keep_scale;
    }
    d.out_a = static_cast<bf16*>(Z_save);
    d.out_b = s != 0.f ? static_cast<bf16*>(w.Zs) : nullptr;
    d.scale_b = s;
    CK(rowproj(d, st));
  }
  // the base product reads the undropped X; the rank-r tail carries the dropped-out branch
  CK(tc_gemm(fwd_desc(M, out, in, X, W0, s != 0.f ? w.Zs : nullptr, B, r, Y, static_cast<const bf16*>(bias),
                      nullptr, w.err),
             st));
  return LORA_OK;
}

lora_status lora_linear_dropout_bwd(const lora_shape* sh, const void* X, const uint8_t* mask, float keep_scale,
                                    const void* W0, const void* A, const void* B, const void* Z_saved,
                                    const void* dY, float s, void* dX, void* dA, void* dB, void* dbias,
                                    void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  if (sh->dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  REQM(sh->M, mask);
  ALN(mask);
  if (!isfinite(keep_scale) || keep_scale < 0.f) return LORA_ERR_INVALID_ARG;
  LinBwdWs w;
  const size_t lin = plan_lin_bwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, lin + dropout_xd_bytes(*sh))) != LORA_OK) return e;
  if (sh->M == 0 || s == 0.f)  // no adapter gradient flows: exactly the plain layer's backward
    return lora_linear_bwd(sh, X, W0, A, B, Z_saved, dY, s, dX, dA, dB, dbias, ws, lin, stream);
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQM(sh->M, dY); REQ(dA); REQ(dB);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(Z_saved); ALN(dY); ALN(dX); ALN(dA); ALN(dB); ALN(dbias);
  if (!isfinite(s)) return LORA_ERR_INVALID_ARG;
  plan_lin_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const bool fused = dropout_fused(*sh);
  const bf16* Xa = static_cast<const bf16*>(X);
  if (!fused) {
    bf16* Xd = reinterpret_cast<bf16*>(static_cast<char*>(ws) + lin);
    CK(apply_mask_bf16(static_cast<const bf16*>(X), mask, keep_scale, M, in, Xd, st));
    Xa = Xd;
  }
  const void* Z = Z_saved;
  if (!Z) {
    RowProjDesc d = rp_desc(M, in, r, Xa, A, false, w.err);
    if (fused) {
      d.mask = mask;
      d.mask_scale = keep_scale;
    }
    d.out_a = static_cast<bf16*>(w.Zrec);
    CK(rowproj(d, st));
    Z = w.Zrec;
  }
  // s G = s dY B, the dB partials dY^T Z and the column sums of dY
  CK(dy_side(w.rc, M, out, r, dY, out, B, Z, r, w.PB, w.splitsB, w.Gp, s, static_cast<bf16*>(w.Gs), r, w.err, st,
             dbias ? w.csum : nullptr));
  if (dX) {  // dY W0 on the tensor cores, then the masked adapter share in its own pass
    CK(tc_gemm(dx_desc(M, in, out, dY, W0, nullptr, A, r, dX, nullptr, w.err), st));
    CK(add_masked_rank_bf16(static_cast<bf16*>(dX), static_cast<const bf16*>(w.Gs), static_cast<const bf16*>(A),
                            mask, keep_scale, M, in, r, st));
  }
  {  // Xd^T (s G)
    ColReduceDesc d = cr_desc(M, in, r, Xa, w.Gs, r, w.PA, w.splitsA, w.err);
    if (fused) {
      d.mask = mask;
      d.mask_scale = keep_scale;
    }
    CK(colreduce(d, st));
  }
  const FinJob fin[2] = {fin_dA(r, in, Partial{w.PA, w.splitsA, r, 0}, 1.f, A, dA),
                         fin_dB(out, r, Partial{w.PB, w.splitsB, r, 0}, s, B, dB)};
  CK(finalize_batch(fin, 2, st));
  if (dbias) CK(sum_splits<bf16>(w.csum, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
  return LORA_OK;
}

// ------------------------------------------------------------------ fused-leaf (QKV) LoRA linear
static lora_status check_leaves(const lora_qkv_shape& sh, const lora_adapter* lv, bool* any_live) {
  REQ(lv);
  *any_live = false;
  for (int l = 0; l < sh.L; ++l) {
    REQ(lv[l].A); REQ(lv[l].B);
    ALN(lv[l].A); ALN(lv[l].B);
    if (!isfinite(lv[l].s)) return LORA_ERR_INVALID_ARG;
    if (lv[l].s != 0.f) *any_live = true;
  }
  return LORA_OK;
}

static LeafPack leaf_pack(const lora_qkv_shape& sh, const lora_adapter* lv, bf16* A_stack, bf16* B_blk) {
  LeafPack p;
  p.L = sh.L;
  p.r = (int)sh.r;
  p.in = sh.d_in;
  p.N = qkv_N(sh);
  int64_t row = 0;
  for (int l = 0; l < sh.L; ++l) {
    p.row0[l] = row;
    row += sh.n[l];
    p.A[l] = static_cast<const bf16*>(lv[l].A);
    p.B[l] = static_cast<const bf16*>(lv[l].B);
    p.s[l] = lv[l].s;
  }
  p.A_stack = A_stack;
  p.B_blk = B_blk;
  return p;
}

// Leaves are handled in groups of at most 64 adapter columns (the width of the rank-r kernels):
// group g covers leaves [first, last) with columns [first r, last r) of Z, G and the partials.
struct LeafGroups {
  int n = 0;
  int first[kMaxLeaves + 1] = {0, 0, 0, 0};
};
static LeafGroups leaf_groups(const lora_qkv_shape& sh) {
  LeafGroups g;
  const int per = (int)(64 / sh.r) > 0 ? (int)(64 / sh.r) : 1;
  for (int l = 0; l < sh.L; l += per) g.first[g.n++] = l;
  g.first[g.n] = (int)sh.L;
  return g;
}

// Z[:, group] = X A_group^T for every group (one pass over X per group; one pass in all when
// L r <= 64)
static lora_status qkv_down(const lora_qkv_shape& sh, const void* X, const bf16* A_stack, bf16* Z, uint32_t* err,
                            cudaStream_t st) {
  const LeafGroups g = leaf_groups(sh);
  const int r = (int)sh.r, R = (int)(sh.L * sh.r);
  for (int i = 0; i < g.n; ++i) {
    const int c0 = g.first[i] * r, Rg = (g.first[i + 1] - g.first[i]) * r;
    RowProjDesc d = rp_desc(sh.M, sh.d_in, Rg, X, A_stack + (int64_t)c0 * sh.d_in, false, err);
    d.out_a = Z + c0;
    d.ldo = R;
    CK(rowproj(d, st));
  }
  return LORA_OK;
}

lora_status lora_qkv_fwd(const lora_qkv_shape* sh, const void* X, const void* W0, const lora_adapter* leaves,
                         const void* bias, void* Y, void* Z_save, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_qkv_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQM(sh->M, Y);
  ALN(X); ALN(W0); ALN(bias); ALN(Y); ALN(Z_save);
  bool live = false;
  if ((e = check_leaves(*sh, leaves, &live)) != LORA_OK) return e;
  QkvFwdWs w;
  if ((e = check_ws(ws, ws_bytes, plan_qkv_fwd(*sh, nullptr, &w))) != LORA_OK) return e;
  plan_qkv_fwd(*sh, static_cast<char*>(ws), &w);
  if (sh->M == 0) return LORA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, N = qkv_N(*sh);
  const int R = (int)(sh->L * sh->r);
  CK(pack_leaves(leaf_pack(*sh, leaves, w.A_stack, w.B_blk), st));
  bf16* Z = Z_save ? static_cast<bf16*>(Z_save) : w.Z;
  if (live || Z_save) {  // every leaf's down-projection (one pass over X when L r <= 64)
    if ((e = qkv_down(*sh, X, w.A_stack, Z, w.err, st)) != LORA_OK) return e;
  }
  // the base product of all leaves and the block-diagonal rank-(L r) tail in one GEMM
  CK(tc_gemm(fwd_desc(M, N, in, X, W0, live ? Z : nullptr, w.B_blk, R, Y, static_cast<const bf16*>(bias), nullptr,
                      w.err),
             st));
  return LORA_OK;
}

lora_status lora_qkv_bwd(const lora_qkv_shape* sh, const void* X, const void* W0, const lora_adapter* leaves,
                         const void* Z_saved, const void* dY, void* dX, void* const* dA, void* const* dB,
                         void* dbias, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_qkv_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQM(sh->M, dY); REQ(dA); REQ(dB);
  ALN(X); ALN(W0); ALN(Z_saved); ALN(dY); ALN(dX); ALN(dbias);
  for (int l = 0; l < sh->L; ++l) {
    REQ(dA[l]); REQ(dB[l]);
    ALN(dA[l]); ALN(dB[l]);
  }
  bool live = false;
  if ((e = check_leaves(*sh, leaves, &live)) != LORA_OK) return e;
  QkvBwdWs w;
  if ((e = check_ws(ws, ws_bytes, plan_qkv_bwd(*sh, nullptr, &w))) != LORA_OK) return e;
  plan_qkv_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, N = qkv_N(*sh);
  const int r = (int)sh->r, R = (int)(sh->L * sh->r);
  if (M == 0 || !live) {
    // no tokens, or every strength 0: adapter gradients vanish; dX is the frozen base's
    for (int l = 0; l < sh->L; ++l) {
      CK(cudaMemsetAsync(dA[l], 0, (size_t)r * in * 2, st));
      CK(cudaMemsetAsync(dB[l], 0, (size_t)sh->n[l] * r * 2, st));
    }
    if (M == 0) {
      if (dbias) CK(cudaMemsetAsync(dbias, 0, (size_t)N * 2, st));
      return LORA_OK;
    }
  }
  int64_t row0[kMaxLeaves] = {0, 0, 0};
  for (int l = 1; l < sh->L; ++l) row0[l] = row0[l - 1] + sh->n[l - 1];
  const bf16* dYb = static_cast<const bf16*>(dY);
  if (!live) {
    if (dX) CK(tc_gemm(dx_desc(M, in, N, dY, W0, nullptr, nullptr, R, dX, nullptr, w.err), st));
    if (dbias) {
      for (int l = 0; l < sh->L; ++l) {
        ColReduceDesc d = cr_desc(M, sh->n[l], 8, dYb + row0[l], dY, N, w.PB[l], w.splitsB[l], w.err);
        d.lds = N;
        d.colsum = w.csum[l];
        CK(colreduce(d, st));
        CK(sum_splits<bf16>(w.csum[l], w.splitsB[l], sh->n[l], nullptr, static_cast<bf16*>(dbias) + row0[l], st));
      }
    }
    return LORA_OK;
  }
  CK(pack_leaves(leaf_pack(*sh, leaves, w.A_stack, nullptr), st));   // A_stack only
  const bf16* Z = static_cast<const bf16*>(Z_saved);
  if (!Z) {
    if ((e = qkv_down(*sh, X, w.A_stack, w.Zrec, w.err, st)) != LORA_OK) return e;
    Z = w.Zrec;
  }
  // leaf by leaf, one pass over its columns of dY: G_l = s_l dY_l B_l into its block of G, the dB
  // partials of the leaf (dY_l^T Z_l) and the column sums of dY_l
  for (int l = 0; l < sh->L; ++l)
    CK(dy_side(w.rc[l], M, sh->n[l], r, dYb + row0[l], N, leaves[l].B, Z + l * r, R, w.PB[l], w.splitsB[l], w.Gp,
               leaves[l].s, w.Gs + l * r, R, w.err, st, dbias ? w.csum[l] : nullptr));
  if (dX) CK(tc_gemm(dx_desc(M, in, N, dY, W0, w.Gs, w.A_stack, R, dX, nullptr, w.err), st));
  // X^T G partials per leaf group: group i's array [splitsA, in, R_i] starts at column offset c0
  const LeafGroups grp = leaf_groups(*sh);
  int grp_of[kMaxLeaves] = {0, 0, 0};
  for (int i = 0; i < grp.n; ++i) {
    const int c0 = grp.first[i] * r, Rg = (grp.first[i + 1] - grp.first[i]) * r;
    CK(colreduce(cr_desc(M, in, Rg, X, w.Gs + c0, R, w.PA + (size_t)w.splitsA * in * c0, w.splitsA, w.err), st));
    for (int l = grp.first[i]; l < grp.first[i + 1]; ++l) grp_of[l] = i;
  }
  FinJob fin[2 * kMaxLeaves];
  for (int l = 0; l < sh->L; ++l) {
    const int gi = grp_of[l], c0 = grp.first[gi] * r, Rg = (grp.first[gi + 1] - grp.first[gi]) * r;
    fin[2 * l] = fin_dA(r, in, Partial{w.PA + (size_t)w.splitsA * in * c0, w.splitsA, Rg, l * r - c0}, 1.f,
                        leaves[l].A, dA[l]);
    fin[2 * l + 1] = fin_dB(sh->n[l], r, Partial{w.PB[l], w.splitsB[l], r, 0}, leaves[l].s, leaves[l].B, dB[l]);
  }
  CK(finalize_batch(fin, 2 * sh->L, st));
  if (dbias)
    for (int l = 0; l < sh->L; ++l)
      CK(sum_splits<bf16>(w.csum[l], w.splitsB[l], sh->n[l], nullptr, static_cast<bf16*>(dbias) + row0[l], st));
  return LORA_OK;
}

// ------------------------------------------------------------------ DoRA
lora_status dora_rownorm2(const lora_shape* sh, const void* W0, float* r0, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  REQ(W0); REQ(r0);
  ALN(W0); ALN(r0);
  cudaStream_t st = (cudaStream_t)stream;
  if (sh->dtype == LORA_BF16) CK(rownorm2<bf16>(static_cast<const bf16*>(W0), sh->d_out, sh->d_in, r0, st));
  else CK(rownorm2<float>(static_cast<const float*>(W0), sh->d_out, sh->d_in, r0, st));
  return LORA_OK;
}

lora_status dora_linear_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                            const void* m, const void* bias, const float* r0, float s, float eps, void* Y,
                            void* Z_save, float* n_save, float* V_save, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQ(m); REQ(r0); REQM(sh->M, Y); REQ(n_save); REQ(V_save);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(m); ALN(bias); ALN(r0); ALN(Y); ALN(Z_save); ALN(n_save); ALN(V_save);
  if (!isfinite(s) || !isfinite(eps) || eps < 0.f) return LORA_ERR_INVALID_ARG;
  DoraFwdWs w;
  const size_t need = plan_dora_fwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_dora_fwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  if (sh->dtype == LORA_BF16) {
    {  // V = W0 A^T (fp32), one pass over W0
      RowProjDesc d = rp_desc(out, in, r, W0, A, false, w.err);
      d.out_f = V_save;
      CK(rowproj(d, st));
    }
    CK(gram_rows<bf16>(static_cast<const bf16*>(A), r, in, w.Kr, st));
    CK(dora_norm<bf16>(out, r, r0, V_save, static_cast<const bf16*>(B), w.Kr, static_cast<const bf16*>(m), s, eps,
                       n_save, w.c, st));
    if (M == 0) return LORA_OK;
    if (s != 0.f || Z_save) {
      RowProjDesc d = rp_desc(M, in, r, X, A, false, w.err);
      d.out_a = static_cast<bf16*>(Z_save);
      d.out_b = s != 0.f ? static_cast<bf16*>(w.Zs) : nullptr;
      d.scale_b = s;
      CK(rowproj(d, st));
    }
    if (s == 0.f)  // strength 0: frozen base X W0^T + bias
      CK(tc_gemm(fwd_desc(M, out, in, X, W0, nullptr, B, r, Y, static_cast<const bf16*>(bias), nullptr, w.err), st));
    else
      CK(tc_gemm(fwd_desc(M, out, in, X, W0, w.Zs, B, r, Y, static_cast<const bf16*>(bias), w.c, w.err), st));
  } else {
    CK(sgemm_f32(sg(out, r, in, W0, in, false, A, in, true, V_save, r), st));
    CK(gram_rows<float>(static_cast<const float*>(A), r, in, w.Kr, st));
    CK(dora_norm<float>(out, r, r0, V_save, static_cast<const float*>(B), w.Kr, static_cast<const float*>(m), s, eps,
                        n_save, w.c, st));
    if (M == 0) return LORA_OK;
    void* Z = Z_save ? Z_save : w.Zs;
    if (s != 0.f || Z_save) CK(sgemm_f32(sg(M, r, in, X, in, false, A, in, true, Z, r), st));
    SgemmDesc d = sg(M, out, in, X, in, false, W0, in, true, Y, out);
    if (s == 0.f) {
      d.bias = static_cast<const float*>(bias);
      CK(sgemm_f32(d, st));
    } else {
      d.cs = w.c;
      CK(sgemm_f32(d, st));
      SgemmDesc d2 = sg(M, out, r, Z, r, false, B, r, true, Y, out, s, 1.f);
      d2.cs = w.c;
      d2.bias = static_cast<const float*>(bias);
      CK(sgemm_f32(d2, st));
    }
  }
  return LORA_OK;
}

lora_status dora_linear_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                            const void* m, const void* bias, const void* Y, const void* Z_saved, const float* n_saved,
                            const float* V_saved, const void* dY, float s, float eps, void* dX, void* dA, void* dB,
                            void* dm, void* dbias, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQ(m); REQM(sh->M, Y); REQ(n_saved); REQ(V_saved); REQM(sh->M, dY);
  REQ(dA); REQ(dB); REQ(dm);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(m); ALN(bias); ALN(Y); ALN(Z_saved); ALN(n_saved); ALN(V_saved); ALN(dY);
  ALN(dX); ALN(dA); ALN(dB); ALN(dm); ALN(dbias);
  if (!isfinite(s) || !isfinite(eps) || eps < 0.f) return LORA_ERR_INVALID_ARG;
  DoraBwdWs w;
  const size_t need = plan_dora_bwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_dora_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const size_t es = sh->dtype == LORA_BF16 ? 2 : 4;
  const bool bf = sh->dtype == LORA_BF16;
  if (M == 0 || s == 0.f) {
    CK(cudaMemsetAsync(dA, 0, (size_t)r * in * es, st));
    CK(cudaMemsetAsync(dB, 0, (size_t)out * r * es, st));
    CK(cudaMemsetAsync(dm, 0, (size_t)out * es, st));
    if (M == 0) {
      if (dbias) CK(cudaMemsetAsync(dbias, 0, (size_t)out * es, st));
      return LORA_OK;
    }
    // strength 0: frozen base, dX = dY W0, dbias = colsum(dY)
    if (bf) {
      if (dX) CK(tc_gemm(dx_desc(M, in, out, dY, W0, nullptr, A, r, dX, nullptr, w.err), st));
      if (dbias) {
        ColReduceDesc d = cr_desc(M, out, 8, dY, dY, out, w.PB, w.splitsB, w.err);
        d.colsum = w.csump;
        CK(colreduce(d, st));
        CK(sum_splits<bf16>(w.csump, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
      }
    } else {
      if (dX) CK(sgemm_f32(sg(M, in, out, dY, out, false, W0, in, false, dX, in), st));
      if (dbias) {
        CK(coldot_f32(static_cast<const float*>(dY), nullptr, M, out, w.csum, nullptr, st));
        CK(sum_splits<float>(w.csum, 1, out, static_cast<float*>(dbias), nullptr, st));
      }
    }
    return LORA_OK;
  }
  if (bf) {
    const bf16* mb = static_cast<const bf16*>(m);
    CK(dora_c<bf16>(out, mb, n_saved, w.c, st, (out + 63) / 64 * 64));
    const void* Z = Z_saved;
    if (!Z) {
      RowProjDesc d = rp_desc(M, in, r, X, A, false, w.err);
      d.out_a = static_cast<bf16*>(w.Zrec);
      CK(rowproj(d, st));
      Z = w.Zrec;
    }
    CK(scale_rows<bf16>(static_cast<const bf16*>(B), out, r, w.c, 1.f, static_cast<bf16*>(w.Bc), st));
    {  // s * G = s (dY o c) B  =  s dY (c o B)
      RowProjDesc d = rp_desc(M, out, r, dY, w.Bc, true, w.err);
      d.out_b = static_cast<bf16*>(w.Gs);
      d.scale_b = s;
      CK(rowproj(d, st));
    }
    // Slab by slab: one pass over dY and Y (dY^T Z partials, colsum(dY), colsum(dY o Y)) that also
    // writes dP = dY o c for the slab's rows, then dX = dP W0 + s G A for those rows from that copy.
    // With the in-GEMM scaling (LORA_GB300_DORA_KSCALE=1) the passes write no copy and one dX GEMM
    // scales each staged dY tile by c in shared memory instead.
    const bool kscale = kscale_dx();
    const char* dYb = static_cast<const char*>(dY);
    const char* Yb = static_cast<const char*>(Y);
    int soff = 0;
    for (int64_t i = 0, row0 = 0; i < w.sl.count; ++i, row0 += w.sl.rows) {
      const int64_t rows = M - row0 < w.sl.rows ? M - row0 : w.sl.rows;
      const int sp = i + 1 < w.sl.count ? w.sl.splits : w.sl.splits_last;
      ColReduceDesc d = cr_desc(rows, out, r, dYb + row0 * out * 2, static_cast<const bf16*>(Z) + row0 * r, r,
                                w.PB + (int64_t)soff * out * r, sp, w.err);
      d.Y = reinterpret_cast<const bf16*>(Yb + row0 * out * 2);
      d.ldy = out;
      d.colsum = w.csump + (int64_t)soff * out;
      d.coldot = w.dotp + (int64_t)soff * out;
      if (dX && !kscale) {
        d.sc = w.c;
        d.sc_out = w.slab;
      }
      CK(colreduce(d, st));
      if (dX && !kscale)
        CK(tc_gemm(dx_desc(rows, in, out, w.slab, W0, static_cast<const bf16*>(w.Gs) + row0 * r, A, r,
                           static_cast<bf16*>(dX) + row0 * in, nullptr, w.err), st));
      soff += sp;
    }
    if (dX && kscale) CK(tc_gemm(dx_desc(M, in, out, dY, W0, w.Gs, A, r, dX, w.c, w.err), st));
    CK(dora_dc<bf16>(out, w.dotp, w.csump, w.splitsB, static_cast<const bf16*>(bias), w.c, n_saved, mb, eps, w.g,
                     static_cast<bf16*>(dm), static_cast<bf16*>(dbias), st));
    CK(scale_rows<bf16>(static_cast<const bf16*>(B), out, r, w.g, 1.f, static_cast<bf16*>(w.gB), st));
    CK(colreduce(cr_desc(M, in, r, X, w.Gs, r, w.PA, w.splitsA, w.err), st));        // X^T (s G)
    CK(colreduce(cr_desc(out, in, r, W0, w.gB, r, w.PW, w.splitsW, w.err), st));     // W0^T (g o B)
    CK(gram_rows<bf16>(static_cast<const bf16*>(A), r, in, w.Kr, st));
    CK(gram_bf16(B, w.gB, out, r, w.Kg, w.Gw, w.err, st));
    FinJob fin[2] = {fin_dA(r, in, Partial{w.PA, w.splitsA, r, 0}, 1.f, A, dA),
                     fin_dB(out, r, Partial{w.PB, w.splitsB, r, 0}, s, B, dB)};
    fin[0].PW = Partial{w.PW, w.splitsW, r, 0};   // + 2s (g o B)^T W0 + 2s^2 (B^T diag(g) B) A
    fin[0].sW = 2.f * s;
    fin[0].Kx = w.Kg;
    fin[0].s2 = 2.f * s * s;
    fin[1].rs = w.c;                               // c o (s dY^T Z) + 2s g o V + 2s^2 g o (B (A A^T))
    fin[1].g = w.g;
    fin[1].V = V_saved;
    fin[1].Kx = w.Kr;
    fin[1].s = s;
    CK(finalize_batch(fin, 2, st));
  } else {
    const float* mf = static_cast<const float*>(m);
    CK(dora_c<float>(out, mf, n_saved, w.c, st));
    const void* Z = Z_saved;
    if (!Z) {
      CK(sgemm_f32(sg(M, r, in, X, in, false, A, in, true, w.Zrec, r), st));
      Z = w.Zrec;
    }
    CK(coldot_f32(static_cast<const float*>(dY), static_cast<const float*>(Y), M, out, w.csum, w.dot, st));
    CK(dora_dc<float>(out, w.dot, w.csum, 1, static_cast<const float*>(bias), w.c, n_saved, mf, eps, w.g,
                      static_cast<float*>(dm), static_cast<float*>(dbias), st));
    {  // G = (dY o c) B
      SgemmDesc d = sg(M, r, out, dY, out, false, B, r, false, w.Gs, r);
      d.kscale = w.c;
      CK(sgemm_f32(d, st));
    }
    if (dX) {
      SgemmDesc d = sg(M, in, out, dY, out, false, W0, in, false, dX, in);
      d.kscale = w.c;
      CK(sgemm_f32(d, st));
      CK(sgemm_f32(sg(M, in, r, w.Gs, r, false, A, in, false, dX, in, s, 1.f), st));
    }
    CK(gram_rows<float>(static_cast<const float*>(A), r, in, w.Kr, st));
    CK(gram_weighted<float>(static_cast<const float*>(B), out, r, w.g, w.Kg, w.Gw, st));
    CK(scale_rows<float>(static_cast<const float*>(B), out, r, w.g, 1.f, static_cast<float*>(w.gB), st));
    CK(sgemm_f32(sg(r, in, M, w.Gs, r, true, X, in, false, dA, in, s), st));                 // s G^T X
    CK(sgemm_f32(sg(r, in, out, w.gB, r, true, W0, in, false, dA, in, 2.f * s, 1.f), st));  // + 2s (gB)^T W0
    CK(sgemm_f32(sg(r, in, r, w.Kg, r, false, A, in, false, dA, in, 2.f * s * s, 1.f), st)); // + 2s^2 Kg A
    {
      SgemmDesc d = sg(out, r, M, dY, out, true, Z, r, false, dB, r, s);  // s c o (dY^T Z)
      d.rscale = w.c;
      CK(sgemm_f32(d, st));
    }
    Partial none{};
    CK(finalize_dB<float>(out, r, none, 0.f, nullptr, w.g, V_saved, static_cast<const float*>(B), w.Kr, s, true,
                          static_cast<float*>(dB), st));
  }
  return LORA_OK;
}

// ------------------------------------------------------------------ DoRA (cols)
lora_status dora_colnorm2(const lora_shape* sh, const void* W0, float* c0, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  if (sh->dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  REQ(W0); REQ(c0);
  ALN(W0); ALN(c0);
  CK(colnorm2_bf16(static_cast<const bf16*>(W0), sh->d_out, sh->d_in, c0, (cudaStream_t)stream));
  return LORA_OK;
}

lora_status dora_cols_fwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                          const void* m, const void* bias, const float* c0, float s, float eps, void* Y, void* Z_save,
                          float* n_save, float* U_save, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  if (sh->dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQ(m); REQ(c0); REQM(sh->M, Y); REQ(n_save); REQ(U_save);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(m); ALN(bias); ALN(c0); ALN(Y); ALN(Z_save); ALN(n_save); ALN(U_save);
  if (!isfinite(s) || !isfinite(eps) || eps < 0.f) return LORA_ERR_INVALID_ARG;
  DoraColsFwdWs w;
  if ((e = check_ws(ws, ws_bytes, plan_dora_cols_fwd(*sh, nullptr, &w))) != LORA_OK) return e;
  plan_dora_cols_fwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const bf16* Ab = static_cast<const bf16*>(A);
  const bf16* Bb = static_cast<const bf16*>(B);
  // U = (B^T W0)^T [in, r] in one pass over W0, K_b = B^T B, then the column norm and c = m / n
  CK(colreduce(cr_desc(out, in, r, W0, B, r, w.PU, w.splitsW, w.err), st));
  CK(sum_splits<float>(w.PU, w.splitsW, in * r, U_save, nullptr, st));
  CK(gram_bf16(B, B, out, r, w.Kb, w.Gw, w.err, st));
  CK(dora_colnorm(in, r, c0, U_save, Ab, w.Kb, static_cast<const bf16*>(m), s, eps, n_save, w.c, w.Ac, st));
  if (M == 0) return LORA_OK;
  if (s != 0.f || Z_save) {
    // one pass over X: Z = X (A diag(c))^T, s Z, and the scaled copy X diag(c) for the GEMM
    RowProjDesc d = rp_desc(M, in, r, X, w.Ac, false, w.err);
    d.out_a = static_cast<bf16*>(Z_save);
    if (s != 0.f) {
      d.out_b = w.Zs;
      d.scale_b = s;
      d.s_scale = w.c;
      d.s_out = w.Xc;
    }
    CK(rowproj(d, st));
  }
  if (s == 0.f)  // strength 0: frozen base X W0^T + bias
    CK(tc_gemm(fwd_desc(M, out, in, X, W0, nullptr, B, r, Y, static_cast<const bf16*>(bias), nullptr, w.err), st));
  else
    CK(tc_gemm(fwd_desc(M, out, in, w.Xc, W0, w.Zs, B, r, Y, static_cast<const bf16*>(bias), nullptr, w.err), st));
  return LORA_OK;
}

lora_status dora_cols_bwd(const lora_shape* sh, const void* X, const void* W0, const void* A, const void* B,
                          const void* m, const void* Z_saved, const float* n_saved, const float* U_saved,
                          const void* dY, float s, float eps, void* dX, void* dA, void* dB, void* dm, void* dbias,
                          void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_shape(sh);
  if (e != LORA_OK) return e;
  if (sh->dtype != LORA_BF16) return LORA_ERR_UNSUPPORTED;
  REQM(sh->M, X); REQ(W0); REQ(A); REQ(B); REQ(m); REQ(n_saved); REQ(U_saved); REQM(sh->M, dY);
  REQ(dA); REQ(dB); REQ(dm);
  ALN(X); ALN(W0); ALN(A); ALN(B); ALN(m); ALN(Z_saved); ALN(n_saved); ALN(U_saved); ALN(dY);
  ALN(dX); ALN(dA); ALN(dB); ALN(dm); ALN(dbias);
  if (!isfinite(s) || !isfinite(eps) || eps < 0.f) return LORA_ERR_INVALID_ARG;
  DoraColsBwdWs w;
  if ((e = check_ws(ws, ws_bytes, plan_dora_cols_bwd(*sh, nullptr, &w))) != LORA_OK) return e;
  plan_dora_cols_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, in = sh->d_in, out = sh->d_out;
  const int r = (int)sh->r;
  const bf16* Ab = static_cast<const bf16*>(A);
  const bf16* Bb = static_cast<const bf16*>(B);
  const bf16* mb = static_cast<const bf16*>(m);
  if (M == 0 || s == 0.f) {
    CK(cudaMemsetAsync(dA, 0, (size_t)r * in * 2, st));
    CK(cudaMemsetAsync(dB, 0, (size_t)out * r * 2, st));
    CK(cudaMemsetAsync(dm, 0, (size_t)in * 2, st));
    if (M == 0) {
      if (dbias) CK(cudaMemsetAsync(dbias, 0, (size_t)out * 2, st));
      return LORA_OK;
    }
    // strength 0: frozen base, dX = dY W0, dbias = colsum(dY)
    if (dX) CK(tc_gemm(dx_desc(M, in, out, dY, W0, nullptr, A, r, dX, nullptr, w.err), st));
    if (dbias) {
      ColReduceDesc d = cr_desc(M, out, 8, dY, dY, out, w.PB, w.splitsB, w.err);
      d.colsum = w.csump;
      CK(colreduce(d, st));
      CK(sum_splits<bf16>(w.csump, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
    }
    return LORA_OK;
  }
  CK(dora_c<bf16>(in, mb, n_saved, w.c, st));
  const void* Z = Z_saved;
  if (!Z) {
    CK(scale_cols_bf16(Ab, r, in, w.c, w.Ac, st));
    RowProjDesc d = rp_desc(M, in, r, X, w.Ac, false, w.err);
    d.out_a = w.Zrec;
    CK(rowproj(d, st));
    Z = w.Zrec;
  }
  // s G = s dY B, the dB partials dY^T Z and the column sums of dY: one rowcol pass over dY
  CK(dy_side(w.rc, M, out, r, dY, out, B, Z, r, w.PB, w.splitsB, w.Gp, s, w.Gs, r, w.err, st,
             dbias ? w.csump : nullptr));
  // dX = (dY W0 + G A) diag(c): the column scale is the GEMM epilogue's
  bf16* dXo = dX ? static_cast<bf16*>(dX) : w.dXt;
  {
    TcGemmDesc d = dx_desc(M, in, out, dY, W0, w.Gs, A, r, dXo, nullptr, w.err);
    d.col_scale = w.c;
    CK(tc_gemm(d, st));
  }
  {  // (X^T G) partials and colsum(X o dX) = c o colsum(X o dXt), one pass over X and dX
    ColReduceDesc d = cr_desc(M, in, r, X, w.Gs, r, w.PA, w.splitsA, w.err);
    d.Y = dXo;
    d.ldy = in;
    d.coldot = w.dotp;
    CK(colreduce(d, st));
  }
  // dc = dot / c (no bias term), dm = dc / n, g = -m dc / (2 n^3)
  CK(dora_dc<bf16>(in, w.dotp, nullptr, w.splitsA, nullptr, w.c, n_saved, mb, eps, w.g, static_cast<bf16*>(dm), nullptr,
                   st));
  CK(gram_bf16(B, B, out, r, w.Kb, w.Gw, w.err, st));
  CK(gram_rows_weighted(Ab, r, in, w.g, w.Kga, st));
  CK(scale_cols_bf16(Ab, r, in, w.g, w.Ag, st));
  {  // W0 diag(g) A^T (fp32), one pass over W0
    RowProjDesc d = rp_desc(out, in, r, W0, w.Ag, false, w.err);
    d.out_f = w.Vg;
    CK(rowproj(d, st));
  }
  Partial pa{w.PA, w.splitsA, r, 0}, pb{w.PB, w.splitsB, r, 0};
  CK(finalize_dA_cols(r, in, pa, w.c, w.g, U_saved, w.Kb, Ab, s, static_cast<bf16*>(dA), st));
  CK(finalize_dB<bf16>(out, r, pb, s, nullptr, nullptr, w.Vg, Bb, w.Kga, s, false, static_cast<bf16*>(dB), st));
  if (dbias) CK(sum_splits<bf16>(w.csump, w.splitsB, out, nullptr, static_cast<bf16*>(dbias), st));
  return LORA_OK;
}

// ------------------------------------------------------------------ SwiGLU MLP
static lora_status check_proj(const lora_proj* p) {
  if (!p || !p->W || !p->A || !p->B) return LORA_ERR_INVALID_ARG;
  if (!al16(p->W) || !al16(p->A) || !al16(p->B)) return LORA_ERR_MISALIGNED;
  if (!isfinite(p->s)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status lora_mlp_swiglu_fwd(const lora_mlp_shape* sh, const void* X, const lora_proj* gate, const lora_proj* up,
                                const lora_proj* down, void* Y, void* e_save, void* u_save, void* h_save,
                                void* Zgu_save, void* Zd_save, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_mlp_shape(sh);
  if (e != LORA_OK) return e;
  if ((e = check_proj(gate)) != LORA_OK || (e = check_proj(up)) != LORA_OK || (e = check_proj(down)) != LORA_OK)
    return e;
  REQM(sh->M, X); REQM(sh->M, Y); REQM(sh->M, e_save); REQM(sh->M, u_save); REQM(sh->M, h_save);
  REQM(sh->M, Zgu_save); REQM(sh->M, Zd_save);
  ALN(X); ALN(Y); ALN(e_save); ALN(u_save); ALN(h_save); ALN(Zgu_save); ALN(Zd_save);
  MlpFwdWs w;
  const size_t need = plan_mlp_fwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_mlp_fwd(*sh, static_cast<char*>(ws), &w);
  if (sh->M == 0) return LORA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, H = sh->H, I = sh->I;
  const int rg = (int)sh->r_g, ru = (int)sh->r_u, rd = (int)sh->r_d, rgu = rg + ru;
  CK(concat_rows_bf16(static_cast<const bf16*>(gate->A), rg, static_cast<const bf16*>(up->A), ru, H, w.Agu, st));
  {  // [Zg | Zu] = X [Ag ; Au]^T (one pass per 64 columns), saved unscaled and scaled per half
    RowProjDesc d = rp_desc(M, H, rgu, X, w.Agu, false, w.err);
    d.out_a = static_cast<bf16*>(Zgu_save);
    d.out_b = w.Zgus;
    d.scale_b = gate->s;
    d.split_col = rg;
    d.scale_b_hi = up->s;
    CK(rowproj(d, st));
  }
  {  // e, u, h = gate/up GEMM with both adapters, gated epilogue
    TcGemmDesc d;
    d.mode = TC_SWIGLU_FWD;
    d.act = sh->act;
    d.M = (int)M;
    d.N = (int)I;
    d.K0 = (int)H;
    d.A0 = X;
    d.lda0 = H;
    d.B0 = gate->W;
    d.B0b = up->W;
    d.ldb0 = H;
    d.has_tail = true;   // tail K = [Zg | Zu] against [Bg | 0] (gate half) and [0 | Bu] (up half)
    d.A1 = w.Zgus;
    d.lda1 = rgu;
    d.K1 = rgu;
    d.K1_a = rgu;
    d.B1 = gate->B;
    d.ldb1 = rg;
    d.K1_b = rg;
    d.B1b = up->B;
    d.ldb1b = ru;
    d.K1_bb = ru;
    d.b1b_x = -rg;       // the up half's columns start after the gate rank (left of them: zero fill)
    d.out[0] = e_save;
    d.out[1] = u_save;
    d.out[2] = h_save;
    d.ldo = I;
    d.err = w.err;
    d.timeout_ns = wait_timeout_ns();
    CK(tc_gemm(d, st));
  }
  {  // Zd = h Ad^T
    RowProjDesc d = rp_desc(M, I, rd, h_save, down->A, false, w.err);
    d.out_a = static_cast<bf16*>(Zd_save);
    d.out_b = w.Zds;
    d.scale_b = down->s;
    CK(rowproj(d, st));
  }
  CK(tc_gemm(fwd_desc(M, H, I, h_save, down->W, w.Zds, down->B, rd, Y, nullptr, nullptr, w.err), st));
  return LORA_OK;
}

lora_status lora_mlp_swiglu_bwd(const lora_mlp_shape* sh, const void* X, const lora_proj* gate, const lora_proj* up,
                                const lora_proj* down, const void* e_saved, const void* u_saved, const void* h_saved,
                                const void* Zgu_saved, const void* Zd_saved, const void* dY, void* dX, void* dAg,
                                void* dBg, void* dAu, void* dBu, void* dAd, void* dBd, void* ws, size_t ws_bytes,
                                void* stream) {
  lora_status e = check_mlp_shape(sh);
  if (e != LORA_OK) return e;
  if ((e = check_proj(gate)) != LORA_OK || (e = check_proj(up)) != LORA_OK || (e = check_proj(down)) != LORA_OK)
    return e;
  REQM(sh->M, X); REQM(sh->M, e_saved); REQM(sh->M, u_saved); REQM(sh->M, h_saved); REQM(sh->M, Zgu_saved);
  REQM(sh->M, Zd_saved); REQM(sh->M, dY);
  REQ(dAg); REQ(dBg); REQ(dAu); REQ(dBu); REQ(dAd); REQ(dBd);
  ALN(X); ALN(e_saved); ALN(u_saved); ALN(h_saved); ALN(Zgu_saved); ALN(Zd_saved); ALN(dY); ALN(dX);
  ALN(dAg); ALN(dBg); ALN(dAu); ALN(dBu); ALN(dAd); ALN(dBd);
  MlpBwdWs w;
  const size_t need = plan_mlp_bwd(*sh, nullptr, &w);
  if ((e = check_ws(ws, ws_bytes, need)) != LORA_OK) return e;
  plan_mlp_bwd(*sh, static_cast<char*>(ws), &w);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t M = sh->M, H = sh->H, I = sh->I, Ip = mlp_ipad(*sh);
  const int rg = (int)sh->r_g, ru = (int)sh->r_u, rd = (int)sh->r_d, rgu = rg + ru;
  if (M == 0) {
    CK(cudaMemsetAsync(dAg, 0, (size_t)rg * H * 2, st));
    CK(cudaMemsetAsync(dAu, 0, (size_t)ru * H * 2, st));
    CK(cudaMemsetAsync(dBg, 0, (size_t)I * rg * 2, st));
    CK(cudaMemsetAsync(dBu, 0, (size_t)I * ru * 2, st));
    CK(cudaMemsetAsync(dAd, 0, (size_t)rd * I * 2, st));
    CK(cudaMemsetAsync(dBd, 0, (size_t)H * rd * 2, st));
    return LORA_OK;
  }
  const bf16* Zgu = static_cast<const bf16*>(Zgu_saved);
  // down projection: dBd partials (dY^T Zd) and sd*Gd = sd dY Bd
  CK(dy_side(w.rcd, M, H, rd, dY, H, down->B, Zd_saved, rd, w.PBd, w.sBd, w.Gpd, down->s, w.Gds, rd, w.err, st));
  if (Ip != I) CK(cudaMemsetAsync(w.dedu, 0, (size_t)M * 2 * Ip * 2, st));
  {  // dh = dY Wd + (sd Gd) Ad, gated backward in the epilogue -> de, du
    TcGemmDesc d;
    d.mode = TC_SWIGLU_BWD;
    d.act = sh->act;
    d.M = (int)M;
    d.N = (int)I;
    d.K0 = (int)H;
    d.A0 = dY;
    d.lda0 = H;
    d.B0 = down->W;
    d.ldb0 = I;
    d.b0_mn = true;
    d.b0_rows = (int)H;
    d.has_tail = true;
    d.b1_mn = true;
    d.A1 = w.Gds;
    d.lda1 = rd;
    d.K1 = rd;
    d.K1_a = rd;
    d.B1 = down->A;
    d.ldb1 = I;
    d.out[0] = w.dedu;
    d.out[1] = w.dedu + Ip;
    d.ldo = 2 * Ip;
    d.e_in = static_cast<const bf16*>(e_saved);
    d.u_in = static_cast<const bf16*>(u_saved);
    d.ld_eu = I;
    d.err = w.err;
    d.timeout_ns = wait_timeout_ns();
    CK(tc_gemm(d, st));
  }
  CK(colreduce(cr_desc(M, I, rd, h_saved, w.Gds, rd, w.PAd, w.sAd, w.err), st));     // h^T (sd Gd)
  // gate and up: the dBg / dBu partials (de^T Zg, du^T Zu) and [sg Gg | su Gu] = [sg de Bg | su du Bu]
  CK(dy_side(w.rcg, M, I, rg, w.dedu, 2 * Ip, gate->B, Zgu, rgu, w.PBg, w.sBg, w.Gpg, gate->s, w.Ggus, rgu, w.err,
             st));
  CK(dy_side(w.rcu, M, I, ru, w.dedu + Ip, 2 * Ip, up->B, Zgu + rg, rgu, w.PBu, w.sBu, w.Gpu, up->s, w.Ggus + rg,
             rgu, w.err, st));
  CK(concat_rows_bf16(static_cast<const bf16*>(gate->A), rg, static_cast<const bf16*>(up->A), ru, H, w.Agu, st));
  if (dX) {  // dX = [de | du] [Wg ; Wu] + [sg Gg | su Gu] [Ag ; Au]
    TcGemmDesc d;
    d.mode = TC_BWD_DX;
    d.M = (int)M;
    d.N = (int)H;
    d.K0 = (int)(2 * Ip);
    d.A0 = w.dedu;
    d.lda0 = 2 * Ip;
    d.B0 = gate->W;
    d.B0b = up->W;
    d.ldb0 = H;
    d.b0_mn = true;
    d.b0_rows = (int)I;
    d.b0b_rows = (int)I;
    d.k0_split = (int)Ip;
    d.has_tail = true;
    d.b1_mn = true;
    d.A1 = w.Ggus;
    d.lda1 = rgu;
    d.K1 = rgu;
    d.K1_a = rgu;
    d.B1 = w.Agu;
    d.ldb1 = H;
    d.out[0] = dX;
    d.ldo = H;
    d.err = w.err;
    d.timeout_ns = wait_timeout_ns();
    CK(tc_gemm(d, st));
  }
  // X^T [sg Gg | su Gu] (one pass over X per 64 columns)
  CK(colreduce(cr_desc(M, H, rgu, X, w.Ggus, rgu, w.PAgu, w.sAgu, w.err), st));
  const FinJob fin[6] = {fin_dA(rg, H, Partial{w.PAgu, w.sAgu, rgu, 0}, 1.f, nullptr, dAg),
                         fin_dA(ru, H, Partial{w.PAgu, w.sAgu, rgu, rg}, 1.f, nullptr, dAu),
                         fin_dA(rd, I, Partial{w.PAd, w.sAd, rd, 0}, 1.f, nullptr, dAd),
                         fin_dB(H, rd, Partial{w.PBd, w.sBd, rd, 0}, down->s, nullptr, dBd),
                         fin_dB(I, rg, Partial{w.PBg, w.sBg, rg, 0}, gate->s, nullptr, dBg),
                         fin_dB(I, ru, Partial{w.PBu, w.sBu, ru, 0}, up->s, nullptr, dBu)};
  CK(finalize_batch(fin, 6, st));
  return LORA_OK;
}

// ------------------------------------------------------------------ W8A8
lora_status w8a8_quantize_rows(int64_t rows, int64_t cols, const void* X, int8_t* Xq, float* sx, const void* A,
                               int64_t r, void* Z, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 8) return rows < 0 || cols <= 0 ? LORA_ERR_INVALID_ARG : LORA_ERR_UNSUPPORTED;
  REQM(rows, X); REQM(rows, Xq); REQM(rows, sx);
  ALN(X); ALN(Xq); ALN(A); ALN(Z);
  if ((A == nullptr) != (Z == nullptr)) return LORA_ERR_INVALID_ARG;
  if (A && (r < 8 || r > 128 || r % 8)) return LORA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  if (rows == 0) return LORA_OK;
  CK(quantize_rows_bf16(static_cast<const bf16*>(X), rows, cols, Xq, sx, st));
  if (A) {
    RowProjDesc d = rp_desc(rows, cols, (int)r, X, A, false, nullptr);  // no workspace: no error word
    d.out_a = static_cast<bf16*>(Z);
    CK(rowproj(d, st));
  }
  return LORA_OK;
}

constexpr int64_t kW8MaxR = 128;   // largest rank of the low-rank term
// K-steps of 64 per exactly summed chunk of the int8 product: every fp32 partial sum of a chunk is
// an integer of magnitude at most 127 * 127 * 1024 < 2^24, hence exact
constexpr int kW8ChunkSteps = 16;

size_t w8a8_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out) {
  if (M < 0 || d_in <= 0 || d_out <= 0) return 0;
  return kErrBytes + al256((size_t)M * d_in * 2) + al256((size_t)d_out * d_in * 2);
}

}  // extern "C"

namespace {
// The int8 product on the bf16 tensor cores and its epilogue, on operands already laid out for it:
// Xb [M, d_in] and Wb [d_out, d_in] the activation and weight codes as bf16 (exact: |code| <= 127).
// The K range goes in chunks of kW8ChunkSteps K-steps, each summed exactly in its own TMEM
// accumulator and added as int32; the rank-r term Z B^T is one more accumulator.
lora_status w8a8_fwd_core(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const bf16* Xb, const float* sx,
                          const bf16* Wb, const float* sw, const void* Z, const void* B, float s, const void* bias,
                          void* Y, int32_t* acc_out, uint32_t* err, cudaStream_t st) {
  TcGemmDesc d;
  d.mode = TC_W8A8K;
  d.M = (int)M;
  d.N = (int)d_out;
  d.K0 = (int)d_in;
  d.A0 = Xb;
  d.lda0 = d_in;
  d.B0 = Wb;
  d.ldb0 = d_in;
  d.out[0] = Y;
  d.ldo = d_out;
  d.bias = static_cast<const bf16*>(bias);
  d.sx = sx;
  d.sw = sw;
  d.ls = s;
  d.acc_out = acc_out;
  d.kc_steps = kW8ChunkSteps;
  d.err = err;
  d.timeout_ns = wait_timeout_ns();
  if (Z) {  // rank-r term Z B^T as a tail K-step into its own accumulator
    d.has_tail = true;
    d.A1 = Z;
    d.lda1 = r;
    d.K1 = (int)r;
    d.K1_a = (int)r;
    d.B1 = B;
    d.ldb1 = r;
    d.K1_b = (int)r;
  }
  CK(tc_gemm(d, st));
  return LORA_OK;
}

lora_status check_w8a8(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const void* Z, const void* B, float s,
                       const void* Y, const int32_t* acc_out, const float* sx, const float* sw) {
  if (M < 0 || d_in <= 0 || d_out <= 0) return LORA_ERR_INVALID_ARG;
  if (d_in % 32 || d_out % 8) return LORA_ERR_UNSUPPORTED;
  if (Y == nullptr && acc_out == nullptr) return LORA_ERR_INVALID_ARG;
  if (Y && (!sx || !sw)) return LORA_ERR_INVALID_ARG;
  if ((Z == nullptr) != (B == nullptr)) return LORA_ERR_INVALID_ARG;
  if (Z && (r < 8 || r > kW8MaxR || r % 8)) return LORA_ERR_UNSUPPORTED;
  if (!isfinite(s)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}
}  // namespace

extern "C" {

lora_status w8a8_lora_fwd(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const int8_t* Xq, const float* sx,
                          const int8_t* Wq, const float* sw, const void* Z, const void* B, float s, const void* bias,
                          void* Y, int32_t* acc_out, void* ws, size_t ws_bytes, void* stream) {
  lora_status e = check_w8a8(M, d_in, d_out, r, Z, B, s, Y, acc_out, sx, sw);
  if (e != LORA_OK) return e;
  REQM(M, Xq); REQ(Wq);
  ALN(Xq); ALN(sx); ALN(Wq); ALN(sw); ALN(Z); ALN(B); ALN(bias); ALN(Y); ALN(acc_out);
  if ((e = check_ws(ws, ws_bytes, w8a8_workspace_bytes(M, d_in, d_out))) != LORA_OK) return e;
  if (M == 0) return LORA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (getenv("LORA_GB300_W8A8_IMMA")) {   // the integer warp-MMA product (s8 x s8 -> s32)
    CK(w8a8_gemm(M, d_in, d_out, Z ? (int)r : 0, Xq, sx, Wq, sw, static_cast<const bf16*>(Z),
                 static_cast<const bf16*>(B), s, static_cast<const bf16*>(bias), static_cast<bf16*>(Y), acc_out, st));
    return LORA_OK;
  }
  Carve c{static_cast<char*>(ws)};
  uint32_t* err = c.take<uint32_t>(kErrBytes / 4);
  bf16* Xb = c.take<bf16>((size_t)M * d_in);
  bf16* Wb = c.take<bf16>((size_t)d_out * d_in);
  CK(i8_to_bf16(Xq, M * d_in, Xb, st));
  CK(i8_to_bf16(Wq, d_out * d_in, Wb, st));
  return w8a8_fwd_core(M, d_in, d_out, r, Xb, sx, Wb, sw, Z, B, s, bias, Y, acc_out, err, st);
}

lora_status w8a8_quantize_rows_bf16(int64_t rows, int64_t cols, const void* X, void* Xcodes, float* sx,
                                    const void* A, int64_t r, void* Z, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 8) return rows < 0 || cols <= 0 ? LORA_ERR_INVALID_ARG : LORA_ERR_UNSUPPORTED;
  REQM(rows, X); REQM(rows, Xcodes); REQM(rows, sx);
  ALN(X); ALN(Xcodes); ALN(A); ALN(Z);
  if ((A == nullptr) != (Z == nullptr)) return LORA_ERR_INVALID_ARG;
  if (A && (r < 8 || r > kW8MaxR || r % 8)) return LORA_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  if (rows == 0) return LORA_OK;
  CK(quantize_rows_bf16(static_cast<const bf16*>(X), rows, cols, nullptr, sx, st, static_cast<bf16*>(Xcodes)));
  if (A) {
    RowProjDesc d = rp_desc(rows, cols, (int)r, X, A, false, nullptr);  // no workspace: no error word
    d.out_a = static_cast<bf16*>(Z);
    CK(rowproj(d, st));
  }
  return LORA_OK;
}

lora_status w8a8_prepack_weight(int64_t d_out, int64_t d_in, const int8_t* Wq, const float* sw, void* Wb, void* Wd,
                                void* stream) {
  if (d_out <= 0 || d_in <= 0) return LORA_ERR_INVALID_ARG;
  if (d_in % 32 || d_out % 8) return LORA_ERR_UNSUPPORTED;
  REQ(Wq);
  if (Wd && !sw) return LORA_ERR_INVALID_ARG;
  ALN(Wq); ALN(sw); ALN(Wb); ALN(Wd);
  cudaStream_t st = (cudaStream_t)stream;
  if (Wb) CK(i8_to_bf16(Wq, d_out * d_in, static_cast<bf16*>(Wb), st));
  if (Wd) CK(i8_dequant_rows_bf16(Wq, sw, d_out, d_in, static_cast<bf16*>(Wd), st));
  return LORA_OK;
}

size_t w8a8_packed_workspace_bytes(int64_t M, int64_t d_out) {
  if (M < 0 || d_out <= 0) return 0;
  return kErrBytes;
}

lora_status w8a8_lora_fwd_packed(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const void* Xcodes,
                                 const float* sx, const void* Wb, const float* sw, const void* Z, const void* B,
                                 float s, const void* bias, void* Y, int32_t* acc_out, void* ws, size_t ws_bytes,
                                 void* stream) {
  lora_status e = check_w8a8(M, d_in, d_out, r, Z, B, s, Y, acc_out, sx, sw);
  if (e != LORA_OK) return e;
  REQM(M, Xcodes); REQ(Wb);
  ALN(Xcodes); ALN(sx); ALN(Wb); ALN(sw); ALN(Z); ALN(B); ALN(bias); ALN(Y); ALN(acc_out);
  if ((e = check_ws(ws, ws_bytes, w8a8_packed_workspace_bytes(M, d_out))) != LORA_OK) return e;
  if (M == 0) return LORA_OK;
  Carve c{static_cast<char*>(ws)};
  uint32_t* err = c.take<uint32_t>(kErrBytes / 4);
  return w8a8_fwd_core(M, d_in, d_out, r, static_cast<const bf16*>(Xcodes), sx, static_cast<const bf16*>(Wb), sw, Z,
                       B, s, bias, Y, acc_out, err, (cudaStream_t)stream);
}

size_t w8a8_bwd_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int64_t r) {
  lora_shape sh{M, d_in, d_out, r, LORA_BF16};
  const size_t lin = lora_workspace_bytes(LORA_OP_LINEAR_BWD, &sh);
  if (lin == 0) return 0;
  return lin + al256((size_t)d_out * d_in * 2);
}

lora_status w8a8_lora_bwd(int64_t M, int64_t d_in, int64_t d_out, int64_t r, const void* X, const int8_t* Wq,
                          const float* sw, const void* A, const void* B, const void* Z_saved, const void* dY,
                          float s, void* dX, void* dA, void* dB, void* dbias, void* ws, size_t ws_bytes,
                          void* stream) {
  lora_shape sh{M, d_in, d_out, r, LORA_BF16};
  lora_status e = check_shape(&sh);
  if (e != LORA_OK) return e;
  if (d_in % 16) return LORA_ERR_UNSUPPORTED;
  REQ(Wq); REQ(sw);
  ALN(Wq); ALN(sw);
  const size_t lin = lora_workspace_bytes(LORA_OP_LINEAR_BWD, &sh);
  if ((e = check_ws(ws, ws_bytes, w8a8_bwd_workspace_bytes(M, d_in, d_out, r))) != LORA_OK) return e;
  // the frozen int8 weight in real units, then the bf16 LoRA backward over it
  bf16* Wd = reinterpret_cast<bf16*>(static_cast<char*>(ws) + lin);
  if (M > 0) CK(i8_dequant_rows_bf16(Wq, sw, d_out, d_in, Wd, (cudaStream_t)stream));
  return lora_linear_bwd(&sh, X, Wd, A, B, Z_saved, dY, s, dX, dA, dB, dbias, ws, lin, stream);
}

}  // extern "C"

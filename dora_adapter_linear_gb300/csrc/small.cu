// Small per-row / per-column kernels of the DoRA norm and the gradient assembly.  They
// touch vectors of length d_out or [d_out, r] / [r, d_in] matrices (kilobytes to a few MB),
// so they are latency-bound one-pass kernels; templated on the storage type (fp32 / bf16).
#include "common.cuh"
#include "internal.h"

namespace lg {

template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i) {
  return to_f<T>(p[i]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int NT>
__device__ __forceinline__ float block_sum(float v) {
  __shared__ float red[NT / 32];
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = l < NT / 32 ? red[l] : 0.f;
    t = warp_sum(t);
  }
  return t;  // valid in thread 0
}

// ------------------------------------------------------------------ rowsum(W^2), one warp per row
template <typename T>
__global__ void rownorm2_kernel(const T* W, int64_t rows, int64_t cols, float* r0) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* w = W + row * cols;
  float acc = 0.f;
  constexpr int V = 16 / sizeof(T);
  for (int64_t k = (int64_t)lane * V; k < cols; k += 32 * V) {
    const uint4 raw = *reinterpret_cast<const uint4*>(w + k);
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const float f = to_f<T>(e[i]);
      acc = fmaf(f, f, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) r0[row] = acc;
}

template <typename T>
cudaError_t rownorm2(const T* W, int64_t rows, int64_t cols, float* r0, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(rownorm2_kernel<T>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, W, rows, cols, r0);
}

// ------------------------------------------------------------------ K = A A^T, one block per (i, j)
template <typename T>
__global__ void gram_rows_kernel(const T* A, int r, int64_t cols, float* K) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int i = blockIdx.x / r, j = blockIdx.x % r;
  if (j < i) return;
  float acc = 0.f;
  for (int64_t k = threadIdx.x; k < cols; k += blockDim.x) acc = fmaf(ldf(A, i * cols + k), ldf(A, j * cols + k), acc);
  acc = block_sum<256>(acc);
  if (threadIdx.x == 0) {
    K[i * r + j] = acc;
    K[j * r + i] = acc;
  }
}
template <typename T>
cudaError_t gram_rows(const T* A, int r, int64_t cols, float* K, cudaStream_t st) {
  return launch_pdl(gram_rows_kernel<T>, dim3(r * r), dim3(256), 0, st, A, r, cols, K);
}

// ------------------------------------------------------------------ Kg = B^T diag(g) B
// Pass 1: block c takes a contiguous chunk of the rows of B, stages 32 rows at a time in shared
// memory and accumulates its share of every entry (i, j); pass 2 sums the chunk partials in a
// fixed order (deterministic, no atomics).
constexpr int kGramChunks = 64;
constexpr int kGramMaxR = 128;
template <typename T>
__global__ void __launch_bounds__(256) gram_partial_kernel(const T* B, int64_t out, int r, const float* g,
                                                           int64_t rows_per, float* part) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  constexpr int NQ = kGramMaxR * kGramMaxR / 256;   // entries (i, j) per thread
  __shared__ float tile[32][kGramMaxR + 1];
  __shared__ float gw[32];
  const int c = blockIdx.x;
  const int64_t o0 = (int64_t)c * rows_per;
  const int64_t o1 = min(out, o0 + rows_per);
  const int rr2 = r * r;
  float acc[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) acc[q] = 0.f;
  for (int64_t ob = o0; ob < o1; ob += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * r; e += 256) {
      const int rr = e / r, j = e - (e / r) * r;
      const int64_t o = ob + rr;
      tile[rr][j] = o < o1 ? ldf(B, o * r + j) : 0.f;
    }
    if (threadIdx.x < 32) {
      const int64_t o = ob + threadIdx.x;
      gw[threadIdx.x] = o < o1 ? (g ? g[o] : 1.f) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int e = threadIdx.x + 256 * q;
      if (e < rr2) {
        const int i = e / r, j = e - (e / r) * r;
        float t = acc[q];
        for (int rr = 0; rr < 32; ++rr) t = fmaf(gw[rr] * tile[rr][i], tile[rr][j], t);
        acc[q] = t;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = threadIdx.x + 256 * q;
    if (e < rr2) part[(int64_t)c * rr2 + e] = acc[q];
  }
}
size_t gram_work_floats(int r) { return (size_t)kGramChunks * r * r; }
template <typename T>
cudaError_t gram_weighted(const T* B, int64_t out, int r, const float* g, float* Kg, float* work, cudaStream_t st) {
  if (r <= 0 || r > kGramMaxR || out <= 0) return cudaErrorInvalidValue;
  int nch = (int)((out + 31) / 32);
  if (nch > kGramChunks) nch = kGramChunks;
  const int64_t rows_per = (out + nch - 1) / nch;
  cudaError_t e = launch_pdl(gram_partial_kernel<T>, dim3(nch), dim3(256), 0, st, B, out, r, g, rows_per, work);
  if (e != cudaSuccess) return e;
  return sum_splits<float>(work, nch, (int64_t)r * r, Kg, nullptr, st);
}

// ------------------------------------------------------------------ closed-form DoRA norm, one warp per row
// Lane j holds B[o, j + 32 h] (h < 4, r <= 128); (B Kr)[o, j] is formed with the row broadcast
// lane by lane; Kr (r x r) sits in shared memory.
constexpr int kNormMaxR = 128;
template <typename T>
__global__ void dora_norm_kernel(int64_t out, int r, const float* r0, const float* V, const T* B, const float* Kr,
                                 const T* m, float s, float eps, float* n_out, float* c) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  extern __shared__ float sKr[];
  for (int i = threadIdx.x; i < r * r; i += blockDim.x) sKr[i] = Kr[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t o = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (o >= out) return;
  float b[4], t1 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int j = lane + 32 * h;
    b[h] = j < r ? ldf(B, o * r + j) : 0.f;
    if (j < r) t1 = fmaf(V[o * r + j], b[h], t1);
  }
  float k[4] = {0.f, 0.f, 0.f, 0.f};
  for (int l = 0; l < r; ++l) {
    const float bl = __shfl_sync(0xffffffffu, b[l >> 5], l & 31);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (lane + 32 * h < r) k[h] = fmaf(bl, sKr[l * r + lane + 32 * h], k[h]);
  }
  float t2 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) t2 = fmaf(k[h], b[h], t2);
  t1 = warp_sum(t1);
  t2 = warp_sum(t2);
  if (lane == 0) {
    const float q = r0[o] + 2.f * s * t1 + s * s * t2;
    const float n = fmaxf(sqrtf(fmaxf(q, 0.f)), eps);
    n_out[o] = n;
    if (c) c[o] = ldf(m, o) / n;
  }
}
// dynamic shared memory for an r x r fp32 matrix (64 KB at r = 128: above the default limit)
template <typename K>
static cudaError_t allow_rr_smem(K kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(kNormMaxR * kNormMaxR * sizeof(float)));
}
template <typename T>
cudaError_t dora_norm(int64_t out, int r, const float* r0, const float* V, const T* B, const float* Kr, const T* m,
                      float s, float eps, float* n_out, float* c, cudaStream_t st) {
  if (out <= 0) return cudaSuccess;
  if (r > kNormMaxR) return cudaErrorInvalidValue;
  const cudaError_t ea = allow_rr_smem(dora_norm_kernel<T>);
  if (ea != cudaSuccess) return ea;
  return launch_pdl(dora_norm_kernel<T>, dim3((unsigned)((out + 7) / 8)), dim3(256), r * r * sizeof(float), st,
                    out, r, r0, V, B, Kr, m, s, eps, n_out, c);
}

// ------------------------------------------------------------------ c = m / n
template <typename T>
__global__ void dora_c_kernel(int64_t out, int64_t padded, const T* m, const float* n, float* c) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o < out) c[o] = ldf(m, o) / n[o];
  else if (o < padded) c[o] = 0.f;
}
template <typename T>
cudaError_t dora_c(int64_t out, const T* m, const float* n, float* c, cudaStream_t st, int64_t padded) {
  if (out <= 0) return cudaSuccess;
  if (padded < out) padded = out;
  return launch_pdl(dora_c_kernel<T>, dim3((unsigned)((padded + 255) / 256)), dim3(256), 0, st, out, padded, m, n, c);
}

// ------------------------------------------------------------------ sum of split partials
template <typename T>
__global__ void sum_splits_kernel(const float* src, int splits, int64_t n, float* dst_f, T* dst_t) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  float a = 0.f;
  for (int s = 0; s < splits; ++s) a += src[(int64_t)s * n + k];
  if (dst_f) dst_f[k] = a;
  if (dst_t) dst_t[k] = from_f<T>(a);
}
template <typename T>
cudaError_t sum_splits(const float* src, int splits, int64_t n, float* dst_f, T* dst_t, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(sum_splits_kernel<T>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    src, splits, n, dst_f, dst_t);
}

// ------------------------------------------------------------------ DoRA dc -> dm, g, dbias
// dot and csum are [splits, out] partial sums (of the row splits of the column pass), added here.
template <typename T>
__global__ void dora_dc_kernel(int64_t out, const float* dot, const float* csum, int splits, const T* bias,
                               const float* c, const float* n, const T* m, float eps, float* g, T* dm, T* dbias) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= out) return;
  float dt = 0.f, cs = 0.f;
  for (int sp = 0; sp < splits; ++sp) dt += dot[(int64_t)sp * out + o];
  if (bias || dbias)
    for (int sp = 0; sp < splits; ++sp) cs += csum[(int64_t)sp * out + o];
  const float b = bias ? ldf(bias, o) : 0.f;
  // P = (Y - bias) / c  =>  sum dY * P = (sum dY*Y - bias * sum dY) / c
  const float dc = (dt - b * cs) / c[o];
  const float nn = n[o];
  dm[o] = from_f<T>(dc / nn);
  g[o] = nn > eps ? -ldf(m, o) * dc / (2.f * nn * nn * nn) : 0.f;
  if (dbias) dbias[o] = from_f<T>(cs);
}
template <typename T>
cudaError_t dora_dc(int64_t out, const float* dot, const float* csum, int splits, const T* bias, const float* c,
                    const float* n, const T* m, float eps, float* g, T* dm, T* dbias, cudaStream_t st) {
  if (out <= 0) return cudaSuccess;
  if ((bias || dbias) && !csum) return cudaErrorInvalidValue;
  return launch_pdl(dora_dc_kernel<T>, dim3((unsigned)((out + 255) / 256)), dim3(256), 0, st,
                    out, dot, csum, splits, bias, c, n, m, eps, g, dm, dbias);
}

// ------------------------------------------------------------------ out = f * scale[o] * B[o, :]
template <typename T>
__global__ void scale_rows_kernel(const T* B, int64_t rows, int r, const float* scale, float f, T* out) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * r) return;
  const int64_t o = i / r;
  const float sc = scale ? scale[o] : 1.f;
  out[i] = from_f<T>(f * sc * ldf(B, i));
}
template <typename T>
cudaError_t scale_rows(const T* B, int64_t rows, int r, const float* scale, float f, T* out, cudaStream_t st) {
  const int64_t n = rows * r;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(scale_rows_kernel<T>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    B, rows, r, scale, f, out);
}

// ------------------------------------------------------------------ gradient assembly
// One entry dA[j, k] of a dA assembly.
template <typename T>
__device__ __forceinline__ float finalize_dA_val(int64_t k, int j, int r, int64_t in, const Partial& PA, float sA,
                                                 const Partial& PW, float sW, const float* Kg, float s2,
                                                 const T* A) {
  float a = 0.f;
  if (PA.p) {
    float t = 0.f;
    for (int s = 0; s < PA.splits; ++s) t += PA.p[((int64_t)s * in + k) * PA.ldp + PA.j0 + j];
    a += sA * t;
  }
  if (PW.p) {
    float t = 0.f;
    for (int s = 0; s < PW.splits; ++s) t += PW.p[((int64_t)s * in + k) * PW.ldp + PW.j0 + j];
    a += sW * t;
  }
  if (Kg) {
    float t = 0.f;
    for (int l = 0; l < r; ++l) t = fmaf(Kg[j * r + l], ldf(A, (int64_t)l * in + k), t);
    a += s2 * t;
  }
  return a;
}

template <typename T>
__device__ __forceinline__ void finalize_dB_elem(int64_t i, int64_t out, int r, const Partial& PB, float sB,
                                                 const float* rs, const float* g, const float* V, const T* B,
                                                 const float* Kr, float s, bool accumulate, T* dB) {
  const int64_t o = i / r;
  const int j = (int)(i - o * r);
  float t = 0.f;
  if (PB.p)
    for (int sp = 0; sp < PB.splits; ++sp) t += PB.p[((int64_t)sp * out + o) * PB.ldp + PB.j0 + j];
  float a = sB * (rs ? rs[o] : 1.f) * t;
  if (accumulate) a += ldf(dB, i);
  if (V) {  // norm terms; g == null: the weights are already inside V and Kr
    const float go = g ? g[o] : 1.f;
    float bk = 0.f;
    for (int l = 0; l < r; ++l) bk = fmaf(ldf(B, o * r + l), Kr[l * r + j], bk);
    a += 2.f * s * go * V[o * r + j] + 2.f * s * s * go * bk;
  }
  dB[i] = from_f<T>(a);
}

template <typename T>
__global__ void finalize_dA_kernel(int r, int64_t in, Partial PA, float sA, Partial PW, float sW, const float* Kg,
                                   float s2, const T* A, T* dA) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // index into dA [r, in]
  if (i >= (int64_t)r * in) return;
  const int j = (int)(i / in);
  const int64_t k = i - (int64_t)j * in;
  dA[i] = from_f<T>(finalize_dA_val<T>(k, j, r, in, PA, sA, PW, sW, Kg, s2, A));
}
template <typename T>
cudaError_t finalize_dA(int r, int64_t in, Partial PA, float sA, Partial PW, float sW, const float* Kg, float s2,
                        const T* A, T* dA, cudaStream_t st) {
  const int64_t n = (int64_t)r * in;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(finalize_dA_kernel<T>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    r, in, PA, sA, PW, sW, Kg, s2, A, dA);
}

template <typename T>
__global__ void finalize_dB_kernel(int64_t out, int r, Partial PB, float sB, const float* rs, const float* g,
                                   const float* V, const T* B, const float* Kr, float s, bool accumulate, T* dB) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // index into dB [out, r]
  if (i < out * r) finalize_dB_elem<T>(i, out, r, PB, sB, rs, g, V, B, Kr, s, accumulate, dB);
}
template <typename T>
cudaError_t finalize_dB(int64_t out, int r, Partial PB, float sB, const float* rs, const float* g, const float* V,
                        const T* B, const float* Kr, float s, bool accumulate, T* dB, cudaStream_t st) {
  const int64_t n = out * r;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(finalize_dB_kernel<T>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    out, r, PB, sB, rs, g, V, B, Kr, s, accumulate, dB);
}

// Several dA / dB assemblies in one launch: job j owns blocks [first[j], first[j + 1]).
struct FinBatch {
  FinJob job[kMaxFinJobs];
  int first[kMaxFinJobs + 1];
  int n = 0;
};
__global__ void finalize_batch_kernel(const __grid_constant__ FinBatch b) {
  pdl_wait();      // the partials come from the previous kernels in the stream
  if (threadIdx.x == 0) pdl_trigger();
  int j = 0;
  while (j + 1 < b.n && (int)blockIdx.x >= b.first[j + 1]) ++j;
  const FinJob& f = b.job[j];
  const int64_t i = (int64_t)(blockIdx.x - b.first[j]) * blockDim.x + threadIdx.x;
  if (f.is_dB) {
    if (i < f.rows * f.r)
      finalize_dB_elem<bf16>(i, f.rows, f.r, f.P, f.sP, f.rs, f.g, f.V, f.M, f.Kx, f.s, false, f.out);
  } else {
    if (i < (int64_t)f.r * f.rows) {
      const int jj = (int)(i / f.rows);
      const int64_t k = i - (int64_t)jj * f.rows;
      f.out[i] = from_f<bf16>(finalize_dA_val<bf16>(k, jj, f.r, f.rows, f.P, f.sP, f.PW, f.sW, f.Kx, f.s2, f.M));
    }
  }
}
cudaError_t finalize_batch(const FinJob* jobs, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n > kMaxFinJobs) return cudaErrorInvalidValue;
  FinBatch b;
  int64_t blocks = 0;
  for (int j = 0; j < n; ++j) {
    b.job[j] = jobs[j];
    b.first[j] = (int)blocks;
    blocks += (jobs[j].rows * jobs[j].r + 255) / 256;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  }
  b.first[n] = (int)blocks;
  b.n = n;
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, finalize_batch_kernel, b);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------ concat / zero
__global__ void concat_rows_kernel(const uint4* X1, int64_t n1, const uint4* X2, int64_t n2, uint4* dst) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n1) dst[i] = X1[i];
  else if (i < n1 + n2) dst[i] = X2[i - n1];
}
cudaError_t concat_rows_bf16(const bf16* X1, int64_t rows1, const bf16* X2, int64_t rows2, int64_t cols, bf16* dst,
                             cudaStream_t st) {
  const int64_t n1 = rows1 * cols / 8, n2 = rows2 * cols / 8;
  if (n1 + n2 <= 0) return cudaSuccess;
  return launch_pdl(concat_rows_kernel, dim3((unsigned)((n1 + n2 + 255) / 256)), dim3(256), 0, st,
                    reinterpret_cast<const uint4*>(X1), n1, reinterpret_cast<const uint4*>(X2), n2,
                    reinterpret_cast<uint4*>(dst));
}
// Fused-leaf operands: A_stack = [A_0; A_1; ...] ([L r, in]) and the block-diagonal
// B_blk [N, L r] whose rows of leaf l hold s_l B_l in columns l r .. l r + r - 1, zeros elsewhere.
__global__ void pack_leaves_kernel(LeafPack p) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int R = p.L * p.r;
  const int64_t nA = (int64_t)R * p.in / 8;   // 16-byte chunks of A_stack
  const int64_t nB = p.B_blk ? p.N * R : 0;   // no B_blk: A_stack only
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nA + nB; i += stride) {
    if (i < nA) {
      const int64_t e = i * 8;
      const int row = (int)(e / p.in);
      const int leaf = row / p.r;
      const int64_t off = (int64_t)(row - leaf * p.r) * p.in + (e - (int64_t)row * p.in);
      *reinterpret_cast<uint4*>(p.A_stack + e) = *reinterpret_cast<const uint4*>(p.A[leaf] + off);
    } else {
      const int64_t e = i - nA;
      const int64_t o = e / R;
      const int j = (int)(e - o * R);
      int leaf = 0;
      while (leaf + 1 < p.L && o >= p.row0[leaf + 1]) ++leaf;
      const int jl = j - leaf * p.r;
      float v = 0.f;
      if (jl >= 0 && jl < p.r) v = p.s[leaf] * __bfloat162float(p.B[leaf][(o - p.row0[leaf]) * p.r + jl]);
      p.B_blk[e] = __float2bfloat16_rn(v);
    }
  }
}
cudaError_t pack_leaves(const LeafPack& p, cudaStream_t st) {
  const int64_t n = (int64_t)p.L * p.r * p.in / 8 + (p.B_blk ? p.N * p.L * p.r : 0);
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  return launch_pdl(pack_leaves_kernel, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, st, p);
}

// ------------------------------------------------------------------ DoRA column variant (bf16)
// c0[k] = sum_o W[o, k]^2: 32 columns per block, 8 row phases reduced through shared memory
__global__ void colnorm2_kernel(const bf16* W, int64_t rows, int64_t cols, float* c0) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  __shared__ float red[8][33];
  const int64_t k = (int64_t)blockIdx.x * 32 + threadIdx.x;
  float acc = 0.f;
  if (k < cols)
    for (int64_t o = threadIdx.y; o < rows; o += 8) {
      const float f = __bfloat162float(W[o * cols + k]);
      acc = fmaf(f, f, acc);
    }
  red[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && k < cols) {
    float t = 0.f;
    for (int y = 0; y < 8; ++y) t += red[y][threadIdx.x];
    c0[k] = t;
  }
}
cudaError_t colnorm2_bf16(const bf16* W, int64_t rows, int64_t cols, float* c0, cudaStream_t st) {
  if (cols <= 0) return cudaSuccess;
  return launch_pdl(colnorm2_kernel, dim3((unsigned)((cols + 31) / 32)), dim3(32, 8), 0, st, W, rows, cols, c0);
}

// closed-form column norm, one warp per input column k (lane j holds A[j + 32 h, k], h < 4):
//   q = c0[k] + 2s sum_j A[j,k] U[k,j] + s^2 sum_j A[j,k] (Kb A)[j,k],  n = max(sqrt(max(q, 0)), eps),
//   c = m / n, and (optionally) A_c[:, k] = bf16(A[:, k] c[k]).
__global__ void dora_colnorm_kernel(int64_t in, int r, const float* c0, const float* U, const bf16* A,
                                    const float* Kb, const bf16* m, float s, float eps, float* n_out, float* c,
                                    bf16* A_c) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  extern __shared__ float sK[];
  for (int i = threadIdx.x; i < r * r; i += blockDim.x) sK[i] = Kb[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t k = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (k >= in) return;
  float a[4], t1 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int j = lane + 32 * h;
    a[h] = j < r ? __bfloat162float(A[(int64_t)j * in + k]) : 0.f;
    if (j < r) t1 = fmaf(a[h], U[k * r + j], t1);
  }
  float kk[4] = {0.f, 0.f, 0.f, 0.f};   // (Kb A)[j, k] for j = lane + 32 h (Kb symmetric)
  for (int l = 0; l < r; ++l) {
    const float al = __shfl_sync(0xffffffffu, a[l >> 5], l & 31);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (lane + 32 * h < r) kk[h] = fmaf(sK[l * r + lane + 32 * h], al, kk[h]);
  }
  float t2 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) t2 = fmaf(a[h], kk[h], t2);
  t1 = warp_sum(t1);
  t2 = warp_sum(t2);
  const float q = c0[k] + 2.f * s * t1 + s * s * t2;
  const float n = fmaxf(sqrtf(fmaxf(q, 0.f)), eps);
  const float cc = __bfloat162float(m[k]) / n;
  if (lane == 0) {
    n_out[k] = n;
    c[k] = cc;
  }
  if (A_c) {
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (lane + 32 * h < r) A_c[(int64_t)(lane + 32 * h) * in + k] = __float2bfloat16_rn(a[h] * cc);
  }
}
cudaError_t dora_colnorm(int64_t in, int r, const float* c0, const float* U, const bf16* A, const float* Kb,
                         const bf16* m, float s, float eps, float* n_out, float* c, bf16* A_c, cudaStream_t st) {
  if (in <= 0) return cudaSuccess;
  if (r > kNormMaxR) return cudaErrorInvalidValue;
  const cudaError_t ea = allow_rr_smem(dora_colnorm_kernel);
  if (ea != cudaSuccess) return ea;
  return launch_pdl(dora_colnorm_kernel, dim3((unsigned)((in + 7) / 8)), dim3(256), r * r * sizeof(float), st,
                    in, r, c0, U, A, Kb, m, s, eps, n_out, c, A_c);
}

// out[j, k] = bf16(A[j, k] * w[k])  (A [r, in])
__global__ void scale_cols_kernel(const bf16* A, int r, int64_t in, const float* w, bf16* out) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)r * in) return;
  out[i] = __float2bfloat16_rn(__bfloat162float(A[i]) * w[i % in]);
}
cudaError_t scale_cols_bf16(const bf16* A, int r, int64_t in, const float* w, bf16* out, cudaStream_t st) {
  const int64_t n = (int64_t)r * in;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(scale_cols_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, A, r, in, w, out);
}

// K = A diag(w) A^T (fp32 [r, r]), one block per (i, j >= i)
__global__ void gram_rows_weighted_kernel(const bf16* A, int r, int64_t cols, const float* w, float* K) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int i = blockIdx.x / r, j = blockIdx.x % r;
  if (j < i) return;
  float acc = 0.f;
  for (int64_t k = threadIdx.x; k < cols; k += blockDim.x)
    acc = fmaf(w[k] * __bfloat162float(A[i * cols + k]), __bfloat162float(A[j * cols + k]), acc);
  acc = block_sum<256>(acc);
  if (threadIdx.x == 0) {
    K[i * r + j] = acc;
    K[j * r + i] = acc;
  }
}
cudaError_t gram_rows_weighted(const bf16* A, int r, int64_t cols, const float* w, float* K, cudaStream_t st) {
  return launch_pdl(gram_rows_weighted_kernel, dim3(r * r), dim3(256), 0, st, A, r, cols, w, K);
}

// dA[j, k] = c[k] sum_s PA[s][k][j] + 2 s g[k] U[k, j] + 2 s^2 g[k] (Kb A)[j, k]
__global__ void finalize_dA_cols_kernel(int r, int64_t in, Partial PA, const float* c, const float* g,
                                        const float* U, const float* Kb, const bf16* A, float s, bf16* dA) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)r * in) return;
  const int j = (int)(i / in);
  const int64_t k = i - (int64_t)j * in;
  float t = 0.f;
  for (int sp = 0; sp < PA.splits; ++sp) t += PA.p[((int64_t)sp * in + k) * PA.ldp + PA.j0 + j];
  float ka = 0.f;
  for (int l = 0; l < r; ++l) ka = fmaf(Kb[j * r + l], __bfloat162float(A[(int64_t)l * in + k]), ka);
  dA[i] = __float2bfloat16_rn(c[k] * t + 2.f * s * g[k] * U[k * r + j] + 2.f * s * s * g[k] * ka);
}
cudaError_t finalize_dA_cols(int r, int64_t in, Partial PA, const float* c, const float* g, const float* U,
                             const float* Kb, const bf16* A, float s, bf16* dA, cudaStream_t st) {
  const int64_t n = (int64_t)r * in;
  if (n <= 0) return cudaSuccess;
  return launch_pdl(finalize_dA_cols_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    r, in, PA, c, g, U, Kb, A, s, dA);
}

// ------------------------------------------------------------------ input dropout (unfused path)
// out = bf16(X o mask * scale), 8 elements (one 16-byte chunk) per thread; cols a multiple of 8
__global__ void apply_mask_kernel(const uint4* X, const uint2* mask, float scale, int64_t n8, uint4* out) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  uint4 v = X[i];
  const uint2 m = mask[i];
  const uint8_t* mb = reinterpret_cast<const uint8_t*>(&m);
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = unpack_bf16x2(w[e]);
    w[e] = pack_bf16x2(mb[2 * e] ? f.x * scale : 0.f, mb[2 * e + 1] ? f.y * scale : 0.f);
  }
  out[i] = v;
}
cudaError_t apply_mask_bf16(const bf16* X, const uint8_t* mask, float scale, int64_t rows, int64_t cols, bf16* out,
                            cudaStream_t st) {
  const int64_t n8 = rows * cols / 8;
  if (n8 <= 0) return cudaSuccess;
  return launch_pdl(apply_mask_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, st,
                    reinterpret_cast<const uint4*>(X), reinterpret_cast<const uint2*>(mask), scale, n8,
                    reinterpret_cast<uint4*>(out));
}

// dX[i, k] += scale * mask[i, k] * sum_j G[i, j] A[j, k]  (the adapter's share of dX when a mask
// sits between X and A), G [rows, r], A [r, cols].  A CTA owns 32 rows x 256 columns: A's
// 256-column slice (bf16) and G's 32 rows (fp32) are staged in shared memory; warp w owns rows w,
// w + 8, w + 16, w + 24 and lane l columns 8 l .. 8 l + 7, so every A value read from shared
// memory feeds four rows and every G value is a warp-wide broadcast.  The thread's dX and mask
// chunks are loaded first, their latency overlapping the staging and the products; dX and the
// mask move once, 512 contiguous bytes of a row per warp access.  (75 us for the 8192 x 4096
// rank-16 case when each thread read its 16 rows of A and of G by itself, 55 us tiled, cold.)
constexpr int kAmrRows = 32, kAmrCols = 256;
__global__ void __launch_bounds__(256) add_masked_rank_kernel(bf16* dX, const bf16* G, const bf16* A,
                                                              const uint8_t* mask, float scale, int64_t rows,
                                                              int64_t cols, int r) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  extern __shared__ uint4 amr_smem[];
  bf16* As = reinterpret_cast<bf16*>(amr_smem);                  // [r][256]
  float* Gs = reinterpret_cast<float*>(As + (size_t)r * kAmrCols);  // [32][r]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r0 = (int64_t)blockIdx.x * kAmrRows;
  const int64_t c0 = (int64_t)blockIdx.y * kAmrCols;
  const int64_t k = c0 + lane * 8;
  uint4 d[4];
  uint2 m[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int64_t row = r0 + warp + 8 * q;
    d[q] = make_uint4(0u, 0u, 0u, 0u);
    m[q] = make_uint2(0u, 0u);
    if (row < rows && k < cols) {
      d[q] = *reinterpret_cast<const uint4*>(dX + row * cols + k);
      m[q] = *reinterpret_cast<const uint2*>(mask + row * cols + k);
    }
  }
  for (int i = tid; i < r * (kAmrCols / 8); i += 256) {   // A slice, 8 columns per 16-byte chunk
    const int j = i / (kAmrCols / 8), c = (i % (kAmrCols / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c0 + c < cols) v = *reinterpret_cast<const uint4*>(A + (int64_t)j * cols + c0 + c);
    *reinterpret_cast<uint4*>(As + j * kAmrCols + c) = v;
  }
  for (int i = tid; i < kAmrRows * r; i += 256) {
    const int rr = i / r;
    Gs[i] = r0 + rr < rows ? __bfloat162float(G[(r0 + rr) * r + (i - rr * r)]) : 0.f;
  }
  __syncthreads();
  float acc[4][8];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[q][e] = 0.f;
  for (int j = 0; j < r; ++j) {
    const uint4 av = *reinterpret_cast<const uint4*>(As + j * kAmrCols + lane * 8);
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&av);
    float af[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(aw[e]);
      af[2 * e] = f.x;
      af[2 * e + 1] = f.y;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float gj = Gs[(warp + 8 * q) * r + j];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[q][e] = fmaf(gj, af[e], acc[q][e]);
    }
  }
  if (k >= cols) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int64_t row = r0 + warp + 8 * q;
    if (row >= rows) break;
    const uint8_t* mb = reinterpret_cast<const uint8_t*>(&m[q]);
    uint32_t* dw = reinterpret_cast<uint32_t*>(&d[q]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(dw[e]);
      dw[e] = pack_bf16x2(f.x + (mb[2 * e] ? scale * acc[q][2 * e] : 0.f),
                          f.y + (mb[2 * e + 1] ? scale * acc[q][2 * e + 1] : 0.f));
    }
    *reinterpret_cast<uint4*>(dX + row * cols + k) = d[q];
  }
}
cudaError_t add_masked_rank_bf16(bf16* dX, const bf16* G, const bf16* A, const uint8_t* mask, float scale,
                                 int64_t rows, int64_t cols, int r, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (r < 1 || r > 128 || cols % 8) return cudaErrorInvalidValue;   // A slice + G rows: at most 80 KB
  const size_t smem = (size_t)r * kAmrCols * 2 + (size_t)kAmrRows * r * 4;
  static size_t opted = 48 * 1024;
  if (smem > opted) {
    const cudaError_t e = cudaFuncSetAttribute(add_masked_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    opted = smem;
  }
  const dim3 grid((unsigned)((rows + kAmrRows - 1) / kAmrRows), (unsigned)((cols + kAmrCols - 1) / kAmrCols));
  return launch_pdl(add_masked_rank_kernel, dim3(grid), dim3(256), smem, st, dX, G, A, mask, scale, rows, cols, r);
}

cudaError_t fill_zero(void* p, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  return cudaMemsetAsync(p, 0, bytes, st);
}

// ------------------------------------------------------------------ bounded-wait test hook
__global__ void debug_wait_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the wait must run out and record the error
    (void)mbar_wait(&bar, 0, timeout_ns, &abort_flag, err, 0x7001);
  }
  __syncthreads();
}
cudaError_t debug_wait_timeout(uint32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ explicit instantiations
#define INST(T)                                                                                                    \
  template cudaError_t rownorm2<T>(const T*, int64_t, int64_t, float*, cudaStream_t);                               \
  template cudaError_t gram_rows<T>(const T*, int, int64_t, float*, cudaStream_t);                                  \
  template cudaError_t gram_weighted<T>(const T*, int64_t, int, const float*, float*, float*, cudaStream_t);                \
  template cudaError_t dora_norm<T>(int64_t, int, const float*, const float*, const T*, const float*, const T*,     \
                                    float, float, float*, float*, cudaStream_t);                                    \
  template cudaError_t dora_c<T>(int64_t, const T*, const float*, float*, cudaStream_t, int64_t);                            \
  template cudaError_t sum_splits<T>(const float*, int, int64_t, float*, T*, cudaStream_t);                         \
  template cudaError_t dora_dc<T>(int64_t, const float*, const float*, int, const T*, const float*, const float*,        \
                                  const T*, float, float*, T*, T*, cudaStream_t);                                   \
  template cudaError_t scale_rows<T>(const T*, int64_t, int, const float*, float, T*, cudaStream_t);                \
  template cudaError_t finalize_dA<T>(int, int64_t, Partial, float, Partial, float, const float*, float, const T*,  \
                                      T*, cudaStream_t);                                                            \
  template cudaError_t finalize_dB<T>(int64_t, int, Partial, float, const float*, const float*, const float*,       \
                                      const T*, const float*, float, bool, T*, cudaStream_t);
INST(float)
INST(bf16)
#undef INST

}  // namespace lg

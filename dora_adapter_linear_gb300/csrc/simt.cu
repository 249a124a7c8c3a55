// fp32 path (LORA_F32): plain SIMT FMA tiles, fp32 accumulation, no TF32.  It serves the
// small fp32 workload whose tolerance (1e-5 relative L2) rules out reduced-precision tensor
// math; the fused structure is the same as the bf16 path (no [d_out, d_in] update is ever
// formed: the low-rank terms are extra thin products accumulated into the same output).
#include "common.cuh"
#include "internal.h"

namespace lg {

constexpr int SG_T = 64;   // output tile
constexpr int SG_K = 16;   // K slab

__global__ void __launch_bounds__(256) sgemm_kernel(SgemmDesc d) {
  __shared__ float As[SG_K][SG_T + 4];
  __shared__ float Bs[SG_K][SG_T + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * SG_T, n0 = (int64_t)blockIdx.x * SG_T;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < d.K; k0 += SG_K) {
    for (int i = threadIdx.x; i < SG_T * SG_K; i += 256) {
      // keep the contiguous global index fastest across threads
      int mm, kk;
      if (d.ta) { mm = i % SG_T; kk = i / SG_T; } else { kk = i % SG_K; mm = i / SG_K; }
      const int64_t m = m0 + mm, k = k0 + kk;
      float v = 0.f;
      if (m < d.M && k < d.K) {
        v = d.ta ? d.A[k * d.lda + m] : d.A[m * d.lda + k];
        if (d.kscale) v *= d.kscale[k];
      }
      As[kk][mm] = v;
    }
    for (int i = threadIdx.x; i < SG_T * SG_K; i += 256) {
      int nn, kk;
      if (d.tb) { kk = i % SG_K; nn = i / SG_K; } else { nn = i % SG_T; kk = i / SG_T; }
      const int64_t n = n0 + nn, k = k0 + kk;
      float v = 0.f;
      if (n < d.N && k < d.K) v = d.tb ? d.B[n * d.ldb + k] : d.B[k * d.ldb + n];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= d.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= d.N) continue;
      float v = acc[i][j] * d.alpha;
      if (d.rscale) v *= d.rscale[m];
      if (d.cs) v *= d.cs[n];
      if (d.bias) v += d.bias[n];
      float* c = d.C + m * d.ldc + n;
      if (d.beta != 0.f) v += d.beta * *c;
      *c = v;
    }
  }
}

cudaError_t sgemm_f32(const SgemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0) return cudaSuccess;
  dim3 grid((unsigned)((d.N + SG_T - 1) / SG_T), (unsigned)((d.M + SG_T - 1) / SG_T));
  sgemm_kernel<<<grid, 256, 0, st>>>(d);
  count_launch();
  return cudaGetLastError();
}

__global__ void coldot_f32_kernel(const float* S, const float* Y, int64_t rows, int64_t K, float* colsum,
                                  float* coldot) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= K) return;
  float a = 0.f, b = 0.f;
  for (int64_t i = 0; i < rows; ++i) {
    const float sv = S[i * K + k];
    a += sv;
    if (Y) b = fmaf(sv, Y[i * K + k], b);
  }
  if (colsum) colsum[k] = a;
  if (coldot) coldot[k] = b;
}

cudaError_t coldot_f32(const float* S, const float* Y, int64_t rows, int64_t K, float* colsum, float* coldot,
                       cudaStream_t st) {
  if (K <= 0) return cudaSuccess;
  coldot_f32_kernel<<<(unsigned)((K + 127) / 128), 128, 0, st>>>(S, Y, rows, K, colsum, coldot);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lg

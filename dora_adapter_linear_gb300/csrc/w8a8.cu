// W8A8 base layer with a LoRA epilogue: the quantiser, the int8 re-layouts and the warp-level
// integer product (an alternative to the chunked bf16 tensor-core product of tc_gemm.cu).
//
// The int8 product is exact: int8 x int8 products summed in int32 by the warp-level integer
// MMA (mma.sync m16n8k32 s8.s8.s32).  sm_103a has no tcgen05 integer kind (the PTX assembler
// rejects .kind::i8 for this target).
// The epilogue works on registers: acc * sx[i] * sw[o] + s * (Z B^T)[i, o] + bias[o] -> bf16,
// where the rank-r term is one more small bf16 MMA per 16-row tile; the int32 [M, d_out]
// product is never written unless the raw-product epilogue (acc_out) is asked for.
// "nunchaku-style kernel fusion" (OneTrainer #1680): the three epilogues over one shared
// 8-bit matmul core, and no int32 materialisation.
#include "common.cuh"
#include "internal.h"

namespace lg {

// ------------------------------------------------------------------ per-row absmax quantisation
// Writes the codes as int8 (Xq) and/or as bf16 values (Xb: the same integers, exact in bf16, ready
// to be the A operand of the tensor-core product); either may be null.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const bf16* X, int64_t cols, int8_t* Xq, float* sx,
                                                            bf16* Xb) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t row = blockIdx.x;
  const bf16* x = X + row * cols;
  float amax = 0.f;
  for (int64_t k = (int64_t)threadIdx.x * 8; k < cols; k += 256 * 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(x + k);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_bf16x2(w[i]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  const float scale = __fdiv_rn(m, 127.0f);  // IEEE round-to-nearest division
  if (threadIdx.x == 0) sx[row] = scale;
  for (int64_t k = (int64_t)threadIdx.x * 8; k < cols; k += 256 * 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(x + k);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
    uint32_t packed[2] = {0u, 0u};
    uint32_t codes[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_bf16x2(w[i]);
      int q0 = 0, q1 = 0;
      if (scale > 0.f) {
        q0 = min(127, max(-127, __float2int_rn(__fdiv_rn(f.x, scale))));
        q1 = min(127, max(-127, __float2int_rn(__fdiv_rn(f.y, scale))));
      }
      packed[i >> 1] |= ((uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8)) << ((i & 1) * 16);
      codes[i] = pack_bf16x2((float)q0, (float)q1);
    }
    if (Xq) *reinterpret_cast<uint2*>(Xq + row * cols + k) = make_uint2(packed[0], packed[1]);
    if (Xb) *reinterpret_cast<uint4*>(Xb + row * cols + k) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  }
}

cudaError_t quantize_rows_bf16(const bf16* X, int64_t rows, int64_t cols, int8_t* Xq, float* sx, cudaStream_t st,
                               bf16* Xb) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(quantize_rows_kernel, dim3((unsigned)rows), dim3(256), 0, st, X, cols, Xq, sx, Xb);
}

// ------------------------------------------------------------------ int8 codes as bf16 tensor-core operands
// Every int8 value is exact in bf16, so the codes are the operands of the bf16 tensor-core product,
// which sums them exactly in 1024-wide K chunks (every partial sum an integer below 2^24).
__global__ void i8_to_bf16_kernel(const int8_t* __restrict__ q, int64_t n16, bf16* __restrict__ out) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 raw = reinterpret_cast<const uint4*>(q)[i];
  const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2((float)b[2 * j], (float)b[2 * j + 1]);
  uint4* o = reinterpret_cast<uint4*>(out) + 2 * i;
  o[0] = make_uint4(w[0], w[1], w[2], w[3]);
  o[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// W_deq[o, k] = bf16(sw[o] * q[o, k]): the int8 base weight in real units, the B operand of
// the backward's dX product (the frozen weight, re-laid out once per call like a k-major copy).
__global__ void i8_dequant_rows_kernel(const int8_t* __restrict__ q, const float* __restrict__ sw, int64_t cols,
                                       int64_t n16, bf16* __restrict__ out) {
  pdl_wait();   // inputs may come from the previous kernel in the stream
  if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const float sc = sw[(i * 16) / cols];
  const uint4 raw = reinterpret_cast<const uint4*>(q)[i];
  const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(sc * (float)b[2 * j], sc * (float)b[2 * j + 1]);
  uint4* o = reinterpret_cast<uint4*>(out) + 2 * i;
  o[0] = make_uint4(w[0], w[1], w[2], w[3]);
  o[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

cudaError_t i8_dequant_rows_bf16(const int8_t* q, const float* sw, int64_t rows, int64_t cols, bf16* out,
                                 cudaStream_t st) {
  const int64_t n16 = rows * cols / 16;  // cols is a multiple of 16: a group never straddles rows
  if (n16 <= 0) return cudaSuccess;
  return launch_pdl(i8_dequant_rows_kernel, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0, st,
                    q, sw, cols, n16, out);
}

cudaError_t i8_to_bf16(const int8_t* q, int64_t n, bf16* out, cudaStream_t st) {
  const int64_t n16 = n / 16;
  if (n16 <= 0) return cudaSuccess;
  return launch_pdl(i8_to_bf16_kernel, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0, st, q, n16, out);
}


// ------------------------------------------------------------------ int8 GEMM + epilogue
namespace w8 {
constexpr int BM = 128, BN = 128, BK = 64;  // BK in bytes (int8 elements)
constexpr int PITCH = BK + 16;              // 80-byte rows: conflict-free ldmatrix
constexpr int STAGES = 4;
constexpr int TILE_BYTES = BM * PITCH;      // 10240
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
}  // namespace w8

__global__ void __launch_bounds__(256) w8a8_gemm_kernel(int64_t M, int64_t K, int64_t N, int r, const int8_t* Xq,
                                                        const float* sx, const int8_t* Wq, const float* sw,
                                                        const bf16* Z, const bf16* Bm, float s, const bf16* bias,
                                                        bf16* Y, int32_t* acc_out) {
  using namespace w8;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp & 1, wn = warp >> 1;  // warp tile: 64 rows x 32 cols
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const int nkc = (int)((K + BK - 1) / BK);

  auto load_stage = [&](int stage, int kc) {
    uint8_t* sa = smem + stage * STAGE_BYTES;
    uint8_t* sb = sa + TILE_BYTES;
    const int64_t k0 = (int64_t)kc * BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int ci = tid + 256 * i;  // 128 rows x 4 chunks
      const int rr = ci >> 2, c = ci & 3;
      const int64_t gk = k0 + c * 16;
      const int64_t ga = m0 + rr, gb = n0 + rr;
      const bool oka = ga < M && gk < K, okb = gb < N && gk < K;
      cp_async16(sa + rr * PITCH + c * 16, oka ? Xq + ga * K + gk : Xq, oka);
      cp_async16(sb + rr * PITCH + c * 16, okb ? Wq + gb * K + gk : Wq, okb);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0;

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < nkc) load_stage(st, st);
    cp_async_commit();
  }
  for (int kc = 0; kc < nkc; ++kc) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const uint32_t sa = smem_u32(smem + (kc % STAGES) * STAGE_BYTES);
    const uint32_t sb = sa + TILE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 32; ++kk) {
      uint32_t a[4][4];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
        ldsm_x4(a[mi][0], a[mi][1], a[mi][2], a[mi][3],
                sa + (wm * 64 + mi * 16 + (lane & 15)) * PITCH + kk * 32 + (lane >> 4) * 16);
#pragma unroll
      for (int nj = 0; nj < 4; nj += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3,
                sb + (wn * 32 + nj * 8 + (lane & 7) + ((lane >> 4) << 3)) * PITCH + kk * 32 + ((lane >> 3) & 1) * 16);
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
          mma_s8_16832(acc[mi][nj], a[mi], b0, b1);
          mma_s8_16832(acc[mi][nj + 1], a[mi], b2, b3);
        }
      }
    }
    const int nxt = kc + STAGES - 1;
    if (nxt < nkc) load_stage(nxt % STAGES, nxt);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // ---- epilogue, one 16-row slab at a time
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
    const int64_t rA = m0 + wm * 64 + mi * 16 + g, rB = rA + 8;
    float lora[4][4];
#pragma unroll
    for (int nj = 0; nj < 4; ++nj) lora[nj][0] = lora[nj][1] = lora[nj][2] = lora[nj][3] = 0.f;
    if (Z != nullptr && Y != nullptr) {
      for (int k16 = 0; k16 < r; k16 += 16) {
        const int kc0 = k16 + 2 * t, kc1 = k16 + 8 + 2 * t;
        uint32_t a[4];
        a[0] = (rA < M && kc0 < r) ? *reinterpret_cast<const uint32_t*>(Z + rA * r + kc0) : 0u;
        a[1] = (rB < M && kc0 < r) ? *reinterpret_cast<const uint32_t*>(Z + rB * r + kc0) : 0u;
        a[2] = (rA < M && kc1 < r) ? *reinterpret_cast<const uint32_t*>(Z + rA * r + kc1) : 0u;
        a[3] = (rB < M && kc1 < r) ? *reinterpret_cast<const uint32_t*>(Z + rB * r + kc1) : 0u;
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
          const int64_t col = n0 + wn * 32 + nj * 8 + g;
          const uint32_t b0 = (col < N && kc0 < r) ? *reinterpret_cast<const uint32_t*>(Bm + col * r + kc0) : 0u;
          const uint32_t b1 = (col < N && kc1 < r) ? *reinterpret_cast<const uint32_t*>(Bm + col * r + kc1) : 0u;
          mma_bf16_16816(lora[nj], a, b0, b1);
        }
      }
    }
#pragma unroll
    for (int nj = 0; nj < 4; ++nj) {
      const int64_t col = n0 + wn * 32 + nj * 8 + 2 * t;
      if (col >= N) continue;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int64_t row = hr ? rB : rA;
        if (row >= M) continue;
        const int a0 = acc[mi][nj][2 * hr], a1 = acc[mi][nj][2 * hr + 1];
        if (acc_out) *reinterpret_cast<int2*>(acc_out + row * N + col) = make_int2(a0, a1);
        if (Y) {
          const float rs = sx[row];
          float y0 = (float)a0 * rs * sw[col] + s * lora[nj][2 * hr];
          float y1 = (float)a1 * rs * sw[col + 1] + s * lora[nj][2 * hr + 1];
          if (bias) {
            y0 += __bfloat162float(bias[col]);
            y1 += __bfloat162float(bias[col + 1]);
          }
          *reinterpret_cast<uint32_t*>(Y + row * N + col) = pack_bf16x2(y0, y1);
        }
      }
    }
  }
}

cudaError_t w8a8_gemm(int64_t M, int64_t K, int64_t N, int r, const int8_t* Xq, const float* sx, const int8_t* Wq,
                      const float* sw, const bf16* Z, const bf16* B, float s, const bf16* bias, bf16* Y,
                      int32_t* acc_out, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int smem = w8::STAGES * w8::STAGE_BYTES;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(w8a8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  dim3 grid((unsigned)((N + w8::BN - 1) / w8::BN), (unsigned)((M + w8::BM - 1) / w8::BM));
  w8a8_gemm_kernel<<<grid, 256, smem, st>>>(M, K, N, r, Xq, sx, Wq, sw, Z, B, s, bias, Y, acc_out);
  count_launch();
  return cudaGetLastError();
}

}  // namespace lg

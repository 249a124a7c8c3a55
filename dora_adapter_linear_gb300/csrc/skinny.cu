// Rank-r ("skinny") kernels of the bf16 path.  These touch every element of a large
// activation once and do 2r flops per element, so they are HBM-bound: the design goal is
// coalesced 16-byte loads, a deep cp.async pipeline and enough CTAs in flight per SM.
// The arithmetic runs on the legacy warp MMA (mma.sync m16n8k16, fp32 accumulate), which
// keeps up with HBM at these ranks.
//
//   rowproj:   T = S U^T           (down-projections Z = X A^T, G = dY B, V = W0 A^T)
//   colreduce: P = S^T T per split (adapter gradients dB = s dY^T Z, dA^T = X^T G,
//                                   DoRA norm gradient W0^T (g o B); column sums / dots)
#include "common.cuh"
#include "internal.h"

namespace lg {

// ============================================================================ rowproj
namespace rp {
constexpr int BMR = 32;        // rows per CTA
constexpr int BKC = 128;       // K per stage (256-byte row segments of S)
constexpr int PITCH = BKC + 8; // padded smem row pitch (elements) -> conflict-free ldmatrix
constexpr int STAGES = 6;      // deep ring: ~43 KB of the streamed operand in flight per CTA
constexpr int S_BYTES = BMR * PITCH * 2;       // 8704
// U chunk: [R(+8 pad rows), BKC] K-major or [BKC, R+8] R-major
template <int R, bool KR>
constexpr int u_bytes() { return KR ? BKC * (R + 8) * 2 : (R + 8) * PITCH * 2; }
template <int R, bool KR>
constexpr int stage_bytes() { return S_BYTES + u_bytes<R, KR>(); }
}  // namespace rp

template <int R, bool U_KR>
__global__ void __launch_bounds__(128) rowproj_kernel(RowProjDesc d) {
  using namespace rp;
  constexpr int STAGE_BYTES = stage_bytes<R, U_KR>();
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp & 1;        // 16-row group
  const int kh = warp >> 1;       // which half of each BKC-wide K chunk
  const int64_t row0 = (int64_t)blockIdx.x * BMR;
  const int nkc = (int)((d.K + BKC - 1) / BKC);
  constexpr int UPITCH = U_KR ? (R + 8) : PITCH;

  auto load_stage = [&](int stage, int kc) {
    uint8_t* sS = smem + stage * STAGE_BYTES;
    uint8_t* sU = sS + S_BYTES;
    const int64_t k0 = (int64_t)kc * BKC;
    constexpr int CPS = BKC / 8;   // 16-byte chunks per staged row
#pragma unroll
    for (int i = 0; i < BMR * CPS / 128; ++i) {
      const int ci = tid + 128 * i;
      const int r = ci / CPS, c = ci % CPS;
      const int64_t gr = row0 + r, gk = k0 + c * 8;
      const bool ok = gr < d.rows && gk < d.K;
      const bf16* src = ok ? d.S + gr * d.lds + gk : d.S;
      cp_async16(sS + (r * PITCH + c * 8) * 2, src, ok);
    }
    if (!U_KR) {  // U [R, K]: R rows x CPS chunks
      for (int ci = tid; ci < R * CPS; ci += 128) {
        const int r = ci / CPS, c = ci % CPS;
        const int64_t gk = k0 + c * 8;
        const bool ok = gk < d.K;
        const bf16* src = ok ? d.U + (int64_t)r * d.ldu + gk : d.U;
        cp_async16(sU + (r * UPITCH + c * 8) * 2, src, ok);
      }
    } else {      // U [K, R]: BKC rows x R/8 chunks
      constexpr int CPR = R / 8;
      for (int ci = tid; ci < BKC * CPR; ci += 128) {
        const int r = ci / CPR, c = ci % CPR;
        const int64_t gk = k0 + r;
        const bool ok = gk < d.K;
        const bf16* src = ok ? d.U + gk * d.ldu + c * 8 : d.U;
        cp_async16(sU + (r * UPITCH + c * 8) * 2, src, ok);
      }
    }
  };

  float acc[R / 8][4];
#pragma unroll
  for (int i = 0; i < R / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nkc) load_stage(s, s);
    cp_async_commit();
  }
  for (int kc = 0; kc < nkc; ++kc) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const int stage = kc % STAGES;
    const uint32_t sS = smem_u32(smem + stage * STAGE_BYTES);
    const uint32_t sU = sS + S_BYTES;
    if (d.s_out) {
      // column-scaled copy of this 32 x 128 tile of S: thread tid owns 16-byte chunk (tid & 15)
      // of rows (tid >> 4) + 8 i
      const int c16 = tid & 15;
      const int64_t gk = (int64_t)kc * BKC + c16 * 8;
      if (gk < d.K) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(d.s_scale + gk));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(d.s_scale + gk + 4));
        const float sc8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        const uint8_t* tile = smem + stage * STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < BMR / 8; ++i) {
          const int r = (tid >> 4) + 8 * i;
          if (row0 + r >= d.rows) break;
          uint4 v = *reinterpret_cast<const uint4*>(tile + (r * PITCH + c16 * 8) * 2);
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            w[e] = pack_bf16x2(f.x * sc8[2 * e], f.y * sc8[2 * e + 1]);
          }
          *reinterpret_cast<uint4*>(d.s_out + (row0 + r) * d.K + gk) = v;
        }
      }
    }
#pragma unroll
    for (int k2 = 0; k2 < BKC / 32; ++k2) {
      const int kk = kh * (BKC / 32) + k2;  // k16 step within the BKC-wide chunk
      uint32_t a[4];
      ldsm_x4(a[0], a[1], a[2], a[3],
              sS + ((rg * 16 + (lane & 15)) * PITCH + kk * 16 + (lane >> 4) * 8) * 2);
#pragma unroll
      for (int nt = 0; nt < R / 8; nt += 2) {
        uint32_t b0, b1, b2, b3;
        if (!U_KR) {
          // rows n (8 + 8), 8 contiguous k at kk*16 and kk*16+8
          const int n = nt * 8 + (lane & 7) + ((lane >> 4) << 3);
          const int kcol = kk * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(b0, b1, b2, b3, sU + (n * UPITCH + kcol) * 2);
        } else {
          const int krow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ncol = nt * 8 + (lane >> 4) * 8;
          ldsm_x4_t(b0, b1, b2, b3, sU + (krow * UPITCH + ncol) * 2);
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
        if (nt + 1 < R / 8) mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
    }
    const int nxt = kc + STAGES - 1;
    if (nxt < nkc) load_stage(nxt % STAGES, nxt);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();

  // combine the two K halves: warps with kh == 1 hand their partial sums over via smem
  float* red = reinterpret_cast<float*>(smem);  // [2 row groups][32 lanes][R/2]
  if (kh == 1) {
#pragma unroll
    for (int nt = 0; nt < R / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[(rg * 32 + lane) * (R / 2) + nt * 4 + e] = acc[nt][e];
  }
  __syncthreads();
  if (kh == 0) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < R / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] += red[(rg * 32 + lane) * (R / 2) + nt * 4 + e];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int64_t grow = row0 + rg * 16 + g + hr * 8;
        if (grow >= d.rows) continue;
        const int col = nt * 8 + 2 * t;
        const int64_t ldo = d.ldo > 0 ? d.ldo : R;
        const float v0 = acc[nt][2 * hr], v1 = acc[nt][2 * hr + 1];
        if (d.out_a)
          *reinterpret_cast<uint32_t*>(d.out_a + grow * ldo + col) = pack_bf16x2(v0 * d.scale_a, v1 * d.scale_a);
        if (d.out_b) {
          const float sb = col >= d.split_col ? d.scale_b_hi : d.scale_b;
          *reinterpret_cast<uint32_t*>(d.out_b + grow * ldo + col) = pack_bf16x2(v0 * sb, v1 * sb);
        }
        if (d.out_f) *reinterpret_cast<float2*>(d.out_f + grow * ldo + col) = make_float2(v0, v1);
      }
    }
  }
}

template <int R, bool KR>
static cudaError_t rowproj_launch(const RowProjDesc& d, cudaStream_t st) {
  const int smem = rp::STAGES * rp::stage_bytes<R, KR>();
  auto k = rowproj_kernel<R, KR>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  const int64_t grid = (d.rows + rp::BMR - 1) / rp::BMR;
  k<<<(unsigned)grid, 128, smem, st>>>(d);
  count_launch();
  return cudaGetLastError();
}

cudaError_t rowproj(const RowProjDesc& d, cudaStream_t st) {
  if (d.rows <= 0) return cudaSuccess;
#define RP_CASE(RR)                                                                   \
  case RR:                                                                            \
    return d.u_kr ? rowproj_launch<RR, true>(d, st) : rowproj_launch<RR, false>(d, st);
  switch (d.R) {
    RP_CASE(8)
    RP_CASE(16)
    RP_CASE(24)
    RP_CASE(32)
    RP_CASE(40)
    RP_CASE(48)
    RP_CASE(56)
    RP_CASE(64)
  }
#undef RP_CASE
  return cudaErrorInvalidValue;
}

// ============================================================================ colreduce
namespace cr {
constexpr int BKC = 64;       // columns (K) per CTA
constexpr int BR = 64;        // rows per stage
constexpr int PITCH = 72;
constexpr int S_BYTES = BR * PITCH * 2;   // 9216
}  // namespace cr

template <int R, bool HAS_Y, bool SUMS>
__global__ void __launch_bounds__(128) colreduce_kernel(ColReduceDesc d, int64_t rows_per_split) {
  using namespace cr;
  constexpr int TPITCH = R + 8;
  constexpr int T_BYTES = BR * TPITCH * 2;
  constexpr int STAGE_BYTES = S_BYTES + T_BYTES + (HAS_Y ? S_BYTES : 0);
  constexpr int STAGES = HAS_Y ? 3 : 4;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k0 = (int64_t)blockIdx.x * BKC;
  const int split = blockIdx.y;
  const int64_t r_begin = (int64_t)split * rows_per_split;
  const int64_t r_end = min(d.rows, r_begin + rows_per_split);
  const int nrc = r_end > r_begin ? (int)((r_end - r_begin + BR - 1) / BR) : 0;

  auto load_stage = [&](int stage, int rc) {
    uint8_t* sS = smem + stage * STAGE_BYTES;
    uint8_t* sT = sS + S_BYTES;
    uint8_t* sY = sT + T_BYTES;
    const int64_t rb = r_begin + (int64_t)rc * BR;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // 64 rows x 8 chunks
      const int ci = tid + 128 * i;
      const int r = ci >> 3, c = ci & 7;
      const int64_t gr = rb + r, gk = k0 + c * 8;
      const bool ok = gr < r_end && gk < d.K;
      cp_async16(sS + (r * PITCH + c * 8) * 2, ok ? d.S + gr * d.lds + gk : d.S, ok);
      if (HAS_Y) cp_async16(sY + (r * PITCH + c * 8) * 2, ok ? d.Y + gr * d.ldy + gk : d.Y, ok);
    }
    constexpr int CPR = R / 8;
    for (int ci = tid; ci < BR * CPR; ci += 128) {
      const int r = ci / CPR, c = ci % CPR;
      const int64_t gr = rb + r;
      const bool ok = gr < r_end;
      cp_async16(sT + (r * TPITCH + c * 8) * 2, ok ? d.T + gr * d.ldt + c * 8 : d.T, ok);
    }
  };

  float acc[R / 8][4];
#pragma unroll
  for (int i = 0; i < R / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float csum = 0.f, cdot = 0.f;
  const int my_col = tid & 63, my_par = tid >> 6;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nrc) load_stage(s, s);
    cp_async_commit();
  }
  for (int rc = 0; rc < nrc; ++rc) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const int stage = rc % STAGES;
    uint8_t* pS = smem + stage * STAGE_BYTES;
    const uint32_t sS = smem_u32(pS);
    const uint32_t sT = sS + S_BYTES;
#pragma unroll
    for (int kk = 0; kk < BR / 16; ++kk) {
      uint32_t a[4];
      {
        const int row = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int col = warp * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(a[0], a[1], a[2], a[3], sS + (row * PITCH + col) * 2);
      }
#pragma unroll
      for (int nt = 0; nt < R / 8; nt += 2) {
        uint32_t b0, b1, b2, b3;
        const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int col = nt * 8 + (lane >> 4) * 8;
        if (nt + 1 < R / 8) {
          ldsm_x4_t(b0, b1, b2, b3, sT + (row * TPITCH + col) * 2);
        } else {
          ldsm_x2_t(b0, b1, sT + (row * TPITCH + nt * 8) * 2);
          b2 = b3 = 0;
        }
        mma_bf16_16816(acc[nt], a, b0, b1);
        if (nt + 1 < R / 8) mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
    }
    if (HAS_Y && d.sc_out) {
      // the column-scaled copy of this 64 x 64 tile: thread tid owns 16-byte chunk (tid & 7) of rows
      // (tid >> 3) + 16 i, so its 8 scales are fixed for the whole kernel
      const int c8 = tid & 7;
      const int64_t gk = k0 + c8 * 8;
      if (gk < d.K) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(d.sc + gk));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(d.sc + gk + 4));
        const float sc8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        const int64_t rb = r_begin + (int64_t)rc * BR;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (tid >> 3) + 16 * i;
          if (rb + r >= r_end) break;
          uint4 v = *reinterpret_cast<const uint4*>(pS + (r * PITCH + c8 * 8) * 2);
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            w[e] = pack_bf16x2(f.x * sc8[2 * e], f.y * sc8[2 * e + 1]);
          }
          *reinterpret_cast<uint4*>(d.sc_out + (rb + r) * d.K + gk) = v;
        }
      }
    }
    if (SUMS) {
      const bf16* ps = reinterpret_cast<const bf16*>(pS);
      const bf16* py = reinterpret_cast<const bf16*>(pS + S_BYTES + T_BYTES);
#pragma unroll 8
      for (int r = my_par; r < BR; r += 2) {
        const float sv = __bfloat162float(ps[r * PITCH + my_col]);
        csum += sv;
        if (HAS_Y) cdot += sv * __bfloat162float(py[r * PITCH + my_col]);
      }
    }
    const int nxt = rc + STAGES - 1;
    __syncthreads();
    if (nxt < nrc) load_stage(nxt % STAGES, nxt);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();

  const int g = lane >> 2, t = lane & 3;
  float* part = d.part + ((int64_t)split * d.K) * R;
#pragma unroll
  for (int nt = 0; nt < R / 8; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int64_t k = k0 + warp * 16 + g + hr * 8;
      if (k < d.K)
        *reinterpret_cast<float2*>(part + k * R + nt * 8 + 2 * t) = make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
    }
  if (SUMS) {
    float* red = reinterpret_cast<float*>(smem);
    if (my_par == 1) {
      red[my_col] = csum;
      red[64 + my_col] = cdot;
    }
    __syncthreads();
    if (my_par == 0) {
      const int64_t k = k0 + my_col;
      if (k < d.K) {
        if (d.colsum) d.colsum[(int64_t)split * d.K + k] = csum + red[my_col];
        if (HAS_Y && d.coldot) d.coldot[(int64_t)split * d.K + k] = cdot + red[64 + my_col];
      }
    }
  }
}

int colreduce_splits(int64_t rows, int64_t K) {
  const int64_t kb = (K + cr::BKC - 1) / cr::BKC;
  int64_t want = (4LL * num_sms_current() + kb - 1) / kb;
  const int64_t maxs = (rows + cr::BR - 1) / cr::BR;
  if (want > maxs) want = maxs;
  if (want < 1) want = 1;
  if (want > 64) want = 64;
  return (int)want;
}

template <int R, bool HAS_Y, bool SUMS>
static cudaError_t colreduce_launch(const ColReduceDesc& d, cudaStream_t st) {
  constexpr int T_BYTES = cr::BR * (R + 8) * 2;
  constexpr int STAGE_BYTES = cr::S_BYTES + T_BYTES + (HAS_Y ? cr::S_BYTES : 0);
  constexpr int STAGES = HAS_Y ? 3 : 4;
  const int smem = STAGES * STAGE_BYTES;
  auto k = colreduce_kernel<R, HAS_Y, SUMS>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  int64_t rps = (d.rows + d.splits - 1) / d.splits;
  rps = (rps + cr::BR - 1) / cr::BR * cr::BR;
  dim3 grid((unsigned)((d.K + cr::BKC - 1) / cr::BKC), (unsigned)d.splits);
  k<<<grid, 128, smem, st>>>(d, rps);
  count_launch();
  return cudaGetLastError();
}

cudaError_t colreduce(const ColReduceDesc& d, cudaStream_t st) {
  if (d.K <= 0) return cudaSuccess;
  const bool has_y = d.Y != nullptr;
  const bool sums = d.colsum != nullptr || d.coldot != nullptr;
#define CR_CASE(RR)                                                          \
  case RR:                                                                   \
    if (has_y) return colreduce_launch<RR, true, true>(d, st);               \
    if (sums) return colreduce_launch<RR, false, true>(d, st);               \
    return colreduce_launch<RR, false, false>(d, st);
  switch (d.R) {
    CR_CASE(8)
    CR_CASE(16)
    CR_CASE(24)
    CR_CASE(32)
    CR_CASE(40)
    CR_CASE(48)
    CR_CASE(56)
    CR_CASE(64)
  }
#undef CR_CASE
  return cudaErrorInvalidValue;
}

}  // namespace lg

// Rank-r ("skinny") kernels of the bf16 path.  These touch every element of a large
// activation once and do 2r flops per element, so they are HBM-bound: tiles arrive by TMA
// (one producer warp per CTA, a deep mbarrier ring) and enough CTAs are in flight per SM.
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
// One CTA owns 32 rows of S and streams them across K in 64-wide stages: a producer warp
// issues one TMA box for the S tile (32 x 64, 128B-swizzled) and one for the matching U tile;
// the consumer warps (16 rows each, two K groups taking alternate stages) run the warp MMAs
// straight from the swizzled tiles, and the second K group's sums are added through shared
// memory at the end.  One K group left the MMA chain of each warp, not the memory system, as
// the limit (3.2 TB/s from L2).
namespace rp {
constexpr int BMR = 32;   // rows per CTA
constexpr int BK = 64;    // K per stage (one 128-byte swizzle row)
constexpr int S_BYTES = BMR * 128;

// byte offset of 16-byte chunk `chunk` of row `row` in a TMA-swizzled tile whose rows are
// `pitch` bytes: the chunk index is XORed with address bits 7.. (mask 7 / 3 / 1 / 0 for the
// 128 / 64 / 32-byte / no swizzle)
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk, uint32_t pitch, uint32_t mask) {
  return row * pitch + ((chunk ^ (((row * pitch) >> 7) & mask)) << 4);
}

template <int R, bool U_KR, bool MASK = false>
struct Cfg {
  // U [K, R]: the TMA box spans RPAD >= R columns (power of two, zero-filled past R)
  static constexpr int RPAD = R <= 8 ? 8 : (R <= 16 ? 16 : (R <= 32 ? 32 : 64));
  static constexpr int UPITCH = U_KR ? RPAD * 2 : 128;
  static constexpr int UMASK = U_KR ? (RPAD == 8 ? 0 : RPAD == 16 ? 1 : RPAD == 32 ? 3 : 7) : 7;
  static constexpr int USWZ = U_KR ? (RPAD == 8 ? 0 : RPAD * 2) : 128;
  static constexpr int UROWS = (R + 15) / 16 * 16;              // U [R, K]: rows reserved (even n-tiles)
  static constexpr int U_BYTES = U_KR ? BK * RPAD * 2 : UROWS * 128;
  static constexpr int U_TX = U_KR ? BK * RPAD * 2 : R * 128;   // bytes the U box delivers
  static constexpr int OFF_M = S_BYTES + U_BYTES;                // keep-mask tile (32 x 64 bytes)
  static constexpr int M_BYTES = MASK ? BMR * BK : 0;
  static constexpr int STAGE = (S_BYTES + U_BYTES + M_BYTES + 1023) / 1024 * 1024;
  // stages in flight: about 96 KB per CTA (two CTAs per SM); 8 stages of the small ranks left
  // the pass latency-bound
  static constexpr int NST = (96 * 1024 / STAGE) > 16 ? 16 : ((96 * 1024 / STAGE) < 8 ? 8 : 96 * 1024 / STAGE);
  // consumer warps: 2 row groups of 16 x NG groups of output columns (split when R / 8 is even
  // and large enough, so that more warps share the MMA work of one tile)
  static constexpr int NG = (R % 16 == 0 && R >= 32) ? 2 : 1;
  static constexpr int NTW = R / 8 / NG;   // n-tiles of 8 per consumer warp
  static constexpr int KG = 2;             // K groups: consumer warp sets taking alternate stages
  static constexpr int NCW = 2 * NG * KG;  // consumer warps; the producer is warp NCW
  static constexpr int THREADS = 32 * (NCW + 1);
  static constexpr int RED = (NCW - 2 * NG) * 32 * NTW * 4 * 4;   // partial sums of the K groups > 0
  static constexpr int SMEM = NST * STAGE + RED + 1024 + 2 * NST * 8 + 16;
};
}  // namespace rp

struct RpParams {
  CUtensorMap tmS;
  CUtensorMap tmU;
  CUtensorMap tmM;   // keep mask (MASK)
  RowProjDesc d;
};

template <int R, bool U_KR, bool MASK>
__global__ void __launch_bounds__(rp::Cfg<R, U_KR, MASK>::THREADS) rowproj_kernel(const __grid_constant__ RpParams P) {
  using namespace rp;
  using C = Cfg<R, U_KR, MASK>;
  const RowProjDesc& d = P.d;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(smem + C::NST * C::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE + C::RED);
  uint64_t* empty = full + C::NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::NST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (int64_t)blockIdx.x * BMR;
  const int nkc = (int)((d.K + BK - 1) / BK);
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2 * C::NG);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();      // S and U may come from the previous kernel in the stream
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == C::NCW) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&P.tmS);
      tma_prefetch_desc(&P.tmU);
      if (MASK) tma_prefetch_desc(&P.tmM);
      bool ok = true;
      for (int kc = 0; kc < nkc; ++kc) {
        const int s = kc % C::NST;
        const uint32_t ph = (uint32_t)(kc / C::NST) & 1u;
        if (kc >= C::NST && !mbar_wait(&empty[s], ph ^ 1u, d.timeout_ns, abort_flag, d.err, 0x301)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * C::STAGE;
        mbar_expect_tx(&full[s], S_BYTES + C::U_TX + C::M_BYTES);
        tma_load_2d(st, &P.tmS, &full[s], kc * BK, (int)row0);
        if (MASK) tma_load_2d(st + C::OFF_M, &P.tmM, &full[s], kc * BK, (int)row0);
        if (U_KR) tma_load_2d(st + S_BYTES, &P.tmU, &full[s], 0, kc * BK);
        else tma_load_2d(st + S_BYTES, &P.tmU, &full[s], kc * BK, 0);
      }
      if (!ok) spin_ns(100000ull);  // unwind: let copies already issued land
    }
    return;
  }

  // ------------------------------------------------------------------ consumers: 16 rows x R / NG each
  constexpr int NTW = C::NTW;
  const int rg = warp & 1;                  // row group (rows 16 rg .. 16 rg + 15 of the tile)
  const int nh = (warp >> 1) % C::NG;       // column group (n-tiles nh NTW .. nh NTW + NTW - 1)
  const int kg = warp / (2 * C::NG);        // K group: stages kg, kg + KG, ...
  float acc[NTW][4];
#pragma unroll
  for (int i = 0; i < NTW; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int c8 = lane & 7;  // the 16-byte chunk this lane copies in the scaled side output
  for (int kc = kg; kc < nkc; kc += C::KG) {
    const int s = kc % C::NST;
    const uint32_t ph = (uint32_t)(kc / C::NST) & 1u;
    if (!mbar_wait(&full[s], ph, d.timeout_ns, abort_flag, d.err, 0x302)) break;
    const uint8_t* tile = smem + s * C::STAGE;
    const uint32_t sS = smem_u32(tile);
    const uint32_t sU = sS + S_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a[0], a[1], a[2], a[3], sS + swz(rg * 16 + (lane & 15), kk * 2 + (lane >> 4), 128, 7));
      if constexpr (MASK) {
        // a[i] holds S[16 rg + g + 8 (i & 1)][16 kk + 2t + 8 (i >> 1) + {0, 1}] (g = lane / 4,
        // t = lane % 4): the matching two mask bytes are adjacent in the 64-byte mask row
        const uint8_t* mrow = tile + C::OFF_M + (rg * 16 + (lane >> 2)) * BK + kk * 16 + 2 * (lane & 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t m2 = *reinterpret_cast<const uint16_t*>(mrow + (i & 1) * 8 * BK + (i >> 1) * 8);
          a[i] = mask_bf16x2(a[i], m2 & 0xffu, m2 >> 8, d.mask_scale);
        }
      }
#pragma unroll
      for (int q = 0; q < NTW; q += 2) {
        const int nt = nh * NTW + q;
        uint32_t b0, b1, b2 = 0, b3 = 0;
        if (!U_KR) {
          const int n = nt * 8 + (lane & 7) + ((lane >> 4) << 3);
          const int c = kk * 2 + ((lane >> 3) & 1);
          if (q + 1 < NTW) ldsm_x4(b0, b1, b2, b3, sU + swz(n, c, 128, 7));
          else ldsm_x2(b0, b1, sU + swz(nt * 8 + (lane & 7), c, 128, 7));
        } else {
          const int krow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          if (q + 1 < NTW) ldsm_x4_t(b0, b1, b2, b3, sU + swz(krow, nt + (lane >> 4), C::UPITCH, C::UMASK));
          else ldsm_x2_t(b0, b1, sU + swz(krow, nt, C::UPITCH, C::UMASK));
        }
        mma_bf16_16816(acc[q], a, b0, b1);
        if (q + 1 < NTW) mma_bf16_16816(acc[q + 1], a, b2, b3);
      }
    }
    if (d.s_out && nh == 0) {
      // column-scaled copy of this warp's 16 x 64 slice of S (lane: chunk c8 of rows lane/8 + 4 i)
      const int64_t gk = (int64_t)kc * BK + c8 * 8;
      if (gk < d.K) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(d.s_scale + gk));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(d.s_scale + gk + 4));
        const float sc8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rg * 16 + (lane >> 3) + 4 * i;
          if (row0 + r >= d.rows) break;
          uint4 v = *reinterpret_cast<const uint4*>(tile + swz(r, c8, 128, 7));
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
    warp_release(&empty[s], lane);
  }

  // add the other K groups' sums into K group 0, which writes the outputs
  {
    const int slot = warp % (2 * C::NG);
    if (kg > 0) {
      float* dst = red + (((kg - 1) * 2 * C::NG + slot) * 32 + lane) * NTW * 4;
#pragma unroll
      for (int q = 0; q < NTW; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[q * 4 + e] = acc[q][e];
    }
    named_bar_sync(1, 32 * C::NCW);
    if (kg > 0) return;
#pragma unroll
    for (int j = 1; j < C::KG; ++j) {
      const float* src = red + (((j - 1) * 2 * C::NG + slot) * 32 + lane) * NTW * 4;
#pragma unroll
      for (int q = 0; q < NTW; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[q][e] += src[q * 4 + e];
    }
  }

  const int g = lane >> 2, t = lane & 3;
  const int64_t ldo = d.ldo > 0 ? d.ldo : R;
#pragma unroll
  for (int q = 0; q < NTW; ++q) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int64_t grow = row0 + rg * 16 + g + hr * 8;
      if (grow >= d.rows) continue;
      const int col = (nh * NTW + q) * 8 + 2 * t;
      const float v0 = acc[q][2 * hr], v1 = acc[q][2 * hr + 1];
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

template <int R, bool KR, bool MASK = false>
static cudaError_t rowproj_launch(const RowProjDesc& d, cudaStream_t st) {
  using C = rp::Cfg<R, KR, MASK>;
  auto k = rowproj_kernel<R, KR, MASK>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    set = true;
  }
  RpParams P;
  memset(&P, 0, sizeof(P));
  P.d = d;
  bool ok = make_tmap_bf16(&P.tmS, d.S, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.lds, rp::BK, rp::BMR, 128);
  if (KR) ok = ok && make_tmap_bf16(&P.tmU, d.U, R, (uint64_t)d.K, (uint64_t)d.ldu, C::RPAD, rp::BK, C::USWZ);
  else ok = ok && make_tmap_bf16(&P.tmU, d.U, (uint64_t)d.K, R, (uint64_t)d.ldu, rp::BK, R, 128);
  if (MASK) ok = ok && make_tmap_u8(&P.tmM, d.mask, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.K, rp::BK, rp::BMR);
  if (!ok) return cudaErrorInvalidValue;
  const int64_t grid = (d.rows + rp::BMR - 1) / rp::BMR;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  // algorithmic HBM bytes: S once, U, the outputs (and the scaled copy of S)
  const double outs = (d.out_a ? 2.0 : 0.0) + (d.out_b ? 2.0 : 0.0) + (d.out_f ? 4.0 : 0.0);
  const double bytes = 2.0 * d.rows * d.K * (d.s_out ? 2.0 : 1.0) + (MASK ? 1.0 * d.rows * d.K : 0.0) +
                       2.0 * R * d.K + outs * d.rows * R;
  prof_mark(st, true, bytes, 1);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, P);
  prof_mark(st, false, 0.0, 1);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t rowproj(const RowProjDesc& d, cudaStream_t st) {
  if (d.rows <= 0) return cudaSuccess;
  if (d.mask && (d.u_kr || d.s_out || d.K % 16)) return cudaErrorInvalidValue;   // masked S: X A^T only
  if (d.R > 64) {   // columns in chunks of 64: one pass over S per chunk
    if (d.R > 512 || d.R % 8) return cudaErrorInvalidValue;
    const int64_t ldo = d.ldo > 0 ? d.ldo : d.R;
    for (int c0 = 0; c0 < d.R; c0 += 64) {
      RowProjDesc c = d;
      c.R = d.R - c0 < 64 ? d.R - c0 : 64;
      c.U = d.u_kr ? d.U + c0 : d.U + (int64_t)c0 * d.ldu;
      c.out_a = d.out_a ? d.out_a + c0 : nullptr;
      c.out_b = d.out_b ? d.out_b + c0 : nullptr;
      c.out_f = d.out_f ? d.out_f + c0 : nullptr;
      c.ldo = ldo;
      c.split_col = d.split_col >= (1 << 29) ? d.split_col : d.split_col - c0;
      if (c0 > 0) {   // the scaled copy of S comes with the first chunk
        c.s_scale = nullptr;
        c.s_out = nullptr;
      }
      const cudaError_t e = rowproj(c, st);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
#define RP_CASE(RR)                                                                   \
  case RR:                                                                            \
    if (d.mask) return rowproj_launch<RR, false, true>(d, st);                        \
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
// One CTA owns 64 columns of S and one split of the rows.  A producer warp brings in, per
// 64-row stage, the 64 x 64 tile of S (and of Y), 128B-swizzled, and the 64 x R tile of T by
// TMA; four consumer warps (16 columns each) run the warp MMAs S^T T straight from the tiles.
namespace cr {
constexpr int BKC = 64;       // columns (K) per CTA
constexpr int BR = 64;        // rows per stage
constexpr int S_BYTES = BR * 128;

template <int R, bool HAS_Y, bool MASK = false>
struct Cfg {
  static constexpr int RPAD = R <= 8 ? 8 : (R <= 16 ? 16 : (R <= 32 ? 32 : 64));
  static constexpr int TPITCH = RPAD * 2;
  static constexpr int TMASK = RPAD == 8 ? 0 : RPAD == 16 ? 1 : RPAD == 32 ? 3 : 7;
  static constexpr int TSWZ = RPAD == 8 ? 0 : RPAD * 2;
  static constexpr int T_BYTES = BR * RPAD * 2;
  static constexpr int OFF_Y = S_BYTES + ((T_BYTES + 1023) / 1024) * 1024;   // Y tile, or the keep mask
  static constexpr int M_BYTES = MASK ? BR * BKC : 0;                          // 64 x 64 mask bytes
  static constexpr int STAGE = OFF_Y + (HAS_Y ? S_BYTES : 0) + M_BYTES;
  static constexpr int TX = S_BYTES + T_BYTES + (HAS_Y ? S_BYTES : 0) + M_BYTES;
  // stages: as many as keep the CTAs per SM of the pass without the mask (three up to rank 32)
  static constexpr int NST = HAS_Y ? 4 : (MASK ? 5 : 6);
  static constexpr int SMEM = NST * STAGE + 1024 + 2 * NST * 8 + 16;
};
}  // namespace cr

struct CrParams {
  CUtensorMap tmS;
  CUtensorMap tmT;
  CUtensorMap tmY;   // Y, or the keep mask (MASK)
  ColReduceDesc d;
  int64_t rows_per_split;
};

template <int R, bool HAS_Y, bool SUMS, bool MASK = false>
__global__ void __launch_bounds__(160) colreduce_kernel(const __grid_constant__ CrParams P) {
  using namespace cr;
  using rp::swz;
  static_assert(!MASK || (!HAS_Y && !SUMS), "masked S: no second input, no column sums");
  using C = Cfg<R, HAS_Y, MASK>;
  constexpr int NST = C::NST;
  const ColReduceDesc& d = P.d;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * C::STAGE);
  uint64_t* empty = full + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k0 = (int64_t)blockIdx.x * BKC;
  const int split = blockIdx.y;
  const int64_t r_begin = (int64_t)split * P.rows_per_split;   // a multiple of BR
  const int64_t r_end = min(d.rows, r_begin + P.rows_per_split);
  const int nrc = r_end > r_begin ? (int)((r_end - r_begin + BR - 1) / BR) : 0;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();      // S, T and Y may come from the previous kernel in the stream
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 4) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&P.tmS);
      tma_prefetch_desc(&P.tmT);
      if (HAS_Y) tma_prefetch_desc(&P.tmY);
      bool ok = true;
      for (int rc = 0; rc < nrc; ++rc) {
        const int s = rc % NST;
        const uint32_t ph = (uint32_t)(rc / NST) & 1u;
        if (rc >= NST && !mbar_wait(&empty[s], ph ^ 1u, d.timeout_ns, abort_flag, d.err, 0x311)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * C::STAGE;
        const int y = (int)(r_begin + (int64_t)rc * BR);
        mbar_expect_tx(&full[s], C::TX);
        tma_load_2d(st, &P.tmS, &full[s], (int)k0, y);
        tma_load_2d(st + S_BYTES, &P.tmT, &full[s], 0, y);
        if (HAS_Y || MASK) tma_load_2d(st + C::OFF_Y, &P.tmY, &full[s], (int)k0, y);
      }
      if (!ok) spin_ns(100000ull);  // unwind: let copies already issued land
    }
    return;
  }

  // ------------------------------------------------------------------ consumers: 16 columns each
  float acc[R / 8][4];
#pragma unroll
  for (int i = 0; i < R / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float csum = 0.f, cdot = 0.f;
  const int my_col = tid & 63, my_par = tid >> 6;   // column sums: 2 row phases x 64 columns
  const int c8 = tid & 7;                            // scaled copy: 16-byte chunk of this thread
  float sc8[8];
  const bool copy = HAS_Y && d.sc_out != nullptr && k0 + c8 * 8 < d.K;
  if (copy) {   // the 8 scales of this thread's chunk (K is a multiple of 8)
    const float4 lo = __ldg(reinterpret_cast<const float4*>(d.sc + k0 + c8 * 8));
    const float4 hi = __ldg(reinterpret_cast<const float4*>(d.sc + k0 + c8 * 8 + 4));
    sc8[0] = lo.x; sc8[1] = lo.y; sc8[2] = lo.z; sc8[3] = lo.w;
    sc8[4] = hi.x; sc8[5] = hi.y; sc8[6] = hi.z; sc8[7] = hi.w;
  }
  for (int rc = 0; rc < nrc; ++rc) {
    const int s = rc % NST;
    const uint32_t ph = (uint32_t)(rc / NST) & 1u;
    if (!mbar_wait(&full[s], ph, d.timeout_ns, abort_flag, d.err, 0x312)) break;
    const uint8_t* tile = smem + s * C::STAGE;
    const uint32_t sS = smem_u32(tile);
    const uint32_t sT = sS + S_BYTES;
#pragma unroll
    for (int kk = 0; kk < BR / 16; ++kk) {
      uint32_t a[4];
      {  // A = S^T: 16 columns of this warp x 16 rows, transposed out of the row-major tile
        const int row = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4_t(a[0], a[1], a[2], a[3], sS + swz(row, warp * 2 + ((lane >> 3) & 1), 128, 7));
      }
      if constexpr (MASK) {
        // a[i] holds S[16 kk + 8 (i >> 1) + 2t + {0, 1}][16 warp + 8 (i & 1) + g] (transposed
        // fragments; g = lane / 4, t = lane % 4): two mask bytes one 64-byte mask row apart
        const uint8_t* mcol = tile + C::OFF_Y + (kk * 16 + 2 * (lane & 3)) * BKC + warp * 16 + (lane >> 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint8_t* mp = mcol + (i >> 1) * 8 * BKC + (i & 1) * 8;
          a[i] = mask_bf16x2(a[i], mp[0], mp[BKC], d.mask_scale);
        }
      }
#pragma unroll
      for (int nt = 0; nt < R / 8; nt += 2) {
        uint32_t b0, b1, b2 = 0, b3 = 0;
        const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        if (nt + 1 < R / 8) ldsm_x4_t(b0, b1, b2, b3, sT + swz(row, nt + (lane >> 4), C::TPITCH, C::TMASK));
        else ldsm_x2_t(b0, b1, sT + swz(row, nt, C::TPITCH, C::TMASK));
        mma_bf16_16816(acc[nt], a, b0, b1);
        if (nt + 1 < R / 8) mma_bf16_16816(acc[nt + 1], a, b2, b3);
      }
    }
    if (copy) {
      // column-scaled copy of the S tile: thread tid owns chunk c8 of rows tid / 8 + 16 i
      const int64_t rb = r_begin + (int64_t)rc * BR;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = (tid >> 3) + 16 * i;
        if (rb + r >= r_end) break;
        uint4 v = *reinterpret_cast<const uint4*>(tile + swz(r, c8, 128, 7));
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(w[e]);
          w[e] = pack_bf16x2(f.x * sc8[2 * e], f.y * sc8[2 * e + 1]);
        }
        *reinterpret_cast<uint4*>(d.sc_out + (rb + r) * d.K + k0 + c8 * 8) = v;
      }
    }
    if (SUMS) {
      // rows past the end of the tensor were zero-filled by the TMA, so they add nothing
#pragma unroll 8
      for (int r = my_par; r < BR; r += 2) {
        const uint32_t o = swz(r, my_col >> 3, 128, 7) + (my_col & 7) * 2;
        const float sv = __bfloat162float(*reinterpret_cast<const bf16*>(tile + o));
        csum += sv;
        if (HAS_Y) cdot += sv * __bfloat162float(*reinterpret_cast<const bf16*>(tile + C::OFF_Y + o));
      }
    }
    warp_release(&empty[s], lane);
  }

  // ------------------------------------------------------------------ partials of this split
  const int g = lane >> 2, t = lane & 3;
  const int64_t ldp = d.ldp > 0 ? d.ldp : R;
  float* part = d.part + ((int64_t)split * d.K) * ldp + d.j0;
#pragma unroll
  for (int nt = 0; nt < R / 8; ++nt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int64_t k = k0 + warp * 16 + g + hr * 8;
      if (k < d.K)
        *reinterpret_cast<float2*>(part + k * ldp + nt * 8 + 2 * t) = make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
    }
  if (SUMS) {
    // the two row phases of each column meet in shared memory; stage 0 is free once all four
    // consumer warps are past their last wait (the producer issues nothing more by then)
    float* red = reinterpret_cast<float*>(smem);
    named_bar_sync(1, 128);
    if (my_par == 1) {
      red[my_col] = csum;
      red[64 + my_col] = cdot;
    }
    named_bar_sync(1, 128);
    if (my_par == 0) {
      const int64_t k = k0 + my_col;
      if (k < d.K) {
        if (d.colsum) d.colsum[(int64_t)split * d.K + k] = csum + red[my_col];
        if (HAS_Y && d.coldot) d.coldot[(int64_t)split * d.K + k] = cdot + red[64 + my_col];
      }
    }
  }
}

// CTAs of colreduce_kernel<R, HAS_Y, *, MASK> resident per SM, from its shared memory (each CTA
// also holds 1 KB reserved by the system; 228 KB per SM).
static int colreduce_ctas_per_sm(int R, bool has_y, bool mask) {
  int smem;
  if (R <= 8) smem = mask ? cr::Cfg<8, false, true>::SMEM : has_y ? cr::Cfg<8, true>::SMEM : cr::Cfg<8, false>::SMEM;
  else if (R <= 16)
    smem = mask ? cr::Cfg<16, false, true>::SMEM : has_y ? cr::Cfg<16, true>::SMEM : cr::Cfg<16, false>::SMEM;
  else if (R <= 32)
    smem = mask ? cr::Cfg<32, false, true>::SMEM : has_y ? cr::Cfg<32, true>::SMEM : cr::Cfg<32, false>::SMEM;
  else smem = mask ? cr::Cfg<64, false, true>::SMEM : has_y ? cr::Cfg<64, true>::SMEM : cr::Cfg<64, false>::SMEM;
  const int n = (228 * 1024) / (smem + 1024);
  return n < 1 ? 1 : n;
}

int colreduce_splits(int64_t rows, int64_t K, int R, bool has_y, bool mask) {
  const int64_t kb = (K + cr::BKC - 1) / cr::BKC;
  // Row splits per column block: with n CTAs resident per SM, a launch of kb * s CTAs runs in
  // ceil(kb s / slots) waves of CTAs that each stream ceil(rows / (64 s)) row stages plus a
  // fixed cost of about four stages (ring fill, partial sums); pick the s with the least total,
  // the fewest splits among equals.  A half-empty last wave cost ~1% of a LoRA step.
  const int64_t slots = (int64_t)colreduce_ctas_per_sm(R, has_y, mask) * num_sms_current();
  int64_t maxs = (rows + cr::BR - 1) / cr::BR;
  if (maxs > 64) maxs = 64;
  int64_t best = 1;
  double best_t = 1e30;
  for (int64_t sp = 1; sp <= maxs; ++sp) {
    const int64_t stages = (rows + cr::BR * sp - 1) / (cr::BR * sp);
    const double t = (double)((kb * sp + slots - 1) / slots) * (double)(stages + 4);
    if (t < best_t - 1e-12) {
      best_t = t;
      best = sp;
    }
  }
  return (int)best;
}

template <int R, bool HAS_Y, bool SUMS, bool MASK = false>
static cudaError_t colreduce_launch(const ColReduceDesc& d, cudaStream_t st) {
  using C = cr::Cfg<R, HAS_Y, MASK>;
  auto k = colreduce_kernel<R, HAS_Y, SUMS, MASK>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    set = true;
  }
  CrParams P;
  memset(&P, 0, sizeof(P));
  P.d = d;
  const int64_t rps = (d.rows + d.splits - 1) / d.splits;
  P.rows_per_split = (rps + cr::BR - 1) / cr::BR * cr::BR;
  bool ok = make_tmap_bf16(&P.tmS, d.S, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.lds, cr::BKC, cr::BR, 128);
  ok = ok && make_tmap_bf16(&P.tmT, d.T, R, (uint64_t)d.rows, (uint64_t)d.ldt, C::RPAD, cr::BR, C::TSWZ);
  if (HAS_Y)
    ok = ok && make_tmap_bf16(&P.tmY, d.Y, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.ldy, cr::BKC, cr::BR, 128);
  if (MASK) ok = ok && make_tmap_u8(&P.tmY, d.mask, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.K, cr::BKC, cr::BR);
  if (!ok) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((d.K + cr::BKC - 1) / cr::BKC), (unsigned)d.splits);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = grid;
  cfg.blockDim = dim3(160, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  // algorithmic HBM bytes: S (and Y, and the scaled copy) once, T, the fp32 partials (and column sums)
  const double bytes = 2.0 * d.rows * d.K * (HAS_Y ? (d.sc_out ? 3.0 : 2.0) : (MASK ? 1.5 : 1.0)) + 2.0 * d.rows * R +
                       4.0 * d.splits * d.K * (R + (SUMS ? 2.0 : 0.0));
  prof_mark(st, true, bytes, 1);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, P);
  prof_mark(st, false, 0.0, 1);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t colreduce(const ColReduceDesc& d, cudaStream_t st) {
  if (d.K <= 0) return cudaSuccess;
  if (d.sc_out && (!d.Y || !d.sc || d.K % 8)) return cudaErrorInvalidValue;   // the copy rides on the Y pass
  if (d.mask && (d.Y || d.colsum || d.coldot || d.sc_out || d.K % 16)) return cudaErrorInvalidValue;
  if (d.R > 64) {   // columns of T in chunks of 64: one pass over S per chunk
    if (d.R > 512 || d.R % 8) return cudaErrorInvalidValue;
    for (int c0 = 0; c0 < d.R; c0 += 64) {
      ColReduceDesc c = d;
      c.R = d.R - c0 < 64 ? d.R - c0 : 64;
      c.T = d.T + c0;
      c.ldp = d.ldp > 0 ? d.ldp : d.R;
      c.j0 = d.j0 + c0;
      if (c0 > 0) {   // the column sums come with the first chunk
        c.Y = nullptr;
        c.colsum = nullptr;
        c.coldot = nullptr;
        c.sc_out = nullptr;   // and so does the scaled copy
      }
      const cudaError_t e = colreduce(c, st);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  const bool has_y = d.Y != nullptr;
  const bool sums = d.colsum != nullptr || d.coldot != nullptr;
#define CR_CASE(RR)                                                          \
  case RR:                                                                   \
    if (d.mask) return colreduce_launch<RR, false, false, true>(d, st);      \
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

// ============================================================================ rowcol
// One pass over S [rows, K] for the two rank-r products that read it (the backward's dY side):
//   row products    gpart[bn][row][j] = sum over the columns k of column group bn of S[row, k] U[k, j]
//   column products part[bm][k][j]    = sum over the rows of row group bm of S[row, k] T[row, j]
//   (+ column sums  colsum[bm][k]     = sum over the same rows of S[row, k])
// with U [K, R] (row k contiguous) and T [rows, R].  The CTAs form a pm x pn grid of at most one
// wave: CTA (bm, bn) owns nb row blocks of 128 rows and the 512 columns of column group bn, and
// streams its 128 x 64 tiles of S (two 64-row TMA boxes), row block by row block, through a TMA
// ring; each stage also carries the T rows of its tile, and the CTA's U rows stay resident in
// shared memory.  (One CTA per SM with 8 KB stages streamed at 3 TB/s; 16 KB stages reach the
// rate of several CTAs per SM.)  Two groups of four consumer warps take alternate column chunks:
// warp i of a group forms rows 32i.. of the row product and columns 16i.. of the column product
// of each tile, both with the warp MMA straight from the swizzled tile (and a ones operand for
// the column sums).  A row block's two group partials meet in shared memory and go out as one
// fp32 partial; the column partials stay in registers until the CTA is done.  gpart is summed
// over bn by gpart_sum, part over bm by the gradient finalisation.
namespace rc {
constexpr int TR = 128;           // rows per tile (two 64-row boxes)
constexpr int TC = 64;            // columns per tile (one 128-byte swizzle row)
constexpr int CN = 512;           // columns per CTA
constexpr int NCH = CN / TC;      // column chunks per row block
constexpr int S_BYTES = TR * 128;
constexpr int NST = 6;            // ring depth (stages)

template <int R>
struct Cfg {
  static constexpr int RPAD = R <= 8 ? 8 : (R <= 16 ? 16 : 32);
  static constexpr int PITCH = RPAD * 2;
  static constexpr int MASK = RPAD == 8 ? 0 : RPAD == 16 ? 1 : 3;
  static constexpr int SWZ = RPAD == 8 ? 0 : RPAD * 2;
  static constexpr int T_BYTES = TR * RPAD * 2;
  static constexpr int STAGE = S_BYTES + (T_BYTES + 1023) / 1024 * 1024;
  static constexpr int U_BYTES = CN * RPAD * 2;
  static constexpr int NTW = R / 8;                          // n-tiles of 8 output columns
  static constexpr int RED = 2 * 4 * 32 * 2 * NTW * 4 * 4;   // two slots of group 1's row partials
  static constexpr int OFF_U = NST * STAGE;
  static constexpr int OFF_RED = OFF_U + U_BYTES;
  static constexpr int OFF_BAR = OFF_RED + RED;
  static constexpr int SMEM = OFF_BAR + (2 * NST + 1) * 8 + 16 + 1024;
  static constexpr int THREADS = 32 * 9;                     // 8 consumer warps + the producer
  static_assert(SMEM <= 232448, "shared memory budget");
};
}  // namespace rc

struct RcParams {
  CUtensorMap tmS;
  CUtensorMap tmU;
  CUtensorMap tmT;
  RowColDesc d;
};

template <int R, bool ROW, bool SUMS>
__global__ void __launch_bounds__(rc::Cfg<R>::THREADS, 1) rowcol_kernel(const __grid_constant__ RcParams P) {
  using namespace rc;
  using rp::swz;
  using C = Cfg<R>;
  constexpr int NTW = C::NTW;
  const RowColDesc& d = P.d;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sUr = smem + C::OFF_U;
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NST;
  uint64_t* ubar = empty + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ubar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bm = blockIdx.x / d.pn, bn = blockIdx.x % d.pn;
  const int64_t r0 = (int64_t)bm * d.nb * TR;
  const int64_t nblk_total = (d.rows + TR - 1) / TR;
  const int nb = (int)min((int64_t)d.nb, nblk_total - (int64_t)bm * d.nb);   // row blocks of this CTA
  const int c0 = bn * CN;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    mbar_init(ubar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();      // S, U and T may come from the previous kernel in the stream
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&P.tmS);
      tma_prefetch_desc(&P.tmT);
      if (ROW) {
        tma_prefetch_desc(&P.tmU);
        mbar_expect_tx(ubar, C::U_BYTES);
        tma_load_2d(sUr, &P.tmU, ubar, 0, c0);
        tma_load_2d(sUr + C::U_BYTES / 2, &P.tmU, ubar, 0, c0 + CN / 2);
      }
      const int n = nb * NCH;
      for (int q = 0; q < n; ++q) {
        const int s = q % NST;
        const uint32_t ph = (uint32_t)(q / NST) & 1u;
        if (q >= NST && !mbar_wait(&empty[s], ph ^ 1u, d.timeout_ns, abort_flag, d.err, 0x321)) break;
        uint8_t* st = smem + s * C::STAGE;
        const int y = (int)(r0 + (int64_t)(q / NCH) * TR);
        const int x = c0 + (q % NCH) * TC;
        mbar_expect_tx(&full[s], S_BYTES + C::T_BYTES);
        tma_load_2d(st, &P.tmS, &full[s], x, y);
        tma_load_2d(st + S_BYTES / 2, &P.tmS, &full[s], x, y + TR / 2);
        tma_load_2d(st + S_BYTES, &P.tmT, &full[s], 0, y);
      }
      if (*abort_flag) spin_ns(100000ull);  // unwind: let copies already issued land
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int grp = warp >> 2;      // chunks grp, grp + 2, ...
  const int wi = warp & 3;        // rows 32 wi.. of the row product, columns 16 wi.. of the column product
  const int g = lane >> 2, t = lane & 3;
  constexpr uint32_t ONES = 0x3F803F80u;   // two bf16 1.0
  float accP[NCH / 2][NTW][4];
  float accS[NCH / 2][4];
#pragma unroll
  for (int j = 0; j < NCH / 2; ++j) {
#pragma unroll
    for (int q = 0; q < NTW; ++q) accP[j][q][0] = accP[j][q][1] = accP[j][q][2] = accP[j][q][3] = 0.f;
    accS[j][0] = accS[j][1] = accS[j][2] = accS[j][3] = 0.f;
  }
  // every lane waits on the barriers itself: the tensor-copy writes are visible to the threads
  // that observe the phase completion
  bool ok = true;
  if (ROW) ok = __all_sync(0xffffffffu, mbar_wait(ubar, 0, d.timeout_ns, abort_flag, d.err, 0x322));
  const uint32_t sU = smem_u32(sUr);
  for (int b = 0; b < nb; ++b) {
    float accG[2][NTW][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int q = 0; q < NTW; ++q) accG[mt][q][0] = accG[mt][q][1] = accG[mt][q][2] = accG[mt][q][3] = 0.f;
#pragma unroll
    for (int j = 0; j < NCH / 2; ++j) {
      const int ch = 2 * j + grp;
      const int q = b * NCH + ch;
      const int s = q % NST;
      const uint32_t ph = (uint32_t)(q / NST) & 1u;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[s], ph, d.timeout_ns, abort_flag, d.err, 0x323));
      if (!ok) continue;
      const uint32_t sS = smem_u32(smem + s * C::STAGE);
      const uint32_t sT = sS + S_BYTES;
      if (ROW) {   // rows 32 wi.. of the tile times U rows ch*64 ..
#pragma unroll
        for (int kk = 0; kk < TC / 16; ++kk) {
          uint32_t a0[4], a1[4];
          ldsm_x4(a0[0], a0[1], a0[2], a0[3], sS + swz(wi * 32 + (lane & 15), kk * 2 + (lane >> 4), 128, 7));
          ldsm_x4(a1[0], a1[1], a1[2], a1[3], sS + swz(wi * 32 + 16 + (lane & 15), kk * 2 + (lane >> 4), 128, 7));
          const int krow = ch * TC + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
          for (int n = 0; n < NTW; n += 2) {
            uint32_t b0, b1, b2 = 0, b3 = 0;
            if (n + 1 < NTW) ldsm_x4_t(b0, b1, b2, b3, sU + swz(krow, n + (lane >> 4), C::PITCH, C::MASK));
            else ldsm_x2_t(b0, b1, sU + swz(krow, n, C::PITCH, C::MASK));
            mma_bf16_16816(accG[0][n], a0, b0, b1);
            mma_bf16_16816(accG[1][n], a1, b0, b1);
            if (n + 1 < NTW) {
              mma_bf16_16816(accG[0][n + 1], a0, b2, b3);
              mma_bf16_16816(accG[1][n + 1], a1, b2, b3);
            }
          }
        }
      }
#pragma unroll
      for (int kk = 0; kk < TR / 16; ++kk) {   // columns 16 wi.. of the tile (rows of S^T) times its T rows
        uint32_t a[4];
        const int row = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4_t(a[0], a[1], a[2], a[3], sS + swz(row, wi * 2 + ((lane >> 3) & 1), 128, 7));
        const int trow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int n = 0; n < NTW; n += 2) {
          uint32_t b0, b1, b2 = 0, b3 = 0;
          if (n + 1 < NTW) ldsm_x4_t(b0, b1, b2, b3, sT + swz(trow, n + (lane >> 4), C::PITCH, C::MASK));
          else ldsm_x2_t(b0, b1, sT + swz(trow, n, C::PITCH, C::MASK));
          mma_bf16_16816(accP[j][n], a, b0, b1);
          if (n + 1 < NTW) mma_bf16_16816(accP[j][n + 1], a, b2, b3);
        }
        if (SUMS) mma_bf16_16816(accS[j], a, ONES, ONES);   // every output column = the column sum
      }
      warp_release(&empty[s], lane);
    }
    if (ROW) {
      // the two groups' row partials of this block meet in shared memory (slot b & 1; a slot is
      // written again two blocks later, after group 0 has passed the next barrier)
      float* slot = red + ((((b & 1) * 4 + wi) * 32 + lane) * 2 * NTW * 4);
      if (grp == 1) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int n = 0; n < NTW; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) slot[(mt * NTW + n) * 4 + e] = accG[mt][n][e];
      }
      named_bar_sync(1, 256);
      if (grp == 0 && ok) {
        float* gp = d.gpart + (int64_t)bn * d.rows * R;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
          for (int n = 0; n < NTW; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) accG[mt][n][e] += slot[(mt * NTW + n) * 4 + e];
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int64_t grow = r0 + (int64_t)b * TR + wi * 32 + mt * 16 + g + hr * 8;
            if (grow >= d.rows) continue;
#pragma unroll
            for (int n = 0; n < NTW; ++n)
              *reinterpret_cast<float2*>(gp + grow * R + n * 8 + 2 * t) =
                  make_float2(accG[mt][n][2 * hr], accG[mt][n][2 * hr + 1]);
          }
        }
      }
    }
  }
  if (!ok) return;

  // ------------------------------------------------------------------ column partials of this row group
  const int64_t ldp = d.ldp > 0 ? d.ldp : R;
  float* part = d.part + ((int64_t)bm * d.K) * ldp + d.j0;
#pragma unroll
  for (int j = 0; j < NCH / 2; ++j) {
    const int64_t kb = (int64_t)c0 + (2 * j + grp) * TC + wi * 16;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int64_t k = kb + g + hr * 8;
      if (k >= d.K) continue;
#pragma unroll
      for (int n = 0; n < NTW; ++n)
        *reinterpret_cast<float2*>(part + k * ldp + n * 8 + 2 * t) = make_float2(accP[j][n][2 * hr], accP[j][n][2 * hr + 1]);
      if (SUMS && t == 0 && d.colsum) d.colsum[(int64_t)bm * d.K + k] = accS[j][2 * hr];
    }
  }
}

RowColPlan rowcol_plan(int64_t rows, int64_t K, int R) {
  RowColPlan p;
  const int64_t pn = (K + rc::CN - 1) / rc::CN;
  const int64_t blocks = (rows + rc::TR - 1) / rc::TR;
  const int64_t sms = num_sms_current();
  // one CTA per SM; cost in tile times: the waves times the longest CTA's tiles plus a ring fill,
  // plus the fp32 partials written in both directions (a 128 x 64 bf16 tile is 16 KB)
  double best = 1e30;
  p.pn = (int)pn;
  p.pm = 1;
  p.nb = (int)(blocks > 0 ? blocks : 1);
  for (int64_t nb = 1; nb <= (blocks > 0 ? blocks : 1); ++nb) {
    const int64_t pm = (blocks + nb - 1) / nb;
    const int64_t waves = (pm * pn + sms - 1) / sms;
    const double partial = 4.0 * R * (double)(pm * K + pn * rows) / (16384.0 * (double)sms);
    const double t = (double)waves * (double)(nb * rc::NCH + 4) + partial;
    if (t < best - 1e-9) {
      best = t;
      p.pm = (int)pm;
      p.nb = (int)nb;
    }
  }
  return p;
}

template <int R, bool ROW, bool SUMS>
static cudaError_t rowcol_launch(const RowColDesc& d, cudaStream_t st) {
  using C = rc::Cfg<R>;
  auto k = rowcol_kernel<R, ROW, SUMS>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    set = true;
  }
  RcParams P;
  memset(&P, 0, sizeof(P));
  P.d = d;
  bool ok = make_tmap_bf16(&P.tmS, d.S, (uint64_t)d.K, (uint64_t)d.rows, (uint64_t)d.lds, rc::TC, rc::TR / 2, 128);
  ok = ok && make_tmap_bf16(&P.tmT, d.T, R, (uint64_t)d.rows, (uint64_t)d.ldt, C::RPAD, rc::TR, C::SWZ);
  if (ROW) ok = ok && make_tmap_bf16(&P.tmU, d.U, R, (uint64_t)d.K, (uint64_t)d.ldu, C::RPAD, rc::CN / 2, C::SWZ);
  else P.tmU = P.tmT;
  if (!ok) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)(d.pm * d.pn), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  // algorithmic HBM bytes: S once, U and T once, the fp32 partials (and column sums)
  const double bytes = 2.0 * d.rows * d.K + 2.0 * R * (d.K + d.rows) +
                       4.0 * R * ((double)d.pm * d.K + (ROW ? (double)d.pn * d.rows : 0.0)) +
                       (SUMS ? 4.0 * d.pm * d.K : 0.0);
  prof_mark(st, true, bytes, 1);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, P);
  prof_mark(st, false, 0.0, 1);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t rowcol(const RowColDesc& d, cudaStream_t st) {
  if (d.rows <= 0 || d.K <= 0) return cudaSuccess;
  if (d.pm <= 0 || d.pn != (int)((d.K + rc::CN - 1) / rc::CN) || d.nb <= 0 ||
      (int64_t)d.pm * d.nb * rc::TR < d.rows || (d.U != nullptr) != (d.gpart != nullptr))
    return cudaErrorInvalidValue;
  const bool row = d.U != nullptr, sums = d.colsum != nullptr;
#define RC_CASE(RR)                                                              \
  case RR:                                                                       \
    if (row) return sums ? rowcol_launch<RR, true, true>(d, st) : rowcol_launch<RR, true, false>(d, st); \
    return sums ? rowcol_launch<RR, false, true>(d, st) : rowcol_launch<RR, false, false>(d, st);
  switch (d.R) {
    RC_CASE(8)
    RC_CASE(16)
    RC_CASE(24)
    RC_CASE(32)
  }
#undef RC_CASE
  return cudaErrorInvalidValue;
}

// out[row][j] (row stride ldo) = bf16(scale * sum_p gpart[p][row][j]) over rows x R elements (R a
// multiple of 8, so a group of four never straddles rows)
__global__ void gpart_sum_kernel(const float* __restrict__ gp, int pn, int64_t n, int R, float scale,
                                 bf16* __restrict__ out, int64_t ldo) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  float4 a = *reinterpret_cast<const float4*>(gp + i);
  for (int p = 1; p < pn; ++p) {
    const float4 v = *reinterpret_cast<const float4*>(gp + (int64_t)p * n + i);
    a.x += v.x;
    a.y += v.y;
    a.z += v.z;
    a.w += v.w;
  }
  *reinterpret_cast<uint2*>(out + (i / R) * ldo + i % R) =
      make_uint2(pack_bf16x2(scale * a.x, scale * a.y), pack_bf16x2(scale * a.z, scale * a.w));
}

cudaError_t gpart_sum(const float* gpart, int pn, int64_t rows, int R, float scale, bf16* out, int64_t ldo,
                      cudaStream_t st) {
  const int64_t n = rows * R;
  if (n <= 0) return cudaSuccess;
  if (R % 8 || pn <= 0 || ldo < R || ldo % 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)((n / 4 + 255) / 256), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_attr(&attr[0]);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gpart_sum_kernel, gpart, pn, n, R, scale, out, ldo);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lg

// Persistent, warp-specialised tcgen05 GEMM engine for sm_103a.
//
//   D[M, N] = A0[M, K0] * op(B0)  +  A1[M, K1] * op(B1)        (fp32 in TMEM, bf16 out)
//
// The first term is the dense base contraction (X W0^T forward, dY W0 backward); the
// optional second ("tail") term is the rank-r up-projection applied as one more K-step of
// tcgen05 MMAs into the same accumulator (s Z B^T forward, s G A backward).  This is how
// the low-rank update is folded into the data GEMM without ever forming B A
// ("LoRA/DoRA fast forward: no weight materialization", What section).
//
// The kernels share the tile shape and the epilogues:
//  * tc_gemm_kernel: one CTA per SM, 128 x 256 tile (cta_group::1).
//  * tc_pair_kernel: a cluster of two CTAs on two SMs computes a 256 x 256 tile with
//    cta_group::2 MMAs issued by the even CTA; each SM stages its 128 rows of A and half of
//    B, so the operand bytes per SM and k-step drop from 48 KB to 32 KB.
//  * tc_gemm_kernel in K-scaling mode: the MN-major dX product whose A operand is scaled along
//    K on its way into shared memory (the DoRA backward's dY o c; see OneCta).
// Roles (per CTA, 6 or 10 warps):
//   warp 0      TMA producer into a STAGES-deep ring of 128B-swizzled tiles
//   warp 1      TMEM allocator; MMA issuer (one thread; in the pair kernel, the even CTA's)
//   warps 2..5  epilogue: TMEM -> registers -> (row scale, bias, SwiGLU) -> bf16 ->
//               swizzled SMEM staging -> TMA store
//   warps 6..9  the plain scale/bias epilogue: second half of each accumulator
// Every mbarrier wait is bounded (global timer); on expiry the CTA records the error in
// the caller's error word, lets its in-flight copies and MMAs finish, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

namespace lg {

struct TcParams {
  CUtensorMap tmA0, tmB0, tmB0b, tmA1, tmB1, tmB1b;
  CUtensorMap tmOut[3];
  int M, N, K0, K1;
  int num_m_tiles, num_n_tiles, group_m;
  int k0_split_steps;   // MN-major B0: k-steps taken from tmB0 before switching to tmB0b
  int tail_b1b_x;       // stacked tail: x coordinate (K shift) of the second half
  int tail_b1_x;        // stacked tail: x coordinate of the first half
  const float* col_scale;
  const bf16* bias;
  const float* a_kscale;
  const bf16* e_in;
  const bf16* u_in;
  int ld_eu;
  const float* sx;      // W8A8: per-row activation scales [M]
  const float* sw;      // W8A8: per-column weight scales [N]
  float ls;             // W8A8: scale of the rank-r term
  int32_t* acc_out;     // W8A8: raw int32 product [M, N] (or null)
  int kc_steps;         // W8A8 chunked: K-steps per exactly summed chunk
  int write_y;          // W8A8: 0 when only the raw product is wanted
  int pair_leader_arms; // CTA pair: the leader posts the transaction bytes of both CTAs
  int act;              // gated MLP activation: 0 SwiGLU, 1 GeGLU
  // down-projection in the GEMM (forward): Z = A0 dn_a^T from the staged A0 tiles, the tail's A
  // operand bf16(dn_s Z) written into the tail stage, bf16(Z) to dn_z (the tiles of N-tile 0)
  const bf16* dn_a;
  int64_t dn_lda;
  float dn_s;
  int dn_r;
  bf16* dn_z;
  uint32_t* err;
  uint64_t timeout_ns;
};

constexpr int BM = 128;     // rows of A per CTA
constexpr int BN = 256;     // accumulator columns per tile
constexpr int BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB

template <int EPI, bool PAIR>
struct EpiCfg;
template <> struct EpiCfg<EPI_SCALE_BIAS, false> { static constexpr int STAGES = 4, STG_BUFS = 2; };
template <> struct EpiCfg<EPI_SWIGLU, false> { static constexpr int STAGES = 3, STG_BUFS = 3; };
template <> struct EpiCfg<EPI_SWIGLU_BWD, false> { static constexpr int STAGES = 4, STG_BUFS = 2; };
template <> struct EpiCfg<EPI_SCALE_BIAS, true> { static constexpr int STAGES = 6, STG_BUFS = 2; };
template <> struct EpiCfg<EPI_SWIGLU, true> { static constexpr int STAGES = 5, STG_BUFS = 3; };
template <> struct EpiCfg<EPI_SWIGLU_BWD, true> { static constexpr int STAGES = 6, STG_BUFS = 2; };
template <> struct EpiCfg<EPI_W8A8K, false> { static constexpr int STAGES = 4, STG_BUFS = 2; };
template <> struct EpiCfg<EPI_W8A8K, true> { static constexpr int STAGES = 6, STG_BUFS = 2; };

template <int EPI, bool PAIR, bool KSCALE = false>
struct Layout {
  static constexpr int STAGES = EpiCfg<EPI, PAIR>::STAGES;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;        // B rows (N) staged by one CTA
  static constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
  static constexpr int OFF_STG = OFF_B + STAGES * B_STAGE_BYTES;
  static constexpr int STG_BYTES = 4 * EpiCfg<EPI, PAIR>::STG_BUFS * 4096;
  static constexpr int KSC_BYTES = BK * 4;                  // K-scaling: a stage's 64 fp32 scales
  static constexpr int OFF_KSC = OFF_STG + STG_BYTES;
  static constexpr int OFF_BAR = OFF_KSC + (KSCALE ? STAGES * KSC_BYTES : 0);
  static constexpr int BAR_BYTES = 8 * (3 * STAGES + 5) + 16;
  static constexpr int TOTAL = OFF_BAR + BAR_BYTES + 1024;  // +1024 for base alignment
  static_assert(TOTAL <= 232448, "shared memory budget");
};

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mt, int& nt) {
  const int group_size = group_m * num_n;
  const int g = t / group_size;
  const int first_m = g * group_m;
  const int gm = min(num_m - first_m, group_m);
  const int r = t - g * group_size;
  mt = first_m + r % gm;
  nt = r / gm;
}

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }

// Write 16 words (32 bf16 = four 16-byte chunks) of one row into a 128B-swizzled 32-row
// staging tile: logical chunk jbase + j of row `row` goes to physical chunk (jbase+j) ^ (row & 7).
__device__ __forceinline__ void stage_row(uint8_t* stg, int row, const uint32_t* w, int jbase) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = jbase + j;
    uint4 v = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    *reinterpret_cast<uint4*>(stg + row * 128 + ((jj ^ (row & 7)) << 4)) = v;
  }
}

// ---------------------------------------------------------------------------- gated activations
// act 0: silu(e) = e sigmoid(e); act 1: gelu(e) = e Phi(e) with the normal CDF
// Phi(e) = (1 + erf(e / sqrt 2)) / 2 (CUDA's expf / erff are called, not re-implemented).
__device__ __forceinline__ float gate_act(float e, int act) {
  if (act == 0) return e / (1.0f + __expf(-e));
  return 0.5f * e * (1.0f + erff(e * 0.70710678118654752f));
}
// a = act(e) and its derivative da
__device__ __forceinline__ void gate_act_grad(float e, int act, float& a, float& da) {
  if (act == 0) {
    const float sg = 1.0f / (1.0f + __expf(-e));
    a = e * sg;
    da = sg * (1.0f + e * (1.0f - sg));
  } else {
    const float cdf = 0.5f * (1.0f + erff(e * 0.70710678118654752f));
    a = e * cdf;
    da = cdf + e * 0.39894228040143268f * __expf(-0.5f * e * e);  // + e * N(0,1) density
  }
}

// ---------------------------------------------------------------------------- epilogue of one tile
// One warp drains its 32 TMEM lanes (rows row0 .. row0 + 31) of the accumulator at t_row.
template <int EPI, int N_OUT>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, uint32_t t_row, int row0, int n0, int lane,
                                              uint8_t* my_stg, uint32_t& chunk_ctr) {
  if constexpr (EPI == EPI_SCALE_BIAS) {
#pragma unroll 1
    for (int c = 0; c < N_OUT / 64; ++c, ++chunk_ctr) {
      // a whole-tile epilogue warp double-buffers its staging; a half-tile one has a single buffer
      uint8_t* stg = my_stg + (N_OUT == BN ? (chunk_ctr & 1) * 4096 : 0);
      if (lane == 0) {
        if (N_OUT == BN) tma_store_wait_read<1>();
        else tma_store_wait_read<0>();
      }
      __syncwarp();
      uint32_t v[32];
      uint32_t w[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld_32x32b_x32(t_row + c * 64 + h * 32, v);
        tmem_ld_wait();
        const int col = n0 + c * 64 + h * 32;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float f0 = u2f(v[j]), f1 = u2f(v[j + 1]);
          if (p.col_scale != nullptr && col + j < p.N) {
            f0 *= __ldg(p.col_scale + col + j);
            f1 *= __ldg(p.col_scale + col + j + 1);
          }
          if (p.bias != nullptr && col + j < p.N) {
            f0 += __bfloat162float(p.bias[col + j]);
            f1 += __bfloat162float(p.bias[col + j + 1]);
          }
          w[h * 16 + j / 2] = pack_bf16x2(f0, f1);
        }
      }
      stage_row(stg, lane, w, 0);
      stage_row(stg, lane, w + 16, 4);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmOut[0], stg, n0 + c * 64, row0);
        tma_store_commit();
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // accumulator columns [0, BN/2) hold e, [BN/2, BN) hold u for outputs n0 .. n0 + BN/2
#pragma unroll 1
    for (int c = 0; c < N_OUT / 64; ++c) {
      uint8_t* se = my_stg;
      uint8_t* su = my_stg + 4096;
      uint8_t* sh = my_stg + 8192;
      if (lane == 0) tma_store_wait_read<0>();
      __syncwarp();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t ve[32], vu[32];
        tmem_ld_32x32b_x32(t_row + c * 64 + h * 32, ve);
        tmem_ld_32x32b_x32(t_row + BN / 2 + c * 64 + h * 32, vu);
        tmem_ld_wait();
        uint32_t we[16], wu[16], wh[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float e0 = u2f(ve[j]), e1 = u2f(ve[j + 1]);
          const float u0 = u2f(vu[j]), u1 = u2f(vu[j + 1]);
          const float h0 = gate_act(e0, p.act) * u0;
          const float h1 = gate_act(e1, p.act) * u1;
          we[j / 2] = pack_bf16x2(e0, e1);
          wu[j / 2] = pack_bf16x2(u0, u1);
          wh[j / 2] = pack_bf16x2(h0, h1);
        }
        stage_row(se, lane, we, h * 4);
        stage_row(su, lane, wu, h * 4);
        stage_row(sh, lane, wh, h * 4);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmOut[0], se, n0 + c * 64, row0);
        tma_store_2d(&p.tmOut[1], su, n0 + c * 64, row0);
        tma_store_2d(&p.tmOut[2], sh, n0 + c * 64, row0);
        tma_store_commit();
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU_BWD) {
    // accumulator = dh; read the saved e, u for this thread's row and form de, du.  The e, u
    // values of the next 32-column slice are loaded while the current one is being processed.
    const int grow = row0 + lane;
    uint32_t ev[16], uv[16], en[16], un[16];
    auto load_eu = [&](int slice, uint32_t* e_, uint32_t* u_) {
      const int col = n0 + slice * 32;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int cc = col + 8 * g;
        if (grow < p.M && cc < p.N) {
          const uint4 a = *reinterpret_cast<const uint4*>(p.e_in + (size_t)grow * p.ld_eu + cc);
          const uint4 b = *reinterpret_cast<const uint4*>(p.u_in + (size_t)grow * p.ld_eu + cc);
          e_[4 * g] = a.x; e_[4 * g + 1] = a.y; e_[4 * g + 2] = a.z; e_[4 * g + 3] = a.w;
          u_[4 * g] = b.x; u_[4 * g + 1] = b.y; u_[4 * g + 2] = b.z; u_[4 * g + 3] = b.w;
        } else {
#pragma unroll
          for (int z = 0; z < 4; ++z) e_[4 * g + z] = u_[4 * g + z] = 0u;
        }
      }
    };
    load_eu(0, ev, uv);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c, ++chunk_ctr) {
      // one staging pair per warp (it buys the GEMM a deeper operand ring): the previous chunk's
      // stores must have read it before it is overwritten
      uint8_t* sde = my_stg;
      uint8_t* sdu = sde + 4096;
      if (lane == 0) tma_store_wait_read<0>();
      __syncwarp();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int slice = c * 2 + h;
        if (slice + 1 < BN / 32) load_eu(slice + 1, en, un);
        uint32_t vd[32];
        tmem_ld_32x32b_x32(t_row + c * 64 + h * 32, vd);
        tmem_ld_wait();
        uint32_t wde[16], wdu[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 e = unpack_bf16x2(ev[j]);
          const float2 u = unpack_bf16x2(uv[j]);
          const float d0 = u2f(vd[2 * j]), d1 = u2f(vd[2 * j + 1]);
          float a0, da0, a1, da1;
          gate_act_grad(e.x, p.act, a0, da0);
          gate_act_grad(e.y, p.act, a1, da1);
          const float de0 = d0 * u.x * da0;
          const float de1 = d1 * u.y * da1;
          const float du0 = d0 * a0;
          const float du1 = d1 * a1;
          wde[j] = pack_bf16x2(de0, de1);
          wdu[j] = pack_bf16x2(du0, du1);
        }
        stage_row(sde, lane, wde, h * 4);
        stage_row(sdu, lane, wdu, h * 4);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          ev[j] = en[j];
          uv[j] = un[j];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmOut[0], sde, n0 + c * 64, row0);
        tma_store_2d(&p.tmOut[1], sdu, n0 + c * 64, row0);
        tma_store_commit();
      }
    }
  }
}

// Chunked W8A8 epilogue of one warp's 32 rows x 128 columns once the exact int32 sums S of its row
// are complete: the raw product to acc_out and/or y = S sx sw (+ s T, the rank-r term read from TMEM
// at t_cols, when TAIL) (+ bias), bf16 through the warp's 32 x 64 staging buffer.
template <bool TAIL>
__device__ __forceinline__ void w8k_final(const TcParams& p, const int (&S)[128], uint32_t t_cols, int row0, int col0,
                                          int lane, uint8_t* stg) {
  const int grow = row0 + lane;
  const bool row_ok = grow < p.M;
  if (p.acc_out != nullptr && row_ok) {
#pragma unroll
    for (int g = 0; g < 32; ++g)
      if (col0 + 4 * g < p.N)
        *reinterpret_cast<int4*>(p.acc_out + (size_t)grow * p.N + col0 + 4 * g) =
            make_int4(S[4 * g], S[4 * g + 1], S[4 * g + 2], S[4 * g + 3]);
  }
  if (!p.write_y) return;
  const float rs = row_ok ? p.sx[grow] : 0.f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {   // unrolled: S is indexed by constants only and stays in registers
    if (lane == 0) tma_store_wait_read<0>();   // the previous chunk's store has read the buffer
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 4; ++h) {   // 16 columns at a time: two 16-byte chunks of the staged row
      uint32_t v[16];
      if (TAIL) {
        tmem_ld_32x32b_x16(t_cols + c * 64 + h * 16, v);
        tmem_ld_wait();
      }
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        float y2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int col = col0 + c * 64 + h * 16 + j + k;
          float y = 0.f;
          if (col < p.N) {
            y = (float)S[c * 64 + h * 16 + j + k] * rs * __ldg(p.sw + col);
            if (TAIL) y += p.ls * u2f(v[j + k]);
            if (p.bias != nullptr) y += __bfloat162float(p.bias[col]);
          }
          y2[k] = y;
        }
        w[j / 2] = pack_bf16x2(y2[0], y2[1]);
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int ch = 2 * h + jj;
        *reinterpret_cast<uint4*>(stg + lane * 128 + ((ch ^ (lane & 7)) << 4)) =
            make_uint4(w[4 * jj], w[4 * jj + 1], w[4 * jj + 2], w[4 * jj + 3]);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&p.tmOut[0], stg, col0 + c * 64, row0);
      tma_store_commit();
    }
  }
}

// Multiply one staged 128 x 64 A tile (128B-swizzled) in place by the 64 scales of its K range
// (staged in shared memory with the tile), then make the writes visible to the tensor core.
// Thread tid of the 128 scaling threads owns physical 16-byte chunk pc = tid & 7 of rows
// tid / 8 + 16 i (i < 8); all of them have the same (row & 7), hence the same logical K-chunk and
// the same 8 scales.
__device__ __forceinline__ void kscale_tile_inplace(uint8_t* a_tile, const float* sc64, int tid) {
  const int pc = tid & 7;
  const int j = pc ^ ((tid >> 3) & 7);
  const float4 lo = reinterpret_cast<const float4*>(sc64)[2 * j];
  const float4 hi = reinterpret_cast<const float4*>(sc64)[2 * j + 1];
  const float sc[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint4* ptr = reinterpret_cast<uint4*>(a_tile + ((tid >> 3) + 16 * i) * 128 + pc * 16);
    uint4 v = *ptr;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_bf16x2(w[e]);
      w[e] = pack_bf16x2(f.x * sc[2 * e], f.y * sc[2 * e + 1]);
    }
    *ptr = v;
  }
  fence_proxy_async_smem();   // visible to the tensor core (async proxy) before the hand-over
}

// ============================================================================ 1-CTA kernel
// Threads of the one-CTA kernel: producer, MMA and 4 epilogue warps; for the plain scale/bias
// epilogue 4 more warps drain the second half of each accumulator (8 epilogue warps, two per
// TMEM lane quarter, finish a tile's epilogue in half the time).
//
// K-scaling mode (DoRA backward, dX = (dY o c) W0 + s G A): the producer brings each main
// step's raw dY tile and, by a plain bulk copy, the 64 scales of its K range into the stage;
// 4 scaling warps (warps 6..9) then multiply the tile in place, 16-byte chunk by chunk, and hand
// the stage to the MMA through `ready` (one arrival per warp, made by its lane 0; rank-r tail
// stages pass through unscaled).  No scaled copy of dY exists anywhere.  The scaling reads and
// writes every A tile once more in shared memory.  It runs on the one-CTA kernel (the CTA pair
// with the same scaling warps measured 1.7x slower).
template <int EPI, bool KSCALE = false, bool ZF = false>
struct OneCta {
  static constexpr bool EPI8 = (EPI == EPI_SCALE_BIAS || EPI == EPI_W8A8K) && !KSCALE;
  static constexpr int THREADS = ((KSCALE || EPI8) ? 320 : 192) + (ZF ? 128 : 0);
};

template <bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE = false, bool ZF = false>
__global__ void __launch_bounds__(OneCta<EPI, KSCALE, ZF>::THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  static_assert(!KSCALE || (EPI == EPI_SCALE_BIAS && !STACKED), "K-scaling: plain dX products only");
  static_assert(!ZF || (EPI == EPI_SCALE_BIAS && !STACKED && !B0_MN && HAS_TAIL && !B1_MN && !KSCALE),
                "down-projection in the GEMM: the plain forward only");
  using C = OneCta<EPI, KSCALE, ZF>;
  using L = Layout<EPI, false, KSCALE>;
  constexpr int STAGES = L::STAGES;
  constexpr int BNB = STACKED ? BN / 2 : BN;          // rows per K-major B box
  constexpr int N_OUT = STACKED ? BN / 2 : BN;        // logical output columns per tile
  constexpr uint32_t TMEM_COLS = 2 * BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + L::OFF_A;
  uint8_t* sB = smem + L::OFF_B;
  uint8_t* sStg = smem + L::OFF_STG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* ready = bars + 2 * STAGES;   // K-scaling: the stage's A tile is scaled
  uint64_t* acc_full = bars + 3 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nk0 = (p.K0 + BK - 1) / BK;
  const int nk = nk0 + (HAS_TAIL ? (p.K1 + BK - 1) / BK : 0);   // the rank-r tail may span several K-steps
  const int t_first = (int)blockIdx.x;
  const int t_step = (int)gridDim.x;
  const int t_count = p.num_m_tiles * p.num_n_tiles;
  auto coords = [&](int t, int& mt, int& nt) { tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // down-projection: full = the producer's two arrivals on a main step, or its one plus the
      // Z warps' on the tail step; empty = the MMA commit plus the four Z warps
      mbar_init(&full[i], ZF ? 2 : 1);
      mbar_init(&empty[i], ZF ? 5 : 1);
      mbar_init(&ready[i], 4);    // K-scaling: one arrival per scaling warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], C::EPI8 ? 8 : 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA0);
    tma_prefetch_desc(&p.tmB0);
    if (HAS_TAIL) {
      tma_prefetch_desc(&p.tmA1);
      tma_prefetch_desc(&p.tmB1);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();      // the operands may come from the previous kernel in the stream
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;         // bit s: stage s has been armed at least once
      uint32_t armed_par = 0;     // bit s: parity of the last arm of stage s
      bool ok = true;
      for (int t = t_first; t < t_count && ok; t += t_step) {
        int mt, nt;
        coords(t, mt, nt);
        const int m0 = mt * BM;
        const int n0 = nt * N_OUT;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x101)) {
            ok = false;
            break;
          }
          const bool tail = HAS_TAIL && ks >= nk0;
          // the W8A8 tail stages only the rank-r B rows of this tile (no second stacked half); a
          // K-scaled main step also brings the 64 scales of its K range
          if constexpr (ZF) {   // the tail's A operand is written by the Z warps, not copied
            mbar_expect_tx(&full[stage], tail ? L::B_STAGE_BYTES : L::STAGE_BYTES);
            if (!tail) mbar_arrive(&full[stage]);
          } else {
            mbar_expect_tx(&full[stage], (KSCALE && !tail) ? L::STAGE_BYTES + L::KSC_BYTES : L::STAGE_BYTES);
          }
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * A_STAGE_BYTES;
          uint8_t* b_dst = sB + stage * L::B_STAGE_BYTES;
          if (!tail) {
            const int kx = ks * BK;
            if constexpr (KSCALE)   // the 64 scales of this K range (zero past K0)
              bulk_load(smem + L::OFF_KSC + stage * L::KSC_BYTES, p.a_kscale + kx, L::KSC_BYTES, &full[stage]);
            tma_load_2d(a_dst, &p.tmA0, &full[stage], kx, m0);
            if (B0_MN) {
              const bool second = ks >= p.k0_split_steps;
              const void* mp = second ? (const void*)&p.tmB0b : (const void*)&p.tmB0;
              const int ky = second ? kx - p.k0_split_steps * BK : kx;
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * 8192, mp, &full[stage], n0 + 64 * j, ky);
            } else if (STACKED) {
              tma_load_2d(b_dst, &p.tmB0, &full[stage], kx, n0);
              tma_load_2d(b_dst + BNB * 128, &p.tmB0b, &full[stage], kx, n0);
            } else {
              tma_load_2d(b_dst, &p.tmB0, &full[stage], kx, n0);
            }
          } else {
            const int kt = (ks - nk0) * BK;   // K offset inside the rank-r tail
            if (!ZF) tma_load_2d(a_dst, &p.tmA1, &full[stage], kt, m0);
            if (B1_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * 8192, &p.tmB1, &full[stage], n0 + 64 * j, kt);
            } else if (STACKED) {
              tma_load_2d(b_dst, &p.tmB1, &full[stage], p.tail_b1_x + kt, n0);
              tma_load_2d(b_dst + BNB * 128, &p.tmB1b, &full[stage], p.tail_b1b_x + kt, n0);
            } else {
              tma_load_2d(b_dst, &p.tmB1, &full[stage], kt, n0);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // unwind: let every copy this thread issued land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) mbar_wait_drain(&full[s], (armed_par >> s) & 1u, 20000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && EPI == EPI_W8A8K) {
      // chunked W8A8: each chunk of kc_steps K-steps (and the rank-r tail) in its own accumulator,
      // the two accumulators alternating across chunks and tiles
      constexpr uint32_t idesc = umma_idesc_bf16(BM, BN, 0, 0);
      const int kc = p.kc_steps;
      const int nch = (nk0 + kc - 1) / kc;
      const int nchunks = nch + (HAS_TAIL ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t u = 0;
      for (int t = t_first; t < t_count && ok; t += t_step) {
        for (int c = 0; c < nchunks && ok; ++c, ++u) {
          const int buf = (int)(u & 1);
          const uint32_t aph = (u >> 1) & 1;
          if (!mbar_wait(&acc_empty[buf], aph ^ 1, p.timeout_ns, abort_flag, p.err, 0x102)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int k_begin = c < nch ? c * kc : nk0;
          const int k_end = c < nch ? min(nk0, (c + 1) * kc) : nk;
          for (int ks = k_begin; ks < k_end; ++ks) {
            if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x103)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
            const uint32_t b_base = smem_u32(sB + stage * L::B_STAGE_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16(d_tmem, umma_smem_desc(a_base + kk * 32, 16, 1024), umma_smem_desc(b_base + kk * 32, 16, 1024),
                        idesc, (ks > k_begin || kk > 0) ? 1u : 0u);
            umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(&acc_full[buf]);
        }
      }
      umma_commit(drain);
      mbar_wait_drain(drain, 0, 20000000ull);
    } else if (lane == 0) {
      constexpr uint32_t idesc0 = umma_idesc_bf16(BM, BN, 0, B0_MN ? 1 : 0);
      constexpr uint32_t idesc1 = umma_idesc_bf16(BM, BN, 0, B1_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = t_first; t < t_count && ok; t += t_step, ++it) {
        const int buf = it & 1;
        const uint32_t acc_phase = (uint32_t)((it >> 1) & 1);
        if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x102)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int ks = 0; ks < nk; ++ks) {
          const bool tail = HAS_TAIL && ks >= nk0;
          if (!mbar_wait(KSCALE ? &ready[stage] : &full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x103)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * L::B_STAGE_BYTES);
          // a fixed count of BK / 16 MMAs per stage, the rank-r tail included: TMA fills the tail
          // tile's columns past the rank with zeros on both operands, so the padding adds exact
          // zeros, and a count that depends on the data made the whole GEMM 6-13% slower
          const bool bmn = tail ? B1_MN : B0_MN;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = umma_smem_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = bmn ? umma_smem_desc(b_base + kk * 2048, 8192, 1024)
                                       : umma_smem_desc(b_base + kk * 32, 16, 1024);
            umma_bf16(d_tmem, adesc, bdesc, tail ? idesc1 : idesc0, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[buf]);
      }
      // make sure no MMA is still reading SMEM / writing TMEM before teardown
      umma_commit(drain);
      mbar_wait_drain(drain, 0, 20000000ull);
    }
    __syncwarp();
  } else if (warp < (C::EPI8 ? 10 : 6)) {
    // ---------------------------------------------------------------- epilogue
    constexpr bool EPI8 = C::EPI8;
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = EPI8 ? (warp - 2) >> 2 : 0;   // with 8 warps: which half of the columns
    uint8_t* my_stg = sStg + (warp - 2) * (EPI8 ? 4096 : EpiCfg<EPI, false>::STG_BUFS * 4096);
    int it = 0;
    uint32_t chunk_ctr = 0;
    if constexpr (EPI == EPI_W8A8K) {
      // chunked W8A8: every integer chunk is added to the row's int32 sums S, held in registers
      // (exact: each chunk's fp32 sum is an integer below 2^24); the tail chunk (or, without one, the
      // last integer chunk) closes the tile.  Warp (q, half): rows 32q.., columns 128 half..
      const int kc = p.kc_steps;
      const int nch = (nk0 + kc - 1) / kc;
      const int nchunks = nch + (HAS_TAIL ? 1 : 0);
      const uint32_t lanes = tmem_base + ((uint32_t)(32 * q) << 16) + half * (BN / 2);
      uint32_t u = 0;
      bool ok = true;
      for (int t = t_first; t < t_count && ok; t += t_step) {
        int mt, nt;
        coords(t, mt, nt);
        const int row0 = mt * BM + 32 * q;
        const int col0 = nt * BN + half * (BN / 2);
        int S[128];
#pragma unroll
        for (int j = 0; j < 128; ++j) S[j] = 0;
        for (int c = 0; c < nchunks; ++c, ++u) {
          const int buf = (int)(u & 1);
          const uint32_t aph = (u >> 1) & 1;
          if (!mbar_wait(&acc_full[buf], aph, p.timeout_ns, abort_flag, p.err, 0x104)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t c_cols = lanes + buf * BN;
          if (c < nch) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t v[16];
              tmem_ld_32x32b_x16(c_cols + j * 16, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) S[j * 16 + e] += __float2int_rn(u2f(v[e]));
            }
          } else {
            w8k_final<true>(p, S, c_cols, row0, col0, lane, my_stg);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (!ok) break;
        if (!HAS_TAIL) w8k_final<false>(p, S, 0, row0, col0, lane, my_stg);
      }
      if (lane == 0) tma_store_wait_all<0>();
      __syncwarp();
    } else
    for (int t = t_first; t < t_count; t += t_step, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (uint32_t)((it >> 1) & 1);
      if (!mbar_wait(&acc_full[buf], acc_phase, p.timeout_ns, abort_flag, p.err, 0x104)) break;
      tc_fence_after();
      int mt, nt;
      coords(t, mt, nt);
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + buf * BN + half * (N_OUT / 2);
      if constexpr (EPI8)
        epilogue_tile<EPI, N_OUT / 2>(p, t_row, mt * BM + 32 * q, nt * N_OUT + half * (N_OUT / 2), lane, my_stg,
                                      chunk_ctr);
      else
        epilogue_tile<EPI, N_OUT>(p, t_row, mt * BM + 32 * q, nt * N_OUT, lane, my_stg, chunk_ctr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  } else if (KSCALE) {
    // ---------------------------------------------------------------- A-tile K-scaling in place
    const int tid = threadIdx.x - 192;   // 0 .. 127
    const float* sKsc = reinterpret_cast<const float*>(smem + L::OFF_KSC);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = t_first; t < t_count && ok; t += t_step) {
      for (int ks = 0; ks < nk; ++ks) {
        if (lane == 0) ok = mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x105);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (!(HAS_TAIL && ks >= nk0))   // the rank-r tail is not scaled
          kscale_tile_inplace(sA + stage * A_STAGE_BYTES, sKsc + stage * BK, tid);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (ZF) {
    // ---------------------------------------------------------------- down-projection Z = A0 dn_a^T
    // Z warp zw forms rows 32 zw .. 32 zw + 31 of the tile's Z with the warp MMA straight from each
    // staged (128B-swizzled) A0 tile; the dn_a fragments come from global memory (L1/L2 resident),
    // loaded while the next stage is awaited.  On the tail step it writes bf16(dn_s Z) as that step's A operand (zeros past
    // the rank) once the stage is free, and bf16(Z) to dn_z for the tiles of N-tile 0.
    const int zw = warp - 10;
    const int g = lane >> 2, t4 = lane & 3;
    const int nzt = p.dn_r / 8;              // n-tiles of 8 (rank 8 .. 32)
    const int64_t K0 = p.K0;
    auto load_b = [&](int ks, uint32_t (&b)[4][4][2]) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const int64_t k = (int64_t)ks * BK + kk * 16 + 2 * t4;
          const bf16* row = p.dn_a + (int64_t)(n * 8 + g) * p.dn_lda;
          const bool okn = n < nzt;
          b[kk][n][0] = (okn && k < K0) ? __ldg(reinterpret_cast<const uint32_t*>(row + k)) : 0u;
          b[kk][n][1] = (okn && k + 8 < K0) ? __ldg(reinterpret_cast<const uint32_t*>(row + k + 8)) : 0u;
        }
    };
    // After a failed wait a warp keeps stepping through its tiles without waiting or working, so
    // that all four still meet at the named barrier of every tail step.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = t_first; t < t_count; t += t_step) {
      int mt, nt;
      coords(t, mt, nt);
      float acc[2][4][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
      uint32_t bcur[4][4][2];
      if (ok) load_b(0, bcur);
      for (int ks = 0; ks < nk0; ++ks) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x106));
        if (ok) {
          const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int row = zw * 32 + i * 16 + (lane & 15);
              const int ch = kk * 2 + (lane >> 4);
              uint32_t a[4];
              ldsm_x4(a[0], a[1], a[2], a[3], a_base + row * 128 + ((ch ^ (row & 7)) << 4));
#pragma unroll
              for (int n = 0; n < 4; ++n)
                if (n < nzt) mma_bf16_16816(acc[i][n], a, bcur[kk][n][0], bcur[kk][n][1]);
            }
          }
          warp_release(&empty[stage], lane);
          // the next K-step's fragments, issued after the release so that its fence does not wait
          // for them
          if (ks + 1 < nk0) load_b(ks + 1, bcur);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      // the tail step: the stage must be free (its previous MMA done) before it is written
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x107));
      uint8_t* a_tile = sA + stage * A_STAGE_BYTES;
      if (ok) {
        const bool save = p.dn_z != nullptr && nt == 0;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int row = zw * 32 + i * 16 + g + 8 * hr;
            const int64_t grow = (int64_t)mt * BM + row;
#pragma unroll
            for (int n = 0; n < 4; ++n) {
              if (n >= nzt) continue;
              const float z0 = acc[i][n][2 * hr], z1 = acc[i][n][2 * hr + 1];
              const int col = n * 8 + 2 * t4;
              *reinterpret_cast<uint32_t*>(a_tile + row * 128 + ((n ^ (row & 7)) << 4) + (col & 7) * 2) =
                  pack_bf16x2(z0 * p.dn_s, z1 * p.dn_s);
              if (save && grow < p.M)
                *reinterpret_cast<uint32_t*>(p.dn_z + grow * p.dn_r + col) = pack_bf16x2(z0, z1);
            }
          }
        const int row = zw * 32 + lane;   // 16-byte chunks past the rank read as zeros
        for (int c = nzt; c < 8; ++c)
          *reinterpret_cast<uint4*>(a_tile + row * 128 + ((c ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();   // visible to the tensor core before the MMA is released
      }
      const bool all_ok = named_bar_or(2, 128, !ok) == false;
      if (all_ok && zw == 0 && lane == 0) mbar_arrive(&full[stage]);
      if (ok) warp_release(&empty[stage], lane);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ============================================================================ CTA-pair kernel
// Cluster of 2: CTA rank 0 (leader) issues cta_group::2 MMAs of M = 256 (its 128 rows of A in
// its SMEM, the peer's 128 rows in the peer's) x N = 256 (B columns 0..127 from the leader's
// SMEM, 128..255 from the peer's); each CTA's TMEM receives its own 128 rows of D.
//   full[s]      leader: 2 arrivals (both producers' expect_tx) + both CTAs' TMA bytes
//   empty[s]     both CTAs: the leader's MMA commit, multicast to the pair
//   acc_full[b]  both CTAs: the leader's MMA commit, multicast
//   acc_empty[b] leader: 4 epilogue warps (8 for the plain scale/bias epilogue) x 2 CTAs
template <bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE = false>
__global__ void __launch_bounds__(OneCta<EPI, KSCALE>::THREADS, 1) tc_pair_kernel(const __grid_constant__ TcParams p) {
  static_assert(!KSCALE || (EPI == EPI_SCALE_BIAS && !STACKED), "K-scaling: plain dX products only");
  using C = OneCta<EPI, KSCALE>;
  using L = Layout<EPI, true, KSCALE>;
  constexpr int STAGES = L::STAGES;
  constexpr int N_OUT = STACKED ? BN / 2 : BN;        // logical output columns per tile
  constexpr uint32_t TMEM_COLS = 2 * BN;
  constexpr int PM = 2 * BM;                          // rows per pair tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + L::OFF_A;
  uint8_t* sB = smem + L::OFF_B;
  uint8_t* sStg = smem + L::OFF_STG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* ready = bars + 2 * STAGES;   // K-scaling (leader): both CTAs' A tiles are scaled
  uint64_t* acc_full = bars + 3 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;   // pair tiles (256 rows each)
  const int nk0 = (p.K0 + BK - 1) / BK;
  const int nk = nk0 + (HAS_TAIL ? (p.K1 + BK - 1) / BK : 0);   // the rank-r tail may span several K-steps

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // K-scaling: each CTA's own loads on its own barrier, waited by its scaling warps
      mbar_init(&full[i], (KSCALE || p.pair_leader_arms) ? 1 : 2);
      mbar_init(&empty[i], 1);
      mbar_init(&ready[i], 8);   // K-scaling: 4 scaling warps x 2 CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], C::EPI8 ? 16 : 8);   // epilogue warps x 2 CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA0);
    tma_prefetch_desc(&p.tmB0);
    if (HAS_TAIL) {
      tma_prefetch_desc(&p.tmA1);
      tma_prefetch_desc(&p.tmB1);
    }
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates the pair's TMEM columns
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();      // the operands may come from the previous kernel in the stream
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
        int mt, nt;
        tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
        const int m0 = mt * PM + (int)rank * BM;
        const int n0 = nt * N_OUT;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait_cl(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x201)) {
            ok = false;
            break;
          }
          const bool tail = HAS_TAIL && ks >= nk0;
          uint32_t bar;
          if constexpr (KSCALE) {   // this CTA's bytes (and the scales of a main step) on its own barrier
            mbar_expect_tx(&full[stage], L::STAGE_BYTES + (tail ? 0 : L::KSC_BYTES));
            bar = mapa_shared(smem_u32(&full[stage]), rank);
            if (!tail)
              bulk_load(smem + L::OFF_KSC + stage * L::KSC_BYTES, p.a_kscale + ks * BK, L::KSC_BYTES, &full[stage]);
          } else {
            bar = mapa_shared(smem_u32(&full[stage]), 0);
            if (!p.pair_leader_arms) mbar_expect_tx_cluster(bar, L::STAGE_BYTES);
            else if (rank == 0) mbar_expect_tx(&full[stage], 2 * L::STAGE_BYTES);  // both CTAs' bytes
          }
          uint8_t* a_dst = sA + stage * A_STAGE_BYTES;
          uint8_t* b_dst = sB + stage * L::B_STAGE_BYTES;
          if (!tail) {
            const int kx = ks * BK;
            tma_load_2d_pair(a_dst, &p.tmA0, bar, kx, m0);
            if (B0_MN) {
              const bool second = ks >= p.k0_split_steps;
              const void* mp = second ? (const void*)&p.tmB0b : (const void*)&p.tmB0;
              const int ky = second ? kx - p.k0_split_steps * BK : kx;
#pragma unroll
              for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(b_dst + j * 8192, mp, bar, n0 + (int)rank * 128 + 64 * j, ky);
            } else if (STACKED) {
              tma_load_2d_pair(b_dst, rank ? (const void*)&p.tmB0b : (const void*)&p.tmB0, bar, kx, n0);
            } else {
              tma_load_2d_pair(b_dst, &p.tmB0, bar, kx, n0 + (int)rank * 128);
            }
          } else {
            const int kt = (ks - nk0) * BK;   // K offset inside the rank-r tail
            tma_load_2d_pair(a_dst, &p.tmA1, bar, kt, m0);
            if (B1_MN) {
#pragma unroll
              for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(b_dst + j * 8192, &p.tmB1, bar, n0 + (int)rank * 128 + 64 * j, kt);
            } else if (STACKED) {
              if (rank == 0) tma_load_2d_pair(b_dst, &p.tmB1, bar, p.tail_b1_x + kt, n0);
              else tma_load_2d_pair(b_dst, &p.tmB1b, bar, p.tail_b1b_x + kt, n0);
            } else {
              tma_load_2d_pair(b_dst, &p.tmB1, bar, kt, n0 + (int)rank * 128);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) spin_ns(100000ull);  // unwind: give copies already issued time to land
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA only)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc0 = umma_idesc_bf16(PM, BN, 0, B0_MN ? 1 : 0);
      constexpr uint32_t idesc1 = umma_idesc_bf16(PM, BN, 0, B1_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cluster_id; t < num_tiles && ok; t += num_clusters, ++it) {
        const int buf = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_cl(&acc_empty[buf], acc_phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x202)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int ks = 0; ks < nk; ++ks) {
          const bool tail = HAS_TAIL && ks >= nk0;
          if (!mbar_wait_cl(KSCALE ? &ready[stage] : &full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x203)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * L::B_STAGE_BYTES);
          const bool bmn = tail ? B1_MN : B0_MN;   // BK / 16 MMAs per stage, as in tc_gemm_kernel
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = umma_smem_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = bmn ? umma_smem_desc(b_base + kk * 2048, 8192, 1024)
                                       : umma_smem_desc(b_base + kk * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, tail ? idesc1 : idesc0, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&acc_full[buf], 0x3);
      }
      umma_commit_pair_mc(drain, 0x1);
      mbar_wait_drain(drain, 0, 20000000ull);
    }
    __syncwarp();
  } else if (warp < (C::EPI8 ? 10 : 6)) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    constexpr bool EPI8 = C::EPI8;
    const int q = warp & 3;                         // TMEM lane quarter this warp may access
    const int half = EPI8 ? (warp - 2) >> 2 : 0;    // with 8 warps: which half of the columns
    uint8_t* my_stg = sStg + (warp - 2) * (EPI8 ? 4096 : EpiCfg<EPI, true>::STG_BUFS * 4096);
    int it = 0;
    uint32_t chunk_ctr = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_cl(&acc_full[buf], acc_phase, p.timeout_ns, abort_flag, p.err, 0x204)) break;
      tc_fence_after();
      int mt, nt;
      tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + buf * BN + half * (N_OUT / 2);
      const int row0 = mt * PM + (int)rank * BM + 32 * q;
      if constexpr (EPI8)
        epilogue_tile<EPI, N_OUT / 2>(p, t_row, row0, nt * N_OUT + half * (N_OUT / 2), lane, my_stg, chunk_ctr);
      else
        epilogue_tile<EPI, N_OUT>(p, t_row, row0, nt * N_OUT, lane, my_stg, chunk_ctr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[buf]), 0));
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  } else if (KSCALE) {
    // ---------------------------------------------------------------- A-tile K-scaling (both CTAs)
    const int tid = threadIdx.x - 192;   // 0 .. 127
    const float* sKsc = reinterpret_cast<const float*>(smem + L::OFF_KSC);
    const uint32_t ready_leader = mapa_shared(smem_u32(ready), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = cluster_id; t < num_tiles && ok; t += num_clusters) {
      for (int ks = 0; ks < nk; ++ks) {
        if (lane == 0) ok = mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x205);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (!(HAS_TAIL && ks >= nk0))   // the rank-r tail is not scaled
          kscale_tile_inplace(sA + stage * A_STAGE_BYTES, sKsc + stage * BK, tid);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(ready_leader + 8u * (uint32_t)stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync_all();   // neither CTA leaves while its peer may still reach into it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ============================================================================ host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor map, inner extent `inner` (contiguous), `outer` rows of `ld` elements,
// box {64, box_rows}, 128-byte swizzle, out-of-bounds elements read as zero.
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc || base == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                    uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  auto enc = get_encode();
  if (!enc || base == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                  uint32_t box_outer) {
  auto enc = get_encode();
  if (!enc || base == nullptr || ld % 16 != 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_current() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// index of the current device in the per-device caches of the launch helpers
static int current_device_slot() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev < 0 || dev >= 64) ? 0 : dev;
}

static int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e ? atoi(e) : dflt;
}

// Programmatic dependent launch for the kernels of the hot path (all of them wait for their
// predecessor before touching global memory); LORA_GB300_PDL=0 launches them plainly.
int pdl_attr(cudaLaunchAttribute* a) {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("LORA_GB300_PDL");
    on = (e && *e) ? (atoi(e) != 0) : 1;
  }
  if (!on) return 0;
  a->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a->val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

template <bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE = false, bool ZF = false>
static cudaError_t launch_one(const TcParams& p, cudaStream_t st, int tiles, int max_ctas) {
  using L = Layout<EPI, false, KSCALE>;
  auto kern = tc_gemm_kernel<B0_MN, STACKED, HAS_TAIL, B1_MN, EPI, KSCALE, ZF>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(OneCta<EPI, KSCALE, ZF>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  static int max_units_dev[64] = {0};   // co-resident CTAs, per device
  int& max_units = max_units_dev[current_device_slot()];
  if (max_units == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    max_units = num_sms_current();
  }
  int units = max_units;
  // test knob: cap the persistent grid so that small problems still run several tiles per CTA
  const int cap = env_int("LORA_GB300_MAX_CTAS", 0);
  if (cap > 0 && cap < units) units = cap;
  if (max_ctas > 0 && max_ctas < units) units = max_ctas;
  if (units > tiles) units = tiles;
  cfg.gridDim = dim3(units, 1, 1);
  cfg.numAttrs += (unsigned)pdl_attr(&attr[cfg.numAttrs]);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE = false>
static cudaError_t launch_pair(const TcParams& p, cudaStream_t st, int tiles, int max_ctas) {
  using L = Layout<EPI, true, KSCALE>;
  auto kern = tc_pair_kernel<B0_MN, STACKED, HAS_TAIL, B1_MN, EPI, KSCALE>;
  static int max_clusters_dev[64] = {0};   // co-resident clusters, per device
  int& max_clusters = max_clusters_dev[current_device_slot()];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(OneCta<EPI, KSCALE>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (const int pol = env_int("LORA_GB300_PAIR_POLICY", 0)) {  // 1 = spread, 2 = load balancing
    attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[1].val.clusterSchedulingPolicyPreference =
        pol == 2 ? cudaClusterSchedulingPolicyLoadBalancing : cudaClusterSchedulingPolicySpread;
    cfg.numAttrs = 2;
  }
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (num_sms_current() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters = n > 0 ? n : 1;
    if (env_int("LORA_GB300_VERBOSE", 0))
      fprintf(stderr, "[lora_gb300] pair GEMM: %d co-resident clusters of 2 CTAs, %d bytes smem\n", n, L::TOTAL);
  }
  int clusters = max_clusters;     // persistent: every cluster resident at once
  const int cap = env_int("LORA_GB300_MAX_CTAS", 0) / 2;
  if (cap > 0 && cap < clusters) clusters = cap;
  if (max_ctas > 1 && max_ctas / 2 < clusters) clusters = max_ctas / 2;
  if (clusters > tiles) clusters = tiles;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.numAttrs += (unsigned)pdl_attr(&attr[cfg.numAttrs]);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// kind: 0 one CTA, 1 CTA pair
template <bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE = false>
static cudaError_t launch_variant(const TcParams& p, cudaStream_t st, int kind, int tiles, int max_ctas) {
  if (kind == 1) return launch_pair<B0_MN, STACKED, HAS_TAIL, B1_MN, EPI, KSCALE>(p, st, tiles, max_ctas);
  return launch_one<B0_MN, STACKED, HAS_TAIL, B1_MN, EPI, KSCALE>(p, st, tiles, max_ctas);
}

static cudaError_t launch_mode(const TcGemmDesc& d, const TcParams& p, cudaStream_t st, int kind, int tiles) {
  const int mc = d.max_ctas;
  switch (d.mode) {
    case TC_FWD:
      if (d.dn_a) return launch_one<false, false, true, false, EPI_SCALE_BIAS, false, true>(p, st, tiles, mc);
      if (d.has_tail) return launch_variant<false, false, true, false, EPI_SCALE_BIAS>(p, st, kind, tiles, mc);
      return launch_variant<false, false, false, false, EPI_SCALE_BIAS>(p, st, kind, tiles, mc);
    case TC_BWD_DX:
      if (d.a_kscale) {   // A tiles scaled in shared memory by the scaling warps
        if (d.has_tail) return launch_variant<true, false, true, true, EPI_SCALE_BIAS, true>(p, st, kind, tiles, mc);
        return launch_variant<true, false, false, true, EPI_SCALE_BIAS, true>(p, st, kind, tiles, mc);
      }
      if (d.has_tail) return launch_variant<true, false, true, true, EPI_SCALE_BIAS>(p, st, kind, tiles, mc);
      return launch_variant<true, false, false, true, EPI_SCALE_BIAS>(p, st, kind, tiles, mc);
    case TC_SWIGLU_FWD:
      return launch_variant<false, true, true, false, EPI_SWIGLU>(p, st, kind, tiles, mc);
    case TC_SWIGLU_BWD:
      return launch_variant<true, false, true, true, EPI_SWIGLU_BWD>(p, st, kind, tiles, mc);
    case TC_W8A8K:  // one-CTA kernel only
      if (d.has_tail) return launch_one<false, false, true, false, EPI_W8A8K>(p, st, tiles, mc);
      return launch_one<false, false, false, false, EPI_W8A8K>(p, st, tiles, mc);
  }
  return cudaErrorInvalidValue;
}

// Kernel choice per mode.  LORA_GB300_GEMM_PAIR=0 / 1 forces the one-CTA / pair kernel for every
// mode (the chunked W8A8 product always runs one-CTA).
static bool use_pair(int mode) {
  const char* e = getenv("LORA_GB300_GEMM_PAIR");
  if (e && *e) return atoi(e) != 0;
  // measured over LLM layer shapes: the pair is 4-7% faster on the K-major products; on the
  // MN-major dX products (one-CTA 168 us against 174 us for the pair at 8192 x 4096 x 4096; with
  // the DoRA K-scaling 0.776 ms against 1.309 ms at 8192 x 11008 x 4096) and the fused W8A8 output
  // path the one-CTA kernel is as fast or faster
  return mode == TC_FWD || mode == TC_SWIGLU_FWD;
}

cudaError_t tc_gemm(const TcGemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0) return cudaSuccess;
  // the down-projection in the GEMM runs on the one-CTA kernel (ranks 8 .. 32, one tail step)
  if (d.dn_a && (d.mode != TC_FWD || !d.has_tail || d.dn_r < 8 || d.dn_r > 32 || d.dn_r % 8 || d.K1 != d.dn_r))
    return cudaErrorInvalidValue;
  const bool pair = use_pair(d.mode) && d.mode != TC_W8A8K && d.dn_a == nullptr;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const bool stacked = d.mode == TC_SWIGLU_FWD;
  // rows of a K-major B box: 256 (one CTA), 128 (stacked halves, or one CTA's half of a pair)
  const int bnb = (stacked || pair) ? BN / 2 : BN;
  bool ok = make_map(&p.tmA0, d.A0, d.K0, d.M, d.lda0, BM);
  if (d.b0_mn) {
    ok = ok && make_map(&p.tmB0, d.B0, d.N, d.b0_rows, d.ldb0, 64);
    if (d.B0b) ok = ok && make_map(&p.tmB0b, d.B0b, d.N, d.b0b_rows, d.ldb0, 64);
  } else {
    ok = ok && make_map(&p.tmB0, d.B0, d.K0, d.N, d.ldb0, bnb);
    if (stacked) ok = ok && make_map(&p.tmB0b, d.B0b, d.K0, d.N, d.ldb0, bnb);
  }
  if (d.has_tail) {
    // the tail's last K-step runs over a whole BK: its columns past K1 must read as TMA zero fill
    if (d.dn_a == nullptr) {   // with the down-projection in the GEMM the tail's A is written on chip
      if (d.K1_a != d.K1) return cudaErrorInvalidValue;
      ok = ok && make_map(&p.tmA1, d.A1, d.K1_a, d.M, d.lda1, BM);
    }
    if (d.b1_mn) ok = ok && make_map(&p.tmB1, d.B1, d.N, d.K1, d.ldb1, 64);
    else {
      ok = ok && make_map(&p.tmB1, d.B1, d.K1_b, d.N, d.ldb1, bnb);
      if (stacked)
        ok = ok && make_map(&p.tmB1b, d.B1b, d.K1_bb > 0 ? d.K1_bb : d.K1_b, d.N, d.ldb1b > 0 ? d.ldb1b : d.ldb1, bnb);
    }
  }
  int nouts = d.mode == TC_SWIGLU_FWD ? 3 : (d.mode == TC_SWIGLU_BWD ? 2 : 1);
  if (d.mode == TC_W8A8K && d.out[0] == nullptr) nouts = 0;   // raw int32 product only
  for (int i = 0; i < nouts; ++i) ok = ok && make_map(&p.tmOut[i], d.out[i], d.N, d.M, d.ldo, 32);
  if (!ok) return cudaErrorInvalidValue;
  p.sx = d.sx;
  p.sw = d.sw;
  p.ls = d.ls;
  p.acc_out = d.acc_out;
  p.kc_steps = d.kc_steps > 0 ? d.kc_steps : 16;
  p.write_y = d.out[0] != nullptr ? 1 : 0;
  p.pair_leader_arms = env_int("LORA_GB300_PAIR_ARM", 1);
  p.act = d.act;
  p.dn_a = d.dn_a;
  p.dn_lda = d.dn_lda;
  p.dn_s = d.dn_s;
  p.dn_r = d.dn_r;
  p.dn_z = d.dn_z;

  p.M = d.M;
  p.N = d.N;
  p.K0 = d.K0;
  p.K1 = d.K1;
  const int tile_m = pair ? 2 * BM : BM;
  p.num_m_tiles = (d.M + tile_m - 1) / tile_m;
  const int n_out = stacked ? BN / 2 : BN;
  p.num_n_tiles = (d.N + n_out - 1) / n_out;
  // raster group in M tiles of the tile sequence (pair tiles of 256 rows, or one-CTA tiles of 128):
  // measured, the MN-major dX products run best with groups of 4-8 one-CTA tiles (8192 x 4096 x
  // 4096: 168-169 us against 176 us with 16)
  const int gm_env = env_int("LORA_GB300_GROUP_M", 0);
  p.group_m = gm_env > 0 ? gm_env : (pair ? 8 : (d.b0_mn ? 8 : 16));
  p.k0_split_steps = d.b0_mn && d.B0b ? (d.k0_split / BK) : (1 << 30);
  p.tail_b1b_x = d.b1b_x;
  p.tail_b1_x = d.b1_x;
  p.col_scale = d.col_scale;
  p.bias = d.bias;
  p.a_kscale = d.a_kscale;

  p.e_in = d.e_in;
  p.u_in = d.u_in;
  p.ld_eu = d.ld_eu;
  p.err = d.err;
  p.timeout_ns = d.timeout_ns;
  const int tiles = p.num_m_tiles * p.num_n_tiles;

  // algorithmic flops of this launch: the base contraction plus the rank-r tail
  const double ntot = stacked ? 2.0 * d.N : (double)d.N;
  const double k1 = d.has_tail ? (stacked ? d.K1 / 2.0 : (double)d.K1) : 0.0;
  const double flops = 2.0 * d.M * ntot * ((double)d.K0 + k1);
  prof_mark(st, true, flops);
  const cudaError_t e = launch_mode(d, p, st, pair ? 1 : 0, tiles);
  prof_mark(st, false, 0.0);
  return e;
}

}  // namespace lg

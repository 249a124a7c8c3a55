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
// Roles (one CTA per SM, 6 or 10 warps):
//   warp 0      TMA producer: 128x64 A tiles and BNx64 B tiles into a STAGES-deep ring
//   warp 1      TMEM allocator + MMA issuer (one thread), double-buffered accumulators
//   warps 2..5  epilogue: TMEM -> registers -> (row scale, bias, SwiGLU) -> bf16 ->
//               swizzled SMEM staging -> TMA store
//   warps 6..9  (DoRA backward only) scale the A tile in SMEM by c[k] along K
// Every mbarrier wait is bounded (global timer); on expiry the CTA records the error in
// the caller's error word, drains its in-flight copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>
#include <stdlib.h>

namespace lg {

struct TcParams {
  CUtensorMap tmA0, tmB0, tmB0b, tmA1, tmB1, tmB1b;
  CUtensorMap tmOut[3];
  int M, N, K0, K1;
  int num_m_tiles, num_n_tiles, group_m;
  int k0_split_steps;   // MN-major B0: k-steps taken from tmB0 before switching to tmB0b
  int tail_b1b_x;       // stacked tail: x coordinate (K shift) of the second half
  const float* col_scale;
  const bf16* bias;
  const float* a_kscale;
  const bf16* e_in;
  const bf16* u_in;
  int ld_eu;
  uint32_t* err;
  uint64_t timeout_ns;
};

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB

template <int EPI>
struct EpiCfg;
template <>
struct EpiCfg<EPI_SCALE_BIAS> { static constexpr int STAGES = 4, STG_BUFS = 2; };
template <>
struct EpiCfg<EPI_SWIGLU> { static constexpr int STAGES = 3, STG_BUFS = 3; };
template <>
struct EpiCfg<EPI_SWIGLU_BWD> { static constexpr int STAGES = 3, STG_BUFS = 4; };

template <int BN, int EPI>
struct Layout {
  static constexpr int STAGES = EpiCfg<EPI>::STAGES;
  static constexpr int B_STAGE_BYTES = BN * BK * 2;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
  static constexpr int OFF_STG = OFF_B + STAGES * B_STAGE_BYTES;
  static constexpr int STG_BYTES = 4 * EpiCfg<EPI>::STG_BUFS * 4096;
  static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
  static constexpr int BAR_BYTES = 8 * (3 * STAGES + 5) + 16;
  static constexpr int TOTAL = OFF_BAR + BAR_BYTES + 1024;  // +1024 for base alignment
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

template <int BN, bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE>
__global__ void __launch_bounds__(KSCALE ? 320 : 192, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using L = Layout<BN, EPI>;
  constexpr int STAGES = L::STAGES;
  constexpr int BNB = STACKED ? BN / 2 : BN;          // rows per K-major B box
  constexpr int N_OUT = STACKED ? BN / 2 : BN;        // logical output columns per tile
  constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(TMEM_COLS <= 512, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + L::OFF_A;
  uint8_t* sB = smem + L::OFF_B;
  uint8_t* sStg = smem + L::OFF_STG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* ready = bars + 2 * STAGES;
  uint64_t* acc_full = bars + 3 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  const int nk0 = (p.K0 + BK - 1) / BK;
  const int nk = nk0 + (HAS_TAIL ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&ready[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;         // bit s: stage s has been armed at least once
      uint32_t armed_par = 0;     // bit s: parity of the last arm of stage s
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
        const int m0 = mt * BM;
        const int n0 = nt * N_OUT;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x101)) {
            ok = false;
            break;
          }
          const bool tail = HAS_TAIL && ks >= nk0;
          mbar_expect_tx(&full[stage], A_STAGE_BYTES + L::B_STAGE_BYTES);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * A_STAGE_BYTES;
          uint8_t* b_dst = sB + stage * L::B_STAGE_BYTES;
          if (!tail) {
            const int kx = ks * BK;
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
            tma_load_2d(a_dst, &p.tmA1, &full[stage], 0, m0);
            if (B1_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * 8192, &p.tmB1, &full[stage], n0 + 64 * j, 0);
            } else if (STACKED) {
              tma_load_2d(b_dst, &p.tmB1, &full[stage], 0, n0);
              tma_load_2d(b_dst + BNB * 128, &p.tmB1b, &full[stage], p.tail_b1b_x, n0);
            } else {
              tma_load_2d(b_dst, &p.tmB1, &full[stage], 0, n0);
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
    if (lane == 0) {
      constexpr uint32_t idesc0 = umma_idesc_bf16(BM, BN, 0, B0_MN ? 1 : 0);
      constexpr uint32_t idesc1 = umma_idesc_bf16(BM, BN, 0, B1_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1, p.timeout_ns, abort_flag, p.err, 0x102)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int ks = 0; ks < nk; ++ks) {
          const bool tail = HAS_TAIL && ks >= nk0;
          // with K-scaling every stage (tail included) is handed over through `ready`, so that
          // barrier completes exactly one phase per use of the stage, in step with `full`
          uint64_t* wb = KSCALE ? &ready[stage] : &full[stage];
          if (!mbar_wait(wb, phase, p.timeout_ns, abort_flag, p.err, 0x103)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * L::B_STAGE_BYTES);
          const int nsub = tail ? (p.K1 + 15) / 16 : BK / 16;
          const bool bmn = tail ? B1_MN : B0_MN;
          for (int kk = 0; kk < nsub; ++kk) {
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
  } else if (warp < 6) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int ew = warp - 2;                // epilogue warp index 0..3 (staging owner)
    uint8_t* my_stg = sStg + ew * (EpiCfg<EPI>::STG_BUFS * 4096);
    int it = 0;
    uint32_t chunk_ctr = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait(&acc_full[buf], acc_phase, p.timeout_ns, abort_flag, p.err, 0x104)) {
        ok = false;
        break;
      }
      tc_fence_after();
      int mt, nt;
      tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
      const int row0 = mt * BM + 32 * q;         // global row of lane 0
      const int n0 = nt * N_OUT;
      const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + buf * BN;

      if constexpr (EPI == EPI_SCALE_BIAS) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c, ++chunk_ctr) {
          uint8_t* stg = my_stg + (chunk_ctr & 1) * 4096;
          if (lane == 0) tma_store_wait_read<1>();
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
              const float h0 = e0 / (1.0f + __expf(-e0)) * u0;
              const float h1 = e1 / (1.0f + __expf(-e1)) * u1;
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
        // accumulator = dh; read the saved e, u for this thread's row and form de, du
        const int grow = row0 + lane;
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c, ++chunk_ctr) {
          uint8_t* sde = my_stg + (chunk_ctr & 1) * 8192;
          uint8_t* sdu = sde + 4096;
          if (lane == 0) tma_store_wait_read<1>();
          __syncwarp();
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t vd[32];
            tmem_ld_32x32b_x32(t_row + c * 64 + h * 32, vd);
            tmem_ld_wait();
            const int col = n0 + c * 64 + h * 32;
            uint32_t ev[16], uv[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const int cc = col + 8 * g;
              if (grow < p.M && cc < p.N) {
                const uint4 a = *reinterpret_cast<const uint4*>(p.e_in + (size_t)grow * p.ld_eu + cc);
                const uint4 b = *reinterpret_cast<const uint4*>(p.u_in + (size_t)grow * p.ld_eu + cc);
                ev[4 * g] = a.x; ev[4 * g + 1] = a.y; ev[4 * g + 2] = a.z; ev[4 * g + 3] = a.w;
                uv[4 * g] = b.x; uv[4 * g + 1] = b.y; uv[4 * g + 2] = b.z; uv[4 * g + 3] = b.w;
              } else {
#pragma unroll
                for (int z = 0; z < 4; ++z) ev[4 * g + z] = uv[4 * g + z] = 0u;
              }
            }
            uint32_t wde[16], wdu[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 e = unpack_bf16x2(ev[j]);
              const float2 u = unpack_bf16x2(uv[j]);
              const float d0 = u2f(vd[2 * j]), d1 = u2f(vd[2 * j + 1]);
              const float s0 = 1.0f / (1.0f + __expf(-e.x));
              const float s1 = 1.0f / (1.0f + __expf(-e.y));
              const float de0 = d0 * u.x * s0 * (1.0f + e.x * (1.0f - s0));
              const float de1 = d1 * u.y * s1 * (1.0f + e.y * (1.0f - s1));
              const float du0 = d0 * e.x * s0;
              const float du1 = d1 * e.y * s1;
              wde[j] = pack_bf16x2(de0, de1);
              wdu[j] = pack_bf16x2(du0, du1);
            }
            stage_row(sde, lane, wde, h * 4);
            stage_row(sdu, lane, wdu, h * 4);
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    (void)ok;
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  } else if (KSCALE) {
    // ---------------------------------------------------------------- A-tile K-scaling (DoRA backward)
    const int tid = threadIdx.x - 192;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      for (int ks = 0; ks < nk; ++ks) {
        const bool tail = HAS_TAIL && ks >= nk0;
        if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err, 0x105)) {
          ok = false;
          break;
        }
        if (tail) {
          // the rank-r tail is not scaled: hand the stage straight on
          mbar_arrive(&ready[stage]);
        } else {
          uint8_t* a = sA + stage * A_STAGE_BYTES;
          const int k0 = ks * BK;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int ci = tid + 128 * i;
            const int r = ci >> 3, pc = ci & 7;
            const int j = pc ^ (r & 7);
            const int kb = k0 + 8 * j;
            uint4* ptr = reinterpret_cast<uint4*>(a + r * 128 + pc * 16);
            uint4 v = *ptr;
            float sc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[e] = (kb + e < p.K0) ? __ldg(p.a_kscale + kb + e) : 0.0f;
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack_bf16x2(w[e]);
              w[e] = pack_bf16x2(f.x * sc[2 * e], f.y * sc[2 * e + 1]);
            }
            *ptr = v;
          }
          fence_proxy_async_smem();
          mbar_arrive(&ready[stage]);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
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

template <int BN, bool B0_MN, bool STACKED, bool HAS_TAIL, bool B1_MN, int EPI, bool KSCALE>
static cudaError_t launch_variant(const TcParams& p, cudaStream_t st, int grid) {
  using L = Layout<BN, EPI>;
  auto kern = tc_gemm_kernel<BN, B0_MN, STACKED, HAS_TAIL, B1_MN, EPI, KSCALE>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, KSCALE ? 320 : 192, L::TOTAL, st>>>(p);
  count_launch();
  return cudaGetLastError();
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

static cudaError_t launch_mode(const TcGemmDesc& d, const TcParams& p, cudaStream_t st, int grid);

cudaError_t tc_gemm(const TcGemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0) return cudaSuccess;
  TcParams p;
  memset(&p, 0, sizeof(p));
  constexpr int BN = 256;
  const bool stacked = d.mode == TC_SWIGLU_FWD;
  const int bnb = stacked ? BN / 2 : BN;
  const bool b0_mn = d.b0_mn, b1_mn = d.b1_mn;
  bool ok = make_map(&p.tmA0, d.A0, d.K0, d.M, d.lda0, BM);
  if (b0_mn) {
    ok = ok && make_map(&p.tmB0, d.B0, d.N, d.b0_rows, d.ldb0, 64);
    if (d.B0b) ok = ok && make_map(&p.tmB0b, d.B0b, d.N, d.b0b_rows, d.ldb0, 64);
  } else {
    ok = ok && make_map(&p.tmB0, d.B0, d.K0, d.N, d.ldb0, bnb);
    if (stacked) ok = ok && make_map(&p.tmB0b, d.B0b, d.K0, d.N, d.ldb0, bnb);
  }
  if (d.has_tail) {
    ok = ok && make_map(&p.tmA1, d.A1, d.K1_a, d.M, d.lda1, BM);
    if (b1_mn) ok = ok && make_map(&p.tmB1, d.B1, d.N, d.K1, d.ldb1, 64);
    else {
      ok = ok && make_map(&p.tmB1, d.B1, d.K1_b, d.N, d.ldb1, bnb);
      if (stacked) ok = ok && make_map(&p.tmB1b, d.B1b, d.K1_b, d.N, d.ldb1, bnb);
    }
  }
  const int nouts = d.mode == TC_SWIGLU_FWD ? 3 : (d.mode == TC_SWIGLU_BWD ? 2 : 1);
  for (int i = 0; i < nouts; ++i) ok = ok && make_map(&p.tmOut[i], d.out[i], d.N, d.M, d.ldo, 32);
  if (!ok) return cudaErrorInvalidValue;

  p.M = d.M;
  p.N = d.N;
  p.K0 = d.K0;
  p.K1 = d.K1;
  p.num_m_tiles = (d.M + BM - 1) / BM;
  const int n_out = stacked ? BN / 2 : BN;
  p.num_n_tiles = (d.N + n_out - 1) / n_out;
  p.group_m = 16;
  p.k0_split_steps = b0_mn && d.B0b ? (d.k0_split / BK) : (1 << 30);
  p.tail_b1b_x = d.b1b_x;
  p.col_scale = d.col_scale;
  p.bias = d.bias;
  p.a_kscale = d.a_kscale;
  p.e_in = d.e_in;
  p.u_in = d.u_in;
  p.ld_eu = d.ld_eu;
  p.err = d.err;
  p.timeout_ns = d.timeout_ns;
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  int grid = num_sms_current();
  if (d.max_ctas > 0 && d.max_ctas < grid) grid = d.max_ctas;
  // test knob: cap the persistent grid so that small problems still run several tiles per CTA
  if (const char* env = getenv("LORA_GB300_MAX_CTAS")) {
    const int v = atoi(env);
    if (v > 0 && v < grid) grid = v;
  }
  if (grid > tiles) grid = tiles;

  // algorithmic flops of this launch: the base contraction plus the rank-r tail
  const double ntot = stacked ? 2.0 * d.N : (double)d.N;
  const double k1 = d.has_tail ? (stacked ? d.K1 / 2.0 : (double)d.K1) : 0.0;
  const double flops = 2.0 * d.M * ntot * ((double)d.K0 + k1);
  prof_mark(st, true, flops);
  const cudaError_t e = launch_mode(d, p, st, grid);
  prof_mark(st, false, 0.0);
  return e;
}

static cudaError_t launch_mode(const TcGemmDesc& d, const TcParams& p, cudaStream_t st, int grid) {
  constexpr int BN = 256;
  switch (d.mode) {
    case TC_FWD:
      if (d.has_tail) return launch_variant<BN, false, false, true, false, EPI_SCALE_BIAS, false>(p, st, grid);
      return launch_variant<BN, false, false, false, false, EPI_SCALE_BIAS, false>(p, st, grid);
    case TC_BWD_DX:
      if (d.a_kscale) {
        if (d.has_tail) return launch_variant<BN, true, false, true, true, EPI_SCALE_BIAS, true>(p, st, grid);
        return launch_variant<BN, true, false, false, true, EPI_SCALE_BIAS, true>(p, st, grid);
      }
      if (d.has_tail) return launch_variant<BN, true, false, true, true, EPI_SCALE_BIAS, false>(p, st, grid);
      return launch_variant<BN, true, false, false, true, EPI_SCALE_BIAS, false>(p, st, grid);
    case TC_SWIGLU_FWD:
      return launch_variant<BN, false, true, true, false, EPI_SWIGLU, false>(p, st, grid);
    case TC_SWIGLU_BWD:
      return launch_variant<BN, true, false, true, true, EPI_SWIGLU_BWD, false>(p, st, grid);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lg

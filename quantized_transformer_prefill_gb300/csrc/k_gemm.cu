// k_gemm.cu -- Q8_0 x Q8_0 block-scaled GEMM on the 5th-generation tensor
// cores (tcgen05.mma kind::f16 with TMEM accumulators, TMA-fed).
//
// What it computes (walkthrough index, master table, row "CPU matmul
// kernels": quantized weight x on-the-fly Q8_0 activations; "05 · Graph
// build", section 2.5: one matmul per projection):
//     y[m][n] = sum_b  da[m][b] * dw[n][b] * sum_{i<32} qa[m][32b+i] * qw[n][32b+i]
//
// How: the int8 codes are stored as fp16 (every integer in [-127, 127] is
// exact in fp16, each product is exact in f32 and a 32-term block sum stays
// below 2^24), so a kind::f16 MMA with f32 accumulation over one 32-wide
// block returns that block's integer dot exactly.  Each K block is
// accumulated into its own TMEM slot; epilogue warps read the slot back
// (tcgen05.ld), scale it by da * dw in f32 registers and add it to the
// running f32 sum.  This keeps the per-block scales of Q8_0 exact where a
// dequantize-first scheme would round the operands.
//
// Warp roles (320 threads, one CTA per SM, persistent over output tiles):
//   warp 0     TMA producer: A/B code tiles (128-byte swizzle) per 64-wide K
//              stage, and the two blocks' scale rows into a separate ring
//   warp 1     TMEM allocator and MMA issuer (one thread)
//   warps 2-9  epilogue: warp w reads TMEM lane quadrant w % 4 (32 rows of
//              the 128-row tile) in the 16x256b fragment shape; warps 2-5
//              take the left half of the N tile, warps 6-9 the right half
// Rings: STAGES A/B stages, free as soon as the MMAs that read them
// completed (TMA latency is ~1.6k cycles, so refills must not wait for the
// epilogue); SSTAGES scale stages, freed by the epilogue; NSLOT TMEM slots
// of BN columns (tfull/tempty).  Every wait is bounded; on
// timeout the kernel records a status code, drains its own TMA loads and
// MMAs, frees TMEM and returns.
#include <algorithm>
#include <cstdio>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // fp16 elements per stage: two Q8_0 blocks
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;

template <int BN>
struct Cfg {
  // four stages of A/B (8 K blocks in flight), measured against 3, 5 and 6:
  // six is 1-2% slower on the 1.5B and 7B shapes, three 1.5% slower on
  // 1.5B/2048, five 0.4% slower on the 0.5B forward
  static constexpr int STAGES = 4;
  static constexpr int SSTAGES = 8;
  static constexpr int NSLOT = 512 / BN;
  static constexpr int CPW = BN / 2;  // columns per epilogue thread
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int SA_BYTES = 2 * kBM * 4;
  static constexpr int SB_BYTES = 2 * BN * 4;
  static constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES;
  static constexpr uint32_t SCALE_TX = SA_BYTES + SB_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SB = OFF_SA + SSTAGES * SA_BYTES;
  static constexpr int OFF_BAR = OFF_SB + SSTAGES * SB_BYTES;
  static constexpr int NBAR = 2 * STAGES + 2 * SSTAGES + 2 * NSLOT;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEM + 16 + 1024;  // + slack to align the base to 1024
  static_assert(OFF_B % 1024 == 0 && OFF_SA % 1024 == 0, "swizzled tiles need 1024-B alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct Args {
  int M, N, nb, n_stages;
  int m_tiles, n_tiles, splits, stages_per_split;
  int epi;
  float* out;
  int64_t ldo, split_stride;
  __half* q_out;
  int64_t ldq;
  float* qs_out;
  int64_t ldqs;
  int64_t n_out_cols;
  int32_t* dots;
  int* err;
  uint64_t wait_ns;  // time limit of every bounded wait
  int skip_stage;    // test hook: a stage CTA 0's producer withholds (-1: none)
  int b_pre;         // B written by no kernel in flight: its first loads precede the grid wait
};

// silu(g) * u = g / (1 + exp(-g)) * u in f32: expf (2 ulp), the add, the
// fast division (2 ulp) and the product stay within 10 units of f32 roundoff
// of the exact value; the gate/up GEMM of the 0.5B shape takes 8% less time
// than with an IEEE division.  (For 1 + exp(-g) above 2^126, g < -87, the
// fast division returns 0, as the exact value ~g e^g is below 1e-35.)
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, expf(-g))), u);
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_q8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA,
                   const __grid_constant__ CUtensorMap tmSB, const Args p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sSA = reinterpret_cast<float*>(smem + C::OFF_SA);
  float* sSB = reinterpret_cast<float*>(smem + C::OFF_SB);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* sfull = empty + C::STAGES;
  uint64_t* sempty = sfull + C::SSTAGES;
  uint64_t* tfull = sempty + C::SSTAGES;
  uint64_t* tempty = tfull + C::NSLOT;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::SSTAGES; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kEpiWarps);
    }
    for (int k = 0; k < C::NSLOT; ++k) {
      mbar_init(&tfull[k], 1);
      mbar_init(&tempty[k], kEpiWarps);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSA);
    tma_prefetch_desc(&tmSB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // set-up above overlaps the previous kernel; global memory only after it,
  // except the producer's first B loads when B is static (below)
  pdl_trigger();
  if (warp != 0) pdl_wait();

  const int total = p.m_tiles * p.n_tiles * p.splits;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0, n_ab = 0, n_s = 0;  // stages issued; A/B loads and scale loads in flight
      bool ok = true;
      // the first stages' B tiles and B scales (weights) before the wait for
      // the previous kernel: their ring slots are free at the start, and the
      // stage barriers complete once the A halves follow
      int npre = 0;
      if (p.b_pre && (int)blockIdx.x < total) {
        const int rest = (int)blockIdx.x / p.m_tiles;
        const int ntile = rest % p.n_tiles;
        const int s0 = (rest / p.n_tiles) * p.stages_per_split;
        const int s1 = min(p.n_stages, s0 + p.stages_per_split);
        npre = min(C::STAGES, s1 - s0);
        for (int j = 0; j < npre; ++j) {
          if (j == p.skip_stage && blockIdx.x == 0) continue;
          mbar_arrive_expect_tx(&full[j], C::STAGE_TX);
          tma_load_2d(sB + j * C::B_BYTES, &tmB, &full[j], (s0 + j) * kBK, ntile * BN);
          mbar_arrive_expect_tx(&sfull[j], C::SCALE_TX);
          tma_load_2d(sSB + j * (C::SB_BYTES / 4), &tmSB, &sfull[j], ntile * BN, 2 * (s0 + j));
        }
      }
      pdl_wait();
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int mt = t % p.m_tiles;
        const int rest = t / p.m_tiles;
        const int ntile = rest % p.n_tiles;
        const int sp = rest / p.n_tiles;
        const int s0 = sp * p.stages_per_split;
        const int s1 = min(p.n_stages, s0 + p.stages_per_split);
        for (int s = s0; s < s1; ++s, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&empty[st], ((it / C::STAGES) & 1) ^ 1, p.err, kDevTimeoutTmaEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          // test hook: withhold this stage (no loads, no arrival), so the
          // consumers' bounded waits on it run out
          if (it == p.skip_stage && blockIdx.x == 0) continue;
          const bool pre = it < npre;  // B half already issued
          if (!pre) mbar_arrive_expect_tx(&full[st], C::STAGE_TX);
          tma_load_2d(sA + st * C::A_BYTES, &tmA, &full[st], s * kBK, mt * kBM);
          if (!pre) tma_load_2d(sB + st * C::B_BYTES, &tmB, &full[st], s * kBK, ntile * BN);
          n_ab = it + 1;
          const int ss = it % C::SSTAGES;
          if (!mbar_wait(&sempty[ss], ((it / C::SSTAGES) & 1) ^ 1, p.err, kDevTimeoutTmaEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          if (!pre) mbar_arrive_expect_tx(&sfull[ss], C::SCALE_TX);
          tma_load_2d(sSA + ss * (C::SA_BYTES / 4), &tmSA, &sfull[ss], mt * kBM, 2 * s);
          if (!pre) tma_load_2d(sSB + ss * (C::SB_BYTES / 4), &tmSB, &sfull[ss], ntile * BN, 2 * s);
          n_s = it + 1;
        }
      }
      if (!ok) {
        // drain the loads that may still be in flight before the CTA exits
        for (int j = max(0, n_ab - C::STAGES); j < n_ab; ++j)
          mbar_wait(&full[j % C::STAGES], (j / C::STAGES) & 1, p.err, kDevTimeoutDrain, p.wait_ns);
        for (int j = max(0, n_s - C::SSTAGES); j < n_s; ++j)
          mbar_wait(&sfull[j % C::SSTAGES], (j / C::SSTAGES) & 1, p.err, kDevTimeoutDrain, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      int it = 0, sit = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const int rest = t / p.m_tiles;
        const int sp = rest / p.n_tiles;
        const int s0 = sp * p.stages_per_split;
        const int s1 = min(p.n_stages, s0 + p.stages_per_split);
        for (int s = s0; s < s1 && ok; ++s, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&full[st], (it / C::STAGES) & 1, p.err, kDevTimeoutMmaFull, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + st * C::A_BYTES);
          const uint32_t b_base = smem_u32(sB + st * C::B_BYTES);
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            const int slot = sit % C::NSLOT;
            if (!mbar_wait(&tempty[slot], ((sit / C::NSLOT) & 1) ^ 1, p.err, kDevTimeoutMmaSlot, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(slot * BN);
#pragma unroll
            for (int k16 = 0; k16 < 2; ++k16) {
              const uint32_t koff = (uint32_t)(blk * 64 + k16 * 32);  // bytes along K
              tc_mma_f16(d, smem_desc_sw128(a_base + koff), smem_desc_sw128(b_base + koff), idesc,
                         (uint32_t)k16);
            }
            tc_commit(&tfull[slot]);
            ++sit;
          }
          if (ok) tc_commit(&empty[st]);
        }
      }
      // every MMA issued must have landed before TMEM is released
      if (sit > 0) {
        const int j = sit - 1;
        mbar_wait(&tfull[j % C::NSLOT], (j / C::NSLOT) & 1, p.err, kDevTimeoutDrain, p.wait_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Fragment layout (tcgen05.ld 16x256b): lane l of warp w holds rows
    // quad*32 + {g, g+8, g+16, g+24} (g = l / 4) and the column pairs
    // 8k + 2(l % 4) + {0, 1}, k < 8, of its 64-column half.  A thread then
    // needs 8 column scales and 4 row scales per K block instead of the 64
    // broadcast column scales of a row-per-thread layout, which keeps the
    // epilogue's shared-memory loads off the port the MMAs read operands from.
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int g = lane >> 2, t4 = lane & 3;
    int it = 0, sit = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int mt = t % p.m_tiles;
      const int rest = t / p.m_tiles;
      const int ntile = rest % p.n_tiles;
      const int sp = rest / p.n_tiles;
      const int s0 = sp * p.stages_per_split;
      const int s1 = min(p.n_stages, s0 + p.stages_per_split);
      const int mrow0 = mt * kBM + quad * 32;
      const int ncol0 = ntile * BN + half * C::CPW;

      float2 acc[4][8];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[rr][k] = make_float2(0.f, 0.f);

      for (int s = s0; s < s1 && ok; ++s, ++it) {
        const int ss = it % C::SSTAGES;
        if (!mbar_wait(&sfull[ss], (it / C::SSTAGES) & 1, p.err, kDevTimeoutEpilogue, p.wait_ns)) {
          ok = false;
          break;
        }
        // both blocks of the stage unrolled (the second block's TMEM load and
        // the first one's FFMAs interleave: 7% fewer cycles per block); each
        // block's scales are read from shared memory before its slot is waited
        // for
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int slot = sit % C::NSLOT;
          const float* sa = sSA + ss * 2 * kBM + blk * kBM + quad * 32 + g;
          const float* dw = sSB + ss * 2 * BN + blk * BN + half * C::CPW + 2 * t4;
          float2 w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = *reinterpret_cast<const float2*>(dw + 8 * k);
          float da4[4];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) da4[rr] = sa[8 * rr];
          if (!mbar_wait_spin(&tfull[slot], (sit / C::NSLOT) & 1, p.err, kDevTimeoutEpilogue, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr =
              tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(slot * BN + half * C::CPW);
          uint32_t ra[32], rb[32];  // rows g, g+8 and g+16, g+24
          tmem_ld16x256(taddr, ra);
          tmem_ld16x256(taddr + (16u << 16), rb);
          tmem_wait_ld();
          // slot read: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[slot]);
          const int b = 2 * s + blk;
          if (EPI == kEpiDots && b < p.nb) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int m = mrow0 + g + 8 * rr;
              if (m >= p.M) continue;
#pragma unroll
              for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int n = ncol0 + 8 * k + 2 * t4 + e;
                  const uint32_t v = rr < 2 ? ra[4 * k + 2 * rr + e] : rb[4 * k + 2 * (rr - 2) + e];
                  if (n < p.N) p.dots[((int64_t)m * p.N + n) * p.nb + b] = __float2int_rn(__uint_as_float(v));
                }
            }
          }
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const float da = da4[rr];
            const float2 da2 = make_float2(da, da);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t* rv = rr < 2 ? &ra[4 * k + 2 * rr] : &rb[4 * k + 2 * (rr - 2)];
              acc[rr][k] = __ffma2_rn(make_float2(__uint_as_float(rv[0]), __uint_as_float(rv[1])),
                                      __fmul2_rn(da2, w[k]), acc[rr][k]);
            }
          }
          ++sit;
        }
        if (!ok) break;
        // this stage's scales are consumed
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[ss]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- store
      if (EPI == kEpiSwiGLU) {
        // the warp's 64 columns hold 32 gate (k < 4) then 32 up (k >= 4) rows
        // of W for the same 32 outputs j0..j0+31: one Q8_0 block per row,
        // spread over the four lanes of a quad
        const int64_t j0 = (int64_t)ncol0 / 2;
        if (j0 < p.n_out_cols) {
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int m = mrow0 + g + 8 * rr;
            float sv[8];
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              sv[2 * k] = silu_mul(acc[rr][k].x, acc[rr][k + 4].x);
              sv[2 * k + 1] = silu_mul(acc[rr][k].y, acc[rr][k + 4].y);
              amax = fmaxf(amax, fmaxf(fabsf(sv[2 * k]), fabsf(sv[2 * k + 1])));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            if (m >= p.M) continue;
            if (p.out) {
              // debug capture: the f32 SwiGLU values this epilogue quantizes
              float* fo = p.out + (int64_t)m * p.ldo + j0 + 2 * t4;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                *reinterpret_cast<float2*>(fo + 8 * k) = make_float2(sv[2 * k], sv[2 * k + 1]);
            }
            const float d = __fdiv_rn(amax, 127.0f);
            const float id = q8_inv(d);
            __half* dst = p.q_out + (int64_t)m * p.ldq + j0 + 2 * t4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<__half2*>(dst + 8 * k) =
                  __floats2half2_rn(q8_code(sv[2 * k], id), q8_code(sv[2 * k + 1], id));
            if (t4 == 0) p.qs_out[(j0 / 32) * p.ldqs + m] = __half2float(__float2half_rn(d));
          }
        }
      } else {
        // column pairs straight to the row-major output: the four lanes of a
        // quad fill one 32-byte sector per row
        float* base = p.out + (int64_t)sp * p.split_stride;
        const bool pairs = (p.ldo & 1) == 0;
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int m = mrow0 + g + 8 * rr;
          if (m >= p.M) continue;
          float* row = base + (int64_t)m * p.ldo;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int n = ncol0 + 8 * k + 2 * t4;
            if (pairs && n + 1 < p.N) {
              *reinterpret_cast<float2*>(row + n) = acc[rr][k];
            } else {
              if (n < p.N) row[n] = acc[rr][k].x;
              if (n + 1 < p.N) row[n + 1] = acc[rr][k].y;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

int make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
             uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return -1;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

template <int BN, int EPI>
cudaError_t launch_bn(const GemmLaunch& g, const GemmMaps& maps, int num_sms, cudaStream_t st) {
  using C = Cfg<BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_q8_kernel<BN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  Args a;
  a.M = (int)g.M;
  a.N = (int)g.N;
  a.nb = g.B.nb;
  a.n_stages = (g.B.nb + 1) / 2;
  a.m_tiles = (int)((g.M + kBM - 1) / kBM);
  a.n_tiles = (int)((g.N + BN - 1) / BN);
  a.splits = std::max(1, std::min(g.plan.splits, a.n_stages));
  a.stages_per_split = (a.n_stages + a.splits - 1) / a.splits;
  a.splits = (a.n_stages + a.stages_per_split - 1) / a.stages_per_split;
  a.epi = g.epi;
  a.out = g.out;
  a.ldo = g.ldo;
  a.split_stride = g.split_stride;
  a.q_out = g.q_out;
  a.ldq = g.ldq;
  a.qs_out = g.qs_out;
  a.ldqs = g.ldqs;
  a.n_out_cols = g.n_out_cols;
  a.dots = g.dots;
  a.err = g.err;
  a.wait_ns = g.wait_ns ? g.wait_ns : kWaitLimitNs;
  a.skip_stage = g.skip_stage;
  a.b_pre = g.b_static ? 1 : 0;
  const int total = a.m_tiles * a.n_tiles * a.splits;
  const int grid = std::max(1, std::min(total, num_sms));
  return launch_pdl(gemm_q8_kernel<BN, EPI>, grid, kThreads, C::SMEM, st, maps.a, maps.b, maps.sa,
                    maps.sb, a);
}

}  // namespace

int tensor_map_2d(CUtensorMap* map, const void* base, bool f32, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  return make_map(map, base, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  inner, outer, row_bytes, box_inner, box_outer,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

GemmPlan gemm_plan(int64_t M, int64_t N, int nb, int num_sms, bool allow_split) {
  GemmPlan p;
  const int64_t mt = (M + kBM - 1) / kBM;
  const int stages = (nb + 1) / 2;
  // one tile width (128 columns) for every shape
  p.bn = 128;
  const int64_t tiles = mt * ((N + p.bn - 1) / p.bn);
  p.splits = 1;
  if (allow_split && tiles < num_sms) {
    // split K so that every SM gets work, keeping >= 2 stages (4 blocks) per split
    int s = (int)std::min<int64_t>(num_sms / std::max<int64_t>(tiles, 1), stages / 2);
    p.splits = std::max(1, s);
  }
  return p;
}

int gemm_make_maps(const GemmOperand& A, const GemmOperand& B, int bn, GemmMaps* maps) {
  const uint64_t kpad = (uint64_t)B.nb * 32;
  int r = 0;
  r |= make_map(&maps->a, A.codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kpad, (uint64_t)A.rows,
                kpad * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  r |= make_map(&maps->b, B.codes, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kpad, (uint64_t)B.rows,
                kpad * 2, kBK, (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_128B);
  r |= make_map(&maps->sa, A.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)A.rows_pad,
                (uint64_t)A.nb, (uint64_t)A.rows_pad * 4, kBM, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
  r |= make_map(&maps->sb, B.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)B.rows_pad,
                (uint64_t)B.nb, (uint64_t)B.rows_pad * 4, (uint32_t)bn, 2,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  return r ? -1 : 0;
}

cudaError_t gemm_launch(const GemmLaunch& g, const GemmMaps& maps, int num_sms,
                        cudaStream_t stream) {
  if (g.A.nb != g.B.nb || g.plan.bn != 128) return cudaErrorInvalidValue;
  switch (g.epi) {
    case kEpiF32: return launch_bn<128, kEpiF32>(g, maps, num_sms, stream);
    case kEpiSwiGLU: return launch_bn<128, kEpiSwiGLU>(g, maps, num_sms, stream);
    case kEpiDots: return launch_bn<128, kEpiDots>(g, maps, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace minfer

// k_attn_tc.cu -- causal GQA attention on the 5th-generation tensor cores
// (tcgen05.mma with TMEM accumulators, TMA-fed), for calls of 64 rows and
// more (the forward uses it from 128 rows on); short calls (the last-row tail,
// single tokens) keep k_attn.cu.
//
// What it computes ("09 · Prefill: the first forward", section 2.2: token t
// attends to positions 0..=pos[t]; "05 · Graph build", section 2.5: GQA,
// scale 1/sqrt(head_dim)):
//     o[t, h] = sum_{j <= pos[t]} softmax_j(q[t,h] . K[j, g] / sqrt(hd)) V[j, g],
//     g = h / (n_head / n_head_kv)
//
// Design.  One CTA per (128 query rows, query head, key split).  Every f32
// operand is split into fp16 hi + lo and the three significant products are
// accumulated (about 22 significant bits, the precision the Q8_0 output
// needs), as in the k_attn.cu kernel:
//   S  = Qh.Kh^T + Qh.Kl^T + Ql.Kh^T        M = 128 rows, N = 64 keys, K = hd
//   Ot = Ph.Vh + Ph.Vl + Pl.Vh              M = 128 rows, N = hd, K = 64 keys
// warp 0 loads the Q tile (hi/lo planes written by the RoPE kernel) and
// streams K (hi/lo shadow planes) and V^T (hi/lo transposed planes) tiles
// with TMA into two-stage rings; one thread of warp 1 issues the S MMAs into
// two TMEM buffers, one thread of warp 10 the P.V MMAs, which accumulate O in
// TMEM over the key tiles.  Warps 2-9 run the softmax, two threads per query
// row (the two warps of a TMEM lane quadrant): both read the whole S row and
// take the same max after the causal mask (log2 units), each exponentiates
// half of the keys into P's hi/lo in shared memory for the P.V MMA, owns half
// of O's columns and keeps its part of the row sum.  The reference max moves
// only when a row's scores rise more than 2^8 above it; O in TMEM is then
// rescaled in place before the next P.V, and every four tiles the tensor-core
// sum is folded into a second TMEM part with round-to-nearest adds.  S of tile
// j+1 is computed while tile j's softmax runs, and P of tile j+1 while P.V of
// tile j runs.
// With few row tiles the key range is split over the CTAs of a cluster,
// merged through distributed shared memory as in k_attn.cu.  The output row
// is normalized and each 32-block quantized to Q8_0 by the thread owning it.
// Every wait is bounded; on timeout the kernel records a status code,
// drains its own TMA loads and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {

constexpr int kTcRows = 128;    // query rows per CTA (MMA M)
constexpr int kTcKeys = 64;     // keys per tile (N of the S MMA, K of the P.V MMA)
constexpr int kTcThreads = 352;  // TMA warp, S issuer, eight softmax warps, P.V issuer
constexpr int kPvWarp = 10;
constexpr int kSmWarps = 8;  // two per TMEM lane quadrant: two threads per query row
constexpr int kTcMaxSplits = 8;  // CTAs per cluster (portable cluster size)

// Largest rise of a row's scores over its reference max (log2 units) that is
// absorbed without rescaling O: P then stays below 2^8.
constexpr float kLazyMax = 8.0f;
// Key tiles accumulated by the tensor core into T before T is folded into R.
constexpr int kFoldTiles = 4;
constexpr uint32_t kTcolT = 128;  // TMEM column of T; R follows at kTcolT + hd
// Two P buffers (fp16 hi/lo, 64 keys: 32 columns each, 64 per buffer) after
// R, so the softmax of tile j+1 need not wait for the P.V of tile j.  (The Q
// tile stays in shared memory: copying it into TMEM as the S MMA's A operand,
// as P is for P.V, cost 0.3% of the 0.5B forward in the copy's latency.)
template <int HD>
struct TcCols {
  static constexpr uint32_t R = kTcolT + HD;
  static constexpr uint32_t P = R + HD;  // buffer b at P + b * kTcKeys
  static constexpr uint32_t END = P + 2 * kTcKeys;
  static_assert(END <= 512, "TMEM columns");
};

template <int HD>
struct TcCfg {
  static constexpr int QSUB = kTcRows * 128;   // bytes of one 64-wide swizzled Q sub-tile
  static constexpr int KSUB = kTcKeys * 128;   // one 64-wide K sub-tile
  static constexpr int Q_BYTES = kTcRows * HD * 2;
  static constexpr int K_BYTES = kTcKeys * HD * 2;
  static constexpr int V_BYTES = HD * kTcKeys * 2;  // V^T tile [hd][64 keys]
  static constexpr int STAGES = 2;
  static constexpr int OFF_QH = 0;
  static constexpr int OFF_QL = OFF_QH + Q_BYTES;
  static constexpr int OFF_K = OFF_QL + Q_BYTES;            // stage s: hi, lo
  static constexpr int OFF_V = OFF_K + STAGES * 2 * K_BYTES;  // stage s: hi, lo
  static constexpr int OFF_P = OFF_V + STAGES * 2 * V_BYTES;  // end of the V ring (P is in TMEM)
  static constexpr int OFF_BAR = OFF_P;
  static constexpr int NBAR = 4 * STAGES + 4 + 3 + 4 + 1 + 2;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEM + 16 + 1024;
  // the split-merge partials reuse the K/V rings: o [128 rows][hd], then
  // (max, sum) [128 rows][2]
  static constexpr int PART_ML = kTcRows * HD;  // float offset of the (max, sum) pairs
  // the two threads of a row exchange their partial sums at the end of the V ring
  static constexpr int OFF_LX = OFF_P - 2 * kTcRows * 4;
  static_assert(OFF_K + kTcRows * (HD + 2) * 4 <= OFF_LX, "sum exchange clear of the partials");
  static_assert(kTcRows * (HD + 2) * 4 <= OFF_P - OFF_K, "partials fit the K/V rings");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0, "1024-B alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM columns: S buffers at 0 and 64, the accumulating O part T at 128,
  // the folded part R after it
  static constexpr uint32_t TCOLS = 512;
};

struct TcArgs {
  const int32_t* pos;
  int r0, r1, nh, nkv, n_ctx;
  int* err;
};

__device__ __forceinline__ uint32_t cluster_rank_tc() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_tc() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t peer_addr_tc(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_peer2_tc(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_peer4_tc(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// 32 lanes x 32 columns of 32-bit TMEM words from registers (thread i -> row
// lane base + i), and the wait for this thread's TMEM stores.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 columns of 32-bit TMEM words from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


template <int HD, bool kGemvOut>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmKh, const __grid_constant__ CUtensorMap tmKl,
                   const __grid_constant__ CUtensorMap tmVh, const __grid_constant__ CUtensorMap tmVl,
                   const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmQl,
                   const TcArgs a, const AttnOut out) {
  using C = TcCfg<HD>;
  constexpr uint32_t kTcolR = kTcolT + (uint32_t)HD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kempty = kfull + C::STAGES;
  uint64_t* vfull = kempty + C::STAGES;
  uint64_t* vempty = vfull + C::STAGES;
  uint64_t* sready = vempty + C::STAGES;  // [2]
  uint64_t* sfree = sready + 2;           // [2]
  uint64_t* pready = sfree + 2;   // [2] P buffer b written by the softmax warps
  uint64_t* oready = pready + 2;  // [2] the P.V that read P buffer b has completed
  uint64_t* qready = oready + 2;
  uint64_t* mdone = qready + 1;  // [2] each issuer's MMAs completed (before TMEM is freed)
  uint64_t* lsum = mdone + 2;    // the two halves of every row have published their sums
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
  __shared__ int s_maxp;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.nh / a.nkv;
  const int ns = (int)gridDim.x;
  const int split = (int)cluster_rank_tc();
  const int tile = (int)gridDim.z - 1 - (int)blockIdx.z;  // longest rows first
  const int h = blockIdx.y;
  const int g = h / G;
  const int rbase = a.r0 + tile * kTcRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sready[b], 1);
      mbar_init(&sfree[b], kSmWarps);
    }
    mbar_init(&pready[0], kSmWarps);
    mbar_init(&pready[1], kSmWarps);
    mbar_init(lsum, kSmWarps);
    mbar_init(&oready[0], 1);
    mbar_init(&oready[1], 1);
    mbar_init(qready, 1);
    mbar_init(&mdone[0], 1);
    mbar_init(&mdone[1], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmKh);
    tma_prefetch_desc(&tmKl);
    tma_prefetch_desc(&tmVh);
    tma_prefetch_desc(&tmVl);
    tma_prefetch_desc(&tmQh);
    tma_prefetch_desc(&tmQl);
    s_maxp = -1;
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_trigger();

  auto clamp_pos = [&](int r) -> int {
    if (r >= a.r1) return -1;
    const int p = a.pos[r];
    return p < 0 ? -1 : (p >= a.n_ctx ? a.n_ctx - 1 : p);
  };
  // the positions are the call's input, written before any kernel: their max
  // is taken while the previous kernel finishes
  if (threadIdx.x < kTcRows) atomicMax(&s_maxp, clamp_pos(rbase + threadIdx.x));
  pdl_wait();
  __syncthreads();
  const int nkeys = s_maxp + 1;
  int share = (nkeys + ns - 1) / ns;
  share = (share + kTcKeys - 1) / kTcKeys * kTcKeys;
  const int kbeg = split * share;
  const int kend = min(nkeys, kbeg + share);
  const int ntile = kend > kbeg ? (kend - kbeg + kTcKeys - 1) / kTcKeys : 0;

  uint8_t* sQh = smem + C::OFF_QH;
  uint8_t* sQl = smem + C::OFF_QL;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0 && ntile > 0) {
      // the Q tile (hi, lo), rows past the call's last are filled with zeros
      mbar_arrive_expect_tx(qready, 2 * C::Q_BYTES);
#pragma unroll
      for (int sub = 0; sub < HD / 64; ++sub) {
        tma_load_2d(sQh + sub * C::QSUB, &tmQh, qready, h * HD + sub * 64, rbase);
        tma_load_2d(sQl + sub * C::QSUB, &tmQl, qready, h * HD + sub * 64, rbase);
      }
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < ntile && ok; ++j) {
        const int st = j % C::STAGES;
        const uint32_t par = ((j / C::STAGES) & 1) ^ 1;
        const int key0 = kbeg + j * kTcKeys;
        if (!mbar_wait(&kempty[st], par, a.err, kDevTimeoutAttn)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kfull[st], 2 * C::K_BYTES);
        uint8_t* kh = smem + C::OFF_K + st * 2 * C::K_BYTES;
#pragma unroll
        for (int sub = 0; sub < HD / 64; ++sub) {
          tma_load_2d(kh + sub * C::KSUB, &tmKh, &kfull[st], g * HD + sub * 64, key0);
          tma_load_2d(kh + C::K_BYTES + sub * C::KSUB, &tmKl, &kfull[st], g * HD + sub * 64, key0);
        }
        if (!mbar_wait(&vempty[st], par, a.err, kDevTimeoutAttn)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&vfull[st], 2 * C::V_BYTES);
        uint8_t* vh = smem + C::OFF_V + st * 2 * C::V_BYTES;
        tma_load_2d(vh, &tmVh, &vfull[st], key0, g * HD);
        tma_load_2d(vh + C::V_BYTES, &tmVl, &vfull[st], key0, g * HD);
        issued = j + 1;
      }
      if (!ok) {
        mbar_wait(qready, 0, a.err, kDevTimeoutAttn);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j) {
          mbar_wait(&kfull[j % C::STAGES], (j / C::STAGES) & 1, a.err, kDevTimeoutAttn);
          mbar_wait(&vfull[j % C::STAGES], (j / C::STAGES) & 1, a.err, kDevTimeoutAttn);
        }
      }
    }
  } else if (warp == 1 || warp == kPvWarp) {
    // ---------------------------------------------------------- MMA issuers
    // S = Q.K^T (warp 1) and O += P.V (warp 10) have an issuing thread each.
    // P is the A operand of P.V straight from TMEM: that MMA then reads only
    // V^T from shared memory; S reads Q and K from shared memory.
    if (lane == 0 && ntile > 0) {
      using TC = TcCols<HD>;
      constexpr uint32_t idS = idesc_f16_f32(kTcRows, kTcKeys);
      constexpr uint32_t idO = idesc_f16_f32(kTcRows, HD);
      const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl);
      const uint32_t ph0 = tmem_base + TC::P;  // P buffer b: hi at ph0 + 64 b, lo 32 columns on
      const uint32_t tO = tmem_base + kTcolT;
      bool ok = true;
      bool committed = false;
      auto issue_s = [&](int j) -> bool {
        const int st = j % C::STAGES, b = j & 1;
        if (!mbar_wait(&kfull[st], (j / C::STAGES) & 1, a.err, kDevTimeoutAttn)) return false;
        if (!mbar_wait(&sfree[b], ((j >> 1) & 1) ^ 1, a.err, kDevTimeoutAttn)) return false;
        tc_fence_after();
        const uint32_t kh = smem_u32(smem + C::OFF_K + st * 2 * C::K_BYTES);
        const uint32_t kl = kh + C::K_BYTES;
        const uint32_t d = tmem_base + (uint32_t)(b * kTcKeys);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const uint32_t B = c == 1 ? kl : kh;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint32_t off = (uint32_t)((k & 3) * 32);
            const uint64_t bd = smem_desc_sw128(B + (k >> 2) * C::KSUB + off);
            const uint32_t A = c == 2 ? ql : qh;
            tc_mma_f16(d, smem_desc_sw128(A + (k >> 2) * C::QSUB + off), bd, idS,
                       (c == 0 && k == 0) ? 0u : 1u);
          }
        }
        tc_commit(&sready[b]);
        tc_commit(&kempty[st]);
        committed = true;
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int st = j % C::STAGES, pb = j & 1;
        if (!mbar_wait(&pready[pb], (j >> 1) & 1, a.err, kDevTimeoutAttn)) return false;
        const uint32_t ph = ph0 + (uint32_t)(pb * kTcKeys), pl = ph + kTcKeys / 2;
        if (!mbar_wait(&vfull[st], (j / C::STAGES) & 1, a.err, kDevTimeoutAttn)) return false;
        tc_fence_after();
        const uint32_t vh = smem_u32(smem + C::OFF_V + st * 2 * C::V_BYTES);
        const uint32_t vl = vh + C::V_BYTES;
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const uint32_t A = c == 2 ? pl : ph;
          const uint32_t B = c == 1 ? vl : vh;
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            const uint32_t off = (uint32_t)(k * 32);
            // T accumulates over the key tiles since the last fold (rescaled in
            // place by the softmax warps); the first tile after a fold restarts it.
            // P in TMEM: 16 keys along K = 8 columns per step.
            tc_mma_f16_ts(tO, A + (uint32_t)(8 * k), smem_desc_sw128(B + off), idO,
                          (j % kFoldTiles == 0 && c == 0 && k == 0) ? 0u : 1u);
          }
        }
        tc_commit(&oready[pb]);
        tc_commit(&vempty[st]);
        committed = true;
        return true;
      };
      if (warp == 1) {
        // Q in shared memory (TMA)
        ok = mbar_wait(qready, 0, a.err, kDevTimeoutAttn);
        if (ok) tc_fence_after();
        for (int j = 0; j < ntile && ok; ++j) ok = issue_s(j);
      } else {
        for (int j = 0; j < ntile && ok; ++j) ok = issue_pv(j);
      }
      // every MMA this thread issued must have landed before TMEM is released
      if (committed) {
        uint64_t* md = &mdone[warp == 1 ? 0 : 1];
        tc_commit(md);
        mbar_wait(md, 0, a.err, kDevTimeoutAttn);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax rows
    // Two threads per row (warps w and w + 4 share a TMEM lane quadrant): both
    // read the whole S row and take the same max; each exponentiates its half
    // of the keys, owns half of O's columns and keeps its part of the sum.
    const int quad = warp & 3;                // TMEM lane quadrant
    const int kh = (warp - 2) >> 2;           // key half of S, column half of O
    const int rl = quad * 32 + lane;          // row within the tile
    const int r = rbase + rl;
    const int pr = clamp_pos(r);
    const int q = a.nh * HD;
    const uint32_t lanebase = (uint32_t)(quad * 32) << 16;

    constexpr int HO = HD / 2;     // O columns of this thread
    const uint32_t ocol = (uint32_t)(kh * HO);
    float m = -INFINITY, l = 0.f;  // reference max (log2 units) and this half's sum of P against it
    // scores in log2 units: s2 = (q.k) / sqrt(hd) * log2(e)
    const float sc = __fmul_rn(__fdiv_rn(1.0f, __fsqrt_rn((float)HD)), 1.4426950408889634f);
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&sready[b], (j >> 1) & 1, a.err, kDevTimeoutAttn)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kTcKeys];
      tmem_ld32(tmem_base + lanebase + (uint32_t)(b * kTcKeys),
                *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tmem_base + lanebase + (uint32_t)(b * kTcKeys + 32),
                *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[b]);
      const int nvalid = pr - (kbeg + j * kTcKeys);  // keys c <= nvalid are visible
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kTcKeys; ++c) {
        const float s2 = (c <= nvalid) ? __fmul_rn(__uint_as_float(sr[c]), sc) : -INFINITY;
        sr[c] = __float_as_uint(s2);
        mx4[c & 3] = fmaxf(mx4[c & 3], s2);
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // The reference max moves only when a score exceeds it by more than
      // kLazyMax (P stays below 2^kLazyMax, well inside f32 and fp16); the O
      // accumulated in TMEM and the sum l are then rescaled by alpha.
      float alpha = 1.f;
      bool resc = false;
      if (mx > m + kLazyMax) {
        if (m != -INFINITY) {
          alpha = exp2f(m - mx);
          resc = true;
        }
        m = mx;
        l *= alpha;
      }
      // this half's P -> fp16 hi/lo words, held until the P buffer is free.  A
      // row whose reference max is still -inf has only -inf scores: exp2(-inf) = 0.
      const float mref = (m == -INFINITY) ? 0.f : m;
      uint32_t hi[kTcKeys / 4], lo[kTcKeys / 4];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t sh[kTcKeys / 2];  // this thread's key half (selected, not indexed, to stay in registers)
#pragma unroll
      for (int i = 0; i < kTcKeys / 2; ++i) sh[i] = kh ? sr[kTcKeys / 2 + i] : sr[i];
#pragma unroll
      for (int i = 0; i < kTcKeys / 4; ++i) {
        const float p0 = exp2f(__fsub_rn(__uint_as_float(sh[2 * i]), mref));
        const float p1 = exp2f(__fsub_rn(__uint_as_float(sh[2 * i + 1]), mref));
        l4[i & 3] += __fadd_rn(p0, p1);
        const __half2 h = __floats2half2_rn(p0, p1);
        const float2 hf = __half22float2(h);
        const __half2 lw = __floats2half2_rn(__fsub_rn(p0, hf.x), __fsub_rn(p1, hf.y));
        hi[i] = *reinterpret_cast<const uint32_t*>(&h);
        lo[i] = *reinterpret_cast<const uint32_t*>(&lw);
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      // O = R + T: T is what the tensor core accumulated since the last fold,
      // R (TMEM too) the sum of the folded parts.  Every kFoldTiles tiles T is
      // added into R with round-to-nearest f32 adds, and the next P.V starts T
      // afresh, so no long sum builds up inside the tensor core.  A fold or a
      // rescale of O needs the previous P.V to have completed; otherwise only
      // the P.V two tiles back, which read the P buffer this tile writes.
      const bool fold = j > 0 && (j % kFoldTiles) == 0;
      const bool touch_o = j > 0 && (fold || __any_sync(0xffffffffu, resc));
      const int jw = touch_o ? j - 1 : j - 2;  // the P.V to wait for
      if (jw >= 0) {
        if (!mbar_wait(&oready[jw & 1], (jw >> 1) & 1, a.err, kDevTimeoutAttn)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      {
        const bool has_r = j > kFoldTiles;  // an earlier fold wrote R
        if (touch_o) {
#pragma unroll
          for (int d0 = 0; d0 < HO; d0 += 32) {
            uint32_t t[32], rr[32];
            tmem_ld32(tmem_base + lanebase + kTcolT + ocol + (uint32_t)d0, t);
            if (has_r) tmem_ld32(tmem_base + lanebase + kTcolR + ocol + (uint32_t)d0, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float rv = has_r ? __uint_as_float(rr[i]) : 0.f;
              const float tv = __uint_as_float(t[i]);
              if (fold) {
                rr[i] = __float_as_uint(__fmul_rn(__fadd_rn(rv, tv), alpha));
              } else {
                // rows whose reference max moved: O *= alpha (alpha = 1 elsewhere)
                rr[i] = __float_as_uint(__fmul_rn(rv, alpha));
                t[i] = __float_as_uint(__fmul_rn(tv, alpha));
              }
            }
            if (fold || has_r) tmem_st32(tmem_base + lanebase + kTcolR + ocol + (uint32_t)d0, rr);
            if (!fold) tmem_st32(tmem_base + lanebase + kTcolT + ocol + (uint32_t)d0, t);
          }
          tmem_wait_st();
        }
      }
      // this half's P (keys kh*32.. of the row, two fp16 per column) into the
      // TMEM columns the P.V MMA reads as its A operand
      const uint32_t pcol = TcCols<HD>::P + (uint32_t)((j & 1) * kTcKeys);
      tmem_st16(tmem_base + lanebase + pcol + (uint32_t)(kh * kTcKeys / 4), hi);
      tmem_st16(tmem_base + lanebase + pcol + kTcKeys / 2 + (uint32_t)(kh * kTcKeys / 4), lo);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[j & 1]);
    }
    // the last P.V completes the O tile
    float o[HO];
#pragma unroll
    for (int d = 0; d < HO; ++d) o[d] = 0.f;
    if (ok && ntile > 0) {
      if (!mbar_wait(&oready[(ntile - 1) & 1], ((ntile - 1) >> 1) & 1, a.err, kDevTimeoutAttn)) {
        ok = false;
      } else {
        tc_fence_after();
        const bool has_r = ntile - 1 >= kFoldTiles;  // some tile folded T into R
#pragma unroll
        for (int d0 = 0; d0 < HO; d0 += 32) {
          uint32_t t[32], rr[32];
          tmem_ld32(tmem_base + lanebase + kTcolT + ocol + (uint32_t)d0, t);
          if (has_r) tmem_ld32(tmem_base + lanebase + kTcolR + ocol + (uint32_t)d0, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            o[d0 + i] = has_r ? __fadd_rn(__uint_as_float(rr[i]), __uint_as_float(t[i]))
                              : __uint_as_float(t[i]);
        }
      }
    }

    // the row's sum: this half's plus the other's (the K/V rings are idle
    // once the last P.V has completed)
    if (ntile > 0) {
      float* lx = reinterpret_cast<float*>(smem + C::OFF_LX);
      lx[kh * kTcRows + rl] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(lsum);
      if (ok && mbar_wait(lsum, 0, a.err, kDevTimeoutAttn))
        l = __fadd_rn(lx[rl], lx[kTcRows + rl]);  // same order on both threads
      else
        ok = false;
    }

    // ------------------------------------------------------- merge + output
    const int nb = q / 32;
    auto emit = [&](const float* v, float inv) {
      if (r >= a.r1) return;
      const int64_t orow = r - out.row_base;
#pragma unroll
      for (int bq = 0; bq < HO / 32; ++bq) {
        float y[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          y[i] = __fmul_rn(v[bq * 32 + i], inv);
          amax = fmaxf(amax, fabsf(y[i]));
        }
        const int k0 = h * HD + (int)ocol + bq * 32;
        const int blk = k0 / 32;
        if (out.f32)
#pragma unroll
          for (int i = 0; i < 32; ++i) out.f32[(int64_t)r * q + k0 + i] = y[i];
        const float dd = __fdiv_rn(amax, 127.0f);
        const float id = q8_inv(dd);
        const float d16 = __half2float(__float2half_rn(dd));
        if (kGemvOut) {
#pragma unroll
          for (int i = 0; i < 32; ++i) out.q8[orow * (int64_t)nb * 32 + k0 + i] = (int8_t)q8_code(y[i], id);
          out.s8[orow * nb + blk] = d16;
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            __half2 c0 = __floats2half2_rn(q8_code(y[i], id), q8_code(y[i + 1], id));
            __half2 c1 = __floats2half2_rn(q8_code(y[i + 2], id), q8_code(y[i + 3], id));
            __half2 c2 = __floats2half2_rn(q8_code(y[i + 4], id), q8_code(y[i + 5], id));
            __half2 c3 = __floats2half2_rn(q8_code(y[i + 6], id), q8_code(y[i + 7], id));
            w.x = *reinterpret_cast<uint32_t*>(&c0);
            w.y = *reinterpret_cast<uint32_t*>(&c1);
            w.z = *reinterpret_cast<uint32_t*>(&c2);
            w.w = *reinterpret_cast<uint32_t*>(&c3);
            *reinterpret_cast<uint4*>(out.q16 + orow * out.ldq + k0 + i) = w;
          }
          out.s16[(int64_t)blk * out.ldqs + orow] = d16;
        }
      }
    };
    if (ns == 1) {
      if (ok) emit(o, l > 0.f ? __fdiv_rn(1.0f, l) : 0.f);
    } else {
      // partials into this CTA's K/V rings (idle now), merged after the cluster barrier
      float* po = reinterpret_cast<float*>(smem + C::OFF_K);
#pragma unroll
      for (int d = 0; d < HO; d += 4)
        *reinterpret_cast<float4*>(po + rl * HD + ocol + d) =
            make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]);
      if (kh == 0) *reinterpret_cast<float2*>(po + C::PART_ML + rl * 2) = make_float2(m, l);
    }
  }

  if (ns > 1) {
    __syncthreads();
    cluster_sync_tc();
    // merge: CTA `split` takes rows rl = split, split + ns, ...; TPR threads
    // per row, 16 consecutive dims each (a 32-block spans two neighbouring
    // threads), so every row of the CTA merges at once: each thread loads the
    // (max, sum) of every split and its 16 values of every split, combines them
    // and quantizes its half block
    constexpr int TPR = HD / 16;
    const uint32_t po_s = smem_u32(smem + C::OFF_K);
    const int q = a.nh * HD;
    const int nb = q / 32;
    const int nrows = (kTcRows - split + ns - 1) / ns;
    const int items = nrows * TPR;
    for (int base = 0; base < items; base += kTcThreads) {  // CTA-uniform bound
      const int idx = base + (int)threadIdx.x;
      const int part = idx % TPR;
      const int rl = split + ns * (idx / TPR);
      const int r = rbase + rl;
      const bool valid = idx < items && r < a.r1;  // equal on both threads of a block
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = 0.f;
      float amax = 0.f;
      if (valid) {
        float ms[kTcMaxSplits], ls[kTcMaxSplits];
        float4 xs[kTcMaxSplits][4];
#pragma unroll
        for (int sdx = 0; sdx < kTcMaxSplits; ++sdx) {
          ms[sdx] = -INFINITY;
          ls[sdx] = 0.f;
          if (sdx < ns) {
            const float2 ml = ld_peer2_tc(
                peer_addr_tc(po_s + (uint32_t)((C::PART_ML + rl * 2) * 4), (uint32_t)sdx));
            ms[sdx] = ml.x;
            ls[sdx] = ml.y;
            const uint32_t pa =
                peer_addr_tc(po_s + (uint32_t)((rl * HD + part * 16) * 4), (uint32_t)sdx);
#pragma unroll
            for (int i = 0; i < 4; ++i) xs[sdx][i] = ld_peer4_tc(pa + 16u * i);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int sdx = 0; sdx < kTcMaxSplits; ++sdx)
          if (sdx < ns) M = fmaxf(M, ms[sdx]);
        float L = 0.f;
#pragma unroll
        for (int sdx = 0; sdx < kTcMaxSplits; ++sdx) {
          if (sdx < ns) {
            const float w = ms[sdx] != -INFINITY ? exp2f(ms[sdx] - M) : 0.f;
            L = fmaf(w, ls[sdx], L);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              y[4 * i + 0] = fmaf(xs[sdx][i].x, w, y[4 * i + 0]);
              y[4 * i + 1] = fmaf(xs[sdx][i].y, w, y[4 * i + 1]);
              y[4 * i + 2] = fmaf(xs[sdx][i].z, w, y[4 * i + 2]);
              y[4 * i + 3] = fmaf(xs[sdx][i].w, w, y[4 * i + 3]);
            }
          }
        }
        const float inv = L > 0.f ? __fdiv_rn(1.0f, L) : 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          y[i] = __fmul_rn(y[i], inv);
          amax = fmaxf(amax, fabsf(y[i]));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      if (valid) {
        const int k0 = h * HD + part * 16;  // first element of this thread in the output row
        const int blk = k0 / 32;
        if (out.f32)
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(out.f32 + (int64_t)r * q + k0 + i) =
                make_float4(y[i], y[i + 1], y[i + 2], y[i + 3]);
        const float dd = __fdiv_rn(amax, 127.0f);
        const float id = q8_inv(dd);
        const float d16 = __half2float(__float2half_rn(dd));
        const int64_t orow = r - out.row_base;
        if (kGemvOut) {
          uint32_t wv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            wv[i] = (uint32_t)(uint8_t)(int8_t)q8_code(y[4 * i], id) |
                    ((uint32_t)(uint8_t)(int8_t)q8_code(y[4 * i + 1], id) << 8) |
                    ((uint32_t)(uint8_t)(int8_t)q8_code(y[4 * i + 2], id) << 16) |
                    ((uint32_t)(uint8_t)(int8_t)q8_code(y[4 * i + 3], id) << 24);
          *reinterpret_cast<uint4*>(out.q8 + orow * (int64_t)nb * 32 + k0) =
              make_uint4(wv[0], wv[1], wv[2], wv[3]);
          if ((part & 1) == 0) out.s8[orow * nb + blk] = d16;
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 8) {
            uint4 w;
            __half2 c0 = __floats2half2_rn(q8_code(y[i], id), q8_code(y[i + 1], id));
            __half2 c1 = __floats2half2_rn(q8_code(y[i + 2], id), q8_code(y[i + 3], id));
            __half2 c2 = __floats2half2_rn(q8_code(y[i + 4], id), q8_code(y[i + 5], id));
            __half2 c3 = __floats2half2_rn(q8_code(y[i + 6], id), q8_code(y[i + 7], id));
            w.x = *reinterpret_cast<uint32_t*>(&c0);
            w.y = *reinterpret_cast<uint32_t*>(&c1);
            w.z = *reinterpret_cast<uint32_t*>(&c2);
            w.w = *reinterpret_cast<uint32_t*>(&c3);
            *reinterpret_cast<uint4*>(out.q16 + orow * out.ldq + k0 + i) = w;
          }
          if ((part & 1) == 0) out.s16[(int64_t)blk * out.ldqs + orow] = d16;
        }
      }
    }
    cluster_sync_tc();  // peers may still be reading this CTA's partials
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TCOLS);
}

}  // namespace

bool attention_tc_supported(const AttnArgs& a) {
  return (a.hd == 64 || a.hd == 128) && a.r1 - a.r0 >= 64 && a.vt[0] && a.vt[1] && a.qp[0] &&
         a.qp[1] && a.vt_ld % 64 == 0 && ((int64_t)a.nkv * a.hd) % 8 == 0;
}

bool attention_tc_preferred(int rows, int nh, int num_sms) {
  // from one full 128-row tile on; shorter calls keep the mma.sync kernel's
  // 16-row tiles
  (void)nh;
  (void)num_sms;
  return rows >= kTcRows;
}

int attention_tc_nsplit(int rows, int nh, int num_sms) {
  const int ctas = (rows + kTcRows - 1) / kTcRows * nh;
  // split the keys when the (row tile, head) pairs leave at least half of the
  // SMs idle: ns CTAs per pair, one wave (0.5B shape, 512 rows: 56 pairs, 2 splits)
  if (2 * ctas > num_sms) return 1;
  const int ns = num_sms / std::max(ctas, 1);
  return ns < 1 ? 1 : (ns > kTcMaxSplits ? kTcMaxSplits : ns);
}

template <int HD, bool kGemvOut>
cudaError_t launch_tc(const AttnArgs& a, const AttnOut& out, int ns, int* err, cudaStream_t st) {
  using C = TcCfg<HD>;
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, kGemvOut>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    set = true;
  }
  const int64_t kvw = (int64_t)a.nkv * HD;
  const int64_t qw = (int64_t)a.nh * HD;
  CUtensorMap mk[2], mv[2], mq[2];
  for (int i = 0; i < 2; ++i) {
    if (tensor_map_2d(&mk[i], a.shadow[i], false, (uint64_t)kvw, (uint64_t)a.n_ctx,
                      (uint64_t)kvw * 2, 64, kTcKeys, true) ||
        tensor_map_2d(&mv[i], a.vt[i], false, (uint64_t)a.vt_ld, (uint64_t)kvw,
                      (uint64_t)a.vt_ld * 2, kTcKeys, HD, true) ||
        tensor_map_2d(&mq[i], a.qp[i], false, (uint64_t)qw, (uint64_t)a.r1, (uint64_t)qw * 2, 64,
                      kTcRows, true))
      return cudaErrorInvalidValue;
  }
  TcArgs t;
  t.pos = a.pos;
  t.r0 = a.r0;
  t.r1 = a.r1;
  t.nh = a.nh;
  t.nkv = a.nkv;
  t.n_ctx = a.n_ctx;
  t.err = err;
  const int rows = a.r1 - a.r0;
  cudaLaunchConfig_t cfg = {};
  // the cluster's CTAs (key splits) along x, heads along y, row tiles along z
  // with the longest rows first, so that every head's longest tiles start in
  // the first wave
  cfg.gridDim = dim3(ns, a.nh, (rows + kTcRows - 1) / kTcRows);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, kGemvOut>, mk[0], mk[1], mv[0], mv[1], mq[0],
                            mq[1], t, out);
}

cudaError_t attention_tc_launch(const AttnArgs& a, const AttnOut& out, int num_sms, int* err,
                                cudaStream_t st) {
  if (!attention_tc_supported(a) || a.nh % a.nkv != 0) return cudaErrorInvalidValue;
  const int ns = attention_tc_nsplit(a.r1 - a.r0, a.nh, num_sms);
  const bool gemv = out.q8 != nullptr;
  if (a.hd == 64)
    return gemv ? launch_tc<64, true>(a, out, ns, err, st) : launch_tc<64, false>(a, out, ns, err, st);
  return gemv ? launch_tc<128, true>(a, out, ns, err, st) : launch_tc<128, false>(a, out, ns, err, st);
}

}  // namespace minfer

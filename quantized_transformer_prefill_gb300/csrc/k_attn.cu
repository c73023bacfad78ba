// k_attn.cu -- causal GQA attention over the persistent KV regions.
//
// What it computes ("09 · Prefill: the first forward", section 2.2: token t
// attends to positions 0..=pos[t]; "05 · Graph build — the IR and the
// builder", section 2.5: GQA, scale 1/sqrt(head_dim)):
//     o[t, h] = sum_{j <= pos[t]} softmax_j(q[t,h] . K[j, g] / sqrt(hd)) V[j, g],
//     g = h / (n_head / n_head_kv)
//
// Design.  One CTA per (16 * R query rows, KV head g, key split): warp w
// serves 16 of the rows for query head g * G + (w % G), so the G heads that
// share a KV head, and R row tiles (R = 8 / G when a group is small), share
// every K/V tile in shared memory.  K/V tiles come from fp16 hi/lo shadow planes of the
// f32 regions (written next to the regions by the RoPE/store kernel), staged
// with double-buffered cp.async.  Scores and P.V run on the tensor cores
// (mma.sync m16n8k16, fp16 operands, f32 accumulate) with every f32 operand
// split as hi + lo and the three significant cross products accumulated
// (about 22 significant bits, the precision the Q8_0 quantization of the
// output needs).  The softmax is online: running row max and sum in f32,
// reduced across the four lanes of a row with warp shuffles.
//
// Short prompts have too few (rows, KV head) tiles to fill the GPU, so the
// key range of each tile is split (the split-KV scheme of the pages' CUDA
// backend) across the CTAs of one thread-block cluster: each CTA covers a
// contiguous share of the keys 0..max position of its rows, leaves its
// unnormalized output and (max, sum) in its own shared memory, and after a
// cluster barrier every CTA merges a share of the (row, head, 32-block)
// units by reading its peers' partials through distributed shared memory,
// normalizes, and quantizes each 32-block of the output row to Q8_0 for the
// o-projection.  No partials go through global memory and no second kernel
// runs; without a split the cluster is one CTA.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {

constexpr int kMaxSplits = 8;  // CTAs per cluster (portable cluster size)
constexpr int kTileQ = 16;     // query rows per CTA
constexpr int kTileKV = 32;  // keys per shared-memory tile

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices, transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_t(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_peer2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// f32 pair -> (hi, lo) fp16x2 words with x = hi + lo to ~22 bits.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  const __half l0 = __float2half_rn(__fsub_rn(x0, __half2float(h0)));
  const __half l1 = __float2half_rn(__fsub_rn(x1, __half2float(h1)));
  hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
  lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
}

template <int HD>
struct Tile {
  static constexpr int RS = HD + 8;            // row stride (halves), conflict-free
  static constexpr int PLANE = kTileKV * RS;   // halves per plane
  static constexpr int STAGE = 4 * PLANE;      // Kh, Kl, Vh, Vl
  static constexpr int BYTES = 2 * STAGE * 2;  // two stages, 2 B per half
  // after the key loop the same bytes hold the CTA's partial result:
  // o [16 rows][G heads][HD] and (max, sum) [16][G][2], f32
  static constexpr int PART_BYTES = (kTileQ * 8 * HD + kTileQ * 8 * 2) * 4;  // G <= 8
  static_assert(PART_BYTES <= BYTES, "partials must fit the staging buffers");
};

template <int HD, bool kGemvOut>
__global__ void __launch_bounds__(256) attn_kernel(const AttnArgs a, const AttnOut out) {
  using T = Tile<HD>;
  extern __shared__ __align__(16) __half smem_h[];
  __shared__ int s_maxp;
  pdl_trigger();
  pdl_wait();

  const int G = a.nh / a.nkv;
  const int ns = (int)gridDim.z;  // key splits = CTAs of this cluster
  const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest rows first
  const int g = blockIdx.y;
  const int split = (int)cluster_rank();
  // R row tiles of 16 per CTA when a KV group has few heads (R * G <= 8
  // warps share every K/V tile); warp = (row tile tl, head hg of the group)
  const int nw = (int)(blockDim.x >> 5);
  const int R = nw / G;
  const int rbase = a.r0 + tile * kTileQ * R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = warp / G, hg = warp - tl * G;
  const int h = g * G + hg;
  const int wbase = rbase + tl * kTileQ;  // this warp's 16 rows
  const int qr = lane >> 2, qc = (lane & 3) * 2;
  const int64_t qw = (int64_t)a.nh * HD;
  const int64_t kw = (int64_t)a.nkv * HD;

  auto clamp_pos = [&](int r) -> int {
    if (r >= a.r1) return -1;
    const int p = a.pos[r];
    return p < 0 ? -1 : (p >= a.n_ctx ? a.n_ctx - 1 : p);
  };
  if (threadIdx.x == 0) s_maxp = -1;
  __syncthreads();
  if (threadIdx.x < kTileQ * R) atomicMax(&s_maxp, clamp_pos(rbase + threadIdx.x));
  __syncthreads();
  // this split's share of the keys 0..max position of the tile's rows
  const int nkeys = s_maxp + 1;
  int share = (nkeys + ns - 1) / ns;
  share = (share + kTileKV - 1) / kTileKV * kTileKV;
  const int kbeg = split * share;
  const int kend = min(nkeys, kbeg + share);
  const int ntile = kend > kbeg ? (kend - kbeg + kTileKV - 1) / kTileKV : 0;

  const int ra = wbase + qr, rb = wbase + qr + 8;
  const int pa = clamp_pos(ra), pb = clamp_pos(rb);

  // stage loader: 32 keys x HD of Kh, Kl, Vh, Vl in 16-byte chunks
  const uint32_t sbase = smem_u32(smem_h);
  auto load_tile = [&](int t, int stage) {
    const int key0 = kbeg + t * kTileKV;
    constexpr int CPR = HD / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < 4 * kTileKV * CPR; c += blockDim.x) {
      const int plane = c / (kTileKV * CPR);
      const int rem = c % (kTileKV * CPR);
      const int j = rem / CPR, ch = rem % CPR;
      const int key = key0 + j;
      const bool ok = key < a.n_ctx;
      const __half* pbase =
          plane == 0 ? a.shadow[0] : (plane == 1 ? a.shadow[1] : (plane == 2 ? a.shadow[2] : a.shadow[3]));
      const __half* src = pbase + (int64_t)(ok ? key : 0) * kw + (int64_t)g * HD + ch * 8;
      const uint32_t dst =
          sbase + 2u * (uint32_t)(stage * T::STAGE + plane * T::PLANE + j * T::RS + ch * 8);
      cp_async16(dst, src, ok);
    }
    cp_async_commit();
  };
  if (ntile > 0) load_tile(0, 0);

  // Q fragments (A operand, row-major 16 x HD), split into fp16 hi/lo
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  {
    const float* qa = a.q + (int64_t)ra * qw + (int64_t)h * HD;
    const float* qb = a.q + (int64_t)rb * qw + (int64_t)h * HD;
    const bool va = ra < a.r1, vb = rb < a.r1;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const int c0 = kk * 16 + qc;
      const float2 x0 = va ? *reinterpret_cast<const float2*>(qa + c0) : make_float2(0.f, 0.f);
      const float2 x1 = vb ? *reinterpret_cast<const float2*>(qb + c0) : make_float2(0.f, 0.f);
      const float2 x2 = va ? *reinterpret_cast<const float2*>(qa + c0 + 8) : make_float2(0.f, 0.f);
      const float2 x3 = vb ? *reinterpret_cast<const float2*>(qb + c0 + 8) : make_float2(0.f, 0.f);
      split2(x0.x, x0.y, qh[kk][0], ql[kk][0]);
      split2(x1.x, x1.y, qh[kk][1], ql[kk][1]);
      split2(x2.x, x2.y, qh[kk][2], ql[kk][2]);
      split2(x3.x, x3.y, qh[kk][3], ql[kk][3]);
    }
  }

  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  // scores are kept in log2 units: s2 = (q.k) / sqrt(hd) * log2(e)
  const float sc = __fmul_rn(__fdiv_rn(1.0f, __fsqrt_rn((float)HD)), 1.4426950408889634f);
  const int mi = lane >> 3, mr = lane & 7;

  for (int t = 0; t < ntile; ++t) {
    const int stage = t & 1;
    if (t + 1 < ntile) {
      load_tile(t + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __half* Kh = smem_h + stage * T::STAGE;
    const __half* Kl = Kh + T::PLANE;
    const uint32_t vh_base = sbase + 2u * (uint32_t)(stage * T::STAGE + 2 * T::PLANE);
    const uint32_t vl_base = vh_base + 2u * (uint32_t)T::PLANE;
    const int key0 = kbeg + t * kTileKV;

    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    // the three products of one accumulator are issued four MMAs apart (one
    // per key group), so consecutive mma.sync never wait on each other
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t bh[4][2], bl[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const __half* kh = Kh + (nt * 8 + qr) * T::RS + kk * 16 + qc;
        const __half* kl = Kl + (nt * 8 + qr) * T::RS + kk * 16 + qc;
        bh[nt][0] = *reinterpret_cast<const uint32_t*>(kh);
        bh[nt][1] = *reinterpret_cast<const uint32_t*>(kh + 8);
        bl[nt][0] = *reinterpret_cast<const uint32_t*>(kl);
        bl[nt][1] = *reinterpret_cast<const uint32_t*>(kl + 8);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) mma16816(s[nt], qh[kk], bh[nt][0], bh[nt][1]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) mma16816(s[nt], qh[kk], bl[nt][0], bl[nt][1]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) mma16816(s[nt], ql[kk], bh[nt][0], bh[nt][1]);
    }

    // mask, online softmax
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = key0 + nt * 8 + qc + c;
        s[nt][c] = (j <= pa) ? __fmul_rn(s[nt][c], sc) : -INFINITY;
        s[nt][2 + c] = (j <= pb) ? __fmul_rn(s[nt][2 + c], sc) : -INFINITY;
        mx_a = fmaxf(mx_a, s[nt][c]);
        mx_b = fmaxf(mx_b, s[nt][2 + c]);
      }
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float ca = (mn_a == -INFINITY) ? 1.f : exp2f(m_a - mn_a);
    const float cb = (mn_b == -INFINITY) ? 1.f : exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;
    l_a *= ca;
    l_b *= cb;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= ca; o[i][1] *= ca;
      o[i][2] *= cb; o[i][3] *= cb;
    }
    uint32_t ph[2][4], pl[2][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = (s[nt][0] == -INFINITY) ? 0.f : exp2f(s[nt][0] - m_a);
      const float p1 = (s[nt][1] == -INFINITY) ? 0.f : exp2f(s[nt][1] - m_a);
      const float p2 = (s[nt][2] == -INFINITY) ? 0.f : exp2f(s[nt][2] - m_b);
      const float p3 = (s[nt][3] == -INFINITY) ? 0.f : exp2f(s[nt][3] - m_b);
      l_a += p0 + p1;
      l_b += p2 + p3;
      const int ks = nt >> 1, hi8 = nt & 1;
      split2(p0, p1, ph[ks][hi8 * 2 + 0], pl[ks][hi8 * 2 + 0]);
      split2(p2, p3, ph[ks][hi8 * 2 + 1], pl[ks][hi8 * 2 + 1]);
    }
    // O += P V: B fragments of V (keys x dims) by transposing ldmatrix
    // four output tiles per group, their three products interleaved as above
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int ng = 0; ng < HD / 8; ng += 4) {
        uint32_t vh[8], vl[8];
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          const uint32_t off = 2u * (uint32_t)((ks * 16 + (mi & 1) * 8 + mr) * T::RS +
                                               (ng + 2 * p2) * 8 + (mi >> 1) * 8);
          ldsm_x4_t(vh_base + off, vh[4 * p2], vh[4 * p2 + 1], vh[4 * p2 + 2], vh[4 * p2 + 3]);
          ldsm_x4_t(vl_base + off, vl[4 * p2], vl[4 * p2 + 1], vl[4 * p2 + 2], vl[4 * p2 + 3]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) mma16816(o[ng + t], ph[ks], vh[2 * t], vh[2 * t + 1]);
#pragma unroll
        for (int t = 0; t < 4; ++t) mma16816(o[ng + t], ph[ks], vl[2 * t], vl[2 * t + 1]);
#pragma unroll
        for (int t = 0; t < 4; ++t) mma16816(o[ng + t], pl[ks], vh[2 * t], vh[2 * t + 1]);
      }
    }
    __syncthreads();  // the next prefetch overwrites this stage's buffer
  }

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

  const int nblk = HD / 32;
  const int q = a.nh * HD;
  const int nb = q / 32;
  const int r_a = wbase + qr, r_b = wbase + qr + 8;
  // Normalized values of this thread's 8 + 8 elements of 32-block bq (rows
  // r_a, r_b; dims bq*32 + i*8 + qc + {0,1}) -> f32 (debug), Q8_0 codes and
  // the block scale.  The four lanes of a row hold the whole block.
  auto emit = [&](int bq, const float (&va)[8], const float (&vb)[8]) {
    float ma = 0.f, mb = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ma = fmaxf(ma, fabsf(va[i]));
      mb = fmaxf(mb, fabsf(vb[i]));
    }
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const int kb = h * HD + bq * 32;  // first element of the block in the output row
    const int b = kb / 32;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? r_b : r_a;
      if (r >= a.r1) continue;
      const float* v = half ? vb : va;
      const float amax = half ? mb : ma;
      const float dd = __fdiv_rn(amax, 127.0f);
      const float id = q8_inv(dd);
      const int64_t orow = r - out.row_base;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = kb + i * 8 + qc;
        if (out.f32) *reinterpret_cast<float2*>(out.f32 + (int64_t)r * q + k) = make_float2(v[2 * i], v[2 * i + 1]);
        const float c0 = q8_code(v[2 * i], id), c1 = q8_code(v[2 * i + 1], id);
        if (kGemvOut) {
          out.q8[orow * (int64_t)nb * 32 + k] = (int8_t)c0;
          out.q8[orow * (int64_t)nb * 32 + k + 1] = (int8_t)c1;
        } else {
          *reinterpret_cast<__half2*>(out.q16 + orow * out.ldq + k) = __floats2half2_rn(c0, c1);
        }
      }
      if ((lane & 3) == 0) {
        const float d16 = __half2float(__float2half_rn(dd));
        if (kGemvOut)
          out.s8[orow * nb + b] = d16;
        else
          out.s16[(int64_t)b * out.ldqs + orow] = d16;
      }
    }
  };

  if (ns == 1) {
    // the whole key range is here: normalize and quantize from registers
    const float ia = l_a > 0.f ? __fdiv_rn(1.0f, l_a) : 0.f;
    const float ib = l_b > 0.f ? __fdiv_rn(1.0f, l_b) : 0.f;
#pragma unroll
    for (int bq = 0; bq < nblk; ++bq) {
      float va[8], vb[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        va[2 * i] = __fmul_rn(o[4 * bq + i][0], ia);
        va[2 * i + 1] = __fmul_rn(o[4 * bq + i][1], ia);
        vb[2 * i] = __fmul_rn(o[4 * bq + i][2], ib);
        vb[2 * i + 1] = __fmul_rn(o[4 * bq + i][3], ib);
      }
      emit(bq, va, vb);
    }
    return;  // a cluster of one: nothing to wait for
  }

  // partial result into this CTA's shared memory (the staging buffers are
  // free once every warp has left the key loop)
  __syncthreads();
  float* po = reinterpret_cast<float*>(smem_h);  // [16][G][HD]
  float* pml = po + kTileQ * nw * HD;            // [16][warps][2]
#pragma unroll
  for (int nd = 0; nd < HD / 8; ++nd) {
    *reinterpret_cast<float2*>(po + ((qr * nw) + warp) * HD + nd * 8 + qc) =
        make_float2(o[nd][0], o[nd][1]);
    *reinterpret_cast<float2*>(po + (((qr + 8) * nw) + warp) * HD + nd * 8 + qc) =
        make_float2(o[nd][2], o[nd][3]);
  }
  if ((lane & 3) == 0) {
    *reinterpret_cast<float2*>(pml + (qr * nw + warp) * 2) = make_float2(m_a, l_a);
    *reinterpret_cast<float2*>(pml + ((qr + 8) * nw + warp) * 2) = make_float2(m_b, l_b);
  }
  cluster_sync_all();

  // merge: the (head, 32-block) units are dealt round the CTAs of the
  // cluster; the warp of that head merges its 16 rows from every CTA's
  // partials (distributed shared memory) at its own fragment positions
  const uint32_t po_s = smem_u32(po), pml_s = smem_u32(pml);
  const uint32_t mla_off = (uint32_t)((qr * nw + warp) * 2 * 4);
  const uint32_t mlb_off = (uint32_t)(((qr + 8) * nw + warp) * 2 * 4);
  for (int bq = 0; bq < nblk; ++bq) {
    if ((warp * nblk + bq) % ns != split) continue;  // warp-uniform
    float2 mla[kMaxSplits], mlb[kMaxSplits];
    float Ma = -INFINITY, Mb = -INFINITY;
#pragma unroll
    for (int sidx = 0; sidx < kMaxSplits; ++sidx) {
      if (sidx < ns) {
        mla[sidx] = ld_peer2(peer_addr(pml_s + mla_off, (uint32_t)sidx));
        mlb[sidx] = ld_peer2(peer_addr(pml_s + mlb_off, (uint32_t)sidx));
        Ma = fmaxf(Ma, mla[sidx].x);
        Mb = fmaxf(Mb, mlb[sidx].x);
      }
    }
    float va[8], vb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) va[i] = vb[i] = 0.f;
    float La = 0.f, Lb = 0.f;
#pragma unroll
    for (int sidx = 0; sidx < kMaxSplits; ++sidx) {
      if (sidx < ns) {
        const float wa = (mla[sidx].x == -INFINITY) ? 0.f : exp2f(mla[sidx].x - Ma);
        const float wb = (mlb[sidx].x == -INFINITY) ? 0.f : exp2f(mlb[sidx].x - Mb);
        La = fmaf(mla[sidx].y, wa, La);
        Lb = fmaf(mlb[sidx].y, wb, Lb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int dim = bq * 32 + i * 8 + qc;
          const float2 xa = ld_peer2(peer_addr(po_s + (uint32_t)(((qr * nw + warp) * HD + dim) * 4), (uint32_t)sidx));
          const float2 xb = ld_peer2(peer_addr(po_s + (uint32_t)((((qr + 8) * nw + warp) * HD + dim) * 4), (uint32_t)sidx));
          va[2 * i] = fmaf(xa.x, wa, va[2 * i]);
          va[2 * i + 1] = fmaf(xa.y, wa, va[2 * i + 1]);
          vb[2 * i] = fmaf(xb.x, wb, vb[2 * i]);
          vb[2 * i + 1] = fmaf(xb.y, wb, vb[2 * i + 1]);
        }
      }
    }
    const float ia = La > 0.f ? __fdiv_rn(1.0f, La) : 0.f;
    const float ib = Lb > 0.f ? __fdiv_rn(1.0f, Lb) : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      va[i] = __fmul_rn(va[i], ia);
      vb[i] = __fmul_rn(vb[i], ib);
    }
    emit(bq, va, vb);
  }
  // peers may still be reading this CTA's partials
  cluster_sync_all();
}

__global__ void split_planes_kernel(const float* __restrict__ x, int64_t count, __half* hi,
                                    __half* lo) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float v = x[i];
    const __half h = __float2half_rn(v);
    hi[i] = h;
    lo[i] = __float2half_rn(__fsub_rn(v, __half2float(h)));
  }
}

// K/V rows of one layer -> fp16 hi/lo shadow planes (count f32 values each).
__global__ void kv_shadow_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                 int64_t count, __half* kh, __half* kl, __half* vh, __half* vl,
                                 __half* vth, __half* vtl, int64_t vt_ld, int row0, int kvw) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = k[i], y = v[i];
    const __half xh = __float2half_rn(x), yh = __float2half_rn(y);
    const __half yl = __float2half_rn(__fsub_rn(y, __half2float(yh)));
    kh[i] = xh;
    kl[i] = __float2half_rn(__fsub_rn(x, __half2float(xh)));
    vh[i] = yh;
    vl[i] = yl;
    const int64_t row = row0 + i / kvw, e = i % kvw;
    vth[e * vt_ld + row] = yh;
    vtl[e * vt_ld + row] = yl;
  }
}

// ---------------------------------------------------------------- one query row
// A call with a single query row (a one-token call, the last row of a prompt)
// has almost no work per KV head: the tiled kernel's 16-row MMA tiles are all
// latency there.  Here one thread-block cluster of CS CTAs (16 where the
// device allows that non-portable size, else 8) serves a KV head; CTA c takes
// the c-th share of the keys 0..pos.  A CTA walks its
// share in chunks of kRowKeys K and V rows of the f32 regions, staged in
// shared memory (the next chunk's loads are in flight while the current one
// is scored); warp h scores the chunk for query head h of the group, one key
// per lane, in f32 on the CUDA cores, keeps the softmax online and
// accumulates P.V with lane l holding dims l + 32 j.  After a cluster barrier
// CTA h merges head h from its peers' (max, sum, O) through distributed
// shared memory, normalizes and quantizes; a second barrier keeps every CTA
// alive until its partials have been read.
constexpr int kRowKeys = 32;    // keys per chunk
constexpr int kRowThreadsA = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int HD, int CS>
__global__ void __launch_bounds__(kRowThreadsA) attn_row_kernel(const AttnArgs a, const AttnOut out) {
  static_assert(CS >= 8, "CTA h merges query head h < G <= 8");
  constexpr int DPL = HD / 32;                      // dims per lane
  constexpr int C4 = HD / 4;                        // float4 per row
  constexpr int PER = kRowKeys * C4 / kRowThreadsA;  // float4 of K (and of V) per thread and chunk
  static_assert(PER * kRowThreadsA == kRowKeys * C4, "whole chunks per thread");
  __shared__ float ks[kRowKeys][HD + 1];  // +1: lane = key reads a column without bank conflicts
  __shared__ __align__(16) float vs[kRowKeys][HD];
  __shared__ float qs[8][HD];
  __shared__ float po[8][HD];  // this CTA's unnormalized O, per query head of the group
  __shared__ float pml[8][2];  // and its (max, sum)
  pdl_trigger();

  const int G = a.nh / a.nkv;
  const int g = blockIdx.y;
  const int split = (int)cluster_rank();
  const int ns = CS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = a.r0;
  const int64_t kw = (int64_t)a.nkv * HD;
  const int64_t qw = (int64_t)a.nh * HD;
  int p = a.pos[r];  // the positions are the call's input, written before any kernel
  p = p < 0 ? -1 : (p >= a.n_ctx ? a.n_ctx - 1 : p);
  const int nkeys = p + 1;
  const int share = (nkeys + ns - 1) / ns;
  const int kbeg = min(nkeys, split * share);
  const int kend = min(nkeys, kbeg + share);
  const int nchunks = (kend - kbeg + kRowKeys - 1) / kRowKeys;
  // scores in log2 units: s = (q.k) / sqrt(hd) * log2(e)
  const float sc = __fmul_rn(__fdiv_rn(1.0f, __fsqrt_rn((float)HD)), 1.4426950408889634f);

  float4 kr[PER], vr[PER];  // the next chunk, in flight
  auto load_chunk = [&](int k0) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = tid + kRowThreadsA * i;
      const int kk = idx / C4, c = idx % C4;
      kr[i] = vr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k0 + kk < kend) {
        const int64_t off = (int64_t)(k0 + kk) * kw + (int64_t)g * HD + 4 * c;
        kr[i] = *reinterpret_cast<const float4*>(a.kreg + off);
        vr[i] = *reinterpret_cast<const float4*>(a.vreg + off);
      }
    }
  };
  // the first chunk before the wait for the previous kernel when none of its
  // rows is the one that kernel wrote (row p)
  const bool early = a.kv_static_below && nchunks > 0 && min(kbeg + kRowKeys, kend) <= p;
  if (early) load_chunk(kbeg);
  pdl_wait();
  // the group's query rows load next to the chunk
  for (int i = tid; i < G * HD; i += kRowThreadsA)
    qs[i / HD][i % HD] = a.q[(int64_t)r * qw + (int64_t)g * G * HD + i];
  if (nchunks > 0 && !early) load_chunk(kbeg);

  float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] = 0.f;
  for (int ci = 0; ci < nchunks; ++ci) {
    const int k0 = kbeg + ci * kRowKeys;
    const int nc = min(kRowKeys, kend - k0);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = tid + kRowThreadsA * i;
      const int kk = idx / C4, c = idx % C4;
      ks[kk][4 * c] = kr[i].x;
      ks[kk][4 * c + 1] = kr[i].y;
      ks[kk][4 * c + 2] = kr[i].z;
      ks[kk][4 * c + 3] = kr[i].w;
      *reinterpret_cast<float4*>(&vs[kk][4 * c]) = vr[i];
    }
    __syncthreads();
    if (ci + 1 < nchunks) load_chunk(k0 + kRowKeys);
    if (warp < G) {
      const int h = warp;
      float d4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial dots: shorter dependency chains
#pragma unroll 8
      for (int d = 0; d < HD; d += 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) d4[e] = fmaf(qs[h][d + e], ks[lane][d + e], d4[e]);
      }
      const float dot = __fadd_rn(__fadd_rn(d4[0], d4[1]), __fadd_rn(d4[2], d4[3]));
      const float s = lane < nc ? __fmul_rn(dot, sc) : -INFINITY;
      const float m_new = fmaxf(m, warp_max(s));
      const float corr = m == -INFINITY ? 1.f : exp2f(m - m_new);
      const float pk = lane < nc ? exp2f(s - m_new) : 0.f;
      l = __fadd_rn(__fmul_rn(l, corr), warp_sum(pk));
      m = m_new;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[j] *= corr;
      for (int kk = 0; kk < nc; ++kk) {
        const float pb = __shfl_sync(0xffffffffu, pk, kk);
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = fmaf(pb, vs[kk][lane + 32 * j], o[j]);
      }
    }
    __syncthreads();  // the next chunk overwrites ks / vs
  }
  if (warp < G) {
#pragma unroll
    for (int j = 0; j < DPL; ++j) po[warp][lane + 32 * j] = o[j];
    if (lane == 0) {
      pml[warp][0] = m;
      pml[warp][1] = l;
    }
  }
  cluster_sync_all();  // every CTA's partials are visible to the cluster

  if (split < G && warp == 0) {
    // merge head h = split from the ns CTAs: weights exp2(m_s - M), then 1 / L
    const int h = split;
    const uint32_t ml_s = smem_u32(&pml[h][0]);
    float ms[CS], ls[CS];
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      const float2 v = ld_peer2(peer_addr(ml_s, (uint32_t)c));
      ms[c] = v.x;
      ls[c] = v.y;
    }
    float x[CS][DPL];
#pragma unroll
    for (int c = 0; c < CS; ++c)
#pragma unroll
      for (int j = 0; j < DPL; ++j)
        x[c][j] = ld_peer(peer_addr(smem_u32(&po[h][lane + 32 * j]), (uint32_t)c));
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CS; ++c) M = fmaxf(M, ms[c]);
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      const float w = ms[c] == -INFINITY ? 0.f : exp2f(ms[c] - M);
      L = fmaf(ls[c], w, L);
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[j] = fmaf(x[c][j], w, acc[j]);
    }
    const float il = L > 0.f ? __fdiv_rn(1.0f, L) : 0.f;
    // Q8_0: block j of head h is dims 32 j .. 32 j + 31, one per lane
    const int q = a.nh * HD;
    const int nb = q / 32;
    const int64_t orow = r - out.row_base;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const float v = __fmul_rn(acc[j], il);
      const int k = (g * G + h) * HD + 32 * j + lane;  // element of the output row
      const int b = k / 32;
      const float amax = warp_max(fabsf(v));
      const float dd = __fdiv_rn(amax, 127.0f);
      const float code = q8_code(v, q8_inv(dd));
      if (out.f32) out.f32[(int64_t)r * q + k] = v;
      const float d16 = __half2float(__float2half_rn(dd));
      if (out.q8) {
        out.q8[orow * (int64_t)nb * 32 + k] = (int8_t)code;
        if (lane == 0) out.s8[orow * nb + b] = d16;
      } else {
        out.q16[orow * out.ldq + k] = __float2half_rn(code);
        if (lane == 0) out.s16[(int64_t)b * out.ldqs + orow] = d16;
      }
    }
  }
  cluster_sync_all();  // peers may still be reading this CTA's partials
}

}  // namespace

// 16-row tiles per CTA: enough to give the CTA 8 warps when a KV group has
// few query heads.
int attn_row_tiles(int G) { return G >= 8 ? 1 : 8 / G; }

int attention_nsplit(int rows, int nkv, int num_sms, int G) {
  const int rtiles = attn_row_tiles(G);
  const int ctas = (rows + kTileQ * rtiles - 1) / (kTileQ * rtiles) * nkv;
  if (ctas >= num_sms) return 1;
  int ns = (2 * num_sms + ctas - 1) / std::max(ctas, 1);
  return ns < 1 ? 1 : (ns > kMaxSplits ? kMaxSplits : ns);
}

template <int HD, bool kGemvOut>
cudaError_t launch_attn(const AttnArgs& a, const AttnOut& out, int rows, cudaStream_t st) {
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, kGemvOut>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Tile<HD>::BYTES);
    if (e != cudaSuccess) return e;
    set = true;
  }
  const int G = a.nh / a.nkv;
  cudaLaunchConfig_t cfg = {};
  const int R = attn_row_tiles(G);
  cfg.gridDim = dim3((rows + kTileQ * R - 1) / (kTileQ * R), a.nkv, a.nsplit);
  cfg.blockDim = dim3(32 * G * R);
  cfg.dynamicSmemBytes = Tile<HD>::BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = a.nsplit;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_kernel<HD, kGemvOut>, a, out);
}

cudaError_t attention_launch(const AttnArgs& a, const AttnOut& out, cudaStream_t st) {
  const int rows = a.r1 - a.r0;
  if (rows <= 0) return cudaSuccess;
  const int G = a.nh / a.nkv;
  if (a.nh % a.nkv != 0 || G > 8 || a.nsplit < 1 || a.nsplit > kMaxSplits)
    return cudaErrorInvalidValue;
  const bool gemv = out.q8 != nullptr;
  if (rows == 1 && a.kreg && a.vreg && reinterpret_cast<uintptr_t>(a.kreg) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(a.vreg) % 16 == 0 && ((int64_t)a.nkv * a.hd) % 4 == 0) {
    // 16 CTAs per cluster where the device allows that size (measured faster
    // than 8 on both single-token shapes), else the portable 8
    static int cs = 0;
    if (cs == 0) {
      cs = 16;
      if (cudaFuncSetAttribute(attn_row_kernel<64, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
              cudaSuccess ||
          cudaFuncSetAttribute(attn_row_kernel<128, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
              cudaSuccess) {
        (void)cudaGetLastError();
        cs = 8;
      }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)a.nkv, 1);
    cfg.blockDim = dim3(kRowThreadsA);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (a.hd == 64)
      return cs == 16 ? cudaLaunchKernelEx(&cfg, attn_row_kernel<64, 16>, a, out)
                      : cudaLaunchKernelEx(&cfg, attn_row_kernel<64, 8>, a, out);
    if (a.hd == 128)
      return cs == 16 ? cudaLaunchKernelEx(&cfg, attn_row_kernel<128, 16>, a, out)
                      : cudaLaunchKernelEx(&cfg, attn_row_kernel<128, 8>, a, out);
    return cudaErrorInvalidValue;
  }
  if (a.hd == 64) return gemv ? launch_attn<64, true>(a, out, rows, st) : launch_attn<64, false>(a, out, rows, st);
  if (a.hd == 128)
    return gemv ? launch_attn<128, true>(a, out, rows, st) : launch_attn<128, false>(a, out, rows, st);
  return cudaErrorInvalidValue;
}

cudaError_t split_planes_launch(const float* x, int64_t count, __half* hi, __half* lo,
                                cudaStream_t st) {
  int64_t g = (count + 255) / 256;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  split_planes_kernel<<<(unsigned)g, 256, 0, st>>>(x, count, hi, lo);
  return cudaGetLastError();
}

cudaError_t kv_shadow_launch(const float* k, const float* v, int64_t count, __half* const* planes,
                             __half* const* vt, int64_t vt_ld, int row0, int kvw,
                             cudaStream_t st) {
  int64_t g = (count + 255) / 256;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  kv_shadow_kernel<<<(unsigned)g, 256, 0, st>>>(k, v, count, planes[0], planes[1], planes[2],
                                                planes[3], vt[0], vt[1], vt_ld, row0, kvw);
  return cudaGetLastError();
}

}  // namespace minfer

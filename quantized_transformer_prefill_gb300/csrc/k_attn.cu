// k_attn.cu -- causal GQA attention over the persistent KV regions.
//
// What it computes ("09 · Prefill: the first forward", section 2.2: token t
// attends to positions 0..=pos[t]; "05 · Graph build — the IR and the
// builder", section 2.5: GQA, scale 1/sqrt(head_dim)):
//     o[t, h] = sum_{j <= pos[t]} softmax_j(q[t,h] . K[j, g] / sqrt(hd)) V[j, g],
//     g = h / (n_head / n_head_kv)
//
// Design: one CTA per (16 query rows, KV head g); warp w of the CTA serves
// query head g * G + w, so the G heads that share a KV head share every K/V
// tile staged in shared memory.  Scores and P.V run on the tensor cores
// (mma.sync m16n8k16, fp16 operands, f32 accumulate) with each f32 operand
// split into an fp16 pair hi + lo and the three significant cross products
// (hi.hi + hi.lo + lo.hi) accumulated, which keeps about 22 significant bits
// -- the precision the following Q8_0 quantization of the output needs.  The
// softmax is online (running row max and sum in f32, reduced across the four
// lanes that share a row with warp shuffles).
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {

constexpr int kTileQ = 16;   // query rows per CTA
constexpr int kTileKV = 32;  // keys per shared-memory tile

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
__global__ void __launch_bounds__(256) attn_kernel(const AttnArgs a) {
  constexpr int KS = HD + 8;       // K tile row stride (halves)
  constexpr int VS = kTileKV + 8;  // V^T tile row stride (halves)
  __shared__ __align__(16) __half sKh[kTileKV * KS];
  __shared__ __align__(16) __half sKl[kTileKV * KS];
  __shared__ __align__(16) __half sVh[HD * VS];
  __shared__ __align__(16) __half sVl[HD * VS];
  __shared__ int s_maxp;

  const int G = a.nh / a.nkv;
  const int g = blockIdx.y;
  const int n_tiles = gridDim.x;
  const int tile = n_tiles - 1 - (int)blockIdx.x;  // longest rows first
  const int rbase = a.r0 + tile * kTileQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = g * G + warp;
  const int qr = lane >> 2, qc = (lane & 3) * 2;
  const int64_t qw = (int64_t)a.nh * HD;
  const int64_t kw = (int64_t)a.nkv * HD;

  auto clamp_pos = [&](int r) -> int {
    if (r >= a.r1) return -1;
    int p = a.pos[r];
    return p < 0 ? -1 : (p >= a.n_ctx ? a.n_ctx - 1 : p);
  };
  const int ra = rbase + qr, rb = rbase + qr + 8;
  const int pa = clamp_pos(ra), pb = clamp_pos(rb);

  if (threadIdx.x == 0) s_maxp = -1;
  __syncthreads();
  if (threadIdx.x < kTileQ) atomicMax(&s_maxp, clamp_pos(rbase + threadIdx.x));
  __syncthreads();
  const int maxp = s_maxp;

  // Q fragments (A operand, row-major 16 x HD), split into fp16 hi/lo.
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  {
    const float* qa = a.q + (int64_t)ra * qw + (int64_t)h * HD;
    const float* qb = a.q + (int64_t)rb * qw + (int64_t)h * HD;
    const bool va = ra < a.r1, vb = rb < a.r1;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const int c0 = kk * 16 + qc;
      float2 x0 = va ? *reinterpret_cast<const float2*>(qa + c0) : make_float2(0.f, 0.f);
      float2 x1 = vb ? *reinterpret_cast<const float2*>(qb + c0) : make_float2(0.f, 0.f);
      float2 x2 = va ? *reinterpret_cast<const float2*>(qa + c0 + 8) : make_float2(0.f, 0.f);
      float2 x3 = vb ? *reinterpret_cast<const float2*>(qb + c0 + 8) : make_float2(0.f, 0.f);
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

  for (int kv0 = 0; kv0 <= maxp; kv0 += kTileKV) {
    __syncthreads();
    // stage K (rows) and V (transposed) of head g, split into fp16 hi/lo
    for (int e = threadIdx.x; e < kTileKV * HD; e += blockDim.x) {
      const int j = e / HD, d = e % HD;
      const int row = kv0 + j;
      float kx = 0.f, vx = 0.f;
      if (row < a.n_ctx) {
        kx = a.k[(int64_t)row * kw + (int64_t)g * HD + d];
        vx = a.v[(int64_t)row * kw + (int64_t)g * HD + d];
      }
      const __half kh = __float2half_rn(kx), vh = __float2half_rn(vx);
      sKh[j * KS + d] = kh;
      sKl[j * KS + d] = __float2half_rn(__fsub_rn(kx, __half2float(kh)));
      sVh[d * VS + j] = vh;
      sVl[d * VS + j] = __float2half_rn(__fsub_rn(vx, __half2float(vh)));
    }
    __syncthreads();

    // S = Q K^T for 32 keys: 4 n-tiles of 8
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const __half* kh = sKh + (nt * 8 + qr) * KS + kk * 16 + qc;
        const __half* kl = sKl + (nt * 8 + qr) * KS + kk * 16 + qc;
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(kh);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(kh + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(kl);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(kl + 8);
        mma16816(s[nt], qh[kk], bh0, bh1);
        mma16816(s[nt], qh[kk], bl0, bl1);
        mma16816(s[nt], ql[kk], bh0, bh1);
      }
    }

    // mask, online softmax
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = kv0 + nt * 8 + qc + c;
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
    // P fragments (A operand of P.V), keys [16 ks, 16 ks + 16)
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
    // O += P V
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int nd = 0; nd < HD / 8; ++nd) {
        const __half* vh = sVh + (nd * 8 + qr) * VS + ks * 16 + qc;
        const __half* vl = sVl + (nd * 8 + qr) * VS + ks * 16 + qc;
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(vh);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(vh + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(vl);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(vl + 8);
        mma16816(o[nd], ph[ks], bh0, bh1);
        mma16816(o[nd], ph[ks], bl0, bl1);
        mma16816(o[nd], pl[ks], bh0, bh1);
      }
    }
  }

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float ia = l_a > 0.f ? __fdiv_rn(1.0f, l_a) : 0.f;
  const float ib = l_b > 0.f ? __fdiv_rn(1.0f, l_b) : 0.f;
  if (ra < a.r1) {
    float* dst = a.o + (int64_t)ra * qw + (int64_t)h * HD + qc;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][0] * ia, o[nd][1] * ia);
  }
  if (rb < a.r1) {
    float* dst = a.o + (int64_t)rb * qw + (int64_t)h * HD + qc;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][2] * ib, o[nd][3] * ib);
  }
}

}  // namespace

cudaError_t attention_launch(const AttnArgs& a, cudaStream_t st) {
  const int rows = a.r1 - a.r0;
  if (rows <= 0) return cudaSuccess;
  const int G = a.nh / a.nkv;
  if (a.nh % a.nkv != 0 || G > 8) return cudaErrorInvalidValue;
  dim3 grid((rows + kTileQ - 1) / kTileQ, a.nkv);
  if (a.hd == 64) attn_kernel<64><<<grid, 32 * G, 0, st>>>(a);
  else if (a.hd == 128) attn_kernel<128><<<grid, 32 * G, 0, st>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace minfer

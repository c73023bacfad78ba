// k_rows.cu -- the memory-bound kernels of the prefill: embedding gather,
// residual-add + RMSNorm + Q8_0 activation quantization, RoPE + KV store,
// input validation, the one-row tail (GEMV, SwiGLU + quantize) and the
// load-time weight quantize/repack kernels.
//
// Q8_0 of a 32-element block (walkthrough index, master table, row "CPU
// matmul kernels": on-the-fly Q8_0 activations; block = 32 int8 codes + one
// fp16 scale): d = amax / 127 (f32), codes = round-half-away(x * (1/d))
// clamped to +-127, stored scale = fp16(d) round-to-nearest-even.  One warp
// owns one block, one lane one element, so amax is a 5-step shuffle max.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {


// ---------------------------------------------------------------- error-free sums
// Knuth's TwoSum and the fma-based TwoProduct: the pair (hi, lo) carries the
// sum of squares to about 48 bits, so the per-row RMS matches a float64
// accumulation.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void ff_add(float& hi, float& lo, float bhi, float blo) {
  float s, e;
  two_sum(hi, bhi, s, e);
  e = __fadd_rn(e, __fadd_rn(lo, blo));
  hi = __fadd_rn(s, e);
  lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// The RMSNorm scale 1 / sqrt(ss / n + eps), rounded to f32, from the sum of
// squares ss held as a float-float pair (hi, lo), in f32 arithmetic only (the
// double pipe of this part is slow, and the scale sits on every row's critical
// path): v = ss / n + eps as a float-float pair (the exact remainder of the
// division by fma), the hardware reciprocal square root of its high part,
// then two Newton-Raphson steps y <- y + y (1 - v y^2) / 2 for 1/sqrt carried
// in float-float, so the result is within a few 2^-47 of the exact value and
// rounds to f32 like a float64 evaluation except that close to a boundary.
__device__ __forceinline__ float rms_scale(float hi, float lo, float n, float eps) {
  const float q1 = __fdiv_rn(hi, n);
  const float r1 = fmaf(-q1, n, hi);  // hi - q1 n, exact
  const float q2 = __fdiv_rn(__fadd_rn(r1, lo), n);
  float vh, vl;
  two_sum(q1, q2, vh, vl);
  ff_add(vh, vl, eps, 0.f);
  if (!(vh > 0.f)) return __frcp_rn(__fsqrt_rn(vh));  // v = 0: inf, as in float64
  float yh = rsqrtf(vh), yl = 0.f;
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    // y^2 = s + se (yl's share to first order)
    const float s = __fmul_rn(yh, yh);
    const float se = fmaf(yh, yh, -s) + 2.0f * yh * yl;
    // v y^2 = t + te
    const float t = __fmul_rn(vh, s);
    const float te = fmaf(vh, s, -t) + (vh * se + vl * s);
    // e = 1 - v y^2 (1 - t is exact: t is close to 1)
    const float e = __fsub_rn(1.0f - t, te);
    // y += y e / 2 as a float-float pair
    const float c = __fmul_rn(0.5f * yh, e) + 0.5f * yl * e;
    float nh, nl;
    two_sum(yh, c, nh, nl);
    yl = nl + yl;
    two_sum(nh, yl, yh, yl);
  }
  return yh;
}

// ---------------------------------------------------------------- row quant
// One CTA of 256 threads per row; thread i holds elements i + 256 k (k < PER,
// all loads issued before any arithmetic).  In step k, warp w holds block
// 8 k + w, so a block's amax is a 5-step shuffle max.  The sum of squares is
// a float-float (hi, lo) pair reduced over the warp, then over the 8 warps.
constexpr int kRowThreads = 256;
constexpr int kMaxPartialSplits = 8;  // split-K partials a row kernel sums (GEMM split cap)

template <bool kGemvOut, int PER>
__global__ void __launch_bounds__(kRowThreads) row_quant_kernel(const RowQuantArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red_hi[kRowThreads / 32], red_lo[kRowThreads / 32];
  __shared__ float s_scale;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const int64_t hr = a.row_offset + r;
  const int64_t n = a.n;
  const int nb = (int)((n + 31) / 32);
  float* hrow = a.h + hr * n;

  float x[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int64_t k = tid + (int64_t)kRowThreads * i;
    x[i] = k < n ? hrow[k] : 0.f;
  }
  if (a.nsplit > 0) {
    float o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int64_t k = tid + (int64_t)kRowThreads * i;
      o[i] = k < n ? a.partials[hr * n + k] : 0.f;
    }
    if constexpr (PER <= 4) {
      // short rows: every split's loads in flight at once, summed in split order
      float ps[kMaxPartialSplits - 1][PER];
#pragma unroll
      for (int s = 1; s < kMaxPartialSplits; ++s) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int64_t k = tid + (int64_t)kRowThreads * i;
          ps[s - 1][i] =
              (s < a.nsplit && k < n) ? a.partials[s * a.split_stride + hr * n + k] : 0.f;
        }
      }
#pragma unroll
      for (int s = 1; s < kMaxPartialSplits; ++s) {
        if (s < a.nsplit) {
#pragma unroll
          for (int i = 0; i < PER; ++i) o[i] = __fadd_rn(o[i], ps[s - 1][i]);
        }
      }
    } else {
      for (int s = 1; s < a.nsplit; ++s) {
        const float* ps = a.partials + s * a.split_stride + hr * n;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int64_t k = tid + (int64_t)kRowThreads * i;
          if (k < n) o[i] = __fadd_rn(o[i], ps[k]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int64_t k = tid + (int64_t)kRowThreads * i;
      if (k < n) {
        x[i] = __fadd_rn(x[i], o[i]);
        hrow[k] = x[i];
      }
    }
  }

  float scale = 1.0f;
  if (a.norm_w) {
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const float p = __fmul_rn(x[i], x[i]);
      ff_add(hi, lo, p, fmaf(x[i], x[i], -p));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float bhi = __shfl_xor_sync(0xffffffffu, hi, o);
      const float blo = __shfl_xor_sync(0xffffffffu, lo, o);
      ff_add(hi, lo, bhi, blo);
    }
    if (lane == 0) {
      red_hi[warp] = hi;
      red_lo[warp] = lo;
    }
    __syncthreads();
    if (tid == 0) {
      float h2 = red_hi[0], l2 = red_lo[0];
      for (int w = 1; w < kRowThreads / 32; ++w) ff_add(h2, l2, red_hi[w], red_lo[w]);
      s_scale = rms_scale(h2, l2, (float)n, a.eps);
    }
    __syncthreads();
    scale = s_scale;
  }

#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int64_t k = tid + (int64_t)kRowThreads * i;
    const int b = 8 * i + warp;
    if (b >= nb) continue;  // warp-uniform
    float y = x[i];
    if (a.norm_w) y = (k < n) ? __fmul_rn(__fmul_rn(y, scale), a.norm_w[k]) : 0.f;
    const float amax = warp_max(fabsf(y));
    const float d = __fdiv_rn(amax, 127.0f);
    const float code = q8_code(y, q8_inv(d));
    const __half d16 = __float2half_rn(d);
    if (kGemvOut) {
      a.q8[r * (int64_t)nb * 32 + k] = (int8_t)code;
      if (lane == 0) {
        a.s8[r * nb + b] = __half2float(d16);
        if (a.s8_bits) a.s8_bits[r * nb + b] = __half_as_ushort(d16);
      }
    } else {
      a.q16[r * a.ldq + k] = __float2half_rn(code);
      if (lane == 0) a.s16[(int64_t)b * a.ldqs + r] = __half2float(d16);
    }
  }
}

// Rows whose length is a multiple of 32 (every hidden width): thread t holds
// the four consecutive elements of chunk t + 256 k (k < PER4; float4 loads and
// stores, all loads issued before any arithmetic), so the 8 chunks of a Q8_0
// block are 8 neighbouring lanes and one warp step quantizes 4 blocks: the
// block amax is a 3-step shuffle and the scale's division and reciprocal are
// issued once per 4 blocks instead of once per block.  Same arithmetic as
// row_quant_kernel element by element (partials summed in split order, then
// the residual add; the sum of squares as float-float pairs; y = (x * r) * w).
// kCG: read h through L2 only (h was written by other CTAs of the running
// grid: the one-row GEMV's fused norm).
template <bool kGemvOut, int PER4, bool kCG>
__device__ __forceinline__ void row_quant4_row(const RowQuantArgs& a, const int64_t r) {
  __shared__ float red_hi[kRowThreads / 32], red_lo[kRowThreads / 32];
  __shared__ float s_scale;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t hr = a.row_offset + r;
  const int64_t n = a.n;
  const int64_t nc = n >> 2;  // float4 chunks of the row
  const int nb = (int)(n >> 5);
  float* hrow = a.h + hr * n;

  float4 x[PER4], w4[PER4];
#pragma unroll
  for (int i = 0; i < PER4; ++i) {
    const int64_t c = tid + (int64_t)kRowThreads * i;
    const float4* src = reinterpret_cast<const float4*>(hrow + 4 * c);
    x[i] = c < nc ? (kCG ? __ldcg(src) : *src) : make_float4(0.f, 0.f, 0.f, 0.f);
    // the norm weights load with the row, ahead of the stores of h (which the
    // compiler cannot move them past)
    w4[i] = (a.norm_w && c < nc) ? *reinterpret_cast<const float4*>(a.norm_w + 4 * c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (a.nsplit > 0) {
    float4 o[PER4];
#pragma unroll
    for (int i = 0; i < PER4; ++i) {
      const int64_t c = tid + (int64_t)kRowThreads * i;
      o[i] = c < nc ? *reinterpret_cast<const float4*>(a.partials + hr * n + 4 * c)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s = 1; s < a.nsplit; ++s) {
      float4 ps[PER4];
#pragma unroll
      for (int i = 0; i < PER4; ++i) {
        const int64_t c = tid + (int64_t)kRowThreads * i;
        ps[i] = c < nc ? *reinterpret_cast<const float4*>(a.partials + s * a.split_stride + hr * n + 4 * c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < PER4; ++i) {
        o[i].x = __fadd_rn(o[i].x, ps[i].x);
        o[i].y = __fadd_rn(o[i].y, ps[i].y);
        o[i].z = __fadd_rn(o[i].z, ps[i].z);
        o[i].w = __fadd_rn(o[i].w, ps[i].w);
      }
    }
#pragma unroll
    for (int i = 0; i < PER4; ++i) {
      const int64_t c = tid + (int64_t)kRowThreads * i;
      if (c < nc) {
        x[i].x = __fadd_rn(x[i].x, o[i].x);
        x[i].y = __fadd_rn(x[i].y, o[i].y);
        x[i].z = __fadd_rn(x[i].z, o[i].z);
        x[i].w = __fadd_rn(x[i].w, o[i].w);
        *reinterpret_cast<float4*>(hrow + 4 * c) = x[i];
      }
    }
  }

  float scale = 1.0f;
  if (a.norm_w) {
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int i = 0; i < PER4; ++i) {
      const float v[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = __fmul_rn(v[e], v[e]);
        ff_add(hi, lo, p, fmaf(v[e], v[e], -p));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float bhi = __shfl_xor_sync(0xffffffffu, hi, o);
      const float blo = __shfl_xor_sync(0xffffffffu, lo, o);
      ff_add(hi, lo, bhi, blo);
    }
    if (lane == 0) {
      red_hi[warp] = hi;
      red_lo[warp] = lo;
    }
    __syncthreads();
    if (tid == 0) {
      float h2 = red_hi[0], l2 = red_lo[0];
      for (int w = 1; w < kRowThreads / 32; ++w) ff_add(h2, l2, red_hi[w], red_lo[w]);
      s_scale = rms_scale(h2, l2, (float)n, a.eps);
    }
    __syncthreads();
    scale = s_scale;
  }

#pragma unroll
  for (int i = 0; i < PER4; ++i) {
    const int64_t c = tid + (int64_t)kRowThreads * i;
    if ((c & ~int64_t(31)) >= nc) continue;  // warp-uniform: nc is a multiple of 8
    const bool in = c < nc;
    float y[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
    if (a.norm_w) {
      const float wv[4] = {w4[i].x, w4[i].y, w4[i].z, w4[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = in ? __fmul_rn(__fmul_rn(y[e], scale), wv[e]) : 0.f;
    }
    float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    if (!in) continue;
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = q8_inv(d);
    const __half d16 = __float2half_rn(d);
    const int b = (int)(c >> 3);
    const bool first = (c & 7) == 0;
    if (kGemvOut) {
      char4 q4;
      q4.x = (signed char)q8_code(y[0], id);
      q4.y = (signed char)q8_code(y[1], id);
      q4.z = (signed char)q8_code(y[2], id);
      q4.w = (signed char)q8_code(y[3], id);
      *reinterpret_cast<char4*>(a.q8 + r * (int64_t)nb * 32 + 4 * c) = q4;
      if (first) {
        a.s8[r * nb + b] = __half2float(d16);
        if (a.s8_bits) a.s8_bits[r * nb + b] = __half_as_ushort(d16);
      }
    } else {
      const __half2 c01 = __floats2half2_rn(q8_code(y[0], id), q8_code(y[1], id));
      const __half2 c23 = __floats2half2_rn(q8_code(y[2], id), q8_code(y[3], id));
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&c01);
      u.y = *reinterpret_cast<const uint32_t*>(&c23);
      *reinterpret_cast<uint2*>(a.q16 + r * a.ldq + 4 * c) = u;
      if (first) a.s16[(int64_t)b * a.ldqs + r] = __half2float(d16);
    }
  }
}

template <bool kGemvOut, int PER4>
__global__ void __launch_bounds__(kRowThreads) row_quant4_kernel(const RowQuantArgs a) {
  pdl_trigger();
  pdl_wait();
  row_quant4_row<kGemvOut, PER4, false>(a, blockIdx.x);
}

template <bool kGemvOut>
cudaError_t row_quant_dispatch(const RowQuantArgs& a, cudaStream_t st) {
  const unsigned grid = (unsigned)a.rows;
  // whole Q8_0 blocks and 16-byte aligned rows: the four-element form
  const bool aligned =
      (a.n % 32) == 0 && (reinterpret_cast<uintptr_t>(a.h) % 16) == 0 &&
      (a.nsplit == 0 || (reinterpret_cast<uintptr_t>(a.partials) % 16 == 0 && a.split_stride % 4 == 0)) &&
      (a.norm_w == nullptr || reinterpret_cast<uintptr_t>(a.norm_w) % 16 == 0) &&
      (kGemvOut ? (reinterpret_cast<uintptr_t>(a.q8) % 4) == 0
                : ((reinterpret_cast<uintptr_t>(a.q16) % 8) == 0 && a.ldq % 4 == 0));
  if (aligned) {
    const int per4 = (int)((a.n / 4 + kRowThreads - 1) / kRowThreads);
    if (per4 <= 1) return launch_pdl(row_quant4_kernel<kGemvOut, 1>, grid, kRowThreads, 0, st, a);
    if (per4 <= 2) return launch_pdl(row_quant4_kernel<kGemvOut, 2>, grid, kRowThreads, 0, st, a);
    if (per4 <= 4) return launch_pdl(row_quant4_kernel<kGemvOut, 4>, grid, kRowThreads, 0, st, a);
  }
  const int per = (int)((a.n + kRowThreads - 1) / kRowThreads);
  if (per <= 1) return launch_pdl(row_quant_kernel<kGemvOut, 1>, grid, kRowThreads, 0, st, a);
  if (per <= 2) return launch_pdl(row_quant_kernel<kGemvOut, 2>, grid, kRowThreads, 0, st, a);
  if (per <= 4) return launch_pdl(row_quant_kernel<kGemvOut, 4>, grid, kRowThreads, 0, st, a);
  if (per <= 8) return launch_pdl(row_quant_kernel<kGemvOut, 8>, grid, kRowThreads, 0, st, a);
  if (per <= 16) return launch_pdl(row_quant_kernel<kGemvOut, 16>, grid, kRowThreads, 0, st, a);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- embedding
__global__ void embed_kernel(const int8_t* __restrict__ q, const float* __restrict__ s,
                             int64_t kpad, int nb, const int32_t* __restrict__ ids, int64_t H,
                             float* __restrict__ h, int n_vocab) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  int id = ids[t];
  id = id < 0 ? 0 : (id >= n_vocab ? n_vocab - 1 : id);  // invalid ids are reported by validation
  const int8_t* qr = q + (int64_t)id * kpad;
  const float* sr = s + (int64_t)id * nb;
  for (int64_t k = threadIdx.x; k < H; k += blockDim.x)
    h[(int64_t)t * H + k] = __fmul_rn(sr[k / 32], (float)qr[k]);
}

// ---------------------------------------------------------------- validation
__global__ void validate_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ pos,
                                int nt, int n_vocab, int n_ctx, uint32_t* seen, int* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int code;
  if (threadIdx.x == 0) code = 0;
  const int words = (n_ctx + 31) / 32;
  for (int i = threadIdx.x; i < words; i += blockDim.x) seen[i] = 0u;
  __syncthreads();
  for (int t = threadIdx.x; t < nt; t += blockDim.x) {
    const int p = pos[t];
    const int id = ids[t];
    if (p < 0 || p >= n_ctx) {
      atomicCAS(&code, 0, MINFER_ERR_POS_OOB);
    } else {
      const uint32_t bit = 1u << (p & 31);
      if (atomicOr(&seen[p >> 5], bit) & bit) atomicCAS(&code, 0, MINFER_ERR_ARG);
    }
    if (id < 0 || id >= n_vocab) atomicCAS(&code, 0, MINFER_ERR_TOKEN_OOB);
  }
  __syncthreads();
  if (threadIdx.x == 0) *status = code;
}

// ---------------------------------------------------------------- RoPE + KV store
// NeoX half-split pairs (x_i, x_{i + hd/2}) rotated by the per-position
// cos/sin table ("09 · Prefill", section 2.2: the positions buffer is the
// rotation angle's input and names the K/V row written).  The products and
// the differences are separate IEEE roundings, as written.
// A rotated Q pair (elements o and o + half of a row) to the f32 output and,
// when present, the fp16 hi/lo planes the tensor-core attention loads by TMA.
__device__ __forceinline__ void store_q(const RopeStoreArgs& a, int64_t o, float v0, float v1,
                                        int half) {
  if (a.q_out) {
    a.q_out[o] = v0;
    a.q_out[o + half] = v1;
  }
  if (a.q_planes[0]) {
    const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
    a.q_planes[0][o] = h0;
    a.q_planes[0][o + half] = h1;
    a.q_planes[1][o] = __float2half_rn(__fsub_rn(v0, __half2float(h0)));
    a.q_planes[1][o + half] = __float2half_rn(__fsub_rn(v1, __half2float(h1)));
  }
}

// Two neighbouring dimensions per thread (i, i + 1 of a head's first half,
// with their partners i + hd/2, i + 1 + hd/2): 8-byte loads and stores, half
// the threads of one per pair, the same arithmetic element by element.
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}
__device__ __forceinline__ void split2(float2 v, __half2& hi, __half2& lo) {
  hi = __floats2half2_rn(v.x, v.y);
  const float2 hf = __half22float2(hi);
  lo = __floats2half2_rn(__fsub_rn(v.x, hf.x), __fsub_rn(v.y, hf.y));
}

__global__ void __launch_bounds__(1024, 2) rope_store_kernel(const RopeStoreArgs a) {
  pdl_trigger();
  const int t = blockIdx.x;
  // the position is the call's input, written before any kernel: read while
  // the previous kernel finishes, so the table rows load with the sums
  const int p_in = a.pos[t];
  pdl_wait();
  // an out-of-range position is reported by validation; it only selects a
  // table row here (clamped) and never a region row
  const bool write_kv =
      status_clear(a.status) && p_in >= 0 && p_in < a.n_ctx;
  const int p = (p_in >= 0 && p_in < a.n_ctx) ? p_in : 0;
  const int half = a.hd >> 1;
  const int qshift = half == 64 ? 5 : 4;  // head_dim is 64 or 128: half/2 dimension pairs per head
  const int W = (a.nh + 2 * a.nkv) * a.hd;
  const int64_t row = (int64_t)t * W;
  const int np2 = (a.nh + a.nkv) * (half >> 1);
  const int kw = a.nkv * a.hd;
  const float* cs = a.cos_t + (int64_t)p * half;
  const float* sn = a.sin_t + (int64_t)p * half;
  for (int pi = threadIdx.x; pi < np2 + (kw >> 1); pi += blockDim.x) {
    if (pi < np2) {
      const int head = pi >> qshift, i = 2 * (pi & ((half >> 1) - 1));
      const int e0 = head * a.hd + i;
      float2 x0 = ld2(a.partials + row + e0), x1 = ld2(a.partials + row + e0 + half);
      for (int s = 1; s < a.nsplit; ++s) {
        const float* ps = a.partials + s * a.split_stride + row;
        x0 = add2(x0, ld2(ps + e0));
        x1 = add2(x1, ld2(ps + e0 + half));
      }
      if (a.bias) {
        x0 = add2(x0, ld2(a.bias + e0));
        x1 = add2(x1, ld2(a.bias + e0 + half));
      }
      const float2 c = ld2(cs + i), sv = ld2(sn + i);
      const float2 v0 = make_float2(__fsub_rn(__fmul_rn(x0.x, c.x), __fmul_rn(x1.x, sv.x)),
                                    __fsub_rn(__fmul_rn(x0.y, c.y), __fmul_rn(x1.y, sv.y)));
      const float2 v1 = make_float2(__fadd_rn(__fmul_rn(x0.x, sv.x), __fmul_rn(x1.x, c.x)),
                                    __fadd_rn(__fmul_rn(x0.y, sv.y), __fmul_rn(x1.y, c.y)));
      __half2 h0, l0, h1, l1;
      split2(v0, h0, l0);
      split2(v1, h1, l1);
      if (head < a.nh) {
        // rotated Q to f32 and, when present, the fp16 hi/lo planes the
        // tensor-core attention loads by TMA
        const int64_t o = (int64_t)t * a.nh * a.hd + e0;
        if (a.q_out) {
          *reinterpret_cast<float2*>(a.q_out + o) = v0;
          *reinterpret_cast<float2*>(a.q_out + o + half) = v1;
        }
        if (a.q_planes[0]) {
          *reinterpret_cast<__half2*>(a.q_planes[0] + o) = h0;
          *reinterpret_cast<__half2*>(a.q_planes[0] + o + half) = h1;
          *reinterpret_cast<__half2*>(a.q_planes[1] + o) = l0;
          *reinterpret_cast<__half2*>(a.q_planes[1] + o + half) = l1;
        }
      } else if (write_kv) {
        const int ke = (head - a.nh) * a.hd + i;
        const int64_t o0 = (int64_t)p * kw + ke;
        *reinterpret_cast<float2*>(a.kreg + o0) = v0;
        *reinterpret_cast<float2*>(a.kreg + o0 + half) = v1;
        *reinterpret_cast<__half2*>(a.shadow[0] + o0) = h0;
        *reinterpret_cast<__half2*>(a.shadow[0] + o0 + half) = h1;
        *reinterpret_cast<__half2*>(a.shadow[1] + o0) = l0;
        *reinterpret_cast<__half2*>(a.shadow[1] + o0 + half) = l1;
      }
    } else if (write_kv) {
      const int e = 2 * (pi - np2);
      const int col = (a.nh + a.nkv) * a.hd + e;
      float2 v = ld2(a.partials + row + col);
      for (int s = 1; s < a.nsplit; ++s) v = add2(v, ld2(a.partials + s * a.split_stride + row + col));
      if (a.bias) v = add2(v, ld2(a.bias + col));
      const int64_t o0 = (int64_t)p * kw + e;
      *reinterpret_cast<float2*>(a.vreg + o0) = v;
      __half2 vh, vl;
      split2(v, vh, vl);
      *reinterpret_cast<__half2*>(a.shadow[2] + o0) = vh;
      *reinterpret_cast<__half2*>(a.shadow[3] + o0) = vl;
      a.vt[0][(int64_t)e * a.vt_ld + p] = __low2half(vh);
      a.vt[0][(int64_t)(e + 1) * a.vt_ld + p] = __high2half(vh);
      a.vt[1][(int64_t)e * a.vt_ld + p] = __low2half(vl);
      a.vt[1][(int64_t)(e + 1) * a.vt_ld + p] = __high2half(vl);
    }
  }
}

// Qwen3: the same with the per-head QK RMSNorm between the bias and RoPE
// ("05 · Graph build", section 3.2, FusedQkvNorm).  One CTA per token: the
// Q and K sums go to shared memory, one warp per head takes the sum of
// squares as float-float pairs, warp 0 turns every head's sum into its scale
// (rms_scale), then the pairs are normalized, weighted and rotated.
constexpr int kMaxQkHeads = 128;

__global__ void __launch_bounds__(1024) rope_store_qknorm_kernel(const RopeStoreArgs a) {
  extern __shared__ float xs[];  // [(nh + nkv) * hd]
  __shared__ float rs[kMaxQkHeads], rl[kMaxQkHeads];  // per head: (hi, lo) sum of squares, then the scale
  pdl_trigger();
  const int t = blockIdx.x;
  const int p_in = a.pos[t];  // the call's input: read before the wait, as above
  pdl_wait();
  const bool write_kv =
      status_clear(a.status) && p_in >= 0 && p_in < a.n_ctx;
  const int p = (p_in >= 0 && p_in < a.n_ctx) ? p_in : 0;
  const int half = a.hd >> 1;
  const int hshift = half == 64 ? 6 : 5;  // head_dim is 64 or 128
  const int nheads = a.nh + a.nkv;
  const int nqk = nheads * a.hd;
  const int W = nqk + a.nkv * a.hd;
  const int64_t row = (int64_t)t * W;
  const int kw = a.nkv * a.hd;
  for (int e = threadIdx.x; e < W; e += blockDim.x) {
    float v = a.partials[row + e];
    for (int s = 1; s < a.nsplit; ++s) v = __fadd_rn(v, a.partials[s * a.split_stride + row + e]);
    if (a.bias) v = __fadd_rn(v, a.bias[e]);
    if (e < nqk) {
      xs[e] = v;
    } else if (write_kv) {
      const int64_t o0 = (int64_t)p * kw + (e - nqk);
      a.vreg[o0] = v;
      const __half vh = __float2half_rn(v);
      const __half vl = __float2half_rn(__fsub_rn(v, __half2float(vh)));
      a.shadow[2][o0] = vh;
      a.shadow[3][o0] = vl;
      a.vt[0][(e - nqk) * a.vt_ld + p] = vh;
      a.vt[1][(e - nqk) * a.vt_ld + p] = vl;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int hh = warp; hh < nheads; hh += nwarps) {
    // the head's sum of squares as float-float pairs (as in the row kernel):
    // the double pipe of this part is too slow for a sum per element
    float hi = 0.f, lo = 0.f;
    for (int i = lane; i < a.hd; i += 32) {
      const float x = xs[hh * a.hd + i];
      const float sq = __fmul_rn(x, x);
      ff_add(hi, lo, sq, fmaf(x, x, -sq));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float bhi = __shfl_xor_sync(0xffffffffu, hi, o);
      const float blo = __shfl_xor_sync(0xffffffffu, lo, o);
      ff_add(hi, lo, bhi, blo);
    }
    if (lane == 0) {
      rs[hh] = hi;
      rl[hh] = lo;
    }
  }
  __syncthreads();
  // the scales of all heads side by side in the lanes of warp 0
  if (warp == 0)
    for (int hh = lane; hh < nheads; hh += 32) rs[hh] = rms_scale(rs[hh], rl[hh], (float)a.hd, a.eps);
  __syncthreads();
  const float* cs = a.cos_t + (int64_t)p * half;
  const float* sn = a.sin_t + (int64_t)p * half;
  for (int pi = threadIdx.x; pi < nheads * half; pi += blockDim.x) {
    const int head = pi >> hshift, i = pi & (half - 1);
    const int e0 = head * a.hd + i;
    const float r = rs[head];
    const float* w = head < a.nh ? a.q_norm : a.k_norm;
    const float x0 = __fmul_rn(__fmul_rn(xs[e0], r), w[i]);
    const float x1 = __fmul_rn(__fmul_rn(xs[e0 + half], r), w[i + half]);
    const float c = cs[i], sv = sn[i];
    const float v0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sv));
    const float v1 = __fadd_rn(__fmul_rn(x0, sv), __fmul_rn(x1, c));
    if (head < a.nh) {
      store_q(a, (int64_t)t * a.nh * a.hd + e0, v0, v1, half);
    } else if (write_kv) {
      const int ke = (head - a.nh) * a.hd + i;
      const int64_t o0 = (int64_t)p * kw + ke;
      a.kreg[o0] = v0;
      a.kreg[o0 + half] = v1;
      const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
      a.shadow[0][o0] = h0;
      a.shadow[0][o0 + half] = h1;
      a.shadow[1][o0] = __float2half_rn(__fsub_rn(v0, __half2float(h0)));
      a.shadow[1][o0 + half] = __float2half_rn(__fsub_rn(v1, __half2float(h1)));
    }
  }
}

// ---------------------------------------------------------------- one-row GEMV
// y[n] = sum_b dw[n][b] * dx[b] * dot_b.  A warp owns R output rows; lane l
// reads bytes 16 l .. 16 l + 15 of each 512-byte chunk of a row's codes (half
// of a Q8_0 block, coalesced across the warp); dp4a gives the integer partial
// and the lane pair (l, l ^ 1) adds up the block's exact int32 dot, which the
// even lane scales by dw * dx.  Every load of a round (U chunks of all R
// rows, U = 4 for R = 1 and 2 above) is issued before the first dp4a: the
// kernel is bound by HBM, and the bytes in flight per warp (R * U * 512) set
// how close it gets.
//
// Fused one-row epilogues (grid-wide, wait-free):
//  - swiglu: the rows are gate/up interleaved in groups of 32, so CTA j (8
//    warps x 8 rows) holds the gate and up sums of outputs 32 j .. 32 j + 31;
//    it quantizes silu(g) * u of them (Q8_0) into q8/s8 and writes no y;
//  - norm_w: after its rows are written each CTA takes a ticket; the CTA that
//    draws the last one RMS-normalizes y[0:N] and quantizes it (Q8_0) into
//    q8/s8, with the row kernel's arithmetic, and returns the ticket to zero.
constexpr int kGemvWarps = 8;

__device__ __forceinline__ float silu_mul_row(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// The dot products of R rows (rows[r] < 0: none) with the activation row:
// after the call every lane holds the full sum of each row in acc[r].
template <int R>
__device__ __forceinline__ void gemv_dot(const GemvArgs& a, const int64_t (&rows)[R], float (&acc)[R]) {
  constexpr int U = R >= 2 ? 2 : 4;  // 512-byte chunks per round
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;
  for (int64_t c = 0; c < a.kpad; c += 512 * U) {
    int4 w[U][R];
    float dw[U][R];
    int4 x[U];
    float dx[U];
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int64_t k = c + 512 * h + 16 * lane;
      const bool in = k < a.kpad;
      const int b = (int)(k >> 5);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int64_t n = rows[r];
        const bool ok = in && n >= 0;
        w[h][r] = ok ? __ldg(reinterpret_cast<const int4*>(a.wq + n * a.kpad + k))
                     : make_int4(0, 0, 0, 0);
        dw[h][r] = ok ? __ldg(a.ws + n * a.nb + b) : 0.f;
      }
    }
    // static weights: their first round is in flight before the wait for the
    // kernel that wrote the activation row
    if (c == 0 && a.w_static) pdl_wait();
#pragma unroll
    for (int h = 0; h < U; ++h) {
      const int64_t k = c + 512 * h + 16 * lane;
      const bool in = k < a.kpad;
      const int b = (int)(k >> 5);
      x[h] = in ? *reinterpret_cast<const int4*>(a.xq + k) : make_int4(0, 0, 0, 0);
      dx[h] = in ? a.xs[b] : 0.f;
    }
#pragma unroll
    for (int h = 0; h < U; ++h)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int isum = __dp4a(w[h][r].x, x[h].x, 0);
        isum = __dp4a(w[h][r].y, x[h].y, isum);
        isum = __dp4a(w[h][r].z, x[h].z, isum);
        isum = __dp4a(w[h][r].w, x[h].w, isum);
        isum += __shfl_xor_sync(0xffffffffu, isum, 1);
        if (!(lane & 1)) acc[r] = fmaf((float)isum, __fmul_rn(dw[h][r], dx[h]), acc[r]);
      }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
}

template <int R>
__global__ void __launch_bounds__(32 * kGemvWarps, R >= 4 ? 2 : (R == 2 ? 4 : 3)) gemv_kernel(const GemvArgs a) {
  __shared__ float part[kGemvWarps][8];
  __shared__ unsigned s_last;
  pdl_trigger();
  if (!a.w_static) pdl_wait();  // else inside gemv_dot, after the first weight loads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n0 = ((int64_t)blockIdx.x * kGemvWarps + warp) * R;
  float acc[R];
  int64_t rows[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rows[r] = n0 + r < a.N ? n0 + r : -1;
  gemv_dot<R>(a, rows, acc);
  float v = acc[0];  // lane r < R: the sum of row n0 + r
#pragma unroll
  for (int r = 1; r < R; ++r)
    if (lane == r) v = acc[r];
  const int64_t n = n0 + lane;
  if (a.swiglu) {
    // part[w][r] = row 8 w + r of the CTA: gate rows in warps 0-3, up in 4-7
    if (lane < R) part[warp][lane] = v;
    __syncthreads();
    if (warp == 0) {
      const float gsum = part[lane >> 3][lane & 7];
      const float usum = part[4 + (lane >> 3)][lane & 7];
      const float sv = silu_mul_row(gsum, usum);
      const float amax = warp_max(fabsf(sv));
      const float d = __fdiv_rn(amax, 127.0f);
      a.q8[(int64_t)blockIdx.x * 32 + lane] = (int8_t)q8_code(sv, q8_inv(d));
      if (lane == 0) a.s8[blockIdx.x] = __half2float(__float2half_rn(d));
    }
    return;
  }
  if (lane < R && n < a.N && status_clear(a.status)) a.y[n] = a.resid ? __fadd_rn(a.resid[n], v) : v;
  if (a.norm_w) {
    __threadfence();  // this CTA's rows of y, device-wide, before its ticket
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    RowQuantArgs rq;
    rq.h = a.y;
    rq.norm_w = a.norm_w;
    rq.eps = a.eps;
    rq.rows = 1;
    rq.n = a.N;
    rq.q8 = a.q8;
    rq.s8 = a.s8;
    row_quant4_row<true, 4, true>(rq, 0);
    if (threadIdx.x == 0) *a.ticket = 0u;
  }
}

// The one-row QKV GEMV with the RoPE/store of its token in the same kernel.
// A warp's four rows are two neighbouring dimension pairs (i, i + 1 and their
// partners i + hd/2, i + 1 + hd/2) of one Q or K head, or four V dimensions,
// so the rotation needs only the warp's own sums.  The raw sums still go to y;
// bias, rotation, the region and plane writes are rope_store_kernel's
// arithmetic element by element.
__global__ void __launch_bounds__(32 * kGemvWarps, 2) gemv_rope_kernel(const GemvArgs a,
                                                                      const RopeStoreArgs ra) {
  pdl_trigger();
  if (!a.w_static) pdl_wait();  // else inside gemv_dot, after the first weight loads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hd = ra.hd, half = hd >> 1;
  const int64_t unit = (int64_t)blockIdx.x * kGemvWarps + warp;
  const int64_t urope = (int64_t)(ra.nh + ra.nkv) * half / 2;  // units of Q and K heads
  const int64_t units = a.N / 4;
  const bool live = unit < units, rope = unit < urope;
  int hh = 0, i0 = 0;
  int64_t rows[4];
  if (rope) {
    hh = (int)(2 * unit / half);
    i0 = (int)(2 * unit % half);
    const int64_t base = (int64_t)hh * hd + i0;
    rows[0] = base;
    rows[1] = base + 1;
    rows[2] = base + half;
    rows[3] = base + half + 1;
  } else {
    const int64_t base = (int64_t)(ra.nh + ra.nkv) * hd + 4 * (unit - urope);
#pragma unroll
    for (int r = 0; r < 4; ++r) rows[r] = live ? base + r : -1;
  }
  float acc[4];
  gemv_dot<4>(a, rows, acc);
  const int r4 = lane & 3;
  const float v = r4 == 0 ? acc[0] : (r4 == 1 ? acc[1] : (r4 == 2 ? acc[2] : acc[3]));
  const int64_t row = r4 == 0 ? rows[0] : (r4 == 1 ? rows[1] : (r4 == 2 ? rows[2] : rows[3]));
  float x = v;
  if (live && ra.bias) x = __fadd_rn(x, ra.bias[row]);
  const float xp = __shfl_xor_sync(0xffffffffu, x, 2);  // the pair partner (lanes 0<->2, 1<->3)
  if (!live || lane >= 4) return;
  a.y[row] = v;
  const int p_in = ra.pos[0];
  const bool write_kv = status_clear(ra.status) && p_in >= 0 && p_in < ra.n_ctx;
  const int p = (p_in >= 0 && p_in < ra.n_ctx) ? p_in : 0;
  const int64_t kw = (int64_t)ra.nkv * hd;
  if (rope) {
    const int i = i0 + (lane & 1);
    const float c = ra.cos_t[(int64_t)p * half + i], sn = ra.sin_t[(int64_t)p * half + i];
    const bool first = lane < 2;
    const float x0 = first ? x : xp, x1 = first ? xp : x;
    const float val = first ? __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn))
                            : __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
    const int e = first ? i : i + half;  // dimension within the head
    const __half hi = __float2half_rn(val);
    const __half lo = __float2half_rn(__fsub_rn(val, __half2float(hi)));
    if (hh < ra.nh) {
      const int64_t o = (int64_t)hh * hd + e;
      ra.q_out[o] = val;
      if (ra.q_planes[0]) {
        ra.q_planes[0][o] = hi;
        ra.q_planes[1][o] = lo;
      }
    } else if (write_kv) {
      const int64_t o0 = (int64_t)p * kw + (int64_t)(hh - ra.nh) * hd + e;
      ra.kreg[o0] = val;
      ra.shadow[0][o0] = hi;
      ra.shadow[1][o0] = lo;
    }
  } else if (write_kv) {
    const int64_t e = row - (int64_t)(ra.nh + ra.nkv) * hd;
    const int64_t o0 = (int64_t)p * kw + e;
    const __half hi = __float2half_rn(x);
    const __half lo = __float2half_rn(__fsub_rn(x, __half2float(hi)));
    ra.vreg[o0] = x;
    ra.shadow[2][o0] = hi;
    ra.shadow[3][o0] = lo;
    ra.vt[0][e * ra.vt_ld + p] = hi;
    ra.vt[1][e * ra.vt_ld + p] = lo;
  }
}

// ---------------------------------------------------------------- load-time kernels
__global__ void quantize_rows_kernel(const float* __restrict__ x, int64_t rows, int64_t n,
                                     int8_t* q, uint16_t* dbits) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = (n + 31) / 32;
  const int64_t total = rows * nb;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < total;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t r = w / nb, b = w % nb;
    const int64_t k = b * 32 + lane;
    const float v = k < n ? x[r * n + k] : 0.f;
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    q[r * nb * 32 + k] = (int8_t)q8_code(v, q8_inv(d));
    if (lane == 0) dbits[r * nb + b] = __half_as_ushort(__float2half_rn(d));
  }
}

__global__ void unpack_q8_0_kernel(const uint8_t* __restrict__ blocks, int64_t rows, int64_t n,
                                   int8_t* q, uint16_t* dbits) {
  const int64_t nb = (n + 31) / 32;
  const int64_t total = rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, b = i % nb;
    const uint8_t* p = blocks + 34 * i;
    dbits[i] = (uint16_t)(p[0] | (p[1] << 8));
    for (int k = 0; k < 32; ++k) q[(r * nb + b) * 32 + k] = (b * 32 + k < n) ? (int8_t)p[2 + k] : 0;
  }
}

__global__ void repack_gemm_kernel(const RepackArgs a) {
  const int64_t kpad = (int64_t)a.nb * 32;
  const int64_t total = a.rows * kpad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kpad, k = i % kpad;
    const int64_t dr = a.interleave ? ((r / kSwiGluGroup) * 2 * kSwiGluGroup +
                                       a.which * kSwiGluGroup + (r % kSwiGluGroup))
                                    : (a.dst_row0 + r);
    a.dst_codes[dr * kpad + k] = __float2half_rn((float)a.q[i]);
    if ((k & 31) == 0) {
      const int b = (int)(k / 32);
      a.dst_scales[(int64_t)b * a.dst_rows_pad + dr] =
          __half2float(__ushort_as_half(a.dbits[r * a.nb + b]));
    }
  }
}

// One-row (GEMV) layout -> tensor-core layout: int8 codes [rows][kpad] and f32
// scales [rows][nb] -> fp16 codes [rows][kpad] and block-major scales
// [nb][rows_pad] (the lm_head when several rows need logits).
__global__ void gemv_to_gemm_kernel(const int8_t* __restrict__ q, const float* __restrict__ s,
                                    int64_t rows, int nb, __half* codes, float* scales,
                                    int64_t rows_pad) {
  const int64_t kpad = (int64_t)nb * 32;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * kpad;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kpad, k = i % kpad;
    codes[i] = __float2half_rn((float)q[i]);
    if ((k & 31) == 0) scales[(k / 32) * rows_pad + r] = s[r * nb + k / 32];
  }
}

// dst = src when the call's status is clean (a rejected call writes no logit).
__global__ void copy_if_ok_kernel(const float* __restrict__ src, float* dst, int64_t n,
                                  const int* status) {
  pdl_trigger();
  pdl_wait();
  if (!status_clear(status)) return;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// interleave: source row r goes to row (r / 32) * 64 + which * 32 + r % 32
// (gate and up rows of the same 32 outputs side by side), else to row r.
__global__ void repack_gemv_kernel(const int8_t* __restrict__ q, const uint16_t* __restrict__ dbits,
                                   int64_t rows, int nb, int8_t* dst_q, float* dst_s, int interleave,
                                   int which) {
  const int64_t kpad = (int64_t)nb * 32;
  const int64_t total = rows * kpad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kpad, k = i % kpad;
    const int64_t dr = interleave ? (r / kSwiGluGroup) * 2 * kSwiGluGroup + which * kSwiGluGroup +
                                        r % kSwiGluGroup
                                  : r;
    dst_q[dr * kpad + k] = q[i];
    if ((k & 31) == 0) dst_s[dr * nb + k / 32] = __half2float(__ushort_as_half(dbits[i / 32]));
  }
}

__global__ void plane_to_q8_kernel(const __half* __restrict__ codes, const float* __restrict__ scales,
                                   int64_t rows, int64_t rows_pad, int nb, int8_t* q,
                                   uint16_t* dbits) {
  const int64_t kpad = (int64_t)nb * 32;
  const int64_t total = rows * kpad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kpad, k = i % kpad;
    q[i] = (int8_t)__half2float(codes[i]);
    if ((k & 31) == 0)
      dbits[r * nb + k / 32] = __half_as_ushort(__float2half_rn(scales[(k / 32) * rows_pad + r]));
  }
}

__global__ void sum_splits_kernel(const float* __restrict__ p, int nsplit, int64_t stride,
                                  int64_t count, float* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    float o = p[i];
    for (int s = 1; s < nsplit; ++s) o = __fadd_rn(o, p[s * stride + i]);
    out[i] = o;
  }
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  if (g > 152 * 32) g = 152 * 32;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t row_quant_launch(const RowQuantArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  return a.q8 ? row_quant_dispatch<true>(a, st) : row_quant_dispatch<false>(a, st);
}

cudaError_t embed_launch(const int8_t* q, const float* s, int64_t kpad, int nb, const int32_t* ids,
                         int nt, int64_t H, int n_vocab, float* h, cudaStream_t st) {
  return launch_pdl(embed_kernel, nt, 128, 0, st, q, s, kpad, nb, ids, H, h, n_vocab);
}

cudaError_t validate_launch(const int32_t* ids, const int32_t* pos, int nt, int n_vocab, int n_ctx,
                            uint32_t* seen, int* status, cudaStream_t st) {
  return launch_pdl(validate_kernel, 1, 1024, 0, st, ids, pos, nt, n_vocab, n_ctx, seen, status);
}

cudaError_t rope_store_launch(const RopeStoreArgs& a, cudaStream_t st) {
  if (a.nt <= 0) return cudaSuccess;
  if (a.q_norm || a.k_norm) {
    const int nheads = a.nh + a.nkv;
    if (!a.q_norm || !a.k_norm || nheads > kMaxQkHeads) return cudaErrorInvalidValue;
    const size_t smem = (size_t)nheads * a.hd * sizeof(float);
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    // up to one thread per element of the token's Q|K|V sums: the loads go
    // out in few rounds and every head's norm gets its own warp
    const int W = (a.nh + 2 * a.nkv) * a.hd;
    const int threads = std::min(1024, std::max(128, (W + 31) / 32 * 32));
    return launch_pdl(rope_store_qknorm_kernel, a.nt, threads, smem, st, a);
  }
  // one thread per two (Q/K pair, V element)s of the token where that fits a
  // CTA: every thread's loads go out in one round instead of several
  const int items = (a.nh + a.nkv) * (a.hd / 4) + a.nkv * a.hd / 2;
  const int threads = std::min(1024, std::max(128, (items + 31) / 32 * 32));
  return launch_pdl(rope_store_kernel, a.nt, threads, 0, st, a);
}

cudaError_t gemv_launch(const GemvArgs& a, cudaStream_t st) {
  if (a.swiglu) {
    // one CTA per 32 outputs: 64 interleaved gate/up rows, 8 per warp
    if (a.N % 64 != 0 || !a.q8 || !a.s8) return cudaErrorInvalidValue;
    return launch_pdl(gemv_kernel<8>, (unsigned)(a.N / 64), 32 * kGemvWarps, 0, st, a);
  }
  if (a.norm_w && (!a.ticket || !gemv_norm_fusable(a.N, a.y, a.norm_w, a.q8)))
    return cudaErrorInvalidValue;
  // the most rows per warp that still gives every SM two CTAs
  const int64_t per_cta[4] = {8 * kGemvWarps, 4 * kGemvWarps, 2 * kGemvWarps, kGemvWarps};
  int pick = 3;
  for (int i = 0; i < 4; ++i)
    if ((a.N + per_cta[i] - 1) / per_cta[i] >= 2 * a.num_sms) {
      pick = i;
      break;
    }
  const unsigned grid = (unsigned)((a.N + per_cta[pick] - 1) / per_cta[pick]);
  switch (pick) {
    case 0: return launch_pdl(gemv_kernel<8>, grid, 32 * kGemvWarps, 0, st, a);
    case 1: return launch_pdl(gemv_kernel<4>, grid, 32 * kGemvWarps, 0, st, a);
    case 2: return launch_pdl(gemv_kernel<2>, grid, 32 * kGemvWarps, 0, st, a);
    default: return launch_pdl(gemv_kernel<1>, grid, 32 * kGemvWarps, 0, st, a);
  }
}

cudaError_t gemv_rope_launch(const GemvArgs& a, const RopeStoreArgs& r, cudaStream_t st) {
  if (r.nt != 1 || r.q_norm || r.nsplit != 1 || (r.hd != 64 && r.hd != 128) ||
      a.N != (int64_t)(r.nh + 2 * r.nkv) * r.hd)
    return cudaErrorInvalidValue;
  const int64_t units = a.N / 4;
  return launch_pdl(gemv_rope_kernel, (unsigned)((units + kGemvWarps - 1) / kGemvWarps),
                    32 * kGemvWarps, 0, st, a, r);
}

bool gemv_norm_fusable(int64_t N, const float* y, const float* norm_w, const int8_t* q8) {
  return N % 32 == 0 && N / 4 <= 4 * kRowThreads && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(norm_w) % 16 == 0 && reinterpret_cast<uintptr_t>(q8) % 4 == 0;
}

cudaError_t gemv_to_gemm_launch(const int8_t* q, const float* sc, int64_t rows, int nb,
                                __half* codes, float* scales, int64_t rows_pad, cudaStream_t st) {
  gemv_to_gemm_kernel<<<grid_for(rows * nb * 32, 256), 256, 0, st>>>(q, sc, rows, nb, codes, scales,
                                                                    rows_pad);
  return cudaGetLastError();
}

cudaError_t copy_if_ok_launch(const float* src, float* dst, int64_t n, const int* status,
                              cudaStream_t st) {
  return launch_pdl(copy_if_ok_kernel, (unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0,
                    st, src, dst, n, status);
}

cudaError_t quantize_rows_launch(const float* x, int64_t rows, int64_t n, int8_t* q,
                                 uint16_t* dbits, cudaStream_t st) {
  const int64_t nb = (n + 31) / 32;
  quantize_rows_kernel<<<grid_for(rows * nb * 32, 256), 256, 0, st>>>(x, rows, n, q, dbits);
  return cudaGetLastError();
}

cudaError_t unpack_q8_0_launch(const uint8_t* blocks, int64_t rows, int64_t n, int8_t* q,
                               uint16_t* dbits, cudaStream_t st) {
  const int64_t nb = (n + 31) / 32;
  unpack_q8_0_kernel<<<grid_for(rows * nb, 256), 256, 0, st>>>(blocks, rows, n, q, dbits);
  return cudaGetLastError();
}

cudaError_t repack_gemm_launch(const RepackArgs& a, cudaStream_t st) {
  repack_gemm_kernel<<<grid_for(a.rows * a.nb * 32, 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t repack_gemv_launch(const int8_t* q, const uint16_t* dbits, int64_t rows, int nb,
                               int8_t* dst_q, float* dst_s, int interleave, int which,
                               cudaStream_t st) {
  repack_gemv_kernel<<<grid_for(rows * nb * 32, 256), 256, 0, st>>>(q, dbits, rows, nb, dst_q, dst_s,
                                                                    interleave, which);
  return cudaGetLastError();
}

cudaError_t gemm_plane_to_q8_launch(const __half* codes, const float* scales, int64_t rows,
                                    int64_t rows_pad, int nb, int8_t* q, uint16_t* dbits,
                                    cudaStream_t st) {
  plane_to_q8_kernel<<<grid_for(rows * nb * 32, 256), 256, 0, st>>>(codes, scales, rows, rows_pad,
                                                                    nb, q, dbits);
  return cudaGetLastError();
}

cudaError_t sum_splits_launch(const float* p, int nsplit, int64_t stride, int64_t count, float* out,
                              cudaStream_t st) {
  sum_splits_kernel<<<grid_for(count, 256), 256, 0, st>>>(p, nsplit, stride, count, out);
  return cudaGetLastError();
}

}  // namespace minfer

// k_attn.cu -- causal GQA attention over the persistent KV regions.
//
// What it computes ("09 · Prefill: the first forward", section 2.2: token t
// attends to positions 0..=pos[t]; "05 · Graph build — the IR and the
// builder", section 2.5: GQA, scale 1/sqrt(head_dim)):
//     o[t, h] = sum_{j <= pos[t]} softmax_j(q[t,h] . K[j, g] / sqrt(hd)) V[j, g],
//     g = h / (n_head / n_head_kv)
//
// Design.  One CTA per (16 query rows, KV head g, key split): warp w serves
// query head g * G + w, so the G heads that share a KV head share every K/V
// tile in shared memory.  K/V tiles come from fp16 hi/lo shadow planes of the
// f32 regions (written next to the regions by the RoPE/store kernel), staged
// with double-buffered cp.async.  Scores and P.V run on the tensor cores
// (mma.sync m16n8k16, fp16 operands, f32 accumulate) with every f32 operand
// split as hi + lo and the three significant cross products accumulated
// (about 22 significant bits, the precision the Q8_0 quantization of the
// output needs).  The softmax is online: running row max and sum in f32,
// reduced across the four lanes of a row with warp shuffles.
//
// Short prompts have too few (rows, KV head) tiles to fill the GPU, so the
// key range is split (the split-KV scheme of the pages' CUDA backend): each
// split writes its unnormalized output and (max, sum) to scratch, and the
// combine kernel merges the splits, normalizes, and quantizes each 32-block
// of the output row to Q8_0 for the o-projection.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace minfer {

namespace {

constexpr int kMaxSplitsSmem = 64;  // key splits one combine CTA can merge
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
};

template <int HD>
__global__ void __launch_bounds__(256) attn_split_kernel(const AttnArgs a) {
  using T = Tile<HD>;
  extern __shared__ __align__(16) __half smem_h[];
  __shared__ int s_maxp;
  pdl_trigger();
  pdl_wait();

  const int G = a.nh / a.nkv;
  const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest rows first
  const int g = blockIdx.y;
  const int split = blockIdx.z;
  const int rbase = a.r0 + tile * kTileQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = g * G + warp;
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
  if (threadIdx.x < kTileQ) atomicMax(&s_maxp, clamp_pos(rbase + threadIdx.x));
  __syncthreads();
  const int maxp = s_maxp;
  const int kbeg = split * a.ksplit;
  if (kbeg > maxp) return;  // uniform across the CTA
  const int kend = min(maxp + 1, kbeg + a.ksplit);
  const int ntile = (kend - kbeg + kTileKV - 1) / kTileKV;

  const int ra = rbase + qr, rb = rbase + qr + 8;
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
  load_tile(0, 0);

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
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const __half* kh = Kh + (nt * 8 + qr) * T::RS + kk * 16 + qc;
        const __half* kl = Kl + (nt * 8 + qr) * T::RS + kk * 16 + qc;
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
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int nd = 0; nd < HD / 8; nd += 2) {
        const uint32_t off =
            2u * (uint32_t)((ks * 16 + (mi & 1) * 8 + mr) * T::RS + nd * 8 + (mi >> 1) * 8);
        uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
        ldsm_x4_t(vh_base + off, h0, h1, h2, h3);
        ldsm_x4_t(vl_base + off, l0, l1, l2, l3);
        mma16816(o[nd], ph[ks], h0, h1);
        mma16816(o[nd], ph[ks], l0, l1);
        mma16816(o[nd], pl[ks], h0, h1);
        mma16816(o[nd + 1], ph[ks], h2, h3);
        mma16816(o[nd + 1], ph[ks], l2, l3);
        mma16816(o[nd + 1], pl[ks], h2, h3);
      }
    }
    __syncthreads();  // the next prefetch overwrites this stage's buffer
  }

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  // partial: unnormalized o, running max (log2 units) and sum per row
  const int nrows = a.r1 - a.r0;
  if (ra < a.r1) {
    const int64_t base = ((int64_t)split * nrows + (ra - a.r0)) * a.nh + h;
    float* dst = a.part_o + base * HD + qc;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][0], o[nd][1]);
    if ((lane & 3) == 0) *reinterpret_cast<float2*>(a.part_ml + base * 2) = make_float2(m_a, l_a);
  }
  if (rb < a.r1) {
    const int64_t base = ((int64_t)split * nrows + (rb - a.r0)) * a.nh + h;
    float* dst = a.part_o + base * HD + qc;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd)
      *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][2], o[nd][3]);
    if ((lane & 3) == 0) *reinterpret_cast<float2*>(a.part_ml + base * 2) = make_float2(m_b, l_b);
  }
}

// One CTA of 256 threads per query row: per-head split weights
// w_s = 2^(m_s - M) / L in shared memory, then every thread merges its
// elements over the splits, and each warp quantizes its 32-block.
constexpr int kCombThreads = 256;
constexpr int kMaxHeads = 64;

template <bool kGemvOut, int PER>
__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(const AttnArgs a, const AttnOut out) {
  __shared__ float s_w[kMaxHeads][kMaxSplitsSmem];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = a.r0 + (int)blockIdx.x;
  const int nrows = a.r1 - a.r0;
  int p = a.pos[r];
  p = p < 0 ? 0 : (p >= a.n_ctx ? a.n_ctx - 1 : p);
  const int nsplit = min(p / a.ksplit + 1, kMaxSplitsSmem);
  const int hd = a.hd;
  const int q = a.nh * hd;
  const int nb = q / 32;
  if (tid < a.nh) {
    const int h = tid;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s)
      M = fmaxf(M, a.part_ml[(((int64_t)s * nrows + (r - a.r0)) * a.nh + h) * 2]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const int64_t base = ((int64_t)s * nrows + (r - a.r0)) * a.nh + h;
      const float m = a.part_ml[base * 2];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      s_w[h][s] = w;
      L = fmaf(a.part_ml[base * 2 + 1], w, L);
    }
    const float inv = L > 0.f ? __fdiv_rn(1.0f, L) : 0.f;
    for (int s = 0; s < nsplit; ++s) s_w[h][s] = __fmul_rn(s_w[h][s], inv);
  }
  __syncthreads();
  float y[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) y[i] = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float* po = a.part_o + ((int64_t)s * nrows + (r - a.r0)) * q;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int k = tid + kCombThreads * i;
      if (k < q) y[i] = fmaf(po[k], s_w[k / hd][s], y[i]);
    }
  }
  const int64_t orow = r - out.row_base;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int k = tid + kCombThreads * i;
    const int b = 8 * i + warp;
    if (b >= nb) continue;  // warp-uniform
    if (out.f32) out.f32[(int64_t)r * q + k] = y[i];
    const float amax = warp_max(fabsf(y[i]));
    const float dd = __fdiv_rn(amax, 127.0f);
    const float code = q8_code(y[i], q8_inv(dd));
    const __half d16 = __float2half_rn(dd);
    if (kGemvOut) {
      out.q8[orow * (int64_t)nb * 32 + k] = (int8_t)code;
      if (lane == 0) out.s8[orow * nb + b] = __half2float(d16);
    } else {
      out.q16[orow * out.ldq + k] = __float2half_rn(code);
      if (lane == 0) out.s16[(int64_t)b * out.ldqs + orow] = __half2float(d16);
    }
  }
}

template <bool kGemvOut>
cudaError_t combine_dispatch(const AttnArgs& a, const AttnOut& out, int rows, cudaStream_t st) {
  const int per = (a.nh * a.hd + kCombThreads - 1) / kCombThreads;
  if (per <= 4) return launch_pdl(attn_combine_kernel<kGemvOut, 4>, rows, kCombThreads, 0, st, a, out);
  if (per <= 8) return launch_pdl(attn_combine_kernel<kGemvOut, 8>, rows, kCombThreads, 0, st, a, out);
  if (per <= 16) return launch_pdl(attn_combine_kernel<kGemvOut, 16>, rows, kCombThreads, 0, st, a, out);
  return cudaErrorInvalidValue;
}

// K/V rows of one layer -> fp16 hi/lo shadow planes (count f32 values each).
__global__ void kv_shadow_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                 int64_t count, __half* kh, __half* kl, __half* vh, __half* vl) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = k[i], y = v[i];
    const __half xh = __float2half_rn(x), yh = __float2half_rn(y);
    kh[i] = xh;
    kl[i] = __float2half_rn(__fsub_rn(x, __half2float(xh)));
    vh[i] = yh;
    vl[i] = __float2half_rn(__fsub_rn(y, __half2float(yh)));
  }
}

}  // namespace

int attention_splits(int rows, int nkv, int n_ctx, int num_sms, int* ksplit) {
  const int tiles = (rows + kTileQ - 1) / kTileQ;
  if (tiles * nkv >= num_sms) {
    *ksplit = (n_ctx + kTileKV - 1) / kTileKV * kTileKV;
    return 1;
  }
  // 128 keys per split, fewer (longer) splits for very long regions
  int ks = (n_ctx + kMaxSplitsSmem - 1) / kMaxSplitsSmem;
  ks = ks < 128 ? 128 : (ks + kTileKV - 1) / kTileKV * kTileKV;
  *ksplit = ks;
  return (n_ctx + ks - 1) / ks;
}

cudaError_t attention_launch(const AttnArgs& a, const AttnOut& out, cudaStream_t st) {
  const int rows = a.r1 - a.r0;
  if (rows <= 0) return cudaSuccess;
  const int G = a.nh / a.nkv;
  if (a.nh % a.nkv != 0 || G > 8 || a.ksplit <= 0 || a.ksplit % kTileKV != 0)
    return cudaErrorInvalidValue;
  const int nsplit = (a.n_ctx + a.ksplit - 1) / a.ksplit;
  const dim3 grid((rows + kTileQ - 1) / kTileQ, a.nkv, nsplit);
  if (a.hd == 64) {
    static bool set = false;
    if (!set) {
      cudaError_t e = cudaFuncSetAttribute(
          attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tile<64>::BYTES);
      if (e != cudaSuccess) return e;
      set = true;
    }
    cudaError_t e = launch_pdl(attn_split_kernel<64>, grid, 32 * G, Tile<64>::BYTES, st, a);
    if (e != cudaSuccess) return e;
  } else if (a.hd == 128) {
    static bool set = false;
    if (!set) {
      cudaError_t e = cudaFuncSetAttribute(
          attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tile<128>::BYTES);
      if (e != cudaSuccess) return e;
      set = true;
    }
    cudaError_t e = launch_pdl(attn_split_kernel<128>, grid, 32 * G, Tile<128>::BYTES, st, a);
    if (e != cudaSuccess) return e;
  } else {
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.nh > kMaxHeads || (a.n_ctx + a.ksplit - 1) / a.ksplit > kMaxSplitsSmem)
    return cudaErrorInvalidValue;
  return out.q8 ? combine_dispatch<true>(a, out, rows, st) : combine_dispatch<false>(a, out, rows, st);
}

cudaError_t kv_shadow_launch(const float* k, const float* v, int64_t count, __half* const* planes,
                             cudaStream_t st) {
  int64_t g = (count + 255) / 256;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  kv_shadow_kernel<<<(unsigned)g, 256, 0, st>>>(k, v, count, planes[0], planes[1], planes[2],
                                                planes[3]);
  return cudaGetLastError();
}

}  // namespace minfer

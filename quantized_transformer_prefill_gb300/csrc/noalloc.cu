// noalloc.cu -- the Q8_0 tensor-core GEMM behind an entry point that
// allocates no device memory.
//
// Some callers cannot call cudaMalloc: a serving process that hands nearly all
// of HBM to its own allocator at start-up (a later cudaMalloc fails or steals
// from that pool), and code that must not stall the device (cudaFree
// synchronizes the whole device).  minfer_op_gemm needs scratch for the
// tensor-core operand planes and the split-K partial sums; this variant keeps
// all of it in one file-scope __device__ array of fixed size instead.
//
// The array is part of the library image: every GPU that loads the library
// holds it until the process exits.  All calls share it and find the previous
// call's contents there; the regions that must start at zero (scale padding,
// the status word) are cleared on every call.  Two calls whose work overlaps
// on the GPU race on the array.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "../../include/minfer.h"
#include "kernels.h"

namespace minfer {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace minfer

using namespace minfer;

extern "C" int minfer_op_gemm_noalloc(const int8_t* d_xq, const uint16_t* d_xd, int64_t M,
                                      const int8_t* d_wq, const uint16_t* d_wd, int64_t N,
                                      int64_t K, float* d_y) {
  if (!d_xq || !d_xd || !d_wq || !d_wd || !d_y || M <= 0 || N <= 0 || K <= 0)
    return MINFER_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MINFER_ERR_CUDA;
  // set-up, once per device, with that device current: the host-side name of
  // the array is not a device address; ask the runtime for the real one
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MINFER_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  int num_sms = 148;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MINFER_ERR_CUDA;

  const int nb = (int)((K + 31) / 32);
  const int64_t kpad = (int64_t)nb * 32;
  const int64_t Mp = (M + 127) / 128 * 128, Np = (N + 127) / 128 * 128;
  GemmPlan plan = gemm_plan(M, N, nb, num_sms, true);
  plan.splits = std::min(plan.splits, 8);
  const int stages = (nb + 1) / 2;
  int splits = std::max(1, std::min(plan.splits, stages));
  const int sps = (stages + splits - 1) / splits;
  splits = (stages + sps - 1) / sps;

  // carve the array: A codes, A scales, B codes, B scales, partials, status
  const size_t sz_ac = align256((size_t)M * kpad * 2), sz_as = align256((size_t)nb * Mp * 4);
  const size_t sz_bc = align256((size_t)N * kpad * 2), sz_bs = align256((size_t)nb * Np * 4);
  const size_t sz_p = align256((size_t)splits * M * N * 4), sz_err = 256;
  if (sz_ac + sz_as + sz_bc + sz_bs + sz_p + sz_err > kNoAllocScratchBytes) return MINFER_ERR_TOO_LARGE;
  unsigned char* p = static_cast<unsigned char*>(base);
  __half* a_codes = reinterpret_cast<__half*>(p);
  float* a_scales = reinterpret_cast<float*>(p + sz_ac);
  __half* b_codes = reinterpret_cast<__half*>(p + sz_ac + sz_as);
  float* b_scales = reinterpret_cast<float*>(p + sz_ac + sz_as + sz_bc);
  float* part = reinterpret_cast<float*>(p + sz_ac + sz_as + sz_bc + sz_bs);
  int* err = reinterpret_cast<int*>(p + sz_ac + sz_as + sz_bc + sz_bs + sz_p);

  cudaError_t e = cudaMemsetAsync(a_scales, 0, sz_as, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(b_scales, 0, sz_bs, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), 0);
  RepackArgs ra;
  ra.q = d_xq;
  ra.dbits = d_xd;
  ra.rows = M;
  ra.nb = nb;
  ra.dst_codes = a_codes;
  ra.dst_scales = a_scales;
  ra.dst_rows_pad = Mp;
  if (e == cudaSuccess) e = repack_gemm_launch(ra, 0);
  RepackArgs rb = ra;
  rb.q = d_wq;
  rb.dbits = d_wd;
  rb.rows = N;
  rb.dst_codes = b_codes;
  rb.dst_scales = b_scales;
  rb.dst_rows_pad = Np;
  if (e == cudaSuccess) e = repack_gemm_launch(rb, 0);
  if (e != cudaSuccess) return MINFER_ERR_CUDA;

  GemmLaunch g;
  g.A.codes = a_codes;
  g.A.scales = a_scales;
  g.A.rows = M;
  g.A.rows_pad = Mp;
  g.A.nb = nb;
  g.B.codes = b_codes;
  g.B.scales = b_scales;
  g.B.rows = N;
  g.B.rows_pad = Np;
  g.B.nb = nb;
  g.M = M;
  g.N = N;
  g.epi = kEpiF32;
  g.plan = plan;
  g.out = part;
  g.ldo = N;
  g.split_stride = M * N;
  g.err = err;
  GemmMaps maps;
  if (gemm_make_maps(g.A, g.B, g.plan.bn, &maps)) return MINFER_ERR_CUDA;
  e = gemm_launch(g, maps, num_sms, 0);
  if (e == cudaSuccess) e = sum_splits_launch(part, splits, M * N, M * N, d_y, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return MINFER_ERR_CUDA;
  int herr = 0;
  if (cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MINFER_ERR_CUDA;
  return herr ? MINFER_ERR_DEVICE : MINFER_OK;
}

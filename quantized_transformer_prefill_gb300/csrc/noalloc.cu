// noalloc.cu -- the Q8_0 tensor-core GEMM behind an entry point that
// allocates no device memory.
//
// Some callers cannot call cudaMalloc: a serving process that hands nearly all
// of HBM to its own memory pool at start-up (a later cudaMalloc fails, or takes
// memory the pool counts on), and code that must not stall the whole device
// (cudaFree synchronizes every stream of the device).  minfer_op_gemm needs
// scratch for the tensor-core operand planes and the split-K partial sums;
// this variant keeps all of it in one file-scope __device__ array of fixed
// size instead, and runs on a non-blocking stream of its own that it waits
// for alone.
//
// The array is part of the library image: every GPU that loads the library
// holds it until the process exits.  All calls share it and find the previous
// call's contents there; the regions that must start at zero (scale padding,
// the status word) are cleared on every call.  Two calls whose work overlapped
// on the GPU would race on the array, so each call holds a process-wide lock
// until its work has finished.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <mutex>

#include "../../include/minfer.h"
#include "kernels.h"

namespace minfer {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up, done once with that device current: the array's device
// address (the host-side name of a __device__ array is only a stand-in, never
// a device address) and the stream the calls run on.
struct DeviceSetup {
  void* scratch = nullptr;
  cudaStream_t stream = nullptr;
  int num_sms = 0;
};
std::mutex g_mu;  // guards g_setup and serializes the calls (the array is shared)
DeviceSetup g_setup[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// a + b into *acc unless the total would pass the array's size
bool add_fits(size_t* acc, size_t b) {
  if (b > kNoAllocScratchBytes || *acc > kNoAllocScratchBytes - b) return false;
  *acc += b;
  return true;
}

}  // namespace
}  // namespace minfer

using namespace minfer;

extern "C" int minfer_op_gemm_noalloc(const int8_t* d_xq, const uint16_t* d_xd, int64_t M,
                                      const int8_t* d_wq, const uint16_t* d_wd, int64_t N,
                                      int64_t K, float* d_y) {
  if (!d_xq || !d_xd || !d_wq || !d_wd || !d_y || M <= 0 || N <= 0 || K <= 0)
    return MINFER_ERR_ARG;
  // the kernels index rows and columns with 32-bit integers
  if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return MINFER_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MINFER_ERR_CUDA;

  std::lock_guard<std::mutex> lk(g_mu);
  DeviceSetup& su = g_setup[dev];
  if (!su.scratch) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MINFER_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MINFER_ERR_CUDA;
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return MINFER_ERR_CUDA;
    su.scratch = p;
    su.stream = st;
    su.num_sms = sms;
  }
  const cudaStream_t st = su.stream;

  const int nb = (int)((K + 31) / 32);
  const int64_t kpad = (int64_t)nb * 32;
  const int64_t Mp = (M + 127) / 128 * 128, Np = (N + 127) / 128 * 128;
  GemmPlan plan = gemm_plan(M, N, nb, su.num_sms, true);
  plan.splits = std::min(plan.splits, 8);
  const int stages = (nb + 1) / 2;
  int splits = std::max(1, std::min(plan.splits, stages));
  const int sps = (stages + splits - 1) / splits;
  splits = (stages + sps - 1) / sps;

  // carve the array: A codes, A scales, B codes, B scales, partials, status;
  // every term is checked against the array's size before it is added, so
  // no product or sum can wrap past the bound
  const double dM = (double)M, dN = (double)N, dk = (double)kpad;
  if (dM * dk * 2 > (double)kNoAllocScratchBytes || dN * dk * 2 > (double)kNoAllocScratchBytes ||
      (double)splits * dM * dN * 4 > (double)kNoAllocScratchBytes)
    return MINFER_ERR_TOO_LARGE;
  const size_t sz_ac = align256((size_t)M * kpad * 2), sz_as = align256((size_t)nb * Mp * 4);
  const size_t sz_bc = align256((size_t)N * kpad * 2), sz_bs = align256((size_t)nb * Np * 4);
  const size_t sz_p = align256((size_t)splits * M * N * 4), sz_err = 256;
  size_t total = 0;
  if (!add_fits(&total, sz_ac) || !add_fits(&total, sz_as) || !add_fits(&total, sz_bc) ||
      !add_fits(&total, sz_bs) || !add_fits(&total, sz_p) || !add_fits(&total, sz_err))
    return MINFER_ERR_TOO_LARGE;
  unsigned char* p = static_cast<unsigned char*>(su.scratch);
  __half* a_codes = reinterpret_cast<__half*>(p);
  float* a_scales = reinterpret_cast<float*>(p + sz_ac);
  __half* b_codes = reinterpret_cast<__half*>(p + sz_ac + sz_as);
  float* b_scales = reinterpret_cast<float*>(p + sz_ac + sz_as + sz_bc);
  float* part = reinterpret_cast<float*>(p + sz_ac + sz_as + sz_bc + sz_bs);
  int* err = reinterpret_cast<int*>(p + sz_ac + sz_as + sz_bc + sz_bs + sz_p);

  cudaError_t e = cudaMemsetAsync(a_scales, 0, sz_as, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(b_scales, 0, sz_bs, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), st);
  RepackArgs ra;
  ra.q = d_xq;
  ra.dbits = d_xd;
  ra.rows = M;
  ra.nb = nb;
  ra.dst_codes = a_codes;
  ra.dst_scales = a_scales;
  ra.dst_rows_pad = Mp;
  if (e == cudaSuccess) e = repack_gemm_launch(ra, st);
  RepackArgs rb = ra;
  rb.q = d_wq;
  rb.dbits = d_wd;
  rb.rows = N;
  rb.dst_codes = b_codes;
  rb.dst_scales = b_scales;
  rb.dst_rows_pad = Np;
  if (e == cudaSuccess) e = repack_gemm_launch(rb, st);
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
  e = gemm_launch(g, maps, su.num_sms, st);
  if (e == cudaSuccess) e = sum_splits_launch(part, splits, M * N, M * N, d_y, st);
  int herr = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&herr, err, sizeof(int), cudaMemcpyDeviceToHost, st);
  // wait for this call's own stream only
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return MINFER_ERR_CUDA;
  return herr ? MINFER_ERR_DEVICE : MINFER_OK;
}

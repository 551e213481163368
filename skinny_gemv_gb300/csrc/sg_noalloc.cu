// gemv_bf16_noalloc: the CUDA-core skinny GEMV for callers that must not allocate
// device memory.
//
// gemv_bf16 keeps its split-K partial sums and arrival counters in a workspace
// that the library allocates with cudaMalloc on the first call.  Some callers
// cannot let that happen: an engine whose device memory is owned by its own
// pool allocator (cudaMalloc would fail or fragment memory the pool expected to
// own), a plug-in running inside a host framework that forbids raw allocations,
// or code that must not pay cudaMalloc's implicit device synchronisation.  This
// entry point runs the same CUDA-core kernel with that scratch in a fixed
// file-scope __device__ array instead.  The array is part of the library's
// device image: every GPU that loads the library holds it until the process
// exits.  The call itself makes no cudaMalloc, cudaFree or other allocating call.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/skinny_gemm.h"
#include "sg_internal.h"

namespace sg {
namespace {

constexpr size_t kScratchPartialBytes = SG_NOALLOC_PARTIAL_BYTES;
constexpr size_t kScratchCounters = SG_NOALLOC_COUNTERS;
constexpr int kMaxDevices = 64;

// [fp32 partial sums | uint32 arrival counters]; zero at load.
static __device__ __align__(256) unsigned char g_scratch[kScratchPartialBytes + kScratchCounters * 4];

std::mutex g_setup_mutex;
void* g_scratch_dev[kMaxDevices] = {};  // device address of g_scratch, per device

// Per-device set-up, done by the first call on each device (with that device
// current): the host-side name g_scratch is only a stand-in, so the array's
// device address is looked up once and passed to the kernel.
int scratch_for_device(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_last_cuda_error(static_cast<int>(e));
      return SG_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return SG_OK;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace
}  // namespace sg

extern "C" int gemv_bf16_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc, sg_stream_t stream) {
  using namespace sg;
  // The same argument rules as gemv_bf16.
  if (M < 0 || N < 0 || K < 0 || M > 64 || N > INT32_MAX || K > INT32_MAX) return SG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SG_OK;
  if (!C || (K > 0 && (!A || !B))) return SG_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N) return SG_ERR_INVALID_ARG;
  if (misaligned(C) || (K > 0 && (misaligned(A) || misaligned(B)))) return SG_ERR_MISALIGNED;
  if ((lda & 7) || (ldb & 7) || (ldc & 7)) return SG_ERR_MISALIGNED;

  int dev = 0, sms = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(static_cast<int>(e));
    return SG_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices || major != 10 || minor != 3) return SG_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) {  // an empty sum: C := 0
    e = cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, s);
    if (e == cudaSuccess) return SG_OK;
    set_last_cuda_error(static_cast<int>(e));
    return SG_ERR_CUDA;
  }

  // Plan every 8-row block first, so a call that would not fit is rejected
  // before anything is launched.
  sg_plan_info plans[8];
  int nblocks = 0;
  for (int64_t m0 = 0; m0 < M; m0 += 8, ++nblocks) {
    const int64_t mb = std::min<int64_t>(8, M - m0);
    if (sg_plan(mb, N, K, sms, SG_PATH_CUDA_CORE, &plans[nblocks]) != SG_OK) return SG_ERR_INVALID_ARG;
    const sg_plan_info& p = plans[nblocks];
    if (p.split_k > 1) {
      const size_t partial_bytes = static_cast<size_t>(p.split_k) * mb * N * sizeof(float);
      if (partial_bytes > kScratchPartialBytes || static_cast<size_t>(p.tiles_m) > kScratchCounters)
        return SG_ERR_INVALID_ARG;  // beyond SG_NOALLOC_PARTIAL_BYTES / SG_NOALLOC_COUNTERS
    }
  }

  void* scratch = nullptr;
  int st = scratch_for_device(dev, &scratch);
  if (st != SG_OK) return st;
  float* partials = static_cast<float*>(scratch);
  uint32_t* counters = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(scratch) + kScratchPartialBytes);

  for (int b = 0; b < nblocks; ++b) {
    const int64_t m0 = static_cast<int64_t>(b) * 8;
    const int64_t mb = std::min<int64_t>(8, M - m0);
    const sg_plan_info& plan = plans[b];
    if (plan.split_k > 1) {
      // The array keeps the previous call's contents.  A kernel that runs to the
      // end leaves its counters at zero, but one that never finished (its launch
      // failed part-way, or its stream was torn down) would leave a count behind
      // that the next call's slices would miscount, so each call clears the
      // counters it uses instead of trusting the last call to have done so.
      e = cudaMemsetAsync(counters, 0, static_cast<size_t>(plan.tiles_m) * sizeof(uint32_t), s);
      if (e != cudaSuccess) {
        set_last_cuda_error(static_cast<int>(e));
        return SG_ERR_CUDA;
      }
    }
    CcParams p{};
    p.A = static_cast<const uint16_t*>(A) + m0 * lda;
    p.B = static_cast<const uint16_t*>(B);
    p.C = static_cast<uint16_t*>(C) + m0 * ldc;
    p.M = static_cast<int32_t>(mb);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.grid_rows = plan.tiles_m;
    p.split_k = plan.split_k;
    p.k_slice = plan.k_steps;
    p.partials = partials;
    p.counters = counters;
    p.prewait = plan.prefetch_steps;
    e = launch_cc_gemv(p, s);
    if (e != cudaSuccess) {
      set_last_cuda_error(static_cast<int>(e));
      return SG_ERR_CUDA;
    }
  }
  return SG_OK;
}

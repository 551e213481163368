// Roofline denominators measured on the card itself (spark-kernels, "how things
// are measured": a loop of tensor-core instructions on resident operands gives
// the usable peak, read at the clock the card actually runs; UwULLM kernel-dev,
// section 1: peak bandwidth and peak matmul rate are measured, never computed).
//
//   tc_peak_kernel     one CTA per SM issues back-to-back tcgen05.mma.kind::f16
//                      128 x 256 x 16 from shared-memory operands that stay
//                      resident, alternating two TMEM accumulators;
//   read_stream_kernel 16-byte non-caching loads over a buffer, folded into one
//                      word so the loads cannot be removed.
#include "sg_internal.h"
#include "sg_ptx.cuh"

namespace sg {
namespace {

constexpr int kPeakN = 256;
// More than half of an SM's shared memory, so exactly one CTA fits per SM
// (each CTA takes all 512 TMEM columns).
constexpr int kPeakSmem = 128 * 1024;
static_assert((kBM + kPeakN) * kBK * 2 + 1024 + 64 <= kPeakSmem, "operands fit");

__global__ void __launch_bounds__(128, 1)
    tc_peak_kernel(int64_t iters, unsigned long long* cycles, unsigned long long* ns, DeviceError* err,
                   uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tile = smem;
  uint8_t* b_tile = smem + kBM * kBK * 2;
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + (kBM + kPeakN) * kBK * 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  // Operands: bf16 values of magnitude < 1 from a per-element hash, so the
  // tensor cores see ordinary data (all-zero operands draw less power).
  for (int i = threadIdx.x; i < (kBM + kPeakN) * kBK; i += blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u + 0x9E3779B9u * (blockIdx.x + 1);
    h ^= h >> 15;
    const uint16_t bits = static_cast<uint16_t>(0x3C00u | (h & 0x7Fu) | ((h >> 8) & 1u) << 15);
    reinterpret_cast<uint16_t*>(smem)[i] = bits;
  }
  fence_proxy_async_smem();  // generic writes -> async-proxy (MMA) reads
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kPeakN);
    const uint32_t a_addr = smem_u32(a_tile), b_addr = smem_u32(b_tile);
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    for (int64_t i = 0; i < iters; ++i) {
      const uint32_t kk = static_cast<uint32_t>(i & 3) * 32u;
      tc_mma_bf16(tmem + static_cast<uint32_t>((i >> 2) & 1) * kPeakN, smem_desc_sw128(a_addr + kk),
                  smem_desc_sw128(b_addr + kk), idesc, i >= 8 ? 1u : 0u);
    }
    tc_commit(done);
    volatile uint32_t never = 0;
    const bool ok = mbar_wait(done, 0, timeout_ns, &never);
    const long long c1 = clock64();
    const uint64_t t1 = globaltimer_ns();
    if (!ok) record_error(err, kDevTimeoutTeardown, 0);
    cycles[blockIdx.x] = static_cast<unsigned long long>(c1 - c0);
    ns[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(512) read_stream_kernel(const uint4* __restrict__ src, int64_t nvec,
                                                          uint32_t* sink) {
  uint32_t acc = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4* p = src + i + u * stride;
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                   : "l"(p));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < nvec; i += stride) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(src + i));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  // Data-dependent store keeps every load live; almost never taken.
  if (acc == 0x9E3779B9u) sink[0] = acc;
}

}  // namespace

cudaError_t launch_tc_peak(int64_t iters, int grid, unsigned long long* cycles, unsigned long long* ns,
                           DeviceError* err, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(tc_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  tc_peak_kernel<<<grid, 128, kPeakSmem, stream>>>(iters, cycles, ns, err, 4000000000ull);
  return cudaGetLastError();
}

cudaError_t launch_read_stream(const void* src, int64_t bytes, void* sink, int grid, cudaStream_t stream) {
  read_stream_kernel<<<grid, 512, 0, stream>>>(static_cast<const uint4*>(src), bytes / 16,
                                               static_cast<uint32_t*>(sink));
  return cudaGetLastError();
}

}  // namespace sg

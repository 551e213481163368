// CUDA-core skinny GEMM (decode GEMV) for M <= 8 activation rows.
//
// C[m, n] = sum_k A[m, k] B[n, k]: each warp owns R consecutive weight rows n and
// streams them along K with 16-byte (8 x bf16) loads, adjacent lanes on adjacent
// 16-byte vectors so one warp instruction reads 512 contiguous bytes of a row.
// Every loaded weight vector is multiplied against all M activation rows before
// the next one is loaded, so each weight byte crosses the memory bus once
// ("The kernels that were there", "The GEMV": parallel over output columns, warps
// stride K with adjacent threads on adjacent weights, 128-bit loads, fp32
// accumulation, bf16 store; the M = 2 kernel feeds both rows from one load).
// Per-lane fp32 partials are combined with warp shuffles.
//
// When there are too few row groups to keep enough bytes in flight, K is cut
// into split_k slices (blockIdx.y).  Each slice writes fp32 partials; the last
// slice of a row group to finish (an arrival counter) sums the slices in slice
// order, stores bf16 and resets the counter, so the result is the same every
// run and nothing needs clearing between calls (spark-kernels, "the decode
// kernel": split K only when the strips are too few, and keep it to one launch).
#include <cuda_bf16.h>

#include "sg_internal.h"

namespace sg {
namespace {

constexpr int kCcWarps = 8;
constexpr int kCcUnroll = 4;

__device__ __forceinline__ uint4 ld_stream_v4(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);             // low half: element 2i
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);  // high half: element 2i+1
  }
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

template <int MT, int R>
__global__ void __launch_bounds__(kCcWarps * 32) cc_gemv_kernel(const CcParams p) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n0 = blockIdx.x * p.rows_per_cta + warp * R;
  const int slice = blockIdx.y;
  const int kb = slice * p.k_slice;
  const int ke = min(p.K, kb + p.k_slice);
  const int kvec_end = kb + ((max(ke - kb, 0)) / 8) * 8;

  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

  bool row_ok[R];
  const uint16_t* brow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    row_ok[r] = (n0 + r) < p.N;
    brow[r] = p.B + static_cast<int64_t>(row_ok[r] ? n0 + r : 0) * p.ldb;
  }

  for (int k = kb + lane * 8; k < kvec_end; k += 32 * 8 * kCcUnroll) {
    uint4 wv[kCcUnroll][R];
#pragma unroll
    for (int u = 0; u < kCcUnroll; ++u) {
      const int kk = k + u * 256;
#pragma unroll
      for (int r = 0; r < R; ++r)
        wv[u][r] = (kk < kvec_end && row_ok[r]) ? ld_stream_v4(brow[r] + kk) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kCcUnroll; ++u) {
      const int kk = k + u * 256;
      if (kk < kvec_end) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < p.M) {
            float a[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.A + static_cast<int64_t>(m) * p.lda + kk)), a);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float w[8];
              bf16x8_to_f32(wv[u][r], w);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[r][m] = fmaf(w[e], a[e], acc[r][m]);
            }
          }
        }
      }
    }
  }
  // K tail (fewer than 8 elements): one element per lane.
  {
    const int k = kvec_end + lane;
    if (k < ke) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float w = row_ok[r] ? bf16_to_f32(brow[r][k]) : 0.f;
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < p.M) acc[r][m] = fmaf(w, bf16_to_f32(p.A[static_cast<int64_t>(m) * p.lda + k]), acc[r][m]);
      }
    }
  }
  // Warp reduction: every lane ends with the full sums.
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      acc[r][m] = v;
    }

  __nv_bfloat16* C = reinterpret_cast<__nv_bfloat16*>(p.C);
  if (p.split_k == 1) {
    // Lane (r * MT + m) stores element (m, n0 + r).
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (lane == r * MT + m && m < p.M && row_ok[r])
          C[static_cast<int64_t>(m) * p.ldc + n0 + r] = __float2bfloat16_rn(acc[r][m]);
    return;
  }

  // Split K: publish this slice's partials, the last slice to arrive finishes.
  float* part = p.partials + static_cast<int64_t>(slice) * p.M * p.N;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (lane == r * MT + m && m < p.M && row_ok[r]) part[static_cast<int64_t>(m) * p.N + n0 + r] = acc[r][m];
  __threadfence();
  __syncthreads();
  __shared__ uint32_t is_last;
  if (threadIdx.x == 0) {
    const uint32_t before = atomicAdd(&p.counters[blockIdx.x], 1u);
    is_last = (before == static_cast<uint32_t>(p.split_k - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int rows = p.rows_per_cta;
  const int nb = blockIdx.x * rows;
  for (int e = threadIdx.x; e < rows * p.M; e += blockDim.x) {
    const int m = e / rows;
    const int n = nb + e % rows;
    if (n >= p.N) continue;
    float s = 0.f;
    for (int sl = 0; sl < p.split_k; ++sl)
      s = (sl == 0) ? __ldcg(p.partials + (static_cast<int64_t>(sl) * p.M + m) * p.N + n)
                    : s + __ldcg(p.partials + (static_cast<int64_t>(sl) * p.M + m) * p.N + n);
    C[static_cast<int64_t>(m) * p.ldc + n] = __float2bfloat16_rn(s);
  }
  if (threadIdx.x == 0) atomicExch(&p.counters[blockIdx.x], 0u);
}

template <int MT>
cudaError_t launch_mt(const CcParams& p, int grid_rows, cudaStream_t stream) {
  dim3 grid(grid_rows, p.split_k);
  const int R = p.rows_per_cta / kCcWarps;
  switch (R) {
    case 1: cc_gemv_kernel<MT, 1><<<grid, kCcWarps * 32, 0, stream>>>(p); break;
    case 2: cc_gemv_kernel<MT, 2><<<grid, kCcWarps * 32, 0, stream>>>(p); break;
    case 4: cc_gemv_kernel<MT, 4><<<grid, kCcWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cc_gemv(const CcParams& p, int grid_rows, cudaStream_t stream) {
  if (p.M <= 1) return launch_mt<1>(p, grid_rows, stream);
  if (p.M <= 2) return launch_mt<2>(p, grid_rows, stream);
  if (p.M <= 4) return launch_mt<4>(p, grid_rows, stream);
  if (p.M <= 8) return launch_mt<8>(p, grid_rows, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sg

// CUDA-core skinny GEMM (decode GEMV) for M <= 8 activation rows per launch (the
// automatic choice sends it M <= 2; beyond that the tcgen05 kernel is faster).
//
// C[m, n] = sum_k A[m, k] B[n, k].  The grid is grid_rows x split_k CTAs.  CTA
// (b, s) owns the contiguous weight rows [b*N/grid_rows, (b+1)*N/grid_rows), so
// every CTA streams one contiguous block of B, and K slice s.  Inside the CTA the 8
// warps split the slice along K; each warp walks the CTA's rows R at a time with
// 16-byte (8 x bf16) non-caching loads, adjacent lanes on adjacent 16-byte vectors
// (512 contiguous bytes per row per warp instruction).  Every loaded weight vector
// is multiplied against all M activation rows before the next is loaded, so each
// weight byte crosses the memory bus once; pairs of weight rows share paired fp32
// FMAs (fma.rn.f32x2, two independent single-rounding FMAs) ("The kernels that were there", "The
// GEMV": parallel over output columns, warps stride K with adjacent threads on
// adjacent weights, 128-bit loads, fp32 accumulation, bf16 store; the M = 2
// kernel feeds both rows from one load).  Lane partials are combined with warp
// shuffles, and the 8 warps' partials are summed in warp order through shared
// memory, so the result does not depend on timing.
//
// When there are too few rows to give every SM two CTAs, K is also split across
// CTAs (split_k > 1).  Each slice writes fp32 partials, and the last slice of a
// row block to finish (an arrival counter) sums the slices in slice order, stores
// bf16 and resets the counter.  Nothing needs clearing between calls, and a call
// is one launch (spark-kernels, "the decode kernel": split K only when the strips
// are too few).
#include <algorithm>
#include <cuda_bf16.h>

#include "sg_internal.h"
#include "sg_ptx.cuh"

namespace sg {
namespace {

constexpr int kCcWarps = 8;

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

// The rows [lo, hi) of the N output rows that one CTA computes, and its weights.
// In a batched launch the host gives every matrix its own run of CTAs
// (cta_begin), so a CTA's rows all belong to one matrix i: row n is row
// n - first of that matrix (first = row_begin[i]).  The matrix is looked up once
// per CTA (and again for the stores, rather than held in registers throughout).
__device__ __forceinline__ int cta_batch(const CcParams& p) {
  int i = 0;
#pragma unroll
  for (int j = 1; j < kMaxBatch; ++j)
    if (j < p.nbatch && static_cast<int>(blockIdx.x) >= p.cta_begin[j]) i = j;
  return i;
}

struct CtaRows {
  const uint16_t* b;
  int64_t ldb;
  int first, lo, hi;
};

template <bool BATCHED>
__device__ __forceinline__ CtaRows cta_rows(const CcParams& p) {
  CtaRows t;
  if constexpr (!BATCHED) {
    t.b = p.B;
    t.ldb = p.ldb;
    t.first = 0;
    t.lo = static_cast<int>((static_cast<int64_t>(blockIdx.x) * p.N) / p.grid_rows);
    t.hi = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * p.N) / p.grid_rows);
    return t;
  }
  const int i = cta_batch(p);
  const int64_t ctas = p.cta_begin[i + 1] - p.cta_begin[i];
  const int64_t b = static_cast<int64_t>(blockIdx.x) - p.cta_begin[i];
  const int64_t rows = p.row_begin[i + 1] - p.row_begin[i];
  t.b = p.Bs[i];
  t.ldb = p.ldbs[i];
  t.first = p.row_begin[i];
  t.lo = t.first + static_cast<int>((b * rows) / ctas);
  t.hi = t.first + static_cast<int>(((b + 1) * rows) / ctas);
  return t;
}

__device__ __forceinline__ const uint16_t* weight_row(const CtaRows& t, int n) {
  return t.b + static_cast<int64_t>(n - t.first) * t.ldb;
}

// Where this CTA's outputs go: output row n, activation row m at
// out + m * ldc + (n - first).
struct CtaOut {
  uint16_t* out;
  int64_t ldc;
  int first;
  __device__ __forceinline__ uint16_t* at(int64_t m, int64_t n) const { return out + m * ldc + (n - first); }
};

template <bool BATCHED>
__device__ __forceinline__ CtaOut cta_out(const CcParams& p) {
  if constexpr (!BATCHED) {
    return {p.C, p.ldc, 0};
  } else {
    const int i = cta_batch(p);
    return {p.Cs[i], p.ldcs[i], p.row_begin[i]};
  }
}

// The residual R[m, n] as fp32 (0 without one); R may be C itself.
__device__ __forceinline__ float residual(const CcParams& p, int64_t m, int64_t n) {
  return p.R != nullptr ? __uint_as_float(static_cast<uint32_t>(p.R[m * p.ldr + n]) << 16) : 0.f;
}

// silu(g) * u = g / (1 + e^-g) * u in fp32 (a signed zero where e^-g is inf).
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// One butterfly step per lane bit OFF = 16, 8, ..., 1 over the N values still
// held: lanes with that bit set keep the upper half, the others the lower half,
// and each kept value gains its partner's copy.  Once one value is left, the
// remaining steps add the partner's value.
template <int N, int OFF>
struct Butterfly {
  __device__ __forceinline__ static void run(float* v, int lane, int& idx) {
    if constexpr (OFF > 0) {
      if constexpr (N > 1) {
        constexpr int H = N / 2;
        const bool upper = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = upper ? v[i] : v[i + H];
          const float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, OFF);
        }
        if (upper) idx += H;
        Butterfly<H, OFF / 2>::run(v, lane, idx);
      } else {
        v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], OFF);
        Butterfly<1, OFF / 2>::run(v, lane, idx);
      }
    }
  }
};

// MT: activation rows held (>= M); R: weight rows per warp pass; U: 16-byte
// vectors per lane per row in flight.  GATED: the CTA's rows are outputs n, each
// from weight row n of B (gate) and of B2 (up); a pass takes R / 2 outputs, their
// gate and up rows sharing each paired FMA, and the result is silu(gate) * up.
template <int MT, int R, int U, bool GATED, bool BATCHED>
__global__ void __launch_bounds__(kCcWarps * 32, 2) cc_gemv_kernel(const CcParams p) {
  extern __shared__ float red[];  // [rows of this CTA (x 2 gated)][MT][kCcWarps]
  constexpr int kRowStep = GATED ? R / 2 : R;  // output rows per pass
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const CtaRows rows_of = cta_rows<BATCHED>(p);
  const int row_lo = rows_of.lo;
  const int row_hi = rows_of.hi;
  const int slice = blockIdx.y;
  const int kb = slice * p.k_slice;
  const int ke = min(p.K, kb + p.k_slice);
  const int nvec = max(ke - kb, 0) / 8;  // whole 16-byte vectors in this slice
  const int v_lo = kb / 8 + (warp * nvec) / kCcWarps;
  const int v_hi = kb / 8 + ((warp + 1) * nvec) / kCcWarps;
  const int tail_k = kb + nvec * 8;  // [tail_k, ke): fewer than 8 elements, warp 0
  if (p.prewait && lane < R && v_hi > v_lo) {
    // The first row pass's weights of this warp's k range, pulled into L2 while
    // the previous launch may still be finishing (a hint: L2 is the point of
    // coherence, so nothing read here can be stale once the wait returns).
    const int r = lane;
    const int n = row_lo + (GATED ? r / 2 : r);
    if (n < row_hi) {
      const uint16_t* row = GATED ? ((r & 1) ? p.B2 : p.B) + static_cast<int64_t>(n) * p.ldb : weight_row(rows_of, n);
      bulk_prefetch_l2(row + 8 * v_lo, static_cast<uint32_t>(v_hi - v_lo) * 16u);
    }
  }
  grid_dependency_wait();  // no global load before the previous kernel has completed

  static_assert(R % 2 == 0, "weight rows are processed in pairs");
  // Without a K split, each thread's outputs are known from the start: elements
  // threadIdx.x + j * blockDim.x of the CTA's rows x M block (at most 8 of them:
  // rows <= 256, M <= 8).  Their residuals are loaded now, behind the stream.
  constexpr int kResidPer = 8;
  float rres[kResidPer];
  if (!GATED && p.R != nullptr && p.split_k == 1) {
#pragma unroll
    for (int j = 0; j < kResidPer; ++j) {
      const int e = threadIdx.x + j * kCcWarps * 32;
      rres[j] = e < (row_hi - row_lo) * p.M ? residual(p, e % p.M, row_lo + e / p.M) : 0.f;
    }
  }
  for (int r0 = row_lo; r0 < row_hi; r0 += kRowStep) {
    // The next launch may start its set-up (and early prefetch) once every CTA is
    // on its last row pass.
    if (r0 + kRowStep >= row_hi) grid_launch_dependents();
    // acc[r / 2][m] holds the fp32 sums of weight rows r (x) and r + 1 (y) for
    // activation row m; one paired FMA updates both.
    float2 acc[R / 2][MT];
#pragma unroll
    for (int r = 0; r < R / 2; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.f, 0.f);
    const uint16_t* brow[R];
    bool row_ok[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if constexpr (GATED) {  // gate and up rows of output r0 + r / 2
        row_ok[r] = r0 + r / 2 < row_hi;
        brow[r] = ((r & 1) ? p.B2 : p.B) + static_cast<int64_t>(row_ok[r] ? r0 + r / 2 : r0) * p.ldb;
      } else {
        row_ok[r] = r0 + r < row_hi;
        brow[r] = weight_row(rows_of, row_ok[r] ? r0 + r : r0);
      }
    }
    for (int v = v_lo + lane; v < v_hi; v += 32 * U) {
      uint4 wv[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vv = v + 32 * u;
#pragma unroll
        for (int r = 0; r < R; ++r)
          wv[u][r] = (vv < v_hi && row_ok[r]) ? ld_stream_v4(brow[r] + 8 * vv) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vv = v + 32 * u;
        if (vv < v_hi) {
          // activations of this k vector for every row (rows past M read as 0)
          float a[MT][8];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 av = m < p.M
                                 ? __ldg(reinterpret_cast<const uint4*>(p.A + static_cast<int64_t>(m) * p.lda + 8 * vv))
                                 : make_uint4(0, 0, 0, 0);
            bf16x8_to_f32(av, a[m]);
          }
          // each weight vector is widened once and used for all MT rows; two
          // weight rows share each paired FMA (the same fp32 operations, in the
          // same order, as two scalar FMAs)
#pragma unroll
          for (int r = 0; r < R / 2; ++r) {
            float w0[8], w1[8];
            bf16x8_to_f32(wv[u][2 * r], w0);
            bf16x8_to_f32(wv[u][2 * r + 1], w1);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
              for (int e = 0; e < 8; ++e)
                acc[r][m] = __ffma2_rn(make_float2(w0[e], w1[e]), make_float2(a[m][e], a[m][e]), acc[r][m]);
          }
        }
      }
    }
    if (warp == 0 && tail_k + lane < ke) {  // K tail: one element per lane
      const int k = tail_k + lane;
#pragma unroll
      for (int r = 0; r < R / 2; ++r) {
        const float w0 = row_ok[2 * r] ? bf16_to_f32(brow[2 * r][k]) : 0.f;
        const float w1 = row_ok[2 * r + 1] ? bf16_to_f32(brow[2 * r + 1][k]) : 0.f;
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < p.M) {
            const float x = bf16_to_f32(p.A[static_cast<int64_t>(m) * p.lda + k]);
            acc[r][m] = __ffma2_rn(make_float2(w0, w1), make_float2(x, x), acc[r][m]);
          }
      }
    }
    // Reduce the R x MT sums across the warp's 32 lanes with a butterfly that
    // also scatters them: at each step a lane keeps half of its values and sends
    // the other half to its partner, so NV values take NV - 1 + (5 - log2 NV)
    // shuffles instead of 5 NV.  Afterwards lane l holds the full sum of value
    // index(l) (flattened r * MT + m), duplicated in lanes 2^(log2 NV) apart.
    constexpr int NV = R * MT;
    static_assert((NV & (NV - 1)) == 0 && NV <= 32, "power-of-two sums per lane");
    float v[NV];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) v[r * MT + m] = (r & 1) ? acc[r / 2][m].y : acc[r / 2][m].x;
    int idx = 0;
    Butterfly<NV, 16>::run(v, lane, idx);
    if ((lane & ((32 / NV) - 1)) == 0) {  // one lane per value index
      const int r = idx / MT, m = idx % MT;
      if constexpr (GATED) {  // red row 2 * output + (0 gate, 1 up)
        if (r0 + r / 2 < row_hi) red[(((r0 - row_lo) * 2 + r) * MT + m) * kCcWarps + warp] = v[0];
      } else {
        if (r0 + r < row_hi) red[((r0 + r - row_lo) * MT + m) * kCcWarps + warp] = v[0];
      }
    }
  }
  __syncthreads();

  // Sum the warps' partials in warp order.  Split-K partials are [slice][gu][M][N]
  // (gu = 0 gate, 1 up; one plane when not gated).
  constexpr int kPlanes = GATED ? 2 : 1;
  const int rows = row_hi - row_lo;
  float* part = p.partials + static_cast<int64_t>(slice) * kPlanes * p.M * p.N;
  // rows * M <= 256 * 8 = kResidPer * blockDim.x: element e = threadIdx.x + j * blockDim.x
#pragma unroll
  for (int j = 0; j < kResidPer; ++j) {
    const int e = threadIdx.x + j * kCcWarps * 32;
    if (e >= rows * p.M) break;
    const int r = e / p.M, m = e % p.M;
    float s[kPlanes];
#pragma unroll
    for (int gu = 0; gu < kPlanes; ++gu) {
      const float* src = red + ((r * kPlanes + gu) * MT + m) * kCcWarps;
      s[gu] = src[0];
#pragma unroll
      for (int w = 1; w < kCcWarps; ++w) s[gu] += src[w];
    }
    if (p.split_k == 1) {
      const int64_t n = row_lo + r;
      const CtaOut o = cta_out<BATCHED>(p);
      const float res = (!GATED && p.R != nullptr) ? rres[j] : 0.f;  // prefetched at the start
      *reinterpret_cast<__nv_bfloat16*>(o.at(m, n)) =
          __float2bfloat16_rn(GATED ? silu_mul(s[0], s[kPlanes - 1]) : s[0] + res);
    } else {
#pragma unroll
      for (int gu = 0; gu < kPlanes; ++gu) part[(static_cast<int64_t>(gu) * p.M + m) * p.N + row_lo + r] = s[gu];
    }
  }
  if (p.split_k == 1) return;

  // Split K across CTAs: the last slice of this row block to arrive finishes.
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
  const CtaOut o = cta_out<BATCHED>(p);
  for (int e = threadIdx.x; e < rows * p.M; e += blockDim.x) {
    const int r = e / p.M, m = e % p.M;
    const int n = row_lo + r;
    float s[kPlanes];
#pragma unroll
    for (int gu = 0; gu < kPlanes; ++gu) {
      s[gu] = 0.f;
      for (int sl = 0; sl < p.split_k; ++sl) {
        const float x = __ldcg(p.partials + ((static_cast<int64_t>(sl) * kPlanes + gu) * p.M + m) * p.N + n);
        s[gu] = (sl == 0) ? x : s[gu] + x;
      }
    }
    *reinterpret_cast<__nv_bfloat16*>(o.at(m, n)) =
        __float2bfloat16_rn(GATED ? silu_mul(s[0], s[kPlanes - 1]) : s[0] + residual(p, m, n));
  }
  if (threadIdx.x == 0) atomicExch(&p.counters[blockIdx.x], 0u);
}

template <int MT, int R, int U, bool GATED, bool BATCHED = false>
cudaError_t launch_one(const CcParams& p, cudaStream_t stream) {
  int rows_max = (p.N + p.grid_rows - 1) / p.grid_rows;
  if (p.nbatch > 0) {  // the largest row block of any matrix's run of CTAs
    rows_max = 0;
    for (int i = 0; i < p.nbatch; ++i) {
      const int rows = p.row_begin[i + 1] - p.row_begin[i];
      const int ctas = p.cta_begin[i + 1] - p.cta_begin[i];
      if (ctas < 1) return cudaErrorInvalidValue;
      rows_max = std::max(rows_max, (rows + ctas - 1) / ctas);
    }
  }
  const size_t smem = static_cast<size_t>(rows_max) * (GATED ? 2 : 1) * MT * kCcWarps * sizeof(float);
  auto kern = cc_gemv_kernel<MT, R, U, GATED, BATCHED>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid_rows, p.split_k, 1);
  cfg.blockDim = dim3(kCcWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int cc_smem_bytes(int64_t M, int64_t N, int grid_rows, bool gated) {
  const int64_t mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  return static_cast<int>(((N + grid_rows - 1) / grid_rows) * (gated ? 2 : 1) * mt * kCcWarps * sizeof(float));
}

cudaError_t launch_cc_gemv(const CcParams& p, cudaStream_t stream) {
  if (p.B2 != nullptr) {
    if (p.M <= 1) return launch_one<1, 8, 2, true>(p, stream);
    if (p.M <= 2) return launch_one<2, 8, 2, true>(p, stream);
    if (p.M <= 4) return launch_one<4, 4, 2, true>(p, stream);
    if (p.M <= 8) return launch_one<8, 2, 2, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (p.nbatch > 0) {
    if (p.M <= 1) return launch_one<1, 8, 2, false, true>(p, stream);
    if (p.M <= 2) return launch_one<2, 8, 2, false, true>(p, stream);
    if (p.M <= 4) return launch_one<4, 4, 2, false, true>(p, stream);
    if (p.M <= 8) return launch_one<8, 2, 2, false, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (p.M <= 1) return launch_one<1, 8, 2, false>(p, stream);
  if (p.M <= 2) return launch_one<2, 8, 2, false>(p, stream);
  if (p.M <= 4) return launch_one<4, 4, 2, false>(p, stream);
  if (p.M <= 8) return launch_one<8, 2, 2, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sg

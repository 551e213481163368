// Decode attention on CUDA cores: the few query rows of one kv-head group (all
// Sq queries of the H / Hkv heads that share a K/V head; at most four rows)
// against a range of the keys, with K and V streamed once by plain 16-byte loads.
//
// spark-kernels, "Fused attention": one decode query against a 4096-token cache
// is bound by reading K and V (the page's 49 us at 1366 GB/s, 89% of that card's
// copy roof).  With one query row, the tensor-core kernel's 128-row score tiles
// are almost all padding, and its per-key-block dependency chain sets the pace
// instead of the memory stream.  Here each CTA takes one (batch, kv head, key
// range), its rows share every K/V byte it reads, and the key ranges (splits)
// are merged by attn_combine_kernel from the same fp32 partials the tensor-core
// kernel writes.
//
// Lane layout: lane = 8 kg + dg, key group kg (4 keys side by side in a warp)
// and dimension group dg (dims 16 dg .. 16 dg + 15, 32 bytes of a key row, so 8
// lanes read one 256-byte row).  Each (warp, key group) keeps its own online
// softmax state (row maximum m and sum l in log2 units, output o over its 16
// dims); the 32 states of a CTA are merged at the end.  Scores are
// (q . k) * scale * log2 e and the weights 2^(s - m) (ex2.approx), in fp32;
// the weights are not rounded to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sg_internal.h"
#include "sg_ptx.cuh"

namespace sg {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kKeysPerStep = kDecWarps * 4;  // keys a CTA takes side by side (key groups x warps)

__device__ __forceinline__ float dec_exp2(float x) {  // 2^x, ex2.approx (2^-inf = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16 bytes of K or V, read once: streamed past L1.
__device__ __forceinline__ uint4 ld_kv_v4(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bf16x8_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&v);
}

// RT: query rows held (>= a.rows); C: keys per lane per step (their K and V
// loads in flight together).  Four rows take one CTA per SM (registers).
template <int RT, int C>
__global__ void __launch_bounds__(kDecThreads, RT >= 4 ? 1 : 2) attn_decode_kernel(const AttnParams p, const AttnDecodeArgs a) {
  __shared__ float sm_m[kDecWarps][RT];
  __shared__ float sm_l[kDecWarps][RT];
  __shared__ float sm_o[kDecWarps][RT][kAttnHeadDim];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int kg = lane >> 3, dg = lane & 7;
  const int G = p.H / p.Hkv;
  const int split = static_cast<int>(blockIdx.x % p.n_splits);
  const int bg = static_cast<int>(blockIdx.x / p.n_splits);
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int ka = split * a.keys_per_split;
  const int kb = min(p.Sk, ka + a.keys_per_split);

  // The first round's K and V rows (256 bytes each), pulled into L2 while the
  // previous launch may still be finishing: a hint only (L2 is the point of
  // coherence, so the loads after the wait see that launch's writes).
  if (dg == 0) {
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int j = ka + kKeysPerStep * c + 4 * warp + kg;
      if (j < kb) {
        const int64_t kvr = static_cast<int64_t>(b) * p.Sk + j;
        bulk_prefetch_l2(a.K + kvr * a.ldk + g * kAttnHeadDim, kAttnHeadDim * 2);
        bulk_prefetch_l2(a.V + kvr * a.ldv + g * kAttnHeadDim, kAttnHeadDim * 2);
      }
    }
  }
  grid_dependency_wait();  // Q, K and V may come from the previous kernel

  // this lane's 16 dims of each query row (bf16 pairs), and each row's last visible key
  uint32_t q[RT][8];
  int lim[RT];
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const int i = r / G, h = g * G + r % G;
    if (r < a.rows) {
      const uint4* src = reinterpret_cast<const uint4*>(a.Q + (static_cast<int64_t>(b) * p.Sq + i) * a.ldq +
                                                        h * kAttnHeadDim + 16 * dg);
      const uint4 v0 = src[0], v1 = src[1];
      q[r][0] = v0.x; q[r][1] = v0.y; q[r][2] = v0.z; q[r][3] = v0.w;
      q[r][4] = v1.x; q[r][5] = v1.y; q[r][6] = v1.z; q[r][7] = v1.w;
      lim[r] = p.causal ? i + (p.Sk - p.Sq) : p.Sk - 1;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[r][e] = 0u;
      lim[r] = -1;  // sees nothing
    }
  }
  float m[RT], l[RT], o[RT][16];
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) o[r][e] = 0.f;
  }
  const int64_t kv_row0 = static_cast<int64_t>(b) * p.Sk;
  const int col = g * kAttnHeadDim + 16 * dg;
  // warp-uniform trip count (the score sums shuffle across the warp)
  for (int base = ka; base < kb; base += kKeysPerStep * C) {
    uint4 kv[C][2], vv[C][2];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int j = base + kKeysPerStep * c + 4 * warp + kg;
      if (j < kb) {
        const uint16_t* kr = a.K + (kv_row0 + j) * a.ldk + col;
        const uint16_t* vr = a.V + (kv_row0 + j) * a.ldv + col;
        kv[c][0] = ld_kv_v4(kr);
        kv[c][1] = ld_kv_v4(kr + 8);
        vv[c][0] = ld_kv_v4(vr);
        vv[c][1] = ld_kv_v4(vr + 8);
      } else {
        kv[c][0] = kv[c][1] = vv[c][0] = vv[c][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // scores s[r][c] in log2 units (-inf: masked or past the range)
    float s[RT][C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      float kf[16];
      bf16x8_f32(kv[c][0], kf);
      bf16x8_f32(kv[c][1], kf + 8);
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dot = fmaf(__uint_as_float(q[r][e] << 16), kf[2 * e], dot);
          dot = fmaf(__uint_as_float(q[r][e] & 0xFFFF0000u), kf[2 * e + 1], dot);
        }
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 2);
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 4);
        const int j = base + kKeysPerStep * c + 4 * warp + kg;
        s[r][c] = (j < kb && j <= lim[r]) ? dot * p.scale_log2 : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float cm = s[r][0];
#pragma unroll
      for (int c = 1; c < C; ++c) cm = fmaxf(cm, s[r][c]);
      if (cm == -INFINITY) continue;  // nothing visible in this step
      const float mn = fmaxf(m[r], cm);
      const float corr = dec_exp2(m[r] - mn);  // 0 while nothing was visible
      m[r] = mn;
      l[r] *= corr;
#pragma unroll
      for (int e = 0; e < 16; ++e) o[r][e] *= corr;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const float w = dec_exp2(s[r][c] - mn);
        l[r] += w;
        float vf[16];
        bf16x8_f32(vv[c][0], vf);
        bf16x8_f32(vv[c][1], vf + 8);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[r][e] = fmaf(w, vf[e], o[r][e]);
      }
    }
  }
  grid_launch_dependents();  // the combine kernel may start its set-up

  // merge the four key groups of the warp (lanes dg, dg + 8, dg + 16, dg + 24)
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    float mw = fmaxf(m[r], __shfl_xor_sync(0xFFFFFFFFu, m[r], 8));
    mw = fmaxf(mw, __shfl_xor_sync(0xFFFFFFFFu, mw, 16));
    const float corr = m[r] == -INFINITY ? 0.f : dec_exp2(m[r] - mw);
    float lw = l[r] * corr;
    lw += __shfl_xor_sync(0xFFFFFFFFu, lw, 8);
    lw += __shfl_xor_sync(0xFFFFFFFFu, lw, 16);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float x = o[r][e] * corr;
      x += __shfl_xor_sync(0xFFFFFFFFu, x, 8);
      x += __shfl_xor_sync(0xFFFFFFFFu, x, 16);
      o[r][e] = x;
    }
    if (kg == 0) {
#pragma unroll
      for (int e = 0; e < 16; ++e) sm_o[warp][r][16 * dg + e] = o[r][e];
      if (dg == 0) {
        sm_m[warp][r] = mw;
        sm_l[warp][r] = lw;
      }
    }
  }
  __syncthreads();

  // merge the warps: thread t takes (row, dim) pairs t, t + 256, ...
  const int64_t rows_all = static_cast<int64_t>(p.B) * p.Sq * p.H;
  for (int t = threadIdx.x; t < a.rows * kAttnHeadDim; t += kDecThreads) {
    const int r = t / kAttnHeadDim, d = t % kAttnHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w][r]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = sm_m[w][r] == -INFINITY ? 0.f : dec_exp2(sm_m[w][r] - M);
        L = fmaf(sm_l[w][r], f, L);
        acc = fmaf(sm_o[w][r][d], f, acc);
      }
    }
    const float out = L > 0.f ? acc / L : 0.f;
    const int i = r / G, h = g * G + r % G;
    const int64_t row = static_cast<int64_t>(b) * p.Sq + i;
    // a warp holds 32 consecutive dims of one row (rows x 128 is a multiple of 32,
    // so every lane of a warp runs this iteration): the odd dim's value comes
    // from the next lane
    const float hi = __shfl_down_sync(0xFFFFFFFFu, out, 1);
    if (p.n_splits == 1) {
      if ((d & 1) == 0) *reinterpret_cast<uint32_t*>(p.O + row * p.ldo + h * kAttnHeadDim + d) = pack2_bf16(out, hi);
    } else {
      const int64_t unit = static_cast<int64_t>(split) * rows_all + row * p.H + h;
      p.part_o[unit * kAttnHeadDim + d] = out;
      if (d == 0) p.part_lse[unit] = L > 0.f ? M + __log2f(L) : -INFINITY;
    }
  }
}

template <int RT, int C>
cudaError_t launch_rows(const AttnParams& p, const AttnDecodeArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(p.B) * p.Hkv * p.n_splits), 1, 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<RT, C>, p, a);
}

}  // namespace

cudaError_t launch_attn_decode(const AttnParams& p, const AttnDecodeArgs& a, cudaStream_t stream) {
  if (a.rows <= 1) return launch_rows<1, 4>(p, a, stream);
  if (a.rows <= 2) return launch_rows<2, 3>(p, a, stream);
  if (a.rows <= kAttnDecodeMaxRows) return launch_rows<4, 4>(p, a, stream);  // one CTA per SM
  return cudaErrorInvalidValue;
}

}  // namespace sg

// Fused scaled dot-product attention (forward) on the 5th-generation tensor
// cores, head dimension 128, bf16 in and out, fp32 softmax and accumulation:
//
//   O[i] = sum_j softmax_j(scale * q_i . k_j over the keys visible to i) v_j
//
// the attention kernel of the spark-kernels page ("attention": flash attention,
// the online softmax between two tensor-core products S = Q K^T and O += P V, P
// rounded to bf16 for the second product, causal tiles above the diagonal never
// loaded, the heaviest query tiles launched first).
//
// One CTA per (128-row query tile, head, batch), or per key split of one.
// Roles:
//   warp 0     TMA producer: the Q tile once (two 64-column boxes, 128-byte
//              swizzle), then per key block a K tile and a V tile (128 keys x
//              128 columns each) into a 3-stage ring
//   warp 1     TMEM allocator and MMA issuer (one thread): S_j = Q K_j^T into one
//              of two 128-column TMEM buffers (K-major A and B from shared
//              memory), then, once the softmax has written P_j, O += P_j V_j with
//              P read from TMEM and V the B operand in MN-major form (the key rows
//              of the V tile as TMA wrote them), so nothing is transposed
//   warps 2-9  softmax, two threads per query row (the row's TMEM lane; warps w
//              and w + 4 share a lane quarter and take 64 columns each, swapping
//              row maxima through shared memory): S row -> scale, mask, running
//              max and sum -> P row as bf16 into one of two TMEM P buffers; at the
//              end O / l is rounded to bf16 and stored
// TMEM columns: S buffers [0, 128) and [128, 256), O [256, 384), P buffers
// [384, 448) and [448, 512) (bf16 pairs).  The tensor core runs S_{j+1} and
// P_j V_j while the softmax works on block j + 1: the softmax never waits for a
// P V product unless the row max grew by more than 2^8 since the max its weights
// are taken against, when O must be rescaled first (the weights themselves stay
// below 2^8, which bf16 and the fp32 sums hold exactly enough).
//
// Key j is visible to query i when j < Sk and, for a causal launch, j <= i +
// (Sk - Sq).  A row that sees no key gets O = 0.  Scores are kept in log2 units
// (scale * log2 e folded into one multiply) and exponentiated with ex2.approx.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sg_internal.h"
#include "sg_ptx.cuh"

namespace sg {
namespace {

constexpr int kAtStages = 3;
constexpr int kAtThreads = 320;           // warp 0 producer, warp 1 MMA, warps 2-9 softmax
constexpr int kAtBox = kAttnTile * 128;   // 128 rows x 128 bytes (64 bf16)
constexpr int kAtQOff = 0;                // Q: two boxes (d 0-63, 64-127)
constexpr int kAtKvOff = 2 * kAtBox;      // per stage: K boxes 0, 1 then V boxes 0, 1
constexpr int kAtStageBytes = 4 * kAtBox;
constexpr int kAtBarOff = kAtKvOff + kAtStages * kAtStageBytes;
// q, k[], v[], kv_empty[], s_full[2], p_ready[2], pv_done[2], teardown
constexpr int kAtNumBars = 1 + 3 * kAtStages + 2 + 2 + 2 + 1;
constexpr int kAtXchgOff = kAtBarOff + kAtNumBars * 8;  // row maxima / sums swapped by the two halves
constexpr int kAtMiscOff = kAtXchgOff + 256 * 4;
constexpr int kAtSmem = kAtMiscOff + 16 + 1024;
constexpr int kAtTmemCols = 512;
constexpr uint32_t kAtOCol = 256;
constexpr uint32_t kAtPCol = 384;         // P buffer b at kAtPCol + 64 b
constexpr float kAtRescaleLog2 = 8.f;     // O is rescaled once the row max grows past the reference by this
static_assert(kAtSmem <= 232448, "shared memory budget");
static_assert(kAttnHeadDim == 128 && kAttnTile == 128, "the tile shapes below assume 128");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Named barrier `id` over `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 2^x by the ex2.approx instruction (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Number of 128-key blocks query tile t must visit.
__device__ __forceinline__ int attn_blocks(const AttnParams& p, int q0) {
  int kend = p.Sk;
  if (p.causal) kend = min(p.Sk, min(q0 + kAttnTile, p.Sq) + (p.Sk - p.Sq));
  return kend > 0 ? (kend + kAttnTile - 1) / kAttnTile : 0;
}

__global__ void __launch_bounds__(kAtThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + kAtBarOff);
  uint64_t* k_full = q_full + 1;
  uint64_t* v_full = k_full + kAtStages;
  uint64_t* kv_empty = v_full + kAtStages;
  uint64_t* s_full = kv_empty + kAtStages;  // [2]
  uint64_t* p_ready = s_full + 2;   // [2]: block j on p_ready[j & 1]
  uint64_t* pv_done = p_ready + 2;  // [2]: P_j V_j complete, on pv_done[j & 1]
  uint64_t* teardown = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAtMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kAtMiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Query tiles in decreasing order: under a causal mask the last tiles see the
  // most keys, so they start first and the short ones fill the tail.
  const int split = static_cast<int>(blockIdx.x) % p.n_splits;
  const int unit = static_cast<int>(blockIdx.x) / p.n_splits;
  const int hb = unit % (p.H * p.B);
  const int t = p.q_tiles - 1 - unit / (p.H * p.B);
  const int h = hb % p.H;
  const int b = hb / p.H;
  const int kvh = h / (p.H / p.Hkv);
  const int q0 = t * kAttnTile;
  // this CTA's key blocks [j_begin, j_begin + nblk)
  const int tile_blocks = attn_blocks(p, q0);
  const int j_begin = split * p.split_blocks;
  const int nblk = max(0, min(tile_blocks - j_begin, p.split_blocks));
  // softmax warps whose 32 rows hold at least one query (the others idle)
  const int active_quarters = min(4, (p.Sq - q0 + 31) / 32);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kAtStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    for (int u = 0; u < 2; ++u) {
      mbar_init(&p_ready[u], 64u * static_cast<uint32_t>(active_quarters));
      mbar_init(&pv_done[u], 1);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kAtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      grid_dependency_wait();
      const int32_t qy = b * p.Sq + q0;
      if (nblk > 0) {  // a tile that sees no key loads nothing
        mbar_arrive_expect_tx(q_full, 2u * kAtBox);
        tma_load_2d(smem + kAtQOff, &tmQ, h * kAttnHeadDim, qy, q_full);
        tma_load_2d(smem + kAtQOff + kAtBox, &tmQ, h * kAttnHeadDim + 64, qy, q_full);
      }
      int j = 0;
      for (; j < nblk; ++j) {
        const uint32_t s = j % kAtStages;
        const uint32_t ph = (j / kAtStages) & 1u;
        if (!mbar_wait(&kv_empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutEmpty, j);
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + kAtKvOff + s * kAtStageBytes;
        const int32_t ky = b * p.Sk + (j_begin + j) * kAttnTile;
        const int32_t kx = kvh * kAttnHeadDim;
        mbar_arrive_expect_tx(&k_full[s], 2u * kAtBox + (j == 0 ? p.inject_extra_tx : 0u));  // + injection
        tma_load_2d(st, &tmK, kx, ky, &k_full[s]);
        tma_load_2d(st + kAtBox, &tmK, kx + 64, ky, &k_full[s]);
        mbar_arrive_expect_tx(&v_full[s], 2u * kAtBox);
        tma_load_2d(st + 2 * kAtBox, &tmV, kx, ky, &v_full[s]);
        tma_load_2d(st + 3 * kAtBox, &tmV, kx + 64, ky, &v_full[s]);
      }
      if (*abort_flag) {
        // Unwinding: let the copies already issued land before the CTA exits.
        volatile uint32_t never = 0;
        if (nblk > 0) mbar_wait(q_full, 0, p.timeout_ns, &never);
        for (int i = (j > kAtStages ? j - kAtStages : 0); i < j; ++i) {
          mbar_wait(&k_full[i % kAtStages], (i / kAtStages) & 1u, p.timeout_ns, &never);
          mbar_wait(&v_full[i % kAtStages], (i / kAtStages) & 1u, p.timeout_ns, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kAttnTile, kAttnTile);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kAttnTile, kAttnHeadDim) | (1u << 16);  // B MN-major
      const uint32_t base = smem_u32(smem);
      bool ok = nblk == 0 || mbar_wait(q_full, 0, p.timeout_ns, abort_flag);
      if (!ok && !*abort_flag) record_error(p.err, kDevTimeoutFull, 0);
      // S_j = Q K_j^T: K = 128 in 8 steps of 16 (32 bytes of a swizzle row; the
      // second 64 columns are the next box).
      auto issue_s = [&](int j) -> bool {
        const uint32_t s = j % kAtStages;
        if (!mbar_wait(&k_full[s], (j / kAtStages) & 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutFull, j);
          return false;
        }
        tc_fence_after();
        const uint32_t kaddr = base + kAtKvOff + s * kAtStageBytes;
        const uint32_t dst = tmem_base + static_cast<uint32_t>(j & 1) * kAttnTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kAtBox + (kk & 3) * 32;
          tc_mma_bf16(dst, smem_desc_sw128(base + kAtQOff + off), smem_desc_sw128(kaddr + off), kIdescS,
                      kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[j & 1]);
        return true;
      };
      if (ok && nblk > 0) ok = issue_s(0);
      for (int j = 0; j < nblk && ok; ++j) {
        // The S buffer of block j + 1 was last read by the softmax of block j - 1,
        // which finished before p_ready of j - 1 (waited for below last round).
        if (j + 1 < nblk && !(ok = issue_s(j + 1))) break;
        if (!mbar_wait(&p_ready[j & 1], (static_cast<uint32_t>(j) >> 1) & 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutTmemEmpty, j);
          ok = false;
          break;
        }
        const uint32_t s = j % kAtStages;
        if (!mbar_wait(&v_full[s], (j / kAtStages) & 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutFull, j);
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P_j V_j: K = 128 keys in 8 steps of 16 keys; P from TMEM (8 columns
        // of bf16 pairs per step), V MN-major (two 8-key atoms, 2048 bytes, per
        // step; the d columns 64-127 are the next box, kAtBox further on).
        const uint32_t vaddr = base + kAtKvOff + s * kAtStageBytes + 2 * kAtBox;
        const uint32_t pcol = tmem_base + kAtPCol + static_cast<uint32_t>(j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_bf16_ts(tmem_base + kAtOCol, pcol + kk * 8, smem_desc_sw128_mn(vaddr + kk * 2048, kAtBox), kIdescO,
                         (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[j & 1]);
        tc_commit(&kv_empty[s]);
      }
      if (!ok) *abort_flag = 1;
      if (*abort_flag) {
        // Unwinding: wait for every tcgen05 operation issued so far before TMEM is freed.
        tc_commit(teardown);
        volatile uint32_t never = 0;
        if (!mbar_wait(teardown, 0, p.timeout_ns, &never)) record_error(p.err, kDevTimeoutTeardown, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Two warps per TMEM lane quarter: warps 2-5 take columns 0-63 of their rows,
    // warps 6-9 columns 64-127; the two threads of a row swap their row maxima
    // through shared memory once per block (named barrier 1 + quarter).
    const int q = warp & 3;                // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;      // which 64 columns of the row
    const int r = q * 32 + lane;           // query row of the tile = TMEM lane
    const int i = q0 + r;                  // query index in the sequence
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t col0 = static_cast<uint32_t>(half * 64);
    // [2 halves][128 rows]: a value written for block j is read before the partner
    // passes the pair barrier at the start of block j + 1, so one buffer serves
    float* xchg = reinterpret_cast<float*>(smem + kAtXchgOff);
    // keys [0, lim) of this CTA's range are visible to this query (rows past Sq
    // compute garbage and store nothing)
    const int lim = (p.causal ? min(p.Sk, i + (p.Sk - p.Sq) + 1) : p.Sk) - j_begin * kAttnTile - half * 64;
    const bool active = q < active_quarters;
    float m_run = -INFINITY;  // the row's reference max (log2 units) the weights are taken against
    float l_run = 0.f;        // running sum of this thread's bf16-rounded weights
    bool ok = true;
    for (int j = 0; j < nblk && active; ++j) {
      const uint64_t limit = p.timeout_ns + 20000ull * static_cast<uint64_t>(j + 1);
      ok = mbar_wait(&s_full[j & 1], (static_cast<uint32_t>(j) >> 1) & 1u, limit, abort_flag);
      // both warps of the pair take the same decision (so both reach the same barriers)
      ok = !bar_sync_or(1 + q, 64, !ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(j & 1) * kAttnTile + col0 + 32 * c, sv[c]);
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld_wait(sv[c]);
      // scale into log2 units, mask (only where the block reaches past the row's
      // visible keys), max over 8 independent partial maxima
      const int kv = lim - j * kAttnTile;  // columns of this half visible: [0, kv)
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
      if (kv >= 64) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(sv[c][e]) * p.scale_log2;
            sv[c][e] = __float_as_uint(x);
            mx8[e & 7] = fmaxf(mx8[e & 7], x);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = (32 * c + e < kv) ? __uint_as_float(sv[c][e]) * p.scale_log2 : -INFINITY;
            sv[c][e] = __float_as_uint(x);
            mx8[e & 7] = fmaxf(mx8[e & 7], x);
          }
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // the row max: this half's and the other half's
      float* xb = xchg;
      xb[half * 128 + r] = mx;
      named_bar_sync(1 + q, 64);
      mx = fmaxf(mx, xb[(half ^ 1) * 128 + r]);
      // The reference moves only when the row max passes it by more than 2^8 (so
      // on the first block that shows a key); the two halves decide alike.
      const bool move = mx > m_run + kAtRescaleLog2;
      const float m_new = move ? mx : m_run;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = move ? fast_exp2(m_run - m_use) : 1.f;  // 0 while nothing was visible yet
      // weights, rounded to bf16 (the P V product's operand); l sums the rounded
      // values (8 independent partial sums, added in a fixed order)
      uint32_t pk[32];
      float rs8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(__uint_as_float(sv[c][2 * e]) - m_use);
          const float p1 = fast_exp2(__uint_as_float(sv[c][2 * e + 1]) - m_use);
          const uint32_t w = pack_bf16x2(p0, p1);
          pk[16 * c + e] = w;
          rs8[e & 7] += bf16_lo(w) + bf16_hi(w);
        }
      const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      l_run = l_run * alpha + rs;
      m_run = m_new;
      // P buffer j & 1 was read by P_{j-2} V_{j-2}; rescaling O needs P_{j-1} V_{j-1}
      // done.  Rows (and so `need`) are the same in both warps of the pair.
      const bool need = j > 0 && __any_sync(0xFFFFFFFFu, move);
      bool okw = true;
      if (j >= 2) okw = mbar_wait(&pv_done[j & 1], (static_cast<uint32_t>(j - 2) >> 1) & 1u, limit, abort_flag);
      if (need && okw)
        okw = mbar_wait(&pv_done[(j - 1) & 1], (static_cast<uint32_t>(j - 1) >> 1) & 1u, limit, abort_flag);
      ok = !bar_sync_or(1 + q, 64, !okw);
      if (!ok) break;
      tc_fence_after();
      if (need) {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(lane_base + kAtOCol + col0 + 32 * c, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st_32x32b_x32(lane_base + kAtOCol + col0 + 32 * c, ov);
        }
      }
      // this half of the P row: keys 64 half + 2c, 2c + 1 in column 32 half + c of
      // P buffer j & 1
      tmem_st_32x32b_x32(lane_base + kAtPCol + static_cast<uint32_t>(j & 1) * 64 + 32 * half, pk);
      tmem_st_wait();
      tc_fence_before();  // order the TMEM stores before the MMA thread's next products
      mbar_arrive(&p_ready[j & 1]);
    }
    if (!ok) *abort_flag = 1;
    // the row's total weight: both halves' sums
    if (active) {
      float* xl = xchg;  // the last block's reads finished before its closing pair barrier
      xl[half * 128 + r] = l_run;
      named_bar_sync(1 + q, 64);
      l_run += xl[(half ^ 1) * 128 + r];
    }
    // epilogue: O / l, rounded to bf16 (or the fp32 part of a key split)
    bool have_o = ok && nblk > 0 && active;
    if (have_o) {
      const uint64_t limit = p.timeout_ns + 20000ull * static_cast<uint64_t>(nblk + 1);
      have_o = mbar_wait(&pv_done[(nblk - 1) & 1], (static_cast<uint32_t>(nblk - 1) >> 1) & 1u, limit, abort_flag);
      have_o = !bar_sync_or(1 + q, 64, !have_o);
      if (!have_o) {
        if (!*abort_flag) record_error(p.err, kDevTimeoutTmemFull, nblk);
        *abort_flag = 1;
      }
      tc_fence_after();
    }
    grid_dependency_wait();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const bool store = active && i < p.Sq && !*abort_flag;
    if (p.n_splits > 1) {
      // normalised fp32 part and the log2-sum-exp of this split's scores
      const int64_t prw = (static_cast<int64_t>(split) * p.B * p.Sq + b * p.Sq + i) * p.H + h;
      if (store && half == 0) p.part_lse[prw] = l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY;
      float* po = p.part_o + prw * kAttnHeadDim + col0;
#pragma unroll 1
      for (int c = 0; c < 2 && active; ++c) {
        uint32_t ov[32];
        if (have_o) {
          tmem_ld_32x32b_x32(lane_base + kAtOCol + col0 + 32 * c, ov);
          tmem_ld_wait(ov);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (store) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<float4*>(po + 32 * c + 4 * g) =
                make_float4(__uint_as_float(ov[4 * g]) * inv, __uint_as_float(ov[4 * g + 1]) * inv,
                            __uint_as_float(ov[4 * g + 2]) * inv, __uint_as_float(ov[4 * g + 3]) * inv);
        }
      }
    } else {
      uint16_t* orow = p.O + static_cast<int64_t>(b * p.Sq + i) * p.ldo + h * kAttnHeadDim + col0;
#pragma unroll 1
      for (int c = 0; c < 2 && active; ++c) {
        uint32_t ov[32];
        if (have_o) {
          tmem_ld_32x32b_x32(lane_base + kAtOCol + col0 + 32 * c, ov);
          tmem_ld_wait(ov);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (store) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[8 * g + 0]) * inv, __uint_as_float(ov[8 * g + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[8 * g + 2]) * inv, __uint_as_float(ov[8 * g + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[8 * g + 4]) * inv, __uint_as_float(ov[8 * g + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[8 * g + 6]) * inv, __uint_as_float(ov[8 * g + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * g) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kAtTmemCols);
  }
}

// One warp per (output row, head): weights 2^(lse_s - max) over the splits
// (lane s holds split s), then each lane sums 4 of the 128 columns over the
// splits in split order and stores them as bf16.  A row no split saw is 0.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Sq * p.H;
  // The next launch may start its set-up (and its early L2 reads) at once: it
  // waits for this grid's completion before it touches memory.
  grid_launch_dependents();
  grid_dependency_wait();
  if (unit >= rows) return;
  const int64_t row = unit / p.H;  // b * Sq + i
  const int h = static_cast<int>(unit % p.H);
  const int64_t split_stride = rows;
  const float l = lane < p.n_splits ? p.part_lse[lane * split_stride + unit] : -INFINITY;
  float mx = l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  const float w = mx == -INFINITY ? 0.f : fast_exp2(l - mx);
  float tot = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
  // Eight splits' loads are issued together, then summed in split order (one
  // load per iteration would put n_splits memory latencies in a row).  A split
  // of zero weight (no visible key, or past n_splits: lanes there hold w = 0) is
  // not read: its part may be stale.
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp0 = 0; sp0 < p.n_splits; sp0 += 8) {
    float ws[8];
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sp = sp0 + u;  // < 32: n_splits <= 32
      ws[u] = __shfl_sync(0xFFFFFFFFu, w, sp);
      v[u] = (sp < p.n_splits && ws[u] != 0.f)
                 ? *reinterpret_cast<const float4*>(p.part_o + (sp * split_stride + unit) * kAttnHeadDim + 4 * lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc.x += ws[u] * v[u].x;
      acc.y += ws[u] * v[u].y;
      acc.z += ws[u] * v[u].z;
      acc.w += ws[u] * v[u].w;
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.O + row * p.ldo + h * kAttnHeadDim + 4 * lane) = out;
}

}  // namespace

cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Sq * p.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, p);
}

cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t grid = static_cast<int64_t>(p.q_tiles) * p.H * p.B * p.n_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kAtThreads, 1, 1);
  cfg.dynamicSmemBytes = kAtSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_fwd_kernel, tmQ, tmK, tmV, p);
}

}  // namespace sg

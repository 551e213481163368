// NVFP4 (W4A4) block-scaled GEMM on the 5th-generation tensor cores:
//
//   C[m][n] = alpha * sum_k  a[m][k] * sa[m][k / 16] * b[n][k] * sb[n][k / 16]
//
// with a, b packed E2M1 values (two per byte, element k in byte k / 2, the low
// nibble holding the even k), sa, sb E4M3 scales of 16-element blocks along K,
// fp32 accumulation and fp16 output, the dense W4A4 GEMM the gemm3 benchmarks page
// times ("Implementations": packed NVFP4 operands, E4M3 scales, 16-element blocks,
// alpha = 1, FP16 output).
//
// Roles (one CTA per SM, persistent over 128 x 256 tiles):
//   warp 0    TMA producer: per stage a 128-row box of A and a 256-row box of B
//             (128 bytes of K each, 128-byte swizzle) and the stage's scale atoms
//             (bulk copies of 512-byte blocks)
//   warp 1    TMEM allocator and MMA issuer: once a stage's operands have landed
//             and its scale columns are written, the four K = 64 block-scaled MMAs
//   warps 2-5 epilogue: each thread reads its accumulator row (two halves of 128
//             columns), releases the accumulator after the second, scales by
//             alpha, rounds to fp16 and stores straight from registers
//   warps 6-9 scale warps: per stage, the scale atoms from shared memory into
//             that stage's TMEM scale columns with tcgen05.st (each warp its lane
//             quarter).  Copying them with tcgen05.cp instead puts the copies in
//             the tensor pipe's queue between the MMAs: a 128 x 256 x 64 MMA
//             issued alone takes 128 cycles, and 200 with its three scale copies.
//             A stage's scale columns are rewritten only after its shared-memory
//             slot was refilled, so after the MMAs that read them completed.
//
// TMEM: the accumulator (256 columns) and per stage 16 columns of A scales and 32
// of B scales.  There is no room for a second 256-column accumulator, so the MMAs
// of the next tile wait only for the epilogue's TMEM reads, not for its stores.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sg_internal.h"
#include "sg_ptx.cuh"

namespace sg {
namespace {

constexpr int kF4Threads = 320;
constexpr int kF4EpiWarps = 4;
constexpr int kF4SfWarp0 = 2 + kF4EpiWarps;   // warps 6-9 write the scale columns
constexpr int kF4ABytes = kF4TileM * 128;                 // 16 KB
constexpr int kF4BBytes = kF4TileN * 128;                 // 32 KB
constexpr int kF4SfaBytes = 4 * kF4AtomBytes;             // 4 atoms (one per K = 64 chunk)
constexpr int kF4SfbBytes = 2 * 4 * kF4AtomBytes;         // 2 row blocks x 4 chunks
constexpr int kF4SfaOff = kF4ABytes + kF4BBytes;
constexpr int kF4SfbOff = kF4SfaOff + kF4SfaBytes;
constexpr int kF4StageBytes = kF4SfbOff + kF4SfbBytes;    // 54 KB, a multiple of 1024
constexpr int kF4BarOff = kF4Stages * kF4StageBytes;
constexpr int kF4MiscOff = kF4BarOff + (3 * kF4Stages + 3) * 8;
constexpr int kF4Smem = kF4MiscOff + 16 + 1024;            // + alignment slack
constexpr int kF4TmemCols = 512;
constexpr int kF4SfCols = 48;                              // per stage: 16 (A) + 32 (B)
static_assert(kF4StageBytes % 1024 == 0, "stage bases keep the 1024-byte swizzle alignment");
static_assert(kF4TileN + kF4Stages * kF4SfCols <= kF4TmemCols, "TMEM budget");
static_assert(kF4Smem <= 232448, "shared memory budget");

// Reads 128 accumulator columns of this thread's TMEM lane (`tacc`), scaled by
// alpha and rounded to fp16 pairs, in two halves; for the last columns of the
// tile (`last`), the warp releases the accumulator through `release` (called by
// lane 0) once they are read.
template <typename Release>
__device__ __forceinline__ void f4_read_acc(uint32_t tacc, float alpha, uint32_t (&hp)[64], bool last,
                                            Release release) {
#pragma unroll
  for (int j2 = 0; j2 < 2; ++j2) {
    uint32_t v0[32], v1[32];
    tmem_ld_32x32b_x32(tacc + 64 * j2, v0);
    tmem_ld_32x32b_x32(tacc + 64 * j2 + 32, v1);
    tmem_ld_wait(v0);
    tmem_ld_wait(v1);
    if (j2 == 1 && last) {
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) release();  // the accumulator may be overwritten now
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const __half2 x0 = __floats2half2_rn(alpha * __uint_as_float(v0[2 * e]), alpha * __uint_as_float(v0[2 * e + 1]));
      const __half2 x1 = __floats2half2_rn(alpha * __uint_as_float(v1[2 * e]), alpha * __uint_as_float(v1[2 * e + 1]));
      hp[32 * j2 + e] = *reinterpret_cast<const uint32_t*>(&x0);
      hp[32 * j2 + 16 + e] = *reinterpret_cast<const uint32_t*>(&x1);
    }
  }
}

// Stores 128 fp16 outputs (hp: column pairs) of one row from column col0,
// clipped at N.
__device__ __forceinline__ void f4_store_row(uint16_t* crow, int col0, int N, const uint32_t (&hp)[64]) {
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    const int c = col0 + 8 * g;
    if (c + 8 <= N) {
      *reinterpret_cast<uint4*>(crow + c) = make_uint4(hp[4 * g], hp[4 * g + 1], hp[4 * g + 2], hp[4 * g + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c + e < N) crow[c + e] = static_cast<uint16_t>(hp[4 * g + e / 2] >> (16 * (e & 1)));
    }
  }
}

// One stage's scale columns, written by the four scale warps (warp w writes the
// TMEM lanes of quarter w % 4), in the layout the block-scaled MMA reads: for
// K = 64 chunk kk, A scales at sfc + 4 kk and B scales (row blocks 0 and 1) at
// sfc + 16 + 8 kk and sfc + 20 + 8 kk, each 4 columns holding, in every lane
// quarter, the 16-byte row (lane % 32) of the chunk's scale atom (rows l, l + 32,
// l + 64, l + 96 of the 128-row block, 4 block scales each).  B row blocks that
// do not exist get zero scales.
__device__ __forceinline__ void f4_write_scales(const uint8_t* st_sfa, const uint8_t* st_sfb, uint32_t sfc_lane,
                                                bool rb0, bool rb1) {
  const int lane = threadIdx.x & 31;
  uint32_t a[16], bw[32];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint4 v = *reinterpret_cast<const uint4*>(st_sfa + kk * kF4AtomBytes + lane * 16);
    a[4 * kk] = v.x;
    a[4 * kk + 1] = v.y;
    a[4 * kk + 2] = v.z;
    a[4 * kk + 3] = v.w;
#pragma unroll
    for (int rb = 0; rb < 2; ++rb) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (rb == 0 ? rb0 : rb1) w = *reinterpret_cast<const uint4*>(st_sfb + (rb * 4 + kk) * kF4AtomBytes + lane * 16);
      bw[8 * kk + 4 * rb] = w.x;
      bw[8 * kk + 4 * rb + 1] = w.y;
      bw[8 * kk + 4 * rb + 2] = w.z;
      bw[8 * kk + 4 * rb + 3] = w.w;
    }
  }
  tmem_st_32x32b_x16(sfc_lane, a);
  tmem_st_32x32b_x32(sfc_lane + 16, bw);
  tmem_st_wait();
}

__global__ void __launch_bounds__(kF4Threads, 1)
    f4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const F4Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kF4BarOff);
  uint64_t* empty = full + kF4Stages;
  uint64_t* tmem_full = full + 2 * kF4Stages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* teardown = tmem_full + 2;
  uint64_t* sf_ready = tmem_full + 3;  // [kF4Stages]: the stage's scale columns written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kF4MiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kF4MiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Schedule& sched = p.sched;
  const int nitems = item_count(sched, static_cast<int>(blockIdx.x));
  const int k_stages = sched.k_steps;
  constexpr uint32_t kIdesc = idesc_nvf4_f32(kF4TileM, kF4TileN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kF4EpiWarps);
    mbar_init(teardown, 1);
    for (int s = 0; s < kF4Stages; ++s) mbar_init(&sf_ready[s], 4);  // one arrival per scale warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kF4TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Nothing above touched global memory: the next launch may start its set-up.
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < nitems && ok; ++i) {
        const WorkItem w = get_item(sched, static_cast<int>(blockIdx.x), i);
        int32_t tm, tn;
        tile_coords(sched, w.tile, tm, tn);
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const uint32_t s = it % kF4Stages;
          const uint32_t ph = (it / kF4Stages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutEmpty, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (it == 0) grid_dependency_wait();
          const int c0 = ks * 4;                      // first K = 64 chunk of the stage
          const int nch = min(4, p.kc - c0);          // chunks that hold data
          const uint32_t sf_bytes = static_cast<uint32_t>(nch * kF4AtomBytes);
          int nrb = 0;                                // B row blocks that exist
          for (int rb = 0; rb < 2; ++rb) nrb += (2 * tn + rb < p.rb_n) ? 1 : 0;
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(kF4ABytes + kF4BBytes) + (1u + nrb) * sf_bytes +
                                              (it == 0 ? p.inject_extra_tx : 0u));  // + failure injection only
          uint8_t* st = smem + s * kF4StageBytes;
          tma_load_2d(st, &tmA, ks * 128, tm * kF4TileM, &full[s]);
          tma_load_2d(st + kF4ABytes, &tmB, ks * 128, tn * kF4TileN, &full[s]);
          bulk_load(st + kF4SfaOff, p.SFA + (static_cast<int64_t>(tm) * p.kc + c0) * kF4AtomBytes, sf_bytes, &full[s]);
          for (int rb = 0; rb < 2; ++rb) {
            const int R = 2 * tn + rb;
            if (R < p.rb_n)
              bulk_load(st + kF4SfbOff + rb * 4 * kF4AtomBytes,
                        p.SFB + (static_cast<int64_t>(R) * p.kc + c0) * kF4AtomBytes, sf_bytes, &full[s]);
          }
        }
      }
      if (!ok) {
        // Unwinding: let the copies already issued land before the CTA exits.
        const uint32_t inflight = it < kF4Stages ? it : kF4Stages;
        for (uint32_t j = 0; j < inflight; ++j) {
          const uint32_t jt = it - 1 - j;
          volatile uint32_t never = 0;
          mbar_wait(&full[jt % kF4Stages], (jt / kF4Stages) & 1u, p.timeout_ns, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors of stage 0; a stage adds its byte offset >> 4, a K = 64 step
      // 32 bytes of the swizzle row (+2), an atom 512 bytes (+32).  Every address
      // stays below 256 KB, so the sums never carry out of the 14-bit field.
      const uint32_t base = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc_sw128(base);
      const uint64_t b_desc0 = smem_desc_sw128(base + kF4ABytes);
      constexpr uint64_t kStageUnits = kF4StageBytes >> 4;
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < nitems && ok; ++i) {
        if (!mbar_wait(tmem_empty, (static_cast<uint32_t>(i) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutTmemEmpty, i);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const uint32_t s = it % kF4Stages;
          const uint32_t ph = (it / kF4Stages) & 1u;
          if (!mbar_wait(&full[s], ph, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutFull, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (!mbar_wait(&sf_ready[s], ph, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutFull, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = s * kStageUnits;
          const uint32_t sfc = tmem_base + kF4TileN + s * kF4SfCols;
          // per K = 64 chunk one block-scaled MMA; the scale warps have written the
          // chunk's A scales at sfc + 4 kk and B scales at sfc + 16 + 8 kk
          auto chunk = [&](int kk) {
            tc_mma_nvf4(tmem_base, a_desc0 + so + 2 * kk, b_desc0 + so + 2 * kk, kIdesc, sfc + 4 * kk,
                        sfc + 16 + 8 * kk, (ks > 0 || kk > 0) ? 1u : 0u);
          };
          if (ks + 1 < k_stages || p.kc % 4 == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) chunk(kk);
          } else {
            const int nch = p.kc - ks * 4;  // the last stage's chunks that hold data
            for (int kk = 0; kk < nch; ++kk) chunk(kk);
          }
          tc_commit(&empty[s]);  // the slot (and its scale columns) are free once these MMAs are done
        }
        if (!ok) break;
        tc_commit(tmem_full);
      }
      if (!ok || *abort_flag) {
        // Unwinding: wait for every tcgen05 operation issued so far before TMEM is freed.
        tc_commit(teardown);
        volatile uint32_t never = 0;
        if (!mbar_wait(teardown, 0, p.timeout_ns, &never)) record_error(p.err, kDevTimeoutTeardown, 0);
      }
    }
  } else if (warp < kF4SfWarp0) {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    for (int i = 0; i < nitems; ++i) {
      const WorkItem w = get_item(sched, static_cast<int>(blockIdx.x), i);
      int32_t tm, tn;
      tile_coords(sched, w.tile, tm, tn);
      const uint64_t limit = p.timeout_ns + static_cast<uint64_t>(k_stages) * 20000ull;
      const bool ready = mbar_wait(tmem_full, static_cast<uint32_t>(i) & 1u, limit, abort_flag);
      if (!ready) {
        if (!*abort_flag) record_error(p.err, kDevTimeoutTmemFull, i);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = tm * kF4TileM + q * 32 + lane;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // accumulator columns [128 half, 128 half + 128)
        uint32_t hp[64];
        f4_read_acc(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + half * 128, p.alpha, hp, half == 1,
                    [&] { mbar_arrive(tmem_empty); });
        if (row < p.M) f4_store_row(p.C + static_cast<int64_t>(row) * p.ldc, tn * kF4TileN + half * 128, p.N, hp);
      }
    }
  } else {
    // ------------------------------------------------------------ scale warps
    const uint32_t sf_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kF4TileN;
    uint32_t it = 0;
    bool ok = true;
    for (int i = 0; i < nitems && ok; ++i) {
      const WorkItem w = get_item(sched, static_cast<int>(blockIdx.x), i);
      int32_t tm, tn;
      tile_coords(sched, w.tile, tm, tn);
      for (int ks = 0; ks < k_stages; ++ks, ++it) {
        const uint32_t s = it % kF4Stages;
        // the slot's copies landed (and, the producer having waited for the slot,
        // the MMAs that read its previous scale columns are done)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (it / kF4Stages) & 1u, p.timeout_ns, abort_flag));
        if (!ok) break;
        const uint8_t* st = smem + s * kF4StageBytes;
        f4_write_scales(st + kF4SfaOff, st + kF4SfbOff, sf_lane + s * kF4SfCols, 2 * tn < p.rb_n, 2 * tn + 1 < p.rb_n);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[s]);
      }
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF4TmemCols);
  }
}

// ------------------------------------------------------------------ CTA pairs
// The paired form: clusters of two CTAs on two SMs share a 256 x 256 output tile
// (tcgen05.mma.cta_group::2, M = 256).  Per stage each CTA loads its 128 rows of A
// and its 128 rows of B (128 bytes of K each; TMA loads that signal the leading
// CTA's full barrier) and the scale atoms of its A rows and of all 256 B rows
// (on its own barrier: its scale warps write them into its own TMEM, then arrive
// on the leader's barrier); the leader's MMA thread issues the MMAs for both.
// Against the one-CTA form this halves the B bytes and the MMA instructions per
// output, but not the scale columns each SM must hold (its A rows and all 256 B
// rows), and the cross-CTA hand-offs make it slower: 64.6 against 39.6 us at
// 4096^3.  It is kept as an explicit path (SG_PATH_GEMM_PAIR).
constexpr int kF4PStages = 5;
constexpr int kF4PABytes = 128 * 128;                        // 16 KB
constexpr int kF4PBBytes = 128 * 128;                        // 16 KB
constexpr int kF4PSfaOff = kF4PABytes + kF4PBBytes;
constexpr int kF4PSfbOff = kF4PSfaOff + 4 * kF4AtomBytes;    // 4 atoms of this CTA's A rows
constexpr int kF4PStageBytes = kF4PSfbOff + 8 * kF4AtomBytes; // + 2 row blocks x 4 atoms of B
constexpr int kF4PBarOff = kF4PStages * kF4PStageBytes;
constexpr int kF4PMiscOff = kF4PBarOff + (4 * kF4PStages + 3) * 8;
constexpr int kF4PSmem = kF4PMiscOff + 16 + 1024;
constexpr uint32_t kF4PStageTx = 2u * kF4PSfaOff;            // both CTAs' A and B bytes, on the leader's barrier
constexpr uint32_t kF4PSfTx = kF4PStageBytes - kF4PSfaOff;    // a CTA's scale atoms, on its own barrier
static_assert(kF4PStageBytes % 1024 == 0, "stage bases keep the 1024-byte swizzle alignment");
static_assert(kF4TileN + kF4PStages * kF4SfCols <= kF4TmemCols, "TMEM budget");
static_assert(kF4PSmem <= 232448, "shared memory budget");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kF4Threads, 1)
    f4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const F4Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kF4PBarOff);
  uint64_t* empty = full + kF4PStages;
  uint64_t* tmem_full = full + 2 * kF4PStages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* teardown = tmem_full + 2;
  uint64_t* sf_full = tmem_full + 3;                // [kF4PStages]: this CTA's scale atoms landed
  uint64_t* sf_ready = sf_full + kF4PStages;        // [kF4PStages] (leader): both CTAs' scale columns written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kF4PMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kF4PMiscOff + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: the pair's MMA issuer
  const int unit = static_cast<int>(blockIdx.x / 2);
  const Schedule& sched = p.sched;
  const int nitems = item_count(sched, unit);
  const int k_stages = sched.k_steps;
  constexpr uint32_t kIdesc = idesc_nvf4_f32(2 * kF4TileM, kF4TileN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4PStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * kF4EpiWarps);
    mbar_init(teardown, 1);
    for (int s = 0; s < kF4PStages; ++s) {
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], 2 * 4);  // one arrival per scale warp of each CTA
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSFA);
    tma_prefetch_desc(&tmSFB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kF4TmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < nitems && ok; ++i) {
        const WorkItem w = get_item(sched, unit, i);
        int32_t tm, tn;
        tile_coords(sched, w.tile, tm, tn);
        const int32_t arow = tm * 2 * kF4TileM + static_cast<int32_t>(rank) * kF4TileM;
        const int32_t brow = tn * kF4TileN + static_cast<int32_t>(rank) * (kF4TileN / 2);
        const int32_t ablk = 2 * tm + static_cast<int32_t>(rank);  // 128-row block of this CTA's A rows
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const uint32_t s = it % kF4PStages;
          const uint32_t ph = (it / kF4PStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutEmpty, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (it == 0) grid_dependency_wait();
          const uint32_t full_leader = mapa_shared(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], kF4PStageTx);
          uint8_t* st = smem + s * kF4PStageBytes;
          tma_load_2d_pair(st, &tmA, ks * 128, arow, full_leader);
          tma_load_2d_pair(st + kF4PABytes, &tmB, ks * 128, brow, full_leader);
          // scale atoms, viewed as rows of 256 bytes: atom (R, c) is rows
          // 2 (R kc + c) and 2 (R kc + c) + 1; a stage takes 4 atoms (8 rows)
          mbar_arrive_expect_tx(&sf_full[s], kF4PSfTx);
          tma_load_2d(st + kF4PSfaOff, &tmSFA, 0, 2 * (ablk * p.kc + 4 * ks), &sf_full[s]);
          for (int rb = 0; rb < 2; ++rb)
            tma_load_2d(st + kF4PSfbOff + rb * 4 * kF4AtomBytes, &tmSFB, 0, 2 * ((2 * tn + rb) * p.kc + 4 * ks),
                        &sf_full[s]);
        }
      }
      if (!ok) {
        // Unwinding: let the copies already issued arrive before the pair exits
        // (both CTAs' A and B bytes land on the leader's barriers, each CTA's scale
        // atoms on its own).
        const uint32_t inflight = it < kF4PStages ? it : kF4PStages;
        for (uint32_t j = 0; j < inflight; ++j) {
          const uint32_t jt = it - 1 - j;
          volatile uint32_t never = 0;
          if (rank == 0) mbar_wait(&full[jt % kF4PStages], (jt / kF4PStages) & 1u, p.timeout_ns, &never);
          mbar_wait(&sf_full[jt % kF4PStages], (jt / kF4PStages) & 1u, p.timeout_ns, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      const uint32_t base = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc_sw128(base);
      const uint64_t b_desc0 = smem_desc_sw128(base + kF4PABytes);
      constexpr uint64_t kStageUnits = kF4PStageBytes >> 4;
      uint32_t it = 0;
      bool ok = true;
      for (int i = 0; i < nitems && ok; ++i) {
        if (!mbar_wait(tmem_empty, (static_cast<uint32_t>(i) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutTmemEmpty, i);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const uint32_t s = it % kF4PStages;
          const uint32_t ph = (it / kF4PStages) & 1u;
          if (!mbar_wait(&full[s], ph, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutFull, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (!mbar_wait_cluster(&sf_ready[s], ph, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutFull, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = s * kStageUnits;
          const uint32_t sfc = tmem_base + kF4TileN + s * kF4SfCols;
          auto chunk = [&](int kk) {
            tc_mma_nvf4_pair(tmem_base, a_desc0 + so + 2 * kk, b_desc0 + so + 2 * kk, kIdesc, sfc + 4 * kk,
                             sfc + 16 + 8 * kk, (ks > 0 || kk > 0) ? 1u : 0u);
          };
          if (ks + 1 < k_stages || p.kc % 4 == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) chunk(kk);
          } else {
            const int nch = p.kc - ks * 4;  // the last stage's chunks that hold data
            for (int kk = 0; kk < nch; ++kk) chunk(kk);
          }
          tc_commit_pair_multicast(&empty[s], 0x3);  // the slot is free in both CTAs
        }
        if (!ok) break;
        tc_commit_pair_multicast(tmem_full, 0x3);  // the accumulator is complete in both CTAs
      }
      if (!ok || *abort_flag) {
        // Unwinding: wait for every tcgen05 operation issued so far before TMEM is freed.
        tc_commit_pair_multicast(teardown, 0x1);
        volatile uint32_t never = 0;
        if (!mbar_wait(teardown, 0, p.timeout_ns, &never)) record_error(p.err, kDevTimeoutTeardown, 0);
      }
    }
  } else if (warp < kF4SfWarp0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    grid_dependency_wait();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t tmem_empty_leader = mapa_shared(smem_u32(tmem_empty), 0);
    for (int i = 0; i < nitems; ++i) {
      const WorkItem w = get_item(sched, unit, i);
      int32_t tm, tn;
      tile_coords(sched, w.tile, tm, tn);
      const uint64_t limit = p.timeout_ns + static_cast<uint64_t>(k_stages) * 20000ull;
      const bool ready = mbar_wait(tmem_full, static_cast<uint32_t>(i) & 1u, limit, abort_flag);
      if (!ready) {
        if (!*abort_flag) record_error(p.err, kDevTimeoutTmemFull, i);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = tm * 2 * kF4TileM + static_cast<int>(rank) * kF4TileM + q * 32 + lane;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // accumulator columns [128 half, 128 half + 128)
        uint32_t hp[64];
        f4_read_acc(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + half * 128, p.alpha, hp, half == 1,
                    [&] { mbar_arrive_cluster(tmem_empty_leader); });
        if (row < p.M) f4_store_row(p.C + static_cast<int64_t>(row) * p.ldc, tn * kF4TileN + half * 128, p.N, hp);
      }
    }
  } else {
    // ------------------------------------------------------------ scale warps (both CTAs)
    const uint32_t sf_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kF4TileN;
    uint32_t it = 0;
    bool ok = true;
    for (int i = 0; i < nitems && ok; ++i) {
      const WorkItem w = get_item(sched, unit, i);
      int32_t tm, tn;
      tile_coords(sched, w.tile, tm, tn);
      for (int ks = 0; ks < k_stages; ++ks, ++it) {
        const uint32_t s = it % kF4PStages;
        // this CTA's scale atoms landed (the producer refilled the slot only after
        // the MMAs that read its previous scale columns completed)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sf_full[s], (it / kF4PStages) & 1u, p.timeout_ns, abort_flag));
        if (!ok) break;
        const uint8_t* st = smem + s * kF4PStageBytes;
        f4_write_scales(st + kF4PSfaOff, st + kF4PSfbOff, sf_lane + s * kF4SfCols, 2 * tn < p.rb_n,
                        2 * tn + 1 < p.rb_n);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sf_ready[s]), 0));
      }
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kF4TmemCols);
  }
}

// One thread per atom byte: atom (R, c), byte o -> row R * 128 + (o / 16) + 32 * ((o % 16) / 4),
// block 4 c + o % 4.
__global__ void f4_pack_scales_kernel(const uint8_t* __restrict__ plain, int64_t rows, int64_t nblk, int64_t ld,
                                      int64_t kc, int64_t total, uint8_t* __restrict__ atoms) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t atom = i / kF4AtomBytes;
  const int o = static_cast<int>(i % kF4AtomBytes);
  const int64_t R = atom / kc, c = atom % kc;
  const int64_t r = R * 128 + o / 16 + 32 * ((o % 16) / 4);
  const int64_t blk = 4 * c + o % 4;
  atoms[i] = (r < rows && blk < nblk) ? plain[r * ld + blk] : 0;
}

}  // namespace

cudaError_t launch_f4_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const F4Params& p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(f4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF4Smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.sched.grid, 1, 1);
  cfg.blockDim = dim3(kF4Threads, 1, 1);
  cfg.dynamicSmemBytes = kF4Smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f4_gemm_kernel, tmA, tmB, p);
}

cudaError_t launch_f4_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                               const CUtensorMap& tmSFB, const F4Params& p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(f4_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF4PSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.sched.grid, 1, 1);
  cfg.blockDim = dim3(kF4Threads, 1, 1);
  cfg.dynamicSmemBytes = kF4PSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f4_gemm_pair_kernel, tmA, tmB, tmSFA, tmSFB, p);
}

cudaError_t launch_f4_pack_scales(const uint8_t* plain, int64_t rows, int64_t K, int64_t ld, uint8_t* atoms,
                                  cudaStream_t stream) {
  const int64_t kc = (K + 63) / 64;
  const int64_t total = ((rows + 127) / 128) * kc * kF4AtomBytes;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  f4_pack_scales_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(
      plain, rows, K / 16, ld, kc, total, atoms);
  return cudaGetLastError();
}

}  // namespace sg

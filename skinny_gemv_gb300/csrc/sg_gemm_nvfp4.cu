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
//   warp 1    TMEM allocator and MMA issuer: copies the stage's scale atoms into
//             that stage's TMEM scale columns (tcgen05.cp), then issues the four
//             K = 64 block-scaled MMAs; a stage's scale columns are rewritten only
//             after its shared-memory slot was refilled, so after the MMAs that
//             read them completed
//   warps 2-9 epilogue: each reads 32 rows x 128 columns of the accumulator into
//             registers, releases the accumulator, then scales by alpha, rounds
//             to fp16 and stores straight from registers
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
constexpr int kF4EpiWarps = 8;
constexpr int kF4ABytes = kF4TileM * 128;                 // 16 KB
constexpr int kF4BBytes = kF4TileN * 128;                 // 32 KB
constexpr int kF4SfaBytes = 4 * kF4AtomBytes;             // 4 atoms (one per K = 64 chunk)
constexpr int kF4SfbBytes = 2 * 4 * kF4AtomBytes;         // 2 row blocks x 4 chunks
constexpr int kF4SfaOff = kF4ABytes + kF4BBytes;
constexpr int kF4SfbOff = kF4SfaOff + kF4SfaBytes;
constexpr int kF4StageBytes = kF4SfbOff + kF4SfbBytes;    // 54 KB, a multiple of 1024
constexpr int kF4BarOff = kF4Stages * kF4StageBytes;
constexpr int kF4MiscOff = kF4BarOff + (2 * kF4Stages + 3) * 8;
constexpr int kF4Smem = kF4MiscOff + 16 + 1024;            // + alignment slack
constexpr int kF4TmemCols = 512;
constexpr int kF4SfCols = 48;                              // per stage: 16 (A) + 32 (B)
static_assert(kF4StageBytes % 1024 == 0, "stage bases keep the 1024-byte swizzle alignment");
static_assert(kF4TileN + kF4Stages * kF4SfCols <= kF4TmemCols, "TMEM budget");
static_assert(kF4Smem <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kF4Threads, 1)
    f4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const F4Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kF4BarOff);
  uint64_t* empty = full + kF4Stages;
  uint64_t* tmem_full = full + 2 * kF4Stages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* teardown = tmem_full + 2;
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
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(kF4ABytes + kF4BBytes) + (1u + nrb) * sf_bytes);
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
      const uint64_t sfa_desc0 = smem_desc_rows16(base + kF4SfaOff);
      const uint64_t sfb_desc0 = smem_desc_rows16(base + kF4SfbOff);
      constexpr uint64_t kStageUnits = kF4StageBytes >> 4;
      constexpr uint64_t kAtomUnits = kF4AtomBytes >> 4;
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
          tc_fence_after();
          const uint64_t so = s * kStageUnits;
          const uint32_t sfc = tmem_base + kF4TileN + s * kF4SfCols;
          // per K = 64 chunk: its A scales, the B scales of both row blocks, then
          // the MMA (a copy is ordered before a later MMA of the same thread)
          auto chunk = [&](int kk) {
            tc_cp_32x128b_warpx4(sfc + 4 * kk, sfa_desc0 + so + kk * kAtomUnits);
            tc_cp_32x128b_warpx4(sfc + 16 + 8 * kk, sfb_desc0 + so + kk * kAtomUnits);
            tc_cp_32x128b_warpx4(sfc + 20 + 8 * kk, sfb_desc0 + so + (4 + kk) * kAtomUnits);
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
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;  // accumulator columns [128 half, 128 half + 128)
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
      uint32_t v[4][32];
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + half * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(tacc + j * 32, v[j]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);  // the accumulator may be overwritten now
      const int row = tm * kF4TileM + q * 32 + lane;
      if (row < p.M) {
        uint16_t* crow = p.C + static_cast<int64_t>(row) * p.ldc;
        const int col0 = tn * kF4TileN + half * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int c = col0 + 32 * j + 8 * g;
            uint32_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 x = __floats2half2_rn(p.alpha * __uint_as_float(v[j][8 * g + 2 * e]),
                                                  p.alpha * __uint_as_float(v[j][8 * g + 2 * e + 1]));
              h[e] = *reinterpret_cast<const uint32_t*>(&x);
            }
            if (c + 8 <= p.N) {
              *reinterpret_cast<uint4*>(crow + c) = make_uint4(h[0], h[1], h[2], h[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (c + e < p.N) crow[c + e] = static_cast<uint16_t>(h[e / 2] >> (16 * (e & 1)));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF4TmemCols);
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

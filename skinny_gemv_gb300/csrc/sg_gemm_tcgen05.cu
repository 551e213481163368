// Persistent tcgen05 GEMM for sm_103a: C[M,N] = A[M,K] . B[N,K]^T, bf16 in,
// fp32 accumulate in tensor memory, bf16 out.
//
// One CTA per SM (two on the swapped variant), warps with fixed roles:
//   warp 0     TMA producer: per k-step waits for a free ring stage, arms its
//              `full` barrier with the stage's byte count and issues two tiled
//              cp.async.bulk.tensor loads (A box 64 x 128, B box 64 x BN, 128-byte
//              swizzle, zero fill outside the matrices);
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma
//              (128 x BN x 16 per instruction, 4 per stage) and commits each stage
//              back to its `empty` barrier and each finished accumulator to
//              `tmem_full`;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, Stream-K partials,
//              fp32 -> bf16 (round to nearest even), 64-byte-swizzled staging and
//              TMA stores (clipped at M and N), then release the accumulator;
//   warps 6-7  (GEMM variants) sum the fp32 partials of Stream-K tiles that this
//              CTA finishes in the middle of its schedule.  A CTA's last item is
//              summed by the epilogue warps from the idle copy ring instead.
// Two accumulators (2 x BN TMEM columns) let the epilogue of one tile overlap the
// main loop of the next.  The single-CTA GEMM comes with BN = 256 or, for GEMMs
// whose 128 x 128 tiles fit in one wave, BN = 128; below one wave K may be split
// into equal pieces, one per CTA (split mode of the schedule).
//
// This is spark-kernels' variant 5 ("the copies were the problem, not the power":
// a producer warp with cp.async.bulk.tensor boxes, 128-byte swizzle, a full and an
// empty barrier per stage, no block-wide barrier in the k-loop) on the Stream-K
// schedule of variant 4 ("stream-k proper"), with the sm_100-class tensor cores:
// operands go TMA -> shared memory -> tcgen05.mma without a trip through
// registers, and the accumulator lives in tensor memory instead of registers.
//
// The paired variant (PAIR = true) runs on clusters of two CTAs on two SMs: one
// 256 x 256 output tile per pair, each CTA loading its 128 rows of A and 128 rows
// of B (32 KB per stage, 6 stages) and holding its 128 x 256 half of the
// accumulator; the even CTA issues tcgen05.mma.cta_group::2 for both.  Per SM this
// moves 2/3 of the bytes of the 128 x 256 single-CTA tile for the same FLOPs.
//
// The swapped variant (SWAP = true) serves the skinny path: the weights B take
// the MMA's M side (64- or 128-row tiles) and the few activation rows of A its N
// side (16, 32 or 64), so every weight byte is loaded once for all rows; its
// epilogue writes C[m, n] = D[n, m] into a shared-memory tile in C's layout and
// stores it with one TMA store.
#include <cuda_bf16.h>

#include "sg_internal.h"
#include "sg_ptx.cuh"
#include "sg_sched.cuh"

namespace sg {
namespace {

// KSUB: consecutive 64-wide k boxes per pipeline stage (one schedule k-step).
// PAIR: B's rows are split between the two CTAs of a pair (BN / 2 each).
// SWAP_ROWS: 0 for the GEMM, else the swapped variant's weight rows per tile.
// GATED: gate and up weights (see the kernel); the swapped variant keeps two
// accumulators side by side in TMEM, gate in columns [0, BN), up in [BN, 2 BN).
template <int BN, int STAGES, int SWAP_ROWS, int KSUB, bool PAIR, bool GATED = false>
struct TcLayout {
  static constexpr bool SWAP = SWAP_ROWS > 0;
  static constexpr int kAMats = (SWAP && GATED) ? 2 : 1;      // A-side boxes per k box
  static constexpr int kAccCols = (SWAP && GATED) ? 2 * BN : BN;  // TMEM columns per accumulator
  // rows of the MMA's A operand per CTA: 128, or 64 / 128 weight rows on the
  // swapped path (an M = 64 accumulator sits in lanes 0-15 of each TMEM lane quarter)
  static constexpr int kARows = SWAP ? SWAP_ROWS : kBM;
  static constexpr int kBRowsPerCta = PAIR ? BN / 2 : BN;
  static constexpr int kASub = kARows * kBK * 2;  // one kARows x 64 box
  static constexpr int kBSub = kBRowsPerCta * kBK * 2;
  static constexpr int kABytes = KSUB * kAMats * kASub;
  static constexpr int kBBytes = KSUB * kBSub;
  // epilogue warps: one per TMEM lane quarter (eight, two per quarter, measured
  // no faster and would cap registers at 168)
  static constexpr int kEpiWarps = 4;
  // GEMM variants: two more warps sum the fp32 partials of Stream-K tiles, so a
  // tile finished in the middle of a CTA's schedule does not hold up the
  // epilogue of the tiles after it (the skinny variant's split pieces end the
  // CTA's schedule and are summed from the idle copy ring instead).
  static constexpr int kFixupWarps = SWAP ? 0 : 2;
  static constexpr int kMaxJobs = kFixupMaxJobs;  // Stream-K pieces per CTA the fixup warps take
  static constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kFixupWarps;
  static constexpr int kColsPerEpiWarp = BN / (kEpiWarps / 4);
  static constexpr int kStagingBufBytes = 32 * 64;  // 32 rows x 32 bf16
  static constexpr int kStagingBufs = 2;            // per epilogue warp
  static constexpr int kAOff = 0;
  static constexpr int kBOff = STAGES * kABytes;
  static constexpr int kStagingOff = kBOff + STAGES * kBBytes;
  // swapped path: one C tile (BN activation rows x kARows weight rows, bf16)
  static constexpr int kStagingBytes = SWAP ? BN * kARows * 2 : kEpiWarps * kStagingBufs * kStagingBufBytes;
  // columns of a Stream-K partial (all of an accumulator's columns)
  static constexpr int kSlotCols = kAccCols;
  static constexpr int kFixStagingOff = kStagingOff + kStagingBytes;
  static constexpr int kFixStagingBytes = kFixupWarps * kStagingBufs * kStagingBufBytes;
  static constexpr int kBarOff = kFixStagingOff + kFixStagingBytes;
  // full[S], empty[S], tmem_full[2], tmem_empty[2], teardown, fixup, job[kMaxJobs]
  static constexpr int kNumBars = 2 * STAGES + 6 + kMaxJobs + 1;  // + the residual tile's load
  static constexpr int kRingBytes = STAGES * (kABytes + kBBytes);
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort, sk flag
  static constexpr int kJobOff = kMiscOff + 16;            // kMaxJobs x {tm, tn, last, -}
  static constexpr int kBytes = kJobOff + kMaxJobs * 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
  static constexpr uint32_t kTmemCols = (2 * kAccCols < 32) ? 32u : static_cast<uint32_t>(2 * kAccCols);
  static constexpr int kChunk = SWAP ? 16 : 32;  // accumulator columns per tcgen05.ld
  // accumulator rows a Stream-K partial holds (an M = 64 accumulator has 64)
  static constexpr int kSlotRows = kARows;
  // CTAs per SM the launch bounds ask for: two when both fit in shared memory
  static constexpr int kMinBlocks = (kAlloc + 1024) * 2 <= 228 * 1024 ? 2 : 1;
  // epilogue arrivals that free an accumulator: 4 warps, of both CTAs when paired
  static constexpr uint32_t kTmemEmptyCount = PAIR ? 2 * kEpiWarps : kEpiWarps;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  static_assert(kFixupWarps == 0 || (kChunk == 32 && kStagingBufs == 2 && kStagingBufBytes == 32 * 64 &&
                                     kFixupWarps * 64 == kBM),
                "fixup warps: 64 rows each, 32-column chunks, two 2 KB store buffers");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM columns");
  static_assert(!(PAIR && SWAP), "the paired variant is the non-swapped GEMM");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<uint32_t*>(&v);
}

// SwiGLU of one output: silu(g) * u = g / (1 + e^-g) * u in fp32; for g far
// below zero e^-g is inf and the result the correct limit, a signed zero.
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Adds the residual R[row, col0 .. col0 + 31] to this thread's 32 values (only
// elements with row < M and column < N are read; 16-byte vectors where all eight
// are inside, single elements at the row's ragged end).  R may be C itself: each
// element is read before the same thread's store writes it.
__device__ __forceinline__ void add_residual_32(float* v, const uint16_t* R, int64_t ldr, int row, int col0, int M,
                                                int N) {
  if (row >= M) return;
  const uint16_t* src = R + static_cast<int64_t>(row) * ldr + col0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (col0 + 8 * c + 8 <= N) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + 8 * c);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * c + 2 * i] += __uint_as_float(w[i] << 16);
        v[8 * c + 2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (col0 + 8 * c + e < N) v[8 * c + e] += __uint_as_float(static_cast<uint32_t>(src[8 * c + e]) << 16);
    }
  }
}

// One warp writes 32 rows x 32 fp32 columns (lane = row) to C as bf16 (round to
// nearest even): 64-byte-swizzled staging in one of two 2 KB buffers, then a TMA
// store clipped at M and N.  With `own` set, the chunk goes through that 2 KB
// buffer instead, one that no earlier store of the warp uses, so nothing is waited for.
__device__ __forceinline__ void store_rows_32x32(const CUtensorMap* tmC, const float* v, int col0, int row0,
                                                 uint8_t* staging, uint32_t& count, int lane, int M, int N,
                                                 uint8_t* own = nullptr) {
  constexpr int kBuf = 32 * 64;
  const uint32_t buf = count & 1u;
  if (own == nullptr) {
    if (lane == 0) bulk_wait_group_read<1>();  // buffer `buf` no longer read by TMA
    __syncwarp();
  }
  uint8_t* const dst = own != nullptr ? own : staging + buf * kBuf;
  const uint32_t base = smem_u32(dst) + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t phys = static_cast<uint32_t>(c) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u);
    st_shared_v4(base + phys * 16, pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                 pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (row0 < M && col0 < N) tma_store_2d_hint(tmC, dst, col0, row0, policy_evict_first());
    bulk_commit_group();
  }
  ++count;
}

// GATED: C = silu(A . G^T) * (A . U^T) with tmW2 mapping the up weights U.  GEMM:
// the B tile is BN / 2 rows of G (tmB) over BN / 2 rows of U for the same output
// columns, and the epilogue writes BN / 2 columns per tile.  Swapped: each k box
// holds a weight box of G (tmA) and one of U, two MMAs fill a gate and an up
// accumulator, and each thread combines its row's two.
template <int BN, int STAGES, int SWAP_ROWS, int KSUB, bool PAIR, bool GATED>
__global__ void __launch_bounds__(TcLayout<BN, STAGES, SWAP_ROWS, KSUB, PAIR, GATED>::kThreads,
                                  TcLayout<BN, STAGES, SWAP_ROWS, KSUB, PAIR, GATED>::kMinBlocks)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW2,
                   const TcParams p, const __grid_constant__ TcBatchMaps bmaps) {
  using L = TcLayout<BN, STAGES, SWAP_ROWS, KSUB, PAIR, GATED>;
  constexpr bool SWAP = L::SWAP;
  // output columns per tile
  constexpr int kOutCols = (GATED && !SWAP) ? BN / 2 : BN;
  // A batched swapped launch: weight tile tm is tile tm - tile_begin[i] of matrix i.
  auto batch_of = [&](int tm) {
    int i = 0;
    while (i + 1 < p.nbatch && tm >= p.tile_begin[i + 1]) ++i;
    return i;
  };
  // Gated accumulators alternate blocks of kHalf gate columns and kHalf up
  // columns: one block each on the swapped path and in a single-CTA tile, and
  // per CTA of a pair (each CTA's B rows are 64 gate over 64 up rows).
  constexpr int kHalf = SWAP ? BN : (PAIR ? 64 : 128);
  // accumulator column of the gate value of output column c (up: + kHalf)
  auto gate_col = [](int c) { return (c / kHalf) * 2 * kHalf + c % kHalf; };
  constexpr int kTileRows = PAIR ? 2 * kBM : L::kARows;  // output rows per tile (the MMA's M)
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileRows, BN);
  const int kboxes = (p.K + kBK - 1) / kBK;  // 64-wide k boxes that hold data

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tmem_full = bars + 2 * STAGES;
  uint64_t* tmem_empty = bars + 2 * STAGES + 2;
  uint64_t* teardown = bars + 2 * STAGES + 4;
  uint64_t* fixup_bar = bars + 2 * STAGES + 5;  // bulk loads of Stream-K partials
  uint64_t* job_bar = bars + 2 * STAGES + 6;    // Stream-K piece j handed to the fixup warps
  uint64_t* resid_bar = job_bar + L::kMaxJobs;  // swapped path: the residual tile's TMA load
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 4);
  volatile uint32_t* sk_last = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 8);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Schedule& sched = p.sched;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 = the pair's MMA issuer
  const int unit = PAIR ? static_cast<int>(blockIdx.x / 2) : static_cast<int>(blockIdx.x);
  const int nitems = item_count(sched, unit);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], L::kTmemEmptyCount);
    }
    mbar_init(teardown, 1);
    mbar_init(fixup_bar, 1);
    for (int j = 0; j < L::kMaxJobs; ++j) mbar_init(&job_bar[j], 1);
    mbar_init(resid_bar, 1);
    *abort_flag = 0;
    *sk_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, L::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, L::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above touched no global memory, so it may overlap the previous
  // kernel's tail.  Each role waits for the previous kernel before its first
  // global access (and before any bounded wait starts its clock); the producer
  // first works out its first copy, so only the copy itself waits.  The GEMM
  // lets the next launch start its set-up at once; the swapped kernel, which
  // streams weights at the memory system's limit, only once its producer has
  // issued its last copy, so the next launch's early weight reads fill its tail
  // instead of competing with its stream.
  if constexpr (!SWAP) grid_launch_dependents();

  // Swapped path with a residual, one tile per CTA: the producer fetches the
  // tile's residual values at the start instead of the epilogue at the end.
  const bool resid_early = SWAP && !PAIR && !GATED && p.R != nullptr && sched.split > 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (SWAP && nitems > 0 && p.prewait_steps > 0) {
        // Before the wait for the previous launch (whose tail this CTA may
        // overlap), the first weight boxes are pulled into L2; the ring's loads
        // then find them there.
        const WorkItem w = get_item(sched, unit, 0);
        int32_t tm, tn;
        tile_coords(sched, w.tile, tm, tn);
        int arow = tm * kTileRows;
        const CUtensorMap* wmap = &tmA;
        if (p.nbatch > 0) {
          const int bi = batch_of(tm);
          wmap = &bmaps.w[bi];
          arow = (tm - p.tile_begin[bi]) * L::kARows;
        }
        const int kend = min(w.k1, w.k0 + p.prewait_steps);
        for (int ks = w.k0; ks < kend; ++ks) {
          const int nsub = min(KSUB, kboxes - ks * KSUB);
          for (int j = 0; j < nsub; ++j) {
            tma_prefetch_l2_2d(wmap, (ks * KSUB + j) * kBK, arow);
            if constexpr (GATED) tma_prefetch_l2_2d(&tmW2, (ks * KSUB + j) * kBK, arow);
          }
        }
      }
      uint32_t it = 0;
      bool ok = true;
      // GEMM operands are read by many tiles: their L2 lines are marked to be
      // evicted last (the output and the partial sums go first).  Measured:
      // 8192^3 615 -> 582 us, DRAM traffic at 4096^3 166.6 -> 153.9 MB per launch.
      const uint64_t keep = policy_evict_last();
      for (int i = 0; i < nitems && ok; ++i) {
        const WorkItem w = get_item(sched, unit, i);
        int32_t tm, tn;
        tile_coords(sched, w.tile, tm, tn);
        int arow = tm * kTileRows + static_cast<int>(rank) * L::kARows;
        const CUtensorMap* wmap = &tmA;
        if (SWAP && p.nbatch > 0) {
          const int bi = batch_of(tm);
          wmap = &bmaps.w[bi];
          arow = (tm - p.tile_begin[bi]) * L::kARows;
        }
        const int brow = tn * kOutCols + static_cast<int>(rank) * (GATED ? L::kBRowsPerCta / 2 : L::kBRowsPerCta);
        for (int ks = w.k0; ks < w.k1; ++ks, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutEmpty, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const int nsub = min(KSUB, kboxes - ks * KSUB);  // boxes past K are skipped
          uint32_t bytes = static_cast<uint32_t>(nsub * (L::kAMats * L::kASub + L::kBSub));
          const uint32_t extra = (it == 0) ? p.inject_extra_tx : 0u;  // failure injection only
          if (it == 0) grid_dependency_wait();
          if constexpr (PAIR) {
            // the leader's full barrier counts both CTAs' bytes
            const uint32_t full_leader = mapa_shared(smem_u32(&full[s]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * bytes + extra);
            for (int j = 0; j < nsub; ++j) {
              const int kx = (ks * KSUB + j) * kBK;
              uint8_t* bdst = smem + L::kBOff + s * L::kBBytes + j * L::kBSub;
              tma_load_2d_pair_hint(smem + L::kAOff + s * L::kABytes + j * L::kASub, &tmA, kx, arow, full_leader,
                                    keep);
              tma_load_2d_pair_hint(bdst, &tmB, kx, brow, full_leader, keep);
              if constexpr (GATED) tma_load_2d_pair_hint(bdst + L::kBSub / 2, &tmW2, kx, brow, full_leader, keep);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], bytes + extra);
            for (int j = 0; j < nsub; ++j) {
              const int kx = (ks * KSUB + j) * kBK;
              uint8_t* bdst = smem + L::kBOff + s * L::kBBytes + j * L::kBSub;
              uint8_t* adst = smem + L::kAOff + s * L::kABytes + j * L::kAMats * L::kASub;
              if constexpr (SWAP) {
                tma_load_2d(adst, wmap, kx, arow, &full[s]);
                if constexpr (GATED) tma_load_2d(adst + L::kASub, &tmW2, kx, arow, &full[s]);
                tma_load_2d(bdst, &tmB, kx, brow, &full[s]);
              } else {
                tma_load_2d_hint(adst, wmap, kx, arow, &full[s], keep);
                tma_load_2d_hint(bdst, &tmB, kx, brow, &full[s], keep);
                // gated: gate rows over up rows of the same output columns
                if constexpr (GATED) tma_load_2d_hint(bdst + L::kBSub / 2, &tmW2, kx, brow, &full[s], keep);
              }
            }
            if (SWAP && !GATED && it == 0 && resid_early) {
              // One tile per CTA: the residual tile goes into the store staging
              // right behind the first weight stage.
              mbar_arrive_expect_tx(resid_bar, static_cast<uint32_t>(BN * L::kARows * 2));
              tma_load_2d(smem + L::kStagingOff, &tmW2, tm * L::kARows, tn * BN, resid_bar);
            }
          }
        }
      }
      if constexpr (SWAP) grid_launch_dependents();
      if (resid_early && it > 0) {
        // The residual load lands before the CTA exits, whether or not this CTA
        // finishes the tile.
        volatile uint32_t never = 0;
        mbar_wait(resid_bar, 0, p.timeout_ns, &never);
      }
      if (!ok && rank == 0) {
        // Unwinding: let the loads already issued land before the CTA exits.
        const uint32_t inflight = it < STAGES ? it : STAGES;
        for (uint32_t j = 0; j < inflight; ++j) {
          const uint32_t jt = it - 1 - j;
          volatile uint32_t never = 0;
          mbar_wait(&full[jt % STAGES], (jt / STAGES) & 1u, p.timeout_ns, &never);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // This thread's loop sets the pace of the tensor pipe: per k-step it waits
    // for the stage, issues the MMAs and commits, and whatever else it does per
    // step adds to the step's time (measured: one extra global store per step cost
    // ~40 of ~560 cycles).  So the items' k-ranges are decoded before the wait
    // for the previous launch, the descriptors are advanced by additions, and, in
    // the GEMM, the next stage's barrier is tested while this step's last MMA is
    // queued.  (The swapped kernel waits on its weight stream instead; there the
    // test measured 4% slower at M = 64.)
    const KRanges kr(sched, unit);
    grid_dependency_wait();
    if (lane == 0 && rank == 0) {
      uint32_t s = 0, ph = 0;  // ring stage and the parity of its current phase
      bool ok = true;
      bool ready = false;      // the next stage's full barrier was seen complete
      // Descriptors of stage 0's first A and B boxes.  A byte offset d moves the
      // address field by d / 16, without carry: shared memory ends below 256 KB.
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + L::kAOff));
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + L::kBOff));
      for (int i = 0; i < nitems && ok; ++i) {
        int32_t k0, k1;
        kr.range(i, k0, k1);
        const uint32_t b = static_cast<uint32_t>(i) & 1u;
        const uint32_t use = static_cast<uint32_t>(i) >> 1;
        if (!mbar_wait(&tmem_empty[b], (use & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) record_error(p.err, kDevTimeoutTmemEmpty, i);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * L::kAccCols;
        uint32_t acc = 0u;  // the item's first MMA overwrites the accumulator
        for (int ks = k0; ks < k1; ++ks) {
          if (!ready && !mbar_wait(&full[s], ph, p.timeout_ns, abort_flag)) {
            if (!*abort_flag) record_error(p.err, kDevTimeoutFull, s);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ready = false;
          tc_fence_after();
          const uint32_t s_next = (s + 1 == STAGES) ? 0u : s + 1;
          const uint32_t ph_next = (s + 1 == STAGES) ? ph ^ 1u : ph;
          const int nsub = min(KSUB, kboxes - ks * KSUB);
          const uint64_t a_st = a_desc0 + s * static_cast<uint32_t>(L::kABytes / 16);
          const uint64_t b_st = b_desc0 + s * static_cast<uint32_t>(L::kBBytes / 16);
          for (int j = 0; j < nsub; ++j) {
            const uint64_t ad = a_st + static_cast<uint32_t>(j * (L::kAMats * L::kASub / 16));
            const uint64_t bd = b_st + static_cast<uint32_t>(j * (L::kBSub / 16));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              if (!SWAP && kk == kBK / 16 - 1 && j == nsub - 1 && ks + 1 < k1)
                ready = mbar_test_wait(&full[s_next], ph_next);
              // +32 bytes (2 in the address field) per 16 bf16 of K inside the 128-byte swizzle row
              if constexpr (PAIR) {
                tc_mma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, kIdesc, acc);
              } else {
                tc_mma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, kIdesc, acc);
                if constexpr (SWAP && GATED)  // the up weights into the up accumulator
                  tc_mma_bf16(d_tmem + BN, ad + L::kASub / 16 + 2 * kk, bd + 2 * kk, kIdesc, acc);
              }
              acc = 1u;
            }
          }
          // the stage is free (in both CTAs) once these MMAs have read it
          if constexpr (PAIR)
            tc_commit_pair_multicast(&empty[s], 0x3);
          else
            tc_commit(&empty[s]);
          s = s_next;
          ph = ph_next;
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair_multicast(&tmem_full[b], 0x3);  // accumulator b complete in both CTAs
        else
          tc_commit(&tmem_full[b]);
      }
      if (!ok || *abort_flag) {
        // Unwinding: wait for every MMA issued so far before TMEM is freed.
        if constexpr (PAIR)
          tc_commit_pair_multicast(teardown, 0x1);
        else
          tc_commit(teardown);
        volatile uint32_t never = 0;
        if (!mbar_wait(teardown, 0, p.timeout_ns, &never)) record_error(p.err, kDevTimeoutTeardown, 0);
      }
    }
  } else if (warp < 2 + L::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int ew = warp - 2;                      // epilogue warp index
    const int chunk_lo = (ew / 4) * (L::kColsPerEpiWarp / L::kChunk);  // this warp's columns
    const int chunk_hi = chunk_lo + L::kColsPerEpiWarp / L::kChunk;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int epi_tid = threadIdx.x - 64;  // 0 .. 32 * kEpiWarps - 1
    uint32_t store_count = 0;
    uint8_t* staging = smem + L::kStagingOff + ew * L::kStagingBufs * L::kStagingBufBytes;
    // the accumulator-free barrier lives in the pair's MMA-issuing CTA
    const uint32_t tmem_empty_addr0 = PAIR ? mapa_shared(smem_u32(&tmem_empty[0]), 0) : smem_u32(&tmem_empty[0]);
    // The threads that hold accumulator rows and the row each holds: an M = 64
    // accumulator has its rows in lanes 0-15 of each lane quarter.
    const bool holds_row = !SWAP || L::kARows == kBM || lane < 16;
    const int slot_row = (SWAP && L::kARows != kBM) ? q * 16 + lane : row;
    constexpr int kEpiThreads = 32 * L::kEpiWarps;
    // Swapped path with a residual: tmW2 maps R like C, and begin_tile loads the
    // tile's R values into the staging tile, which the chunks then add to and
    // overwrite with their outputs.
    const bool swap_resid = SWAP && !GATED && p.R != nullptr;

    // The CTA's last item, when a whole tile: its MMAs have read the copy ring
    // for the last time, so each chunk is staged in a 2 KB buffer of its own
    // carved from the ring (kOutCols / 32 per warp), and the stores of the
    // launch's tail do not wait for one another.
    uint8_t* last_staging = nullptr;
    static_assert(SWAP || L::kEpiWarps * (kOutCols / 32) * 2048 <= L::kRingBytes, "last tile staged in the ring");
    // Writes one chunk of kChunk fp32 columns (per thread: one row) to C.
    auto emit_chunk = [&](float* v, int tm, int tn, int j) {
      if constexpr (!SWAP) {
        const int col0 = tn * kOutCols + j * 32;
        const int row0 = tm * kTileRows + static_cast<int>(rank) * kBM + q * 32;
        if (!GATED && p.R != nullptr) add_residual_32(v, p.R, p.ldr, row0 + lane, col0, p.M, p.N);
        store_rows_32x32(&tmC, v, col0, row0, staging, store_count, lane, p.M, p.N,
                         last_staging != nullptr ? last_staging + j * 2048 : nullptr);
      } else {
        // D[n][m]: this thread's row is weight row n, its columns activation rows
        // m; the staging tile is C's layout (row m, 64 consecutive n), so a warp's
        // 16 rows land in 32 contiguous bytes per m.
        if (holds_row) {
          __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(smem + L::kStagingOff);
#pragma unroll
          for (int e = 0; e < L::kChunk; ++e) {
            __nv_bfloat16& o = st[(j * L::kChunk + e) * L::kARows + slot_row];
            float x = v[e];
            if (swap_resid) x += __bfloat162float(o);  // R[m][n], loaded by begin_tile
            o = __float2bfloat16_rn(x);
          }
        }
      }
    };
    // Swapped path: a tile's outputs are gathered in shared memory and written by
    // one TMA store (rows past M and columns past N are clipped by the copy).
    uint32_t resid_phase = 0;
    auto begin_tile = [&](int tm, int tn) {
      if constexpr (SWAP) {
        if (epi_tid == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
        named_bar_sync(2, kEpiThreads);
        if (swap_resid) {
          if (epi_tid == 0 && !resid_early) {
            mbar_arrive_expect_tx(resid_bar, static_cast<uint32_t>(BN * L::kARows * 2));
            tma_load_2d(smem + L::kStagingOff, &tmW2, tm * L::kARows, tn * BN, resid_bar);
          }
          const bool landed = mbar_wait(resid_bar, resid_phase, p.timeout_ns, abort_flag);
          if (!landed && !*abort_flag) record_error(p.err, kDevTimeoutFull, 4000);
          if (bar_sync_or(2, kEpiThreads, !landed)) *abort_flag = 1;  // the tile is then stored unfinished
          resid_phase ^= 1u;
        }
      }
    };
    auto end_tile = [&](int tm, int tn) {
      if constexpr (SWAP) {
        fence_proxy_async_smem();
        named_bar_sync(2, kEpiThreads);
        if (epi_tid == 0) {
          if (p.nbatch > 0) {
            const int bi = batch_of(tm);
            tma_store_2d(&bmaps.c[bi], smem + L::kStagingOff, (tm - p.tile_begin[bi]) * L::kARows, tn * BN);
          } else {
            tma_store_2d(&tmC, smem + L::kStagingOff, tm * L::kARows, tn * BN);
          }
          bulk_commit_group();
        }
      }
    };

    // Asynchronous TMEM load of one chunk (kChunk columns of this thread's row);
    // its registers are valid after tmem_ld_wait(r).
    auto issue_chunk = [&](uint32_t taddr, uint32_t (&r)[L::kChunk]) {
      if constexpr (L::kChunk == 32)
        tmem_ld_32x32b_x32(taddr, r);
      else
        tmem_ld_32x32b_x16(taddr, r);
    };
    auto load_chunk = [&](uint32_t taddr, float* v) {
      uint32_t r[L::kChunk];
      issue_chunk(taddr, r);
      tmem_ld_wait(r);
#pragma unroll
      for (int e = 0; e < L::kChunk; ++e) v[e] = __uint_as_float(r[e]);
    };

    auto release_accumulator = [&](uint32_t b) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(tmem_empty_addr0 + b * 8);
        else
          mbar_arrive(&tmem_empty[b]);
      }
    };

    constexpr int kQuads = L::kChunk / 4;
    constexpr int kSR = L::kSlotRows;
    constexpr int64_t kSlotFloats = static_cast<int64_t>(kSR) * L::kSlotCols;  // one CTA's share of a tile
    for (int i = 0; i < nitems; ++i) {
      const WorkItem w = get_item(sched, unit, i);
      int32_t tm, tn;
      tile_coords(sched, w.tile, tm, tn);
      const uint32_t b = static_cast<uint32_t>(i) & 1u;
      const uint32_t use = static_cast<uint32_t>(i) >> 1;
      // An accumulator is ready after its k-steps have run: allow 20 us per k-step
      // on top of the base bound (a k-step normally takes well under 1 us).
      const uint64_t limit = p.timeout_ns + static_cast<uint64_t>(w.k1 - w.k0) * 20000ull;
      const bool ready = mbar_wait(&tmem_full[b], use & 1u, limit, abort_flag);
      if (!ready && !*abort_flag) record_error(p.err, kDevTimeoutTmemFull, i);
      if (bar_sync_or(1, kEpiThreads, !ready)) {  // all epilogue threads give up together
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + b * L::kAccCols;
      float v[L::kChunk];
      if (!SWAP && w.npieces == 1 && i == nitems - 1)
        last_staging = smem + L::kAOff + ew * (kOutCols / 32) * 2048;
      if (GATED && w.npieces == 1) {
        // Whole gated tile: output chunk j combines accumulator columns j * kChunk
        // (gate) and kOutCols + j * kChunk (up) of this thread's row.
        begin_tile(tm, tn);
#pragma unroll 1
        for (int jo = 0; jo < kOutCols / L::kChunk; ++jo) {
          uint32_t rg[L::kChunk], ru[L::kChunk];
          const int gcol = gate_col(jo * L::kChunk);
          issue_chunk(tacc + gcol, rg);
          issue_chunk(tacc + gcol + kHalf, ru);
          tmem_ld_wait(rg);
          tmem_ld_wait(ru);
#pragma unroll
          for (int e = 0; e < L::kChunk; ++e) v[e] = silu_mul(__uint_as_float(rg[e]), __uint_as_float(ru[e]));
          emit_chunk(v, tm, tn, jo);
        }
        release_accumulator(b);
        end_tile(tm, tn);
      } else if (w.npieces == 1) {
        // Whole tile: the TMEM load of chunk j + 1 is in flight while chunk j is
        // converted and stored.
        constexpr int kChunks = L::kColsPerEpiWarp / L::kChunk;
        begin_tile(tm, tn);
        uint32_t ra[L::kChunk], rb[L::kChunk];
        issue_chunk(tacc + chunk_lo * L::kChunk, ra);
        tmem_ld_wait(ra);
#pragma unroll
        for (int jj = 0; jj < kChunks; ++jj) {
          uint32_t(&cur)[L::kChunk] = (jj & 1) ? rb : ra;
          uint32_t(&nxt)[L::kChunk] = (jj & 1) ? ra : rb;
          if (jj + 1 < kChunks) issue_chunk(tacc + (chunk_lo + jj + 1) * L::kChunk, nxt);
#pragma unroll
          for (int e = 0; e < L::kChunk; ++e) v[e] = __uint_as_float(cur[e]);
          emit_chunk(v, tm, tn, chunk_lo + jj);
          if (jj + 1 < kChunks) tmem_ld_wait(nxt);
        }
        release_accumulator(b);
        end_tile(tm, tn);
      } else {
        // Stream-K piece: publish this CTA's fp32 partial, then count arrivals.
        // Slots and counters are per CTA of a pair (each holds its own rows).
        const int64_t my_slot = PAIR ? 2 * static_cast<int64_t>(w.slot) + rank : w.slot;
        const int counter = PAIR ? 2 * w.sk_index + static_cast<int>(rank) : w.sk_index;
        float4* slot = reinterpret_cast<float4*>(p.partials + my_slot * kSlotFloats);
        for (int j = 0; j < L::kAccCols / L::kChunk; ++j) {  // every accumulator column
          load_chunk(tacc + j * L::kChunk, v);
          if (holds_row) {
#pragma unroll
            for (int q4 = 0; q4 < kQuads; ++q4)
              slot[(j * kQuads + q4) * kSR + slot_row] =
                  make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          }
        }
        release_accumulator(b);
        fence_proxy_async_global();  // the finisher may read these bytes with bulk copies
        __threadfence();
        named_bar_sync(1, 32 * L::kEpiWarps);
        if (epi_tid == 0) {
          const uint32_t before = atomicAdd(&p.counters[counter], 1u);
          *sk_last = (before == static_cast<uint32_t>(w.npieces - 1)) ? 1u : 0u;
        }
        named_bar_sync(1, 32 * L::kEpiWarps);
        // The CTA's last item, when this CTA finishes its tile: the epilogue warps
        // sum it themselves from the idle copy ring (below), since nothing follows
        // for them to overlap it with.
        constexpr int64_t kChunkFloats = static_cast<int64_t>(kQuads) * kSR * 4;  // one piece's 32 columns
        const bool take_last = !SWAP && !GATED && *sk_last && i == nitems - 1 &&
                               static_cast<int64_t>(w.npieces) * kChunkFloats * 4 <= L::kRingBytes;
        if (L::kFixupWarps > 0 && i < L::kMaxJobs) {
          // Hand the piece to the fixup warps (the sum, if this piece arrived last,
          // runs there while this epilogue goes on to the next tile).
          if (epi_tid == 0) {
            int32_t* job = reinterpret_cast<int32_t*>(smem + L::kJobOff) + 4 * i;
            job[0] = tm;
            job[1] = tn;
            job[2] = static_cast<int32_t>(*sk_last && !take_last);
            mbar_arrive(&job_bar[i]);
          }
          if (!take_last) continue;
        }
        if (take_last) {
          // Chunk j (32 columns) of every piece's partial is bulk-copied into the
          // ring under fixup_bar's phase j, two chunks' buffers in turn when they
          // fit, then summed in k order and stored.  The piece's loads in flight
          // are whole 16 KB chunks instead of one row per thread.
          __threadfence();
          float* ring = reinterpret_cast<float*>(smem);
          constexpr int kNChunks = L::kAccCols / L::kChunk;
          const int64_t buf_floats = static_cast<int64_t>(w.npieces) * kChunkFloats;
          const bool two_bufs = 2 * buf_floats * 4 <= L::kRingBytes;
          auto fetch = [&](int j) {
            if (epi_tid == 0) {
              float* dst = ring + ((two_bufs && (j & 1)) ? buf_floats : 0);
              fence_proxy_async_global();
              mbar_arrive_expect_tx(fixup_bar, static_cast<uint32_t>(buf_floats * 4));
              for (int pj = 0; pj < w.npieces; ++pj) {
                const int64_t sl = piece_slot(sched, w.sk_index, pj);
                bulk_load(dst + pj * kChunkFloats,
                          p.partials + (PAIR ? 2 * sl + rank : sl) * kSlotFloats + j * kChunkFloats,
                          static_cast<uint32_t>(kChunkFloats * 4), fixup_bar);
              }
            }
          };
          fetch(0);
          for (int j = 0; j < kNChunks; ++j) {
            const bool landed = mbar_wait(fixup_bar, static_cast<uint32_t>(j) & 1u, p.timeout_ns, abort_flag);
            if (!landed && !*abort_flag) record_error(p.err, kDevTimeoutFull, 1000 + i);
            if (bar_sync_or(1, kEpiThreads, !landed)) {  // every thread is past chunk j - 1
              *abort_flag = 1;
              break;
            }
            if (two_bufs && j + 1 < kNChunks) fetch(j + 1);
            const float4* src =
                reinterpret_cast<const float4*>(ring + ((two_bufs && (j & 1)) ? buf_floats : 0));
            float acc[L::kChunk];
            for (int pj = 0; pj < w.npieces; ++pj) {  // k order
#pragma unroll
              for (int q4 = 0; q4 < kQuads; ++q4) {
                const float4 x = src[pj * (kChunkFloats / 4) + q4 * kSR + slot_row];
                float* a4 = &acc[4 * q4];
                if (pj == 0) {
                  a4[0] = x.x; a4[1] = x.y; a4[2] = x.z; a4[3] = x.w;
                } else {
                  a4[0] += x.x; a4[1] += x.y; a4[2] += x.z; a4[3] += x.w;
                }
              }
            }
            emit_chunk(acc, tm, tn, j);
            if (!two_bufs && j + 1 < kNChunks) {
              named_bar_sync(1, kEpiThreads);  // the one buffer has been read
              fetch(j + 1);
            }
          }
          if (epi_tid == 0) atomicExch(&p.counters[counter], 0u);
          continue;
        }
        if constexpr (GATED && !SWAP) {
          // the gated plan gives no CTA more Stream-K pieces than the fixup warps take
          if (epi_tid == 0) record_error(p.err, kDevTimeoutFull, 3000 + i);
          continue;
        }
        // Writes output chunk jo from the summed accumulator chunks: chunk jo, or
        // silu(chunk jo) * chunk jo + kOutCols / kChunk when gated.
        auto emit_summed = [&](auto&& sum_chunk) {
#pragma unroll 1
          for (int jo = 0; jo < kOutCols / L::kChunk; ++jo) {
            float acc[L::kChunk];
            sum_chunk(GATED ? gate_col(jo * L::kChunk) / L::kChunk : jo, acc);
            if constexpr (GATED) {
              float up[L::kChunk];
              sum_chunk((gate_col(jo * L::kChunk) + kHalf) / L::kChunk, up);
#pragma unroll
              for (int e = 0; e < L::kChunk; ++e) acc[e] = silu_mul(acc[e], up[e]);
            }
            emit_chunk(acc, tm, tn, jo);
          }
        };
        // The finisher's last item: the copy ring is idle (every stage of this CTA
        // has been consumed), so all pieces' partials are fetched into it with
        // bulk copies under one barrier instead of dependent rounds of loads.
        const bool ring_fixup = *sk_last && i == nitems - 1 &&
                                static_cast<int64_t>(w.npieces) * kSlotFloats * 4 <= L::kRingBytes;
        if (ring_fixup) {
          __threadfence();
          float* ring = reinterpret_cast<float*>(smem);
          if (epi_tid == 0) {
            fence_proxy_async_global();
            const uint32_t slot_bytes = static_cast<uint32_t>(kSlotFloats * 4);
            mbar_arrive_expect_tx(fixup_bar, slot_bytes * static_cast<uint32_t>(w.npieces));
            for (int pj = 0; pj < w.npieces; ++pj) {
              const int64_t sl = piece_slot(sched, w.sk_index, pj);
              bulk_load(ring + pj * kSlotFloats, p.partials + (PAIR ? 2 * sl + rank : sl) * kSlotFloats, slot_bytes,
                        fixup_bar);
            }
          }
          const bool landed = mbar_wait(fixup_bar, 0, p.timeout_ns, abort_flag);
          if (!landed && !*abort_flag) record_error(p.err, kDevTimeoutFull, 1000 + i);
          if (bar_sync_or(1, kEpiThreads, !landed)) {
            *abort_flag = 1;
          } else {
            begin_tile(tm, tn);
            const float4* rs = reinterpret_cast<const float4*>(ring);
            emit_summed([&](int j, float* acc) {
#pragma unroll
              for (int e = 0; e < L::kChunk; ++e) acc[e] = 0.f;
              for (int pj = 0; pj < w.npieces && holds_row; ++pj) {  // k order
                const float4* src = rs + pj * (kSlotFloats / 4);
#pragma unroll
                for (int q4 = 0; q4 < kQuads; ++q4) {
                  const float4 x = src[(j * kQuads + q4) * kSR + slot_row];
                  float* a4 = &acc[4 * q4];
                  if (pj == 0) {
                    a4[0] = x.x; a4[1] = x.y; a4[2] = x.z; a4[3] = x.w;
                  } else {
                    a4[0] += x.x; a4[1] += x.y; a4[2] += x.z; a4[3] += x.w;
                  }
                }
              }
            });
            end_tile(tm, tn);
          }
          if (epi_tid == 0) atomicExch(&p.counters[counter], 0u);
        } else if (*sk_last) {
          // Last arrival: sum all pieces in k order, then store.
          __threadfence();
          // Loads in flight per batch: kBatch pieces x kBQuads float4 of one chunk.
          constexpr int kBatch = (kQuads <= 4 && !GATED) ? 4 : 2;  // pieces per batch (8-16 loads in flight)
          constexpr int kBQuads = kQuads;                // float4 per piece per batch: the whole chunk
          begin_tile(tm, tn);
          emit_summed([&](int j, float* acc) {
#pragma unroll
            for (int e = 0; e < L::kChunk; ++e) acc[e] = 0.f;
#pragma unroll
            for (int h = 0; h < kQuads / kBQuads; ++h) {
              for (int pj = 0; pj < w.npieces && holds_row; pj += kBatch) {
                float4 x[kBatch][kBQuads];
#pragma unroll
                for (int bi = 0; bi < kBatch; ++bi) {
                  if (pj + bi < w.npieces) {
                    const int64_t sl = piece_slot(sched, w.sk_index, pj + bi);
                    const float4* src =
                        reinterpret_cast<const float4*>(p.partials + (PAIR ? 2 * sl + rank : sl) * kSlotFloats);
#pragma unroll
                    for (int q4 = 0; q4 < kBQuads; ++q4)
                      x[bi][q4] = __ldcg(&src[(j * kQuads + h * kBQuads + q4) * kSR + slot_row]);
                  }
                }
#pragma unroll
                for (int bi = 0; bi < kBatch; ++bi) {  // k order: pieces pj, pj + 1, ...
                  if (pj + bi < w.npieces) {
#pragma unroll
                    for (int q4 = 0; q4 < kBQuads; ++q4) {
                      float* a4 = &acc[4 * (h * kBQuads + q4)];
                      if (pj + bi == 0) {
                        a4[0] = x[bi][q4].x; a4[1] = x[bi][q4].y; a4[2] = x[bi][q4].z; a4[3] = x[bi][q4].w;
                      } else {
                        a4[0] += x[bi][q4].x; a4[1] += x[bi][q4].y; a4[2] += x[bi][q4].z; a4[3] += x[bi][q4].w;
                      }
                    }
                  }
                }
              }
            }
          });
          end_tile(tm, tn);
          if (epi_tid == 0) atomicExch(&p.counters[counter], 0u);
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // stores complete before the CTA exits
  } else {
    // ------------------------------------------------------------ Stream-K fixup
    // Takes the CTA's Stream-K pieces in order.  For a piece whose tile this CTA
    // finished last, sums every piece's fp32 partial in k order (each thread one
    // row, 64 rows per warp) and stores bf16.
    grid_dependency_wait();
    const int fw = warp - 2 - L::kEpiWarps;
    uint8_t* fstaging = smem + L::kFixStagingOff + fw * L::kStagingBufs * L::kStagingBufBytes;
    uint32_t fstore_count = 0;
    constexpr int64_t kSlotFloats = static_cast<int64_t>(kBM) * BN;
    constexpr int kQuads = 8;  // float4 per 32-column chunk
    const int njobs = min(sk_count(sched, unit), L::kMaxJobs);
    for (int jidx = 0; jidx < njobs; ++jidx) {
      const WorkItem w = get_item(sched, unit, jidx);
      if (w.npieces <= 1) continue;  // a whole tile: the epilogue stored it
      // the job is posted once this piece's accumulator is ready, after at most
      // jidx + 1 items of this CTA: allow 20 us per k-step of those
      const uint64_t limit = p.timeout_ns + static_cast<uint64_t>((jidx + 1) * sched.k_steps) * 20000ull;
      const bool posted = mbar_wait(&job_bar[jidx], 0, limit, abort_flag);
      if (!posted && !*abort_flag) record_error(p.err, kDevTimeoutTmemFull, 2000 + jidx);
      if (bar_sync_or(3, 32 * L::kFixupWarps, !posted)) {
        *abort_flag = 1;
        break;
      }
      const int32_t* job = reinterpret_cast<const int32_t*>(smem + L::kJobOff) + 4 * jidx;
      const int tm = job[0], tn = job[1];
      if (!job[2]) continue;
      __threadfence();  // the other pieces' partials were published before their arrivals
      // Sums 32-column chunk j of every piece's partial for row frow, in k order.
      constexpr int kFB = GATED ? 1 : 4;  // pieces whose loads are in flight together
      auto sum_chunk = [&](int j, int frow, float* acc) {
        for (int pj = 0; pj < w.npieces; pj += kFB) {
          float4 x[kFB][kQuads];
#pragma unroll
          for (int bi = 0; bi < kFB; ++bi) {
            if (pj + bi < w.npieces) {
              const int64_t sl = piece_slot(sched, w.sk_index, pj + bi);
              const float4* src =
                  reinterpret_cast<const float4*>(p.partials + (PAIR ? 2 * sl + rank : sl) * kSlotFloats);
#pragma unroll
              for (int q4 = 0; q4 < kQuads; ++q4) x[bi][q4] = __ldcg(&src[(j * kQuads + q4) * kBM + frow]);
            }
          }
#pragma unroll
          for (int bi = 0; bi < kFB; ++bi) {  // k order: pieces pj, pj + 1, ...
            if (pj + bi < w.npieces) {
#pragma unroll
              for (int q4 = 0; q4 < kQuads; ++q4) {
                float* a4 = &acc[4 * q4];
                if (pj + bi == 0) {
                  a4[0] = x[bi][q4].x; a4[1] = x[bi][q4].y; a4[2] = x[bi][q4].z; a4[3] = x[bi][q4].w;
                } else {
                  a4[0] += x[bi][q4].x; a4[1] += x[bi][q4].y; a4[2] += x[bi][q4].z; a4[3] += x[bi][q4].w;
                }
              }
            }
          }
        }
      };
#pragma unroll 1
      for (int j = 0; j < kOutCols / 32; ++j) {
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          const int frow = fw * 64 + g * 32 + lane;
          float acc[32];
          sum_chunk(GATED ? gate_col(j * 32) / 32 : j, frow, acc);
          if constexpr (GATED) {
            float up[32];
            sum_chunk((gate_col(j * 32) + kHalf) / 32, frow, up);
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = silu_mul(acc[e], up[e]);
          }
          const int frow0 = tm * kTileRows + static_cast<int>(rank) * kBM + fw * 64 + g * 32;
          if (!GATED && p.R != nullptr) add_residual_32(acc, p.R, p.ldr, frow0 + lane, tn * kOutCols + j * 32, p.M, p.N);
          store_rows_32x32(&tmC, acc, tn * kOutCols + j * 32, frow0, fstaging, fstore_count, lane, p.M, p.N);
        }
      }
      if (fw == 0 && lane == 0) atomicExch(&p.counters[PAIR ? 2 * w.sk_index + static_cast<int>(rank) : w.sk_index], 0u);
    }
    if (lane == 0) bulk_wait_group<0>();  // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, L::kTmemCols);
    else
      tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int BN, int STAGES, int SWAP_ROWS, int KSUB, bool PAIR, bool GATED = false>
cudaError_t launch_variant(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const TcParams& p,
                           cudaStream_t stream, const CUtensorMap* b2 = nullptr,
                           const TcBatchMaps* batch = nullptr) {
  static const TcBatchMaps kNoBatch{};
  using L = TcLayout<BN, STAGES, SWAP_ROWS, KSUB, PAIR, GATED>;
  auto kern = tc_gemm_kernel<BN, STAGES, SWAP_ROWS, KSUB, PAIR, GATED>;
  static bool configured = false;  // the attribute is per function, process-wide
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((PAIR ? 2 : 1) * p.sched.grid, 1, 1);
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a, b, c, b2 ? *b2 : b, p, batch ? *batch : kNoBatch);
}

}  // namespace

cudaError_t launch_tc_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const TcParams& p, cudaStream_t stream) {
  return launch_variant<kGemmBN, kGemmStages, 0, 1, false>(tmA, tmB, tmC, p, stream);
}

cudaError_t launch_tc_gemm_narrow(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                                  const TcParams& p, cudaStream_t stream) {
  return launch_variant<kGemmNarrowBN, kGemmNarrowStages, 0, 1, false>(tmA, tmB, tmC, p, stream);
}

cudaError_t launch_tc_gemm_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmG, const CUtensorMap& tmU,
                                  const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
  return launch_variant<kGemmBN, kGemmStages, 0, 1, false, true>(tmA, tmG, tmC, p, stream, &tmU);
}

cudaError_t launch_tc_gemm_swiglu_pair(const CUtensorMap& tmA, const CUtensorMap& tmG, const CUtensorMap& tmU,
                                       const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
  return launch_variant<kGemmBN, kPairStages, 0, 1, true, true>(tmA, tmG, tmC, p, stream, &tmU);
}

cudaError_t launch_tc_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                                const TcParams& p, cudaStream_t stream) {
  return launch_variant<kGemmBN, kPairStages, 0, 1, true>(tmA, tmB, tmC, p, stream);
}

template <int BN, int ROWS>
cudaError_t launch_skinny(const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmC, const TcParams& p,
                          cudaStream_t stream, const CUtensorMap* tmR, const TcBatchMaps* batch) {
  static_assert(TcLayout<BN, skinny_stages(BN, ROWS), ROWS, skinny_ksub(ROWS), false>::kMinBlocks == kSkinnyCtasPerSm,
                "the skinny plan counts on two resident CTAs per SM");
  return launch_variant<BN, skinny_stages(BN, ROWS), ROWS, skinny_ksub(ROWS), false>(tmW, tmX, tmC, p, stream, tmR,
                                                                                     batch);
}

template <int BN>
cudaError_t launch_skinny_swiglu(const CUtensorMap& tmG, const CUtensorMap& tmU, const CUtensorMap& tmX,
                                 const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
  constexpr int kS = skinny_stages_gated(BN);
  static_assert(TcLayout<BN, kS, 64, 1, false, true>::kMinBlocks == kSkinnyCtasPerSm,
                "the skinny plan counts on two resident CTAs per SM");
  return launch_variant<BN, kS, 64, 1, false, true>(tmG, tmX, tmC, p, stream, &tmU);
}

cudaError_t launch_tc_skinny_swiglu(int bn, const CUtensorMap& tmG, const CUtensorMap& tmU, const CUtensorMap& tmX,
                                    const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch_skinny_swiglu<16>(tmG, tmU, tmX, tmC, p, stream);
    case 32: return launch_skinny_swiglu<32>(tmG, tmU, tmX, tmC, p, stream);
    case 64: return launch_skinny_swiglu<64>(tmG, tmU, tmX, tmC, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc_skinny(int bn, int rows, const CUtensorMap& tmW, const CUtensorMap& tmX,
                             const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream, const CUtensorMap* tmR,
                             const TcBatchMaps* batch) {
  if (rows == 64) {
    switch (bn) {
      case 16: return launch_skinny<16, 64>(tmW, tmX, tmC, p, stream, tmR, batch);
      case 32: return launch_skinny<32, 64>(tmW, tmX, tmC, p, stream, tmR, batch);
      case 64: return launch_skinny<64, 64>(tmW, tmX, tmC, p, stream, tmR, batch);
      default: return cudaErrorInvalidValue;
    }
  }
  if (rows == 128) {
    switch (bn) {
      case 16: return launch_skinny<16, 128>(tmW, tmX, tmC, p, stream, tmR, batch);
      case 32: return launch_skinny<32, 128>(tmW, tmX, tmC, p, stream, tmR, batch);
      case 64: return launch_skinny<64, 128>(tmW, tmX, tmC, p, stream, tmR, batch);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace sg

// Host side of the C ABI declared in include/skinny_gemm.h: argument checks,
// per-device state (properties, workspace, error word), tensor-map encoding,
// launch planning and dispatch.  Nothing here computes any part of C: every
// output element is produced by the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/skinny_gemm.h"
#include "sg_internal.h"
#include "sg_ptx.cuh"
#include "sg_sched.cuh"

namespace sg {
namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<uint32_t> g_inject_missing_tx{0};  // consumed by the next tcgen05 GEMM, one-CTA NVFP4 or attention launch

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return SG_ERR_CUDA;
}

// ----------------------------------------------------------------- device state
constexpr int kMaxDevices = 64;
constexpr size_t kPartialBytes = size_t(64) << 20;  // Stream-K / split-K fp32 partials
constexpr size_t kNumCounters = 16384;
constexpr int64_t kCcMaxRowsPerCta = 256;

struct DeviceState {
  bool props_ready = false;
  int sm_count = 0, cc_major = 0, cc_minor = 0, smem_optin = 0, l2_bytes = 0;
  void* workspace = nullptr;  // [partials | counters | error word]
  float* partials = nullptr;
  uint32_t* counters = nullptr;
  DeviceError* err = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

int current_device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return SG_ERR_UNSUPPORTED_DEVICE;
  DeviceState& d = g_devices[dev];
  if (!d.props_ready) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.props_ready) {
      int v[5];
      const cudaDeviceAttr attrs[5] = {cudaDevAttrMultiProcessorCount, cudaDevAttrComputeCapabilityMajor,
                                       cudaDevAttrComputeCapabilityMinor, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                       cudaDevAttrL2CacheSize};
      for (int i = 0; i < 5; ++i) {
        e = cudaDeviceGetAttribute(&v[i], attrs[i], dev);
        if (e != cudaSuccess) return cuda_fail(e);
      }
      d.sm_count = v[0];
      d.cc_major = v[1];
      d.cc_minor = v[2];
      d.smem_optin = v[3];
      d.l2_bytes = v[4];
      d.props_ready = true;
    }
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return SG_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  if (dev_out) *dev_out = dev;
  return SG_OK;
}

// Allocates the workspace on first use.  Refused while `stream` is capturing.
int ensure_workspace(DeviceState& d, cudaStream_t stream) {
  if (d.workspace) return SG_OK;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (d.workspace) return SG_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e);
  if (cap != cudaStreamCaptureStatusNone) return SG_ERR_INVALID_ARG;
  const size_t bytes = kPartialBytes + kNumCounters * sizeof(uint32_t) + 256;
  void* p = nullptr;
  e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    return SG_ERR_OUT_OF_MEMORY;
  }
  uint8_t* base = static_cast<uint8_t*>(p);
  e = cudaMemsetAsync(base + kPartialBytes, 0, bytes - kPartialBytes, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaFree(p);
    return cuda_fail(e);
  }
  d.partials = reinterpret_cast<float*>(base);
  d.counters = reinterpret_cast<uint32_t*>(base + kPartialBytes);
  d.err = reinterpret_cast<DeviceError*>(base + kPartialBytes + kNumCounters * sizeof(uint32_t));
  d.workspace = p;
  return SG_OK;
}

// ----------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  uint64_t cols, rows, ld;
  uint32_t box_cols, box_rows, swizzle;
  int dev;
  uint32_t elem_bytes;  // 2: bf16 / fp16 elements, 1: bytes (packed fp4)
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && cols == o.cols && rows == o.rows && ld == o.ld && box_cols == o.box_cols &&
           box_rows == o.box_rows && swizzle == o.swizzle && dev == o.dev && elem_bytes == o.elem_bytes;
  }
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
};

constexpr int kMapCacheSize = 64;
std::mutex g_map_mutex;
MapEntry g_map_cache[kMapCacheSize];
int g_map_used = 0, g_map_next = 0;

// A 2-D bf16 tensor of `rows` rows x `cols` columns with a row pitch of `ld`
// elements, read or written in boxes of box_rows x box_cols.
// 2-D tensor map of a row-major matrix of 16-bit elements (elem_bytes 2) or of
// bytes (elem_bytes 1); cols, ld and box_cols count elements.
int make_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
             uint32_t box_cols, CUtensorMapSwizzle swz, int dev, uint32_t elem_bytes = 2) {
  const MapKey key{ptr, cols, rows, ld, box_cols, box_rows, static_cast<uint32_t>(swz), dev, elem_bytes};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_cache[i].key == key) {
        *out = g_map_cache[i].map;
        return SG_OK;
      }
  }
  EncodeTiledFn enc = get_encoder();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = enc(&m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  *out = m;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  MapEntry& slot = g_map_cache[g_map_used < kMapCacheSize ? g_map_used++ : (g_map_next++ % kMapCacheSize)];
  slot.key = key;
  slot.map = m;
  return SG_OK;
}

// ----------------------------------------------------------------- planning
void fill_sched(sg_plan_info* o, const Schedule& s) {
  o->tiles_m = s.tiles_m;
  o->tiles_n = s.tiles_n;
  o->k_steps = s.k_steps;
  o->grid = s.grid;
  o->dp_tiles = s.dp_tiles;
  o->sk_tiles = s.sk_tiles;
  o->sk_units = s.sk_units;
  o->group_m = s.group_m;
}

Schedule sched_from_plan(const sg_plan_info& o) {
  Schedule s{};
  s.tiles_m = o.tiles_m;
  s.tiles_n = o.tiles_n;
  s.k_steps = o.k_steps;
  s.grid = o.grid;
  s.dp_tiles = o.dp_tiles;
  s.sk_tiles = o.sk_tiles;
  s.sk_units = o.sk_units;
  s.group_m = o.group_m;
  s.split = (o.path == SG_PATH_TENSOR_CORE || o.path == SG_PATH_GEMM || o.path == SG_PATH_GEMM_PAIR) ? o.split_k : 0;
  s.sk_q = s.sk_units > 0 ? static_cast<int32_t>(s.sk_units / s.grid) : 0;
  s.sk_r = s.sk_units > 0 ? static_cast<int32_t>(s.sk_units % s.grid) : 0;
  return s;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Single-CTA tiles are 128 columns wide when the 128 x 128 tiles fit in one wave
// of SMs, else 256.  Such a GEMM then spreads over up to twice as many SMs, each
// with half the MMA work per k-step, and splits K less often.  Measured
// (graph-timed): 512^3 6.4 -> 5.3 us, 1024^3 9.5 -> 8.0 us, 1536^3 12.4 -> 11.2 us,
// 128 x 4096 x 4096 83.3 -> 26.4 us, 512 x 4096 x 4096 38.8 -> 22.4 us,
// 128 x 11008 x 4096 56.8 -> 22.7 us; past one wave they lose (1792^3 14.0 -> 19.9 us).
bool narrow_tiles(int64_t M, int64_t N, int sms) {
  return ceil_div(M, kBM) * ceil_div(N, kGemmNarrowBN) <= static_cast<int64_t>(sms);
}

// tcgen05 GEMM plan.  pair: 256 x 256 tiles on clusters of two CTAs (the
// schedule counts clusters); else 128 x 256 or 128 x 128 tiles, one CTA each.
void plan_tc_gemm(int64_t M, int64_t N, int64_t K, int sms, bool pair, sg_plan_info* o) {
  std::memset(o, 0, sizeof *o);
  const bool narrow = !pair && narrow_tiles(M, N, sms);
  o->path = pair ? SG_PATH_GEMM_PAIR : SG_PATH_GEMM;
  o->tile_m = pair ? 2 * kBM : kBM;
  o->tile_n = narrow ? kGemmNarrowBN : kGemmBN;
  o->tile_k = kBK;
  o->stages = pair ? kPairStages : (narrow ? kGemmNarrowStages : kGemmStages);
  o->cluster_size = pair ? 2 : 1;
  const int32_t units = pair ? std::max(1, sms / 2) : sms;
  const int32_t tm = static_cast<int32_t>(ceil_div(M, o->tile_m)), tn = static_cast<int32_t>(ceil_div(N, o->tile_n));
  const int32_t ks = static_cast<int32_t>(ceil_div(K, kBK));
  // Raster groups of 8 tile rows: a wave of 76 pair tiles then spans ~8 rows x
  // ~10 columns of tiles, the fewest A and B bytes per wave (measured: MLP
  // 4096 x 11008 x 4096 204.6 -> 199.5 us and 4096 x 4096 x 11008 210.1 -> 202.1 us
  // against groups of 4; 4096^3 and 8192^3 unchanged within noise).
  Schedule s = make_schedule(tm, tn, ks, units, 4, std::min<int32_t>(tm, 8), false);
  o->split_k = 0;
  const int64_t T = static_cast<int64_t>(tm) * tn;
  if (T < units && s.sk_tiles == T && s.dp_tiles == 0) {
    // Fewer tiles than units, and K worth splitting: every tile is cut into
    // `split` equal k pieces, one per unit (split mode), so each unit runs one
    // piece and the piece that finishes a tile is its unit's last item, summed
    // from the idle copy ring.  Stream-K ranges over the same units would cross
    // tile boundaries, and a piece that finishes a tile in the middle of its
    // unit's schedule is summed by the fixup warps, at a fraction of the
    // bandwidth.  Measured with the ring sum: 384 x 512 x 8192 56.3 -> 19.6 us,
    // 300 x 1000 x 2048 36.1 -> 15.6 us, 256 x 256 x 65536 135 -> 51 us.  At most
    // kGemmMaxSplit pieces per tile: their 32-column chunks fit the ring together.
    const int32_t split = std::min<int32_t>(s.grid / static_cast<int32_t>(T), kGemmMaxSplit);
    if (split >= 2) {
      s = make_split_schedule(tm, tn, ks, split);
      o->split_k = split;
    }
  }
  fill_sched(o, s);
  o->ctas_per_sm = 1;
  o->wave_efficiency = wave_efficiency(T, units);
}

// The automatic GEMM kernel for M > 64: CTA pairs from M = 256, except where
// 128 x 128 single-CTA tiles fit in one wave (above), or where at most 32 k-steps
// of 256 x 256 pair tiles fall short of a wave while 128 x 256 single-CTA tiles
// fit in one: the pairs' set-up then weighs more than their lighter operand
// traffic (2048^3 16.3 -> 15.8 us, 1792^3 14.35 -> 13.96 us; at 64 k-steps the
// pairs stay ahead, 1024 x 4096 x 4096 25.3 against 27.5 us).
bool auto_pair(int64_t M, int64_t N, int64_t K, int sms) {
  if (M < 2 * kBM || narrow_tiles(M, N, sms)) return false;
  const bool short_sub_wave = ceil_div(K, kBK) <= 32 && ceil_div(M, 2 * kBM) * ceil_div(N, kGemmBN) < sms / 2 &&
                              ceil_div(M, kBM) * ceil_div(N, kGemmBN) <= sms;
  return !short_sub_wave;
}

// Most Stream-K pieces any CTA of the schedule runs.
int32_t max_sk_items(const Schedule& s) {
  int32_t m = 0;
  for (int32_t c = 0; c < s.grid; ++c) m = std::max(m, sk_count(s, c));
  return m;
}

// Gated GEMM plan (silu(A . G^T) * (A . U^T)): tiles of 128 (single CTA) or 256
// (CTA pair) rows x 128 output columns, each computed from 128 gate and 128 up
// weight rows.  Stream-K stays only where no CTA gets more pieces than the fixup
// warps take.
void plan_tc_swiglu(int64_t M, int64_t N, int64_t K, int sms, bool pair, sg_plan_info* o) {
  std::memset(o, 0, sizeof *o);
  o->path = pair ? SG_PATH_GEMM_PAIR : SG_PATH_GEMM;
  o->tile_m = pair ? 2 * kBM : kBM;
  o->tile_n = kGemmBN / 2;
  o->tile_k = kBK;
  o->stages = pair ? kPairStages : kGemmStages;
  o->cluster_size = pair ? 2 : 1;
  o->ctas_per_sm = 1;
  const int32_t units = pair ? std::max(1, sms / 2) : sms;
  const int32_t tm = static_cast<int32_t>(ceil_div(M, o->tile_m)), tn = static_cast<int32_t>(ceil_div(N, kGemmBN / 2));
  const int32_t ks = static_cast<int32_t>(ceil_div(K, kBK));
  Schedule s = make_schedule(tm, tn, ks, units, 4, std::min<int32_t>(tm, pair ? 4 : 8), false);
  if (s.sk_tiles > 0 && max_sk_items(s) > kFixupMaxJobs) {
    s.dp_tiles += s.sk_tiles;
    s.sk_tiles = 0;
    s.sk_units = 0;
    s.sk_q = s.sk_r = 0;
  }
  fill_sched(o, s);
  o->split_k = 0;
  o->wave_efficiency = wave_efficiency(static_cast<int64_t>(tm) * tn, units);
}

int skinny_bn(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// Swapped skinny plan: 128-row (M <= 16) or 64-row weight tiles, two CTAs per SM.  When every tile
// fits in the resident slots, each tile is cut into split_k equal k pieces, one
// CTA per piece, and all CTAs run at once (split mode); past that, a persistent
// grid of two CTAs per SM walks the tiles with a Stream-K remainder.
// Weight rows per tile.  Each tile's MMAs are thin (N = 16 to 64 activation
// rows), and a thin tcgen05.mma costs about the same whatever its N, so wider
// weight tiles mean fewer MMAs for the same bytes.  128-row tiles pay at M <= 16
// (11008 x 4096 weights 18.3 -> 17.6 us, 4096 x 11008 18.8 -> 18.6 us); at M = 64
// they hold only three stages and split K nine ways with 32 KB partial sums
// (20.3 -> 21.9 us and 21.5 -> 27.1 us), so 64-row tiles stay there.
int skinny_rows(int64_t M) { return M <= 16 ? 128 : 64; }

void plan_tc_skinny(int64_t M, int64_t N, int64_t K, int sms, sg_plan_info* o, bool gated = false) {
  std::memset(o, 0, sizeof *o);
  const int rows = gated ? 64 : skinny_rows(M);  // gated: 64 outputs from 64 gate + 64 up rows
  o->path = SG_PATH_TENSOR_CORE;
  o->tile_m = rows;
  o->tile_n = skinny_bn(M);
  o->tile_k = gated ? kBK : kBK * skinny_ksub(rows);
  o->stages = gated ? skinny_stages_gated(o->tile_n) : skinny_stages(o->tile_n, rows);
  o->cluster_size = 1;
  o->ctas_per_sm = kSkinnyCtasPerSm;
  const int32_t tm = static_cast<int32_t>(ceil_div(N, rows));
  const int32_t ks = static_cast<int32_t>(ceil_div(K, o->tile_k));
  const int32_t slots = kSkinnyCtasPerSm * sms;
  if (tm <= slots) {
    const int32_t split = std::max(1, std::min(slots / tm, ks / (kSkinnyMinPieceK / o->tile_k)));
    const Schedule s = make_split_schedule(tm, 1, ks, split);
    fill_sched(o, s);
    o->split_k = s.split;
  } else {
    const Schedule s = make_schedule(tm, 1, ks, slots, 2, 1, true);
    fill_sched(o, s);
    o->split_k = 0;
  }
  o->wave_efficiency = wave_efficiency(o->grid, slots);
  // Early L2 reads of the first weights pay when the next launch's CTAs can only
  // start as this one's leave (the grid fills most slots); with many slots free,
  // they start at once and compete with the running launch's stream (measured
  // slower at N = 11,008 and 12,288, K = 4,096: 172 and 192 CTAs on 304 slots).
  o->prefetch_steps = o->grid * 10 >= kPreWaitMinFill * slots ? kPreWaitSteps : 0;
}

// CUDA-core plan: two CTAs per SM, each owning a contiguous block of weight rows
// (at most kCcMaxRowsPerCta); K is split across CTAs only when there are fewer
// row blocks than that.
void plan_cc(int64_t M, int64_t N, int64_t K, int sms, sg_plan_info* o, bool gated = false) {
  std::memset(o, 0, sizeof *o);
  o->path = SG_PATH_CUDA_CORE;
  o->cluster_size = 1;
  o->ctas_per_sm = 2;
  const int64_t target = 2 * static_cast<int64_t>(sms);
  int64_t rows_grid = std::min<int64_t>(N, target);
  rows_grid = std::max<int64_t>(rows_grid, ceil_div(N, kCcMaxRowsPerCta));
  int64_t split = 1;
  if (rows_grid < target && K >= 2048) split = std::max<int64_t>(1, std::min<int64_t>(ceil_div(target, rows_grid), K / 1024));
  int64_t k_slice = ceil_div(ceil_div(K, split), 8) * 8;
  if (k_slice < 8) k_slice = 8;
  split = ceil_div(K, k_slice);
  if (split < 1) split = 1;
  const int64_t mrows = std::min<int64_t>(M, 8);
  if (split > 1 && (static_cast<size_t>(split) * mrows * N * 4 * (gated ? 2 : 1) > kPartialBytes ||
                    static_cast<size_t>(rows_grid) > kNumCounters)) {
    split = 1;
    k_slice = ceil_div(K, 8) * 8;
  }
  o->rows_per_cta = static_cast<int32_t>(ceil_div(N, rows_grid));
  o->tile_m = o->rows_per_cta;
  o->tile_n = static_cast<int32_t>(mrows);
  o->tile_k = 8;
  o->split_k = static_cast<int32_t>(split);
  o->tiles_m = static_cast<int32_t>(rows_grid);
  o->tiles_n = 1;
  o->k_steps = static_cast<int32_t>(k_slice);  // elements per K slice
  o->grid = static_cast<int32_t>(rows_grid * split);
  o->wave_efficiency = wave_efficiency(o->grid, 2 * static_cast<int64_t>(sms));
  o->prefetch_steps = o->grid * 10 >= kPreWaitMinFill * target ? 1 : 0;  // one row pass
}

// The CUDA-core kernel spends M/2 paired fp32 FMAs per weight element; measured
// on the 7B-model decode shapes it keeps up with the weight stream at M <= 2,
// beyond which the tcgen05 kernel (same single pass over the weights) is faster.
constexpr int64_t kCudaCoreMaxRows = 2;
int choose_skinny_path(int64_t M) { return M <= kCudaCoreMaxRows ? SG_PATH_CUDA_CORE : SG_PATH_TENSOR_CORE; }

// The gated entry's automatic kernel: the skinny kernels up to M = 64, then the
// GEMM, on CTA pairs from M = 256 (as gemm_bf16).
int swiglu_path(int64_t M) {
  return M <= 64 ? choose_skinny_path(M) : (M >= 2 * kBM ? SG_PATH_GEMM_PAIR : SG_PATH_GEMM);
}

// ----------------------------------------------------------------- validation
int validate(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
             int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return SG_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return SG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SG_OK;
  if (!C || (K > 0 && (!A || !B))) return SG_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N) return SG_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(C) || (K > 0 && (misaligned(A) || misaligned(B)))) return SG_ERR_MISALIGNED;
  if ((lda & 7) || (ldb & 7) || (ldc & 7)) return SG_ERR_MISALIGNED;
  return SG_OK;
}

TcParams base_params(DeviceState& d, int64_t M, int64_t N, int64_t K, int64_t ldc, void* C) {
  TcParams p{};
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.ldc = ldc;
  p.C = C;
  p.partials = d.partials;
  p.counters = d.counters;
  p.err = d.err;
  p.timeout_ns = g_timeout_ns.load();
  return p;
}

int run_tc_gemm(DeviceState& d, int dev, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                int64_t lda, int64_t ldb, int64_t ldc, bool pair, cudaStream_t stream, const void* R = nullptr,
                int64_t ldr = 0) {
  sg_plan_info plan;
  plan_tc_gemm(M, N, K, d.sm_count, pair, &plan);
  CUtensorMap ta, tb, tc;
  const uint32_t b_rows = pair ? kGemmBN / 2 : static_cast<uint32_t>(plan.tile_n);  // B rows each CTA loads per tile
  int st = make_map(&ta, A, M, K, lda, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tb, B, N, K, ldb, b_rows, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tc, C, M, N, ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, dev);
  if (st != SG_OK) return st;
  TcParams p = base_params(d, M, N, K, ldc, C);
  p.sched = sched_from_plan(plan);
  p.inject_extra_tx = g_inject_missing_tx.exchange(0);
  p.R = static_cast<const uint16_t*>(R);
  p.ldr = ldr;
  cudaError_t e = pair                              ? launch_tc_gemm_pair(ta, tb, tc, p, stream)
                  : plan.tile_n == kGemmNarrowBN ? launch_tc_gemm_narrow(ta, tb, tc, p, stream)
                                                 : launch_tc_gemm(ta, tb, tc, p, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int run_tc_swiglu(DeviceState& d, int dev, const void* A, const void* Wg, const void* Wu, void* C, int64_t M,
                  int64_t N, int64_t K, int64_t lda, int64_t ldw, int64_t ldc, bool pair, cudaStream_t stream) {
  sg_plan_info plan;
  plan_tc_swiglu(M, N, K, d.sm_count, pair, &plan);
  // each CTA loads 128 (single) or 64 (pair) rows of each of Wg and Wu per tile
  const uint32_t w_rows = pair ? kGemmBN / 4 : kGemmBN / 2;
  CUtensorMap ta, tg, tu, tc;
  int st = make_map(&ta, A, M, K, lda, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tg, Wg, N, K, ldw, w_rows, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tu, Wu, N, K, ldw, w_rows, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tc, C, M, N, ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, dev);
  if (st != SG_OK) return st;
  TcParams p = base_params(d, M, N, K, ldc, C);
  p.sched = sched_from_plan(plan);
  cudaError_t e = pair ? launch_tc_gemm_swiglu_pair(ta, tg, tu, tc, p, stream)
                       : launch_tc_gemm_swiglu(ta, tg, tu, tc, p, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int run_tc_skinny_swiglu(DeviceState& d, int dev, const void* A, const void* Wg, const void* Wu, void* C, int64_t M,
                         int64_t N, int64_t K, int64_t lda, int64_t ldw, int64_t ldc, cudaStream_t stream) {
  sg_plan_info plan;
  plan_tc_skinny(M, N, K, d.sm_count, &plan, true);
  CUtensorMap tg, tu, tx, tc;
  int st = make_map(&tg, Wg, N, K, ldw, plan.tile_m, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tu, Wu, N, K, ldw, plan.tile_m, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tx, A, M, K, lda, plan.tile_n, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tc, C, M, N, ldc, plan.tile_n, plan.tile_m, CU_TENSOR_MAP_SWIZZLE_NONE, dev);
  if (st != SG_OK) return st;
  TcParams p = base_params(d, M, N, K, ldc, C);
  p.sched = sched_from_plan(plan);
  p.prewait_steps = plan.prefetch_steps;
  cudaError_t e = launch_tc_skinny_swiglu(plan.tile_n, tg, tu, tx, tc, p, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int run_tc_skinny(DeviceState& d, int dev, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, cudaStream_t stream, const void* R = nullptr,
                  int64_t ldr = 0) {
  sg_plan_info plan;
  plan_tc_skinny(M, N, K, d.sm_count, &plan);
  CUtensorMap tw, tx, tc;
  int st = make_map(&tw, B, N, K, ldb, plan.tile_m, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tx, A, M, K, lda, plan.tile_n, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tc, C, M, N, ldc, plan.tile_n, plan.tile_m, CU_TENSOR_MAP_SWIZZLE_NONE, dev);
  if (st != SG_OK) return st;
  CUtensorMap tr;
  if (R != nullptr) {
    st = make_map(&tr, R, M, N, ldr, plan.tile_n, plan.tile_m, CU_TENSOR_MAP_SWIZZLE_NONE, dev);
    if (st != SG_OK) return st;
  }
  TcParams p = base_params(d, M, N, K, ldc, C);
  p.sched = sched_from_plan(plan);
  p.R = static_cast<const uint16_t*>(R);
  p.ldr = ldr;
  p.prewait_steps = plan.prefetch_steps;
  cudaError_t e = launch_tc_skinny(plan.tile_n, plan.tile_m, tw, tx, tc, p, stream, R ? &tr : nullptr);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int run_cc(DeviceState& d, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
           int64_t ldb, int64_t ldc, cudaStream_t stream, const void* B2 = nullptr, const void* R = nullptr,
           int64_t ldr = 0) {
  // At most 8 activation rows per launch; larger M runs as consecutive row blocks.
  for (int64_t m0 = 0; m0 < M; m0 += 8) {
    const int64_t mb = std::min<int64_t>(8, M - m0);
    sg_plan_info plan;
    plan_cc(mb, N, K, d.sm_count, &plan, B2 != nullptr);
    CcParams p{};
    p.A = static_cast<const uint16_t*>(A) + m0 * lda;
    p.B = static_cast<const uint16_t*>(B);
    p.B2 = static_cast<const uint16_t*>(B2);
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
    p.partials = d.partials;
    p.counters = d.counters;
    p.R = R ? static_cast<const uint16_t*>(R) + m0 * ldr : nullptr;
    p.ldr = ldr;
    p.prewait = plan.prefetch_steps;
    cudaError_t e = launch_cc_gemv(p, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return SG_OK;
}

// The CUDA-core kernel's CTAs for a batched launch: matrix i gets a run of
// cb[i + 1] - cb[i] of them, in proportion to its rows, at least one and at least
// enough for kCcMaxRowsPerCta rows each; any CTAs left over go, one at a time, to
// the matrix with the most rows per CTA.  Returns the total, G unless the minimums
// ask for more.
int64_t split_batch_ctas(const int64_t* N, int count, int64_t ntot, int64_t G, int32_t* cb) {
  int64_t g[kMaxBatch];
  int64_t sum = 0;
  for (int i = 0; i < count; ++i) {
    g[i] = std::max<int64_t>({1, ceil_div(N[i], kCcMaxRowsPerCta), (G * N[i]) / ntot});
    sum += g[i];
  }
  while (sum < G) {  // at most `count` rounds: each floor above lost less than one
    int best = 0;
    for (int i = 1; i < count; ++i)
      if (N[i] * g[best] > N[best] * g[i]) best = i;
    ++g[best];
    ++sum;
  }
  cb[0] = 0;
  for (int i = 0; i < count; ++i) cb[i + 1] = static_cast<int32_t>(cb[i] + g[i]);
  return sum;
}

// One launch over `count` weight matrices against the same activations A: the
// CUDA-core kernel with a run of CTAs per matrix (each CTA's rows inside one
// matrix), or the swapped tcgen05 kernel over their concatenated 64-row tiles
// (each tile inside one matrix).
int run_batched(DeviceState& d, int dev, const void* A, int64_t M, int64_t K, int64_t lda, const void* const* B,
                const int64_t* N, const int64_t* ldb, void* const* C, const int64_t* ldc, int count, int path,
                cudaStream_t stream) {
  if (path == SG_PATH_CUDA_CORE) {
    int64_t ntot = 0;
    for (int i = 0; i < count; ++i) ntot += N[i];
    for (int64_t m0 = 0; m0 < M; m0 += 8) {
      const int64_t mb = std::min<int64_t>(8, M - m0);
      sg_plan_info plan;
      plan_cc(mb, ntot, K, d.sm_count, &plan);
      CcParams p{};
      p.A = static_cast<const uint16_t*>(A) + m0 * lda;
      p.M = static_cast<int32_t>(mb);
      p.N = static_cast<int32_t>(ntot);
      p.K = static_cast<int32_t>(K);
      p.lda = lda;
      p.grid_rows = plan.tiles_m;
      p.split_k = plan.split_k;
      p.k_slice = plan.k_steps;
      p.partials = d.partials;
      p.counters = d.counters;
      p.prewait = plan.prefetch_steps;
      p.nbatch = count;
      int64_t r = 0;
      for (int i = 0; i < count; ++i) {
        p.row_begin[i] = static_cast<int32_t>(r);
        r += N[i];
        p.Bs[i] = static_cast<const uint16_t*>(B[i]);
        p.Cs[i] = static_cast<uint16_t*>(C[i]) + m0 * ldc[i];
        p.ldbs[i] = ldb[i];
        p.ldcs[i] = ldc[i];
      }
      p.row_begin[count] = static_cast<int32_t>(r);
      p.grid_rows = static_cast<int32_t>(split_batch_ctas(N, count, ntot, plan.tiles_m, p.cta_begin));
      cudaError_t e = launch_cc_gemv(p, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return SG_OK;
  }
  // tensor cores: plan over the concatenated tiles
  const int64_t rows = skinny_rows(M);
  int64_t tiles = 0;
  for (int i = 0; i < count; ++i) tiles += ceil_div(N[i], rows);
  sg_plan_info plan;
  plan_tc_skinny(M, tiles * rows, K, d.sm_count, &plan);
  TcBatchMaps maps{};
  CUtensorMap tx;
  int st = make_map(&tx, A, M, K, lda, plan.tile_n, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  TcParams p = base_params(d, M, tiles * rows, K, 0, nullptr);
  p.sched = sched_from_plan(plan);
  p.prewait_steps = plan.prefetch_steps;
  p.nbatch = count;
  int64_t t = 0;
  for (int i = 0; i < count && st == SG_OK; ++i) {
    p.tile_begin[i] = static_cast<int32_t>(t);
    t += ceil_div(N[i], rows);
    st = make_map(&maps.w[i], B[i], N[i], K, ldb[i], rows, kBK, CU_TENSOR_MAP_SWIZZLE_128B, dev);
    if (st == SG_OK) st = make_map(&maps.c[i], C[i], M, N[i], ldc[i], plan.tile_n, rows, CU_TENSOR_MAP_SWIZZLE_NONE, dev);
  }
  if (st != SG_OK) return st;
  p.tile_begin[count] = static_cast<int32_t>(t);
  cudaError_t e = launch_tc_skinny(plan.tile_n, plan.tile_m, maps.w[0], tx, maps.c[0], p, stream, nullptr, &maps);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

// NVFP4 plan: 128 x 256 tiles, 256 of K per stage, whole tiles round-robin over
// one CTA per SM in a grouped raster.
// NVFP4 kernel choice: the one-CTA kernel unless the pairs are asked for (they
// measured slower at every size tried: 64.6 against 39.6 us at 4096^3).
bool nvfp4_pair(int64_t, int path) { return path == SG_PATH_GEMM_PAIR; }

void plan_nvfp4(int64_t M, int64_t N, int64_t K, int sms, bool pair, sg_plan_info* o) {
  std::memset(o, 0, sizeof *o);
  o->path = pair ? SG_PATH_GEMM_PAIR : SG_PATH_GEMM;
  o->tile_m = pair ? 2 * kF4TileM : kF4TileM;
  o->tile_n = kF4TileN;
  o->tile_k = kF4StageK;
  o->stages = pair ? 5 : kF4Stages;
  o->cluster_size = pair ? 2 : 1;
  o->ctas_per_sm = 1;
  Schedule s{};
  s.tiles_m = static_cast<int32_t>(ceil_div(M, o->tile_m));
  s.tiles_n = static_cast<int32_t>(ceil_div(N, kF4TileN));
  s.k_steps = static_cast<int32_t>(ceil_div(K, kF4StageK));
  s.group_m = std::max<int32_t>(1, std::min<int32_t>(s.tiles_m, 8));
  const int64_t T = static_cast<int64_t>(s.tiles_m) * s.tiles_n;
  const int64_t units = pair ? sms / 2 : sms;  // clusters or CTAs
  s.grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(T, units)));
  s.dp_tiles = static_cast<int32_t>(T);
  fill_sched(o, s);
  o->split_k = 0;
  o->wave_efficiency = wave_efficiency(T, units);
}

int run_nvfp4(DeviceState& d, int dev, const void* A, const void* SFA, const void* B, const void* SFB, void* C,
              int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, float alpha,
              bool pair, cudaStream_t stream) {
  sg_plan_info plan;
  plan_nvfp4(M, N, K, d.sm_count, pair, &plan);
  const int64_t kc = ceil_div(K, 64);
  CUtensorMap ta, tb, tsa, tsb;
  int st = make_map(&ta, A, M, K / 2, lda, kF4TileM, 128, CU_TENSOR_MAP_SWIZZLE_128B, dev, 1);
  if (st == SG_OK)
    st = make_map(&tb, B, N, K / 2, ldb, pair ? kF4TileN / 2 : kF4TileN, 128, CU_TENSOR_MAP_SWIZZLE_128B, dev, 1);
  if (pair) {
    // scale atoms as rows of 256 bytes, 8 rows (4 atoms, one stage) per box
    if (st == SG_OK)
      st = make_map(&tsa, SFA, 2 * ceil_div(M, 128) * kc, 256, 256, 8, 256, CU_TENSOR_MAP_SWIZZLE_NONE, dev, 1);
    if (st == SG_OK)
      st = make_map(&tsb, SFB, 2 * ceil_div(N, 128) * kc, 256, 256, 8, 256, CU_TENSOR_MAP_SWIZZLE_NONE, dev, 1);
  }
  if (st != SG_OK) return st;
  F4Params p{};
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.kc = static_cast<int32_t>(ceil_div(K, 64));
  p.rb_n = static_cast<int32_t>(ceil_div(N, 128));
  p.ldc = ldc;
  p.C = static_cast<uint16_t*>(C);
  p.SFA = static_cast<const uint8_t*>(SFA);
  p.SFB = static_cast<const uint8_t*>(SFB);
  p.alpha = alpha;
  p.sched = sched_from_plan(plan);
  p.err = d.err;
  p.timeout_ns = g_timeout_ns.load();
  if (!pair) p.inject_extra_tx = g_inject_missing_tx.exchange(0);
  const cudaError_t e = pair ? launch_f4_gemm_pair(ta, tb, tsa, tsb, p, stream) : launch_f4_gemm(ta, tb, p, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

// C := 0 (no residual) or C := R, the value of an empty sum plus the residual.
int empty_sum(void* C, int64_t M, int64_t N, int64_t ldc, const void* R, int64_t ldr, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (R == nullptr)
    e = cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, stream);
  else if (R != C)
    e = cudaMemcpy2DAsync(C, ldc * 2, R, ldr * 2, N * 2, M, cudaMemcpyDeviceToDevice, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int skinny_dispatch(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                    int64_t ldb, int64_t ldc, int path, cudaStream_t stream, const void* R = nullptr,
                    int64_t ldr = 0) {
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (K == 0) return empty_sum(C, M, N, ldc, R, ldr, stream);
  st = ensure_workspace(*d, stream);
  if (st != SG_OK) return st;
  if (path == SG_PATH_AUTO) path = choose_skinny_path(M);
  if (path == SG_PATH_CUDA_CORE) return run_cc(*d, A, B, C, M, N, K, lda, ldb, ldc, stream, nullptr, R, ldr);
  return run_tc_skinny(*d, dev, A, B, C, M, N, K, lda, ldb, ldc, stream, R, ldr);
}

// gemm_bf16_path and gemm_bf16_residual_path after their argument checks.
int gemm_dispatch(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                  int64_t ldc, int path, cudaStream_t s, const void* R, int64_t ldr) {
  if (path == SG_PATH_AUTO && M <= 64) return skinny_dispatch(A, B, C, M, N, K, lda, ldb, ldc, SG_PATH_AUTO, s, R, ldr);
  if (path == SG_PATH_CUDA_CORE || path == SG_PATH_TENSOR_CORE)
    return skinny_dispatch(A, B, C, M, N, K, lda, ldb, ldc, path, s, R, ldr);
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (K == 0) return empty_sum(C, M, N, ldc, R, ldr, s);
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  const bool pair = path == SG_PATH_GEMM_PAIR || (path == SG_PATH_AUTO && auto_pair(M, N, K, d->sm_count));
  return run_tc_gemm(*d, dev, A, B, C, M, N, K, lda, ldb, ldc, pair, s, R, ldr);
}

// Key splits of an attention launch: when the (query tile, head, batch) units
// leave SMs idle, each unit's key blocks are cut into n_splits equal runs (one
// CTA each, at most one CTA per SM in all), provided the fp32 partial outputs
// and log-sum-exps fit the workspace's partial slots.
void attn_splits(int64_t B, int64_t Sq, int64_t Sk, int64_t H, int causal, int sms, int32_t* n_splits,
                 int32_t* split_blocks) {
  const int64_t units = ceil_div(Sq, kAttnTile) * H * B;
  const int64_t max_blocks = ceil_div(Sk, kAttnTile);  // the last query tile sees the most keys
  (void)causal;
  int64_t n = units >= sms ? 1 : std::max<int64_t>(1, sms / units);
  n = std::min<int64_t>(n, std::min<int64_t>(max_blocks, 32));
  const int64_t per_split_bytes = B * Sq * H * (kAttnHeadDim + 1) * 4 + 256;
  while (n > 1 && n * per_split_bytes > static_cast<int64_t>(kPartialBytes)) --n;
  const int64_t bps = ceil_div(max_blocks, n);
  *n_splits = static_cast<int32_t>(ceil_div(max_blocks, bps));
  *split_blocks = static_cast<int32_t>(bps);
}

// Key splits of the decode kernel: enough (batch, kv head, split) CTAs to fill the
// resident slots (two per SM, one with more than two rows), at most 32 splits (the
// combine kernel's lanes) of at least 128 keys, within the partials workspace.
// Each split's keys are a multiple of 32 (one key per lane group and warp).
void attn_decode_splits(int64_t B, int64_t Sq, int64_t Sk, int64_t H, int64_t Hkv, int64_t rows, int sms,
                        int32_t* n_splits, int32_t* keys_per_split) {
  const int64_t slots = (rows > 2 ? 1 : 2) * static_cast<int64_t>(sms);
  const int64_t units = B * Hkv;
  int64_t n = units >= slots ? 1 : slots / units;
  n = std::min<int64_t>({n, 32, std::max<int64_t>(1, ceil_div(Sk, 128))});
  const int64_t per_split_bytes = B * Sq * H * (kAttnHeadDim + 1) * 4 + 256;
  while (n > 1 && n * per_split_bytes > static_cast<int64_t>(kPartialBytes)) --n;
  const int64_t kps = ceil_div(ceil_div(Sk, n), 32) * 32;
  *keys_per_split = static_cast<int32_t>(kps);
  *n_splits = static_cast<int32_t>(ceil_div(Sk, kps));
}

// The decode kernel takes a launch whose query rows per kv head (Sq x H / Hkv) fit
// its registers.
bool attn_decode_fits(int64_t Sq, int64_t H, int64_t Hkv) { return Sq * (H / Hkv) <= kAttnDecodeMaxRows; }

// attention_bf16's choice of the decode kernel, by measurement against a
// 4096-key cache (32 query heads): one row per kv head 16.1 us against 17.1 (32
// kv heads), four rows 13.5 against 14.5 (8 kv heads; 45.6 against 68.2 at batch
// 8); two rows 18.1 against 17.5, so two rows stay on the tcgen05 kernel.
bool attn_decode_auto(int64_t Sq, int64_t H, int64_t Hkv) {
  return attn_decode_fits(Sq, H, Hkv) && Sq * (H / Hkv) != 2;
}

int run_attention(DeviceState& d, int dev, const void* Q, const void* K, const void* V, void* O, int64_t B,
                  int64_t Sq, int64_t Sk, int64_t H, int64_t Hkv, int64_t ldq, int64_t ldk, int64_t ldv,
                  int64_t ldo, int causal, float scale, int path, cudaStream_t stream) {
  if (path == SG_PATH_CUDA_CORE) {
    AttnParams p{};
    p.B = static_cast<int32_t>(B);
    p.Sq = static_cast<int32_t>(Sq);
    p.Sk = static_cast<int32_t>(Sk);
    p.H = static_cast<int32_t>(H);
    p.Hkv = static_cast<int32_t>(Hkv);
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.O = static_cast<uint16_t*>(O);
    p.ldo = ldo;
    p.err = d.err;
    p.timeout_ns = g_timeout_ns.load();
    AttnDecodeArgs a{};
    a.Q = static_cast<const uint16_t*>(Q);
    a.K = static_cast<const uint16_t*>(K);
    a.V = static_cast<const uint16_t*>(V);
    a.ldq = ldq;
    a.ldk = ldk;
    a.ldv = ldv;
    a.rows = static_cast<int32_t>(Sq * (H / Hkv));
    attn_decode_splits(B, Sq, Sk, H, Hkv, a.rows, d.sm_count, &p.n_splits, &a.keys_per_split);
    p.part_lse = d.partials;
    p.part_o = d.partials + ceil_div(static_cast<int64_t>(p.n_splits) * B * Sq * H, 64) * 64;
    cudaError_t e = launch_attn_decode(p, a, stream);
    if (e == cudaSuccess && p.n_splits > 1) e = launch_attn_combine(p, stream);
    return e == cudaSuccess ? SG_OK : cuda_fail(e);
  }
  CUtensorMap tq, tk, tv;
  int st = make_map(&tq, Q, B * Sq, H * kAttnHeadDim, ldq, kAttnTile, 64, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tk, K, B * Sk, Hkv * kAttnHeadDim, ldk, kAttnTile, 64, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st == SG_OK) st = make_map(&tv, V, B * Sk, Hkv * kAttnHeadDim, ldv, kAttnTile, 64, CU_TENSOR_MAP_SWIZZLE_128B, dev);
  if (st != SG_OK) return st;
  AttnParams p{};
  p.B = static_cast<int32_t>(B);
  p.Sq = static_cast<int32_t>(Sq);
  p.Sk = static_cast<int32_t>(Sk);
  p.H = static_cast<int32_t>(H);
  p.Hkv = static_cast<int32_t>(Hkv);
  p.q_tiles = static_cast<int32_t>(ceil_div(Sq, kAttnTile));
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.inject_extra_tx = g_inject_missing_tx.exchange(0);
  p.O = static_cast<uint16_t*>(O);
  p.ldo = ldo;
  p.err = d.err;
  p.timeout_ns = g_timeout_ns.load();
  attn_splits(B, Sq, Sk, H, causal, d.sm_count, &p.n_splits, &p.split_blocks);
  p.part_lse = d.partials;
  p.part_o = d.partials + ceil_div(static_cast<int64_t>(p.n_splits) * B * Sq * H, 64) * 64;
  cudaError_t e = launch_attention(tq, tk, tv, p, stream);
  if (e == cudaSuccess && p.n_splits > 1) e = launch_attn_combine(p, stream);
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

}  // namespace

void set_last_cuda_error(int e) { g_last_cuda_error = e; }

}  // namespace sg

using namespace sg;

extern "C" {

int gemm_bf16_path(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                   int64_t ldb, int64_t ldc, int path, sg_stream_t stream) {
  if (path < SG_PATH_AUTO || path > SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if ((path == SG_PATH_CUDA_CORE || path == SG_PATH_TENSOR_CORE) && M > 64) return SG_ERR_INVALID_ARG;
  int st = validate(A, B, C, M, N, K, lda, ldb, ldc);
  if (st != SG_OK || M == 0 || N == 0) return st;
  return gemm_dispatch(A, B, C, M, N, K, lda, ldb, ldc, path, reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

int gemm_bf16_residual_path(const void* A, const void* B, const void* R, void* C, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldr, int64_t ldc, int path, sg_stream_t stream) {
  if (path < SG_PATH_AUTO || path > SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if ((path == SG_PATH_CUDA_CORE || path == SG_PATH_TENSOR_CORE) && M > 64) return SG_ERR_INVALID_ARG;
  int st = validate(A, B, C, M, N, K, lda, ldb, ldc);
  if (st != SG_OK || M == 0 || N == 0) return st;
  if (!R || ldr < N) return SG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(R) & 15u) || (ldr & 7)) return SG_ERR_MISALIGNED;
  if (R == C && ldr != ldc) return SG_ERR_INVALID_ARG;  // in place only with the same layout
  return gemm_dispatch(A, B, C, M, N, K, lda, ldb, ldc, path, reinterpret_cast<cudaStream_t>(stream), R, ldr);
}

int gemm_bf16_residual(const void* A, const void* B, const void* R, void* C, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldr, int64_t ldc, sg_stream_t stream) {
  return gemm_bf16_residual_path(A, B, R, C, M, N, K, lda, ldb, ldr, ldc, SG_PATH_AUTO, stream);
}

int gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              int64_t ldc, sg_stream_t stream) {
  return gemm_bf16_path(A, B, C, M, N, K, lda, ldb, ldc, SG_PATH_AUTO, stream);
}

int gemv_bf16_path(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                   int64_t ldb, int64_t ldc, int path, sg_stream_t stream) {
  if (path < SG_PATH_AUTO || path > SG_PATH_TENSOR_CORE) return SG_ERR_INVALID_ARG;
  if (M > 64) return SG_ERR_INVALID_ARG;
  int st = validate(A, B, C, M, N, K, lda, ldb, ldc);
  if (st != SG_OK || M == 0 || N == 0) return st;
  return skinny_dispatch(A, B, C, M, N, K, lda, ldb, ldc, path, reinterpret_cast<cudaStream_t>(stream));
}

int gemv_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              int64_t ldc, sg_stream_t stream) {
  return gemv_bf16_path(A, B, C, M, N, K, lda, ldb, ldc, SG_PATH_AUTO, stream);
}

int gemm_bf16_swiglu_path(const void* A, const void* Wg, const void* Wu, void* C, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldw, int64_t ldc, int path, sg_stream_t stream) {
  if (path < SG_PATH_AUTO || path > SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if ((path == SG_PATH_CUDA_CORE || path == SG_PATH_TENSOR_CORE) && M > 64) return SG_ERR_INVALID_ARG;
  int st = validate(A, Wg, C, M, N, K, lda, ldw, ldc);
  if (st == SG_OK && M > 0 && N > 0 && K > 0) {
    if (!Wu) return SG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(Wu) & 15u) return SG_ERR_MISALIGNED;
  }
  if (st != SG_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* d = nullptr;
  int dev = 0;
  st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (K == 0) {  // silu(0) * 0 = 0
    cudaError_t e = cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, s);
    return e == cudaSuccess ? SG_OK : cuda_fail(e);
  }
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  if (path == SG_PATH_AUTO) path = swiglu_path(M);
  if (path == SG_PATH_CUDA_CORE) return run_cc(*d, A, Wg, C, M, N, K, lda, ldw, ldc, s, Wu);
  if (path == SG_PATH_TENSOR_CORE) return run_tc_skinny_swiglu(*d, dev, A, Wg, Wu, C, M, N, K, lda, ldw, ldc, s);
  return run_tc_swiglu(*d, dev, A, Wg, Wu, C, M, N, K, lda, ldw, ldc, path == SG_PATH_GEMM_PAIR, s);
}

int gemm_bf16_swiglu(const void* A, const void* Wg, const void* Wu, void* C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldw, int64_t ldc, sg_stream_t stream) {
  return gemm_bf16_swiglu_path(A, Wg, Wu, C, M, N, K, lda, ldw, ldc, SG_PATH_AUTO, stream);
}

int64_t nvfp4_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return -1;
  return ceil_div(rows, 128) * ceil_div(K, 64) * kF4AtomBytes;
}

int nvfp4_pack_scales(const void* plain, int64_t rows, int64_t K, int64_t ld, void* atoms, sg_stream_t stream) {
  if (rows < 0 || K < 0 || K % 16 != 0 || ld < K / 16) return SG_ERR_INVALID_ARG;
  if (rows == 0 || K == 0) return SG_OK;
  if (!plain || !atoms) return SG_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const int st = current_device_state(&d, nullptr);
  if (st != SG_OK) return st;
  const cudaError_t e = launch_f4_pack_scales(static_cast<const uint8_t*>(plain), rows, K, ld,
                                              static_cast<uint8_t*>(atoms), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SG_OK : cuda_fail(e);
}

int gemm_nvfp4_path(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc, float alpha, int path, sg_stream_t stream) {
  if (path != SG_PATH_AUTO && path != SG_PATH_GEMM && path != SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return SG_ERR_INVALID_ARG;
  if (K % 16 != 0) return SG_ERR_INVALID_ARG;  // whole 16-element scale blocks
  if (M == 0 || N == 0) return SG_OK;
  if (!C || (K > 0 && (!A || !B || !SFA || !SFB))) return SG_ERR_INVALID_ARG;
  if (ldc < N || lda < K / 2 || ldb < K / 2) return SG_ERR_INVALID_ARG;
  auto misaligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
  if (misaligned(C) || (ldc & 7)) return SG_ERR_MISALIGNED;
  if (K > 0 && (misaligned(A) || misaligned(B) || misaligned(SFA) || misaligned(SFB) || (lda & 15) || (ldb & 15)))
    return SG_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (K == 0) return empty_sum(C, M, N, ldc, nullptr, 0, s);  // +0.0 in fp16 is all zero bits
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  return run_nvfp4(*d, dev, A, SFA, B, SFB, C, M, N, K, lda, ldb, ldc, alpha, nvfp4_pair(M, path), s);
}

int gemm_nvfp4(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int64_t M, int64_t N,
               int64_t K, int64_t lda, int64_t ldb, int64_t ldc, float alpha, sg_stream_t stream) {
  return gemm_nvfp4_path(A, SFA, B, SFB, C, M, N, K, lda, ldb, ldc, alpha, SG_PATH_AUTO, stream);
}

int sg_plan_nvfp4(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t path, sg_plan_info* out) {
  if (!out || M < 0 || N < 0 || K < 0 || num_sms < 2) return SG_ERR_INVALID_ARG;
  if (path != SG_PATH_AUTO && path != SG_PATH_GEMM && path != SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  plan_nvfp4(M, N, K, num_sms, nvfp4_pair(M, path), out);
  return SG_OK;
}

int sg_plan_swiglu(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t entry, sg_plan_info* out) {
  if (!out || M < 0 || N < 0 || K < 0 || num_sms < 1) return SG_ERR_INVALID_ARG;
  if (entry < SG_PATH_AUTO || entry > SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if ((entry == SG_PATH_CUDA_CORE || entry == SG_PATH_TENSOR_CORE) && M > 64) return SG_ERR_INVALID_ARG;
  const int path = entry == SG_PATH_AUTO ? swiglu_path(M) : entry;
  if (path == SG_PATH_CUDA_CORE)
    plan_cc(std::min<int64_t>(std::max<int64_t>(M, 1), 8), N, K, num_sms, out, true);
  else if (path == SG_PATH_TENSOR_CORE)
    plan_tc_skinny(M, N, K, num_sms, out, true);
  else
    plan_tc_swiglu(M, N, K, num_sms, path == SG_PATH_GEMM_PAIR, out);
  return SG_OK;
}

int gemv_bf16_batched(const void* A, int64_t M, int64_t K, int64_t lda, const void* const* B, const int64_t* N,
                      const int64_t* ldb, void* const* C, const int64_t* ldc, int count, int path, sg_stream_t stream) {
  if (count < 1 || count > kMaxBatch || !B || !N || !ldb || !C || !ldc) return SG_ERR_INVALID_ARG;
  if (path != SG_PATH_AUTO && path != SG_PATH_CUDA_CORE && path != SG_PATH_TENSOR_CORE) return SG_ERR_INVALID_ARG;
  if (M > 64) return SG_ERR_INVALID_ARG;
  int64_t ntot = 0;
  for (int i = 0; i < count; ++i) {
    const int st = validate(A, B[i], C[i], M, N[i], K, lda, ldb[i], ldc[i]);
    if (st != SG_OK) return st;
    ntot += N[i];
  }
  if (ntot > INT32_MAX / 2) return SG_ERR_INVALID_ARG;
  if (M == 0 || ntot == 0) return SG_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (K == 0) {
    for (int i = 0; i < count && st == SG_OK; ++i)
      if (N[i] > 0) st = empty_sum(C[i], M, N[i], ldc[i], nullptr, 0, s);
    return st;
  }
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  // Automatic kernel: the CUDA-core kernel only at M = 1.  Measured on three
  // 4096 x 4096 weights (a decode step's Q, K and V): M = 1 17.8 us against 18.4
  // on tensor cores, M = 2 20.3 us against 18.4.
  if (path == SG_PATH_AUTO) path = M <= 1 ? SG_PATH_CUDA_CORE : SG_PATH_TENSOR_CORE;
  // matrices with no rows take no part
  const void* b2[kMaxBatch];
  void* c2[kMaxBatch];
  int64_t n2[kMaxBatch], lb2[kMaxBatch], lc2[kMaxBatch];
  int cnt = 0;
  for (int i = 0; i < count; ++i)
    if (N[i] > 0) {
      b2[cnt] = B[i];
      c2[cnt] = C[i];
      n2[cnt] = N[i];
      lb2[cnt] = ldb[i];
      lc2[cnt] = ldc[i];
      ++cnt;
    }
  return run_batched(*d, dev, A, M, K, lda, b2, n2, lb2, c2, lc2, cnt, path, s);
}

const char* sg_status_string(int status) {
  switch (status) {
    case SG_OK: return "SG_OK";
    case SG_ERR_INVALID_ARG: return "SG_ERR_INVALID_ARG: invalid argument";
    case SG_ERR_MISALIGNED: return "SG_ERR_MISALIGNED: pointer or leading dimension not 16-byte aligned";
    case SG_ERR_UNSUPPORTED_DEVICE: return "SG_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3 (sm_103a)";
    case SG_ERR_CUDA: return "SG_ERR_CUDA: a CUDA call failed (see sg_last_cuda_error)";
    case SG_ERR_TIMEOUT: return "SG_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    case SG_ERR_OUT_OF_MEMORY: return "SG_ERR_OUT_OF_MEMORY: workspace allocation failed";
    default: return "unknown sg_status";
  }
}

int attention_bf16(const void* Q, const void* K, const void* V, void* O, int64_t batch, int64_t seq_q,
                   int64_t seq_k, int64_t heads, int64_t kv_heads, int64_t head_dim, int64_t ldq, int64_t ldk,
                   int64_t ldv, int64_t ldo, int causal, float scale, sg_stream_t stream) {
  return attention_bf16_path(Q, K, V, O, batch, seq_q, seq_k, heads, kv_heads, head_dim, ldq, ldk, ldv, ldo, causal,
                             scale, SG_PATH_AUTO, stream);
}

int attention_bf16_path(const void* Q, const void* K, const void* V, void* O, int64_t batch, int64_t seq_q,
                        int64_t seq_k, int64_t heads, int64_t kv_heads, int64_t head_dim, int64_t ldq, int64_t ldk,
                        int64_t ldv, int64_t ldo, int causal, float scale, int path, sg_stream_t stream) {
  if (path != SG_PATH_AUTO && path != SG_PATH_TENSOR_CORE && path != SG_PATH_CUDA_CORE) return SG_ERR_INVALID_ARG;
  if (batch < 0 || seq_q < 0 || seq_k < 0 || heads < 0 || kv_heads < 0) return SG_ERR_INVALID_ARG;
  if (head_dim != kAttnHeadDim || !std::isfinite(scale)) return SG_ERR_INVALID_ARG;
  if (batch == 0 || seq_q == 0 || heads == 0) return SG_OK;
  if (kv_heads == 0 || heads % kv_heads != 0) return SG_ERR_INVALID_ARG;
  if (path == SG_PATH_CUDA_CORE && !attn_decode_fits(seq_q, heads, kv_heads)) return SG_ERR_INVALID_ARG;
  // every row index and grid size in int32
  const int64_t tiles = ceil_div(seq_q, kAttnTile) * heads * batch;
  if (batch * seq_q > INT32_MAX || batch * seq_k > INT32_MAX || heads * head_dim > INT32_MAX || tiles > INT32_MAX)
    return SG_ERR_INVALID_ARG;
  if (!O || ldo < heads * head_dim) return SG_ERR_INVALID_ARG;
  if (seq_k > 0 && (!Q || !K || !V || ldq < heads * head_dim || ldk < kv_heads * head_dim ||
                    ldv < kv_heads * head_dim))
    return SG_ERR_INVALID_ARG;
  auto misaligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
  if (misaligned(O) || (ldo & 7)) return SG_ERR_MISALIGNED;
  if (seq_k > 0 && (misaligned(Q) || misaligned(K) || misaligned(V) || (ldq & 7) || (ldk & 7) || (ldv & 7)))
    return SG_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  if (seq_k == 0) {  // no query sees a key: O = 0
    const cudaError_t e = cudaMemset2DAsync(O, ldo * 2, 0, heads * head_dim * 2, batch * seq_q, s);
    return e == cudaSuccess ? SG_OK : cuda_fail(e);
  }
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  if (path == SG_PATH_AUTO) path = attn_decode_auto(seq_q, heads, kv_heads) ? SG_PATH_CUDA_CORE : SG_PATH_TENSOR_CORE;
  return run_attention(*d, dev, Q, K, V, O, batch, seq_q, seq_k, heads, kv_heads, ldq, ldk, ldv, ldo, causal,
                       scale, path, s);
}

int sg_last_cuda_error(void) { return g_last_cuda_error; }

void sg_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns); }

void sg_debug_inject_missing_tx(uint32_t bytes) { g_inject_missing_tx.store(bytes); }

int sg_check_device_errors(sg_stream_t stream, uint32_t detail[4]) {
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (detail) std::memset(detail, 0, 4 * sizeof(uint32_t));
  if (!d->workspace) return SG_OK;
  DeviceError h{};
  e = cudaMemcpyAsync(&h, d->err, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (h.code == 0) return SG_OK;
  if (detail) {
    detail[0] = h.code;
    detail[1] = h.block;
    detail[2] = h.role;
    detail[3] = h.where;
  }
  // Clear the error word and every arrival counter an aborted launch may have left.
  e = cudaMemsetAsync(d->counters, 0, kNumCounters * sizeof(uint32_t) + sizeof(DeviceError), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  return SG_ERR_TIMEOUT;
}

int sg_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t entry, sg_plan_info* out) {
  if (!out || M < 0 || N < 0 || K < 0 || num_sms < 1) return SG_ERR_INVALID_ARG;
  if (entry < SG_PATH_AUTO || entry > SG_PATH_GEMM_PAIR) return SG_ERR_INVALID_ARG;
  if (entry == SG_PATH_GEMM || entry == SG_PATH_GEMM_PAIR || (entry == SG_PATH_AUTO && M > 64)) {
    plan_tc_gemm(M, N, K, num_sms,
                 entry == SG_PATH_GEMM_PAIR || (entry == SG_PATH_AUTO && auto_pair(M, N, K, num_sms)), out);
    return SG_OK;
  }
  if (M > 64) return SG_ERR_INVALID_ARG;
  const int path = entry == SG_PATH_AUTO ? choose_skinny_path(M) : entry;
  if (path == SG_PATH_CUDA_CORE)
    plan_cc(std::min<int64_t>(std::max<int64_t>(M, 1), 8), N, K, num_sms, out);
  else
    plan_tc_skinny(M, N, K, num_sms, out);
  return SG_OK;
}

int sg_plan_item(const sg_plan_info* plan, int32_t cta, int32_t index, int32_t out[9]) {
  if (!plan || !out || plan->path == SG_PATH_CUDA_CORE) return -1;
  const Schedule s = sched_from_plan(*plan);
  if (cta < 0 || cta >= s.grid) return -1;
  const int32_t n = item_count(s, cta);
  if (index < 0 || index >= n) return -1;
  const WorkItem w = get_item(s, cta, index);
  int32_t tm, tn;
  tile_coords(s, w.tile, tm, tn);
  const int32_t vals[9] = {w.tile, w.k0, w.k1, w.piece, w.npieces, w.slot, w.sk_index, tm, tn};
  std::memcpy(out, vals, sizeof vals);
  return n;
}

double sg_wave_efficiency(int64_t ctas, int64_t slots) { return wave_efficiency(ctas, slots); }

int sg_device_query(sg_device_info* out) {
  if (!out) return SG_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  int clk = 0, mclk = 0, bus = 0;
  cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev);
  cudaDeviceGetAttribute(&mclk, cudaDevAttrMemoryClockRate, dev);
  cudaDeviceGetAttribute(&bus, cudaDevAttrGlobalMemoryBusWidth, dev);
  out->sm_count = prop.multiProcessorCount;
  out->cc_major = prop.major;
  out->cc_minor = prop.minor;
  out->smem_optin_bytes = static_cast<int32_t>(prop.sharedMemPerBlockOptin);
  out->l2_bytes = prop.l2CacheSize;
  out->global_mem_bytes = static_cast<int64_t>(prop.totalGlobalMem);
  out->clock_khz = clk;
  out->mem_clock_khz = mclk;
  out->mem_bus_bits = bus;
  return SG_OK;
}

int sg_bench_tcgen05_peak(int64_t iters, double* tflops, double* sm_mhz, sg_stream_t stream) {
  if (iters < 16 || !tflops || !sm_mhz) return SG_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int dev = 0;
  int st = current_device_state(&d, &dev);
  if (st != SG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = ensure_workspace(*d, s);
  if (st != SG_OK) return st;
  const int grid = d->sm_count;
  unsigned long long* buf = nullptr;
  cudaError_t e = cudaMalloc(&buf, 2 * grid * sizeof(unsigned long long));
  if (e != cudaSuccess) return cuda_fail(e);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  e = launch_tc_peak(std::min<int64_t>(iters, 1024), grid, buf, buf + grid, d->err, s);  // warm-up
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) e = launch_tc_peak(iters, grid, buf, buf + grid, d->err, s);
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  std::vector<unsigned long long> h(2 * grid);
  if (e == cudaSuccess) e = cudaMemcpy(h.data(), buf, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(buf);
  if (e != cudaSuccess) return cuda_fail(e);
  const double flops = 2.0 * kBM * 256 * 16 * static_cast<double>(iters) * grid;
  *tflops = flops / (ms * 1e-3) / 1e12;
  double mhz = 0;
  for (int i = 0; i < grid; ++i) mhz += static_cast<double>(h[i]) / static_cast<double>(h[grid + i]) * 1e3;
  *sm_mhz = mhz / grid;
  return SG_OK;
}

namespace {
double median_of(std::vector<float>& v) {
  std::sort(v.begin(), v.end());
  return v.size() % 2 ? v[v.size() / 2] : 0.5 * (v[v.size() / 2 - 1] + v[v.size() / 2]);
}
}  // namespace

int sg_bench_copy(void* dst, const void* src, int64_t bytes, int32_t reps, double* gbps, sg_stream_t stream) {
  if (!dst || !src || bytes <= 0 || reps < 1 || !gbps) return SG_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  std::vector<float> t;
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);  // warm-up
  for (int i = 0; i < reps && e == cudaSuccess; ++i) {
    float ms = 0;
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    t.push_back(ms);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(e);
  *gbps = 2.0 * static_cast<double>(bytes) / (median_of(t) * 1e-3) / 1e9;
  return SG_OK;
}

int sg_bench_read(const void* src, int64_t bytes, int32_t reps, void* sink, double* gbps, sg_stream_t stream) {
  if (!src || !sink || bytes < 16 || (bytes % 16) || reps < 1 || !gbps) return SG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return SG_ERR_MISALIGNED;
  DeviceState* d = nullptr;
  int st = current_device_state(&d, nullptr);
  if (st != SG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int grid = d->sm_count * 4;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  std::vector<float> t;
  cudaError_t e = launch_read_stream(src, bytes, sink, grid, s);  // warm-up
  for (int i = 0; i < reps && e == cudaSuccess; ++i) {
    float ms = 0;
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = launch_read_stream(src, bytes, sink, grid, s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    t.push_back(ms);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(e);
  *gbps = static_cast<double>(bytes) / (median_of(t) * 1e-3) / 1e9;
  return SG_OK;
}

}  // extern "C"

// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sg_sched.cuh"

namespace sg {

struct DeviceError;

// Most weight matrices one batched skinny launch takes.
constexpr int kMaxBatch = 8;

constexpr int kBM = 128;  // MMA M (tile rows; weight rows on the swapped path)
constexpr int kBK = 64;   // bf16 per k-step: one 128-byte swizzle row
constexpr int kGemmBN = 256;
// Single-CTA tiles 128 columns wide, for GEMMs whose 128 x 128 tiles fit in one wave
// (six 32 KB stages).
constexpr int kGemmNarrowBN = 128;
constexpr int kGemmNarrowStages = 6;
// Most k pieces per tile in a GEMM split-mode plan: the pieces' 32-column chunks
// of fp32 partial sums (16 KB each) must fit the copy ring together.
constexpr int kGemmMaxSplit = 8;
constexpr int kGemmStages = 4;
constexpr int kPairStages = 6;  // paired tiles: 32 KB per stage per CTA
// Stream-K pieces per CTA that the GEMM's fixup warps take (more fall back to
// the epilogue warps; the gated GEMM's plans never give more).
constexpr int kFixupMaxJobs = 4;
// Skinny (swapped) path: two CTAs per SM, each with at most kSkinnySmemBytes of
// copy ring plus output staging (two such CTAs and their barriers fit in an SM's
// 228 KB).  A weight tile is `rows` = 64 or 128 weight rows (MMA M); each stage
// holds skinny_ksub(rows) consecutive 64-wide k boxes of it (a 64-row tile reads
// 256 contiguous bytes of each weight row per stage) plus the matching
// activation boxes; the staging holds one bf16 output tile (bn x rows).
constexpr int kSkinnyCtasPerSm = 2;
constexpr int kSkinnySmemBytes = 111 * 1024;
constexpr int skinny_ksub(int rows) { return rows == 64 ? 2 : 1; }
constexpr int skinny_stages(int bn, int rows) {
  return (kSkinnySmemBytes - bn * rows * 2) / (skinny_ksub(rows) * (rows + bn) * kBK * 2) < 2
             ? 2
             : (kSkinnySmemBytes - bn * rows * 2) / (skinny_ksub(rows) * (rows + bn) * kBK * 2);
}
// Gated skinny kernel: 64 output rows per tile, each k box a 64-row box of the
// gate weights and one of the up weights (one 64-wide k box per stage).
constexpr int skinny_stages_gated(int bn) {
  return (kSkinnySmemBytes - bn * 64 * 2) / ((2 * 64 + bn) * kBK * 2) < 2
             ? 2
             : (kSkinnySmemBytes - bn * 64 * 2) / ((2 * 64 + bn) * kBK * 2);
}
// Smallest K range a split piece of the skinny path gets (each piece's partial
// sum is written, counted and read back once).
constexpr int kSkinnyMinPieceK = 512;
// Swapped skinny kernel: k-steps of weights each CTA pulls into L2 before it waits
// for the previous launch in the stream, when the grid holds at least
// kPreWaitMinFill tenths of the resident slots.
constexpr int kPreWaitSteps = 8;
constexpr int kPreWaitMinFill = 7;
// tcgen05 kernels: warp 0 TMA producer, warp 1 MMA issuer, then the epilogue warps.

// Everything a tcgen05 launch needs besides its tensor maps.
struct TcParams {
  int32_t M, N, K;       // C is M x N (output terms)
  int64_t ldc;           // elements
  void* C;               // used by the swapped epilogue's direct stores
  Schedule sched;
  float* partials;       // Stream-K slots, 2 * grid of them
  uint32_t* counters;    // one arrival counter per Stream-K tile
  DeviceError* err;
  uint64_t timeout_ns;
  uint32_t inject_extra_tx;  // failure injection: extra bytes expected on the first stage
  const uint16_t* R;     // non-null: residual, C = A . B^T + R (R[m * ldr + n], may be C)
  int64_t ldr;
  // Batched swapped launch (nbatch > 0): weight tiles [tile_begin[i], tile_begin[i + 1])
  // belong to matrix i, read through batch maps w[i] and stored through c[i].
  int32_t nbatch;
  int32_t tile_begin[kMaxBatch + 1];
  // Swapped kernel: k-steps of its first weight tile each CTA prefetches into L2
  // before it waits for the previous launch.
  int32_t prewait_steps;
};

// Tensor maps of a batched swapped launch: matrix i's weights and output.
struct TcBatchMaps {
  CUtensorMap w[kMaxBatch];
  CUtensorMap c[kMaxBatch];
};

// Non-swapped GEMM: A-operand = A (rows M), B-operand = B (rows N), BN = 256.
cudaError_t launch_tc_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const TcParams& p, cudaStream_t stream);
cudaError_t launch_tc_gemm_narrow(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const TcParams& p, cudaStream_t stream);

// Gated GEMM: C = silu(A . G^T) * (A . U^T); each 128 x 256 B tile is 128 rows of
// G over 128 rows of U (boxes 64 x 128 each), 128 output columns per tile.
cudaError_t launch_tc_gemm_swiglu(const CUtensorMap& tmA, const CUtensorMap& tmG, const CUtensorMap& tmU,
                                  const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream);

// Gated paired GEMM: 256 x 128-output tiles on clusters of two CTAs; each CTA's
// B rows are 64 of G over 64 of U (boxes 64 x 64 each).
cudaError_t launch_tc_gemm_swiglu_pair(const CUtensorMap& tmA, const CUtensorMap& tmG, const CUtensorMap& tmU,
                                       const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream);

// Paired GEMM over clusters of two CTAs: 256 x 256 tiles, p.sched counts pairs.
cudaError_t launch_tc_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                                const TcParams& p, cudaStream_t stream);

// Swapped skinny GEMM: A-operand = weights B (rows N, tiles of `rows` in {64, 128}),
// B-operand = activations A (rows M <= bn), bn in {16, 32, 64}; tmC stores C in
// boxes of bn rows x `rows` columns.
cudaError_t launch_tc_skinny(int bn, int rows, const CUtensorMap& tmW, const CUtensorMap& tmX,
                             const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream,
                             const CUtensorMap* tmR = nullptr,  // tmR: the residual, mapped like C
                             const TcBatchMaps* batch = nullptr);


// Gated swapped skinny GEMM: C = silu(X . G^T) * (X . U^T) for M <= bn activation
// rows X; tmG / tmU map the gate / up weights in 64-row boxes.
cudaError_t launch_tc_skinny_swiglu(int bn, const CUtensorMap& tmG, const CUtensorMap& tmU, const CUtensorMap& tmX,
                                    const CUtensorMap& tmC, const TcParams& p, cudaStream_t stream);

// CUDA-core skinny kernel.
struct CcParams {
  const uint16_t* A;
  const uint16_t* B;
  const uint16_t* B2;    // non-null: gated, C = silu(A . B^T) * (A . B2^T), B2 with B's ldb
  uint16_t* C;
  int32_t M, N, K;
  int64_t lda, ldb, ldc;
  int32_t grid_rows;     // CTAs along N; CTA b owns rows [b*N/grid_rows, (b+1)*N/grid_rows)
  int32_t split_k;       // K slices; > 1 uses the partial/counter fixup
  int32_t k_slice;       // k elements per slice (multiple of 8)
  float* partials;       // split_k * M * N fp32 when split_k > 1
  uint32_t* counters;    // one per CTA row group
  const uint16_t* R;     // non-null: residual added to the result (R[m * ldr + n], may be C)
  int64_t ldr;
  // Batched launch (nbatch > 0): output rows [row_begin[i], row_begin[i + 1]) of the
  // N rows belong to matrix i (weights Bs[i], ldbs[i]; outputs Cs[i], ldcs[i]) and
  // are split over CTAs [cta_begin[i], cta_begin[i + 1]) (at least one each;
  // cta_begin[nbatch] = grid_rows).
  int32_t nbatch;
  int32_t row_begin[kMaxBatch + 1];
  int32_t cta_begin[kMaxBatch + 1];
  const uint16_t* Bs[kMaxBatch];
  uint16_t* Cs[kMaxBatch];
  int64_t ldbs[kMaxBatch];
  int64_t ldcs[kMaxBatch];
  // Non-zero: each warp prefetches its k range of the CTA's first row pass into L2
  // before it waits for the previous launch.
  int32_t prewait;
};

cudaError_t launch_cc_gemv(const CcParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- NVFP4 GEMM
// Tiles of 128 x 256 outputs; a stage is 256 fp4 of K (128 bytes per row, 4 MMAs
// of K = 64) with its scale atoms.  A scale atom is 512 bytes holding the E4M3
// scales of 128 rows x 4 blocks of 16 (64 of K): row r, block j at byte
// (r % 32) * 16 + (r / 32) * 4 + j; atom (row block R, k chunk c) of a matrix with
// kc = ceil(K / 64) chunks sits at byte (R * kc + c) * 512.
constexpr int kF4TileM = 128;
constexpr int kF4TileN = 256;
constexpr int kF4StageK = 256;
constexpr int kF4Stages = 4;
constexpr int kF4AtomBytes = 512;

struct F4Params {
  int32_t M, N, K;
  int32_t kc;            // 64-element k chunks: ceil(K / 64)
  int32_t rb_n;          // 128-row blocks of B: ceil(N / 128)
  int64_t ldc;           // elements
  uint16_t* C;           // fp16 bit patterns
  const uint8_t* SFA;    // scale atoms of A (ceil(M / 128) * kc of them)
  const uint8_t* SFB;    // scale atoms of B (rb_n * kc of them)
  float alpha;
  Schedule sched;        // whole tiles, round-robin
  DeviceError* err;
  uint64_t timeout_ns;
  uint32_t inject_extra_tx;  // failure injection (one-CTA kernel): extra bytes expected on the first stage
};

cudaError_t launch_f4_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const F4Params& p, cudaStream_t stream);

// Paired form: clusters of two CTAs, 256 x 256 tiles (p.sched counts pair tiles
// and clusters); tmB in 128-row boxes; tmSFA / tmSFB view the scale atoms as rows
// of 256 bytes in boxes of 8 rows (4 atoms).
cudaError_t launch_f4_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                               const CUtensorMap& tmSFB, const F4Params& p, cudaStream_t stream);

// Plain row-major scales (rows x K/16 bytes, pitch ld) to scale atoms; padding
// bytes (rows past `rows`, blocks past K/16) are written as 0.
cudaError_t launch_f4_pack_scales(const uint8_t* plain, int64_t rows, int64_t K, int64_t ld, uint8_t* atoms,
                                  cudaStream_t stream);

// ---------------------------------------------------------------- attention
// Fused attention forward for head dimension 128: query tiles of 128 rows, key
// blocks of 128.  Q rows are tokens b * Sq + i with head h at columns
// [128 h, 128 h + 128); K and V rows are tokens b * Sk + j with kv head g at
// columns [128 g, 128 g + 128).
constexpr int kAttnTile = 128;
constexpr int kAttnHeadDim = 128;

struct AttnParams {
  int32_t B, Sq, Sk, H, Hkv;
  int32_t q_tiles;       // ceil(Sq / 128)
  int32_t causal;        // key j visible to query i iff j <= i + (Sk - Sq)
  float scale_log2;      // softmax scale x log2(e)
  uint16_t* O;           // bf16 output, rows b * Sq + i, head h at columns 128 h
  int64_t ldo;           // elements between consecutive rows of O
  // Split along the keys (n_splits > 1): CTA split s of a tile takes key blocks
  // [s * split_blocks, (s + 1) * split_blocks) and writes its normalised fp32
  // output part_o[((s * B * Sq + row) * H + h) * 128 + d] and the log2-sum-exp
  // of its scores part_lse[(s * B * Sq + row) * H + h] (-inf: no visible key);
  // attn_combine merges the splits.
  int32_t n_splits;
  int32_t split_blocks;
  float* part_o;
  float* part_lse;
  DeviceError* err;
  uint64_t timeout_ns;
  uint32_t inject_extra_tx;  // failure injection: extra bytes expected on the first K tile
};

// Decode attention on CUDA cores (sg_attention_decode.cu): CTA (b, kv head g,
// split s) takes the rows = Sq x H / Hkv query rows of heads g H / Hkv .. and keys
// [s keys_per_split, (s + 1) keys_per_split); Q, K and V are read directly (row
// pitches ldq, ldk, ldv elements, 16-byte aligned).  With n_splits > 1 it writes
// the same partials as the tensor-core kernel for launch_attn_combine.
constexpr int kAttnDecodeMaxRows = 4;
struct AttnDecodeArgs {
  const uint16_t* Q;
  const uint16_t* K;
  const uint16_t* V;
  int64_t ldq, ldk, ldv;
  int32_t rows;
  int32_t keys_per_split;
};
cudaError_t launch_attn_decode(const AttnParams& p, const AttnDecodeArgs& a, cudaStream_t stream);

// Merges the n_splits partial results of a split launch into O (bf16).
cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t stream);

cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, cudaStream_t stream);

// Dynamic shared memory of the CUDA-core kernel for M rows over grid_rows row blocks.
int cc_smem_bytes(int64_t M, int64_t N, int grid_rows, bool gated = false);

// Records a CUDA error for sg_last_cuda_error() (this host thread).
void set_last_cuda_error(int e);

// Microbenchmark kernels.
cudaError_t launch_tc_peak(int64_t iters, int grid, unsigned long long* cycles, unsigned long long* ns,
                           DeviceError* err, cudaStream_t stream);
cudaError_t launch_read_stream(const void* src, int64_t bytes, void* sink, int grid, cudaStream_t stream);

}  // namespace sg

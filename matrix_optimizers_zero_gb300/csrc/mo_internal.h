// Internal layout shared by the host planner and the CUDA kernels.
// Nothing here is part of the public ABI (include/mo.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "mo.h"

namespace mo {

// Newton-Schulz GEMM tiling: 256 x 256 output tiles computed by a pair of
// CTAs (UMMA M=256 across the pair, N=256), 64-element (128-byte, one
// swizzle row) K blocks.
constexpr int kBM = 256;
constexpr int kBN = 256;
constexpr int kBK = 64;

// Muon prologue norm items (momentum + sum of squares): flat chunks of the
// row-major stored matrix; cast items (normalise + bf16 cast, transposed for tall
// matrices): 64 x 128 tiles of the stored matrix.
constexpr int64_t kNrmChunk = 131072;
constexpr int kPrologueCtasPerSm = 2;   // launch bound of the prologue's norm kernel
constexpr int kCastTR = 64;
constexpr int kCastTC = 128;

// Supported maximum sizes (the A and B buffers are m x m).
constexpr int64_t kMaxDim = int64_t(1) << 22;   // rows or cols
constexpr int64_t kMaxM = 65536;                 // min(rows, cols)
constexpr int kMaxNsSteps = 100;                 // Newton-Schulz iterations per step
constexpr int kMaxNsLaunches = 3 * kMaxNsSteps;  // three grouped GEMM launches per iteration

// A Newton-Schulz launch with at least this many tiles per CTA pair takes its
// tiles from a device counter; shorter ones assign them statically (pair c
// runs tiles c, c + pairs, ...). Over a long launch the static assignment
// lets the pairs drift apart until the tiles in flight span more operand
// panels than L2 holds; on short launches it is the faster of the two.
constexpr int64_t kCounterTilesPerPair = 256;
// The last launch (weight update) streams W through L2 beside its operands;
// from this many tiles per pair the drifting static assignment lets that
// stream evict X column panels (measured: +2% reads at 47 tiles per pair, +45%
// at 142), so it takes the counter earlier.
constexpr int64_t kCounterTilesPerPairLast = 128;

// Test support of muon_owner_step_coverage: per-tile execution counters and a
// forced tile schedule (mo_ns_schedule).
struct StepHooks {
  uint32_t* coverage;
  int64_t coverage_len;
  int32_t schedule;
};

// Gram products longer than this along their reduction (n) are split into
// slices of this many columns: each slice accumulates its own fp32 partial
// (tcgen05 accumulation over very long reductions drops products far below
// the running sum: measured on a 1 x 2^20 matrix, a 4% error), and a
// reduction launch sums the partials in a fixed order.
constexpr int64_t kGramSliceK = 32768;

// Number of CUtensorMap objects per matrix: X ping, X pong, A, B.
constexpr int kMapsPerMat = 4;
constexpr size_t kTensorMapBytes = 128;

// Device-side description of one matrix of the table.
struct DevMat {
  float* W;                 // [R, C] fp32
  const uint16_t* G;        // [R, C] bf16
  float* V;                 // [R, C] fp32
  uint16_t* X[2];           // [m, ldx] bf16 ping-pong Newton-Schulz iterates
  uint16_t* A;              // [m, lda] bf16 Gram
  uint16_t* B;              // [m, lda] bf16 b A + c A A; appendix form: [m, ldx] bf16 A X
  int32_t R, C;             // stored shape
  int32_t m, n;             // iteration shape (m <= n)
  int32_t ldx, lda;         // row strides in elements (multiples of 64)
  int32_t tall;             // R > C: X = V^T
  int32_t vec_ok;           // C % 4 == 0 (16-byte vector access along rows)
  int32_t cast_tiles_c;     // normalise/cast tiles along C
  float shape_scale;        // sqrt(max(1, R/C))
  float rms_scale;          // 0.2 sqrt(max(R, C)) (match_rms_adamw)
  int64_t nrm_base;         // first sum-of-squares chunk (global index)
  int64_t nrm_count;        // sum-of-squares chunks of this matrix
  int32_t gram_partial;     // a Gram slice entry: n is the slice length, X points at its first
                            // column, A is its fp32 [m, lda] partial (upper tiles, no mirror)
  int32_t pad0;
};

// One long matrix whose Gram is summed from slice partials.
struct GramReduce {
  uint16_t* A;              // [m, lda] bf16 result (upper part and mirror)
  const float* parts;       // `slices` fp32 [m, lda] partials, part_stride floats apart
  int64_t part_stride;
  int64_t block_base;       // first 64 x 64 upper block of this matrix in the launch
  int32_t m, lda, slices, pad;
};

// Newton-Schulz launch kinds beyond the public MO_PHASE_* values: the two
// m x n products of the appendix form of the iteration, B = A X and
// X' = a X + b B + c A B. Both use the MO_PHASE_UPDATE tile schedule.
constexpr int kPhaseAX = 3;
constexpr int kPhaseABX = 4;

// Identical layout to mo_tile.
struct TileRec {
  uint32_t mat;
  uint16_t tm;
  uint16_t tn;
};
static_assert(sizeof(TileRec) == 8, "TileRec layout");
static_assert(sizeof(mo_tile) == 8, "mo_tile layout");

}  // namespace mo

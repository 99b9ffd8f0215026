// Launch interface between the C-ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mo_internal.h"

namespace mo {

// ---------------------------------------------------------------- NS GEMMs
struct NsParams {
  const DevMat* mats;
  const CUtensorMap* tmaps;   // kMapsPerMat per matrix: X[0], X[1], A, B
  const TileRec* tiles;
  int* status;                // device status word
  int32_t ntiles;
  int32_t cur;                // X buffer read by this launch
  float a, b, c;
  float lr;
  float wd;
  const float* lr_dev;        // when set, the learning rate is read from this device float instead of `lr`
  int32_t lr_adjust;          // mo_lr_adjust: which per-matrix scale the update uses
  uint64_t timeout_ns;
  uint32_t* coverage;         // tests only (null otherwise): per tile, two execution counters (even, odd CTA)
  uint32_t* tile_ctr;         // this launch's tile counter (zero on entry)
  int32_t counter_tiles;      // 1: CTA pairs take tiles in list order from tile_ctr; 0: pair c runs c, c + pairs, ...
};

// 256 x 256 tiles on CTA pairs; grid must be even (two CTAs per cluster).
// phase: MO_PHASE_GRAM, MO_PHASE_POLY, MO_PHASE_UPDATE, kPhaseAX or kPhaseABX;
// last (UPDATE and ABX only) applies the weight update in the epilogue.
cudaError_t launch_ns_phase(int phase, bool last, const NsParams& p, int grid, cudaStream_t stream);
// A = bf16(sum of the slice partials) for the long matrices, upper part and
// mirror; `blocks` 64 x 64 upper blocks over the `count` records.
cudaError_t launch_gram_reduce(const GramReduce* reduces, int32_t count, int64_t blocks, int grid,
                               cudaStream_t stream);
// Writes kMapsPerMat CUtensorMap; with MO_NS_APPENDIX the B buffer is m x n.
bool encode_matrix_maps(const DevMat& d, int ns_form, void* out_maps);
cudaError_t device_status_ptr(int** out);
cudaError_t launch_bounded_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream);

// ---------------------------------------------------------------- Muon prologue
struct ProParams {
  const DevMat* mats;
  const int64_t* nrm_prefix;  // n + 1 prefix sums of the matrices' norm chunks
  const int64_t* cast_prefix; // n + 1 prefix sums of the matrices' cast tiles
  float* partials;            // one sum of squares per chunk
  uint32_t* counters;         // per matrix, zero on entry, zero again on exit
  uint32_t* ready;            // per matrix, set once its scale is final (zero on entry)
  uint32_t* abort;            // unused by the prologue (zero on entry)
  float* scales;              // 1 / (||U||_F + eps), U = V_new or G + mu V_new
  int* status;                // device status word
  int32_t n;
  int64_t nrm_total, cast_total;
  float mu, eps;
  int32_t nesterov;           // orthogonalise G + mu V_new instead of V_new
  uint64_t timeout_ns;
};
// Two launches: the momentum/norm chunks, then (programmatic dependent
// launch) the normalise/cast tiles, whose scales are final by then.
cudaError_t launch_muon_prologue(const ProParams& p, int max_grid, cudaStream_t stream);

// ---------------------------------------------------------------- RMNP
constexpr int kRmnpMaxEntries = 512;
struct RmnpEntry {
  float* W;
  const uint16_t* G;
  float* V;
  int32_t R, C;
  float scale;
  int32_t vec_ok;
};
struct RmnpParams {
  RmnpEntry e[kRmnpMaxEntries];
  int64_t row_prefix[kRmnpMaxEntries + 1];
  int32_t n;
  float lr, wd, mu, eps;
  float power;                // HTRMNP: rows scaled by max(||V_i||, eps)^(power - 1); 0 for RMNP
  const float* lr_dev;        // when set, the learning rate is read from this device float instead of `lr`
};
// Rows of at least kRmnpLongRow elements go to the CTA-per-row kernel (its
// grid: CTAs), the others to the warp-per-row kernel (grid: CTAs of 8 warps).
constexpr int kRmnpLongRow = 8192;
cudaError_t launch_rmnp(const RmnpParams& p, bool row_per_cta, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- column-cut RMNP
struct ColcutParams {
  RmnpEntry e[kRmnpMaxEntries];
  int64_t row_prefix[kRmnpMaxEntries + 1];   // prefix sums of shard rows (= partial offsets)
  int16_t first[kRmnpMaxEntries];            // first and last entry of each entry's group
  int16_t last[kRmnpMaxEntries];
  float* partials;
  int32_t n;
  float lr, wd, mu, eps;
};
cudaError_t launch_rmnp_colcut(const ColcutParams& p, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- AdamW
constexpr int kAdamMaxSegs = 256;
constexpr int kAdamItem = 4096;   // elements per work item (1024 float4)
struct AdamSeg {
  float* p;
  const float* g;
  float* m;
  float* v;
  int64_t numel;
};
struct AdamParams {
  AdamSeg s[kAdamMaxSegs];
  int64_t item_prefix[kAdamMaxSegs + 1];
  int32_t n;
  float lr, wd;
  int64_t step;              // t after the increment (>= 1)
  const float* lr_dev;       // when set, lr is read from this device float
  const int64_t* step_dev;   // when set, t is read from this device int64
  float beta1, beta2, eps;
};
cudaError_t launch_adamw(const AdamParams& p, int grid, cudaStream_t stream);

}  // namespace mo

// Host-only planning: argument validation, Newton-Schulz tile schedules and
// the Muon workspace layout. No CUDA calls, so all of it runs (and is tested)
// on a machine without a GPU.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "mo_internal.h"

namespace mo {

struct MuonLayout {
  int32_t n = 0;                     // matrices of the table; mats[n..] are Gram slice entries
  int32_t ns_form = MO_NS_GRAM;
  std::vector<DevMat> mats;          // buffer pointers hold workspace OFFSETS until bound
  // Prologue work: the momentum/norm chunks of every matrix, in table order,
  // for the norm launch; the normalise/cast tiles for the cast launch (which
  // takes them from the last matrix back). Prefix sums over the matrices.
  std::vector<int64_t> nrm_prefix, cast_prefix;   // n + 1
  std::vector<int64_t> nrm_items, cast_items;     // per matrix
  std::vector<TileRec> tiles[3];     // per phase, launch order (Gram tiles may name slice entries)
  std::vector<GramReduce> reduces;   // long matrices (pointer fields hold offsets until bound)
  int64_t reduce_blocks = 0;         // 64 x 64 upper blocks over all long matrices
  int64_t nrm_total = 0;
  int64_t cast_total = 0;
  size_t off_meta = 0, off_tmaps = 0, off_nrm_prefix = 0, off_cast_prefix = 0, off_counters = 0, off_ready = 0,
         off_abort = 0;
  size_t off_tile_ctr = 0;           // kMaxNsLaunches tile counters, one per Newton-Schulz launch of a step
  size_t off_lr = 0;                 // one fp32: the learning rate a planned step reads (mo_muon_plan)
  size_t off_reduces = 0;
  size_t off_tiles[3] = {0, 0, 0};
  size_t header_bytes = 0;           // [0, header_bytes) is uploaded by every call
  size_t off_partials = 0, off_scales = 0, off_buffers = 0;
  size_t total_bytes = 0;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int validate_matrix_table(const mo_matrix* tbl, int32_t n);
int validate_muon_params(const mo_muon_params* p);
int validate_rmnp_params(const mo_rmnp_params* p);
int validate_adamw(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* p);

// Tile schedule of one phase (MO_PHASE_*), sorted into launch order; bm is
// the output tile height (128 rows for one CTA, 256 for a CTA pair).
void build_tiles(const mo_matrix* tbl, int32_t n, int phase, int bm, std::vector<TileRec>& out);

// Gram work entries: the matrices with n <= kGramSliceK, and one slice entry
// per kGramSliceK columns of the longer ones. Entry e < n is matrix e; slice
// entries follow in (matrix, slice) order.
struct GramEntry {
  int32_t parent;
  int32_t slice;     // -1 for a whole matrix
  int64_t k0, k;     // first column and length along the reduction
};
std::vector<GramEntry> gram_slices(const mo_matrix* tbl, int32_t n);

// Gram tile schedule over the entries above (TileRec::mat = entry index).
void build_gram_tiles(const mo_matrix* tbl, int32_t n, int bm, std::vector<TileRec>& out);

// Layout of the Muon workspace for a validated table; ns_form (mo_ns_form)
// sets the size of the B buffers (m x m, or m x n for the appendix form).
void plan_muon(const mo_matrix* tbl, int32_t n, int bm, int ns_form, MuonLayout& L);

}  // namespace mo

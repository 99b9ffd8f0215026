// Host-only planning for the owner-local optimizer step (see plan.h).
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <utility>

namespace mo {

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite(float x) { return std::isfinite(x); }

struct Range {
  uintptr_t lo, hi;
};

// True if any two of the byte ranges overlap.
bool any_overlap(std::vector<Range>& r) {
  std::sort(r.begin(), r.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < r.size(); ++i)
    if (r[i].lo < r[i - 1].hi) return true;
  return false;
}

}  // namespace

int validate_matrix_table(const mo_matrix* tbl, int32_t n) {
  if (n < 0) return MO_ERR_BAD_SHAPE;
  if (n == 0) return MO_OK;
  if (!tbl) return MO_ERR_NULL_POINTER;
  std::vector<Range> written;
  std::vector<Range> read;
  written.reserve(2 * size_t(n));
  for (int32_t i = 0; i < n; ++i) {
    const mo_matrix& e = tbl[i];
    if (!e.W || !e.G || !e.V) return MO_ERR_NULL_POINTER;
    if (e.rows < 1 || e.cols < 1 || e.rows > kMaxDim || e.cols > kMaxDim) return MO_ERR_BAD_SHAPE;
    if (std::min(e.rows, e.cols) > kMaxM) return MO_ERR_BAD_SHAPE;
    if (!aligned16(e.W) || !aligned16(e.G) || !aligned16(e.V)) return MO_ERR_MISALIGNED;
    const uintptr_t el = uintptr_t(e.rows) * uintptr_t(e.cols);
    written.push_back({uintptr_t(e.W), uintptr_t(e.W) + 4 * el});
    written.push_back({uintptr_t(e.V), uintptr_t(e.V) + 4 * el});
    read.push_back({uintptr_t(e.G), uintptr_t(e.G) + 2 * el});
  }
  if (any_overlap(written)) return MO_ERR_OVERLAP;
  // a gradient must not alias any written state
  std::vector<Range> all = written;
  for (const Range& g : read) {
    auto it = std::upper_bound(all.begin(), all.end(), g.lo,
                               [](uintptr_t v, const Range& r) { return v < r.lo; });
    if (it != all.end() && it->lo < g.hi) return MO_ERR_OVERLAP;
    if (it != all.begin() && std::prev(it)->hi > g.lo) return MO_ERR_OVERLAP;
  }
  return MO_OK;
}

int validate_muon_params(const mo_muon_params* p) {
  if (!p) return MO_ERR_NULL_POINTER;
  if (!finite(p->lr) || !finite(p->wd) || !finite(p->mu) || !finite(p->a) || !finite(p->b) ||
      !finite(p->c) || !finite(p->eps))
    return MO_ERR_BAD_PARAM;
  if (p->eps < 0.f) return MO_ERR_BAD_PARAM;
  if (p->ns_steps < 1 || p->ns_steps > kMaxNsSteps) return MO_ERR_BAD_PARAM;
  if (p->ns_form != MO_NS_GRAM && p->ns_form != MO_NS_APPENDIX) return MO_ERR_BAD_PARAM;
  if (p->lr_adjust != MO_LR_ORIGINAL && p->lr_adjust != MO_LR_MATCH_RMS_ADAMW) return MO_ERR_BAD_PARAM;
  if (p->nesterov != 0 && p->nesterov != 1) return MO_ERR_BAD_PARAM;
  return MO_OK;
}

int validate_rmnp_params(const mo_rmnp_params* p) {
  if (!p) return MO_ERR_NULL_POINTER;
  if (!finite(p->lr) || !finite(p->wd) || !finite(p->mu) || !finite(p->eps) || p->eps < 0.f)
    return MO_ERR_BAD_PARAM;
  return MO_OK;
}

int validate_adamw(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* p) {
  if (!p) return MO_ERR_NULL_POINTER;
  if (!finite(p->lr) || !finite(p->wd) || !finite(p->beta1) || !finite(p->beta2) ||
      !finite(p->eps) || p->eps < 0.f)
    return MO_ERR_BAD_PARAM;
  if (p->beta1 < 0.f || p->beta1 >= 1.f || p->beta2 < 0.f || p->beta2 >= 1.f) return MO_ERR_BAD_PARAM;
  if (p->step < 1) return MO_ERR_BAD_PARAM;
  if (n < 0) return MO_ERR_BAD_SHAPE;
  if (n == 0) return MO_OK;
  if (!segs) return MO_ERR_NULL_POINTER;
  std::vector<Range> written;
  std::vector<Range> read;
  for (int32_t i = 0; i < n; ++i) {
    const mo_tail_seg& s = segs[i];
    if (s.numel < 0 || s.numel > (int64_t(1) << 40)) return MO_ERR_BAD_SHAPE;
    if (s.numel == 0) continue;
    if (!s.p || !s.g || !s.m || !s.v) return MO_ERR_NULL_POINTER;
    if (!aligned16(s.p) || !aligned16(s.g) || !aligned16(s.m) || !aligned16(s.v)) return MO_ERR_MISALIGNED;
    const uintptr_t b = 4 * uintptr_t(s.numel);
    written.push_back({uintptr_t(s.p), uintptr_t(s.p) + b});
    written.push_back({uintptr_t(s.m), uintptr_t(s.m) + b});
    written.push_back({uintptr_t(s.v), uintptr_t(s.v) + b});
    read.push_back({uintptr_t(s.g), uintptr_t(s.g) + b});
  }
  if (any_overlap(written)) return MO_ERR_OVERLAP;
  for (const Range& g : read) {
    auto it = std::upper_bound(written.begin(), written.end(), g.lo,
                               [](uintptr_t v, const Range& r) { return v < r.lo; });
    if (it != written.end() && it->lo < g.hi) return MO_ERR_OVERLAP;
    if (it != written.begin() && std::prev(it)->hi > g.lo) return MO_ERR_OVERLAP;
  }
  return MO_OK;
}

void build_tiles(const mo_matrix* tbl, int32_t n, int phase, int bm, std::vector<TileRec>& out) {
  struct Key {
    int64_t k;
    TileRec t;
  };
  std::vector<Key> keys;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t R = tbl[i].rows, C = tbl[i].cols;
    const int64_t m = std::min(R, C), nn = std::max(R, C);
    const int64_t tiles_m = ceil_div(m, bm);
    if (phase == MO_PHASE_UPDATE) {
      const int64_t tiles_n = ceil_div(nn, kBN);
      for (int64_t tm = 0; tm < tiles_m; ++tm)
        for (int64_t tn = 0; tn < tiles_n; ++tn)
          keys.push_back({m, {uint32_t(i), uint16_t(tm), uint16_t(tn)}});
    } else {
      // symmetric m x m output: keep tiles whose column range ends after the
      // first row of the tile, i.e. tiles that touch the upper triangle.
      const int64_t tiles_n = ceil_div(m, kBN);
      const int64_t k = (phase == MO_PHASE_GRAM) ? nn : m;
      for (int64_t tm = 0; tm < tiles_m; ++tm)
        for (int64_t tn = 0; tn < tiles_n; ++tn)
          if ((tn + 1) * kBN > tm * bm) keys.push_back({k, {uint32_t(i), uint16_t(tm), uint16_t(tn)}});
    }
  }
  // Longest K first, then by matrix. Within a matrix the symmetric phases go
  // row-block by row-block; the m x n products go column-block by
  // column-block, so the tiles in flight at once share a few X column panels
  // and all of B's rows (on the 8B table's 4096 x 14336 matrices the
  // row-major order kept ~70 panels of 2 MB in flight, more than L2 holds;
  // measured 5.7% faster NS there, neutral on GPT-2 Large).
  const bool col_major = phase == MO_PHASE_UPDATE;
  std::sort(keys.begin(), keys.end(), [col_major](const Key& a, const Key& b) {
    if (a.k != b.k) return a.k > b.k;
    if (a.t.mat != b.t.mat) return a.t.mat < b.t.mat;
    if (col_major) {
      if (a.t.tn != b.t.tn) return a.t.tn < b.t.tn;
      return a.t.tm < b.t.tm;
    }
    if (a.t.tm != b.t.tm) return a.t.tm < b.t.tm;
    return a.t.tn < b.t.tn;
  });
  out.resize(keys.size());
  for (size_t j = 0; j < keys.size(); ++j) out[j] = keys[j].t;
}

std::vector<GramEntry> gram_slices(const mo_matrix* tbl, int32_t n) {
  std::vector<GramEntry> out;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t nn = std::max(tbl[i].rows, tbl[i].cols);
    if (nn <= kGramSliceK) continue;
    for (int64_t k0 = 0, s = 0; k0 < nn; k0 += kGramSliceK, ++s)
      out.push_back({i, int32_t(s), k0, std::min(kGramSliceK, nn - k0)});
  }
  return out;
}

void build_gram_tiles(const mo_matrix* tbl, int32_t n, int bm, std::vector<TileRec>& out) {
  struct Key {
    int64_t k;
    TileRec t;
  };
  std::vector<Key> keys;
  auto add = [&](int64_t m, int64_t k, uint32_t idx) {
    const int64_t tiles_m = ceil_div(m, bm), tiles_n = ceil_div(m, kBN);
    for (int64_t tm = 0; tm < tiles_m; ++tm)
      for (int64_t tn = 0; tn < tiles_n; ++tn)
        if ((tn + 1) * kBN > tm * bm) keys.push_back({k, {idx, uint16_t(tm), uint16_t(tn)}});
  };
  for (int32_t i = 0; i < n; ++i) {
    const int64_t m = std::min(tbl[i].rows, tbl[i].cols), nn = std::max(tbl[i].rows, tbl[i].cols);
    if (nn <= kGramSliceK) add(m, nn, uint32_t(i));
  }
  const std::vector<GramEntry> sl = gram_slices(tbl, n);
  for (size_t j = 0; j < sl.size(); ++j) {
    const mo_matrix& t = tbl[sl[j].parent];
    add(std::min(t.rows, t.cols), sl[j].k, uint32_t(n) + uint32_t(j));
  }
  // longest reduction first, then entry, tile row, tile column
  std::sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
    if (a.k != b.k) return a.k > b.k;
    if (a.t.mat != b.t.mat) return a.t.mat < b.t.mat;
    if (a.t.tm != b.t.tm) return a.t.tm < b.t.tm;
    return a.t.tn < b.t.tn;
  });
  out.resize(keys.size());
  for (size_t j = 0; j < keys.size(); ++j) out[j] = keys[j].t;
}

void plan_muon(const mo_matrix* tbl, int32_t n, int bm, int ns_form, MuonLayout& L) {
  L.n = n;
  L.ns_form = ns_form;
  L.mats.assign(size_t(n), DevMat{});
  std::vector<int64_t> chunks(static_cast<size_t>(n), 0), casts(static_cast<size_t>(n), 0);
  int64_t nrm = 0, cast = 0;
  for (int32_t i = 0; i < n; ++i) {
    DevMat& d = L.mats[size_t(i)];
    const int64_t R = tbl[i].rows, C = tbl[i].cols;
    d.W = tbl[i].W;
    d.G = static_cast<const uint16_t*>(tbl[i].G);
    d.V = tbl[i].V;
    d.R = int32_t(R);
    d.C = int32_t(C);
    d.tall = R > C ? 1 : 0;
    d.m = int32_t(std::min(R, C));
    d.n = int32_t(std::max(R, C));
    d.ldx = int32_t(align_up(size_t(d.n), 64));
    d.lda = int32_t(align_up(size_t(d.m), 64));
    d.vec_ok = (C % 4 == 0) ? 1 : 0;
    d.cast_tiles_c = int32_t(ceil_div(C, kCastTC));
    d.shape_scale = float(std::sqrt(std::max(1.0, double(R) / double(C))));
    d.rms_scale = float(0.2 * std::sqrt(double(std::max(R, C))));
    d.nrm_base = nrm;
    d.nrm_count = ceil_div(R * C, kNrmChunk);
    chunks[size_t(i)] = d.nrm_count;
    casts[size_t(i)] = ceil_div(R, kCastTR) * ceil_div(C, kCastTC);
    nrm += d.nrm_count;
    cast += casts[size_t(i)];
  }
  L.nrm_total = nrm;
  L.cast_total = cast;
  L.nrm_items = chunks;
  L.cast_items = casts;
  L.nrm_prefix.assign(size_t(n) + 1, 0);
  L.cast_prefix.assign(size_t(n) + 1, 0);
  for (int32_t i = 0; i < n; ++i) {
    L.nrm_prefix[size_t(i) + 1] = L.nrm_prefix[size_t(i)] + chunks[size_t(i)];
    L.cast_prefix[size_t(i) + 1] = L.cast_prefix[size_t(i)] + casts[size_t(i)];
  }
  build_gram_tiles(tbl, n, bm, L.tiles[MO_PHASE_GRAM]);
  build_tiles(tbl, n, MO_PHASE_POLY, bm, L.tiles[MO_PHASE_POLY]);
  build_tiles(tbl, n, MO_PHASE_UPDATE, bm, L.tiles[MO_PHASE_UPDATE]);
  // Gram slice entries of the long matrices (buffers assigned below)
  const std::vector<GramEntry> slices = gram_slices(tbl, n);
  for (const GramEntry& e : slices) {
    DevMat d = L.mats[size_t(e.parent)];
    d.n = int32_t(e.k);
    d.gram_partial = 1;
    L.mats.push_back(d);
  }
  const size_t nall = L.mats.size();
  L.reduces.clear();
  L.reduce_blocks = 0;

  size_t off = 0;
  L.off_meta = off;
  off = align_up(off + sizeof(DevMat) * nall, 128);
  L.off_tmaps = off;
  off = align_up(off + kTensorMapBytes * kMapsPerMat * nall, 256);
  L.off_nrm_prefix = off;
  off = align_up(off + sizeof(int64_t) * L.nrm_prefix.size(), 256);
  L.off_cast_prefix = off;
  off = align_up(off + sizeof(int64_t) * L.cast_prefix.size(), 256);
  L.off_counters = off;
  off = align_up(off + sizeof(uint32_t) * size_t(n), 256);
  L.off_ready = off;
  off = align_up(off + sizeof(uint32_t) * size_t(n), 256);
  L.off_abort = off;
  off = align_up(off + sizeof(uint32_t), 256);
  L.off_tile_ctr = off;
  off = align_up(off + sizeof(uint32_t) * size_t(kMaxNsLaunches), 256);
  L.off_lr = off;
  off = align_up(off + sizeof(float), 256);
  {
    // one reduction record per long matrix
    int32_t prev = -1;
    for (const GramEntry& e : slices)
      if (e.parent != prev) {
        prev = e.parent;
        GramReduce r{};
        r.m = L.mats[size_t(e.parent)].m;
        r.lda = L.mats[size_t(e.parent)].lda;
        r.slices = int32_t(ceil_div(std::max(tbl[e.parent].rows, tbl[e.parent].cols), kGramSliceK));
        r.block_base = L.reduce_blocks;
        const int64_t nb = ceil_div(r.m, 64);
        L.reduce_blocks += nb * (nb + 1) / 2;
        L.reduces.push_back(r);
      }
  }
  L.off_reduces = off;
  off = align_up(off + sizeof(GramReduce) * L.reduces.size(), 256);
  for (int ph = 0; ph < 3; ++ph) {
    L.off_tiles[ph] = off;
    off = align_up(off + sizeof(TileRec) * L.tiles[ph].size(), 256);
  }
  L.header_bytes = off;
  L.off_partials = off;
  off = align_up(off + sizeof(float) * size_t(nrm), 256);
  L.off_scales = off;
  off = align_up(off + sizeof(float) * size_t(n), 1024);
  L.off_buffers = off;
  for (int32_t i = 0; i < n; ++i) {
    DevMat& d = L.mats[size_t(i)];
    const size_t xb = size_t(d.m) * size_t(d.ldx) * 2;
    const size_t ab = size_t(d.m) * size_t(d.lda) * 2;
    const size_t bb = (ns_form == MO_NS_APPENDIX) ? xb : ab;
    // offsets are stored in the pointer fields until the workspace is bound
    d.X[0] = reinterpret_cast<uint16_t*>(off);
    off = align_up(off + xb, 1024);
    d.X[1] = reinterpret_cast<uint16_t*>(off);
    off = align_up(off + xb, 1024);
    d.A = reinterpret_cast<uint16_t*>(off);
    off = align_up(off + ab, 1024);
    d.B = reinterpret_cast<uint16_t*>(off);
    off = align_up(off + bb, 1024);
  }
  // slice entries: X at the slice's first column of the matrix's iterates,
  // A at the slice's fp32 partial (S consecutive partials per long matrix)
  size_t r = 0;
  for (size_t j = 0; j < slices.size(); ++j) {
    const GramEntry& e = slices[j];
    const DevMat& par = L.mats[size_t(e.parent)];
    DevMat& d = L.mats[size_t(n) + j];
    d.X[0] = reinterpret_cast<uint16_t*>(reinterpret_cast<uintptr_t>(par.X[0]) + size_t(e.k0) * 2);
    d.X[1] = reinterpret_cast<uint16_t*>(reinterpret_cast<uintptr_t>(par.X[1]) + size_t(e.k0) * 2);
    d.B = par.B;
    const size_t pb = size_t(par.m) * size_t(par.lda) * 4;
    if (e.slice == 0) {   // the reduction records follow the long matrices in table order
      L.reduces[r].A = par.A;
      L.reduces[r].parts = reinterpret_cast<const float*>(off);
      L.reduces[r].part_stride = int64_t(align_up(pb, 1024) / 4);
      ++r;
    }
    d.A = reinterpret_cast<uint16_t*>(off);
    off = align_up(off + pb, 1024);
  }
  L.total_bytes = off;
}

}  // namespace mo

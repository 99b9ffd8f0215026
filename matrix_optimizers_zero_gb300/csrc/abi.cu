// extern "C" entry points of include/mo.h: validation, planning, workspace
// binding and kernel launches. No entry point allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "mo.h"
#include "mo_internal.h"
#include "plan.h"

namespace {

thread_local int t_last_cuda_error = 0;


int cuda_fail(cudaError_t e) {
  t_last_cuda_error = int(e);
  return MO_ERR_CUDA;
}

// Per-device facts looked up once: compute capability, SM count, the
// device-side status word.
struct DeviceInfo {
  int checked = 0;
  int supported = 0;
  int sms = 0;
  int* status = nullptr;
};
std::array<DeviceInfo, 64> g_dev;
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= int(g_dev.size())) return MO_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[size_t(dev)];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    int* st = nullptr;
    if ((e = mo::device_status_ptr(&st)) != cudaSuccess) return cuda_fail(e);
    d.supported = (major == 10 && minor == 3) ? 1 : 0;
    d.sms = sms;
    d.status = st;
    d.checked = 1;
  }
  if (!d.supported) return MO_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return MO_OK;
}

// ---------------------------------------------------------------- plan cache
//
// Planning a table (tile schedules, tensor maps, header image) costs about a
// millisecond of host time for the GPT-2 Large table and ~20 ms for a Llama
// 8B table, so plans are cached per (device, table, workspace address). A hit
// only re-uploads the immutable header image, from pinned memory when
// available. The header is uploaded on every call, so the workspace contents
// between calls never matter.
struct PlanEntry {
  int dev = -1;
  std::vector<mo_matrix> table;
  uintptr_t ws = 0;
  mo::MuonLayout L;                  // offsets and schedules (pointers bound to `ws`)
  std::vector<uint8_t> header;       // pageable header image
  void* pinned = nullptr;            // pinned copy of the header, or null
  cudaEvent_t uploaded = nullptr;    // recorded after the latest upload from `pinned`
  uint64_t last_use = 0;
};

constexpr size_t kPlanCacheEntries = 8;
std::mutex g_plan_mu;
std::vector<PlanEntry*> g_plans;
uint64_t g_plan_clock = 0;

bool same_table(const PlanEntry& e, int dev, const mo_matrix* tbl, int32_t n, int ns_form, const void* ws) {
  return e.dev == dev && e.ws == reinterpret_cast<uintptr_t>(ws) && e.L.ns_form == ns_form &&
         e.table.size() == size_t(n) &&
         std::memcmp(e.table.data(), tbl, sizeof(mo_matrix) * size_t(n)) == 0;
}

void free_entry(PlanEntry* e) {
  if (e->uploaded) {
    cudaEventSynchronize(e->uploaded);   // the pinned image may still be in flight
    cudaEventDestroy(e->uploaded);
  }
  if (e->pinned) cudaFreeHost(e->pinned);
  delete e;
}

// Binds a planned layout to `ws` and builds its header image.
int bind_header(mo::MuonLayout& L, void* ws, std::vector<uint8_t>& header) {
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  header.assign(L.header_bytes, 0);
  // the table's matrices, then the Gram slice entries of the long ones
  for (size_t i = 0; i < L.mats.size(); ++i) {
    mo::DevMat& d = L.mats[i];
    d.X[0] = reinterpret_cast<uint16_t*>(wsb + reinterpret_cast<uintptr_t>(d.X[0]));
    d.X[1] = reinterpret_cast<uint16_t*>(wsb + reinterpret_cast<uintptr_t>(d.X[1]));
    d.A = reinterpret_cast<uint16_t*>(wsb + reinterpret_cast<uintptr_t>(d.A));
    d.B = reinterpret_cast<uint16_t*>(wsb + reinterpret_cast<uintptr_t>(d.B));
    if (!mo::encode_matrix_maps(d, L.ns_form, header.data() + L.off_tmaps + i * mo::kMapsPerMat * mo::kTensorMapBytes))
      return cuda_fail(cudaErrorInvalidValue);
  }
  for (mo::GramReduce& r : L.reduces) {
    r.A = reinterpret_cast<uint16_t*>(wsb + reinterpret_cast<uintptr_t>(r.A));
    r.parts = reinterpret_cast<const float*>(wsb + reinterpret_cast<uintptr_t>(r.parts));
  }
  if (!L.reduces.empty())
    std::memcpy(header.data() + L.off_reduces, L.reduces.data(), sizeof(mo::GramReduce) * L.reduces.size());
  std::memcpy(header.data() + L.off_meta, L.mats.data(), sizeof(mo::DevMat) * L.mats.size());
  std::memcpy(header.data() + L.off_nrm_prefix, L.nrm_prefix.data(), sizeof(int64_t) * L.nrm_prefix.size());
  std::memcpy(header.data() + L.off_cast_prefix, L.cast_prefix.data(), sizeof(int64_t) * L.cast_prefix.size());
  for (int ph = 0; ph < 3; ++ph)
    if (!L.tiles[ph].empty())
      std::memcpy(header.data() + L.off_tiles[ph], L.tiles[ph].data(), sizeof(mo::TileRec) * L.tiles[ph].size());
  return MO_OK;
}

int build_entry(PlanEntry& E, const mo_matrix* tbl, int32_t n, void* ws) {
  const int st = bind_header(E.L, ws, E.header);
  if (st != MO_OK) return st;
  E.table.assign(tbl, tbl + n);
  E.ws = reinterpret_cast<uintptr_t>(ws);
  return MO_OK;
}

PlanEntry* find_plan(int dev, const mo_matrix* tbl, int32_t n, int ns_form, const void* ws) {
  for (PlanEntry* e : g_plans)
    if ((dev < 0 || e->dev == dev) && same_table(*e, e->dev, tbl, n, ns_form, ws)) return e;
  return nullptr;
}

// Inserts a freshly planned entry (caller holds g_plan_mu), evicting the least
// recently used one when the cache is full.
int insert_plan(PlanEntry* e, const mo_matrix* tbl, int32_t n, void* ws, bool want_pinned) {
  const int st = build_entry(*e, tbl, n, ws);
  if (st != MO_OK) return st;
  e->pinned = nullptr;
  e->uploaded = nullptr;
  if (want_pinned && cudaHostAlloc(&e->pinned, e->header.size(), cudaHostAllocDefault) == cudaSuccess) {
    std::memcpy(e->pinned, e->header.data(), e->header.size());
    if (cudaEventCreateWithFlags(&e->uploaded, cudaEventDisableTiming) != cudaSuccess) {
      e->uploaded = nullptr;
      cudaFreeHost(e->pinned);
      e->pinned = nullptr;
    }
  } else {
    e->pinned = nullptr;
    (void)cudaGetLastError();
  }
  if (g_plans.size() >= kPlanCacheEntries) {
    size_t victim = 0;
    for (size_t i = 1; i < g_plans.size(); ++i)
      if (g_plans[i]->last_use < g_plans[victim]->last_use) victim = i;
    free_entry(g_plans[victim]);
    g_plans.erase(g_plans.begin() + long(victim));
  }
  g_plans.push_back(e);
  return MO_OK;
}

}  // namespace

namespace mo {

int enqueue_muon(const mo::MuonLayout& L, uint8_t* wsb, const mo_muon_params* prm, const float* lr_dev,
                 DeviceInfo* dev, cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end,
                 const StepHooks* hooks);

// Tile-execution counters of one step (muon_owner_step_coverage): two per
// tile of every Newton-Schulz GEMM launch, launches in order.
int64_t coverage_counters(const mo::MuonLayout& L, const mo_muon_params* prm) {
  const int mid = prm->ns_form == MO_NS_APPENDIX ? MO_PHASE_UPDATE : MO_PHASE_POLY;
  return 2 * int64_t(prm->ns_steps) *
         int64_t(L.tiles[MO_PHASE_GRAM].size() + L.tiles[mid].size() + L.tiles[MO_PHASE_UPDATE].size());
}

int muon_step_impl(const mo_matrix* tbl, int32_t n, const mo_muon_params* prm, void* ws, size_t ws_bytes,
                   cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end, bool allow_pinned,
                   const StepHooks* hooks) {
  int st = mo::validate_muon_params(prm);
  if (st != MO_OK) return st;
  if ((st = mo::validate_matrix_table(tbl, n)) != MO_OK) return st;
  if (n == 0) {
    cudaError_t e;
    if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess) return cuda_fail(e);
    if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess) return cuda_fail(e);
    return MO_OK;
  }
  if (!ws) return MO_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MO_ERR_MISALIGNED;

  std::lock_guard<std::mutex> lock(g_plan_mu);
  // Host-only part first: a rejected call makes no CUDA call.
  PlanEntry* E = find_plan(-1, tbl, n, prm->ns_form, ws);
  PlanEntry* fresh = nullptr;
  if (E == nullptr) {
    fresh = new PlanEntry();
    mo::plan_muon(tbl, n, mo::kBM, prm->ns_form, fresh->L);
  }
  const size_t need = (E ? E->L : fresh->L).total_bytes;
  if (ws_bytes < need) {
    delete fresh;
    return MO_ERR_WORKSPACE_TOO_SMALL;
  }
  if (hooks != nullptr && hooks->coverage != nullptr &&
      hooks->coverage_len < coverage_counters(E ? E->L : fresh->L, prm)) {
    delete fresh;
    return MO_ERR_BAD_SHAPE;
  }
  DeviceInfo* dev = nullptr;
  int dev_id = 0;
  if ((st = device_info(&dev)) != MO_OK || cudaGetDevice(&dev_id) != cudaSuccess) {
    delete fresh;
    return st != MO_OK ? st : cuda_fail(cudaErrorInvalidDevice);
  }
  if (E != nullptr && E->dev != dev_id) {
    // same addresses on another device: look for that device's entry
    E = find_plan(dev_id, tbl, n, prm->ns_form, ws);
    if (E == nullptr) {
      fresh = new PlanEntry();
      mo::plan_muon(tbl, n, mo::kBM, prm->ns_form, fresh->L);
    }
  }
  if (E == nullptr) {
    fresh->dev = dev_id;
    if ((st = insert_plan(fresh, tbl, n, ws, allow_pinned)) != MO_OK) {
      delete fresh;
      return st;
    }
    E = fresh;
  }
  E->last_use = ++g_plan_clock;
  const mo::MuonLayout& L = E->L;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const bool use_pinned = allow_pinned && E->pinned != nullptr;
  cudaError_t e = cudaMemcpyAsync(ws, use_pinned ? E->pinned : static_cast<const void*>(E->header.data()),
                                  L.header_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (use_pinned && (e = cudaEventRecord(E->uploaded, stream)) != cudaSuccess) return cuda_fail(e);

  return enqueue_muon(L, wsb, prm, nullptr, dev, stream, ev_begin, ev_end, hooks);
}

// The prologue and Newton-Schulz launches of one step whose workspace header
// is in place; the learning rate comes from `lr_dev` when it is set.
int enqueue_muon(const mo::MuonLayout& L, uint8_t* wsb, const mo_muon_params* prm, const float* lr_dev,
                 DeviceInfo* dev, cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end,
                 const StepHooks* hooks) {
  cudaError_t e;
  uint32_t* coverage = hooks ? hooks->coverage : nullptr;
  const int32_t schedule = hooks ? hooks->schedule : MO_SCHED_AUTO;
  const mo::DevMat* d_mats = reinterpret_cast<const mo::DevMat*>(wsb + L.off_meta);
  float* d_scales = reinterpret_cast<float*>(wsb + L.off_scales);

  mo::ProParams pp{};
  pp.mats = d_mats;
  pp.nrm_prefix = reinterpret_cast<const int64_t*>(wsb + L.off_nrm_prefix);
  pp.cast_prefix = reinterpret_cast<const int64_t*>(wsb + L.off_cast_prefix);
  pp.partials = reinterpret_cast<float*>(wsb + L.off_partials);
  pp.counters = reinterpret_cast<uint32_t*>(wsb + L.off_counters);
  pp.ready = reinterpret_cast<uint32_t*>(wsb + L.off_ready);
  pp.abort = reinterpret_cast<uint32_t*>(wsb + L.off_abort);
  pp.scales = d_scales;
  pp.status = dev->status;
  pp.n = L.n;
  pp.nrm_total = L.nrm_prefix.back();
  pp.cast_total = L.cast_prefix.back();
  pp.mu = prm->mu;
  pp.eps = prm->eps;
  pp.nesterov = prm->nesterov;
  pp.timeout_ns = 2000000000ull;
  if ((e = mo::launch_muon_prologue(pp, 0, stream)) != cudaSuccess) return cuda_fail(e);
  if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess) return cuda_fail(e);

  mo::NsParams np{};
  np.mats = d_mats;
  np.tmaps = reinterpret_cast<const CUtensorMap*>(wsb + L.off_tmaps);
  np.status = dev->status;
  np.a = prm->a;
  np.b = prm->b;
  np.c = prm->c;
  np.lr = prm->lr;
  np.wd = prm->wd;
  np.lr_dev = lr_dev;
  np.lr_adjust = prm->lr_adjust;
  np.timeout_ns = 2000000000ull;
  // Launch kinds of one iteration and the tile schedule each one uses.
  const bool appendix = prm->ns_form == MO_NS_APPENDIX;
  const int kinds[3] = {MO_PHASE_GRAM, appendix ? mo::kPhaseAX : MO_PHASE_POLY,
                        appendix ? mo::kPhaseABX : MO_PHASE_UPDATE};
  const int sched[3] = {MO_PHASE_GRAM, appendix ? MO_PHASE_UPDATE : MO_PHASE_POLY, MO_PHASE_UPDATE};
  int cur = 0;
  for (int it = 0; it < prm->ns_steps; ++it) {
    np.cur = cur;
    for (int k = 0; k < 3; ++k) {
      np.tiles = reinterpret_cast<const mo::TileRec*>(wsb + L.off_tiles[sched[k]]);
      np.ntiles = int32_t(L.tiles[sched[k]].size());
      const bool last = (k == 2) && (it == prm->ns_steps - 1);
      const int grid = 2 * std::max(1, std::min(np.ntiles, dev->sms / 2));
      np.coverage = coverage;
      if (coverage != nullptr) coverage += 2 * size_t(np.ntiles);
      np.tile_ctr = reinterpret_cast<uint32_t*>(wsb + L.off_tile_ctr) + (3 * it + k);
      np.counter_tiles = schedule == MO_SCHED_COUNTER ? 1
                         : schedule == MO_SCHED_STATIC ? 0
                         : (int64_t(np.ntiles) >= (last ? mo::kCounterTilesPerPairLast : mo::kCounterTilesPerPair) *
                                                         int64_t(grid / 2)
                                ? 1 : 0);
      if ((e = mo::launch_ns_phase(kinds[k], last, np, grid, stream)) != cudaSuccess) return cuda_fail(e);
      if (k == 0 && L.reduce_blocks > 0) {
        // long matrices: A = sum of the slice partials
        const int rgrid = int(std::max<int64_t>(1, std::min<int64_t>(L.reduce_blocks, int64_t(dev->sms) * 4)));
        if ((e = mo::launch_gram_reduce(reinterpret_cast<const mo::GramReduce*>(wsb + L.off_reduces),
                                        int32_t(L.reduces.size()), L.reduce_blocks, rgrid, stream)) != cudaSuccess)
          return cuda_fail(e);
      }
    }
    cur ^= 1;
  }
  if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess) return cuda_fail(e);
  return MO_OK;
}

}  // namespace mo

namespace {

int rmnp_impl(const mo_matrix* tbl, const float* scales, int32_t n, const mo_rmnp_params* prm, float power,
              const float* lr_dev, cudaStream_t stream) {
  int st = mo::validate_rmnp_params(prm);
  if (st != MO_OK) return st;
  if (!std::isfinite(power) || power < 0.f || power > 1.f) return MO_ERR_BAD_PARAM;
  if ((st = mo::validate_matrix_table(tbl, n)) != MO_OK) return st;
  if (scales)
    for (int32_t i = 0; i < n; ++i)
      if (!std::isfinite(scales[i])) return MO_ERR_BAD_PARAM;
  if (n == 0) return MO_OK;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MO_OK) return st;
  static thread_local mo::RmnpParams rp;   // ~25 KB: keep off the stack
  // Two passes over the table: entries with short rows (warp per row), then
  // entries with long rows (CTA per row); up to kRmnpMaxEntries per launch.
  for (int pass = 0; pass < 2; ++pass) {
    const bool long_rows = pass == 1;
    int32_t b = 0;
    while (b < n) {
      std::memset(&rp, 0, sizeof(rp));
      rp.lr = prm->lr;
      rp.wd = prm->wd;
      rp.lr_dev = lr_dev;
      rp.mu = prm->mu;
      rp.eps = prm->eps;
      rp.power = power;
      int64_t rows = 0;
      int32_t cnt = 0;
      for (; b < n && cnt < mo::kRmnpMaxEntries; ++b) {
        const mo_matrix& t = tbl[b];
        if ((t.cols >= mo::kRmnpLongRow) != long_rows) continue;
        mo::RmnpEntry& E = rp.e[cnt];
        E.W = t.W;
        E.G = static_cast<const uint16_t*>(t.G);
        E.V = t.V;
        E.R = int32_t(t.rows);
        E.C = int32_t(t.cols);
        E.scale = scales ? scales[b] : float(std::sqrt(std::max(1.0, double(t.rows) / double(t.cols))));
        E.vec_ok = (t.cols % 4 == 0) ? 1 : 0;
        rp.row_prefix[cnt] = rows;
        rows += t.rows;
        ++cnt;
      }
      rp.n = cnt;
      rp.row_prefix[cnt] = rows;
      if (cnt == 0) continue;
      const int64_t ctas = long_rows ? rows : (rows + 7) / 8;
      const int grid = int(std::max<int64_t>(1, std::min<int64_t>(ctas, int64_t(dev->sms) * 8)));
      cudaError_t e = mo::launch_rmnp(rp, long_rows, grid, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  return MO_OK;
}

}  // namespace

namespace mo {
void note_cuda_error(int e) { t_last_cuda_error = e; }
}  // namespace mo

// A Muon step planned once: the layout bound to its workspace (header
// uploaded at creation) and the hyperparameters.
struct mo_muon_plan_s {
  int dev = -1;
  mo::MuonLayout L;
  mo_muon_params params{};
  uint8_t* ws = nullptr;
};

namespace {

// AdamW over the segments; t and lr by value, or from device memory when
// step_dev / lr_dev are set (the kernel forms the per-step factors either way).
int adamw_impl(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* params, const int64_t* step_dev,
               const float* lr_dev, cudaStream_t stream) {
  DeviceInfo* dev = nullptr;
  const int st = device_info(&dev);
  if (st != MO_OK) return st;
  static thread_local mo::AdamParams ap;
  int32_t i = 0;
  while (i < n) {
    std::memset(&ap, 0, sizeof(ap));
    ap.lr = params->lr;
    ap.wd = params->wd;
    ap.step = params->step;
    ap.lr_dev = lr_dev;
    ap.step_dev = step_dev;
    ap.beta1 = params->beta1;
    ap.beta2 = params->beta2;
    ap.eps = params->eps;
    int32_t cnt = 0;
    int64_t items = 0;
    for (; i < n && cnt < mo::kAdamMaxSegs; ++i) {
      const mo_tail_seg& s = segs[i];
      if (s.numel == 0) continue;
      ap.s[cnt] = mo::AdamSeg{s.p, s.g, s.m, s.v, s.numel};
      ap.item_prefix[cnt] = items;
      items += (s.numel + mo::kAdamItem - 1) / mo::kAdamItem;
      ++cnt;
    }
    ap.item_prefix[cnt] = items;
    ap.n = cnt;
    if (cnt == 0) break;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items, int64_t(dev->sms) * 8)));
    cudaError_t e = mo::launch_adamw(ap, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return MO_OK;
}

}  // namespace

extern "C" {

int mo_muon_plan_create(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, void* ws, size_t ws_bytes,
                        cudaStream_t stream, mo_muon_plan* out) {
  if (!out) return MO_ERR_NULL_POINTER;
  int st = mo::validate_muon_params(params);
  if (st != MO_OK) return st;
  if ((st = mo::validate_matrix_table(tbl, n)) != MO_OK) return st;
  if (n == 0) return MO_ERR_BAD_SHAPE;
  if (!ws) return MO_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MO_ERR_MISALIGNED;
  mo_muon_plan_s* P = new mo_muon_plan_s();
  mo::plan_muon(tbl, n, mo::kBM, params->ns_form, P->L);
  if (ws_bytes < P->L.total_bytes) {
    delete P;
    return MO_ERR_WORKSPACE_TOO_SMALL;
  }
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MO_OK || cudaGetDevice(&P->dev) != cudaSuccess) {
    delete P;
    return st != MO_OK ? st : cuda_fail(cudaErrorInvalidDevice);
  }
  std::vector<uint8_t> header;
  if ((st = bind_header(P->L, ws, header)) != MO_OK) {
    delete P;
    return st;
  }
  std::memcpy(header.data() + P->L.off_lr, &params->lr, sizeof(float));
  // pageable source: the copy is staged before cudaMemcpyAsync returns
  const cudaError_t e = cudaMemcpyAsync(ws, header.data(), P->L.header_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) {
    delete P;
    return cuda_fail(e);
  }
  P->params = *params;
  P->ws = static_cast<uint8_t*>(ws);
  *out = P;
  return MO_OK;
}

int mo_muon_plan_step(mo_muon_plan plan, cudaStream_t stream) {
  if (!plan) return MO_ERR_NULL_POINTER;
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != MO_OK) return st;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->dev) return MO_ERR_BAD_PARAM;
  const mo::MuonLayout& L = plan->L;
  // the prologue's counters and flags and the Newton-Schulz tile counters
  // start from zero (a per-call upload would have reset them)
  cudaError_t e = cudaMemsetAsync(plan->ws + L.off_counters, 0, L.off_lr - L.off_counters, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return mo::enqueue_muon(L, plan->ws, &plan->params, reinterpret_cast<const float*>(plan->ws + L.off_lr), dev,
                          stream, nullptr, nullptr, nullptr);
}

float* mo_muon_plan_lr_ptr(mo_muon_plan plan) {
  return plan ? reinterpret_cast<float*>(plan->ws + plan->L.off_lr) : nullptr;
}

int mo_muon_plan_destroy(mo_muon_plan plan) {
  delete plan;
  return MO_OK;
}

size_t mo_muon_workspace_bytes(const mo_matrix* tbl, int32_t n, const mo_muon_params* params) {
  if (mo::validate_muon_params(params) != MO_OK) return 0;
  if (mo::validate_matrix_table(tbl, n) != MO_OK) return 0;
  if (n == 0) return 0;
  mo::MuonLayout L;
  mo::plan_muon(tbl, n, mo::kBM, params->ns_form, L);
  return L.total_bytes;
}

int muon_owner_step(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  return mo::muon_step_impl(tbl, n, params, ws, ws_bytes, stream, nullptr, nullptr, true, nullptr);
}

int muon_owner_step_timed(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, void* ws,
                          size_t ws_bytes, cudaStream_t stream, cudaEvent_t ev_ns_begin, cudaEvent_t ev_ns_end) {
  return mo::muon_step_impl(tbl, n, params, ws, ws_bytes, stream, ev_ns_begin, ev_ns_end, true, nullptr);
}

int muon_owner_step_coverage(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, void* ws,
                             size_t ws_bytes, uint32_t* coverage, int64_t coverage_len, int32_t schedule,
                             int64_t* needed, cudaStream_t stream) {
  if (!needed) return MO_ERR_NULL_POINTER;
  if (schedule != MO_SCHED_AUTO && schedule != MO_SCHED_STATIC && schedule != MO_SCHED_COUNTER)
    return MO_ERR_BAD_PARAM;
  int st = mo::validate_muon_params(params);
  if (st != MO_OK) return st;
  if ((st = mo::validate_matrix_table(tbl, n)) != MO_OK) return st;
  if (n == 0) {
    *needed = 0;
    return MO_OK;
  }
  mo::MuonLayout L;
  mo::plan_muon(tbl, n, mo::kBM, params->ns_form, L);
  *needed = mo::coverage_counters(L, params);
  if (coverage == nullptr) return MO_OK;   // size query
  const mo::StepHooks hooks{coverage, coverage_len, schedule};
  return mo::muon_step_impl(tbl, n, params, ws, ws_bytes, stream, nullptr, nullptr, true, &hooks);
}

int rmnp_step(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, cudaStream_t stream) {
  return rmnp_impl(tbl, nullptr, n, params, 0.0f, nullptr, stream);
}

int rmnp_step_scaled(const mo_matrix* tbl, const float* scales, int32_t n, const mo_rmnp_params* params,
                     cudaStream_t stream) {
  if (n > 0 && !scales) return MO_ERR_NULL_POINTER;
  return rmnp_impl(tbl, scales, n, params, 0.0f, nullptr, stream);
}

int htrmnp_step(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, float power, cudaStream_t stream) {
  return rmnp_impl(tbl, nullptr, n, params, power, nullptr, stream);
}

int rmnp_step_dev(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, float power, const float* d_lr,
                  cudaStream_t stream) {
  if (!d_lr || !params) return MO_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(d_lr) & 3u) != 0) return MO_ERR_MISALIGNED;
  mo_rmnp_params q = *params;   // lr comes from device memory
  q.lr = 0.0f;
  return rmnp_impl(tbl, nullptr, n, &q, power, d_lr, stream);
}

size_t mo_rmnp_colcut_workspace_bytes(const mo_matrix* shards, int32_t n) {
  if (mo::validate_matrix_table(shards, n) != MO_OK) return 0;
  int64_t rows = 0;
  for (int32_t i = 0; i < n; ++i) rows += shards[i].rows;
  return size_t((rows * 4 + 255) / 256 * 256);
}

int rmnp_colcut_step(const mo_matrix* shards, const int32_t* group, const float* scales, int32_t n,
                     const mo_rmnp_params* params, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int st = mo::validate_rmnp_params(params);
  if (st != MO_OK) return st;
  if ((st = mo::validate_matrix_table(shards, n)) != MO_OK) return st;
  if (n > mo::kRmnpMaxEntries) return MO_ERR_BAD_SHAPE;
  if (n == 0) return MO_OK;
  if (!group || !scales || !ws) return MO_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return MO_ERR_MISALIGNED;
  for (int32_t i = 0; i < n; ++i) {
    if (!std::isfinite(scales[i])) return MO_ERR_BAD_PARAM;
    if (i > 0 && group[i] != group[i - 1]) {
      for (int32_t j = 0; j < i; ++j)
        if (group[j] == group[i]) return MO_ERR_BAD_PARAM;   // a group must be consecutive
    }
    if (i > 0 && group[i] == group[i - 1] && shards[i].rows != shards[i - 1].rows) return MO_ERR_BAD_SHAPE;
  }
  if (ws_bytes < mo_rmnp_colcut_workspace_bytes(shards, n)) return MO_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != MO_OK) return st;
  static thread_local mo::ColcutParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.n = n;
  cp.lr = params->lr;
  cp.wd = params->wd;
  cp.mu = params->mu;
  cp.eps = params->eps;
  cp.partials = static_cast<float*>(ws);
  int64_t rows = 0;
  for (int32_t i = 0; i < n; ++i) {
    const mo_matrix& t = shards[i];
    mo::RmnpEntry& E = cp.e[i];
    E.W = t.W;
    E.G = static_cast<const uint16_t*>(t.G);
    E.V = t.V;
    E.R = int32_t(t.rows);
    E.C = int32_t(t.cols);
    E.scale = scales[i];
    E.vec_ok = (t.cols % 4 == 0) ? 1 : 0;
    cp.row_prefix[i] = rows;
    rows += t.rows;
    int32_t a = i, b = i;
    while (a > 0 && group[a - 1] == group[i]) --a;
    while (b + 1 < n && group[b + 1] == group[i]) ++b;
    cp.first[i] = int16_t(a);
    cp.last[i] = int16_t(b);
  }
  cp.row_prefix[n] = rows;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, int64_t(dev->sms) * 8)));
  cudaError_t e = mo::launch_rmnp_colcut(cp, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return MO_OK;
}


int adamw_tail_step(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* params, cudaStream_t stream) {
  const int st = mo::validate_adamw(segs, n, params);
  if (st != MO_OK) return st;
  if (n == 0) return MO_OK;
  return adamw_impl(segs, n, params, nullptr, nullptr, stream);
}

int adamw_tail_step_dev(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* params, const int64_t* d_step,
                        const float* d_lr, cudaStream_t stream) {
  if (!params) return MO_ERR_NULL_POINTER;
  mo_adamw_params q = *params;   // the values read from device memory are not validated here
  q.step = 1;
  if (d_lr) q.lr = 0.0f;
  const int st = mo::validate_adamw(segs, n, &q);
  if (st != MO_OK) return st;
  params = &q;
  if (!d_step) return MO_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(d_step) & 7u) != 0 || (reinterpret_cast<uintptr_t>(d_lr) & 3u) != 0)
    return MO_ERR_MISALIGNED;
  if (n == 0) return MO_OK;
  return adamw_impl(segs, n, params, d_step, d_lr, stream);
}

int mo_last_device_error(cudaStream_t stream) {
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != MO_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int val = 0;
  if ((e = cudaMemcpy(&val, dev->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (val != 0) {
    const int zero = 0;
    if ((e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e);
  }
  return val;
}

int mo_last_cuda_error(void) { return t_last_cuda_error; }

const char* mo_status_string(int status) {
  switch (status) {
    case MO_OK: return "ok";
    case MO_ERR_NULL_POINTER: return "null pointer";
    case MO_ERR_BAD_SHAPE: return "bad shape or size";
    case MO_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MO_ERR_BAD_PARAM: return "hyperparameter NaN/Inf or out of range";
    case MO_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MO_ERR_OVERLAP: return "written buffers overlap";
    case MO_ERR_CUDA: return "CUDA runtime error";
    case MO_ERR_DEVICE_TIMEOUT: return "bounded device-side wait expired";
    case MO_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103";
    case MO_ERR_SCRATCH_LIMIT: return "table needs more scratch than the built-in array holds (mo_static_scratch_bytes)";
    default: return "unknown status";
  }
}

int mo_abi_version(void) { return MO_ABI_VERSION; }

int mo_muon_tile_schedule(const mo_matrix* tbl, int32_t n, int32_t phase, mo_tile* out, int64_t cap,
                          int64_t* count) {
  if (!count) return MO_ERR_NULL_POINTER;
  if (phase < 0 || phase > 2) return MO_ERR_BAD_PARAM;
  int st = mo::validate_matrix_table(tbl, n);
  if (st != MO_OK) return st;
  std::vector<mo::TileRec> tiles;
  if (phase == MO_PHASE_GRAM) {
    // slice entries are reported with their matrix's index
    mo::build_gram_tiles(tbl, n, mo::kBM, tiles);
    const std::vector<mo::GramEntry> sl = mo::gram_slices(tbl, n);
    for (mo::TileRec& t : tiles)
      if (t.mat >= uint32_t(n)) t.mat = uint32_t(sl[t.mat - uint32_t(n)].parent);
  } else {
    mo::build_tiles(tbl, n, phase, mo::kBM, tiles);
  }
  *count = int64_t(tiles.size());
  if (cap < int64_t(tiles.size())) return MO_ERR_BAD_SHAPE;
  if (!tiles.empty()) {
    if (!out) return MO_ERR_NULL_POINTER;
    std::memcpy(out, tiles.data(), tiles.size() * sizeof(mo_tile));
  }
  return MO_OK;
}

int mo_selftest_bounded_wait(int64_t timeout_ns, cudaStream_t stream) {
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != MO_OK) return st;
  const int64_t t = std::min<int64_t>(std::max<int64_t>(timeout_ns, 1000), 10000000000ll);
  cudaError_t e = mo::launch_bounded_wait_selftest(dev->status, uint64_t(t), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return MO_OK;
}

}  // extern "C"

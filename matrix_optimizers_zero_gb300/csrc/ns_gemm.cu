// Grouped Newton-Schulz GEMMs on the 5th-generation tensor cores (sm_103a).
//
// One launch computes one of the three products of a quintic iteration for
// every matrix of the owner's table ("Optimizers In A Sharded World", section
// 1 and appendix: five iterations of three products; the coefficients
// (a, b, c) and the wide orientation m <= n):
//   GRAM    A  = X X^T              (upper-triangle tiles, mirrored store)
//   POLY    B  = b A + c (A A)      (upper-triangle tiles, mirrored store)
//   UPDATE  X' = a X + B X          (all tiles; the last iteration applies
//                                    W <- W (1 - lr wd) - lr s X' instead)
// X0 = bf16(V / (||V||_F + eps)) is written by the prologue.
//
// Kernel structure: persistent clusters of two CTAs on two SMs (tcgen05
// cta_group::2), 256 x 256 output tiles, taken in list order from a counter
// per launch on long launches (the even CTA takes them and shares them with
// its peer through a ring in shared memory) and assigned statically on short
// ones, 10 warps per CTA:
//   warp 0      TMA producer: this CTA's 128-row halves of the A and B
//               operands in 64 x 64 boxes (128-byte swizzle) into a 6-stage
//               shared-memory ring; completion counted on the even CTA's
//               barriers
//   warp 1      TMEM allocation (both CTAs); the even CTA's lane 0 issues
//               tcgen05.mma (M=256, N=256, K=16, fp32 accumulate) and
//               multicasts the completion commits to both CTAs
//   warps 2-9   epilogue: tcgen05.ld of this CTA's accumulator rows (one TMEM
//               lane and 128 columns per thread), fused arithmetic, stores
// The two 256-column accumulators in TMEM let the epilogue of one tile run
// under the main loop of the next.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "kernels.h"
#include "mo_internal.h"
#include "ptx.cuh"

namespace mo {

__device__ int g_mo_status = 0;

namespace {

constexpr uint32_t kBoxBytes = 64 * 64 * 2;                 // one TMA box: 64 x 64 bf16
constexpr int kEpiWarps = 8;                                 // two per TMEM lane quarter
constexpr int kEpiCols = kBN / 2;                            // accumulator columns per epilogue thread
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;                         // 2 accumulators x 256 fp32 columns
static_assert(kBM == 256 && kBN == 256 && kBK == 64, "tile shape baked into the descriptors");

// ------------------------------------------------------------------ epilogues
// Each epilogue thread owns one accumulator row (TMEM lane) and kEpiCols
// consecutive columns of it, processed in chunks of 32. Operand loads for the
// next chunk are issued before the current chunk's accumulator is read, and
// every load of a chunk is issued before its stores. Row accesses use 32-byte
// vectors: a warp instruction then moves whole 32-byte sectors (one per row),
// which measurably leaves more L2 bandwidth to the TMA operand stream than
// 16-byte accesses do.

// Loads the 32 bf16 values of `row_ptr[col0 .. col0+32)` as two 32-byte
// vectors when the whole chunk is inside the row (valid = row in range).
__device__ __forceinline__ void prefetch_chunk(const uint16_t* row_ptr, int col0, int ncols, bool valid,
                                               uint32_t (&dst)[16]) {
  if (valid && col0 + 32 <= ncols) {
    uint32_t (&lo)[8] = *reinterpret_cast<uint32_t (*)[8]>(&dst[0]);
    uint32_t (&hi)[8] = *reinterpret_cast<uint32_t (*)[8]>(&dst[8]);
    ptx::ld_global_v8(row_ptr + col0, lo);
    ptx::ld_global_v8(row_ptr + col0 + 16, hi);
  }
}

__device__ __forceinline__ void chunk_operand(const uint16_t* row_ptr, int col0, int ncols,
                                              const uint32_t (&pre)[16], float (&x)[32]) {
  if (col0 + 32 <= ncols) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      x[2 * j] = bf16_bits_to_float(pre[j] & 0xFFFFu);
      x[2 * j + 1] = bf16_bits_to_float(pre[j] >> 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = (col0 + i < ncols) ? bf16_bits_to_float(row_ptr[col0 + i]) : 0.0f;
  }
}

// Stores 32 values as bf16 with two 32-byte vectors.
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float (&v)[32]) {
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    lo[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    hi[j] = pack_bf16x2(v[16 + 2 * j], v[16 + 2 * j + 1]);
  }
  ptx::st_global_v8(dst, lo);
  ptx::st_global_v8(dst + 16, hi);
}

__device__ __forceinline__ void tmem_chunk(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  __syncwarp();
  ptx::tmem_ld_32x32b_x32(taddr, r);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Pulls the W elements the last update's epilogue will read for this
// thread's row and 128 columns into L2 while the main loop still runs.
__device__ __forceinline__ void prefetch_w_rows(const DevMat& M, int row, int cbase) {
  const int lane = int(threadIdx.x & 31);
  if (row >= M.m || cbase >= M.n) return;
  if (!M.tall) {
    const float* w = M.W + size_t(row) * size_t(M.C) + cbase;
    const int cols = min(kEpiCols, M.n - cbase);
    for (int c = 0; c < cols; c += 32) ptx::prefetch_l2(w + c);
  } else {
    // W is [n, m]: the warp's 32 rows are one 128-byte line per column
    const int row_base = row - lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = cbase + lane * 4 + q;
      if (col < M.n) ptx::prefetch_l2(M.W + size_t(col) * size_t(M.C) + row_base);
    }
  }
}

// GRAM: A = acc.  POLY: B = b A + c acc.  Stored bf16 to the upper triangle
// (col >= row) and mirrored to the strict lower triangle, so every element of
// the symmetric result is written exactly once. The mirrored stores are one
// element per lane; across a warp (32 consecutive rows) each is one
// contiguous 64-byte segment. (Staging the mirror through shared memory was
// measured slower: the main loop needs the shared-memory bandwidth.)
template <int PHASE>
__device__ __forceinline__ void epilogue_symmetric(const NsParams& p, const DevMat& M, int row, int cbase,
                                                   uint32_t tb) {
  const int m = M.m;
  const size_t ld = size_t(M.lda);
  const bool rv = row < m;
  uint16_t* out = (PHASE == MO_PHASE_GRAM) ? M.A : M.B;
  const uint16_t* a_row = M.A + size_t(rv ? row : 0) * ld;
  uint32_t pre[16], nxt[16];
  if (PHASE == MO_PHASE_POLY) prefetch_chunk(a_row, cbase, m, rv, nxt);
#pragma unroll 1
  for (int ch = 0; ch < kEpiCols / 32; ++ch) {
    const int col0 = cbase + ch * 32;
    if (PHASE == MO_PHASE_POLY) {
#pragma unroll
      for (int q = 0; q < 16; ++q) pre[q] = nxt[q];
      if (ch + 1 < kEpiCols / 32) prefetch_chunk(a_row, col0 + 32, m, rv, nxt);
    }
    float v[32];
    tmem_chunk(tb + uint32_t(ch * 32), v);
    if (!rv || col0 >= m) continue;
    if (PHASE == MO_PHASE_GRAM && M.gram_partial) {
      // a slice of a long Gram: the fp32 tile as is (no rounding, no mirror)
      float* o = reinterpret_cast<float*>(M.A) + size_t(row) * ld + col0;
      if (col0 + 32 <= m) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) w8[j] = __float_as_uint(v[8 * q + j]);
          ptx::st_global_v8(o + 8 * q, w8);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < m) o[i] = v[i];
      }
      continue;
    }
    if (PHASE == MO_PHASE_POLY) {
      float a[32];
      chunk_operand(a_row, col0, m, pre, a);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = fmaf(p.b, a[i], p.c * v[i]);
    }
    uint16_t* o_row = out + size_t(row) * ld + col0;
    if (col0 + 32 <= m && col0 >= row) {
      store_bf16x32(o_row, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i >= row && col0 + i < m) o_row[i] = float_to_bf16_bits(v[i]);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int col = col0 + i;
      if (col > row && col < m) out[size_t(col) * ld + row] = float_to_bf16_bits(v[i]);
    }
  }
}

// UPDATE: X' = a X + acc (bf16 to the other X buffer), or in the last
// iteration W <- W decay - lr s X' on the stored orientation (decay = 1 - lr wd).
template <int PHASE, bool LAST>
__device__ __forceinline__ void epilogue_update(const NsParams& p, const DevMat& M, int row, int cbase,
                                                uint32_t tb) {
  // UPDATE: X' = a X + acc.  AX: B = acc.  ABX: X' = a X + b B + c acc.
  constexpr bool kReadX = PHASE != kPhaseAX;
  constexpr bool kReadB = PHASE == kPhaseABX;
  const int m = M.m, n = M.n;
  const bool rv = row < m;
  const size_t roff = size_t(rv ? row : 0) * size_t(M.ldx);
  const uint16_t* x_row = M.X[p.cur] + roff;
  const uint16_t* b_row = M.B + roff;
  uint32_t pre[16], nxt[16], preb[16], nxtb[16];
  if (kReadX) prefetch_chunk(x_row, cbase, n, rv, nxt);
  if (kReadB) prefetch_chunk(b_row, cbase, n, rv, nxtb);
#pragma unroll 1
  for (int ch = 0; ch < kEpiCols / 32; ++ch) {
    const int col0 = cbase + ch * 32;
    if (kReadX) {
#pragma unroll
      for (int q = 0; q < 16; ++q) pre[q] = nxt[q];
      if (ch + 1 < kEpiCols / 32) prefetch_chunk(x_row, col0 + 32, n, rv, nxt);
    }
    if (kReadB) {
#pragma unroll
      for (int q = 0; q < 16; ++q) preb[q] = nxtb[q];
      if (ch + 1 < kEpiCols / 32) prefetch_chunk(b_row, col0 + 32, n, rv, nxtb);
    }
    float v[32];
    tmem_chunk(tb + uint32_t(ch * 32), v);
    if (!rv || col0 >= n) continue;
    const bool full = col0 + 32 <= n;
    if (kReadB) {
      float bb[32];
      chunk_operand(b_row, col0, n, preb, bb);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = fmaf(p.b, bb[i], p.c * v[i]);
    }
    if (kReadX) {
      float x[32];
      chunk_operand(x_row, col0, n, pre, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = fmaf(p.a, x[i], v[i]);
    }
    if (!LAST) {
      uint16_t* o_row = (PHASE == kPhaseAX ? M.B : M.X[p.cur ^ 1]) + size_t(row) * size_t(M.ldx) + col0;
      if (full) {
        store_bf16x32(o_row, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < n) o_row[i] = float_to_bf16_bits(v[i]);
      }
    } else {
      const float lr = p.lr_dev != nullptr ? *p.lr_dev : p.lr;
      const float decay = decay_factor(lr, p.wd);
      const float step = lr * (p.lr_adjust == MO_LR_MATCH_RMS_ADAMW ? M.rms_scale : M.shape_scale);
      // W is read and written once here: evict-first keeps the operand
      // panels the main loop re-reads in L2 (measured: 0.7 GB less DRAM
      // traffic and ~4% off this launch on the GPT-2 Large table)
      const uint64_t pol = ptx::policy_evict_first();
      if (!M.tall) {
        // W is [m, n]: element (row, col)
        float* w_row = M.W + size_t(row) * size_t(M.C) + col0;
        if (full && (reinterpret_cast<uintptr_t>(w_row) & 31u) == 0) {
          uint32_t w8[4][8];
#pragma unroll
          for (int q = 0; q < 4; ++q) ptx::ld_global_v8_hint(w_row + 8 * q, w8[q], pol);
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              w8[q][j] = __float_as_uint(fmaf(__uint_as_float(w8[q][j]), decay, -step * v[8 * q + j]));
#pragma unroll
          for (int q = 0; q < 4; ++q) ptx::st_global_v8_hint(w_row + 8 * q, w8[q], pol);
        } else {
          float w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = (col0 + i < n) ? w_row[i] : 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + i < n) w_row[i] = fmaf(w[i], decay, -step * v[i]);
        }
      } else {
        // W is [n, m]: element (col, row); the lanes of a warp hold
        // consecutive rows, so each access below is one 128-byte line
        float* w_col = M.W + size_t(col0) * size_t(M.C) + row;
        float w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = (col0 + i < n) ? ptx::ld_f32_hint(w_col + size_t(i) * size_t(M.C), pol) : 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < n) ptx::st_f32_hint(w_col + size_t(i) * size_t(M.C), fmaf(w[i], decay, -step * v[i]), pol);
      }
    }
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// Same three products with 256 x 256 output tiles computed by a cluster of
// two CTAs on two SMs (tcgen05 cta_group::2). Each CTA stages its 128-row half
// of the A operand and its 128-row (or 128-column) half of the B operand, so
// a 256 x 256 tile streams 64 KB per K block instead of the 96 KB two
// independent 128 x 256 tiles would need. The even CTA issues the MMAs and
// multicasts their completion to both CTAs; each CTA's epilogue drains the
// accumulator rows of its own A half from its own TMEM.
constexpr int kPairStages = 6;
constexpr uint32_t kPairHalfBytes = 128 * kBK * 2;                  // 16 KB
constexpr uint32_t kPairStageBytes = 2 * kPairHalfBytes;            // A half + B half
constexpr int kSchedSlots = 16;            // ring of published tile numbers
constexpr int kSchedAhead = 3;             // tiles published ahead of the one the producers load
constexpr uint32_t kSchedConsumers = 1 + kEpiWarps + 1 + kEpiWarps;   // MMA + epilogues, peer producer + epilogues
constexpr uint32_t kPairNumBars = 2 * kPairStages + 5 + 2 * kSchedSlots;
// barriers; TMEM slot, abort flag, the peer's report (2 words); the tile ring
constexpr uint32_t kPairCtrlBytes = 512;
static_assert(8 * kPairNumBars + 16 + 4 * kSchedSlots <= kPairCtrlBytes, "control block");
static_assert(kSchedAhead >= 1 && kSchedAhead < kSchedSlots, "a slot is republished only after its tile was loaded");
constexpr size_t kPairSmem = 1024 + size_t(kPairStages) * kPairStageBytes + kPairCtrlBytes;

// COUNTER: the tile schedule (p.counter_tiles), compiled separately so that
// neither variant carries the other's branches.
template <int PHASE, bool LAST, bool COUNTER>
__global__ void __launch_bounds__(kThreads, 1) ns_gemm_pair_kernel(const __grid_constant__ NsParams p) {
  // m x n outputs (B operand X or A X, MN-major, K = m) vs symmetric m x m ones
  constexpr bool kWide = PHASE == MO_PHASE_UPDATE || PHASE == kPhaseAX || PHASE == kPhaseABX;
  static_assert(!LAST || PHASE == MO_PHASE_UPDATE || PHASE == kPhaseABX, "LAST applies to the final product");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + uint32_t(kPairStages) * kPairStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + size_t(kPairStages) * kPairStageBytes + 8 * kPairNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // written by the peer CTA at the end: [0] it gave up, [1] its producer's issued stage count
  volatile uint32_t* peer_report = tmem_slot + 2;
  // tile numbers in launch order, written into both CTAs by the even CTA's producer
  volatile uint32_t* sched_tile = tmem_slot + 4;
  auto full_bar = [&](int s) { return bars + 8u * uint32_t(s); };
  auto empty_bar = [&](int s) { return bars + 8u * uint32_t(kPairStages + s); };
  auto tfull_bar = [&](int s) { return bars + 8u * uint32_t(2 * kPairStages + s); };
  auto tempty_bar = [&](int s) { return bars + 8u * uint32_t(2 * kPairStages + 2 + s); };
  const uint32_t drain_bar = bars + 8u * uint32_t(2 * kPairStages + 4);
  auto sfull_bar = [&](int s) { return bars + 8u * uint32_t(2 * kPairStages + 5 + s); };
  auto sempty_bar = [&](int s) { return bars + 8u * uint32_t(2 * kPairStages + 5 + kSchedSlots + s); };

  const int warp = int(threadIdx.x >> 5);
  const int lane = int(threadIdx.x & 31);
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(tfull_bar(s), 1);
      ptx::mbar_init(tempty_bar(s), 2 * kEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    for (int s = 0; s < kSchedSlots; ++s) {
      ptx::mbar_init(sfull_bar(s), 1);
      ptx::mbar_init(sempty_bar(s), kSchedConsumers);
    }
    *abort_flag = 0;
    peer_report[0] = 0u;
    peer_report[1] = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The setup above overlaps the previous launch's last tiles; its outputs
  // are read only after it has completed.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  // Tile schedule. With COUNTER the CTA pairs take the launch's
  // tiles in list order from one counter, so the pairs work on neighbouring
  // tiles (shared operand panels stay in L2) and finish within a tile or two
  // of each other. The even CTA's producer takes the tile numbers and
  // publishes each in a ring of kSchedSlots slots in both CTAs, kSchedAhead
  // tiles before the producers load it; every other role reads it there,
  // and a number >= ntiles ends the role's loop. The even CTA's own roles
  // synchronise on the ring at CTA scope, the odd CTA's at cluster scope.
  // Without it every role of pair c runs tiles c, c + pairs, ... by itself.
  const uint32_t ntiles = uint32_t(p.ntiles);
  constexpr bool by_counter = COUNTER;
  uint32_t static_next = ptx::cluster_id_x();
  const uint32_t npairs = ptx::nclusters_x();
  int sslot = 0;
  uint32_t sph = 0;
  // Takes the next tile number (a consumer role: the MMA issuer, an
  // epilogue warp, the odd CTA's producer; with the static schedule every
  // role). From the ring: waits for the slot, reads it, and releases the
  // slot to the even CTA's producer, one lane per warp.
  auto next_tile = [&](uint32_t& t) -> bool {
    if (!by_counter) {
      t = static_next;
      static_next += npairs;
      return true;
    }
    bool ok = true;
    if (lane == 0) {
      ok = leader ? mbar_wait_bounded<false>(sfull_bar(sslot), sph, abort_flag, p.status, p.timeout_ns)
                  : mbar_wait_bounded<true>(sfull_bar(sslot), sph, abort_flag, p.status, p.timeout_ns);
      if (ok) {
        t = sched_tile[sslot];
        if (leader)
          ptx::mbar_arrive(sempty_bar(sslot));
        else
          ptx::mbar_arrive_cluster(ptx::mapa_shared(sempty_bar(sslot), 0));
      }
    }
    if (warp >= 2) {
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      t = __shfl_sync(0xFFFFFFFFu, t, 0);
    }
    if (++sslot == kSchedSlots) {
      sslot = 0;
      sph ^= 1u;
    }
    return ok;
  };

  uint32_t n_issued = 0;      // producer: operand stages issued (stage j % S, phase parity (j / S) & 1)
  bool mma_issued = false;    // MMA issuer: any MMA issued
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer (both CTAs)
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t last_mat = 0xFFFFFFFFu;
      // even CTA: the publishing position in the ring, and the next tile
      // number, taken from the counter one publication early
      int pslot = 0;
      uint32_t pph = 0;
      bool published_end = false;
      const bool publisher = leader && by_counter;
      uint32_t ahead = publisher ? atomicAdd(p.tile_ctr, 1u) : 0u;
      auto publish = [&]() -> bool {
        if (published_end) return true;
        if (!mbar_wait_bounded<true>(sempty_bar(pslot), pph ^ 1u, abort_flag, p.status, p.timeout_ns))
          return false;
        const uint32_t v = ahead;
        sched_tile[pslot] = v;
        ptx::mbar_arrive(sfull_bar(pslot));
        ptx::st_shared_cluster_u32(ptx::mapa_shared(ptx::smem_addr(const_cast<uint32_t*>(sched_tile + pslot)), 1u), v);
        ptx::mbar_arrive_cluster(ptx::mapa_shared(sfull_bar(pslot), 1u));
        if (++pslot == kSchedSlots) {
          pslot = 0;
          pph ^= 1u;
        }
        if (v >= ntiles)
          published_end = true;
        else
          ahead = atomicAdd(p.tile_ctr, 1u);
        return true;
      };
      if (publisher)
        for (int i = 0; ok && i < kSchedAhead; ++i) ok = publish();
      while (ok) {
        uint32_t t;
        if (publisher) {
          // this thread published the slot itself; it is republished only
          // kSchedSlots - kSchedAhead tiles after this read
          t = sched_tile[sslot];
          if (++sslot == kSchedSlots) sslot = 0;
          if (t < ntiles && !publish()) break;
        } else if (!next_tile(t)) {
          break;
        }
        if (t >= ntiles) break;
        const TileRec tr = p.tiles[t];
        const DevMat& M = p.mats[tr.mat];
        const CUtensorMap* maps = p.tmaps + size_t(tr.mat) * kMapsPerMat;
        const void* mapA;
        const void* mapB;
        int K;
        if (PHASE == MO_PHASE_GRAM) {
          mapA = mapB = &maps[p.cur];
          K = M.n;
        } else if (PHASE == MO_PHASE_POLY) {
          mapA = mapB = &maps[2];
          K = M.m;
        } else if (PHASE == MO_PHASE_UPDATE) {
          mapA = &maps[3];
          mapB = &maps[p.cur];
          K = M.m;
        } else if (PHASE == kPhaseAX) {
          mapA = &maps[2];
          mapB = &maps[p.cur];
          K = M.m;
        } else {
          mapA = &maps[2];
          mapB = &maps[3];
          K = M.m;
        }
        if (tr.mat != last_mat) {
          ptx::fence_tmap_acquire(mapA);
          ptx::fence_tmap_acquire(mapB);
          last_mat = tr.mat;
        }
        const int nk = (K + kBK - 1) / kBK;
        const int arow = int(tr.tm) * 256 + int(rank) * 128;   // this CTA's A rows
        const int bcol = int(tr.tn) * 256 + int(rank) * 128;   // this CTA's B rows / columns
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), ph ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = full_bar(stage);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, 2 * kPairStageBytes);
          const uint32_t fb = ptx::mapa_shared(fb_local, 0);
          const uint32_t sa = base + uint32_t(stage) * kPairStageBytes;
          const uint32_t sb = sa + kPairHalfBytes;
          const int k0 = kb * kBK;
          ptx::tma_load_2d_pair(sa, mapA, fb, k0, arow);
          ptx::tma_load_2d_pair(sa + kBoxBytes, mapA, fb, k0, arow + 64);
          if (!kWide) {
            ptx::tma_load_2d_pair(sb, mapB, fb, k0, bcol);
            ptx::tma_load_2d_pair(sb + kBoxBytes, mapB, fb, k0, bcol + 64);
          } else {
            ptx::tma_load_2d_pair(sb, mapB, fb, bcol, k0);
            ptx::tma_load_2d_pair(sb + kBoxBytes, mapB, fb, bcol + 64, k0);
          }
          ++n_issued;
          if (++stage == kPairStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (even CTA)
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(256, kBN, 0u, kWide ? 1u : 0u);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      uint32_t t;
      while (ok && next_tile(t) && t < ntiles) {
        const TileRec tr = p.tiles[t];
        const DevMat& M = p.mats[tr.mat];
        const int K = (PHASE == MO_PHASE_GRAM) ? M.n : M.m;
        const int nk = (K + kBK - 1) / kBK;
        if (!mbar_wait_bounded(tempty_bar(acc), aph ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc) * uint32_t(kBN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), ph, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = base + uint32_t(stage) * kPairStageBytes;
          const uint32_t sb = sa + kPairHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(sa + uint32_t(kk) * 32u, 16u, 1024u);
            const uint64_t bd = kWide
                                    ? ptx::smem_desc_sw128(sb + uint32_t(kk) * 2048u, kBoxBytes, 1024u)
                                    : ptx::smem_desc_sw128(sb + uint32_t(kk) * 32u, 16u, 1024u);
            ptx::umma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::umma_commit_pair(empty_bar(stage), 0x3);
          mma_issued = true;
          if (++stage == kPairStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit_pair(tfull_bar(acc), 0x3);
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r_in = quarter * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    uint32_t t;
    while (next_tile(t) && t < ntiles) {
      const TileRec tr = p.tiles[t];
      const DevMat& M = p.mats[tr.mat];
      if (LAST) prefetch_w_rows(M, int(tr.tm) * 256 + int(rank) * 128 + r_in, int(tr.tn) * kBN + half * kEpiCols);
      bool ok = mbar_wait_bounded(tfull_bar(acc), aph, abort_flag, p.status, p.timeout_ns);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row = int(tr.tm) * 256 + int(rank) * 128 + r_in;
      const int cbase = int(tr.tn) * kBN + half * kEpiCols;
      const uint32_t tb = tmem_base + uint32_t(acc) * uint32_t(kBN) + uint32_t(half * kEpiCols) +
                          (uint32_t(quarter * 32) << 16);
      if (kWide)
        epilogue_update<PHASE, LAST>(p, M, row, cbase, tb);
      else
        epilogue_symmetric<PHASE>(p, M, row, cbase, tb);
      // hand the accumulator back: its reads are complete (tcgen05.wait::ld)
      // and fenced; the tile's global stores need no ordering inside the
      // launch, so the arrive releases at CTA scope and does not wait for them
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote_cta(ptx::mapa_shared(tempty_bar(acc), 0));
      if (p.coverage != nullptr && warp == 2 && lane == 0) atomicAdd(p.coverage + 2 * size_t(t) + rank, 1u);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();   // every role has finished: this CTA's abort flag and issue count are final
  // Each CTA tells its peer whether it gave up and how many operand stages
  // its producer issued (thread 0 is the producer lane).
  if (threadIdx.x == 0)
    ptx::st_shared_cluster_v2(ptx::mapa_shared(ptx::smem_addr(const_cast<uint32_t*>(peer_report)), rank ^ 1u),
                              *abort_flag != 0 ? 1u : 0u, n_issued);
  ptx::cluster_sync();
  if (*abort_flag != 0 || peer_report[0] != 0u) {   // the same decision on both CTAs
    // Nothing may still be writing into either CTA's shared memory or TMEM
    // when they exit. The even CTA waits for its MMAs, then for every
    // operand stage either producer left in flight: all copies of both CTAs
    // count their bytes on the even CTA's full barriers, so it settles each
    // stage the two producers did not both fill (arming the ones only the
    // peer filled, completing the peer's share of the ones only it filled)
    // and waits for the stage's phase. Each producer waits for the MMAs to
    // consume a stage before refilling it, so the two issue counts differ by
    // at most S and only the last S stages can be in flight. The second
    // cluster barrier keeps the odd CTA resident until the drain is over.
    if (leader && warp == 1 && lane == 0 && mma_issued) {
      ptx::umma_commit_pair(drain_bar, 0x1);
      mbar_wait_drain(drain_bar, 0u, p.timeout_ns);
    }
    if (leader && threadIdx.x == 0) {
      const uint32_t L = n_issued, P = peer_report[1];
      const uint32_t M = L > P ? L : P;
      for (uint32_t j = M > uint32_t(kPairStages) ? M - uint32_t(kPairStages) : 0u; j < M; ++j) {
        const int s = int(j % uint32_t(kPairStages));
        if (j >= L)
          ptx::mbar_arrive_expect_tx(full_bar(s), kPairStageBytes);   // only the peer's half is coming
        else if (j >= P)
          ptx::mbar_complete_tx(full_bar(s), kPairStageBytes);        // the peer's half never will
        mbar_wait_drain(full_bar(s), (j / uint32_t(kPairStages)) & 1u, p.timeout_ns);
      }
    }
    ptx::cluster_sync();
  }
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
}

// A = bf16(sum over slices of the fp32 partials) for each long matrix: one
// 64 x 64 upper block (column block >= row block) per iteration, partials
// summed in slice order, the upper part stored directly and the strict lower
// part through a shared-memory transpose, so every element of A is written
// once.
__global__ void __launch_bounds__(256) gram_reduce_kernel(const GramReduce* __restrict__ recs, int32_t count,
                                                          int64_t blocks) {
  __shared__ float tile[64][65];
  const int tid = int(threadIdx.x), tx = tid & 15, ty = tid >> 4;
  for (int64_t b = blockIdx.x; b < blocks; b += gridDim.x) {
    int lo = 0, hi = count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (recs[mid].block_base <= b) lo = mid; else hi = mid - 1;
    }
    const GramReduce R = recs[lo];
    const int64_t local = b - R.block_base;
    // upper blocks are numbered row by row; row br starts at br nb - br (br - 1) / 2
    const int nb = (R.m + 63) / 64;
    int br = 0, hb = nb - 1;
    while (br < hb) {
      const int mid = (br + hb + 1) >> 1;
      if (int64_t(mid) * nb - int64_t(mid) * (mid - 1) / 2 <= local) br = mid; else hb = mid - 1;
    }
    const int bc = br + int(local - (int64_t(br) * nb - int64_t(br) * (br - 1) / 2));
    const int r0 = br * 64, c0 = bc * 64 + tx * 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    for (int sl = 0; sl < R.slices; ++sl) {
      const float* P = R.parts + int64_t(sl) * R.part_stride;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty * 4 + i;
        if (r < R.m) {
          const float4 x = *reinterpret_cast<const float4*>(P + size_t(r) * size_t(R.lda) + c0);
          acc[i][0] += x.x;
          acc[i][1] += x.y;
          acc[i][2] += x.z;
          acc[i][3] += x.w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + ty * 4 + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        tile[ty * 4 + i][tx * 4 + j] = acc[i][j];
        const int c = c0 + j;
        if (r < R.m && c < R.m && c >= r) R.A[size_t(r) * size_t(R.lda) + c] = float_to_bf16_bits(acc[i][j]);
      }
    }
    __syncthreads();
    // mirror: A[c][r] = value at (r, c) for c > r
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = bc * 64 + ty * 4 + i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = r0 + tx * 4 + j;
        if (c < R.m && r < R.m && c > r)
          R.A[size_t(c) * size_t(R.lda) + r] = float_to_bf16_bits(tile[tx * 4 + j][ty * 4 + i]);
      }
    }
    __syncthreads();
  }
}

// Single-CTA kernel that waits on a barrier nothing completes; exercises the
// bounded-wait path.
__global__ void bounded_wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(ptx::smem_addr(&bar), 0u, reinterpret_cast<volatile int*>(&abort_flag), status,
                      timeout_ns);
  __syncthreads();
}

template <int PHASE, bool LAST>
cudaError_t launch_pair(const NsParams& p, int grid, cudaStream_t stream) {
  auto kern = p.counter_tiles != 0 ? ns_gemm_pair_kernel<PHASE, LAST, true> : ns_gemm_pair_kernel<PHASE, LAST, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPairSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: CTAs start their setup (barriers, TMEM)
  // as SMs leave the previous launch, then wait for it in griddep_wait()
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_phase(int phase, bool last, const NsParams& p, int grid, cudaStream_t stream) {
  if (p.ntiles <= 0) return cudaSuccess;
  switch (phase) {
    case MO_PHASE_GRAM:
      return launch_pair<MO_PHASE_GRAM, false>(p, grid, stream);
    case MO_PHASE_POLY:
      return launch_pair<MO_PHASE_POLY, false>(p, grid, stream);
    case kPhaseAX:
      return launch_pair<kPhaseAX, false>(p, grid, stream);
    case kPhaseABX:
      return last ? launch_pair<kPhaseABX, true>(p, grid, stream) : launch_pair<kPhaseABX, false>(p, grid, stream);
    default:
      return last ? launch_pair<MO_PHASE_UPDATE, true>(p, grid, stream)
                  : launch_pair<MO_PHASE_UPDATE, false>(p, grid, stream);
  }
}

cudaError_t launch_gram_reduce(const GramReduce* reduces, int32_t count, int64_t blocks, int grid,
                               cudaStream_t stream) {
  if (count <= 0 || blocks <= 0) return cudaSuccess;
  gram_reduce_kernel<<<grid, 256, 0, stream>>>(reduces, count, blocks);
  return cudaGetLastError();
}

cudaError_t device_status_ptr(int** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_mo_status);
}

cudaError_t launch_bounded_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ tensor maps

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode_bf16_2d(CUtensorMap* map, void* gaddr, uint64_t cols, uint64_t rows, uint64_t ld_elems) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld_elems * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, gaddr, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_matrix_maps(const DevMat& d, int ns_form, void* out_maps) {
  static_assert(sizeof(CUtensorMap) == kTensorMapBytes, "CUtensorMap size");
  CUtensorMap* maps = static_cast<CUtensorMap*>(out_maps);
  const bool wide_b = ns_form == MO_NS_APPENDIX;   // B = A X is m x n
  return encode_bf16_2d(&maps[0], d.X[0], uint64_t(d.n), uint64_t(d.m), uint64_t(d.ldx)) &&
         encode_bf16_2d(&maps[1], d.X[1], uint64_t(d.n), uint64_t(d.m), uint64_t(d.ldx)) &&
         encode_bf16_2d(&maps[2], d.A, uint64_t(d.m), uint64_t(d.m), uint64_t(d.lda)) &&
         (wide_b ? encode_bf16_2d(&maps[3], d.B, uint64_t(d.n), uint64_t(d.m), uint64_t(d.ldx))
                 : encode_bf16_2d(&maps[3], d.B, uint64_t(d.m), uint64_t(d.m), uint64_t(d.lda)));
}

}  // namespace mo

// Memory-bound kernels of the owner-local step: the two Muon prologue passes
// (momentum + Frobenius sum of squares; normalise + bf16 cast/transpose), RMNP
// and AdamW. All accesses along rows are 16-byte vectors where the row length
// allows it; every kernel is a grid-stride loop over a flat work list sized to
// a multiple of the SM count.
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "kernels.h"
#include "mo_internal.h"

namespace mo {

namespace {

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// ------------------------------------------------------------------ Muon prologue
//
// Two launches over the owner's table:
//   norm launch  momentum V <- mu V + G ("Optimizers In A Sharded World",
//                section 1) over flat kNrmChunk-element chunks of every
//                stored matrix, with one fp32 sum of squares of U per chunk,
//                where U = V, or U = G + mu V with Nesterov momentum (the
//                default update of torch.optim.Muon, which "MatrixFSDP"
//                section 5.1 runs). The CTA that completes a matrix's last
//                chunk sums that matrix's partials in a fixed order
//                (deterministic, no float atomics) and writes the Frobenius
//                scale 1 / (||U|| + eps) (eps added to the norm, as in the
//                same page's appendix).
//   cast launch  X0 = bf16(U * scale) for 64 x 128 tiles, written in the wide
//                orientation (transposed through shared memory when
//                rows > cols, appendix of the same page). It is a
//                programmatic dependent launch that waits for the norm
//                launch to complete, so every scale is final and nothing
//                waits inside it; tiles are taken from the last matrix back,
//                last row block first, so the momentum the norm launch wrote
//                last is read while it is still in L2.
// Both are grid-stride streams with many 16-byte loads in flight per thread
// (the norm launch 16 vectors of V and 16 of G, at two CTAs per SM), which is
// what a memory-bound kernel needs here to keep HBM busy. (A single launch
// that interleaves the casts with the norms, to re-read the momentum from L2,
// moves fewer bytes but has to make casts wait for their matrix's norm.)


// 16-byte vectors of V (and the matching 8 bytes of G) per thread loaded
// before use in each round of a norm item
constexpr int kNrmBatch = 16;

template <bool NEST>
__device__ void prologue_norm_item(const ProParams& p, int mi, int64_t local, float* red, int* last_flag) {
  const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  const DevMat& M = p.mats[mi];
  const int64_t e0 = local * kNrmChunk;
  const int64_t left = int64_t(M.R) * int64_t(M.C) - e0;
  const int cnt = left < kNrmChunk ? int(left) : int(kNrmChunk);
  float* __restrict__ V = M.V + e0;
  const uint16_t* __restrict__ G = M.G + e0;
  float ss = 0.f;
#pragma unroll 1
  for (int base = 0; base < cnt; base += kNrmBatch * 256 * 4) {
    float4 v[kNrmBatch];
    uint2 g[kNrmBatch];
#pragma unroll
    for (int j = 0; j < kNrmBatch; ++j) {
      const int e = base + (j * 256 + tid) * 4;
      if (e + 4 <= cnt) {
        v[j] = *reinterpret_cast<const float4*>(V + e);
        g[j] = *reinterpret_cast<const uint2*>(G + e);
      }
    }
#pragma unroll
    for (int j = 0; j < kNrmBatch; ++j) {
      const int e = base + (j * 256 + tid) * 4;
      if (e + 4 <= cnt) {
        const float g0 = bf16_bits_to_float(g[j].x & 0xFFFFu), g1 = bf16_bits_to_float(g[j].x >> 16);
        const float g2 = bf16_bits_to_float(g[j].y & 0xFFFFu), g3 = bf16_bits_to_float(g[j].y >> 16);
        float4 n4;
        n4.x = fmaf(p.mu, v[j].x, g0);
        n4.y = fmaf(p.mu, v[j].y, g1);
        n4.z = fmaf(p.mu, v[j].z, g2);
        n4.w = fmaf(p.mu, v[j].w, g3);
        *reinterpret_cast<float4*>(V + e) = n4;
        float4 u4 = n4;
        if (NEST) {
          u4.x = fmaf(p.mu, n4.x, g0);
          u4.y = fmaf(p.mu, n4.y, g1);
          u4.z = fmaf(p.mu, n4.z, g2);
          u4.w = fmaf(p.mu, n4.w, g3);
        }
        ss = fmaf(u4.x, u4.x, ss);
        ss = fmaf(u4.y, u4.y, ss);
        ss = fmaf(u4.z, u4.z, ss);
        ss = fmaf(u4.w, u4.w, ss);
      } else {
        for (int k = e; k < cnt && k < e + 4; ++k) {
          const float gk = bf16_bits_to_float(G[k]);
          const float vn = fmaf(p.mu, V[k], gk);
          V[k] = vn;
          const float u = NEST ? fmaf(p.mu, vn, gk) : vn;
          ss = fmaf(u, u, ss);
        }
      }
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    p.partials[M.nrm_base + local] = tot;
    __threadfence();
    const uint32_t prev = atomicAdd(&p.counters[mi], 1u);
    *last_flag = (int64_t(prev) + 1 == M.nrm_count) ? 1 : 0;
  }
  __syncthreads();
  if (*last_flag) {
    __threadfence();
    float acc = 0.f;
    for (int64_t k = tid; k < M.nrm_count; k += 256) acc += __ldcg(p.partials + M.nrm_base + k);
    acc = warp_sum(acc);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) tot += red[w];
      p.scales[mi] = 1.0f / (sqrtf(tot) + p.eps);
      p.counters[mi] = 0u;
      __threadfence();
      atomicExch(&p.ready[mi], 1u);
    }
  }
  __syncthreads();
}

// U = V, or G + mu V (Nesterov), for four consecutive elements at `off`.
template <bool NEST>
__device__ __forceinline__ float4 load_u4(const ProParams& p, const DevMat& M, size_t off) {
  float4 u = __ldcg(reinterpret_cast<const float4*>(M.V + off));
  if (NEST) {
    const uint2 g = *reinterpret_cast<const uint2*>(M.G + off);
    u.x = fmaf(p.mu, u.x, bf16_bits_to_float(g.x & 0xFFFFu));
    u.y = fmaf(p.mu, u.y, bf16_bits_to_float(g.x >> 16));
    u.z = fmaf(p.mu, u.z, bf16_bits_to_float(g.y & 0xFFFFu));
    u.w = fmaf(p.mu, u.w, bf16_bits_to_float(g.y >> 16));
  }
  return u;
}

template <bool NEST>
__device__ __forceinline__ float load_u1(const ProParams& p, const DevMat& M, size_t off) {
  const float v = __ldcg(M.V + off);
  return NEST ? fmaf(p.mu, v, bf16_bits_to_float(M.G[off])) : v;
}

template <bool NEST>
__device__ void prologue_cast_item(const ProParams& p, int mi, int64_t local, uint16_t (*tbuf)[kCastTR + 8]) {
  const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  const DevMat& M = p.mats[mi];
  const int r0 = int(local / M.cast_tiles_c) * kCastTR;
  const int c0 = int(local % M.cast_tiles_c) * kCastTC;
  const int R = M.R, C = M.C;
  const float sc = __ldcg(p.scales + mi);
  uint16_t* X = M.X[0];
  const size_t ldx = size_t(M.ldx);
  if (!M.tall) {
    // warp w covers rows w, w+8, ...; lanes cover 4 consecutive columns each.
    // All eight rows' loads are issued before their stores (the stores could alias the loads as far as the
    // compiler knows, which would otherwise serialise every row on a full
    // memory latency).
    const int c = c0 + lane * 4;
    if (c < C && M.vec_ok && c + 4 <= C) {
#pragma unroll 1
      for (int i0 = 0; i0 < kCastTR / 8; i0 += 8) {
        float4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = r0 + warp + 8 * (i0 + i);
          if (r < R) u[i] = load_u4<NEST>(p, M, size_t(r) * size_t(C) + size_t(c));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = r0 + warp + 8 * (i0 + i);
          if (r < R)
            *reinterpret_cast<uint2*>(X + size_t(r) * ldx + size_t(c)) =
                make_uint2(pack_bf16x2(u[i].x * sc, u[i].y * sc), pack_bf16x2(u[i].z * sc, u[i].w * sc));
        }
      }
    } else if (c < C) {
      for (int i = 0; i < kCastTR / 8; ++i) {
        const int r = r0 + warp + 8 * i;
        if (r >= R) break;
        const size_t off = size_t(r) * size_t(C) + size_t(c);
        uint16_t* xp = X + size_t(r) * ldx + size_t(c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < C) xp[q] = float_to_bf16_bits(load_u1<NEST>(p, M, off + q) * sc);
      }
    }
  } else {
    // X is [C, R]: X[c][r] = bf16(V[r][c] * scale). Thread = (row rl, 32-column
    // quarter cq): lanes hold consecutive rows, so the shared-memory writes
    // tbuf[c][rl] of a warp are contiguous; each lane reads its 128-byte row
    // segment with 32-byte vectors.
    const int rl = tid & (kCastTR - 1);
    const int cq = tid >> 6;
    const int r = r0 + rl;
    const int cb = cq * 32;
    if (r < R) {
      const size_t roff = size_t(r) * size_t(C) + size_t(c0 + cb);
      const float* vrow = M.V + roff;
      if (c0 + cb + 32 <= C && (reinterpret_cast<uintptr_t>(vrow) & 31u) == 0) {
        uint32_t w8[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) ptx::ld_global_v8_cg(vrow + 8 * j, w8[j]);
        if (NEST) {
          // the matching 8 bf16 of G per 32-byte V vector (16-byte aligned)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 g = *reinterpret_cast<const uint4*>(M.G + roff + 8 * j);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float gq = bf16_bits_to_float((q & 1) ? (gw[q >> 1] >> 16) : (gw[q >> 1] & 0xFFFFu));
              w8[j][q] = __float_as_uint(fmaf(p.mu, __uint_as_float(w8[j][q]), gq));
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int q = 0; q < 8; ++q) tbuf[cb + 8 * j + q][rl] = float_to_bf16_bits(__uint_as_float(w8[j][q]) * sc);
      } else {
        for (int j = 0; j < 32; ++j)
          tbuf[cb + j][rl] = (c0 + cb + j < C) ? float_to_bf16_bits(load_u1<NEST>(p, M, roff + j) * sc) : uint16_t(0);
      }
    }
    __syncthreads();
    // 16-byte segments of 8 rows per X row
    for (int k = tid; k < kCastTC * (kCastTR / 8); k += 256) {
      const int cc = k >> 3, seg = k & 7;
      const int xc = c0 + cc;
      const int xr = r0 + seg * 8;
      if (xc < C && xr < R) {
        uint16_t* xp = X + size_t(xc) * ldx + size_t(xr);
        const uint16_t* sp = &tbuf[cc][seg * 8];
        if (xr + 8 <= R) {
          *reinterpret_cast<uint4*>(xp) = *reinterpret_cast<const uint4*>(sp);
        } else {
          for (int j = 0; j < 8; ++j)
            if (xr + j < R) xp[j] = sp[j];
        }
      }
    }
    __syncthreads();
  }
}

// Index of the matrix whose prefix range [prefix[i], prefix[i+1]) holds t.
__device__ __forceinline__ int prologue_matrix(const int64_t* prefix, int n, int64_t t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <bool NEST>
__global__ void __launch_bounds__(256, kPrologueCtasPerSm) muon_norm_kernel(const __grid_constant__ ProParams p) {
  ptx::griddep_launch_dependents();   // the cast launch is scheduled early; it waits for this grid to finish
  __shared__ float red[8];
  __shared__ int flag;
  for (int64_t t = blockIdx.x; t < p.nrm_total; t += gridDim.x) {
    const int mi = prologue_matrix(p.nrm_prefix, p.n, t);
    prologue_norm_item<NEST>(p, mi, t - p.nrm_prefix[mi], red, &flag);
  }
}

template <bool NEST>
__global__ void __launch_bounds__(256) muon_cast_kernel(const __grid_constant__ ProParams p) {
  __shared__ __align__(16) uint16_t tbuf[kCastTC][kCastTR + 8];
  ptx::griddep_wait();                // the norm launch's momentum and scales
  ptx::griddep_launch_dependents();   // the first Gram launch may start its setup as CTAs finish
  for (int64_t t = blockIdx.x; t < p.cast_total; t += gridDim.x) {
    const int64_t r = p.cast_total - 1 - t;   // from the last tile of the last matrix back
    const int mi = prologue_matrix(p.cast_prefix, p.n, r);
    prologue_cast_item<NEST>(p, mi, r - p.cast_prefix[mi], tbuf);
  }
}

// ------------------------------------------------------------------ RMNP

// lr s / max(||V_i||, eps) for RMNP; lr s max(||V_i||, eps)^(power - 1) for
// HTRMNP (a reading of "Optimizers In A Sharded World" section 7, which names
// the power scaling without printing a formula).
// max(norm, eps) that keeps a NaN norm (a NaN anywhere in the row) as NaN,
// as F.normalize's clamp does; fmaxf would return eps for it
__device__ __forceinline__ float clamp_norm(float nrm, float eps) { return nrm < eps ? eps : nrm; }

__device__ __forceinline__ float rmnp_factor(const RmnpParams& p, float lr, float scale, float sum_sq) {
  const float nrm = clamp_norm(sqrtf(sum_sq), p.eps);
  return p.power == 0.0f ? lr * scale / nrm : lr * scale * powf(nrm, p.power - 1.0f);
}
//
// One warp per stored row ("Optimizers In A Sharded World", section 1 and the
// appendix rmnp_local): V_i <- mu V_i + G_i, D_i = V_i / max(||V_i||_2, eps),
// W_i <- W_i (1 - lr wd) - lr s D_i. Pass 1 writes V_i and accumulates its sum
// of squares in fp32 (lane-strided, then a fixed xor-shuffle tree, so a row's
// result does not depend on which other rows share the launch); pass 2 re-reads
// V_i (just written, served from L2) and updates W_i.
__global__ void __launch_bounds__(256) rmnp_kernel(const __grid_constant__ RmnpParams p) {
  const float lr = p.lr_dev != nullptr ? *p.lr_dev : p.lr;
  const float decay = decay_factor(lr, p.wd);
  const int lane = int(threadIdx.x & 31);
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = p.row_prefix[p.n];
  for (int64_t row = gw; row < total; row += nw) {
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.row_prefix[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const RmnpEntry& E = p.e[lo];
    const int C = E.C;
    const size_t off = size_t(row - p.row_prefix[lo]) * size_t(C);
    float* __restrict__ Vr = E.V + off;
    float* __restrict__ Wr = E.W + off;
    const uint16_t* __restrict__ Gr = E.G + off;
    float ss = 0.f;
    if (E.vec_ok) {
      for (int cb = lane * 4; cb < C; cb += 4 * 128) {
        float4 v[4];
        uint2 g[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            g[u] = *reinterpret_cast<const uint2*>(Gr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            float4 n4;
            n4.x = fmaf(p.mu, v[u].x, bf16_bits_to_float(g[u].x & 0xFFFFu));
            n4.y = fmaf(p.mu, v[u].y, bf16_bits_to_float(g[u].x >> 16));
            n4.z = fmaf(p.mu, v[u].z, bf16_bits_to_float(g[u].y & 0xFFFFu));
            n4.w = fmaf(p.mu, v[u].w, bf16_bits_to_float(g[u].y >> 16));
            *reinterpret_cast<float4*>(Vr + cc) = n4;
            ss = fmaf(n4.x, n4.x, ss);
            ss = fmaf(n4.y, n4.y, ss);
            ss = fmaf(n4.z, n4.z, ss);
            ss = fmaf(n4.w, n4.w, ss);
          }
        }
      }
    } else {
      for (int cc = lane; cc < C; cc += 32) {
        const float vn = fmaf(p.mu, Vr[cc], bf16_bits_to_float(Gr[cc]));
        Vr[cc] = vn;
        ss = fmaf(vn, vn, ss);
      }
    }
    ss = warp_sum(ss);
    const float k = rmnp_factor(p, lr, E.scale, ss);
    if (E.vec_ok) {
      for (int cb = lane * 4; cb < C; cb += 4 * 128) {
        float4 v[4], w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            w[u] = *reinterpret_cast<const float4*>(Wr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            float4 o;
            o.x = w[u].x * decay - k * v[u].x;
            o.y = w[u].y * decay - k * v[u].y;
            o.z = w[u].z * decay - k * v[u].z;
            o.w = w[u].w * decay - k * v[u].w;
            *reinterpret_cast<float4*>(Wr + cc) = o;
          }
        }
      }
    } else {
      for (int cc = lane; cc < C; cc += 32) Wr[cc] = Wr[cc] * decay - k * Vr[cc];
    }
  }
}

// The same RMNP step with one CTA per stored row, for long rows: a warp per
// row keeps up to 64 rows per SM in flight, which for rows of ~14 K elements
// (57 KB) is more than L2 holds between the two passes; a CTA per row keeps
// 8 per SM. The row's sum of squares is reduced in a fixed order (per-thread
// strided sums, a fixed xor tree per warp, the 8 warps in order), so a row's
// result does not depend on the launch either.
__global__ void __launch_bounds__(256) rmnp_row_cta_kernel(const __grid_constant__ RmnpParams p) {
  const float lr = p.lr_dev != nullptr ? *p.lr_dev : p.lr;
  const float decay = decay_factor(lr, p.wd);
  __shared__ float red[8];
  const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  const int64_t total = p.row_prefix[p.n];
  for (int64_t row = blockIdx.x; row < total; row += gridDim.x) {
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.row_prefix[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const RmnpEntry& E = p.e[lo];
    const int C = E.C;
    const size_t off = size_t(row - p.row_prefix[lo]) * size_t(C);
    float* __restrict__ Vr = E.V + off;
    float* __restrict__ Wr = E.W + off;
    const uint16_t* __restrict__ Gr = E.G + off;
    float ss = 0.f;
    if (E.vec_ok) {
      for (int cb = tid * 4; cb < C; cb += 4 * 1024) {
        float4 v[4];
        uint2 g[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 1024;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            g[u] = *reinterpret_cast<const uint2*>(Gr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 1024;
          if (cc < C) {
            float4 n4;
            n4.x = fmaf(p.mu, v[u].x, bf16_bits_to_float(g[u].x & 0xFFFFu));
            n4.y = fmaf(p.mu, v[u].y, bf16_bits_to_float(g[u].x >> 16));
            n4.z = fmaf(p.mu, v[u].z, bf16_bits_to_float(g[u].y & 0xFFFFu));
            n4.w = fmaf(p.mu, v[u].w, bf16_bits_to_float(g[u].y >> 16));
            *reinterpret_cast<float4*>(Vr + cc) = n4;
            ss = fmaf(n4.x, n4.x, ss);
            ss = fmaf(n4.y, n4.y, ss);
            ss = fmaf(n4.z, n4.z, ss);
            ss = fmaf(n4.w, n4.w, ss);
          }
        }
      }
    } else {
      for (int cc = tid; cc < C; cc += 256) {
        const float vn = fmaf(p.mu, Vr[cc], bf16_bits_to_float(Gr[cc]));
        Vr[cc] = vn;
        ss = fmaf(vn, vn, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    __syncthreads();   // red is rewritten by the next row
    const float k = rmnp_factor(p, lr, E.scale, tot);
    if (E.vec_ok) {
      for (int cb = tid * 4; cb < C; cb += 4 * 1024) {
        float4 v[4], w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 1024;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            w[u] = *reinterpret_cast<const float4*>(Wr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 1024;
          if (cc < C) {
            float4 o;
            o.x = w[u].x * decay - k * v[u].x;
            o.y = w[u].y * decay - k * v[u].y;
            o.z = w[u].z * decay - k * v[u].z;
            o.w = w[u].w * decay - k * v[u].w;
            *reinterpret_cast<float4*>(Wr + cc) = o;
          }
        }
      }
    } else {
      for (int cc = tid; cc < C; cc += 256) Wr[cc] = Wr[cc] * decay - k * Vr[cc];
    }
  }
}

// ------------------------------------------------------------------ column-cut RMNP
//
// Rows cut into column shards ("Optimizers In A Sharded World", section 3):
// pass 1 updates each shard's momentum and writes one fp32 sum of squares per
// shard row; pass 2 adds, for every row, the partials of all shards of its
// matrix in table order (in place of the page's all-reduce), clamps the
// square root at eps and applies the update to the shard. Warp per row, as
// rmnp_kernel.

__device__ __forceinline__ int colcut_entry(const ColcutParams& p, int64_t row) {
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.row_prefix[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(256) colcut_partial_kernel(const __grid_constant__ ColcutParams p) {
  const int lane = int(threadIdx.x & 31);
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = p.row_prefix[p.n];
  for (int64_t row = gw; row < total; row += nw) {
    const int ei = colcut_entry(p, row);
    const RmnpEntry& E = p.e[ei];
    const int C = E.C;
    const size_t off = size_t(row - p.row_prefix[ei]) * size_t(C);
    float* __restrict__ Vr = E.V + off;
    const uint16_t* __restrict__ Gr = E.G + off;
    float ss = 0.f;
    if (E.vec_ok) {
      // four 16-byte vectors per lane, all loaded before use
      for (int cb = lane * 4; cb < C; cb += 4 * 128) {
        float4 v[4];
        uint2 g[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            g[u] = *reinterpret_cast<const uint2*>(Gr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            float4 n4;
            n4.x = fmaf(p.mu, v[u].x, bf16_bits_to_float(g[u].x & 0xFFFFu));
            n4.y = fmaf(p.mu, v[u].y, bf16_bits_to_float(g[u].x >> 16));
            n4.z = fmaf(p.mu, v[u].z, bf16_bits_to_float(g[u].y & 0xFFFFu));
            n4.w = fmaf(p.mu, v[u].w, bf16_bits_to_float(g[u].y >> 16));
            *reinterpret_cast<float4*>(Vr + cc) = n4;
            ss = fmaf(n4.x, n4.x, ss);
            ss = fmaf(n4.y, n4.y, ss);
            ss = fmaf(n4.z, n4.z, ss);
            ss = fmaf(n4.w, n4.w, ss);
          }
        }
      }
    } else {
      for (int cc = lane; cc < C; cc += 32) {
        const float vn = fmaf(p.mu, Vr[cc], bf16_bits_to_float(Gr[cc]));
        Vr[cc] = vn;
        ss = fmaf(vn, vn, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) p.partials[row] = ss;
  }
}

__global__ void __launch_bounds__(256) colcut_apply_kernel(const __grid_constant__ ColcutParams p) {
  const float decay = decay_factor(p.lr, p.wd);
  const int lane = int(threadIdx.x & 31);
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = p.row_prefix[p.n];
  for (int64_t row = gw; row < total; row += nw) {
    const int ei = colcut_entry(p, row);
    const RmnpEntry& E = p.e[ei];
    const int64_t r = row - p.row_prefix[ei];
    float sum = 0.f;
    for (int s = p.first[ei]; s <= p.last[ei]; ++s) sum += p.partials[p.row_prefix[s] + r];
    const float k = p.lr * E.scale / clamp_norm(sqrtf(sum), p.eps);
    const int C = E.C;
    const size_t off = size_t(r) * size_t(C);
    const float* __restrict__ Vr = E.V + off;
    float* __restrict__ Wr = E.W + off;
    if (E.vec_ok) {
      for (int cb = lane * 4; cb < C; cb += 4 * 128) {
        float4 v[4], w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            v[u] = *reinterpret_cast<const float4*>(Vr + cc);
            w[u] = *reinterpret_cast<const float4*>(Wr + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = cb + u * 128;
          if (cc < C) {
            float4 o;
            o.x = w[u].x * decay - k * v[u].x;
            o.y = w[u].y * decay - k * v[u].y;
            o.z = w[u].z * decay - k * v[u].z;
            o.w = w[u].w * decay - k * v[u].w;
            *reinterpret_cast<float4*>(Wr + cc) = o;
          }
        }
      }
    } else {
      for (int cc = lane; cc < C; cc += 32) Wr[cc] = Wr[cc] * decay - k * Vr[cc];
    }
  }
}

// ------------------------------------------------------------------ AdamW
//
// Decoupled AdamW with bias correction on the packed tail ("MatrixFSDP",
// sections 3 and 5.1). Work items of 4096 elements; each thread handles four
// 16-byte vectors per item, loads issued before use.
// Per-step factors of AdamW, formed on the device from lr, wd and t (by
// value, or read from device memory): decay 1 - lr wd, step size
// lr / (1 - beta1^t) and 1 / sqrt(1 - beta2^t), each rounded once from double.
struct AdamFactors {
  float decay, step_size, inv_bc2_sqrt;
};

// b^e for e >= 0 by square-and-multiply (at most 2 log2(e) double products:
// far shorter than a general power on the few FP64 units)
__device__ __forceinline__ double pow_int(double b, int64_t e) {
  double r = 1.0;
  while (e > 0) {
    if (e & 1) r = __dmul_rn(r, b);
    b = __dmul_rn(b, b);
    e >>= 1;
  }
  return r;
}

__device__ __forceinline__ AdamFactors adam_factors(const AdamParams& p) {
  const float lr = p.lr_dev != nullptr ? *p.lr_dev : p.lr;
  const int64_t t = p.step_dev != nullptr ? *p.step_dev : p.step;
  const double bc1 = 1.0 - pow_int(double(p.beta1), t);
  const double bc2 = 1.0 - pow_int(double(p.beta2), t);
  AdamFactors f;
  f.decay = decay_factor(lr, p.wd);
  f.step_size = float(double(lr) / bc1);
  f.inv_bc2_sqrt = float(1.0 / sqrt(bc2));
  return f;
}

__device__ __forceinline__ void adam_elem(const AdamParams& p, const AdamFactors& f, float& pp, float g, float& m,
                                          float& v) {
  m = fmaf(p.beta1, m, (1.0f - p.beta1) * g);
  v = fmaf(p.beta2, v, (1.0f - p.beta2) * g * g);
  const float denom = fmaf(sqrtf(v), f.inv_bc2_sqrt, p.eps);
  pp = pp * f.decay - f.step_size * (m / denom);
}

__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamParams p) {
  // one thread forms the factors (double pow: slow FP64 units, so not per thread)
  __shared__ AdamFactors sf;
  if (threadIdx.x == 0) sf = adam_factors(p);
  __syncthreads();
  const AdamFactors f = sf;
  const int64_t total = p.item_prefix[p.n];
  for (int64_t it = blockIdx.x; it < total; it += gridDim.x) {
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.item_prefix[mid] <= it) lo = mid; else hi = mid - 1;
    }
    const AdamSeg& S = p.s[lo];
    const int64_t e0 = (it - p.item_prefix[lo]) * kAdamItem;
    float4 P[4], G[4], Mm[4], Vv[4];
    bool full[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t e = e0 + int64_t(u * 256 + int(threadIdx.x)) * 4;
      full[u] = e + 4 <= S.numel;
      if (full[u]) {
        P[u] = *reinterpret_cast<const float4*>(S.p + e);
        G[u] = *reinterpret_cast<const float4*>(S.g + e);
        Mm[u] = *reinterpret_cast<const float4*>(S.m + e);
        Vv[u] = *reinterpret_cast<const float4*>(S.v + e);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t e = e0 + int64_t(u * 256 + int(threadIdx.x)) * 4;
      if (full[u]) {
        adam_elem(p, f, P[u].x, G[u].x, Mm[u].x, Vv[u].x);
        adam_elem(p, f, P[u].y, G[u].y, Mm[u].y, Vv[u].y);
        adam_elem(p, f, P[u].z, G[u].z, Mm[u].z, Vv[u].z);
        adam_elem(p, f, P[u].w, G[u].w, Mm[u].w, Vv[u].w);
        *reinterpret_cast<float4*>(S.p + e) = P[u];
        *reinterpret_cast<float4*>(S.m + e) = Mm[u];
        *reinterpret_cast<float4*>(S.v + e) = Vv[u];
      } else if (e < S.numel) {
        for (int64_t j = e; j < S.numel && j < e + 4; ++j) {
          float pp = S.p[j], mm = S.m[j], vv = S.v[j];
          adam_elem(p, f, pp, S.g[j], mm, vv);
          S.p[j] = pp;
          S.m[j] = mm;
          S.v[j] = vv;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_muon_prologue(const ProParams& p, int max_grid, cudaStream_t stream) {
  if (p.nrm_total <= 0) return cudaSuccess;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const void* norm = p.nesterov ? reinterpret_cast<const void*>(muon_norm_kernel<true>)
                                : reinterpret_cast<const void*>(muon_norm_kernel<false>);
  const void* cast = p.nesterov ? reinterpret_cast<const void*>(muon_cast_kernel<true>)
                                : reinterpret_cast<const void*>(muon_cast_kernel<false>);
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm, 256, 0)) != cudaSuccess) return e;
  int64_t grid = int64_t(sms) * int64_t(std::max(per_sm, 1));
  if (max_grid > 0) grid = std::min<int64_t>(grid, max_grid);
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, p.nrm_total));
  ProParams copy = p;
  void* args[] = {&copy};
  if ((e = cudaLaunchKernel(norm, dim3(unsigned(grid)), dim3(256), args, 0, stream)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cast, 256, 0)) != cudaSuccess) return e;
  int64_t cgrid = int64_t(sms) * int64_t(std::max(per_sm, 1));
  if (max_grid > 0) cgrid = std::min<int64_t>(cgrid, max_grid);
  cgrid = std::max<int64_t>(1, std::min<int64_t>(cgrid, p.cast_total));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cgrid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, cast, args);
}

cudaError_t launch_rmnp(const RmnpParams& p, bool row_per_cta, int grid, cudaStream_t stream) {
  if (p.n <= 0 || p.row_prefix[p.n] <= 0) return cudaSuccess;
  if (row_per_cta)
    rmnp_row_cta_kernel<<<grid, 256, 0, stream>>>(p);
  else
    rmnp_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rmnp_colcut(const ColcutParams& p, int grid, cudaStream_t stream) {
  if (p.n <= 0 || p.row_prefix[p.n] <= 0) return cudaSuccess;
  colcut_partial_kernel<<<grid, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colcut_apply_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_adamw(const AdamParams& p, int grid, cudaStream_t stream) {
  if (p.n <= 0 || p.item_prefix[p.n] <= 0) return cudaSuccess;
  adamw_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mo

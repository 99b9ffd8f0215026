"""Seeded synthetic workloads for the owner-local optimizer step.

This module only describes and generates inputs: shape tables, tail sizes and
seeded random tensors with the distributions of the five benchmark
configurations, plus the work counts (flops, bytes) used to express timings as
throughput. It contains none of the optimizer arithmetic, so both the CPU
oracle tests and the GPU path can draw identical inputs from it.

Shapes follow the model families the method is evaluated on:
  * GPT-2 Large (hidden 1280, 36 layers, four 2D matrices per layer), the matrix
    set of "Optimizers In A Sharded World: Muon's O(mn) Vs RMNP's Zero",
    section 5 and its appendix benchmark script (LAYER_SHAPES).
  * Llama-style 8B and a 32B-scale owner share (hidden 5120, FFN 27648): model
    sizes of "MatrixFSDP" (arXiv 2607.05895), Table 4.
Every matrix is stored [out, in] row-major, fp32 master weight W, bf16
gradient G and fp32 momentum V.

Seeding: base seed 0 ("fixed seed 0", MatrixFSDP section 5.1), with an
independent numpy stream per (config, matrix index, role) so that any single
matrix can be regenerated without generating the rest.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

BASE_SEED = 0

# role ids for per-tensor seed streams
_ROLE_W, _ROLE_G, _ROLE_V, _ROLE_SPEC = 1, 2, 3, 4
_ROLE_TP, _ROLE_TG, _ROLE_TM, _ROLE_TV = 11, 12, 13, 14

CONFIG_NAMES = ("smoke", "gpt2l", "llama8b", "spectrum", "share32b")


@dataclasses.dataclass(frozen=True)
class MatrixSpec:
    rows: int
    cols: int
    role: str
    # "normal": W ~ N(0, w_std), G ~ N(0, g_std); "haar": G = U diag(s) V^T with
    # log-uniform s; "orthorows": G = diag(z^2) Q with orthonormal rows Q.
    kind: str = "normal"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    matrices: Tuple[MatrixSpec, ...]
    tail: Tuple[int, ...]          # AdamW tail segment sizes (fp32 elements)
    w_std: float
    g_std: float
    tail_p_std: float
    tail_g_std: float
    # hyperparameters of the configuration
    mu: float = 0.95
    ns_steps: int = 5
    lr: float = 0.02
    wd: float = 0.01
    adam_lr: float = 1e-3
    adam_wd: float = 1e-2
    beta1: float = 0.9
    beta2: float = 0.95
    adam_eps: float = 1e-8

    @property
    def n_elements(self) -> int:
        return sum(s.rows * s.cols for s in self.matrices)

    @property
    def tail_elements(self) -> int:
        return sum(self.tail)


def _gpt2l(layers: int = 36) -> Tuple[Tuple[MatrixSpec, ...], Tuple[int, ...]]:
    h = 1280
    per_layer = [MatrixSpec(3 * h, h, "qkv"), MatrixSpec(h, h, "attn_proj"),
                 MatrixSpec(4 * h, h, "fc"), MatrixSpec(h, 4 * h, "fc_proj")]
    mats = tuple(per_layer * layers)
    # Non-matrix tail: two LayerNorms (weight + bias) and the four linear biases
    # per layer, plus the final LayerNorm.
    tail_layer = [h, h, h, h, 3 * h, h, 4 * h, h]
    tail = tuple(tail_layer * layers + [h, h])
    return mats, tail


def _llama8b() -> Tuple[Tuple[MatrixSpec, ...], Tuple[int, ...]]:
    h, kv, ffn, layers, vocab = 4096, 1024, 14336, 32, 128256
    per_layer = [MatrixSpec(h, h, "q"), MatrixSpec(kv, h, "k"), MatrixSpec(kv, h, "v"),
                 MatrixSpec(h, h, "o"), MatrixSpec(ffn, h, "gate"), MatrixSpec(ffn, h, "up"),
                 MatrixSpec(h, ffn, "down")]
    mats = tuple(per_layer * layers)
    # Tail: 2 RMSNorm vectors per layer + the final norm, then the embedding and
    # the LM head, both as packed fp32 AdamW segments.
    tail = tuple([h] * (2 * layers + 1) + [vocab * h, vocab * h])
    return mats, tail


def _share32b() -> Tuple[Tuple[MatrixSpec, ...], Tuple[int, ...]]:
    h, kv, ffn, layers = 5120, 1024, 27648, 4
    per_layer = [MatrixSpec(h, h, "q"), MatrixSpec(kv, h, "k"), MatrixSpec(kv, h, "v"),
                 MatrixSpec(h, h, "o"), MatrixSpec(ffn, h, "gate"), MatrixSpec(ffn, h, "up"),
                 MatrixSpec(h, ffn, "down")]
    return tuple(per_layer * layers), (2_000_000,)


def _spectrum() -> Tuple[Tuple[MatrixSpec, ...], Tuple[int, ...]]:
    mats = ([MatrixSpec(4096, 4096, "sq", "haar")] * 16
            + [MatrixSpec(2048, 8192, "wide", "haar")] * 16
            + [MatrixSpec(8192, 2048, "tall", "haar")] * 16
            + [MatrixSpec(1024, 4096, "orthorows", "orthorows")] * 8)
    return tuple(mats), ()


def get_workload(name: str) -> Workload:
    if name == "smoke":
        return Workload("smoke", 0, (MatrixSpec(128, 256, "w"),), (1024,),
                        w_std=1.0, g_std=1.0, tail_p_std=1.0, tail_g_std=1.0)
    if name == "gpt2l":
        m, t = _gpt2l()
        return Workload("gpt2l", 1, m, t, w_std=0.02, g_std=1e-3, tail_p_std=0.02, tail_g_std=1e-3)
    if name.startswith("gpt2l_") and name.endswith("layers") and name[6:-6].isdigit():
        # the first N layers of the GPT-2 Large set (gpt2l_4layers: the same
        # kernels on a ~2 GB working set, each bf16 iterate buffer (157 MB)
        # still larger than L2; used for profiler captures)
        m, t = _gpt2l(int(name[6:-6]))
        return Workload(name, 5, m, t, w_std=0.02, g_std=1e-3, tail_p_std=0.02, tail_g_std=1e-3)
    if name == "llama8b":
        m, t = _llama8b()
        return Workload("llama8b", 2, m, t, w_std=0.02, g_std=1e-3, tail_p_std=0.02, tail_g_std=1e-3)
    if name == "gram_slices":
        # one 4096 x 40000 matrix: its Gram (n = 40000 > 32768) is summed from
        # two fp32 slice partials (2 x 64 MB, larger than L2); used to profile
        # the slice reduction
        return Workload("gram_slices", 7, (MatrixSpec(4096, 40000, "long"),), (4096,), w_std=0.02, g_std=1e-3,
                        tail_p_std=0.02, tail_g_std=1e-3)
    if name == "llama8b_1layer":
        # one layer of the Llama-style 8B set (7 matrices, 218 M elements) and a
        # tail of its two RMSNorm vectors plus one eighth of the embedding
        # (65.7 M elements, 1.05 GB of AdamW state): the same kernels on a
        # ~5 GB working set, every buffer still larger than L2; used for
        # profiler captures, whose traffic scales by 32 to the full table
        m, t = _llama8b()
        return Workload("llama8b_1layer", 6, m[:7], (4096, 4096, 128256 * 512), w_std=0.02, g_std=1e-3,
                        tail_p_std=0.02, tail_g_std=1e-3)
    if name == "spectrum":
        m, t = _spectrum()
        return Workload("spectrum", 3, m, t, w_std=0.02, g_std=1.0, tail_p_std=0.02, tail_g_std=1e-3)
    if name == "share32b":
        m, t = _share32b()
        return Workload("share32b", 4, m, t, w_std=0.02, g_std=1e-3, tail_p_std=0.02, tail_g_std=1e-3)
    raise KeyError(name)


def custom_workload(shapes: Sequence[Tuple[int, int]], tail: Sequence[int] = (),
                    w_std: float = 0.02, g_std: float = 1e-3, config_id: int = 99) -> Workload:
    """An ad-hoc table (odd and ragged shapes for edge-case tests)."""
    mats = tuple(MatrixSpec(int(r), int(c), f"m{i}") for i, (r, c) in enumerate(shapes))
    return Workload("custom", config_id, mats, tuple(int(t) for t in tail),
                    w_std=w_std, g_std=g_std, tail_p_std=w_std, tail_g_std=g_std)


# ---------------------------------------------------------------------------
# seeded generation (host, numpy)
# ---------------------------------------------------------------------------

def _rng(config_id: int, index: int, role: int, seed: int = BASE_SEED) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, config_id, index, role])))


def _haar(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """rows x cols (rows >= cols) with orthonormal columns: Haar-distributed
    via QR of a Gaussian matrix with the sign of diag(R) folded in."""
    z = rng.standard_normal((rows, cols))
    q, r = np.linalg.qr(z)
    return q * np.sign(np.diag(r))[None, :]


def spectral_factors(wl: Workload, index: int, seed: int = BASE_SEED):
    """For "haar" matrices: (U, s, Vt) in fp64 with G_exact = U diag(s) Vt.
    For "orthorows" matrices: (d, Q) with G_exact = diag(d) Q."""
    spec = wl.matrices[index]
    rng = _rng(wl.config_id, index, _ROLE_SPEC, seed)
    r, c = spec.rows, spec.cols
    k = min(r, c)
    if spec.kind == "haar":
        u = _haar(rng, r, k)
        v = _haar(rng, c, k)
        s = np.exp(rng.uniform(np.log(1e-4), np.log(1.0), size=k))
        return u, s, v.T
    if spec.kind == "orthorows":
        q = _haar(rng, c, r).T          # r x c, orthonormal rows (r <= c)
        z = rng.normal(1.0, 0.3, size=r)
        return z * z, q
    raise ValueError(spec.kind)


def exact_matrix(wl: Workload, index: int, seed: int = BASE_SEED) -> np.ndarray:
    """fp64 pre-cast gradient for the structured-spectrum matrices."""
    spec = wl.matrices[index]
    if spec.kind == "haar":
        u, s, vt = spectral_factors(wl, index, seed)
        return (u * s[None, :]) @ vt
    if spec.kind == "orthorows":
        d, q = spectral_factors(wl, index, seed)
        return d[:, None] * q
    raise ValueError(spec.kind)


def host_matrix(wl: Workload, index: int, seed: int = BASE_SEED, v_std: float = 0.0):
    """Seeded host tensors for matrix `index`: (W fp32, G bf16, V fp32) as torch
    CPU tensors. V is zero (first step) unless v_std > 0."""
    import torch
    spec = wl.matrices[index]
    shape = (spec.rows, spec.cols)
    w = _rng(wl.config_id, index, _ROLE_W, seed).standard_normal(shape, dtype=np.float32) * np.float32(wl.w_std)
    if spec.kind == "normal":
        g32 = _rng(wl.config_id, index, _ROLE_G, seed).standard_normal(shape, dtype=np.float32) * np.float32(wl.g_std)
    else:
        g32 = exact_matrix(wl, index, seed).astype(np.float32)
    if v_std > 0:
        v = _rng(wl.config_id, index, _ROLE_V, seed).standard_normal(shape, dtype=np.float32) * np.float32(v_std)
    else:
        v = np.zeros(shape, dtype=np.float32)
    w, g32, v = (np.ascontiguousarray(x) for x in (w, g32, v))
    return (torch.from_numpy(w), torch.from_numpy(g32).to(torch.bfloat16), torch.from_numpy(v))


def host_tail(wl: Workload, seg: int, seed: int = BASE_SEED, state_std: float = 0.0):
    """Seeded AdamW tail segment: (p, g, m, v) fp32 torch CPU tensors; m = v = 0
    unless state_std > 0 (then m ~ N(0, state_std), v = m^2 + |N(0, state_std)|)."""
    import torch
    n = wl.tail[seg]
    base = 1000 + seg
    p = _rng(wl.config_id, base, _ROLE_TP, seed).standard_normal(n, dtype=np.float32) * np.float32(wl.tail_p_std)
    g = _rng(wl.config_id, base, _ROLE_TG, seed).standard_normal(n, dtype=np.float32) * np.float32(wl.tail_g_std)
    if state_std > 0:
        m = _rng(wl.config_id, base, _ROLE_TM, seed).standard_normal(n, dtype=np.float32) * np.float32(state_std)
        e = _rng(wl.config_id, base, _ROLE_TV, seed).standard_normal(n, dtype=np.float32) * np.float32(state_std)
        v = m * m + np.abs(e)
    else:
        m = np.zeros(n, dtype=np.float32)
        v = np.zeros(n, dtype=np.float32)
    return tuple(torch.from_numpy(x) for x in (p, g, m, v))


# ---------------------------------------------------------------------------
# seeded generation on a CUDA device (benchmark-scale tables)
# ---------------------------------------------------------------------------

def device_matrices(wl: Workload, device, seed: int = BASE_SEED, v_std: float = 0.0):
    """W, G, V for every matrix, generated directly on `device` with torch's
    seeded generator. Used for benchmark-scale tables where host generation
    would dominate; the values differ from host_matrix()."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + wl.config_id)
    out = []
    for spec in wl.matrices:
        shape = (spec.rows, spec.cols)
        w = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(wl.w_std)
        g = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(wl.g_std).to(torch.bfloat16)
        if v_std > 0:
            v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(v_std)
        else:
            v = torch.zeros(shape, device=device, dtype=torch.float32)
        out.append((w, g, v))
    return out


def _device_haar(gen, rows: int, cols: int, device):
    """rows x cols (rows >= cols) with orthonormal columns on `device`: QR of
    a Gaussian matrix with the sign of diag(R) folded in (Haar-distributed),
    in fp32."""
    import torch
    z = torch.randn((rows, cols), generator=gen, device=device, dtype=torch.float32)
    q, r = torch.linalg.qr(z)
    return q * torch.sign(torch.diagonal(r))[None, :]


def device_structured_matrices(wl: Workload, device, seed: int = BASE_SEED):
    """W, G, V for every matrix of a table, generated on `device` with the
    structure its kind states: "haar" G = U diag(s) V^T with Haar U, V and s
    log-uniform on [1e-4, 1]; "orthorows" G = diag(z^2) Q with orthonormal
    rows Q and z ~ N(1, 0.3); "normal" G ~ N(0, g_std). W ~ N(0, w_std), V = 0.
    Used for the structured-spectrum batch at full size, where host QR of
    every matrix would dominate; the values differ from host_matrix()."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + wl.config_id + 700)
    out = []
    for spec in wl.matrices:
        r, c = spec.rows, spec.cols
        k = min(r, c)
        w = torch.randn((r, c), generator=gen, device=device, dtype=torch.float32).mul_(wl.w_std)
        if spec.kind == "haar":
            u = _device_haar(gen, r, k, device)
            v = _device_haar(gen, c, k, device)
            s = torch.empty(k, device=device, dtype=torch.float32).uniform_(math.log(1e-4), 0.0, generator=gen).exp_()
            g = (u * s[None, :]) @ v.T
        elif spec.kind == "orthorows":
            q = _device_haar(gen, c, r, device).T          # r x c, orthonormal rows (r <= c)
            z = torch.randn(r, generator=gen, device=device, dtype=torch.float32).mul_(0.3).add_(1.0)
            g = (z * z)[:, None] * q
        else:
            g = torch.randn((r, c), generator=gen, device=device, dtype=torch.float32).mul_(wl.g_std)
        out.append((w, g.to(torch.bfloat16).contiguous(), torch.zeros_like(w)))
    return out


def device_tail(wl: Workload, device, seed: int = BASE_SEED):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + wl.config_id + 500)
    out = []
    for n in wl.tail:
        p = torch.randn(n, generator=gen, device=device).mul_(wl.tail_p_std)
        g = torch.randn(n, generator=gen, device=device).mul_(wl.tail_g_std)
        out.append((p, g, torch.zeros_like(p), torch.zeros_like(p)))
    return out


# ---------------------------------------------------------------------------
# work counts used to express timings as throughput
# ---------------------------------------------------------------------------

def ns_shape(rows: int, cols: int) -> Tuple[int, int]:
    """(m, n) of the Newton-Schulz operand: m = min, n = max."""
    return (rows, cols) if rows <= cols else (cols, rows)


def ns_alg_flops(rows: int, cols: int, steps: int = 5) -> int:
    """Algorithmic flops of `steps` quintic iterations on one matrix, counting
    only the unique half of the symmetric products: per iteration m^2 n (Gram,
    upper triangle) + m^3 (A.A, upper triangle) + 2 m^2 n (B.X)."""
    m, n = ns_shape(rows, cols)
    return steps * (3 * m * m * n + m ** 3)


def ns_dense_flops(rows: int, cols: int, steps: int = 5) -> int:
    """Dense-equivalent flops: 2 m^2 n + 2 m^3 + 2 m^2 n per iteration."""
    m, n = ns_shape(rows, cols)
    return steps * (4 * m * m * n + 2 * m ** 3)


# algorithmic HBM bytes per element
PROLOGUE_BYTES_PER_EL = 12       # G 2 + V 4+4 + X0 2 (momentum, norm, bf16 cast)
MUON_NONGEMM_BYTES_PER_EL = 20   # the prologue's 12 + W 4+4 (update)
RMNP_BYTES_PER_EL = 18           # G 2 + V 4+4 + W 4+4
ADAMW_BYTES_PER_EL = 28          # p, m, v read + write (24) + g read (4)


def workload_alg_flops(wl: Workload, steps: Optional[int] = None) -> int:
    st = wl.ns_steps if steps is None else steps
    return sum(ns_alg_flops(s.rows, s.cols, st) for s in wl.matrices)


def owner_roles(wl: Workload, matrices_per_block: int) -> List[Tuple[int, int, int]]:
    """Planner roles (numel, block, is_tail) of a table whose matrices come in
    blocks of `matrices_per_block` (one transformer layer per block); each
    block's tail role is its share of the tail segments, in order."""
    nblocks = len(wl.matrices) // matrices_per_block
    roles = []
    for b in range(nblocks):
        for s in wl.matrices[b * matrices_per_block:(b + 1) * matrices_per_block]:
            roles.append((s.rows * s.cols, b, 0))
    if wl.tail:
        per = max(1, len(wl.tail) // max(1, nblocks))
        for b in range(nblocks):
            seg = wl.tail[b * per:(b + 1) * per] if b < nblocks - 1 else wl.tail[b * per:]
            if seg:
                roles.append((sum(seg), b, 1))
    return roles

"""GPU parity of rmnp_step and adamw_tail_step (through the C ABI) against the
CPU oracle: max |gpu - ref| / max |ref| <= 1e-5 for every fp32 output, plus
the row-sharded exactness of RMNP (max difference exactly 0, "Optimizers In A
Sharded World", section 5)."""
import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import FP32_MAX_REL_TOL, f64, max_rel, shape_scale, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def rmnp_check(host_mats, params):
    dev = to_device(host_mats, DEV)
    mo.rmnp_step(dev, params)
    torch.cuda.synchronize()
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host_mats, dev):
        Wn, Vn, D = oracle.rmnp_matrix_step(f64(Wh), f64(Gh), f64(Vh), lr=params.lr, wd=params.wd,
                                            mu=params.mu, eps=params.eps)
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        assert max_rel(f64(Wd), Wn) <= FP32_MAX_REL_TOL
    return dev


def test_rmnp_smoke():
    wl = workloads.get_workload("smoke")
    rmnp_check([workloads.host_matrix(wl, 0)], mo.RmnpParams(lr=0.02, wd=0.01, mu=0.95))


@pytest.mark.parametrize("shape", [(130, 257), (1, 9), (9, 1), (33, 4096), (16, 27648), (5, 14336), (7, 130)])
def test_rmnp_shapes_direction(shape):
    """W = 0, lr = 1, wd = 0 exposes -s D directly."""
    wl = workloads.custom_workload([shape], w_std=0.0, g_std=1.0)
    host = [workloads.host_matrix(wl, 0, v_std=0.5)]
    dev = to_device(host, DEV)
    mo.rmnp_step(dev, mo.RmnpParams(lr=1.0, wd=0.0, mu=0.9))
    torch.cuda.synchronize()
    W, G, V = host[0]
    _, Vn, D = oracle.rmnp_matrix_step(f64(W), f64(G), f64(V), lr=1.0, wd=0.0, mu=0.9)
    got = -f64(dev[0][0]) / shape_scale(*shape)
    assert max_rel(got, D) <= FP32_MAX_REL_TOL
    assert max_rel(f64(dev[0][2]), Vn) <= FP32_MAX_REL_TOL


def test_rmnp_zero_row():
    W = torch.zeros(4, 64, device=DEV)
    G = torch.zeros(4, 64, device=DEV, dtype=torch.bfloat16)
    G[1] = 1.0
    V = torch.zeros(4, 64, device=DEV)
    mo.rmnp_step([(W, G, V)], mo.RmnpParams(lr=1.0, wd=0.0, mu=0.0))
    torch.cuda.synchronize()
    assert torch.all(W[0] == 0) and torch.all(W[2:] == 0)
    assert torch.allclose(W[1], torch.full((64,), -1.0 / 8.0, device=DEV))


def test_rmnp_heterogeneous_gpt2l_layer():
    wl = workloads.get_workload("gpt2l")
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(4)]
    rmnp_check(host, mo.RmnpParams())


def test_rmnp_row_sharded_exact():
    """Virtual row shards (row blocks as separate table entries, with the
    whole matrix's scale) give bit-identical updates to the unsharded call
    (the page's exactness check: 512 x 384, seed 7, 8 shards)."""
    m, n, shards = 512, 384, 8
    full = torch.randn(m, n, generator=torch.Generator().manual_seed(7))
    W1 = torch.zeros(m, n, device=DEV)
    V1 = full.to(DEV)
    G1 = torch.zeros(m, n, device=DEV, dtype=torch.bfloat16)
    W2, V2, G2 = W1.clone(), V1.clone(), G1.clone()
    p = mo.RmnpParams(lr=1.0, wd=0.0, mu=1.0)
    mo.rmnp_step([(W1, G1, V1)], p)
    blocks = [(W2[r * m // shards:(r + 1) * m // shards], G2[r * m // shards:(r + 1) * m // shards],
               V2[r * m // shards:(r + 1) * m // shards]) for r in range(shards)]
    mo.rmnp_step_scaled(blocks, [shape_scale(m, n)] * shards, p)
    torch.cuda.synchronize()
    assert float((W1 - W2).abs().max()) == 0.0
    assert torch.equal(V1, V2)


def test_rmnp_gpt2l_full_table_sampled():
    wl = workloads.get_workload("gpt2l")
    dev = workloads.device_matrices(wl, DEV, v_std=1e-3)
    sample = [0, 1, 2, 3, 100]
    snap = {i: tuple(f64(t) for t in dev[i]) for i in sample}
    p = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
    mo.rmnp_step(dev, p)
    torch.cuda.synchronize()
    for i in sample:
        W0, G0, V0 = snap[i]
        Wn, Vn, _ = oracle.rmnp_matrix_step(W0, G0, V0, lr=p.lr, wd=p.wd, mu=p.mu)
        assert max_rel(f64(dev[i][0]), Wn) <= FP32_MAX_REL_TOL
        assert max_rel(f64(dev[i][2]), Vn) <= FP32_MAX_REL_TOL


# ---------------------------------------------------------------- AdamW

def adam_check(sizes, steps=3, state_std=0.0, params=None):
    wl = workloads.custom_workload([], tail=sizes)
    host = [workloads.host_tail(wl, i, state_std=state_std) for i in range(len(sizes))]
    dev = [tuple(t.to(DEV) for t in seg) for seg in host]
    ref = [(f64(pp), f64(m), f64(v)) for (pp, _, m, v) in host]
    base = params or mo.AdamWParams()
    for step in range(1, steps + 1):
        p = mo.AdamWParams(lr=base.lr, wd=base.wd, beta1=base.beta1, beta2=base.beta2, eps=base.eps, step=step)
        gs = [torch.randn(n, generator=torch.Generator().manual_seed(50 + step)).mul_(1e-3) for n in sizes]
        dev = [(pp, g.to(DEV), m, v) for (pp, _, m, v), g in zip(dev, gs)]
        mo.adamw_tail_step(dev, p)
        ref = [oracle.adamw_step(pp, f64(g), m, v, lr=p.lr, wd=p.wd, beta1=p.beta1, beta2=p.beta2,
                                 eps=p.eps, step=step) for (pp, m, v), g in zip(ref, gs)]
    torch.cuda.synchronize()
    for (pd, _, md, vd), (pr, mr, vr) in zip(dev, ref):
        assert max_rel(f64(pd), pr) <= FP32_MAX_REL_TOL
        assert max_rel(f64(md), mr) <= FP32_MAX_REL_TOL
        assert max_rel(f64(vd), vr) <= FP32_MAX_REL_TOL


def test_adamw_smoke_tail():
    adam_check([1024], steps=1)


def test_adamw_odd_sizes_and_many_segments():
    adam_check([1, 3, 4, 5, 4095, 4097, 10_000, 123_457], steps=3)


def test_adamw_gpt2l_tail():
    wl = workloads.get_workload("gpt2l")
    adam_check(list(wl.tail), steps=2, state_std=1e-3)


def test_adamw_update_direction_exposed():
    """p = 0, wd = 0: the first step writes -lr g / (|g| + eps) exactly."""
    n = 70_001
    g = torch.randn(n, generator=torch.Generator().manual_seed(3)).mul_(1e-2)
    p, m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    mo.adamw_tail_step([(p, g.to(DEV), m, v)], mo.AdamWParams(lr=1.0, wd=0.0, step=1))
    torch.cuda.synchronize()
    ref = -g.double().numpy() / (np.abs(g.double().numpy()) + 1e-8)
    assert max_rel(f64(p), ref) <= FP32_MAX_REL_TOL


def test_adamw_more_than_one_launch_of_segments():
    adam_check([17] * 300, steps=1)


# ---------------------------------------------------------------- column-cut RMNP

def _cut(t, widths):
    out, c = [], 0
    for w in widths:
        out.append(t[:, c:c + w].contiguous())
        c += w
    return out


def test_rmnp_colcut_parity_and_equivalence():
    """Rows cut into column shards (the page's column-cut layout: 8 shards of
    a 3840 x 1280 qkv-shaped matrix, plus an uneven 2-way cut): each shard
    matches the oracle's column-cut step, and reassembled they match the
    unsharded RMNP step within fp32 reassociation."""
    p = mo.RmnpParams(lr=0.02, wd=0.01, mu=0.95, eps=1e-7)
    specs = [((3840, 1280), [160] * 8), ((64, 128), [100, 28]), ((33, 257), [257])]
    shards, groups, scales, refs = [], [], [], []
    for gi, ((R, C), widths) in enumerate(specs):
        wl = workloads.custom_workload([(R, C)], g_std=1e-3, config_id=70 + gi)
        W, G, V = workloads.host_matrix(wl, 0, v_std=1e-3)
        Ws, Gs, Vs = _cut(W, widths), _cut(G, widths), _cut(V, widths)
        for w, g, v in zip(Ws, Gs, Vs):
            shards.append((w.to(DEV), g.to(DEV), v.to(DEV)))
            groups.append(gi)
            scales.append(shape_scale(R, C))
        refs.append(((R, C), widths, oracle.rmnp_colcut_matrix_step(
            [f64(w) for w in Ws], [f64(g) for g in Gs], [f64(v) for v in Vs], R, C, lr=p.lr, wd=p.wd, mu=p.mu,
            eps=p.eps), (W, G, V)))
    mo.rmnp_colcut_step(shards, groups, scales, p)
    torch.cuda.synchronize()
    k = 0
    for (R, C), widths, (Wn, Vn, _), (W, G, V) in refs:
        got_w, got_v = [], []
        for j in range(len(widths)):
            assert max_rel(f64(shards[k][0]), Wn[j]) <= FP32_MAX_REL_TOL
            assert max_rel(f64(shards[k][2]), Vn[j]) <= FP32_MAX_REL_TOL
            got_w.append(f64(shards[k][0]))
            got_v.append(f64(shards[k][2]))
            k += 1
        # reassembled: the unsharded RMNP step on the whole matrix
        Wd, Gd, Vd = W.to(DEV), G.to(DEV), V.to(DEV)
        mo.rmnp_step([(Wd, Gd, Vd)], mo.RmnpParams(lr=p.lr, wd=p.wd, mu=p.mu))
        torch.cuda.synchronize()
        assert max_rel(np.concatenate(got_w, axis=1), f64(Wd)) <= FP32_MAX_REL_TOL
        assert max_rel(np.concatenate(got_v, axis=1), f64(Vd)) <= FP32_MAX_REL_TOL


def test_rmnp_colcut_validation():
    W = torch.zeros(8, 16, device=DEV)
    G = torch.zeros(8, 16, device=DEV, dtype=torch.bfloat16)
    V = torch.zeros(8, 16, device=DEV)
    W2, G2, V2 = W.clone(), G.clone(), V.clone()
    with pytest.raises(mo.MoError):      # a group split across the table
        mo.rmnp_colcut_step([(W, G, V), (W2, G2, V2), (W.clone(), G.clone(), V.clone())], [0, 1, 0], [1, 1, 1])
    with pytest.raises(mo.MoError):      # shards of one matrix with different rows
        mo.rmnp_colcut_step([(W, G, V), (W2[:4], G2[:4], V2[:4])], [0, 0], [1, 1])


# ---------------------------------------------------------------- HTRMNP (a reading: see include/mo.h)

@pytest.mark.parametrize("shape", [(130, 257), (1, 9), (33, 4096), (16, 27648), (5, 14336), (7, 130)])
@pytest.mark.parametrize("power", [0.125, 0.5])
def test_htrmnp_direction(shape, power):
    """W = 0, lr = 1, wd = 0 exposes -s D; rows of 8192 elements or more run
    on the CTA-per-row kernel, the others on the warp-per-row one."""
    wl = workloads.custom_workload([shape], w_std=0.0, g_std=1.0)
    host = [workloads.host_matrix(wl, 0, v_std=0.5)]
    dev = to_device(host, DEV)
    mo.htrmnp_step(dev, mo.RmnpParams(lr=1.0, wd=0.0, mu=0.9), power=power)
    torch.cuda.synchronize()
    W, G, V = host[0]
    _, Vn, D = oracle.htrmnp_matrix_step(f64(W), f64(G), f64(V), lr=1.0, wd=0.0, mu=0.9, power=power)
    got = -f64(dev[0][0]) / shape_scale(*shape)
    assert max_rel(got, D) <= FP32_MAX_REL_TOL
    assert max_rel(f64(dev[0][2]), Vn) <= FP32_MAX_REL_TOL


def test_htrmnp_power_zero_is_rmnp_bit_exactly():
    wl = workloads.custom_workload([(64, 1280), (17, 9000)], g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(2)]
    a, b = to_device(host, DEV), to_device(host, DEV)
    mo.rmnp_step(a, mo.RmnpParams())
    mo.htrmnp_step(b, mo.RmnpParams(), power=0.0)
    torch.cuda.synchronize()
    for (Wa, _, Va), (Wb, _, Vb) in zip(a, b):
        assert torch.equal(Wa, Wb) and torch.equal(Va, Vb)


def test_htrmnp_gpt2l_layer():
    wl = workloads.get_workload("gpt2l")
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(4)]
    dev = to_device(host, DEV)
    p = mo.RmnpParams()
    mo.htrmnp_step(dev, p)
    torch.cuda.synchronize()
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host, dev):
        Wn, Vn, _ = oracle.htrmnp_matrix_step(f64(Wh), f64(Gh), f64(Vh), lr=p.lr, wd=p.wd, mu=p.mu, eps=p.eps)
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        assert max_rel(f64(Wd), Wn) <= FP32_MAX_REL_TOL


def test_rmnp_more_than_one_launch_of_entries():
    """700 entries (two launches of at most 512), short and long rows mixed
    (both RMNP kernels, each with its own launches)."""
    rng = np.random.default_rng(78)
    shapes = [(int(rng.integers(1, 9)), int(rng.choice([7, 64, 1000, 8192, 9001]))) for _ in range(700)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    rmnp_check(host, mo.RmnpParams())

"""AdamW and RMNP with device-resident hyperparameters (adamw_tail_step_dev,
rmnp_step_dev), captured in CUDA graphs and replayed under a schedule. The
device-parameter entry points run the same kernels as the by-value ones and
form the same per-step factors on the device, so the bar is exact equality
with the by-value entry points given the same step counts and learning rates
(which the other GPU tests hold to the oracle)."""
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TAIL = [1, 5, 4097, 10_000, 123_457]
LRS = [1e-3, 8e-4, 5e-4, 2e-4]


def _tail_pair():
    wl = workloads.custom_workload([], tail=TAIL)
    host = [workloads.host_tail(wl, i, state_std=1e-3) for i in range(len(TAIL))]
    return ([tuple(t.to(DEV) for t in seg) for seg in host], [tuple(t.to(DEV) for t in seg) for seg in host])


def _tail_grads(step):
    gen = torch.Generator().manual_seed(70 + step)
    return [torch.randn(n, generator=gen).mul_(1e-3) for n in TAIL]


def test_adamw_device_step_and_lr_in_graph():
    """Step 1 eagerly, then a graph holding `step += 1` and the AdamW launch,
    replayed for steps 2..4 with new gradients and learning rates."""
    ref, got = _tail_pair()
    for t, lr in enumerate(LRS, start=1):
        for (_, g, _, _), gn in zip(ref, _tail_grads(t)):
            g.copy_(gn.to(DEV))
        mo.adamw_tail_step(ref, mo.AdamWParams(lr=lr, step=t))

    params = mo.AdamWParams(lr=123.0, step=99)            # both ignored: read from device memory
    step = torch.ones(1, dtype=torch.int64, device=DEV)
    lr = torch.full((1,), LRS[0], dtype=torch.float32, device=DEV)
    table = mo.TailTable(got)
    for (_, g, _, _), gn in zip(got, _tail_grads(1)):
        g.copy_(gn.to(DEV))
    mo.adamw_tail_step_dev(table, params, step, lr)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.add_(1)
        mo.adamw_tail_step_dev(table, params, step, lr)
    for t, lr_t in enumerate(LRS[1:], start=2):
        for (_, g, _, _), gn in zip(got, _tail_grads(t)):
            g.copy_(gn.to(DEV))
        lr.fill_(lr_t)
        graph.replay()
    torch.cuda.synchronize()
    assert int(step.item()) == len(LRS)
    for a, b in zip(ref, got):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_adamw_device_step_without_device_lr():
    ref, got = _tail_pair()
    p = mo.AdamWParams(lr=7e-4, step=3)
    for (_, g, _, _), gn in zip(ref, _tail_grads(3)):
        g.copy_(gn.to(DEV))
    for (_, g, _, _), gn in zip(got, _tail_grads(3)):
        g.copy_(gn.to(DEV))
    mo.adamw_tail_step(ref, p)
    mo.adamw_tail_step_dev(got, mo.AdamWParams(lr=7e-4, step=1), torch.full((1,), 3, dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("power", [0.0, 0.125])
def test_rmnp_device_lr_in_graph(power):
    """RMNP (power 0) and the HTRMNP reading: a captured launch replayed with
    new gradients and learning rates, against the by-value entry points.
    Short and long rows (two kernels) are both in the table."""
    shapes = [(130, 257), (16, 9000), (64, 64)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    ref = [tuple(t.to(DEV) for t in m) for m in host]
    got = [tuple(t.to(DEV) for t in m) for m in host]
    gen = torch.Generator().manual_seed(3)
    grads = [[(torch.randn(W.shape, generator=gen) * 1e-3).to(torch.bfloat16) for W, _, _ in host] for _ in LRS]
    for lr_t, gs in zip(LRS, grads):
        for (_, G, _), g in zip(ref, gs):
            G.copy_(g.to(DEV))
        p = mo.RmnpParams(lr=lr_t)
        if power == 0.0:
            mo.rmnp_step(ref, p)
        else:
            mo.htrmnp_step(ref, p, power=power)

    table = mo.MuonTable(got)
    lr = torch.full((1,), LRS[0], dtype=torch.float32, device=DEV)
    params = mo.RmnpParams(lr=float("nan"))             # ignored: lr is read from device memory
    for (_, G, _), g in zip(got, grads[0]):
        G.copy_(g.to(DEV))
    mo.rmnp_step_dev(table, params, lr, power=power)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mo.rmnp_step_dev(table, params, lr, power=power)
    for lr_t, gs in zip(LRS[1:], grads[1:]):
        for (_, G, _), g in zip(got, gs):
            G.copy_(g.to(DEV))
        lr.fill_(lr_t)
        graph.replay()
    torch.cuda.synchronize()
    for (Wa, _, Va), (Wb, _, Vb) in zip(ref, got):
        assert torch.equal(Wa, Wb) and torch.equal(Va, Vb)

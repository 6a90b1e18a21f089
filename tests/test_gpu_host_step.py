"""vsa_train_step_host (the step from host buffers, head slices pipelined
with the copies): its outputs equal the device path's bit for bit -- every
head is an independent problem and each slice runs the same kernels -- and
the device path is checked against the oracle by the parity tests. One
small case is also checked against the oracle directly."""
import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, make_tensors
from oracle import oracle as orc
from tests.helpers import GRAD_TOL, OUT_TOL, check_tol, plan_for, to_device

pytestmark = pytest.mark.gpu


def cases():
    return [
        (Problem("host-bshd-gqa", "bshd", 2, 8, 4, 128, 256, 256, 3, 5, q_var=[256, 256, 200],
                 kv_var=[256, 77, 256, 0, 256], topk=3, seed=71), 2),
        (Problem("host-bhsd", "bhsd", 2, 6, 6, 128, 128, 256, 4, 3, q_var=[128] * 4, kv_var=[256, 130, 9],
                 topk=2, seed=72), 3),
        (Problem("host-tnd-fp16", "tnd", 3, 4, 2, 128, 256, 128, 3, 5, dtype="fp16", q_lens=[300, 17, 513],
                 kv_lens=[540, 23, 200], topk=3, seed=73), 2),
        (Problem("host-one-group", "bshd", 1, 2, 1, 128, 256, 256, 2, 3, q_var=[256, 256], kv_var=[256] * 3,
                 topk=2, seed=74), 1),
        (Problem("host-gated-ragged", "bshd", 1, 4, 4, 128, 256, 256, 3, 5, q_var=[256, 160, 256],
                 kv_var=[256, 160, 64, 40, 256], topk=3, gate="uniform_token_head", seed=75), 2),
        (Problem("host-twelve-heads", "bshd", 1, 12, 12, 128, 256, 256, 2, 4, q_var=[256, 256],
                 kv_var=[256, 256, 100, 256], topk=2, seed=76), 4),
    ]


def host(x):
    return x.detach().cpu().contiguous().pin_memory()


@pytest.mark.parametrize("case", cases(), ids=lambda c: c[0].name)
def test_host_step_equals_device_path(case):
    p, groups = case
    t = make_tensors(p)
    g = to_device(t)
    plan = plan_for(p)
    plan.build_block_map(g["q"], g["k"], p.topk)
    gate = g.get("gate")
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=gate)
    dq, dk, dv = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=gate)
    torch.cuda.synchronize()

    hp = plan_for(p)
    h_out = torch.empty(g["q"].shape, dtype=g["q"].dtype, pin_memory=True)
    h_lse = torch.empty(tuple(lse.shape), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.Stream()
    o2, l2, dq2, dk2, dv2 = hp.train_step_host(host(g["q"]), host(g["k"]), host(g["v"]), host(g["dO"]), p.topk,
                                               groups, gate=None if gate is None else host(gate), out=h_out,
                                               lse=h_lse, stream=stream)
    stream.synchronize()
    assert hp.host_step_status(stream) == 0
    for name, a, b in (("out", out, o2), ("dq", dq, dq2), ("dk", dk, dk2), ("dv", dv, dv2)):
        assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16)), name
    assert torch.equal(lse.cpu(), l2)

    if p.name in ("host-one-group", "host-gated-ragged"):  # and directly against the oracle
        ref = orc.run_full(p, t)
        check_tol("host out", ref["out"], o2.double().numpy(), OUT_TOL)
        for n, x in (("dq", dq2), ("dk", dk2), ("dv", dv2)):
            check_tol(f"host {n}", ref[n], x.double().numpy(), GRAD_TOL)


@pytest.mark.parametrize("case", [c for c in cases() if c[0].name in ("host-bshd-gqa", "host-tnd-fp16",
                                                                      "host-gated-ragged")],
                         ids=lambda c: c[0].name)
def test_fwd_step_host_equals_device_forward(case):
    """vsa_fwd_step_host (inference: block map without the KV-owned index,
    forward) equals the device forward bit for bit."""
    p, groups = case
    t = make_tensors(p)
    g = to_device(t)
    plan = plan_for(p)
    plan.build_block_map(g["q"], g["k"], p.topk, need_bwd_index=False)
    gate = g.get("gate")
    out, lse, _ = plan.forward(g["q"], g["k"], g["v"], gate=gate)
    torch.cuda.synchronize()
    hp = plan_for(p)
    h_lse = torch.empty(tuple(lse.shape), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.Stream()
    o2, l2 = hp.fwd_step_host(host(g["q"]), host(g["k"]), host(g["v"]), p.topk, groups,
                              gate=None if gate is None else host(gate), lse=h_lse, stream=stream)
    stream.synchronize()
    assert hp.host_step_status(stream) == 0
    assert torch.equal(out.cpu().view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse.cpu(), l2)

"""The failure path of the bounded mbarrier waits, exercised on the GPU
without a fault: a wait on a barrier that nothing arrives on gives up after
its limit, records its site code in the status word, and the context keeps
working (a block map + forward + backward right after is still correct)."""
import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300 import vsa
from bwd_tile_mean_gb300.inputs import config, make_tensors
from oracle import oracle as orc
from tests.helpers import GRAD_TOL, OUT_TOL, check_tol, plan_for, to_device

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_reports():
    p = config(1)
    plan = plan_for(p)
    assert plan.device_status() == 0
    assert vsa.check_wait_timeout(plan.workspace, limit_ns=50_000_000) == 0   # gave up, did not "complete"
    assert plan.device_status() == 0x7E57                                      # the site code, then cleared
    assert plan.device_status() == 0
    # the context is intact: the full path still matches the oracle
    t = make_tensors(p)
    g = to_device(t)
    plan.build_block_map(g["q"], g["k"], p.topk)
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"])
    dq, dk, dv = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref = orc.run_full(p, t)
    assert np.array_equal(plan.q_idx.cpu().numpy(), ref["q_idx"])
    check_tol("out", ref["out"], out.double().cpu().numpy(), OUT_TOL)
    for n, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tol(n, ref[n], x.double().cpu().numpy(), GRAD_TOL)

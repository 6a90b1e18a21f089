"""Kernels whose shared memory grows with the problem (the compression
passes) must launch for a larger problem after a smaller one in the same
process: the dynamic shared-memory limit a first launch sets has to be
raised, not kept. Run in a fresh process, where no earlier launch has
raised the limit already."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import torch
    from bwd_tile_mean_gb300.inputs import Problem, make_tensors
    from tests.helpers import plan_for, to_device
    # small first (a few KB of shared memory), then one past 48 KB
    for nkv in (4, 600):
        p = Problem(f"gated-{{nkv}}", "bshd", 1, 2, 2, 128, 256, 256, 3, nkv, q_var=[256, 200, 256],
                    kv_var=[256] * (nkv - 1) + [77], topk=2, gate="randn01", seed=nkv)
        g = to_device(make_tensors(p))
        plan = plan_for(p)
        plan.build_block_map(g["q"], g["k"], p.topk)
        out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=g["gate"])
        dq, dk, dv = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=g["gate"])
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert all(torch.isfinite(x).all() for x in (out, dq, dk, dv))
    print("ok")
""")


def test_growing_shared_memory_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]

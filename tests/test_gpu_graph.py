"""A whole training step (block map, forward, backward) captured in a CUDA
graph and replayed gives bit-identical results to running it eagerly: no
call on the path allocates, synchronises or depends on host-side state that
changes between calls."""
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, config, make_tensors
from tests.helpers import plan_for, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("p", [config(1),
                               Problem("graph-gated", "bshd", 1, 4, 2, 128, 256, 256, 3, 5, q_var=[256, 160, 256],
                                       kv_var=[256, 160, 64, 40, 256], topk=3, gate="uniform_token_head", seed=81)],
                         ids=lambda p: p.name)
def test_step_in_cuda_graph_matches_eager(p):
    t = to_device(make_tensors(p))
    plan = plan_for(p)
    gate = t.get("gate")
    out = torch.empty_like(t["q"])
    osp = torch.empty_like(t["q"]) if gate is not None else None
    lse = torch.empty(plan.lse_shape(), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])

    def step():
        plan.build_block_map(t["q"], t["k"], p.topk)
        plan.forward(t["q"], t["k"], t["v"], gate=gate, out=out, lse=lse, o_sparse=osp)
        plan.backward(t["dO"], t["q"], t["k"], t["v"], osp if gate is not None else out, lse, gate=gate,
                      dq=dq, dk=dk, dv=dv)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager, on the capture stream (first launches set kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (out, lse, dq, dk, dv, plan.block_map, plan.q_idx)]
    for x in (out, dq, dk, dv):
        x.zero_()
    lse.zero_()
    plan.block_map.zero_()
    plan.q_idx.zero_()
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv", "map", "q_idx"), eager,
                          (out, lse, dq, dk, dv, plan.block_map, plan.q_idx)):
        assert torch.equal(a, b), name

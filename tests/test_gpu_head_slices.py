"""A problem's heads split with vsa_head_slice (the split that puts each
slice on its own GPU, with no exchange between them) give, slice by slice,
results bitwise equal to the whole problem's: block map, both indices, O,
LSE, dQ, dK and dV. Every (batch, head) is an independent problem (Ascend
test_npu_block_sparse_attention_backward.py, the per-(batch, head) loops of
the TND/GQA golden, key/value head h // (Hq / Hkv)). Runs the slices one
after another on one GPU."""
import pytest
import torch

from bwd_tile_mean_gb300 import vsa
from bwd_tile_mean_gb300.inputs import DTYPES, Problem, make_tensors, tnd_problem
from tests.helpers import plan_for, to_device

pytestmark = pytest.mark.gpu


def _step(plan, t, topk):
    plan.build_block_map(t["q"], t["k"], topk, need_bwd_index=True)
    out, lse, osp = plan.forward(t["q"], t["k"], t["v"])
    dq, dk, dv = plan.backward(t["dO"], t["q"], t["k"], t["v"], osp, lse)
    torch.cuda.synchronize()
    return dict(block_map=plan.block_map.clone(), q_idx=plan.q_idx.clone(), q_cnt=plan.q_cnt.clone(),
                kv_ptr=plan.kv_ptr.clone(), kv_qidx=plan.kv_qidx.clone(), out=out, lse=lse, dq=dq, dk=dk, dv=dv)


def _head_dim(p, name):
    if name in ("block_map", "q_idx", "q_cnt", "kv_ptr", "kv_qidx"):
        return 1
    if name == "lse":
        return 0 if p.layout == "tnd" else 1
    return {"bhsd": 1, "bshd": 2, "tnd": 1}[p.layout]


@pytest.mark.parametrize("layout,groups", [("bshd", 2), ("bhsd", 4), ("tnd", 2)])
def test_head_slices_equal_the_whole_problem(layout, groups):
    if layout == "tnd":
        p = tnd_problem("slices-tnd", [300, 7, 129], [50, 520, 256], 8, 4, dtype="bf16", topk=2, seed=71)
    else:
        p = Problem("slices", layout, 2, 8, 4, 128, 256, 256, 4, 6, q_var=[256, 61, 199, 256],
                    kv_var=[256, 173, 0, 79, 256, 12], topk=3, seed=71)
    t = to_device(make_tensors(p))
    whole = _step(plan_for(p), t, p.topk)
    ref = plan_for(p)
    parts = []
    for g in range(groups):
        sd, q0, kv0 = vsa.vsa_head_slice(ref.desc, groups, g)
        hd = {"bhsd": 1, "bshd": 2, "tnd": 1}[p.layout]
        ts = {n: x.narrow(hd, q0 if n in ("q", "dO") else kv0, sd.Hq if n in ("q", "dO") else sd.Hkv).contiguous()
              for n, x in t.items()}
        plan = vsa.Plan(p.layout, DTYPES[p.dtype], p.B, sd.Hq, sd.Hkv, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV,
                        p.Sq, p.Skv, p.cap, q_var=ref.q_var, kv_var=ref.kv_var, cu_seqlens_q=ref.cu_q,
                        cu_seqlens_kv=ref.cu_kv, scale=p.scale, device="cuda")
        parts.append(_step(plan, ts, p.topk))
    for name, want in whole.items():
        got = torch.cat([x[name] for x in parts], dim=_head_dim(p, name))
        assert torch.equal(got, want), name

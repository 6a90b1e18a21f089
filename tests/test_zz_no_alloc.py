"""vsa_build_block_map_static: the block-map entry point for callers that
may not allocate device memory (a runtime or memory pool that owns all of
it, an allocator that forbids outside allocations, a path where an
allocation could synchronise or fail). Its scratch is a fixed array inside
the library. It must give the same
block map and indices as vsa_build_block_map, bit for bit, on two calls in
a row (the array keeps the previous call's contents)."""
import pytest
import torch

from bwd_tile_mean_gb300 import vsa
from bwd_tile_mean_gb300.inputs import Problem, make_tensors, tnd_problem
from tests.helpers import plan_for

pytestmark = pytest.mark.gpu


def _outputs(plan):
    return [plan.block_map.clone(), plan.q_idx.clone(), plan.q_cnt.clone(), plan.kv_ptr.clone(),
            plan.kv_qidx.clone()]


def test_static_scratch_matches_workspace_entry_point_twice():
    problems = [
        Problem("noalloc-a", "bshd", 1, 4, 2, 128, 256, 256, 6, 9, q_var=[256, 61, 199, 256, 0, 256],
                kv_var=[256, 173, 0, 79, 256, 256, 12, 256, 128], topk=3, seed=41),
        Problem("noalloc-b", "bhsd", 2, 2, 2, 128, 128, 128, 5, 7, q_var=[128] * 5,
                kv_var=[128, 5, 128, 0, 77, 128, 1], topk=2, seed=42, dtype="fp16"),
        tnd_problem("noalloc-tnd", [300, 17, 129, 256], [540, 23, 200, 383], 6, 3, dtype="fp16", topk=2,
                    seed=43),
        # just under the array's size: 16 * 1000 * 128 * 2 = 4,096,000 of 4,194,304 floats
        Problem("noalloc-near-limit", "bshd", 1, 16, 16, 128, 128, 128, 1000, 1000, q_var=[128] * 1000,
                kv_var=[128] * 999 + [77], topk=8, seed=44),
    ]
    for p in problems:  # two calls in a row, on different problems, reuse the array
        t = make_tensors(p, device="cuda")
        ref = plan_for(p)
        ref.build_block_map(t["q"], t["k"], p.topk, need_bwd_index=True)
        want = _outputs(ref)
        for _ in range(2):
            got = plan_for(p)
            vsa.vsa_build_block_map_static(got.desc, t["q"], t["k"], got.q_var, got.kv_var, p.topk, True,
                                           got.block_map, got.q_idx, got.q_cnt, got.idx_cap, got.kv_ptr,
                                           got.kv_qidx)
            torch.cuda.synchronize()
            for a, b in zip(want, _outputs(got)):
                assert torch.equal(a, b)


def test_static_scratch_rejects_problems_beyond_its_size():
    p = Problem("too-big", "bshd", 1, 64, 64, 128, 256, 256, 300, 300, q_var=[256] * 300, kv_var=[256] * 300,
                topk=4)
    plan = plan_for(p)
    q = torch.zeros(p.shape(True), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vsa.VsaError) as e:
        vsa.vsa_build_block_map_static(plan.desc, q, q, plan.q_var, plan.kv_var, p.topk, False, plan.block_map,
                                       plan.q_idx, plan.q_cnt, plan.idx_cap, None, None)
    assert e.value.code == 10

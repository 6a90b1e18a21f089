"""vsa_check_inputs: the opt-in validation of device-resident arguments.

Valid inputs (the library's own block map and indices, padded and varlen)
pass. Each kind of bad input, made on the host, gives VSA_ERR_SHAPE and its
own code: tile fills outside [0, tile] (a fill counts valid slots,
FastVideo block_sparse_attn_cute_fwd.py, _vbs_mask_mod), decreasing
sequence offsets, counts past idx_cap, entries outside the tile range or
out of order, and a KV-owned index that is not the transpose of the
Q-owned one (same page, _build_sparse_tensors). Only the checker sees the
bad values: it reads nothing outside the declared sizes, and no attention
kernel is run on them."""
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, make_tensors, tnd_problem
from tests.helpers import plan_for, to_device

pytestmark = pytest.mark.gpu

SHAPE = 2


def _built(p):
    t = to_device(make_tensors(p))
    plan = plan_for(p)
    plan.build_block_map(t["q"], t["k"], p.topk, need_bwd_index=True)
    torch.cuda.synchronize()
    return plan


def _padded():
    return Problem("chk", "bshd", 1, 4, 2, 128, 256, 256, 5, 7, q_var=[256, 61, 199, 256, 256],
                   kv_var=[256, 173, 0, 79, 256, 256, 12], topk=3, seed=61)


def test_valid_inputs_pass():
    plan = _built(_padded())
    assert plan.check_inputs() == (0, 0)
    assert plan.check_inputs(with_index=False) == (0, 0)      # KV-owned index alone: no transpose check
    assert plan.check_inputs(with_bwd_index=False) == (0, 0)
    p = tnd_problem("chk-tnd", [300, 7, 0, 129], [50, 520, 11, 256], 4, 2, dtype="bf16", topk=2, seed=62)
    assert _built(p).check_inputs() == (0, 0)


@pytest.mark.parametrize("which,value,code", [("kv_var", 300, 0xC002), ("kv_var", -1, 0xC002),
                                              ("q_var", 257, 0xC001)])
def test_tile_fill_out_of_range(which, value, code):
    plan = _built(_padded())
    getattr(plan, which)[2] = value
    assert plan.check_inputs(with_index=False, with_bwd_index=False) == (SHAPE, code)
    assert plan.check_inputs(with_index=False, with_bwd_index=False) == (SHAPE, code)  # the word was cleared


def test_sequence_offsets_not_ascending():
    p = tnd_problem("chk-cu", [300, 7, 129], [50, 520, 256], 2, 2, dtype="bf16", topk=2, seed=63)
    plan = _built(p)
    plan.cu_q[2] = plan.cu_q[1] - 1
    assert plan.check_inputs(with_index=False, with_bwd_index=False) == (SHAPE, 0xC003)
    plan.cu_q[2] = plan.cu_q[1]
    plan.cu_kv[3] = p.Skv + 1                                  # past the total tokens
    assert plan.check_inputs(with_index=False, with_bwd_index=False) == (SHAPE, 0xC004)


def test_q_index_counts_and_entries():
    plan = _built(_padded())
    plan.q_cnt[0, 1, 2] = plan.idx_cap + 1
    assert plan.check_inputs(with_bwd_index=False) == (SHAPE, 0xC005)
    plan.q_cnt[0, 1, 2] = -1
    assert plan.check_inputs(with_bwd_index=False) == (SHAPE, 0xC005)
    plan = _built(_padded())
    plan.q_idx[0, 3, 1, 0] = 7                                 # nKV = 7: out of range
    assert plan.check_inputs(with_bwd_index=False) == (SHAPE, 0xC006)
    plan = _built(_padded())
    row = plan.q_idx[0, 0, 0].clone()
    plan.q_idx[0, 0, 0, 0], plan.q_idx[0, 0, 0, 1] = row[1], row[0]   # not ascending
    assert plan.check_inputs(with_bwd_index=False) == (SHAPE, 0xC006)
    plan = _built(_padded())
    plan.q_idx[0, 2, 4] = torch.tensor([0, 2, 3], dtype=torch.int32)  # kv_var[2] = 0: no valid token
    plan.q_cnt[0, 2, 4] = 3
    assert plan.check_inputs(with_bwd_index=False) == (SHAPE, 0xC006)


def test_kv_index_offsets_entries_and_transpose():
    plan = _built(_padded())
    ptr = plan.kv_ptr[0, 1]
    j = int(torch.nonzero(ptr[1:] > ptr[:-1])[0])               # a KV tile with a non-empty list
    ptr[j + 1] = ptr[j] - 1                                    # decreasing offsets
    assert plan.check_inputs() == (SHAPE, 0xC007)
    plan = _built(_padded())
    plan.kv_ptr[0, 0, 0] = 1                                   # must start at 0
    assert plan.check_inputs() == (SHAPE, 0xC007)
    plan = _built(_padded())
    plan.kv_qidx[0, 2, 0] = 5                                  # nQ = 5: out of range
    assert plan.check_inputs() == (SHAPE, 0xC008)
    # a valid-looking KV-owned list that disagrees with the Q-owned index
    plan = _built(_padded())
    ptr = plan.kv_ptr[0, 3].tolist()
    lst = plan.kv_qidx[0, 3].tolist()
    for jj in range(7):
        a, b = ptr[jj], ptr[jj + 1]
        if 0 < b - a < 5:
            missing = [i for i in range(5) if i not in lst[a:b]]
            lst[a] = missing[0]
            lst[a:b] = sorted(lst[a:b])
            break
    plan.kv_qidx[0, 3] = torch.as_tensor(lst, dtype=torch.int32, device="cuda")
    assert plan.check_inputs(with_index=False) == (0, 0)       # in range and ascending on its own
    assert plan.check_inputs() == (SHAPE, 0xC009)

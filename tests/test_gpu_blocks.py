"""Query blocks smaller than a tile ([32, 128] and [64, 128] block shapes
with an explicit block mask, as on the Ascend block-sparse-attention test
page): GPU against the oracle run with tile_q = block_q, so that every
query block carries its own key list there (no union, no bit masks)."""
import math

import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, make_tensors
from oracle import oracle as orc
from tests.helpers import GRAD_TOL, OUT_TOL, check_tol, plan_for, to_device

pytestmark = pytest.mark.gpu

LSE_ATOL = 2e-3


def cases():
    return [
        (Problem("blk32-bhsd-gqa", "bhsd", 2, 4, 2, 128, 128, 128, 3, 4, q_var=[128] * 3, kv_var=[128] * 4,
                 seed=51), 32),
        (Problem("blk64-bshd-ragged", "bshd", 1, 2, 2, 128, 128, 128, 2, 5, q_var=[128] * 2,
                 kv_var=[128, 77, 128, 5, 128], seed=52), 64),
        (Problem("blk64-tnd-tail", "tnd", 3, 4, 2, 128, 128, 128, 1, 2, dtype="fp16", q_lens=[65, 127, 3],
                 kv_lens=[129, 11, 64], seed=53), 64),
        (Problem("blk32-tnd", "tnd", 3, 4, 2, 128, 128, 128, 3, 5, dtype="fp16", q_lens=[300, 17, 129],
                 kv_lens=[540, 23, 200], seed=54), 32),
        (Problem("blk32-bhsd-one-each", "bhsd", 1, 2, 2, 128, 128, 128, 2, 2, q_var=[128] * 2, kv_var=[128] * 2,
                 seed=55), 32),
    ]


def block_mask(p, bq):
    nqb = (p.nQ * p.tile_q) // bq if p.layout != "tnd" else math.ceil(max(p.q_lens) / bq)
    rng = np.random.default_rng(p.seed + 100)
    if p.name.endswith("one-each"):  # each query block attends exactly one KV block
        m = np.zeros((p.B, p.Hq, nqb, p.nKV), dtype=np.uint8)
        for b in range(p.B):
            for h in range(p.Hq):
                for i in range(nqb):
                    m[b, h, i, (i + b + h) % p.nKV] = 1
        return m
    m = (rng.random((p.B, p.Hq, nqb, p.nKV)) < 0.5).astype(np.uint8)
    m[:, :, 1, :] = 0  # a block that selects nothing: O = 0, LSE = -inf, no gradient
    return m


def block_problem(p, bq, nqb):
    """The same problem with query tiles of block_q rows (for the oracle)."""
    return Problem(p.name + "-oracle", p.layout, p.B, p.Hq, p.Hkv, p.D, bq, p.tile_kv, nqb, p.nKV, dtype=p.dtype,
                   q_var=None if p.layout == "tnd" else [bq] * nqb, kv_var=p.kv_var, q_lens=p.q_lens,
                   kv_lens=p.kv_lens, seed=p.seed)


@pytest.mark.parametrize("case", cases(), ids=lambda c: c[0].name)
def test_query_blocks_parity(case):
    p, bq = case
    t = make_tensors(p)
    m = block_mask(p, bq)
    pb = block_problem(p, bq, m.shape[2])
    ref = orc.run_full(pb, t, mask=m)

    plan = plan_for(p)
    g = to_device(t)
    plan.mask_to_index_blocks(bq, torch.as_tensor(m).cuda())
    out, lse = plan.forward_blocks(g["q"], g["k"], g["v"])
    dq, dk, dv = plan.backward_blocks(g["dO"], g["q"], g["k"], g["v"], out, lse)
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    # the tile map is the union of each tile's blocks (blocks past a sequence's end ignored)
    ns = p.tile_q // bq
    union = np.zeros((p.B, p.Hq, p.nQ, p.nKV), dtype=np.uint8)
    for i in range(p.nQ):
        for s in range(ns):
            blk = i * ns + s
            if blk >= m.shape[2]:
                continue
            for b in range(p.B):
                if p.layout == "tnd" and i * p.tile_q + s * bq >= p.q_lens[b]:
                    continue
                union[b, :, i] |= m[b, :, blk]
    assert np.array_equal(plan.block_map.cpu().numpy(), union)

    check_tol(f"{p.name} out", ref["out"], out.double().cpu().numpy(), OUT_TOL)
    lg, lr = lse.double().cpu().numpy(), ref["lse"]
    fin = np.isfinite(lr)
    assert np.all(lg[~fin & ~np.isnan(lr)] == -np.inf)
    assert np.max(np.abs(lg[fin] - lr[fin]), initial=0.0) < LSE_ATOL
    for n, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tol(f"{p.name} {n}", ref[n], x.double().cpu().numpy(), GRAD_TOL)

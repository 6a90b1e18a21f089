"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (one block-map + forward + backward step through the C
ABI). The whole block map and both indices are compared bit for bit with
the oracle; outputs are compared on samples the oracle computes one by one:
query rows (O, LSE, dQ; random tiles plus the last two query tiles) and
whole KV tiles (dK, dV: the most-selected, a median and the least-selected
tile, and the most-selected partial one when tiles are ragged) of the first
and the last head, each head checked on a one-head slice of the problem
(heads are independent)."""
import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, config, make_tensors
from oracle import oracle as orc
from tests.helpers import GRAD_TOL, OUT_TOL, check_tol, plan_for

pytestmark = pytest.mark.gpu

LSE_ATOL = 2e-3


def _one_head(p, t, h):
    """The problem restricted to query head h (and its KV head), as host
    tensors of the same layout."""
    g = p.Hq // p.Hkv
    ph = Problem(p.name + f"-h{h}", p.layout, p.B, 1, 1, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV,
                 dtype=p.dtype, q_var=p.q_var, kv_var=p.kv_var, topk=p.topk, gate=p.gate, seed=p.seed)
    hd = 2 if p.layout == "bshd" else 1
    th = {}
    for n, x in t.items():
        hh = h if n in ("q", "dO", "gate") else h // g
        th[n] = x.narrow(hd, hh, 1).contiguous().cpu()
    return ph, th


def _sample_rows(p, rng, n):
    """n rows of distinct random query tiles, plus the first and last rows
    of the last two query tiles (the end of the grid)."""
    tiles = rng.choice(p.nQ, size=min(n, p.nQ), replace=False)
    rows = [int(i) * p.tile_q + int(rng.integers(p.tile_q)) for i in tiles]
    for i in (p.nQ - 2, p.nQ - 1):
        rows += [i * p.tile_q, i * p.tile_q + p.tile_q - 1]
    return np.asarray([(0, 0, s) for s in sorted(set(rows))], dtype=np.int32)


def _pick(x, p, h, s):
    """Row s of head h of a full-problem GPU tensor, as float64 numpy."""
    return (x[0, s, h] if p.layout == "bshd" else x[0, h, s]).double().cpu().numpy()


def _run_full_size(p, heads, backward=True, n_rows=48):
    dev = torch.device("cuda")
    t = make_tensors(p, device=dev)
    plan = plan_for(p)
    plan.build_block_map(t["q"], t["k"], p.topk, need_bwd_index=backward)
    out, lse, osp = plan.forward(t["q"], t["k"], t["v"], gate=t.get("gate"))
    if backward:
        dq, dk, dv = plan.backward(t["dO"], t["q"], t["k"], t["v"], osp, lse, gate=t.get("gate"))
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    # whole block map and indices, bit for bit
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    assert np.array_equal(plan.block_map.cpu().numpy(), m)
    assert np.array_equal(plan.q_cnt.cpu().numpy(), qc)
    assert np.array_equal(plan.q_idx.cpu().numpy(), qi)
    if backward:
        kp, kq = orc.transpose(p, qi, qc, p.cap)
        assert np.array_equal(plan.kv_ptr.cpu().numpy(), kp)
        assert np.array_equal(plan.kv_qidx.cpu().numpy(), kq)

    rng = np.random.default_rng(7)
    for h in heads:
        ph, th = _one_head(p, t, h)
        _, qih, qch, _ = orc.build_block_map(ph, th["q"], th["k"], ph.topk, ph.cap)
        assert np.array_equal(qih[0, 0], qi[0, h]) and np.array_equal(qch[0, 0], qc[0, h])
        rows = _sample_rows(ph, rng, n_rows)
        ro, _, rl = orc.forward_rows(ph, th["q"], th["k"], th["v"], qih, qch, ph.cap, gate=th.get("gate"),
                                     rows=rows)
        got_o = np.stack([_pick(out, p, h, int(s)) for s in rows[:, 2]])
        check_tol(f"{p.name} h{h} out", ro, got_o, OUT_TOL)
        got_l = np.asarray([float(lse[0, h, int(s)]) for s in rows[:, 2]])
        assert np.max(np.abs(got_l - rl)) < LSE_ATOL
        if not backward:
            continue
        cg = orc.compress_grads(ph, th["dO"], th["gate"], th["q"], th["k"], th["v"]) if "gate" in th else None
        rdq = orc.backward_dq_rows(ph, th["dO"], th["q"], th["k"], th["v"], qih, qch, ph.cap, gate=th.get("gate"),
                                   rows=rows, cgrads=cg)
        got_dq = np.stack([_pick(dq, p, h, int(s)) for s in rows[:, 2]])
        check_tol(f"{p.name} h{h} dq", rdq, got_dq, GRAD_TOL)
        if h % (p.Hq // p.Hkv):
            continue
        # KV tiles of this head's KV-owned index: the most-selected one (the
        # longest KV-owned work list, many barrier-phase wraps), a median one
        # and the least-selected non-empty one; with ragged tiles also the
        # most-selected partial tile
        kp1, _ = orc.transpose(ph, qih, qch, ph.cap)
        cnt = np.diff(kp1[0, 0])
        cand = sorted((j for j in range(ph.nKV) if cnt[j] > 0 and ph.kv_var[j] > 0), key=lambda jj: (cnt[jj], jj))
        picks = [cand[-1], cand[len(cand) // 2], cand[0]]
        ragged = [j for j in cand if ph.kv_var[j] < ph.tile_kv]
        if ragged:
            picks.append(ragged[-1])
        picks = list(dict.fromkeys(picks))
        rdk, rdv = orc.backward_dkdv_tiles(ph, th["dO"], th["q"], th["k"], th["v"], qih, qch, ph.cap,
                                           gate=th.get("gate"), tiles=np.asarray([(0, 0, j) for j in picks]),
                                           cgrads=cg)
        hk = h // (p.Hq // p.Hkv)
        for n, j in enumerate(picks):
            keys = range(j * p.tile_kv, (j + 1) * p.tile_kv)
            got_dk = np.stack([_pick(dk, p, hk, s) for s in keys])
            got_dv = np.stack([_pick(dv, p, hk, s) for s in keys])
            tag = f"{p.name} h{h} tile {j} ({cnt[j]} query tiles, {ph.kv_var[j]} keys)"
            check_tol(f"{tag} dk", rdk[n], got_dk, GRAD_TOL)
            check_tol(f"{tag} dv", rdv[n], got_dv, GRAD_TOL)


def test_video_dit_76800_full_size():
    _run_full_size(config(3), heads=[0, 39])


def test_gated_ragged_full_size():
    _run_full_size(config(4), heads=[0, 23])


def test_long_video_inference_full_size():
    p = config(5)
    _run_full_size(p, heads=[5, 23], backward=False)


def test_long_video_literal_grid_full_size():
    # 32 x 60 x 128 tiled 4 x 8 x 8: 1,024 tiles, the last tile row of every
    # frame block half full (128 tokens)
    p = config(6)
    assert p.nKV == 1024 and sorted(set(p.kv_var.tolist())) == [128, 256] and int((p.kv_var == 128).sum()) == 128
    _run_full_size(p, heads=[0, 23], backward=False)


def test_all_kv_tiles_empty():
    p = Problem("all-empty", "bshd", 1, 2, 1, 128, 256, 256, 2, 3, q_var=[256, 100], kv_var=[0, 0, 0], topk=2,
                gate="randn01", seed=51)
    t = {n: x.cuda() for n, x in make_tensors(p).items()}
    plan = plan_for(p)
    plan.build_block_map(t["q"], t["k"], p.topk)
    out, lse, osp = plan.forward(t["q"], t["k"], t["v"], gate=t["gate"])
    dq, dk, dv = plan.backward(t["dO"], t["q"], t["k"], t["v"], osp, lse, gate=t["gate"])
    torch.cuda.synchronize()
    assert torch.all(plan.q_cnt == 0)
    assert torch.all(out == 0) and torch.all(osp == 0)
    assert torch.all(torch.isneginf(lse))
    for x in (dq, dk, dv):
        assert torch.all(x == 0)


def test_varlen_with_empty_sequences():
    from bwd_tile_mean_gb300.inputs import tnd_problem
    from tests.helpers import to_device
    p = tnd_problem("tnd-empty", [0, 130, 7], [50, 0, 300], 4, 2, dtype="bf16", topk=2, seed=52)
    t = make_tensors(p)
    plan = plan_for(p)
    g = to_device(t)
    plan.build_block_map(g["q"], g["k"], p.topk)
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"])
    dq, dk, dv = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse)
    torch.cuda.synchronize()
    ref = orc.run_full(p, t)
    assert np.array_equal(plan.q_idx.cpu().numpy(), ref["q_idx"])
    check_tol("out", ref["out"], out.double().cpu().numpy(), OUT_TOL)
    lr, lg = ref["lse"], lse.double().cpu().numpy()
    fin = np.isfinite(lr)
    assert np.all(np.isneginf(lg[~fin])) and np.max(np.abs(lg[fin] - lr[fin])) < LSE_ATOL
    for n, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tol(n, ref[n], x.double().cpu().numpy(), GRAD_TOL)

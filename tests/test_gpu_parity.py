"""GPU parity: the CUDA path through the C ABI against the CPU oracle on
the same seeded inputs. Block maps and indices bit-exact; O within
(avg_abs 1e-3, max_rel 0.2); dQ/dK/dV within (1e-3, 0.25); LSE within 2e-3
absolute (fp32 softmax statistics over bf16/fp16 inputs)."""
import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, config, make_mask, make_tensors, tnd_problem
from oracle import oracle as orc
from tests.helpers import (GRAD_TOL, OUT_TOL, check_tol, load_golden, npu_problem, page_problem, plan_for,
                           to_device)

pytestmark = pytest.mark.gpu

LSE_ATOL = 2e-3


def page_cases():
    g = load_golden("vsa_page_cases.json")
    return [page_problem(c, lay) for c in g["cases"] for lay in ("bhsd", "bshd")]


def topk_varlen():
    return tnd_problem("tnd-topk", [300, 17, 129, 256], [540, 23, 200, 383], 12, 3, dtype="fp16", topk=2,
                       seed=6)


def extra_cases():
    return [
        config(1),
        Problem("gqa-ragged", "bshd", 2, 8, 2, 128, 256, 256, 5, 7, q_var=[256, 0, 61, 256, 199],
                kv_var=[256, 0, 1, 129, 128, 255, 256], topk=3, seed=21),
        Problem("tile128", "bhsd", 1, 4, 4, 128, 128, 128, 6, 9, q_var=[128] * 6,
                kv_var=[128, 5, 128, 0, 77, 128, 128, 128, 1], topk=4, seed=22, dtype="fp16"),
        Problem("topk-ge-nkv", "bshd", 1, 2, 1, 128, 256, 256, 2, 3, q_var=[256, 256], kv_var=[256, 40, 0],
                topk=5, seed=23),
        topk_varlen(),
        # chunks with exactly 64 and 65 valid keys on both sides of the
        # 64-key form of dQ (first and second chunk of a 256-token tile),
        # every non-empty tile selected
        Problem("chunk-64-edges", "bshd", 1, 4, 2, 128, 256, 256, 3, 8, q_var=[256, 256, 256],
                kv_var=[64, 65, 192, 193, 256, 63, 129, 0], topk=7, seed=24),
        tnd_problem("tnd-chunk-64-edges", [300, 256, 129], [320, 449, 192], 4, 4, dtype="bf16", tile=256,
                    topk=2, seed=25),
    ]


MAP_CASES = page_cases() + extra_cases()


def run_map(p, t, need_bwd=True):
    g = to_device(t)
    plan = plan_for(p)
    plan.build_block_map(g["q"], g["k"], p.topk, need_bwd_index=need_bwd)
    return plan, g


@pytest.mark.parametrize("p", MAP_CASES, ids=lambda p: p.name)
def test_block_map_bit_exact(p):
    t = make_tensors(p)
    plan, _ = run_map(p, t)
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    kp, kq = orc.transpose(p, qi, qc, p.cap)
    torch.cuda.synchronize()
    assert np.array_equal(plan.block_map.cpu().numpy(), m)
    assert np.array_equal(plan.q_cnt.cpu().numpy(), qc)
    assert np.array_equal(plan.q_idx.cpu().numpy(), qi)
    assert np.array_equal(plan.kv_ptr.cpu().numpy(), kp)
    assert np.array_equal(plan.kv_qidx.cpu().numpy(), kq)


def tie_cases():
    """Selections decided by ties: duplicated K tiles (equal scores for every
    query), an all-zero K tile (score exactly 0), an all-zero Q tile (every
    score 0), empty KV tiles (-inf), more KV tiles than a warp's lanes, and
    topk above the number of valid tiles."""
    a = Problem("ties-40kv", "bshd", 1, 4, 2, 128, 256, 256, 3, 40, q_var=[256, 256, 256],
                kv_var=[256] * 3 + [0] + [256] * 26 + [0] + [256] * 9, topk=10, seed=31)
    b = Problem("ties-topk-gt-valid", "bhsd", 1, 2, 2, 128, 256, 256, 2, 6, q_var=[256, 256],
                kv_var=[256, 0, 120, 0, 256, 0], topk=5, seed=32)
    return [a, b]


def make_ties(p, t):
    k, q = t["k"].clone(), t["q"].clone()
    T = p.tile_kv

    def tile(x, j):  # token range of tile j in the layout
        return (slice(None), slice(None), slice(j * T, (j + 1) * T)) if p.layout == "bhsd" else \
            (slice(None), slice(j * T, (j + 1) * T))
    for j in (7, 13, 21, 33):
        if j < p.nKV:
            k[tile(k, j)] = k[tile(k, 0)]
    k[tile(k, 2)] = 0
    if p.nKV > 5:
        k[tile(k, 5)] = k[tile(k, 4)]
    q[tile(q, 1)] = 0
    t = dict(t)
    t["k"], t["q"] = k, q
    return t


def test_block_map_many_kv_tiles_bit_exact():
    """2,600 KV tiles (past the point where the selection kernel keeps one
    query tile per warp to fit shared memory; 21 staging chunks), topk 100."""
    nkv = 2600
    kv_var = [128] * nkv
    kv_var[5], kv_var[1000], kv_var[2599] = 0, 17, 1
    p = Problem("many-kv", "bshd", 1, 2, 1, 128, 128, 128, 4, nkv, q_var=[128] * 4, kv_var=kv_var, topk=100, seed=33)
    t = make_tensors(p)
    plan, _ = run_map(p, t)
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    kp, kq = orc.transpose(p, qi, qc, p.cap)
    torch.cuda.synchronize()
    assert np.array_equal(plan.block_map.cpu().numpy(), m)
    assert np.array_equal(plan.q_cnt.cpu().numpy(), qc)
    assert np.array_equal(plan.q_idx.cpu().numpy(), qi)
    assert np.array_equal(plan.kv_ptr.cpu().numpy(), kp)
    assert np.array_equal(plan.kv_qidx.cpu().numpy(), kq)


@pytest.mark.parametrize("p", tie_cases(), ids=lambda p: p.name)
def test_block_map_ties_bit_exact(p):
    t = make_ties(p, make_tensors(p))
    plan, _ = run_map(p, t)
    m, qi, qc, sc = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    kp, kq = orc.transpose(p, qi, qc, p.cap)
    torch.cuda.synchronize()
    # the constructed ties are really there: equal scores across duplicated
    # tiles, or (topk above the valid tiles) the lowest empty tiles chosen
    if p.nKV > 7:
        assert np.any(sc[..., 0] == sc[..., 7])
    else:
        assert np.all(m[..., 1] == 1) and np.all(m[..., 3] == 1) and not np.any(m[..., 5])
    assert np.array_equal(plan.block_map.cpu().numpy(), m)
    assert np.array_equal(plan.q_cnt.cpu().numpy(), qc)
    assert np.array_equal(plan.q_idx.cpu().numpy(), qi)
    assert np.array_equal(plan.kv_ptr.cpu().numpy(), kp)
    assert np.array_equal(plan.kv_qidx.cpu().numpy(), kq)


def test_mask_index_bit_exact_varlen():
    p = config(2)
    t = make_tensors(p)
    mask = make_mask(p)
    plan = plan_for(p)
    plan.mask_to_index(torch.as_tensor(mask).cuda(), need_bwd_index=True)
    qi, qc = orc.mask_index(p, mask, p.cap)
    kp, kq = orc.transpose(p, qi, qc, p.cap)
    torch.cuda.synchronize()
    assert np.array_equal(plan.q_cnt.cpu().numpy(), qc)
    assert np.array_equal(plan.q_idx.cpu().numpy(), qi)
    assert np.array_equal(plan.kv_ptr.cpu().numpy(), kp)
    assert np.array_equal(plan.kv_qidx.cpu().numpy(), kq)


def _fwd_check(p, t, plan, g, qi, qc):
    gate = g.get("gate")
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=gate)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    rows = p.rows()
    ro, rosp, rl = orc.forward_rows(p, t["q"], t["k"], t["v"], qi, qc, p.cap, gate=t.get("gate"), rows=rows)
    out_ref = orc._scatter_rows(p, rows, ro)
    osp_ref = orc._scatter_rows(p, rows, rosp)
    lse_ref = orc._scatter_rows(p, rows, rl, lse_mode=True)
    check_tol(f"{p.name} out", out_ref, out.double().cpu().numpy(), OUT_TOL)
    check_tol(f"{p.name} o_sparse", osp_ref, osp.double().cpu().numpy(), OUT_TOL)
    lg = lse.double().cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.all(lg[~fin & ~np.isnan(lse_ref)] == -np.inf)
    assert np.max(np.abs(lg[fin] - lse_ref[fin]), initial=0.0) < LSE_ATOL
    return out, lse, osp


FWD_CASES = page_cases() + extra_cases()


@pytest.mark.parametrize("p", FWD_CASES, ids=lambda p: p.name)
def test_forward_parity(p):
    t = make_tensors(p)
    plan, g = run_map(p, t)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    _fwd_check(p, t, plan, g, qi, qc)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_scores_far_above_the_first_chunk(dtype):
    # Every row's scores on the last KV tile lie far above its max over the
    # first chunk (q has a common component, that tile's keys are 6 plus half
    # their drawn values), by more than a 16-bit P relative to that max can
    # hold: the forward must move its reference (the tiles are recomputed by
    # the kernel that does) and the outputs and gradients still match the
    # oracle.
    p = Problem(f"far-scores-{dtype}", "bshd", 1, 2, 2, 128, 256, 256, 2, 4, q_var=[256, 256],
                kv_var=[256, 256, 200, 256], topk=4, seed=81, dtype=dtype)
    t = make_tensors(p)
    T = t["q"].dtype
    t["q"] = (t["q"].float() * 0.5 + 1.0).to(T)
    k = t["k"].float()
    k[:, 3 * 256:] = 6.0 + 0.5 * k[:, 3 * 256:]
    t["k"] = k.to(T)
    plan, g = run_map(p, t)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    assert np.all(qc == 4)  # every query tile attends to every KV tile, the far one last
    _fwd_check(p, t, plan, g, qi, qc)
    ref = orc.run_full(p, t)
    _bwd_check(p, t, plan, g, ref)


def test_far_scores_on_some_tiles_of_several_redo_groups():
    # 20 query tiles per head: the forward's recompute launch gives each CTA
    # 16 consecutive tiles of a head, so this spans a full group and a
    # partial one. Every third query tile has the common component that puts
    # its scores on the last KV tile far above its first chunk's max (those
    # tiles are recomputed), the rest do not; the recomputed tiles of a
    # group are computed one after the other by one CTA. Outputs and
    # gradients match the oracle.
    p = Problem("far-scores-groups", "bshd", 1, 2, 2, 128, 256, 256, 20, 4, q_var=[256] * 20,
                kv_var=[256, 256, 200, 256], topk=4, seed=82)
    t = make_tensors(p)
    T = t["q"].dtype
    q = t["q"].float()
    for i in range(0, p.nQ, 3):
        q[:, i * 256:(i + 1) * 256] = q[:, i * 256:(i + 1) * 256] * 0.5 + 1.0
    t["q"] = q.to(T)
    k = t["k"].float()
    k[:, 3 * 256:] = 6.0 + 0.5 * k[:, 3 * 256:]
    t["k"] = k.to(T)
    plan, g = run_map(p, t)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    assert np.all(qc == 4)
    _fwd_check(p, t, plan, g, qi, qc)
    ref = orc.run_full(p, t)
    _bwd_check(p, t, plan, g, ref)


@pytest.mark.parametrize("p", [config(2)] + [npu_problem(c) for c in load_golden("npu_tnd_cases.json")["cases"]],
                         ids=lambda p: p.name)
def test_forward_parity_varlen_mask(p):
    t = make_tensors(p)
    mask = make_mask(p)
    plan = plan_for(p)
    g = to_device(t)
    plan.mask_to_index(torch.as_tensor(mask).cuda(), need_bwd_index=True)
    qi, qc = orc.mask_index(p, mask, p.cap)
    _fwd_check(p, t, plan, g, qi, qc)


def test_forward_separate_o_sparse_without_gate():
    """O as the only output goes out through shared memory and box stores; a
    separate o_sparse buffer without a gate takes the per-thread stores for
    both. The two must agree bit for bit, with each other and across runs,
    and match the oracle."""
    p = extra_cases()[1]  # BSHD, 256-token tiles, GQA, ragged and empty tiles
    t = make_tensors(p)
    plan, g = run_map(p, t)
    out1, lse1, _ = plan.forward(g["q"], g["k"], g["v"])
    out2 = torch.empty_like(g["q"])
    osp2 = torch.empty_like(g["q"])
    plan.forward(g["q"], g["k"], g["v"], out=out2, o_sparse=osp2)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(out1, out2) and torch.equal(out1, osp2)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    rows = p.rows()
    ro, _, _ = orc.forward_rows(p, t["q"], t["k"], t["v"], qi, qc, p.cap, rows=rows)
    check_tol(f"{p.name} out", orc._scatter_rows(p, rows, ro), out1.double().cpu().numpy(), OUT_TOL)


def test_gated_tiles_without_chunks():
    """Gated padded layout from an explicit block mask in which some query
    tiles select nothing, or only a tile without valid keys: their out is
    gate (*) c alone, with the gate read directly (no chunk ran), next to
    tiles whose gate rows are copied in once their last S MMA is done. Out,
    o_sparse and the gradients match the oracle."""
    p = Problem("gated-mask-no-chunks", "bshd", 1, 4, 2, 128, 256, 256, 4, 5, q_var=[256, 256, 200, 256],
                kv_var=[256, 173, 0, 79, 256], gate="randn01", seed=61)
    t = make_tensors(p)
    m = (np.random.default_rng(61).random((p.B, p.Hq, p.nQ, p.nKV)) < 0.6).astype(np.uint8)
    m[0, 0, 1, :] = 0      # nothing selected
    m[0, 1, 0, :] = 0
    m[0, 1, 0, 2] = 1      # only the tile without valid keys
    m[0, 2, 3, :] = 1      # everything
    plan = plan_for(p)
    g = to_device(t)
    plan.mask_to_index(torch.as_tensor(m).cuda(), need_bwd_index=True)
    ref = orc.run_full(p, t, mask=m)
    assert ref["q_cnt"][0, 0, 1] == 0 and ref["q_cnt"][0, 1, 0] == 0
    dq, dk, dv = _bwd_check(p, t, plan, g, ref)
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=g["gate"])
    torch.cuda.synchronize()
    check_tol(f"{p.name} o_sparse", ref["o_sparse"], osp.double().cpu().numpy(), OUT_TOL)
    assert torch.all(osp[0, 256:512, 0] == 0) and torch.all(osp[0, 0:256, 1] == 0)


def test_forward_bhsd_equals_bshd_and_inference_equals_training():
    p = config(1)
    t = make_tensors(p)
    plan, g = run_map(p, t, need_bwd=True)
    out1, lse1, _ = plan.forward(g["q"], g["k"], g["v"])
    plan_inf, _ = run_map(p, t, need_bwd=False)
    out2, lse2, _ = plan_inf.forward(g["q"], g["k"], g["v"])
    pb = Problem("tiny-bshd", "bshd", 1, 2, 2, 128, 256, 256, 3, 4, q_var=p.q_var, kv_var=p.kv_var, topk=2)
    tb = {n: x.transpose(1, 2).contiguous() for n, x in t.items()}
    plan_b, gb = run_map(pb, tb)
    out3, lse3, _ = plan_b.forward(gb["q"], gb["k"], gb["v"])
    out4, lse4, _ = plan.forward(g["q"], g["k"], g["v"])
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)          # inference == training
    assert torch.equal(out1, out3.transpose(1, 2)) and torch.equal(lse1, lse3)  # BHSD == BSHD
    assert torch.equal(out1, out4) and torch.equal(lse1, lse4)          # run to run


def gated_cases():
    kv = [256, 160, 64, 40, 256, 256, 160, 64, 256]
    return [
        Problem("gated-ragged-small", "bshd", 1, 4, 2, 128, 256, 256, 5, 9, q_var=kv[:5], kv_var=kv, topk=3,
                gate="uniform_token_head", seed=31),
        Problem("gated-bhsd-gqa", "bhsd", 2, 6, 3, 128, 256, 256, 3, 4, q_var=[256, 61, 199],
                kv_var=[256, 173, 0, 79], topk=2, gate="randn01", seed=32),
        tnd_problem("gated-tnd-topk", [300, 17, 129], [540, 23, 200], 4, 2, dtype="fp16", topk=2,
                    gate="randn01", seed=33),
        # the CTA-pair forward's gated epilogue: fp16 through the staged box
        # stores, and varlen 256-token tiles through its per-thread stores
        Problem("gated-fp16-bshd", "bshd", 1, 4, 2, 128, 256, 256, 4, 6, q_var=[256, 200, 256, 97],
                kv_var=[256, 64, 160, 0, 256, 40], topk=3, gate="randn01", seed=34, dtype="fp16"),
        tnd_problem("gated-tnd-256", [300, 517, 129], [540, 260, 700], 4, 2, dtype="bf16", tile=256, topk=2,
                    gate="randn01", seed=35),
    ]


BWD_CASES = page_cases() + extra_cases() + gated_cases()


def _bwd_check(p, t, plan, g, ref):
    gate = g.get("gate")
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=gate)
    dq, dk, dv = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=gate)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    check_tol(f"{p.name} out", ref["out"], out.double().cpu().numpy(), OUT_TOL)
    for n, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_tol(f"{p.name} {n}", ref[n], x.double().cpu().numpy(), GRAD_TOL)
    return dq, dk, dv


@pytest.mark.parametrize("p", BWD_CASES, ids=lambda p: p.name)
def test_backward_parity(p):
    t = make_tensors(p)
    plan, g = run_map(p, t)
    ref = orc.run_full(p, t)
    assert np.array_equal(plan.q_idx.cpu().numpy(), ref["q_idx"])
    _bwd_check(p, t, plan, g, ref)


@pytest.mark.parametrize("p", [config(2)] + [npu_problem(c) for c in load_golden("npu_tnd_cases.json")["cases"]],
                         ids=lambda p: p.name)
def test_backward_parity_varlen_mask(p):
    t = make_tensors(p)
    mask = make_mask(p)
    plan = plan_for(p)
    g = to_device(t)
    plan.mask_to_index(torch.as_tensor(mask).cuda(), need_bwd_index=True)
    ref = orc.run_full(p, t, mask=mask)
    _bwd_check(p, t, plan, g, ref)


def test_backward_bitwise_deterministic():
    p = gated_cases()[0]
    t = make_tensors(p)
    plan, g = run_map(p, t)
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=g["gate"])
    r1 = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=g["gate"])
    r2 = plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=g["gate"])
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("p", gated_cases(), ids=lambda p: p.name)
def test_gate_grad_parity(p):
    """dgate = dO (*) c from vsa_gate_grad against the oracle (fp64), with
    the gradient tolerance; rows outside TND sequences stay untouched."""
    t = make_tensors(p)
    g = to_device(t)
    plan = plan_for(p)
    dgate = torch.full_like(g["dO"], 7.0)
    plan.gate_grad(g["dO"], g["q"], g["k"], g["v"], dgate=dgate)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref = orc.gate_grad(p, t["dO"], t["q"], t["k"], t["v"])
    got = dgate.double().cpu().numpy()
    if p.layout == "tnd":
        assert got.shape[0] == p.cu_q[-1]
    check_tol(f"{p.name} dgate", ref, got, GRAD_TOL)


@pytest.mark.parametrize("p", gated_cases(), ids=lambda p: p.name)
def test_gated_step_pools_once(p):
    """A gated step through the plan pools q and k once (block map) and v
    once (forward); the backward pools nothing. Outputs are bitwise those of
    the calls that recompute every tile mean (reuse = 0). After an in-place
    write to q the plan recomputes q's and k's means, again bitwise equal to
    reuse = 0 on the new q."""
    from bwd_tile_mean_gb300 import vsa
    t = make_tensors(p)
    plan, g = run_map(p, t)
    q, k, v, dO, gate = g["q"], g["k"], g["v"], g["dO"], g["gate"]

    def recompute(qq):
        out, lse, osp = torch.empty_like(qq), torch.empty(plan.lse_shape(), dtype=torch.float32, device="cuda"), \
            torch.empty_like(qq)
        vsa.vsa_fwd(plan.desc, qq, k, v, plan.q_idx, plan.q_cnt, plan.idx_cap, plan.q_var, plan.kv_var, gate, out,
                    lse, osp, plan.workspace)
        grads = [torch.empty_like(x) for x in (qq, k, v)]
        vsa.vsa_bwd(plan.desc, dO, qq, k, v, osp, lse, plan.q_idx, plan.q_cnt, plan.idx_cap, plan.kv_ptr,
                    plan.kv_qidx, plan.q_var, plan.kv_var, gate, *grads, plan.workspace)
        return [out, lse, osp] + grads

    ref = recompute(q)
    plan.build_block_map(q, k, p.topk)
    with vsa.profile() as prof:
        out, lse, osp = plan.forward(q, k, v, gate=gate)
        grads = plan.backward(dO, q, k, v, osp, lse, gate=gate)
    torch.cuda.synchronize()
    assert [n for n, _ in prof.records].count("pool") == 1  # v, in the forward
    for a, b in zip(ref, [out, lse, osp] + list(grads)):
        assert torch.equal(a, b)

    q.mul_(-0.5)  # new q: its means (and so c and the gated outputs) change
    ref2 = recompute(q)
    plan.build_block_map(q, k, p.topk)
    q.add_(0.25)  # written again after the block map pooled it
    ref3 = recompute(q)
    with vsa.profile() as prof:
        out, lse, osp = plan.forward(q, k, v, gate=gate)
        grads = plan.backward(dO, q, k, v, osp, lse, gate=gate)
    torch.cuda.synchronize()
    assert [n for n, _ in prof.records].count("pool") == 1  # q and k, in the forward (v's means are kept)
    assert not torch.equal(ref2[0], ref3[0])
    for a, b in zip(ref3, [out, lse, osp] + list(grads)):
        assert torch.equal(a, b)
    assert plan.device_status() == 0


@pytest.mark.parametrize("p", [extra_cases()[1], gated_cases()[0], topk_varlen()], ids=lambda p: p.name)
def test_backward_writes_every_key_row(p):
    """The dK/dV pass runs its units longest first (a permutation computed
    on the device from kv_ptr): every unit must run exactly once. dQ, dK and
    dV start as NaN and must come back finite everywhere, equal to a second
    run (keys no query selected, and padded slots, get 0)."""
    t = make_tensors(p)
    plan, g = run_map(p, t)
    gate = g.get("gate")
    out, lse, osp = plan.forward(g["q"], g["k"], g["v"], gate=gate)
    runs = []
    for _ in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (g["q"], g["k"], g["v"]))
        plan.backward(g["dO"], g["q"], g["k"], g["v"], osp, lse, gate=gate, dq=dq, dk=dk, dv=dv)
        runs.append((dq, dk, dv))
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for x in runs[0]:
        assert torch.isfinite(x).all()
    for a_, b_ in zip(*runs):
        assert torch.equal(a_, b_)

"""Pins of the CPU oracle against things other than itself: library
routines (torch SDPA / autograd in float64, numpy's sequential
accumulate), exact rational arithmetic, brute force, closed forms,
finite differences and invariants. CPU only."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bwd_tile_mean_gb300.inputs import Problem, make_mask, make_tensors, tnd_problem
from oracle import oracle as orc
from tests.helpers import (exact_fmaf, key_mask, load_golden, masked_attention_f64, npu_problem,
                           page_problem, to_bhsd)


def _np(x, dt=np.float64):
    return x.detach().to(torch.float64).numpy().astype(dt)


def small(layout="bhsd", kv_var=(256, 173, 0, 79, 256), q_var=(256, 61, 199), H=2, Hkv=2, topk=2,
          seed=3, D=128, tile=256, gate=None, dtype="bf16"):
    return Problem("small", layout, 1, H, Hkv, D, tile, tile, len(q_var), len(kv_var), dtype=dtype,
                   q_var=list(q_var), kv_var=list(kv_var), topk=topk, seed=seed, gate=gate)


# ------------------------------------------------------------ O1 pooling

@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_pool_bit_exact_vs_sequential_accumulate(layout):
    p = small(layout)
    t = make_tensors(p)
    q = _np(t["q"], np.float32)
    k = _np(t["k"], np.float32)
    pq = orc.pool_f32(p, q, True)
    pk = orc.pool_f32(p, k, False)
    qb, kb = to_bhsd(p, q, True).numpy().astype(np.float32), to_bhsd(p, k, False).numpy().astype(np.float32)
    for (x, pooled, var, T) in ((qb, pq, p.q_var, p.tile_q), (kb, pk, p.kv_var, p.tile_kv)):
        for t_, vv in enumerate(var):
            if vv == 0:
                assert np.all(pooled[:, :, t_] == 0)
                continue
            seg = x[:, :, t_ * T:t_ * T + vv, :]
            ref = np.add.accumulate(seg, axis=2, dtype=np.float32)[:, :, -1, :] / np.float32(vv)
            assert np.array_equal(pooled[:, :, t_], ref)


def test_pool_varlen_tiles_cut_at_sequence_end():
    p = tnd_problem("t", [5, 9], [7, 3], 2, 1, tile=4)
    t = make_tensors(p)
    k = _np(t["k"], np.float32)
    pk = orc.pool_f32(p, k, False)
    cu = p.cu_kv
    for b in range(2):
        for j in range(p.nKV):
            vv = p.tile_var(False, b, j)
            seg = k[cu[b] + 4 * j: cu[b] + 4 * j + vv]
            if vv == 0:
                assert np.all(pk[b, :, j] == 0)
            else:
                ref = np.add.accumulate(seg, axis=0, dtype=np.float32)[-1] / np.float32(vv)
                assert np.array_equal(pk[b, :, j], ref)


# ----------------------------------------------------- O2 scores, O3 top-k

def test_scores_bit_exact_vs_exact_rational_fma():
    p = small(kv_var=(256, 100, 0), q_var=(256, 17), H=1, Hkv=1)
    t = make_tensors(p)
    pq = orc.pool_f32(p, t["q"], True)
    pk = orc.pool_f32(p, t["k"], False)
    _, _, _, sc = orc.select(p, pq, pk, 2, 2)
    for i in range(p.nQ):
        for j in range(p.nKV):
            if p.kv_var[j] == 0:
                assert sc[0, 0, i, j] == -np.inf
                continue
            r = np.float32(0.0)
            for e in range(p.D):
                r = exact_fmaf(pq[0, 0, i, e], pk[0, 0, j, e], r)
            assert sc[0, 0, i, j] == r, (i, j)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_topk_equals_bruteforce_full_sort(seed):
    p = small(kv_var=(256, 173, 0, 79, 256, 12, 256), q_var=(256, 0, 199), topk=3, seed=seed)
    t = make_tensors(p)
    m, qi, qc, sc = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    for h in range(p.Hq):
        for i in range(p.nQ):
            r = sc[0, h, i]
            order = sorted(range(p.nKV), key=lambda j: (-float(r[j]), j))
            chosen = set(order[:min(p.topk, p.nKV)])
            assert set(np.nonzero(m[0, h, i])[0].tolist()) == chosen
            nonempty = sorted(j for j in chosen if p.kv_var[j] > 0)
            assert qc[0, h, i] == len(nonempty)
            assert qi[0, h, i, :len(nonempty)].tolist() == nonempty
            assert np.all(qi[0, h, i, len(nonempty):] == -1)


def test_topk_ties_go_to_lowest_index():
    p = small(kv_var=(0, 256, 256, 256, 256), q_var=(256, 256), topk=2)
    t = make_tensors(p)
    k = torch.zeros_like(t["k"])                  # every score is exactly 0
    m, qi, qc, _ = orc.build_block_map(p, t["q"], k, 2, 2)
    assert np.all(qi[..., :2] == np.array([1, 2]))  # tile 0 is empty (-inf)
    # duplicated tiles: tile 3 copies tile 1, so wherever both tie tile 1 wins
    k2 = t["k"].clone()
    k2[:, :, 3 * 256:4 * 256] = k2[:, :, 1 * 256:2 * 256]
    m2, _, _, sc = orc.build_block_map(p, t["q"], k2, 2, 2)
    assert np.array_equal(sc[..., 1], sc[..., 3])
    assert not np.any((m2[..., 3] == 1) & (m2[..., 1] == 0))


def test_topk_at_least_nkv_selects_everything():
    p = small(kv_var=(256, 0, 79, 256), q_var=(256, 256), topk=9)
    t = make_tensors(p)
    m, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], 9, 4)
    assert np.all(m == 1)
    assert np.all(qc == 3)
    assert np.all(qi[..., :3] == np.array([0, 2, 3]))


def test_selection_agrees_with_fp64_up_to_ties():
    """Every place where the fp32 selection differs from one made on exact
    (fp64) tile means lies within rounding of a tie."""
    p = small(kv_var=tuple([256] * 24), q_var=(256,) * 6, topk=5, seed=9)
    t = make_tensors(p)
    m, _, _, sc = orc.build_block_map(p, t["q"], t["k"], 5, 5)
    qb = to_bhsd(p, _np(t["q"]), True).numpy()
    kb = to_bhsd(p, _np(t["k"]), False).numpy()
    pq = qb.reshape(1, 2, 6, 256, 128).mean(axis=3)
    pk = kb.reshape(1, 2, 24, 256, 128).mean(axis=3)
    r64 = np.einsum("bhid,bhjd->bhij", pq, pk)
    for h in range(2):
        for i in range(6):
            sel = m[0, h, i] == 1
            lo, hi = r64[0, h, i][sel].min(), r64[0, h, i][~sel].max()
            assert lo >= hi - 1e-5 * np.abs(r64[0, h, i]).max()


# ------------------------------------------------------------ O4 transpose

def test_transpose_round_trips_to_q_lists():
    p = small(kv_var=(256, 173, 0, 79, 256, 12), q_var=(256, 61, 199, 5), topk=3, H=3, Hkv=1)
    t = make_tensors(p)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], 3, 3)
    kp, kq = orc.transpose(p, qi, qc, 3)
    for h in range(p.Hq):
        back = {i: [] for i in range(p.nQ)}
        for j in range(p.nKV):
            lst = kq[0, h, kp[0, h, j]:kp[0, h, j + 1]].tolist()
            assert lst == sorted(lst)
            for i in lst:
                back[i].append(j)
        for i in range(p.nQ):
            assert back[i] == qi[0, h, i, :qc[0, h, i]].tolist()


@pytest.mark.parametrize("bad", [("kv", 300), ("kv", -1), ("q", 257)])
def test_tile_fill_outside_the_tile_is_rejected(bad):
    # a fill counts valid slots (key n valid iff n mod tile < vbs); outside
    # [0, tile] it has no meaning on the pages, so the oracle refuses it
    side, v = bad
    kv, qv = [256, 173, 79], [256, 100]
    (kv if side == "kv" else qv)[1] = v
    p = small(kv_var=kv, q_var=qv)
    with pytest.raises(ValueError):
        orc.pool_f32(p, np.zeros(p.shape(side == "q"), np.float32), side == "q")


def test_mask_index_ignores_blocks_past_sequence_ends():
    p = tnd_problem("t", [130, 5, 300], [20, 400, 129], 2, 1, tile=128)
    mask = np.ones((p.B, p.Hq, p.nQ, p.nKV), dtype=np.uint8)
    qi, qc = orc.mask_index(p, mask, p.nKV)
    for b in range(p.B):
        nq = -(-p.q_lens[b] // 128)
        nk = -(-p.kv_lens[b] // 128)
        for i in range(p.nQ):
            want = list(range(nk)) if i < nq else []
            assert qi[b, 0, i, :qc[b, 0, i]].tolist() == want


# ------------------------------------------------------------- O5 forward

def _fwd(p, t, gate=None, mask=None):
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    if mask is None:
        _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
        cap = p.cap
    else:
        cap = p.nKV
        qi, qc = orc.mask_index(p, mask, cap)
    return qi, qc, cap, orc.forward_rows(p, q, k, v, qi, qc, cap, gate=gate)


@pytest.mark.parametrize("layout,Hkv", [("bhsd", 2), ("bshd", 2), ("bshd", 1)])
def test_dense_forward_equals_sdpa(layout, Hkv):
    p = small(layout, kv_var=(256, 256, 256), q_var=(256, 256), topk=3, Hkv=Hkv)
    t = make_tensors(p)
    _, _, _, (out, osp, lse) = _fwd(p, t)
    q, k, v = (to_bhsd(p, _np(t[n]), n == "q") for n in "qkv")
    g = p.Hq // p.Hkv
    k, v = k.repeat_interleave(g, 1), v.repeat_interleave(g, 1)
    mask = torch.ones(p.Sq, p.Skv, dtype=torch.bool)
    ro, rl = masked_attention_f64(q, k, v, mask, p.scale)
    rows = p.rows()
    np.testing.assert_allclose(out, ro[0, rows[:, 1], rows[:, 2]].numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, rl[0, rows[:, 1], rows[:, 2]].numpy(), rtol=1e-13, atol=1e-12)
    assert np.array_equal(out, osp)


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_sparse_forward_equals_masked_sdpa(layout):
    g = load_golden("vsa_page_cases.json")
    for case in g["cases"]:
        p = page_problem(case, layout)
        t = make_tensors(p)
        qi, qc, cap, (out, osp, lse) = _fwd(p, t)
        q, k, v = (to_bhsd(p, _np(t[n]), n == "q") for n in "qkv")
        rows = p.rows()
        for h in range(p.Hq):
            m = key_mask(p, qi, qc, 0, h)
            ro, rl = masked_attention_f64(q[:, h], k[:, h], v[:, h], m, p.scale)
            sel = rows[:, 1] == h
            np.testing.assert_allclose(osp[sel], ro[0, rows[sel, 2]].numpy(), rtol=0, atol=1e-11)
            np.testing.assert_allclose(lse[sel], rl[0, rows[sel, 2]].numpy(), rtol=1e-13, atol=1e-12)


def test_varlen_gqa_forward_equals_per_sequence_masked_sdpa():
    p = tnd_problem("t", [130, 5, 300, 64], [20, 400, 129, 250], 4, 2, tile=128, seed=5)
    t = make_tensors(p)
    mask = make_mask(p)
    qi, qc, cap, (out, osp, lse) = _fwd(p, t, mask=mask)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    rows = p.rows()
    r = 0
    for b in range(p.B):
        qs, ks = p.cu_q[b], p.cu_kv[b]
        lq, lk = p.q_lens[b], p.kv_lens[b]
        for h in range(p.Hq):
            hk = h // 2
            full = torch.as_tensor(mask[b, h]).bool().repeat_interleave(128, 0).repeat_interleave(128, 1)
            mm = full[:lq, :lk]
            qq = torch.as_tensor(q[qs:qs + lq, h])
            kk = torch.as_tensor(k[ks:ks + lk, hk])
            vv = torch.as_tensor(v[ks:ks + lk, hk])
            ro, rl = masked_attention_f64(qq, kk, vv, mm, p.scale)
            assert np.array_equal(rows[r:r + lq, :2], np.tile([b, h], (lq, 1)))
            np.testing.assert_allclose(osp[r:r + lq], ro.numpy(), rtol=0, atol=1e-11)
            fin = np.isfinite(rl.numpy())
            np.testing.assert_allclose(lse[r:r + lq][fin], rl.numpy()[fin], rtol=1e-13, atol=1e-12)
            assert np.all(lse[r:r + lq][~fin] == -np.inf)
            r += lq


def test_single_valid_key_gives_v_and_its_score():
    p = small(kv_var=(1,), q_var=(256,), topk=1)
    t = make_tensors(p)
    _, _, _, (out, _, lse) = _fwd(p, t)
    q, k, v = (to_bhsd(p, _np(t[n]), n == "q") for n in "qkv")
    rows = p.rows()
    np.testing.assert_array_equal(out, v[0, rows[:, 1], 0].numpy())
    s = (q[0, rows[:, 1], rows[:, 2]] * k[0, rows[:, 1], 0]).sum(-1) * p.scale
    np.testing.assert_allclose(lse, s.numpy(), rtol=0, atol=1e-12)


def test_padded_kv_slots_contribute_nothing():
    p = small(kv_var=(256, 173, 79, 256), q_var=(256, 256, 256), topk=2, gate="randn01")
    t = make_tensors(p)
    cap = p.cap
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, cap)
    g = torch.Generator().manual_seed(99)
    t2 = dict(t)
    for n in ("k", "v"):
        x = t[n].clone()
        for j, vv in enumerate(p.kv_var):
            x[:, :, j * 256 + vv:(j + 1) * 256] = torch.randn(x[:, :, j * 256 + vv:(j + 1) * 256].shape, generator=g).to(x.dtype) * 7
        t2[n] = x
    args = lambda tt: (_np(tt["dO"]), _np(tt["q"]), _np(tt["k"]), _np(tt["v"]), qi, qc, cap)
    o1 = orc.forward_rows(p, _np(t["q"]), _np(t["k"]), _np(t["v"]), qi, qc, cap, gate=_np(t["gate"]))
    o2 = orc.forward_rows(p, _np(t2["q"]), _np(t2["k"]), _np(t2["v"]), qi, qc, cap, gate=_np(t["gate"]))
    for a, b in zip(o1, o2):
        assert np.array_equal(a, b)
    g1 = orc.backward_dkdv_tiles(p, *args(t), gate=_np(t["gate"]))
    g2 = orc.backward_dkdv_tiles(p, *args(t2), gate=_np(t["gate"]))
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)
        for j, vv in enumerate(p.kv_var):           # tiles listed (b, hk, j) with j fastest
            assert np.all(a[j::p.nKV, vv:] == 0)


def test_probabilities_sum_to_one_over_unmasked_keys():
    p = small(kv_var=(256, 173, 79, 256), q_var=(256, 61, 199), topk=2)
    t = make_tensors(p)
    qi, qc, cap, (_, _, lse) = _fwd(p, t)
    q, k = to_bhsd(p, _np(t["q"]), True), to_bhsd(p, _np(t["k"]), False)
    rows = p.rows()
    for h in range(p.Hq):
        m = key_mask(p, qi, qc, 0, h)
        s = (q[0, h] @ k[0, h].T) * p.scale
        lse_h = torch.as_tensor(lse[rows[:, 1] == h])
        tot = torch.where(m, torch.exp(s - lse_h[:, None]), torch.zeros_like(s)).sum(-1)
        np.testing.assert_allclose(tot.numpy(), 1.0, rtol=0, atol=1e-12)


# ------------------------------------------------------ O6 compression

def test_compression_gate_zero_gives_sparse_output():
    p = small(kv_var=(256, 173, 79, 256), q_var=(256, 61, 199), topk=2, gate="randn01")
    t = make_tensors(p)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    out, osp, _ = orc.forward_rows(p, _np(t["q"]), _np(t["k"]), _np(t["v"]), qi, qc, p.cap,
                                   gate=np.zeros(p.shape(True)))
    assert np.array_equal(out, osp)


def test_compression_single_tile_and_identical_keys_closed_forms():
    p = small(kv_var=(0, 90, 0), q_var=(256, 40), topk=1, gate="randn01")
    t = make_tensors(p)
    c = orc.compress_c(p, _np(t["q"]), _np(t["k"]), _np(t["v"]))
    v = to_bhsd(p, _np(t["v"]), False).numpy()
    np.testing.assert_allclose(c[0, :, 0], v[0, :, 256:256 + 90].mean(axis=1), rtol=0, atol=1e-14)
    np.testing.assert_allclose(c[0, :, 1], v[0, :, 256:256 + 90].mean(axis=1), rtol=0, atol=1e-14)
    # identical pooled keys: the softmax is uniform over the non-empty tiles
    p2 = small(kv_var=(256, 100, 0, 256), q_var=(256,), topk=1, gate="randn01")
    t2 = make_tensors(p2)
    k2 = torch.ones_like(t2["k"])
    for j, vv in enumerate(p2.kv_var):
        k2[:, :, j * 256 + vv:(j + 1) * 256] = 0
    c2 = orc.compress_c(p2, _np(t2["q"]), _np(k2), _np(t2["v"]))
    v2 = to_bhsd(p2, _np(t2["v"]), False).numpy()
    means = [v2[0, :, j * 256:j * 256 + vv].mean(axis=1) for j, vv in enumerate(p2.kv_var) if vv > 0]
    np.testing.assert_allclose(c2[0, :, 0], np.mean(means, axis=0), rtol=0, atol=1e-14)


# ------------------------------------------------------------- O7 backward

def _bwd(p, t, qi, qc, cap, gate=None):
    a = (_np(t["dO"]), _np(t["q"]), _np(t["k"]), _np(t["v"]), qi, qc, cap)
    dq = orc.backward_dq_rows(p, *a, gate=gate)
    dk, dv = orc.backward_dkdv_tiles(p, *a, gate=gate)
    return dq, orc._scatter_kv(p, p.kv_tiles(), dk), orc._scatter_kv(p, p.kv_tiles(), dv)


@pytest.mark.parametrize("layout,Hkv", [("bhsd", 2), ("bshd", 1)])
def test_rowsum_do_o_equals_sum_p_dp(layout, Hkv):
    """The identity behind the backward preprocess: with O_t = sum_u P_tu v_u,
    dO_t . O_t = sum_u P_tu (dO_t . v_u). The left side uses the oracle's O,
    the right side its LSE through P_tu = exp(scale q_t . k_u - LSE_t) over
    the allowed keys, computed here in fp64 -- so the oracle's two forward
    outputs are checked against each other (an empty tile and partial tiles
    included)."""
    p = small(layout, kv_var=(256, 173, 0, 79, 256), q_var=(256, 61, 199), topk=3, Hkv=Hkv)
    t = make_tensors(p)
    qi, qc, cap, (_, osp, lse) = _fwd(p, t)
    q, k, v, dO = (to_bhsd(p, _np(t[n]), n in ("q", "dO")).numpy() for n in ("q", "k", "v", "dO"))
    g = p.Hq // p.Hkv
    rows = p.rows()
    checked = 0
    for b in range(p.B):
        for h in range(p.Hq):
            sel = (rows[:, 0] == b) & (rows[:, 1] == h)
            s_idx = rows[sel, 2]
            m = key_mask(p, qi, qc, b, h).numpy()[s_idx]            # [rows, Skv]
            S = p.scale * q[b, h, s_idx] @ k[b, h // g].T
            L = lse[sel][:, None]
            P = np.where(m, np.exp(np.where(m, S, 0.0) - np.where(np.isfinite(L), L, 0.0)), 0.0)
            dP = dO[b, h, s_idx] @ v[b, h // g].T
            rhs = (P * dP).sum(axis=1)
            lhs = (dO[b, h, s_idx] * osp[sel]).sum(axis=1)
            np.testing.assert_allclose(lhs, rhs, rtol=1e-9, atol=1e-12)
            checked += len(s_idx)
    assert checked == len(rows)


@pytest.mark.parametrize("layout,Hkv", [("bhsd", 2), ("bshd", 1)])
def test_sparse_grads_equal_torch_autograd(layout, Hkv):
    p = small(layout, kv_var=(256, 173, 79, 256), q_var=(256, 61, 199), topk=2, Hkv=Hkv)
    t = make_tensors(p)
    qi, qc, cap, _ = _fwd(p, t)
    dq, dk, dv = _bwd(p, t, qi, qc, cap)
    q, k, v = (to_bhsd(p, _np(t[n]), n == "q").requires_grad_(True) for n in "qkv")
    dO = to_bhsd(p, _np(t["dO"]), True)
    g = p.Hq // p.Hkv
    ke, ve = k.repeat_interleave(g, 1), v.repeat_interleave(g, 1)
    loss = 0
    for h in range(p.Hq):
        m = key_mask(p, qi, qc, 0, h)
        o, _ = masked_attention_f64(q[:, h], ke[:, h], ve[:, h], m, p.scale)
        loss = loss + (o * dO[:, h]).sum()
    loss.backward()
    rows = p.rows()
    np.testing.assert_allclose(dq, q.grad[0, rows[:, 1], rows[:, 2]].numpy(), rtol=0, atol=1e-10)
    kg, vg = k.grad.numpy(), v.grad.numpy()
    if layout == "bshd":
        kg, vg = kg.transpose(0, 2, 1, 3), vg.transpose(0, 2, 1, 3)
    np.testing.assert_allclose(dk, kg, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, vg, rtol=0, atol=1e-10)


def test_gated_grads_match_central_finite_differences():
    """fp64 central differences of L = sum(out * dO) on a tiny problem with
    ragged tiles, GQA and the gate, block index held fixed."""
    p = Problem("fd", "bshd", 1, 2, 1, 8, 4, 4, 2, 3, q_var=[4, 2], kv_var=[4, 3, 1], topk=2,
                gate="randn01", seed=4)
    t = make_tensors(p)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], 2, 2)
    rng = np.random.default_rng(0)
    x = {n: rng.standard_normal(p.shape(n in ("q", "dO", "gate"))) for n in ("q", "k", "v", "dO", "gate")}
    for n, var, T in (("q", p.q_var, 4), ("k", p.kv_var, 4), ("v", p.kv_var, 4)):
        for j, vv in enumerate(var):
            x[n][:, j * T + vv:(j + 1) * T] = 0.0

    def loss(xx):
        out, _, _ = orc.forward_rows(p, xx["q"], xx["k"], xx["v"], qi, qc, 2, gate=xx["gate"])
        return float((out * xx["dO"][0].reshape(-1, p.Hq, p.D)[p.rows()[:, 2], p.rows()[:, 1]]).sum())

    a = (x["dO"], x["q"], x["k"], x["v"], qi, qc, 2)
    dq = orc.backward_dq_rows(p, *a, gate=x["gate"])
    dk, dv = orc.backward_dkdv_tiles(p, *a, gate=x["gate"])
    dq = orc._scatter_rows(p, p.rows(), dq)
    dk, dv = orc._scatter_kv(p, p.kv_tiles(), dk), orc._scatter_kv(p, p.kv_tiles(), dv)
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        for idx in np.ndindex(x[name].shape):
            xp = {n: a_.copy() for n, a_ in x.items()}
            xm = {n: a_.copy() for n, a_ in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            fd = (loss(xp) - loss(xm)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_gqa_equals_repeated_mha():
    pg = small("bshd", kv_var=(256, 173, 79, 256), q_var=(256, 61), topk=2, H=4, Hkv=2, gate="randn01")
    t = make_tensors(pg)
    pm = small("bshd", kv_var=(256, 173, 79, 256), q_var=(256, 61), topk=2, H=4, Hkv=4, gate="randn01")
    tm = dict(t)
    tm["k"] = t["k"].repeat_interleave(2, dim=2)
    tm["v"] = t["v"].repeat_interleave(2, dim=2)
    rg = orc.run_full(pg, t)
    rm = orc.run_full(pm, tm)
    assert np.array_equal(rg["map"], rm["map"])
    for n in ("out", "lse", "dq"):
        np.testing.assert_allclose(rg[n], rm[n], rtol=0, atol=1e-12)
    for n in ("dk", "dv"):
        s = rm[n].reshape(1, pg.Skv, 2, 2, pg.D).sum(axis=3)
        np.testing.assert_allclose(rg[n], s, rtol=0, atol=1e-12)


def test_varlen_equals_per_sequence_runs():
    lens_q, lens_kv = [130, 5, 77], [20, 300, 129]
    p = tnd_problem("t", lens_q, lens_kv, 4, 2, tile=128, seed=8, topk=2, gate="randn01")
    t = make_tensors(p)
    r = orc.run_full(p, t)
    for b in range(3):
        pb = tnd_problem("t1", [lens_q[b]], [lens_kv[b]], 4, 2, tile=128, topk=2, gate="randn01")
        qs, ks = slice(p.cu_q[b], p.cu_q[b + 1]), slice(p.cu_kv[b], p.cu_kv[b + 1])
        tb = {n: t[n][qs] for n in ("q", "dO", "gate")}
        tb.update({n: t[n][ks] for n in ("k", "v")})
        rb = orc.run_full(pb, tb)
        nq = rb["q_cnt"].shape[2]
        assert np.array_equal(r["q_cnt"][b, :, :nq], rb["q_cnt"][0])
        np.testing.assert_allclose(r["out"][qs], rb["out"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(r["lse"][:, qs], rb["lse"], rtol=0, atol=1e-13)
        for n in ("dq",):
            np.testing.assert_allclose(r[n][qs], rb[n], rtol=0, atol=1e-12)
        for n in ("dk", "dv"):
            np.testing.assert_allclose(r[n][ks], rb[n], rtol=0, atol=1e-12)


def test_npu_page_length_lists_run_with_patterned_mask():
    """The varlen GQA cases of the Ascend page with its sparse mask pattern
    (each Q block attends block (i+b+n) mod nkv_b, plus the next one when
    i+n is even); forward equals the per-sequence masked SDPA."""
    g = load_golden("npu_tnd_cases.json")
    for case in g["cases"][:2]:
        p = npu_problem(case)
        t = make_tensors(p)
        mask = np.zeros((p.B, p.Hq, p.nQ, p.nKV), dtype=np.uint8)
        for b in range(p.B):
            nk = -(-p.kv_lens[b] // 128)
            for h in range(p.Hq):
                for i in range(p.nQ):
                    mask[b, h, i, (i + b + h) % nk] = 1
                    if nk > 1 and (i + h) % 2 == 0:
                        mask[b, h, i, (i + b + h + 1) % nk] = 1
        qi, qc, cap, (out, _, lse) = _fwd(p, t, mask=mask)
        q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
        gsz = p.Hq // p.Hkv
        r = 0
        for b in range(p.B):
            lq, lk = p.q_lens[b], p.kv_lens[b]
            for h in range(p.Hq):
                full = torch.as_tensor(mask[b, h]).bool().repeat_interleave(128, 0).repeat_interleave(128, 1)
                ro, _ = masked_attention_f64(torch.as_tensor(q[p.cu_q[b]:p.cu_q[b] + lq, h]),
                                             torch.as_tensor(k[p.cu_kv[b]:p.cu_kv[b] + lk, h // gsz]),
                                             torch.as_tensor(v[p.cu_kv[b]:p.cu_kv[b] + lk, h // gsz]),
                                             full[:lq, :lk], p.scale)
                np.testing.assert_allclose(out[r:r + lq], ro.numpy(), rtol=0, atol=1e-11)
                r += lq


# ------------------------------------------------------------ 3D video tiling

def test_tile3d_divisible_grid_is_the_block_permutation():
    """On a grid the box divides, tiling is the plain block permutation
    (tiles in raster order, tokens in raster order inside each tile),
    written here as one reshape/transpose, independent of the oracle's
    per-tile loop."""
    from oracle import tile3d
    rng = np.random.default_rng(3)
    B, T, H, W, R = 2, 8, 16, 24, 5
    x = rng.standard_normal((B, T, H, W, R)).astype(np.float32)
    tiled, var = tile3d.tile_3d(x, (4, 8, 8))
    ref = x.reshape(B, 2, 4, 2, 8, 3, 8, R).transpose(0, 1, 3, 5, 2, 4, 6, 7).reshape(B, -1, R)
    np.testing.assert_array_equal(tiled, ref)
    assert (var == 256).all() and var.size == 12


def test_tile3d_gated_ragged_grid_counts():
    """The gated-ragged workload's KV grid 21x45x80 tiled 4x8x8 gives 360
    tiles with valid counts 256 x 250, 160 x 50, 64 x 50 and 40 x 10, the
    same list, in the same raster order, as the workload's kv_var."""
    from oracle import tile3d
    x = np.zeros((1, 21, 45, 80, 1), dtype=np.float32)
    _, var = tile3d.tile_3d(x, (4, 8, 8))
    vals, counts = np.unique(var, return_counts=True)
    assert dict(zip(vals.tolist(), counts.tolist())) == {40: 10, 64: 50, 160: 50, 256: 250}
    assert tile3d.tile_count(21, 45, 80) == 360
    from bwd_tile_mean_gb300.inputs import config
    assert var.tolist() == list(config(4).kv_var)


def test_tile3d_round_trip_and_zero_padding():
    """untile(tile(x)) == x on ragged grids; every slot past a tile's count
    is zero; the counts sum to the number of tokens."""
    from oracle import tile3d
    rng = np.random.default_rng(4)
    for grid in [(5, 9, 7), (1, 1, 1), (4, 8, 8), (6, 17, 3)]:
        x = rng.standard_normal((2,) + grid + (3,)).astype(np.float32) + 1.0
        tiled, var = tile3d.tile_3d(x, (4, 8, 8))
        np.testing.assert_array_equal(tile3d.untile_3d(tiled, grid, (4, 8, 8)), x)
        assert int(var.sum()) == grid[0] * grid[1] * grid[2]
        slots = tiled.reshape(2, var.size, 256, 3)
        for k, n in enumerate(var):
            assert (slots[:, k, n:] == 0).all() and (slots[:, k, :n] != 0).all()


# ----------------------------------------------- compression gate gradient

def test_gate_grad_matches_finite_differences_of_the_forward():
    """dgate from the oracle's closed form equals the central difference of
    the oracle's gated forward output (out = O + gate (*) c is linear in the
    gate, so the difference is exact up to rounding), at positions in full,
    partial and padding slots of several tiles and heads."""
    p = Problem("gate-fd", "bshd", 1, 2, 2, 128, 256, 256, 3, 4, q_var=[256, 100, 7],
                kv_var=[256, 40, 0, 199], topk=2, gate="randn01", seed=41)
    t = make_tensors(p)
    q, k, v, dO, gate = (_np(t[n]).astype(np.float64) for n in ("q", "k", "v", "dO", "gate"))
    dg = orc.gate_grad(p, dO, q, k, v)
    _, qi, qc, _ = orc.build_block_map(p, t["q"], t["k"], p.topk, p.cap)
    eps = 0.5
    for (s, h, d) in [(0, 0, 0), (300, 1, 17), (511, 0, 127), (600, 1, 64), (767, 0, 5)]:
        rows = np.asarray([[0, h, s]], dtype=np.int32)
        gp, gm = gate.copy(), gate.copy()
        gp[0, s, h, d] += eps
        gm[0, s, h, d] -= eps
        op = orc.forward_rows(p, q, k, v, qi, qc, p.cap, gate=gp, rows=rows)[0]
        om = orc.forward_rows(p, q, k, v, qi, qc, p.cap, gate=gm, rows=rows)[0]
        fd = (op[0, d] - om[0, d]) / (2 * eps) * dO[0, s, h, d]
        assert abs(fd - dg[0, s, h, d]) <= 1e-12 * max(1.0, abs(fd)), (s, h, d, fd, dg[0, s, h, d])
        # nothing else in the row moves with this gate element
        others = np.delete(np.arange(128), d)
        assert np.allclose(op[0, others], om[0, others], rtol=0, atol=1e-12)

"""Shared test helpers: problem builders from the page fixtures, error
metrics, and float64 torch references used to pin the oracle."""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

from bwd_tile_mean_gb300.inputs import Problem, tnd_problem

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def page_problem(case, layout, dtype="bf16"):
    g = load_golden("vsa_page_cases.json")
    return Problem(f"{case['name']}-{layout}", layout, 1, g["heads"], g["heads"], g["head_dim"],
                   g["tile"], g["tile"], len(case["q_var"]), len(case["kv_var"]), dtype=dtype,
                   q_var=case["q_var"], kv_var=case["kv_var"], topk=case["topk"], seed=case["seed"],
                   gate=case["gate"])


def npu_problem(case, dtype="fp16", seed=42):
    return tnd_problem(case["name"], case["q_lengths"], case["kv_lengths"], case["num_heads"],
                       case["num_kv_heads"], dtype=dtype, seed=seed)


# ------------------------------------------------------------------ metrics

def metrics(ref, got):
    """(avg_abs, max_rel): mean |got - ref| and max |got - ref| / max |ref|.

    The pages name these two numbers but do not show their definition; this
    is the reading the tests use (relative to the tensor's largest entry,
    so that near-zero entries do not dominate)."""
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    diff = np.abs(got - ref)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    avg = float(diff.mean()) if ref.size else 0.0
    mx = float(diff.max() / scale) if ref.size and scale > 0 else float(diff.max() if ref.size else 0.0)
    return avg, mx


def check_tol(tag, ref, got, tol):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{tag}: non-finite values"
    avg, mx = metrics(ref, got)
    assert avg < tol[0], f"{tag}: avg_abs {avg:.3e} >= {tol[0]:.3e}"
    assert mx < tol[1], f"{tag}: max_rel {mx:.3e} >= {tol[1]:.3e}"
    return avg, mx


OUT_TOL = (1e-3, 0.2)
GRAD_TOL = (1e-3, 0.25)


# ------------------------------------------------- exact fp32 arithmetic

def round_to_f32(x: Fraction) -> np.float32:
    """Correctly rounded (ties to even) float32 nearest to the rational x."""
    if x == 0:
        return np.float32(0.0)
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]

    def key(c):
        lsb = int(np.frombuffer(np.float32(c).tobytes(), dtype=np.uint32)[0]) & 1
        return (abs(Fraction(float(c)) - x), lsb)

    return np.float32(min(cands, key=key))


def exact_fmaf(a, b, c) -> np.float32:
    """fmaf from its definition: a*b + c computed exactly, rounded once."""
    return round_to_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


# ------------------------------------------------ float64 torch references

def to_bhsd(p, x, q_side):
    """[B, H, S, D] float64 view of a padded-layout tensor."""
    x = torch.as_tensor(np.asarray(x, dtype=np.float64))
    if p.layout == "bshd":
        x = x.transpose(1, 2)
    return x.contiguous()


def key_mask(p, q_idx, q_cnt, b, h):
    """Boolean [Sq, Skv] mask of (row, key) pairs the sparse pattern allows,
    for one batch entry and head of a padded-layout problem."""
    m = torch.zeros(p.Sq, p.Skv, dtype=torch.bool)
    for i in range(p.nQ):
        for n in range(int(q_cnt[b, h, i])):
            j = int(q_idx[b, h, i, n])
            vv = p.tile_var(False, b, j)
            m[i * p.tile_q:(i + 1) * p.tile_q, j * p.tile_kv:j * p.tile_kv + vv] = True
    return m


def masked_attention_f64(q, k, v, mask, scale):
    """Library softmax attention (torch SDPA, float64) with a boolean mask;
    rows with no allowed key are returned as 0 with LSE -inf."""
    import torch.nn.functional as F
    out = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    empty = ~mask.any(dim=-1)
    out = torch.where(empty[..., None], torch.zeros_like(out), out)
    return out, lse


# ------------------------------------------------------- GPU path plumbing

def plan_for(p, device="cuda"):
    """A libvsa Plan for problem p (descriptor, workspace, index buffers)."""
    from bwd_tile_mean_gb300 import vsa
    from bwd_tile_mean_gb300.inputs import DTYPES
    dev = torch.device(device)
    i32 = dict(dtype=torch.int32, device=dev)
    kw = {}
    if p.varlen:
        kw.update(cu_seqlens_q=torch.as_tensor(p.cu_q, **i32), cu_seqlens_kv=torch.as_tensor(p.cu_kv, **i32))
    else:
        kw.update(q_var=torch.as_tensor(p.q_var, **i32), kv_var=torch.as_tensor(p.kv_var, **i32))
    return vsa.Plan(p.layout, DTYPES[p.dtype], p.B, p.Hq, p.Hkv, p.D, p.tile_q, p.tile_kv, p.nQ, p.nKV, p.Sq,
                    p.Skv, p.cap, gate=p.gate is not None, scale=p.scale, device=dev, **kw)


def to_device(t, device="cuda"):
    return {n: x.to(device) for n, x in t.items()}

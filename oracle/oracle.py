"""ctypes bindings of the plain-C oracle (vsa_oracle.c).

TEST INFRASTRUCTURE. Only tests/, the smoke check and the benchmark's CPU
baseline leg import this module. It never touches the CUDA library.

Every function takes a ``Problem`` (bwd_tile_mean_gb300.inputs) and host
arrays (numpy, or CPU/GPU torch tensors, which are copied to the host).
The selection step reads float32 images of the inputs; attention and
gradients read and return float64.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsa_oracle.c")
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_LAYOUT = {"bhsd": 0, "bshd": 1, "tnd": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction, no fast-math)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_SO)
    return _lib


class _Desc(C.Structure):
    _fields_ = [("layout", C.c_int), ("B", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int),
                ("D", C.c_int), ("Sq", C.c_int), ("Skv", C.c_int), ("tile_q", C.c_int),
                ("tile_kv", C.c_int), ("nQ", C.c_int), ("nKV", C.c_int),
                ("cu_q", C.c_void_p), ("cu_kv", C.c_void_p), ("q_var", C.c_void_p),
                ("kv_var", C.c_void_p), ("scale", C.c_double)]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


class _Bound:
    """A filled descriptor plus the arrays it points to (kept alive)."""

    def __init__(self, p):
        self.keep = []

        def arr(x):
            if x is None:
                return None
            x = np.ascontiguousarray(x, dtype=np.int32)
            self.keep.append(x)
            return _ptr(x)

        if p.layout != "tnd":
            # a tile fill is a count of valid slots in [0, tile] (FastVideo
            # block_sparse_attn_cute_fwd.py, _vbs_mask_mod: key n valid iff
            # n mod tile < vbs); the pages give no meaning to other values
            for name, var, tile in (("q_var", p.q_var, p.tile_q), ("kv_var", p.kv_var, p.tile_kv)):
                v = np.asarray(var)
                if v.size and (int(v.min()) < 0 or int(v.max()) > tile):
                    raise ValueError(f"{name} outside [0, {tile}]")
        self.p = p
        self.d = _Desc(_LAYOUT[p.layout], p.B, p.Hq, p.Hkv, p.D, p.Sq, p.Skv, p.tile_q, p.tile_kv,
                       p.nQ, p.nKV, arr(p.cu_q), arr(p.cu_kv), arr(p.q_var), arr(p.kv_var),
                       float(p.scale))

    @property
    def ref(self):
        return C.byref(self.d)


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().double().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


# --------------------------------------------------------------- selection

def pool_f32(p, x, q_side: bool) -> np.ndarray:
    """O1: fp32 tile means, [B, H, nT, D]."""
    bd = _Bound(p)
    H, nT = (p.Hq, p.nQ) if q_side else (p.Hkv, p.nKV)
    out = np.zeros((p.B, H, nT, p.D), dtype=np.float32)
    x = _f32(x)
    lib().orc_pool_f32(bd.ref, C.c_int(int(q_side)), _ptr(x), _ptr(out))
    return out


def select(p, pq, pk, topk: int, cap: int):
    """O2 + O3: returns (map u8 [B,Hq,nQ,nKV], q_idx i32 [B,Hq,nQ,cap],
    q_cnt i32 [B,Hq,nQ], scores f32 [B,Hq,nQ,nKV])."""
    bd = _Bound(p)
    pq, pk = _f32(pq), _f32(pk)
    m = np.zeros((p.B, p.Hq, p.nQ, p.nKV), dtype=np.uint8)
    qi = np.zeros((p.B, p.Hq, p.nQ, cap), dtype=np.int32)
    qc = np.zeros((p.B, p.Hq, p.nQ), dtype=np.int32)
    sc = np.zeros((p.B, p.Hq, p.nQ, p.nKV), dtype=np.float32)
    lib().orc_select(bd.ref, _ptr(pq), _ptr(pk), C.c_int(topk), _ptr(m), _ptr(qi), _ptr(qc),
                     C.c_int(cap), _ptr(sc))
    return m, qi, qc, sc


def build_block_map(p, q, k, topk: int, cap: int = None):
    """Pool + select, the whole block-map step of the oracle."""
    cap = cap if cap is not None else min(topk, p.nKV)
    pq = pool_f32(p, q, True)
    pk = pool_f32(p, k, False)
    return select(p, pq, pk, topk, cap)


def mask_index(p, mask, cap: int):
    bd = _Bound(p)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    qi = np.zeros((p.B, p.Hq, p.nQ, cap), dtype=np.int32)
    qc = np.zeros((p.B, p.Hq, p.nQ), dtype=np.int32)
    lib().orc_mask_index(bd.ref, _ptr(mask), _ptr(qi), _ptr(qc), C.c_int(cap))
    return qi, qc


def transpose(p, q_idx, q_cnt, cap: int):
    """O4: returns (kv_ptr [B,Hq,nKV+1], kv_qidx [B,Hq,nQ*cap])."""
    bd = _Bound(p)
    q_idx, q_cnt = _i32(q_idx), _i32(q_cnt)
    kp = np.zeros((p.B, p.Hq, p.nKV + 1), dtype=np.int32)
    kq = np.zeros((p.B, p.Hq, p.nQ * cap), dtype=np.int32)
    lib().orc_transpose(bd.ref, _ptr(q_idx), _ptr(q_cnt), C.c_int(cap), _ptr(kp), _ptr(kq))
    return kp, kq


# --------------------------------------------------------------- attention

def compress_c(p, q, k, v) -> np.ndarray:
    bd = _Bound(p)
    c = np.zeros((p.B, p.Hq, p.nQ, p.D), dtype=np.float64)
    lib().orc_compress_c(bd.ref, _ptr(_f64(q)), _ptr(_f64(k)), _ptr(_f64(v)), _ptr(c))
    return c


def forward_rows(p, q, k, v, q_idx, q_cnt, cap, gate=None, rows=None):
    """O5/O6 on the listed rows ((b, h, s) triples; default all rows).
    Returns (out [n, D], o_sparse [n, D], lse [n]) in float64."""
    bd = _Bound(p)
    rows = p.rows() if rows is None else _i32(rows).reshape(-1, 3)
    q, k, v, gate = _f64(q), _f64(k), _f64(v), _f64(gate)
    q_idx, q_cnt = _i32(q_idx), _i32(q_cnt)
    c = compress_c(p, q, k, v) if gate is not None else None
    n = rows.shape[0]
    out = np.zeros((n, p.D)), np.zeros((n, p.D)), np.zeros(n)
    lib().orc_forward_rows(bd.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(q_cnt),
                           C.c_int(cap), _ptr(gate), _ptr(c), _ptr(rows), C.c_long(n),
                           _ptr(out[0]), _ptr(out[1]), _ptr(out[2]))
    return out


def gate_grad(p, dO, q, k, v) -> np.ndarray:
    """Gradient of the compression gate, float64 in dO's shape: out = O +
    gate (*) c_i over every slot of query tile i, hence dgate = dO (*) c_i
    (padded layouts: every slot; TND: rows inside a sequence, zero
    elsewhere)."""
    c = compress_c(p, q, k, v)
    dO = _f64(dO)
    dg = np.zeros_like(dO)
    for b, h, s in p.rows():
        i = s // p.tile_q
        if p.layout == "bhsd":
            dg[b, h, s] = dO[b, h, s] * c[b, h, i]
        elif p.layout == "bshd":
            dg[b, s, h] = dO[b, s, h] * c[b, h, i]
        else:
            dg[p.cu_q[b] + s, h] = dO[p.cu_q[b] + s, h] * c[b, h, i]
    return dg


def compress_grads(p, dO, gate, q, k, v):
    bd = _Bound(p)
    dpq = np.zeros((p.B, p.Hq, p.nQ, p.D))
    dpk = np.zeros((p.B, p.Hkv, p.nKV, p.D))
    dpv = np.zeros((p.B, p.Hkv, p.nKV, p.D))
    lib().orc_compress_grads(bd.ref, _ptr(_f64(dO)), _ptr(_f64(gate)), _ptr(_f64(q)),
                             _ptr(_f64(k)), _ptr(_f64(v)), _ptr(dpq), _ptr(dpk), _ptr(dpv))
    return dpq, dpk, dpv


def backward_dq_rows(p, dO, q, k, v, q_idx, q_cnt, cap, gate=None, rows=None, cgrads=None):
    """O7 (+O8) dQ of the listed rows, [n, D] float64."""
    bd = _Bound(p)
    rows = p.rows() if rows is None else _i32(rows).reshape(-1, 3)
    dO, q, k, v, gate = _f64(dO), _f64(q), _f64(k), _f64(v), _f64(gate)
    dpq = None
    if gate is not None:
        cgrads = cgrads if cgrads is not None else compress_grads(p, dO, gate, q, k, v)
        dpq = cgrads[0]
    n = rows.shape[0]
    dq = np.zeros((n, p.D))
    lib().orc_backward_dq_rows(bd.ref, _ptr(dO), _ptr(q), _ptr(k), _ptr(v), _ptr(_i32(q_idx)),
                               _ptr(_i32(q_cnt)), C.c_int(cap), _ptr(dpq), _ptr(rows),
                               C.c_long(n), _ptr(dq))
    return dq


def backward_dkdv_tiles(p, dO, q, k, v, q_idx, q_cnt, cap, gate=None, tiles=None, cgrads=None):
    """O7 (+O8) dK, dV of the listed KV tiles ((b, hk, j) triples; default
    all), each [n, tile_kv, D] float64."""
    bd = _Bound(p)
    tiles = p.kv_tiles() if tiles is None else _i32(tiles).reshape(-1, 3)
    dO, q, k, v, gate = _f64(dO), _f64(q), _f64(k), _f64(v), _f64(gate)
    dpk = dpv = None
    if gate is not None:
        cgrads = cgrads if cgrads is not None else compress_grads(p, dO, gate, q, k, v)
        dpk, dpv = cgrads[1], cgrads[2]
    n = tiles.shape[0]
    dk = np.zeros((n, p.tile_kv, p.D))
    dv = np.zeros((n, p.tile_kv, p.D))
    lib().orc_backward_dkdv_tiles(bd.ref, _ptr(dO), _ptr(q), _ptr(k), _ptr(v), _ptr(_i32(q_idx)),
                                  _ptr(_i32(q_cnt)), C.c_int(cap), _ptr(dpk), _ptr(dpv),
                                  _ptr(tiles), C.c_long(n), _ptr(dk), _ptr(dv))
    return dk, dv


# ------------------------------------------------------ whole-problem runs

def _scatter_rows(p, rows, vals, lse_mode=False):
    """Place packed per-row values into the problem's layout (indexing only)."""
    b, h, s = rows[:, 0], rows[:, 1], rows[:, 2]
    if lse_mode:
        if p.varlen:
            out = np.full(p.lse_shape(), np.nan)
            out[h, p.cu_q[b] + s] = vals
        else:
            out = np.full(p.lse_shape(), np.nan)
            out[b, h, s] = vals
        return out
    out = np.zeros(p.shape(True), dtype=np.float64)
    if p.layout == "bhsd":
        out[b, h, s] = vals
    elif p.layout == "bshd":
        out[b, s, h] = vals
    else:
        out[p.cu_q[b] + s, h] = vals
    return out


def _scatter_kv(p, tiles, vals):
    out = np.zeros(p.shape(False), dtype=np.float64)
    for n, (b, hk, j) in enumerate(tiles):
        vv = p.tile_var(False, int(b), int(j)) if p.varlen else p.tile_kv
        s0 = j * p.tile_kv
        if p.layout == "bhsd":
            out[b, hk, s0:s0 + vv] = vals[n, :vv]
        elif p.layout == "bshd":
            out[b, s0:s0 + vv, hk] = vals[n, :vv]
        else:
            base = p.cu_kv[b] + s0
            out[base:base + vv, hk] = vals[n, :vv]
    return out


def run_full(p, t, mask=None, with_backward=True):
    """Oracle block map (or the given mask's index), forward and backward of
    the whole problem; outputs placed in the problem's layouts."""
    q, k, v = _f64(t["q"]), _f64(t["k"]), _f64(t["v"])
    gate = _f64(t.get("gate"))
    res = {}
    if mask is None:
        cap = p.cap
        m, qi, qc, sc = build_block_map(p, t["q"], t["k"], p.topk, cap)
        res.update(map=m, scores=sc)
    else:
        cap = p.nKV
        qi, qc = mask_index(p, mask, cap)
    kp, kq = transpose(p, qi, qc, cap)
    res.update(q_idx=qi, q_cnt=qc, kv_ptr=kp, kv_qidx=kq, cap=cap)
    rows = p.rows()
    out, osp, lse = forward_rows(p, q, k, v, qi, qc, cap, gate=gate, rows=rows)
    res["out"] = _scatter_rows(p, rows, out)
    res["o_sparse"] = _scatter_rows(p, rows, osp)
    res["lse"] = _scatter_rows(p, rows, lse, lse_mode=True)
    if with_backward:
        dO = _f64(t["dO"])
        cg = compress_grads(p, dO, gate, q, k, v) if gate is not None else None
        dq = backward_dq_rows(p, dO, q, k, v, qi, qc, cap, gate=gate, rows=rows, cgrads=cg)
        tiles = p.kv_tiles()
        dk, dv = backward_dkdv_tiles(p, dO, q, k, v, qi, qc, cap, gate=gate, tiles=tiles, cgrads=cg)
        res["dq"] = _scatter_rows(p, rows, dq)
        res["dk"] = _scatter_kv(p, tiles, dk)
        res["dv"] = _scatter_kv(p, tiles, dv)
    return res


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

"""Python binding of libvsa.so (include/vsa.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels. PyTorch provides device memory and streams. The
functions named like the C entry points (``vsa_build_block_map``,
``vsa_mask_to_index``, ``vsa_fwd``, ``vsa_bwd``, ...) take torch tensors
and pass their device pointers; ``Plan`` wraps a problem's descriptor,
workspace and index buffers for convenient use. There is no fallback: a
missing library raises.
"""
from __future__ import annotations

import ctypes as C
import math
import os
import weakref
from typing import Optional

import torch

from . import build as _build

LAYOUTS = {"bhsd": 0, "bshd": 1, "tnd": 2}
DTYPES = {torch.bfloat16: 0, torch.float16: 1}

STATUS = {0: "VSA_OK", 1: "VSA_ERR_NULL", 2: "VSA_ERR_SHAPE", 3: "VSA_ERR_DTYPE", 4: "VSA_ERR_LAYOUT",
          5: "VSA_ERR_UNSUPPORTED", 6: "VSA_ERR_MISSING_SEQLENS", 7: "VSA_ERR_WORKSPACE",
          8: "VSA_ERR_CUDA", 9: "VSA_ERR_DEVICE", 10: "VSA_ERR_SCRATCH"}

EXPORTS = ("vsa_workspace_size", "vsa_build_block_map", "vsa_build_block_map_static", "vsa_mask_to_index",
           "vsa_fwd", "vsa_bwd",
           "vsa_status_string", "vsa_last_cuda_error", "vsa_device_status", "vsa_profile_enable", "vsa_profile_count",
           "vsa_profile_name", "vsa_profile_ms", "vsa_profile_reset", "vsa_launch_count",
           "vsa_tile_3d_count", "vsa_tile_3d", "vsa_untile_3d", "vsa_gate_grad",
           "vsa_mask_to_index_blocks", "vsa_fwd_blocks", "vsa_bwd_blocks", "vsa_check_wait_timeout",
           "vsa_train_step_host_size", "vsa_train_step_host", "vsa_fwd_step_host", "vsa_step_host_status",
           "vsa_check_inputs", "vsa_head_slice", "vsa_fwd_reuse", "vsa_bwd_reuse")

REUSE_QK_MEANS, REUSE_V_MEANS = 1, 2  # vsa_fwd_reuse / vsa_bwd_reuse mask bits


class VsaError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = f"{fn} failed: {STATUS.get(code, code)} ({_lib.vsa_status_string(code).decode()})"
        if code == 8:
            msg += f": {_lib.vsa_last_cuda_error().decode()}"
        super().__init__(msg)


class VsaDesc(C.Structure):
    _fields_ = [("layout", C.c_int32), ("dtype", C.c_int32), ("B", C.c_int32), ("Hq", C.c_int32),
                ("Hkv", C.c_int32), ("D", C.c_int32), ("Sq", C.c_int32), ("Skv", C.c_int32),
                ("tile_q", C.c_int32), ("tile_kv", C.c_int32), ("nQ", C.c_int32), ("nKV", C.c_int32),
                ("cu_seqlens_q", C.c_void_p), ("cu_seqlens_kv", C.c_void_p), ("scale", C.c_float)]


_lib = None
P = C.c_void_p


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libvsa.so (built in-tree by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libvsa.so is not built ({path}); run __graft_entry__.build()")
        L = C.CDLL(path)
        L.vsa_workspace_size.restype = C.c_size_t
        L.vsa_workspace_size.argtypes = [C.POINTER(VsaDesc), C.c_int]
        L.vsa_build_block_map.restype = C.c_int
        L.vsa_build_block_map.argtypes = [C.POINTER(VsaDesc), P, P, P, P, C.c_int, C.c_int, P, P, P, C.c_int,
                                          P, P, P, C.c_size_t, P]
        L.vsa_build_block_map_static.restype = C.c_int
        L.vsa_build_block_map_static.argtypes = [C.POINTER(VsaDesc), P, P, P, P, C.c_int, C.c_int, P, P, P,
                                                 C.c_int, P, P, P]
        L.vsa_mask_to_index.restype = C.c_int
        L.vsa_mask_to_index.argtypes = [C.POINTER(VsaDesc), P, P, P, C.c_int, P, P, C.c_int, P, P, P]
        L.vsa_fwd.restype = C.c_int
        L.vsa_fwd.argtypes = [C.POINTER(VsaDesc), P, P, P, P, P, C.c_int, P, P, P, P, P, P, P, C.c_size_t, P]
        L.vsa_bwd.restype = C.c_int
        L.vsa_bwd.argtypes = [C.POINTER(VsaDesc), P, P, P, P, P, P, P, P, C.c_int, P, P, P, P, P, P, P, P, P,
                              C.c_size_t, P]
        L.vsa_fwd_reuse.restype = C.c_int
        L.vsa_fwd_reuse.argtypes = [C.POINTER(VsaDesc), P, P, P, P, P, C.c_int, P, P, P, P, P, P, C.c_int, P,
                                    C.c_size_t, P]
        L.vsa_bwd_reuse.restype = C.c_int
        L.vsa_bwd_reuse.argtypes = [C.POINTER(VsaDesc), P, P, P, P, P, P, P, P, C.c_int, P, P, P, P, P, P, P, P,
                                    C.c_int, P, C.c_size_t, P]
        L.vsa_status_string.restype = C.c_char_p
        L.vsa_status_string.argtypes = [C.c_int]
        L.vsa_last_cuda_error.restype = C.c_char_p
        L.vsa_device_status.restype = C.c_int
        L.vsa_device_status.argtypes = [P, P, C.POINTER(C.c_int32)]
        L.vsa_profile_enable.argtypes = [C.c_int]
        L.vsa_profile_count.restype = C.c_int
        L.vsa_profile_name.restype = C.c_char_p
        L.vsa_profile_name.argtypes = [C.c_int]
        L.vsa_profile_ms.restype = C.c_float
        L.vsa_profile_ms.argtypes = [C.c_int]
        L.vsa_launch_count.restype = C.c_longlong
        L.vsa_check_wait_timeout.restype = C.c_int
        L.vsa_check_wait_timeout.argtypes = [P, C.c_ulonglong, P, P]
        L.vsa_mask_to_index_blocks.restype = C.c_int
        L.vsa_mask_to_index_blocks.argtypes = [C.POINTER(VsaDesc), C.c_int, C.c_int, P, P, P, C.c_int, P, P, P, P,
                                               C.c_int, P, P, P, P]
        L.vsa_fwd_blocks.restype = C.c_int
        L.vsa_fwd_blocks.argtypes = [C.POINTER(VsaDesc), C.c_int, P, P, P, P, P, P, C.c_int, P, P, P, P, P,
                                     C.c_size_t, P]
        L.vsa_bwd_blocks.restype = C.c_int
        L.vsa_bwd_blocks.argtypes = [C.POINTER(VsaDesc), C.c_int, P, P, P, P, P, P, P, P, P, C.c_int, P, P, P, P,
                                     P, P, P, P, P, C.c_size_t, P]
        L.vsa_gate_grad.restype = C.c_int
        L.vsa_gate_grad.argtypes = [C.POINTER(VsaDesc), P, P, P, P, P, P, P, P, C.c_size_t, P]
        L.vsa_tile_3d_count.restype = C.c_int
        L.vsa_tile_3d_count.argtypes = [C.c_int] * 6
        L.vsa_tile_3d.restype = C.c_int
        L.vsa_tile_3d.argtypes = [C.c_int] * 8 + [P, P, P, P]
        L.vsa_untile_3d.restype = C.c_int
        L.vsa_untile_3d.argtypes = [C.c_int] * 8 + [P, P, P]
        L.vsa_train_step_host_size.restype = C.c_size_t
        L.vsa_train_step_host_size.argtypes = [C.POINTER(VsaDesc), C.c_int, C.c_int, C.c_int]
        L.vsa_train_step_host.restype = C.c_int
        L.vsa_train_step_host.argtypes = [C.POINTER(VsaDesc), C.c_int, P, P, P, P, P, P, P, C.c_int, P, P, P, P, P,
                                          P, C.c_size_t, P]
        L.vsa_step_host_status.restype = C.c_int
        L.vsa_step_host_status.argtypes = [C.POINTER(VsaDesc), C.c_int, C.c_int, C.c_int, P, P, C.POINTER(C.c_int32)]
        L.vsa_check_inputs.restype = C.c_int
        L.vsa_check_inputs.argtypes = [C.POINTER(VsaDesc), P, P, P, P, C.c_int, P, P, P, C.c_size_t, P,
                                       C.POINTER(C.c_int32)]
        L.vsa_head_slice.restype = C.c_int
        L.vsa_head_slice.argtypes = [C.POINTER(VsaDesc), C.c_int, C.c_int, C.POINTER(VsaDesc), C.POINTER(C.c_int32),
                                     C.POINTER(C.c_int32)]
        L.vsa_fwd_step_host.restype = C.c_int
        L.vsa_fwd_step_host.argtypes = [C.POINTER(VsaDesc), C.c_int, P, P, P, P, P, P, C.c_int, P, P, P, C.c_size_t,
                                        P]
        _lib = L
    return _lib


def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(fn, code):
    if code != 0:
        raise VsaError(fn, code)


# ------------------------------------------------------------- raw entry points

def vsa_workspace_size(desc: VsaDesc, with_gate: bool) -> int:
    return int(lib().vsa_workspace_size(C.byref(desc), int(bool(with_gate))))


def vsa_build_block_map(desc, q, k, q_var, kv_var, topk, need_bwd_index, block_map, q_idx, q_cnt, idx_cap,
                        kv_ptr, kv_qidx, workspace, stream=None):
    _check("vsa_build_block_map", lib().vsa_build_block_map(
        C.byref(desc), _p(q), _p(k), _p(q_var), _p(kv_var), int(topk), int(bool(need_bwd_index)),
        _p(block_map), _p(q_idx), _p(q_cnt), int(idx_cap), _p(kv_ptr), _p(kv_qidx), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def vsa_build_block_map_static(desc, q, k, q_var, kv_var, topk, need_bwd_index, block_map, q_idx, q_cnt,
                               idx_cap, kv_ptr, kv_qidx, stream=None):
    """vsa_build_block_map without a workspace: for callers that cannot
    allocate device memory (the scratch is a fixed array in the library)."""
    _check("vsa_build_block_map_static", lib().vsa_build_block_map_static(
        C.byref(desc), _p(q), _p(k), _p(q_var), _p(kv_var), int(topk), int(bool(need_bwd_index)),
        _p(block_map), _p(q_idx), _p(q_cnt), int(idx_cap), _p(kv_ptr), _p(kv_qidx), _stream(stream)))


def vsa_mask_to_index(desc, block_map, q_var, kv_var, need_bwd_index, q_idx, q_cnt, idx_cap, kv_ptr, kv_qidx,
                      stream=None):
    _check("vsa_mask_to_index", lib().vsa_mask_to_index(
        C.byref(desc), _p(block_map), _p(q_var), _p(kv_var), int(bool(need_bwd_index)), _p(q_idx), _p(q_cnt),
        int(idx_cap), _p(kv_ptr), _p(kv_qidx), _stream(stream)))


def vsa_fwd(desc, q, k, v, q_idx, q_cnt, idx_cap, q_var, kv_var, gate, out, lse, o_sparse, workspace,
            stream=None, reuse=0):
    """vsa_fwd (reuse = 0) or vsa_fwd_reuse (reuse: REUSE_* bits)."""
    args = (C.byref(desc), _p(q), _p(k), _p(v), _p(q_idx), _p(q_cnt), int(idx_cap), _p(q_var), _p(kv_var),
            _p(gate), _p(out), _p(lse), _p(o_sparse))
    tail = (_p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if reuse:
        _check("vsa_fwd_reuse", lib().vsa_fwd_reuse(*args, int(reuse), *tail))
    else:
        _check("vsa_fwd", lib().vsa_fwd(*args, *tail))


def vsa_bwd(desc, dO, q, k, v, o_sparse, lse, q_idx, q_cnt, idx_cap, kv_ptr, kv_qidx, q_var, kv_var, gate,
            dq, dk, dv, workspace, stream=None, reuse=0):
    """vsa_bwd (reuse = 0) or vsa_bwd_reuse (reuse: REUSE_* bits)."""
    args = (C.byref(desc), _p(dO), _p(q), _p(k), _p(v), _p(o_sparse), _p(lse), _p(q_idx), _p(q_cnt),
            int(idx_cap), _p(kv_ptr), _p(kv_qidx), _p(q_var), _p(kv_var), _p(gate), _p(dq), _p(dk), _p(dv))
    tail = (_p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if reuse:
        _check("vsa_bwd_reuse", lib().vsa_bwd_reuse(*args, int(reuse), *tail))
    else:
        _check("vsa_bwd", lib().vsa_bwd(*args, *tail))


def vsa_gate_grad(desc, dO, q, k, v, q_var, kv_var, dgate, workspace, stream=None):
    _check("vsa_gate_grad", lib().vsa_gate_grad(
        C.byref(desc), _p(dO), _p(q), _p(k), _p(v), _p(q_var), _p(kv_var), _p(dgate), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def vsa_check_inputs(desc, q_var, kv_var, q_idx, q_cnt, idx_cap, kv_ptr, kv_qidx, workspace, stream=None):
    """Opt-in validation of the device-resident arguments (synchronises).
    Returns (status, code): status 0 = all in range, 2 = a check failed
    (code names it), 9 = the status word already held another failure."""
    code = C.c_int32(0)
    st = lib().vsa_check_inputs(C.byref(desc), _p(q_var), _p(kv_var), _p(q_idx), _p(q_cnt), int(idx_cap),
                                _p(kv_ptr), _p(kv_qidx), _p(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream), C.byref(code))
    if st not in (0, 2, 9):
        raise VsaError("vsa_check_inputs", st)
    return int(st), int(code.value)


def vsa_head_slice(desc, groups, g):
    """Slice g of a problem's heads cut into `groups` (GQA groups whole):
    returns (slice descriptor, first query head, first key/value head)."""
    out, q0, kv0 = VsaDesc(), C.c_int32(0), C.c_int32(0)
    _check("vsa_head_slice", lib().vsa_head_slice(C.byref(desc), int(groups), int(g), C.byref(out), C.byref(q0),
                                                  C.byref(kv0)))
    return out, int(q0.value), int(kv0.value)


def vsa_device_status(workspace, stream=None) -> int:
    code = C.c_int32(0)
    lib().vsa_device_status(_p(workspace), _stream(stream), C.byref(code))
    return int(code.value)


def vsa_launch_count() -> int:
    return int(lib().vsa_launch_count())


class profile:
    """Context manager collecting per-kernel CUDA-event times (ms)."""

    def __enter__(self):
        L = lib()
        L.vsa_profile_reset()
        L.vsa_profile_enable(1)
        self.records = []
        return self

    def __exit__(self, *exc):
        L = lib()
        L.vsa_profile_enable(0)
        self.records = [(L.vsa_profile_name(i).decode(), float(L.vsa_profile_ms(i)))
                        for i in range(L.vsa_profile_count())]
        L.vsa_profile_reset()
        return False


# ----------------------------------------------------------------------- Plan

def describe(layout, dtype, B, Hq, Hkv, D, Sq, Skv, tile_q, tile_kv, nQ, nKV, cu_seqlens_q=None, cu_seqlens_kv=None,
             scale=0.0) -> VsaDesc:
    """A vsa_desc: layout "bhsd" | "bshd" | "tnd", dtype torch.bfloat16 |
    torch.float16, sizes as in include/vsa.h (TND offsets: int32 device
    tensors)."""
    return VsaDesc(LAYOUTS[layout], DTYPES[dtype], B, Hq, Hkv, D, Sq, Skv, tile_q, tile_kv, nQ, nKV,
                   _p(cu_seqlens_q), _p(cu_seqlens_kv), float(scale))


class Plan:
    """Descriptor, workspace and index buffers of one problem.

    layout: "bhsd" | "bshd" | "tnd"; sizes as in vsa_desc. For TND pass
    cu_seqlens_q / cu_seqlens_kv (int32 device tensors, [B+1]) and
    max_seqlen_q / max_seqlen_kv (host ints) instead of Sq / Skv per batch.

    With a gate, the plan's methods keep the tile means in its workspace
    between calls (vsa_fwd_reuse / vsa_bwd_reuse). It tracks what its own
    calls pooled and reuses means only for the same tensor objects whose
    torch version counter has not moved. Two things it cannot see must be
    followed by build_block_map before the next gated forward or backward:
    a module-level call that writes plan.workspace with other tensors, and
    a write to q, k or v that bypasses the version counter (through a raw
    pointer or .data).
    """

    def __init__(self, layout, dtype, B, Hq, Hkv, D, tile_q, tile_kv, nQ, nKV, Sq, Skv, idx_cap, gate=False,
                 cu_seqlens_q=None, cu_seqlens_kv=None, q_var=None, kv_var=None, scale=0.0, device="cuda"):
        self.layout, self.dtype = layout, dtype
        self.B, self.Hq, self.Hkv, self.D = B, Hq, Hkv, D
        self.tile_q, self.tile_kv, self.nQ, self.nKV = tile_q, tile_kv, nQ, nKV
        self.Sq, self.Skv, self.idx_cap, self.gate = Sq, Skv, idx_cap, gate
        self.cu_q, self.cu_kv = cu_seqlens_q, cu_seqlens_kv
        self.q_var, self.kv_var = q_var, kv_var
        self.device = torch.device(device)
        self.desc = describe(layout, dtype, B, Hq, Hkv, D, Sq, Skv, tile_q, tile_kv, nQ, nKV, cu_seqlens_q,
                             cu_seqlens_kv, scale)
        ws = vsa_workspace_size(self.desc, gate)
        if ws == 0:
            raise ValueError("invalid problem description")
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=self.device)
        i32 = dict(dtype=torch.int32, device=self.device)
        self.block_map = torch.zeros((B, Hq, nQ, nKV), dtype=torch.uint8, device=self.device)
        self.q_idx = torch.empty((B, Hq, nQ, idx_cap), **i32)
        self.q_cnt = torch.empty((B, Hq, nQ), **i32)
        self.kv_ptr = torch.empty((B, Hq, nKV + 1), **i32)
        self.kv_qidx = torch.empty((B, Hq, nQ * idx_cap), **i32)
        # Tile means the workspace holds: {"qk": key of (q, k), "v": key of v}
        # as left by the last call that pooled them. A later gated call
        # passes the matching reuse bit only for the same tensor objects,
        # unmodified since: torch bumps a tensor's version counter on every
        # in-place write, through any view of it.
        self._means = {}

    @staticmethod
    def _key(*ts):
        return tuple((weakref.ref(t), t._version) for t in ts)

    def _holds(self, which, *ts):
        key = self._means.get(which)
        return key is not None and len(key) == len(ts) and all(
            r() is t and ver == t._version for (r, ver), t in zip(key, ts))

    def _reuse(self, q, k, v):
        return (REUSE_QK_MEANS if self._holds("qk", q, k) else 0) | (REUSE_V_MEANS if self._holds("v", v) else 0)

    def _pooled(self, q=None, k=None, v=None):
        if q is not None:
            self._means["qk"] = self._key(q, k)
        if v is not None:
            self._means["v"] = self._key(v)

    def lse_shape(self):
        return (self.Hq, self.Sq) if self.layout == "tnd" else (self.B, self.Hq, self.Sq)

    def build_block_map(self, q, k, topk, need_bwd_index=True, stream=None):
        self._means.clear()  # a step starts here: only the means this call pools are kept
        vsa_build_block_map(self.desc, q, k, self.q_var, self.kv_var, topk, need_bwd_index, self.block_map,
                            self.q_idx, self.q_cnt, self.idx_cap, self.kv_ptr if need_bwd_index else None,
                            self.kv_qidx if need_bwd_index else None, self.workspace, stream)
        self._pooled(q, k)

    def mask_to_index(self, block_map, need_bwd_index=True, stream=None):
        self.block_map = block_map
        vsa_mask_to_index(self.desc, block_map, self.q_var, self.kv_var, need_bwd_index, self.q_idx, self.q_cnt,
                          self.idx_cap, self.kv_ptr if need_bwd_index else None,
                          self.kv_qidx if need_bwd_index else None, stream)

    def forward(self, q, k, v, gate=None, out=None, lse=None, o_sparse=None, stream=None):
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty(self.lse_shape(), dtype=torch.float32, device=q.device) if lse is None else lse
        if gate is not None and o_sparse is None:
            o_sparse = torch.empty_like(q)
        reuse = self._reuse(q, k, v) if gate is not None else 0
        if gate is not None:
            self._means.clear()
        vsa_fwd(self.desc, q, k, v, self.q_idx, self.q_cnt, self.idx_cap, self.q_var, self.kv_var, gate, out, lse,
                o_sparse, self.workspace, stream, reuse=reuse)
        if gate is not None:
            self._pooled(q, k, v)
        return out, lse, (o_sparse if o_sparse is not None else out)

    def backward(self, dO, q, k, v, o_sparse, lse, gate=None, dq=None, dk=None, dv=None, stream=None):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        reuse = self._reuse(q, k, v) if gate is not None else 0
        if gate is not None:
            self._means.clear()
        vsa_bwd(self.desc, dO, q, k, v, o_sparse, lse, self.q_idx, self.q_cnt, self.idx_cap, self.kv_ptr,
                self.kv_qidx, self.q_var, self.kv_var, gate, dq, dk, dv, self.workspace, stream, reuse=reuse)
        if gate is not None:
            self._pooled(q, k, v)
        return dq, dk, dv

    def mask_to_index_blocks(self, block_q, block_mask, need_bwd_index=True, stream=None):
        """Index from a query-block mask [B, Hq, nQb, nKV] (block_q rows per
        block); keeps the per-entry block bits for forward_blocks /
        backward_blocks."""
        self.block_q = block_q
        i32 = dict(dtype=torch.int32, device=self.device)
        self.q_sub = torch.empty_like(self.q_idx)
        self.kv_qsub = torch.empty_like(self.kv_qidx)
        _check("vsa_mask_to_index_blocks", lib().vsa_mask_to_index_blocks(
            C.byref(self.desc), int(block_q), int(block_mask.shape[2]), _p(block_mask), _p(self.q_var),
            _p(self.kv_var), int(bool(need_bwd_index)), _p(self.block_map), _p(self.q_idx), _p(self.q_cnt),
            _p(self.q_sub), int(self.idx_cap), _p(self.kv_ptr if need_bwd_index else None),
            _p(self.kv_qidx if need_bwd_index else None), _p(self.kv_qsub if need_bwd_index else None),
            _stream(stream)))

    def forward_blocks(self, q, k, v, out=None, lse=None, stream=None):
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty(self.lse_shape(), dtype=torch.float32, device=q.device) if lse is None else lse
        _check("vsa_fwd_blocks", lib().vsa_fwd_blocks(
            C.byref(self.desc), int(self.block_q), _p(q), _p(k), _p(v), _p(self.q_idx), _p(self.q_cnt),
            _p(self.q_sub), int(self.idx_cap), _p(self.q_var), _p(self.kv_var), _p(out), _p(lse),
            _p(self.workspace), self.workspace.numel() * self.workspace.element_size(), _stream(stream)))
        return out, lse

    def backward_blocks(self, dO, q, k, v, out, lse, dq=None, dk=None, dv=None, stream=None):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        _check("vsa_bwd_blocks", lib().vsa_bwd_blocks(
            C.byref(self.desc), int(self.block_q), _p(dO), _p(q), _p(k), _p(v), _p(out), _p(lse), _p(self.q_idx),
            _p(self.q_cnt), _p(self.q_sub), int(self.idx_cap), _p(self.kv_ptr), _p(self.kv_qidx), _p(self.kv_qsub),
            _p(self.q_var), _p(self.kv_var), _p(dq), _p(dk), _p(dv), _p(self.workspace),
            self.workspace.numel() * self.workspace.element_size(), _stream(stream)))
        return dq, dk, dv

    def gate_grad(self, dO, q, k, v, dgate=None, stream=None):
        """dgate = dO (*) c (the plan must have been made with gate=True)."""
        dgate = torch.empty_like(dO) if dgate is None else dgate
        self._means.clear()
        vsa_gate_grad(self.desc, dO, q, k, v, self.q_var, self.kv_var, dgate, self.workspace, stream)
        self._pooled(q, k, v)
        return dgate

    def check_inputs(self, with_index=True, with_bwd_index=True, stream=None):
        """vsa_check_inputs on this plan's tile fills / offsets and (when
        asked) its index buffers; returns (status, code)."""
        return vsa_check_inputs(self.desc, self.q_var, self.kv_var, self.q_idx if with_index else None,
                                self.q_cnt if with_index else None, self.idx_cap,
                                self.kv_ptr if with_bwd_index else None, self.kv_qidx if with_bwd_index else None,
                                self.workspace, stream)

    def device_status(self, stream=None) -> int:
        return vsa_device_status(self.workspace, stream)

    def _staging(self, groups, topk, gated):
        """Zeroed device staging memory for the host-buffer steps (kept and
        reused; its status words start at 0)."""
        need = int(lib().vsa_train_step_host_size(C.byref(self.desc), int(groups), int(topk), int(gated)))
        if need == 0:
            raise ValueError("invalid descriptor, groups or topk for the host-buffer step")
        buf = getattr(self, "_host_step_buf", None)
        if buf is None or buf.numel() < need:
            buf = self._host_step_buf = torch.zeros(need, dtype=torch.uint8, device=self.device)
        self._host_step_args = (int(groups), int(topk), int(gated))
        return buf, need

    def host_step_status(self, stream=None) -> int:
        """vsa_step_host_status for the last host-buffer step: synchronises
        and returns the first failure code of its staging slots (0 = none)."""
        groups, topk, gated = self._host_step_args
        code = C.c_int32(0)
        rc = lib().vsa_step_host_status(C.byref(self.desc), groups, topk, gated, _p(self._host_step_buf),
                                        _stream(stream), C.byref(code))
        if rc not in (0, 9):
            raise VsaError("vsa_step_host_status", rc)
        return int(code.value)

    def train_step_host(self, q, k, v, dO, topk, groups, gate=None, out=None, lse=None, dq=None, dk=None,
                        dv=None, stream=None):
        """vsa_train_step_host: one step (block map, forward, backward; with
        a gate also the gated compression branch) from host tensors (pin
        them for overlap), heads in `groups` slices whose copies overlap the
        kernels. Outputs are host tensors (allocated pinned when not given);
        `stream` is left ordered after the last copy back, so synchronise it
        before reading them. Returns (out, lse, dq, dk, dv); out / lse only
        if passed in."""
        buf, need = self._staging(groups, topk, gate is not None)
        dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True) if dq is None else dq
        dk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True) if dk is None else dk
        dv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True) if dv is None else dv
        for t in (q, k, v, dO, gate, out, lse, dq, dk, dv):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("vsa_train_step_host takes contiguous host tensors")
        _check("vsa_train_step_host", lib().vsa_train_step_host(
            C.byref(self.desc), int(groups), _p(q), _p(k), _p(v), _p(dO), _p(gate), _p(self.q_var), _p(self.kv_var),
            int(topk), _p(out), _p(lse), _p(dq), _p(dk), _p(dv), _p(buf), need, _stream(stream)))
        return out, lse, dq, dk, dv

    def fwd_step_host(self, q, k, v, topk, groups, gate=None, out=None, lse=None, stream=None):
        """vsa_fwd_step_host: block map and forward from host tensors, head
        slices overlapped with the copies; returns host (out, lse) (out
        allocated pinned when not given; lse only if passed in)."""
        buf, need = self._staging(groups, topk, gate is not None)
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True) if out is None else out
        for t in (q, k, v, gate, out, lse):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("vsa_fwd_step_host takes contiguous host tensors")
        _check("vsa_fwd_step_host", lib().vsa_fwd_step_host(
            C.byref(self.desc), int(groups), _p(q), _p(k), _p(v), _p(gate), _p(self.q_var), _p(self.kv_var),
            int(topk), _p(out), _p(lse), _p(buf), need, _stream(stream)))
        return out, lse


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


# ------------------------------------------------------------- 3D video tiling

def vsa_tile_3d_count(T, H, W, tile=(4, 8, 8)):
    return int(lib().vsa_tile_3d_count(T, H, W, *tile))


def tile_3d(latent: torch.Tensor, tile=(4, 8, 8), out=None, tile_var=None, stream=None):
    """latent [B, T, H, W, heads, D] (or [..., row] with any trailing shape)
    -> (tiled [B, nTiles * prod(tile), heads, D], tile_var [nTiles] int32)."""
    if not latent.is_contiguous():
        raise ValueError("tile_3d: latent must be contiguous")
    B, T, H, W = latent.shape[:4]
    rest = tuple(latent.shape[4:])
    n = vsa_tile_3d_count(T, H, W, tile)
    slots = n * tile[0] * tile[1] * tile[2]
    row_bytes = latent[0, 0, 0, 0].numel() * latent.element_size()
    if out is None:
        out = torch.empty((B, slots) + rest, dtype=latent.dtype, device=latent.device)
    if tile_var is None:
        tile_var = torch.empty(n, dtype=torch.int32, device=latent.device)
    _check("vsa_tile_3d", lib().vsa_tile_3d(B, T, H, W, row_bytes, *tile, _p(latent), _p(out),
                                            _p(tile_var), _stream(stream)))
    return out, tile_var


def untile_3d(tiled: torch.Tensor, grid, tile=(4, 8, 8), out=None, stream=None):
    """tiled [B, nTiles * prod(tile), ...] -> latent [B, T, H, W, ...] for grid = (T, H, W)."""
    if not tiled.is_contiguous():
        raise ValueError("untile_3d: tiled must be contiguous")
    T, H, W = grid
    B = tiled.shape[0]
    rest = tuple(tiled.shape[2:])
    row_bytes = tiled[0, 0].numel() * tiled.element_size()
    if out is None:
        out = torch.empty((B, T, H, W) + rest, dtype=tiled.dtype, device=tiled.device)
    _check("vsa_untile_3d", lib().vsa_untile_3d(B, T, H, W, row_bytes, *tile, _p(tiled), _p(out),
                                                _stream(stream)))
    return out


def check_wait_timeout(workspace: torch.Tensor, limit_ns: int = 50_000_000, stream=None) -> int:
    """Run the bounded-wait failure check; returns the device's completed flag
    (0: the wait timed out as it should)."""
    done = torch.full((1,), -1, dtype=torch.int32, device=workspace.device)
    _check("vsa_check_wait_timeout", lib().vsa_check_wait_timeout(_p(workspace), int(limit_ns), _p(done),
                                                                    _stream(stream)))
    return int(done.item())

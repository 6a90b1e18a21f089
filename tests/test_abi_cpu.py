"""The C-ABI library loads on a machine without a GPU, exports every entry
point include/vsa.h declares, and rejects bad arguments on the host before
any CUDA call."""
import ctypes as C
import os
import re

import pytest

from bwd_tile_mean_gb300 import build as libbuild
from bwd_tile_mean_gb300 import vsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return vsa.lib()


def declared():
    src = open(os.path.join(ROOT, "include", "vsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared()
    assert set(vsa.EXPORTS) == set(names), (names, vsa.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def desc(**kw):
    d = dict(layout=1, dtype=0, B=1, Hq=2, Hkv=2, D=128, Sq=768, Skv=1024, tile_q=256, tile_kv=256, nQ=3, nKV=4,
             cu_seqlens_q=None, cu_seqlens_kv=None, scale=0.0)
    d.update(kw)
    return vsa.VsaDesc(*[d[f] for f, _ in vsa.VsaDesc._fields_])


def test_workspace_size(L):
    assert vsa.vsa_workspace_size(desc(), False) > 0
    assert vsa.vsa_workspace_size(desc(), True) > vsa.vsa_workspace_size(desc(), False)
    assert vsa.vsa_workspace_size(desc(D=64), False) == 0
    assert vsa.vsa_workspace_size(desc(Hq=3, Hkv=2), False) == 0


# 16-byte aligned and never dereferenced: every call below fails host
# validation before any CUDA call, so this file is safe on a GPU machine too.
FAKE = C.c_void_p(1 << 20)


def fwd(L, d, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, q_idx=FAKE, q_cnt=FAKE, cap=2, q_var=FAKE, kv_var=FAKE, gate=None, out=FAKE,
             lse=FAKE, osp=None, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return L.vsa_fwd(C.byref(d), a["q"], a["k"], a["v"], a["q_idx"], a["q_cnt"], a["cap"], a["q_var"],
                     a["kv_var"], a["gate"], a["out"], a["lse"], a["osp"], a["ws"], a["wsb"], None)


def test_host_validation_errors(L):
    assert fwd(L, desc(D=64)) == 5                       # VSA_ERR_UNSUPPORTED
    assert fwd(L, desc(tile_q=64)) == 5
    assert fwd(L, desc(dtype=7)) == 3                    # VSA_ERR_DTYPE
    assert fwd(L, desc(layout=9)) == 4                   # VSA_ERR_LAYOUT
    assert fwd(L, desc(layout=2, Sq=100, Skv=200)) == 6  # TND without seqlens
    assert fwd(L, desc(Sq=700)) == 2                     # Sq != nQ * tile_q
    assert fwd(L, desc(), q=None) == 1                   # VSA_ERR_NULL
    assert fwd(L, desc(), kv_var=None) == 1
    assert fwd(L, desc(), gate=FAKE) == 1                # gated needs a separate o_sparse
    assert fwd(L, desc(), q=C.c_void_p((1 << 20) + 2)) == 4
    assert fwd(L, desc(), wsb=16) == 7                   # workspace too small
    assert fwd(L, desc(), ws=C.c_void_p((1 << 20) + 16)) == 7
    assert fwd(L, desc(), cap=9) == 2                    # idx_cap > nKV
    assert L.vsa_build_block_map(C.byref(desc()), FAKE, FAKE, FAKE, FAKE, 0, 0, FAKE, FAKE, FAKE, 2, None, None,
                                 FAKE, 1 << 30, None) == 2   # topk < 1
    assert L.vsa_build_block_map(C.byref(desc()), FAKE, FAKE, FAKE, FAKE, 2, 1, FAKE, FAKE, FAKE, 2, None, None,
                                 FAKE, 1 << 30, None) == 1   # bwd index needs kv_ptr / kv_qidx
    assert L.vsa_mask_to_index(C.byref(desc()), FAKE, None, FAKE, 0, FAKE, FAKE, 3, None, None, None) == 2
    assert L.vsa_status_string(5).decode().startswith("unsupported")
    big = desc(nKV=4000, Skv=4000 * 256)
    assert L.vsa_build_block_map(C.byref(big), FAKE, FAKE, FAKE, FAKE, 2, 0, FAKE, FAKE, FAKE, 2, None, None,
                                 FAKE, 1 << 40, None) == 5   # nKV past the selection kernel limit


def test_train_step_host_validation(L):
    d = desc(Hq=4, Hkv=2)
    size = lambda dd, g, k, gate=0: L.vsa_train_step_host_size(C.byref(dd), g, k, gate)
    one, two = size(d, 1, 2), size(d, 2, 2)
    assert one > two > 0                               # two slots of a half-size slice
    assert size(d, 2, 2, 1) > two                      # the gate, o_sparse and gated workspace
    assert size(d, 3, 2) == 0                          # groups must divide Hkv
    assert size(d, 0, 2) == 0
    assert size(d, 2, 0) == 0                          # topk < 1
    assert size(desc(D=64), 1, 2) == 0

    def call(groups=2, topk=2, q=FAKE, dq=FAKE, buf=C.c_void_p(1 << 20), nbytes=two, dd=d, gate=None):
        return L.vsa_train_step_host(C.byref(dd), groups, q, FAKE, FAKE, FAKE, gate, FAKE, FAKE, topk, None, None,
                                     dq, FAKE, FAKE, buf, nbytes, None)
    assert call(groups=3) == 2                         # VSA_ERR_SHAPE
    assert call(topk=0) == 2
    assert call(q=None) == 1                           # VSA_ERR_NULL
    assert call(dq=None) == 1
    assert call(buf=None) == 7                         # VSA_ERR_WORKSPACE
    assert call(buf=C.c_void_p((1 << 20) + 16)) == 7   # staging not 256-byte aligned
    assert call(nbytes=two - 1) == 7
    assert call(gate=FAKE) == 7                        # a gate needs the larger staging buffer
    assert call(dd=desc(Hq=4, Hkv=2, dtype=5)) == 3    # the descriptor is checked too (VSA_ERR_DTYPE)
    # the forward-only pipeline: out is required, the rest as above
    fwd = lambda out=FAKE, buf=C.c_void_p(1 << 20): L.vsa_fwd_step_host(C.byref(d), 2, FAKE, FAKE, FAKE, None, FAKE,
                                                                         FAKE, 2, out, None, buf, two, None)
    assert fwd(out=None) == 1
    assert fwd(buf=None) == 7
    # reading the staging slots' status words: arguments checked on the host
    code = C.c_int32(0)
    assert L.vsa_step_host_status(C.byref(d), 2, 2, 0, None, None, C.byref(code)) == 1
    assert L.vsa_step_host_status(C.byref(d), 3, 2, 0, FAKE, None, C.byref(code)) == 2


def test_static_block_map_checks_like_the_workspace_entry_point(L):
    # the allocation-free entry point runs the same host validation: every
    # descriptor or argument error gives the same status from both calls
    def both(d, topk=2, cap=2, need=0, kv_ptr=None):
        ws = L.vsa_build_block_map(C.byref(d), FAKE, FAKE, FAKE, FAKE, topk, need, FAKE, FAKE, FAKE, cap, kv_ptr,
                                   kv_ptr, FAKE, 1 << 30, None)
        st = L.vsa_build_block_map_static(C.byref(d), FAKE, FAKE, FAKE, FAKE, topk, need, FAKE, FAKE, FAKE, cap,
                                          kv_ptr, kv_ptr, None)
        return ws, st
    cases = [desc(scale=float("inf")), desc(scale=-1.0), desc(scale=float("nan")), desc(D=64), desc(dtype=3),
             desc(layout=2, Sq=-5, Skv=100, cu_seqlens_q=FAKE, cu_seqlens_kv=FAKE), desc(Sq=700),
             desc(layout=2, Sq=100, Skv=100), desc(Hq=3, Hkv=2), desc(nKV=4000, Skv=4000 * 256)]
    for d in cases:
        ws, st = both(d)
        assert ws == st != 0, (ws, st)
    assert both(desc(), topk=0) == (2, 2)
    assert both(desc(), cap=1) == (2, 2)
    assert both(desc(), need=1) == (1, 1)


def test_check_inputs_host_validation(L):
    code = C.c_int32(0)

    def call(d=None, q_var=FAKE, kv_var=FAKE, q_idx=None, q_cnt=None, cap=2, kv_ptr=None, kv_qidx=None, ws=FAKE,
             wsb=256, code_p=C.byref(code)):
        return L.vsa_check_inputs(C.byref(d or desc()), q_var, kv_var, q_idx, q_cnt, cap, kv_ptr, kv_qidx, ws, wsb,
                                  None, code_p)
    assert call(d=desc(D=64)) == 5
    assert call(kv_var=None) == 1                       # padded layouts need both fills
    assert call(code_p=None) == 1
    assert call(q_idx=FAKE) == 1                        # half of the Q-owned index
    assert call(kv_ptr=FAKE) == 1                       # half of the KV-owned index
    assert call(q_idx=FAKE, q_cnt=FAKE, cap=0) == 2
    assert call(q_idx=FAKE, q_cnt=FAKE, cap=5) == 2     # idx_cap > nKV
    assert call(ws=None) == 7
    assert call(ws=C.c_void_p((1 << 20) + 16)) == 7
    assert call(wsb=128) == 7


def test_head_slice_host_logic(L):
    d = desc(Hq=12, Hkv=3, Sq=768, Skv=1024)
    seen = []
    for g in range(3):
        s, q0, kv0 = vsa.vsa_head_slice(d, 3, g)
        assert (s.Hq, s.Hkv, q0, kv0) == (4, 1, 4 * g, g)
        assert (s.B, s.D, s.Sq, s.Skv, s.nQ, s.nKV, s.tile_q) == (d.B, d.D, d.Sq, d.Skv, d.nQ, d.nKV, d.tile_q)
        seen += list(range(q0, q0 + s.Hq))
    assert seen == list(range(12))
    for groups, g, code in ((2, 0, 2), (0, 0, 2), (3, 3, 2), (3, -1, 2)):   # Hkv % 2 != 0; groups < 1; g out of range
        with pytest.raises(vsa.VsaError) as e:
            vsa.vsa_head_slice(d, groups, g)
        assert e.value.code == code
    with pytest.raises(vsa.VsaError) as e:
        vsa.vsa_head_slice(desc(D=64), 1, 0)
    assert e.value.code == 5

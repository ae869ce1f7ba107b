"""The C ABI without a GPU: the library loads, exports every function include/moestep.h
declares, and its host-side validation returns the documented codes before any launch."""
import ctypes
import os
import re

import pytest

import moe_expert_step_gb300 as ms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(ms.library_path()):
        ms.build()
    return ms.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "moestep.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|long long|const char\s*\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert sorted(ms.EXPORTS) == names


def test_error_strings(L):
    for code in [ms.OK, ms.EINVAL, ms.EWORKSPACE, ms.EALIGN, ms.ECUDA, ms.EDEVICE, ms.EUNSUPPORTED, ms.ETIMEOUT,
                 ms.EDEVINPUT]:
        assert ms.error_string(code) != "unknown error"


CLOVER = ms.ModelDims(H=2048, E=256, k=8, I=512, Is=512, V=152064, P=32, dtype=ms.BF16)
TINY = ms.ModelDims(H=256, E=16, k=4, I=128, Is=128, V=1024, P=8, dtype=ms.F32)


def test_workspace_size(L):
    n1 = ms.workspace_size(CLOVER, 1)
    n16 = ms.workspace_size(CLOVER, 16)
    assert 0 < n1 < n16 < 1 << 31
    assert ms.workspace_size(TINY, 1) > 0


@pytest.mark.parametrize("bad,code", [
    (dict(k=0), ms.EINVAL), (dict(H=0), ms.EINVAL), (dict(dtype=7), ms.EINVAL),
    (dict(k=33, E=64), ms.EUNSUPPORTED), (dict(k=9, E=8), ms.EUNSUPPORTED), (dict(E=2048), ms.EUNSUPPORTED),
    (dict(H=2000), ms.EUNSUPPORTED), (dict(I=500), ms.EUNSUPPORTED), (dict(P=2048), ms.EUNSUPPORTED),
])
def test_bad_dims(L, bad, code):
    d = ms.ModelDims(**{**CLOVER.__dict__, **bad})
    n = ctypes.c_size_t(0)
    assert L.moestep_workspace_size(ctypes.byref(d.c()), 1, ctypes.byref(n)) == code


def test_bad_arguments_rejected_before_launch(L):
    d = CLOVER.c()
    fake = 1 << 20          # an aligned, never-dereferenced address
    ws_bytes = ms.workspace_size(CLOVER, 1)
    rc = L.moe_block_route(ctypes.byref(d), 32, fake, fake, fake, fake, fake, None, None, ws_bytes, None)
    assert rc == ms.EWORKSPACE
    rc = L.moe_block_route(ctypes.byref(d), 32, fake + 4, fake, fake, fake, fake, None, fake, ws_bytes, None)
    assert rc == ms.EALIGN
    rc = L.moe_block_route(ctypes.byref(d), 0, fake, fake, fake, fake, fake, None, fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.moe_block_route(ctypes.byref(d), 32, fake, fake, fake, fake, fake, None, fake, ws_bytes - 256, None)
    assert rc == ms.EWORKSPACE
    rc = L.moe_block_route(ctypes.byref(d), 32, fake, fake, fake, fake, fake, None, fake + 128, ws_bytes, None)
    assert rc == ms.EWORKSPACE
    for thr in [0.0, -0.5, 1.5, float("nan")]:
        rc = L.lm_head_commit(ctypes.byref(d), 1, fake, fake, 1.0, thr, fake, fake, fake, fake, fake, fake, None,
                              fake, ws_bytes, None)
        assert rc == ms.EINVAL
    lay = ms.Layer(fake, fake, fake, None, None)  # shared expert declared but missing
    rc = L.moe_block_ffn(ctypes.byref(d), 1, fake, ctypes.byref(lay), fake, fake, fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.coreset_select(ctypes.byref(d), 0, fake, fake, fake, fake, fake, fake, fake, fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.block_embed(ctypes.byref(d), 1, fake, fake, fake, fake, -1, fake, None)
    assert rc == ms.EINVAL
    rc = L.block_decode_step(ctypes.byref(d), 1, 2, None, fake, fake, 1.0, 0.95, fake, None, fake, fake, fake, fake,
                             fake, fake, None, fake, ws_bytes, None)
    assert rc == ms.EINVAL


def test_binding_raises_on_error(L):
    with pytest.raises(ms.MoeStepError) as ei:
        ms.workspace_size(ms.ModelDims(H=2048, E=256, k=0, I=512, Is=512, V=10), 1)
    assert ei.value.code == ms.EINVAL

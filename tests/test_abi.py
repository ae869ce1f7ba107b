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


CLOVER8 = ms.ModelDims(H=2048, E=256, k=8, I=512, Is=512, V=152064, P=32, dtype=ms.FP8)


def test_fp8_dims_and_workspace(L):
    """FP8 expert weights keep 2-byte activations: the same workspace as bf16."""
    assert ms.workspace_size(CLOVER8, 1) == ms.workspace_size(CLOVER, 1)
    assert ms.workspace_size(CLOVER8, 16) == ms.workspace_size(CLOVER, 16)
    for bad in (dict(H=2000), dict(I=500)):
        d = ms.ModelDims(**{**CLOVER8.__dict__, **bad})
        n = ctypes.c_size_t(0)
        assert L.moestep_workspace_size(ctypes.byref(d.c()), 1, ctypes.byref(n)) == ms.EUNSUPPORTED


def test_fp8_layer_checks_before_launch(L):
    """An FP8 layer needs its four row-scale tensors (three when there is no shared
    expert is not allowed: Is > 0 needs the shared scales) and K blocks of 128."""
    fake = 1 << 20
    d = CLOVER8.c()
    ws_bytes = ms.workspace_size(CLOVER8, 1)
    no_scales = ms.Layer(fake, fake, fake, fake, fake)
    rc = L.moe_block_ffn(ctypes.byref(d), 1, fake, ctypes.byref(no_scales), fake, fake, fake, ws_bytes, None)
    assert rc == ms.EINVAL
    no_shared_scales = ms.Layer(fake, fake, fake, fake, fake, fake, fake, None, None)
    rc = L.moe_block_ffn(ctypes.byref(d), 1, fake, ctypes.byref(no_shared_scales), fake, fake, fake, ws_bytes, None)
    assert rc == ms.EINVAL
    odd = ms.ModelDims(**{**CLOVER8.__dict__, "I": 192}).c()      # I % 64 == 0 but not % 128
    full = ms.Layer(fake, fake, fake, fake, fake, fake, fake, fake, fake)
    rc = L.moe_block_ffn(ctypes.byref(odd), 1, fake, ctypes.byref(full), fake, fake, fake,
                         ms.workspace_size(ms.ModelDims(**{**CLOVER8.__dict__, "I": 192}), 1), None)
    assert rc == ms.EUNSUPPORTED
    arr = (ms.Layer * 1)(no_scales)
    rc = L.block_decode_step(ctypes.byref(d), 1, 1, arr, fake, fake, 1.0, 0.95, fake, None, fake, fake, fake, fake,
                             fake, fake, None, fake, ws_bytes, None)
    assert rc == ms.EINVAL


def test_loop_and_fusion_arguments(L):
    fake = 1 << 20
    d = CLOVER.c()
    ws_bytes = ms.workspace_size(CLOVER, 1)
    arr = (ms.Layer * 1)(ms.Layer(fake, fake, fake, fake, fake))
    # negative round cap, missing rounds output, missing embedding
    rc = L.block_decode_loop(ctypes.byref(d), 1, 1, arr, fake, fake, fake, 5, fake, 1.0, 0.95, -1, fake, fake, fake,
                             fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.block_decode_loop(ctypes.byref(d), 1, 1, arr, fake, fake, fake, 5, fake, 1.0, 0.95, 8, fake, fake, None,
                             fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.block_decode_loop(ctypes.byref(d), 1, 1, arr, fake, None, fake, 5, fake, 1.0, 0.95, 8, fake, fake, fake,
                             fake, ws_bytes, None)
    assert rc == ms.EINVAL
    rc = L.block_decode_loop(ctypes.byref(d), 1, 1, arr, fake, fake, fake, 5, fake, 1.0, 0.95, 8, fake, fake, fake,
                             fake, ws_bytes - 256, None)
    assert rc == ms.EWORKSPACE
    prev = L.moestep_route_fusion()
    assert prev == ms.FUSED_COMBINE_HEAD                       # the default
    for mode in (ms.SEPARATE_HEAD, ms.FUSED_COMBINE_HEAD):
        assert L.moestep_set_route_fusion(mode) == ms.OK and L.moestep_route_fusion() == mode
    for bad in (1, 3, -1):
        assert L.moestep_set_route_fusion(bad) == ms.EINVAL
    assert L.moestep_route_fusion() == ms.FUSED_COMBINE_HEAD


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with the shared library missing, the first call raises."""
    from moe_expert_step_gb300 import _build
    monkeypatch.setattr(ms, "_LIB", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libmoestep_missing.so"))
    with pytest.raises(ms.MoeStepError):
        ms.lib()
    with pytest.raises(ms.MoeStepError):
        ms.set_route_fusion(ms.FUSED_COMBINE_HEAD)


def test_layer_struct_keeps_its_tensors_alive():
    """ms.layer() returns raw pointers for the C ABI; the struct also holds the tensors, so a
    caller that keeps only the struct (e.g. [ms.layer(**device_layer(...)) for ...]) cannot
    leave the library reading freed memory."""
    import gc
    import weakref

    import torch
    w = torch.zeros(8)
    ref = weakref.ref(w)
    lay = ms.layer(w, w, w)
    del w
    gc.collect()
    assert ref() is not None and lay.Wr == ref().data_ptr()
    del lay
    gc.collect()
    assert ref() is None

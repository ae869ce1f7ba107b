"""Block-diffusion MoE denoising step for GB300 (sm_103a): Python binding of libmoestep.

Every function here marshals torch tensors into the C ABI declared in
``include/moestep.h`` and calls it; all computation happens in the library's
CUDA kernels.  There is no Python or CPU fallback: if the library is not
built, importing works but every call raises ``MoeStepError``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import _build

BF16 = 0
F32 = 1
FP8 = 2

OK = 0
EINVAL = -1
EWORKSPACE = -2
EALIGN = -3
ECUDA = -4
EDEVICE = -5
EUNSUPPORTED = -6
ETIMEOUT = -7
EDEVINPUT = -8

PROF_KERNELS = ["route", "coreset", "gather", "expert_ffn", "expert_down", "combine", "lm_head", "commit", "other"]

EXPORTS = [
    "moestep_workspace_size", "moestep_workspace_init", "moe_block_route", "moe_route_from_logits", "coreset_select", "moe_block_ffn",
    "lm_head_commit", "lm_commit_from_logits", "block_embed", "block_decode_step", "block_decode_loop",
    "moestep_read_device_error",
    "moestep_error_string", "moestep_last_cuda_error", "moestep_prof_enable", "moestep_prof_read",
    "moestep_set_wait_timeout_ns", "moestep_set_route_fusion", "moestep_route_fusion", "moestep_launch_count",
    "moe_block_route_noalloc",
]


class MoeStepError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        # the library's text for the code, once it is loaded (loading it may be what failed)
        text = error_string(code) if _LIB is not None else "library not loaded"
        super().__init__(f"{what}: {text} ({code})")


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("H", "E", "k", "I", "Is", "V", "P", "dtype")]


class Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("Wr", "Wgu", "Wd", "Wsgu", "Wsd", "Sgu", "Sd", "Ssgu", "Ssd")]


class Trace(ctypes.Structure):
    _fields_ = [("n_sel", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("hidden", ctypes.c_void_p),
                ("sel", ctypes.c_void_p), ("x", ctypes.c_void_p), ("h", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libmoestep.so (raises MoeStepError if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise MoeStepError(EDEVICE, f"{_build.LIB} is not built (run __graft_entry__.build())")
        L = ctypes.CDLL(_build.LIB)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        D = ctypes.POINTER(Dims)
        sig = {
            "moestep_workspace_size": [D, i, ctypes.POINTER(sz)],
            "moestep_workspace_init": [vp, sz, vp],
            "moe_block_route": [D, i, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_route_from_logits": [D, i, vp, vp, vp, vp, vp, sz, vp],
            "moe_block_route_noalloc": [D, i, vp, vp, vp, vp, vp, vp, vp],
            "coreset_select": [D, i, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_block_ffn": [D, i, vp, ctypes.POINTER(Layer), vp, vp, vp, sz, vp],
            "lm_head_commit": [D, i, vp, vp, f, f, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "lm_commit_from_logits": [D, i, vp, f, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "block_embed": [D, i, vp, vp, vp, vp, i, vp, vp],
            "block_decode_step": [D, i, i, ctypes.POINTER(Layer), vp, vp, f, f, vp, vp, vp, vp, vp, vp, vp, vp,
                                  ctypes.POINTER(Trace), vp, sz, vp],
            "block_decode_loop": [D, i, i, ctypes.POINTER(Layer), vp, vp, vp, i, vp, f, f, i, vp, vp, vp, vp, sz, vp],
            "moestep_read_device_error": [vp, sz, vp, ctypes.POINTER(i)],
            "moestep_error_string": [i],
            "moestep_last_cuda_error": [],
            "moestep_prof_enable": [i],
            "moestep_prof_read": [i, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_double)],
            "moestep_set_wait_timeout_ns": [ctypes.c_ulonglong],
            "moestep_set_route_fusion": [ctypes.c_int],
            "moestep_route_fusion": [],
            "moestep_launch_count": [],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = {"moestep_error_string": ctypes.c_char_p,
                          "moestep_launch_count": ctypes.c_longlong}.get(name, ctypes.c_int)
        _LIB = L
    return _LIB


def error_string(code: int) -> str:
    try:
        return lib().moestep_error_string(code).decode()
    except MoeStepError:
        return "library not built"


def _check(rc: int, what: str) -> None:
    if rc != OK:
        if rc == ECUDA:
            what = f"{what} (cudaError {lib().moestep_last_cuda_error()})"
        raise MoeStepError(rc, what)


def _p(t):
    """Raw pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    return t.data_ptr()


def _s(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass(frozen=True)
class ModelDims:
    H: int
    E: int
    k: int
    I: int
    Is: int
    V: int
    P: int = 32
    dtype: int = BF16

    def c(self) -> Dims:
        return Dims(self.H, self.E, self.k, self.I, self.Is, self.V, self.P, self.dtype)


def layer(Wr, Wgu, Wd, Wsgu=None, Wsd=None, Sgu=None, Sd=None, Ssgu=None, Ssd=None) -> Layer:
    """Device pointers of one layer; the four row-scale tensors only with FP8 expert weights.
    The returned struct holds references to the tensors, so their memory stays allocated for
    as long as the struct is alive."""
    lay = Layer(_p(Wr), _p(Wgu), _p(Wd), _p(Wsgu), _p(Wsd), _p(Sgu), _p(Sd), _p(Ssgu), _p(Ssd))
    lay._tensors = (Wr, Wgu, Wd, Wsgu, Wsd, Sgu, Sd, Ssgu, Ssd)
    return lay


def workspace_size(d: ModelDims, R: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moestep_workspace_size(ctypes.byref(d.c()), R, ctypes.byref(n)), "moestep_workspace_size")
    return n.value


def workspace_init(ws, stream=None) -> None:
    _check(lib().moestep_workspace_init(_p(ws), ws.numel(), _s(stream)), "moestep_workspace_init")


def workspace(d: ModelDims, R: int, device="cuda", stream=None):
    """Allocate (through torch) and initialise a workspace for R requests."""
    import torch
    ws = torch.empty(workspace_size(d, R), dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def moe_block_route(d: ModelDims, x, Wr, idx, mass, gate, ws, logits=None, stream=None) -> None:
    _check(lib().moe_block_route(ctypes.byref(d.c()), x.shape[0], _p(x), _p(Wr), _p(idx), _p(mass), _p(gate),
                                 _p(logits), _p(ws), ws.numel(), _s(stream)), "moe_block_route")


def moe_block_route_noalloc(d: ModelDims, x, Wr, idx, mass, gate, logits=None, stream=None) -> None:
    """The router without a workspace (scratch in a fixed array inside the library); for callers
    that cannot allocate device memory.  Calls that overlap on the GPU race on that array."""
    _check(lib().moe_block_route_noalloc(ctypes.byref(d.c()), x.shape[0], _p(x), _p(Wr), _p(idx), _p(mass),
                                         _p(gate), _p(logits), _s(stream)), "moe_block_route_noalloc")


def moe_route_from_logits(d: ModelDims, logits, idx, mass, gate, ws, stream=None) -> None:
    _check(lib().moe_route_from_logits(ctypes.byref(d.c()), logits.shape[0], _p(logits), _p(idx), _p(mass),
                                       _p(gate), _p(ws), ws.numel(), _s(stream)), "moe_route_from_logits")


def coreset_select(d: ModelDims, R: int, top_p, idx, mass, n_sel, sel, survive, gate_rr, ws, stream=None) -> None:
    _check(lib().coreset_select(ctypes.byref(d.c()), R, _p(top_p), _p(idx), _p(mass), _p(n_sel), _p(sel),
                                _p(survive), _p(gate_rr), _p(ws), ws.numel(), _s(stream)), "coreset_select")


def moe_block_ffn(d: ModelDims, R: int, x, lay: Layer, gate_rr, out, ws, stream=None) -> None:
    _check(lib().moe_block_ffn(ctypes.byref(d.c()), R, _p(x), ctypes.byref(lay), _p(gate_rr), _p(out), _p(ws),
                               ws.numel(), _s(stream)), "moe_block_ffn")


def lm_head_commit(d: ModelDims, R: int, hidden, Wlm, threshold, tokens, masked, choice, conf, accept, n_committed,
                   ws, logit_scale=1.0, logits=None, stream=None) -> None:
    _check(lib().lm_head_commit(ctypes.byref(d.c()), R, _p(hidden), _p(Wlm), float(logit_scale), float(threshold),
                                _p(tokens), _p(masked), _p(choice), _p(conf), _p(accept), _p(n_committed),
                                _p(logits), _p(ws), ws.numel(), _s(stream)), "lm_head_commit")


def lm_commit_from_logits(d: ModelDims, R: int, logits, threshold, tokens, masked, choice, conf, accept, n_committed,
                          ws, stream=None) -> None:
    _check(lib().lm_commit_from_logits(ctypes.byref(d.c()), R, _p(logits), float(threshold), _p(tokens), _p(masked),
                                       _p(choice), _p(conf), _p(accept), _p(n_committed), _p(ws), ws.numel(),
                                       _s(stream)), "lm_commit_from_logits")


def block_embed(d: ModelDims, R: int, tokens, masked, emb, pos, mask_id: int, h, stream=None) -> None:
    _check(lib().block_embed(ctypes.byref(d.c()), R, _p(tokens), _p(masked), _p(emb), _p(pos), int(mask_id), _p(h),
                             _s(stream)), "block_embed")


def block_decode_step(d: ModelDims, R: int, layers, Wlm, top_p, threshold, h_in, tokens, masked, choice, conf,
                      accept, n_committed, ws, h_out=None, logit_scale=1.0, trace_n_sel=None, trace_idx=None,
                      trace_hidden=None, trace_sel=None, trace_x=None, trace_h=None, stream=None) -> None:
    """One denoising round; the optional trace_* tensors receive the per-layer records of
    moestep_trace (trace_x: each layer's MoE input, trace_h: the residual entering it)."""
    arr = (Layer * max(1, len(layers)))(*layers)
    tr = Trace(_p(trace_n_sel), _p(trace_idx), _p(trace_hidden), _p(trace_sel), _p(trace_x), _p(trace_h))
    _check(lib().block_decode_step(ctypes.byref(d.c()), R, len(layers), arr, _p(Wlm), _p(top_p), float(logit_scale),
                                   float(threshold), _p(h_in), _p(h_out), _p(tokens), _p(masked), _p(choice),
                                   _p(conf), _p(accept), _p(n_committed), ctypes.byref(tr), _p(ws), ws.numel(),
                                   _s(stream)), "block_decode_step")


def block_decode_loop(d: ModelDims, R: int, layers, Wlm, emb, pos, mask_id: int, top_p, threshold, tokens, masked,
                      rounds, ws, max_rounds=None, logit_scale=1.0, stream=None) -> None:
    """Every LowConfidence round of the block on the device (CUDA-graph while loop); rounds[0] = rounds run."""
    arr = (Layer * max(1, len(layers)))(*layers)
    mr = d.P if max_rounds is None else int(max_rounds)
    _check(lib().block_decode_loop(ctypes.byref(d.c()), R, len(layers), arr, _p(Wlm), _p(emb), _p(pos), int(mask_id),
                                   _p(top_p), float(logit_scale), float(threshold), mr, _p(tokens), _p(masked),
                                   _p(rounds), _p(ws), ws.numel(), _s(stream)), "block_decode_loop")


def read_device_error(ws, stream=None) -> int:
    w = ctypes.c_int(0)
    _check(lib().moestep_read_device_error(_p(ws), ws.numel(), _s(stream), ctypes.byref(w)),
           "moestep_read_device_error")
    return w.value


SEPARATE_HEAD, FUSED_COMBINE_HEAD = 0, 2


def set_route_fusion(mode) -> None:
    """What block_decode_step runs between expert launches: SEPARATE_HEAD (0) the combine /
    router / coreset / gather launches; FUSED_COMBINE_HEAD (2, the default) the combine inside
    the router's launch (bit-identical results)."""
    _check(lib().moestep_set_route_fusion(int(mode)), "moestep_set_route_fusion")


def route_fusion() -> int:
    """The mode last set by set_route_fusion."""
    return int(lib().moestep_route_fusion())


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().moestep_set_wait_timeout_ns(int(ns)), "moestep_set_wait_timeout_ns")


def prof_enable(kernels=None) -> None:
    """Time the named kernels (None = all, [] = off) with CUDA events on their stream."""
    names = PROF_KERNELS if kernels is None else list(kernels)
    mask = 0
    for n in names:
        mask |= 1 << PROF_KERNELS.index(n)
    _check(lib().moestep_prof_enable(mask), "moestep_prof_enable")


def launch_count() -> int:
    return int(lib().moestep_launch_count())


def prof_read() -> dict:
    """{kernel name: (launches, total ms)} of everything launched while profiling was on."""
    out = {}
    for kid, name in enumerate(PROF_KERNELS):
        n = ctypes.c_int(0)
        ms = ctypes.c_double(0.0)
        _check(lib().moestep_prof_read(kid, ctypes.byref(n), ctypes.byref(ms)), "moestep_prof_read")
        out[name] = (n.value, ms.value)
    return out


def build(quiet: bool = True) -> str:
    global _LIB
    _LIB = None
    return _build.build(quiet=quiet)

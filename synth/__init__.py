"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This module only *generates inputs*.  It holds none of the decoding method's
arithmetic (no routing, no softmax, no expert FFN, no commit rule): the CPU
oracle under ``oracle/`` and the CUDA library under ``moe_expert_step_gb300/``
each compute the method on their own; the only thing they share is the
tensors made here.

Generator (identical bits on three implementations: numpy below,
``synth_host.c`` with OpenMP, ``synth_dev.cu`` on the GPU):

* element ``i`` of a tensor with 64-bit key ``K`` is output ``i`` of a
  SplitMix64 stream seeded with ``K`` (Steele, Lea & Flood, OOPSLA 2014);
* "normal" values are Irwin-Hall(4) sums of the output's four 16-bit fields,
  centred, converted exactly to binary32 and scaled by one binary32 multiply;
  the scale makes the standard deviation the requested ``std`` (the
  distribution is bounded at about 3.46 std; it approximates N(0, std^2));
* bf16 tensors are that binary32 value rounded to nearest-even; on the host
  they are held as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Iterable

import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
# std of the sum of four independent uniforms on {0..65535}
_IH4_STD = math.sqrt((2.0 ** 32 - 1.0) / 3.0)
_IH4_MEAN = 131070

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_DIR = os.path.join(_HERE, "lib")
HOST_LIB = os.path.join(LIB_DIR, "libsynth_host.so")
DEV_LIB = os.path.join(LIB_DIR, "libsynth_dev.so")


# ----------------------------------------------------------------------------------------------
# keys
# ----------------------------------------------------------------------------------------------
def _mix(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def tensor_key(seed: int, *parts) -> int:
    """64-bit key of one synthetic tensor, from a seed and a path of ints/strings."""
    k = _mix((seed * GAMMA + GAMMA) & M64)
    for p in parts:
        if isinstance(p, str):
            for b in p.encode():
                k = _mix((k ^ b) + GAMMA)
            k = _mix(k ^ 0xFF)
        else:
            k = _mix((k ^ (int(p) & M64)) + GAMMA)
    return k


def scale_for_std(std: float) -> np.float32:
    """The binary32 multiplier that turns a centred Irwin-Hall(4) integer into std units."""
    return np.float32(std / _IH4_STD)


# ----------------------------------------------------------------------------------------------
# numpy reference implementation (slow; used to pin the C and CUDA copies)
# ----------------------------------------------------------------------------------------------
def np_u64(key: int, start: int, n: int) -> np.ndarray:
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def np_normal_f32(key: int, start: int, n: int, std: float) -> np.ndarray:
    u = np_u64(key, start, n)
    m = np.uint64(0xFFFF)
    s = ((u & m).astype(np.int64) + ((u >> np.uint64(16)) & m).astype(np.int64)
         + ((u >> np.uint64(32)) & m).astype(np.int64) + (u >> np.uint64(48)).astype(np.int64))
    c = (s - _IH4_MEAN).astype(np.float32)
    return c * scale_for_std(std)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round binary32 to bfloat16 (nearest-even), returned as uint16 bit patterns."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = b + np.uint32(0x7FFF) + lsb
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def np_normal_bf16(key: int, start: int, n: int, std: float) -> np.ndarray:
    return f32_to_bf16_bits(np_normal_f32(key, start, n, std))


def f32_to_e4m3(f: np.ndarray) -> np.ndarray:
    """binary32 -> FP8 E4M3 codes (bias 7, 3 mantissa bits, max 448, subnormals m * 2^-9),
    nearest-even, saturated to +-448 (the host and device copies' definition)."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    sign = ((b >> np.uint32(31)) << np.uint32(7)).astype(np.uint32)
    a = b & np.uint32(0x7FFFFFFF)
    with np.errstate(over="ignore"):
        r = (a + np.uint32(0x7FFFF) + ((a >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20)
        normal = np.minimum(r - np.uint32(120 << 3), np.uint32(0x7E))
    sub = np.rint(a.view(np.float32) * np.float32(512.0)).astype(np.uint32)
    code = np.where(a >= np.uint32(0x7F800000), np.uint32(0x7E),
                    np.where(a >= np.uint32(0x3C800000), normal, sub))
    return (code | sign).astype(np.uint8)


def e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    """Values of FP8 E4M3 codes (0x7F / 0xFF, the NaN codes, are never generated)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int32)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m.astype(np.float64) * 2.0 ** -9, (8 + m).astype(np.float64) * np.exp2(e - 10.0))
    return np.where(c & 0x80, -mag, mag).astype(np.float32)


def np_e4m3(key: int, start: int, n: int, std: float) -> np.ndarray:
    return f32_to_e4m3(np_normal_f32(key, start, n, std))


def np_row_scales(key: int, start: int, n: int) -> np.ndarray:
    """Per-row scales (16 + (u & 15)) * 2^-16, exact binary32."""
    return ((16 + (np_u64(key, start, n) & np.uint64(15)).astype(np.int64)).astype(np.float32)
            * np.float32(2.0 ** -16))


def np_uniform01(key: int, start: int, n: int) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each output."""
    return (np_u64(key, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


# ----------------------------------------------------------------------------------------------
# native copies
# ----------------------------------------------------------------------------------------------
def build(quiet: bool = True, device: bool = True) -> None:
    """Compile the host (gcc + OpenMP) and device (nvcc, sm_103a) generators in-tree."""
    os.makedirs(LIB_DIR, exist_ok=True)
    out = subprocess.DEVNULL if quiet else None
    jobs = [subprocess.Popen(
        ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
         os.path.join(_HERE, "synth_host.c"), "-o", HOST_LIB], stdout=out)]
    if device:
        jobs.append(subprocess.Popen(
            ["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-std=c++17",
             "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
             os.path.join(_HERE, "synth_dev.cu"), "-o", DEV_LIB], stdout=out))
    for j in jobs:
        if j.wait() != 0:
            raise RuntimeError(f"synth build failed: {j.args}")


_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build(device=False)
        lib = ctypes.CDLL(HOST_LIB)
        u64, i64, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float
        vp = ctypes.c_void_p
        lib.synth_host_u64.argtypes = [u64, u64, i64, vp]
        lib.synth_host_normal_f32.argtypes = [u64, u64, i64, f32, vp]
        lib.synth_host_normal_bf16.argtypes = [u64, u64, i64, f32, vp]
        lib.synth_host_bf16_to_f64.argtypes = [vp, i64, vp]
        lib.synth_host_e4m3.argtypes = [u64, u64, i64, f32, vp]
        lib.synth_host_row_scales.argtypes = [u64, u64, i64, vp]
        lib.synth_host_f32_to_e4m3.argtypes = [vp, i64, vp]
        lib.synth_host_threads.restype = ctypes.c_int
        _host = lib
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError("synth device library not built (run __graft_entry__.build())")
        lib = ctypes.CDLL(DEV_LIB)
        lib.synth_dev_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_float,
                                              ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_dev_fill_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                                           ctypes.c_void_p]
        lib.synth_dev_fill_row_scales.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                                                  ctypes.c_void_p]
        _dev = lib
    return _dev


def host_normal(key: int, start: int, n: int, std: float, dtype: str) -> np.ndarray:
    """Host copy: float32 array (dtype 'f32'), uint16 bf16 bits ('bf16') or uint8 FP8 E4M3 codes ('e4m3')."""
    lib = host_lib()
    if dtype == "e4m3":
        out = np.empty(n, np.uint8)
        lib.synth_host_e4m3(key, start, n, float(scale_for_std(std)), out.ctypes.data)
    elif dtype == "f32":
        out = np.empty(n, np.float32)
        lib.synth_host_normal_f32(key, start, n, float(scale_for_std(std)), out.ctypes.data)
    elif dtype == "bf16":
        out = np.empty(n, np.uint16)
        lib.synth_host_normal_bf16(key, start, n, float(scale_for_std(std)), out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out


def host_normal_f64(key: int, start: int, n: int, std: float, dtype: str) -> np.ndarray:
    """The same values as float64 (what an fp64 consumer is fed)."""
    a = host_normal(key, start, n, std, dtype)
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "e4m3":
        return e4m3_to_f32(a).astype(np.float64)
    out = np.empty(n, np.float64)
    host_lib().synth_host_bf16_to_f64(a.ctypes.data, n, out.ctypes.data)
    return out


def host_f32_to_e4m3(f: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(a.size, np.uint8)
    host_lib().synth_host_f32_to_e4m3(a.ctypes.data, a.size, out.ctypes.data)
    return out


def host_row_scales(key: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    host_lib().synth_host_row_scales(key, start, n, out.ctypes.data)
    return out


def host_u64(key: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    host_lib().synth_host_u64(key, start, n, out.ctypes.data)
    return out


def host_threads() -> int:
    return int(host_lib().synth_host_threads())


def dev_fill_normal(ptr: int, key: int, start: int, n: int, std: float, dtype: str, stream: int = 0) -> None:
    rc = dev_lib().synth_dev_fill_normal(key, start, n, float(scale_for_std(std)),
                                         {"bf16": 0, "f32": 1, "e4m3": 2}[dtype], ptr, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_normal failed: cudaError {rc}")


def dev_fill_row_scales(ptr: int, key: int, start: int, n: int, stream: int = 0) -> None:
    rc = dev_lib().synth_dev_fill_row_scales(key, start, n, ptr, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_row_scales failed: cudaError {rc}")


def dev_fill_u64(ptr: int, key: int, start: int, n: int, stream: int = 0) -> None:
    rc = dev_lib().synth_dev_fill_u64(key, start, n, ptr, stream)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_u64 failed: cudaError {rc}")


def as_f64(bits_or_f32: np.ndarray, dtype: str) -> np.ndarray:
    return (bf16_bits_to_f32(bits_or_f32) if dtype == "bf16" else bits_or_f32).astype(np.float64)


__all__: Iterable[str] = [
    "tensor_key", "scale_for_std", "np_u64", "np_normal_f32", "np_normal_bf16", "np_uniform01",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "build", "host_normal", "host_normal_f64", "host_u64",
    "host_threads", "dev_fill_normal", "dev_fill_u64", "as_f64", "f32_to_e4m3", "e4m3_to_f32", "np_e4m3",
    "np_row_scales", "host_row_scales", "dev_fill_row_scales",
]

"""Synthetic workloads: shapes, seeds and value distributions of every configuration.

Input generation only (no step of the method is computed here).  Weights use
the interleaved gate/up layout of the library: Wgu[e] is [I][2][H] with row
2i = gate row i and row 2i+1 = up row i.

Configurations (all seeds 0, tensors keyed by (seed, family, layer, name)):

* tiny_fp32      H=256, E=16, k=4, I=Is=128, V=1024, P=8, fp32 weights N(0, 0.05^2),
                 embeddings / positions / activations N(0, 1); coreset top_p in {1.0, 0.9, 0.5}.
* clover_layer   H=2048, E=256, k=8, I=Is=512, one shared expert, bf16 weights,
                 Wr and experts N(0, 0.02^2), block of 32 tokens, activations N(0, 1);
                 top_p in {1.0, 0.9, 0.7}.
* clover_stack40 40 layers shaped as clover_layer (64.4 GB of bf16 expert weights),
                 top_p 0.9, residual h0 ~ N(0, 1).
* lm_head        H=2048, V=152064, Wlm N(0, 0.02^2) bf16.
* batched        R in {1, 4, 16} requests x 32 tokens through clover_stack40.
* clover_layer_fp8, clover_stack40_fp8
                 the same shapes with FP8 E4M3 expert weights (routed and shared):
                 codes = e4m3(N(0, 64^2)), one fp32 scale per weight row
                 (16 + u) * 2^-16 with u uniform on 0..15, so a dequantised weight
                 has std ~0.023; router, LM head and activations as in the bf16
                 configs.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

from . import host_normal, host_normal_f64, host_row_scales, np_uniform01, tensor_key


@dataclass(frozen=True)
class Config:
    name: str
    family: str
    H: int
    E: int
    k: int
    I: int
    Is: int
    V: int
    P: int
    dtype: str          # "bf16" or "f32"
    w_std: float
    wr_std: float
    lm_std: float
    n_layers: int = 1
    top_ps: tuple = (1.0,)
    R: int = 1

    @property
    def T(self) -> int:
        return self.R * self.P

    @property
    def act_dtype(self) -> str:
        """Element type of the router, activations and LM head."""
        return "f32" if self.dtype == "f32" else "bf16"


TINY = Config("tiny_fp32", "tiny", 256, 16, 4, 128, 128, 1024, 8, "f32", 0.05, 0.05, 0.05, 1, (1.0, 0.9, 0.5))
LAYER = Config("clover_layer", "clover", 2048, 256, 8, 512, 512, 152064, 32, "bf16", 0.02, 0.02, 0.02, 1,
               (1.0, 0.9, 0.7))
STACK = replace(LAYER, name="clover_stack40", n_layers=40, top_ps=(0.9,))
LMHEAD = LAYER
LAYER_FP8 = replace(LAYER, name="clover_layer_fp8", dtype="fp8")
STACK_FP8 = replace(STACK, name="clover_stack40_fp8", dtype="fp8")
CONFIGS = {c.name: c for c in (TINY, LAYER, STACK, LAYER_FP8, STACK_FP8)}
FP8_CODE_STD = 64.0  # std of the E4M3 codes before the row scale
EXPERT_TENSORS = ("Wgu", "Wd", "Wsgu", "Wsd")
SCALE_OF = {"Wgu": "Sgu", "Wd": "Sd", "Wsgu": "Ssgu", "Wsd": "Ssd"}

SEED = 0


def key(cfg: Config, *parts, seed: int = SEED) -> int:
    return tensor_key(seed, cfg.family, *parts)


# ------------------------------------------------------------------------------------ shapes
def layer_shapes(cfg: Config) -> dict:
    H, E, I, Is = cfg.H, cfg.E, cfg.I, cfg.Is
    s = {"Wr": (E, H), "Wgu": (E, I, 2, H), "Wd": (E, H, I), "Wsgu": (Is, 2, H), "Wsd": (H, Is)}
    if cfg.dtype == "fp8":
        s.update({"Sgu": (E, 2 * I), "Sd": (E, H), "Ssgu": (2 * Is,), "Ssd": (H,)})
    return s


def layer_std(cfg: Config, name: str) -> float:
    if cfg.dtype == "fp8" and name in EXPERT_TENSORS:
        return FP8_CODE_STD
    return cfg.wr_std if name == "Wr" else cfg.w_std


def tensor_dtype(cfg: Config, name: str) -> str:
    """Storage of one layer tensor: 'bf16' / 'f32', 'e4m3' codes, or 'scale' (fp32 row scales)."""
    if cfg.dtype != "fp8":
        return cfg.dtype
    if name in EXPERT_TENSORS:
        return "e4m3"
    return "scale" if name.startswith("S") else "bf16"


# ------------------------------------------------------------------------------------ host copies
def host_tensor(cfg: Config, layer: int, name: str, start: int = 0, n: int | None = None) -> np.ndarray:
    """float64 values of (a slice of) one layer tensor, flattened; FP8 expert tensors are
    dequantised (code value times its row's scale)."""
    shape = layer_shapes(cfg)[name]
    total = int(np.prod(shape))
    n = total - start if n is None else n
    dt = tensor_dtype(cfg, name)
    if n == 0:
        return np.zeros(0, np.float64)
    if dt == "scale":
        return host_row_scales(key(cfg, layer, name), start, n).astype(np.float64)
    v = host_normal_f64(key(cfg, layer, name), start, n, layer_std(cfg, name), dt)
    if dt == "e4m3":
        row = shape[-1]                      # elements per weight row
        assert start % row == 0 and n % row == 0
        sc = host_tensor(cfg, layer, SCALE_OF[name], start // row, n // row)
        v = (v.reshape(-1, row) * sc[:, None]).reshape(-1)
    return v


class HostLayer:
    """float64 accessors of one layer's weights, regenerated on demand (nothing cached)."""

    def __init__(self, cfg: Config, layer: int):
        self.cfg, self.layer = cfg, layer
        self.Wr = host_tensor(cfg, layer, "Wr").reshape(cfg.E, cfg.H)

    def expert(self, e: int):
        c = self.cfg
        gu = host_tensor(c, self.layer, "Wgu", e * c.I * 2 * c.H, c.I * 2 * c.H).reshape(c.I, 2, c.H)
        wd = host_tensor(c, self.layer, "Wd", e * c.H * c.I, c.H * c.I).reshape(c.H, c.I)
        return gu[:, 0, :], gu[:, 1, :], wd

    def shared(self):
        c = self.cfg
        gu = host_tensor(c, self.layer, "Wsgu").reshape(c.Is, 2, c.H)
        return gu[:, 0, :], gu[:, 1, :], host_tensor(c, self.layer, "Wsd").reshape(c.H, c.Is)


def host_lm_head(cfg: Config, rows: slice | None = None) -> np.ndarray:
    """float64 LM-head weights [V][H] (or a row range)."""
    r0, r1 = (0, cfg.V) if rows is None else (rows.start, rows.stop)
    v = host_normal_f64(key(cfg, "Wlm"), r0 * cfg.H, (r1 - r0) * cfg.H, cfg.lm_std, cfg.act_dtype)
    return v.reshape(r1 - r0, cfg.H)


def host_activations(cfg: Config, name: str, rows: int, std: float = 1.0, dtype: str | None = None) -> np.ndarray:
    """[rows][H] activations (bf16 bits / float32 in the given dtype) as stored on the device."""
    dt = dtype or cfg.act_dtype
    return host_normal(key(cfg, name), 0, rows * cfg.H, std, dt).reshape(rows, cfg.H)


def host_h0(cfg: Config, R: int, tag: str = "h0", correlation: float = 0.0) -> np.ndarray:
    """fp32 residual-stream input of a block step, [R*P][H] ~ N(0, 1).  With correlation a > 0
    every token of request r is a*c_r + sqrt(1 - a^2)*n_t (c_r, n_t independent N(0, 1) rows),
    so the tokens of a block route alike (fewer distinct experts per block)."""
    n = host_normal(key(cfg, tag, R), 0, R * cfg.P * cfg.H, 1.0, "f32").reshape(R, cfg.P, cfg.H)
    if correlation <= 0.0:
        return n.reshape(R * cfg.P, cfg.H)
    c = host_normal(key(cfg, tag + "_common", R), 0, R * cfg.H, 1.0, "f32").reshape(R, 1, cfg.H)
    a = float(correlation)
    h = a * c.astype(np.float64) + np.sqrt(1.0 - a * a) * n.astype(np.float64)
    return h.astype(np.float32).reshape(R * cfg.P, cfg.H)


def tiny_tables(cfg: Config):
    """Embedding [V][H] and positional [P][H] tables (fp32 N(0, 1)) of the tiny round-loop model."""
    emb = host_normal(key(cfg, "emb"), 0, cfg.V * cfg.H, 1.0, "f32").reshape(cfg.V, cfg.H)
    pos = host_normal(key(cfg, "pos"), 0, cfg.P * cfg.H, 1.0, "f32").reshape(cfg.P, cfg.H)
    return emb, pos


def masked_subset(cfg: Config, R: int, p_masked: float = 0.75, tag: str = "masked") -> np.ndarray:
    """Seeded mask over R*P positions: each masked with probability p, at least one per request."""
    u = np_uniform01(key(cfg, tag, R), 0, R * cfg.P).reshape(R, cfg.P)
    m = u < p_masked
    for r in range(R):
        if not m[r].any():
            m[r, int(np.argmin(u[r]))] = True
    return m.reshape(-1)


# ------------------------------------------------------------------------------------ device copies
def device_layer(cfg: Config, layer: int, device="cuda"):
    """Fill one layer's weights directly in device memory (bit-identical to the host copies)."""
    import torch

    from . import dev_fill_normal, dev_fill_row_scales
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.uint8, "scale": torch.float32}
    out = {}
    stream = torch.cuda.current_stream(device).cuda_stream
    for name, shape in layer_shapes(cfg).items():
        dt = tensor_dtype(cfg, name)
        t = torch.empty(shape, dtype=tdt[dt], device=device)
        if dt == "scale":
            dev_fill_row_scales(t.data_ptr(), key(cfg, layer, name), 0, t.numel(), stream)
        else:
            dev_fill_normal(t.data_ptr(), key(cfg, layer, name), 0, t.numel(), layer_std(cfg, name), dt, stream)
        out[name] = t
    return out


def device_lm_head(cfg: Config, device="cuda"):
    import torch

    from . import dev_fill_normal
    tdt = torch.bfloat16 if cfg.act_dtype == "bf16" else torch.float32
    t = torch.empty((cfg.V, cfg.H), dtype=tdt, device=device)
    dev_fill_normal(t.data_ptr(), key(cfg, "Wlm"), 0, t.numel(), cfg.lm_std, cfg.act_dtype,
                    torch.cuda.current_stream(device).cuda_stream)
    return t


def to_device(a: np.ndarray, dtype: str, device="cuda"):
    """Host array (float32, or uint16 bf16 bits) -> device tensor of that dtype."""
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)

"""Seeded synthetic workloads for the materialised-probability SDPA forward.

This module only draws inputs; it holds none of the operation's arithmetic, so
both the CUDA path and the CPU oracle can be fed from it without sharing code.

Shapes follow the benchmark shapes of FlagOS-OP PR #10 "feat: add sdpa_math
operator" (performance tables: prefill 1k D64, prefill 2k D128, GQA 1k D128,
decode and tail100), with Q/K/V drawn i.i.d. N(0, 1) in float32 and then cast to
the working dtype.  Draw order is q, k, v, then the mask, from one CPU
``torch.Generator`` seeded per workload.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" | "f16" | "bf16"
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    is_causal: bool = False
    mask: Optional[str] = None   # None | "bool_keep0.8_rows5pct" | "additive"
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_dtype(self, dtype: str) -> "Workload":
        return dataclasses.replace(self, dtype=dtype, name=f"{self.name.rsplit('_', 1)[0]}_{dtype}")

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["scale"] = self.scale
        return d


# The six benchmark shapes (plus the small fp32 oracle check).
TINY = Workload("tiny_f32", "f32", 1, 2, 2, 64, 64, 64, False, None, seed=0)
PREFILL_1K_D64 = Workload("prefill1k_d64_f16", "f16", 2, 8, 8, 1024, 1024, 64, True, None, seed=1)
PREFILL_2K_D128 = Workload("prefill2k_d128_f16", "f16", 1, 16, 16, 2048, 2048, 128, True, None, seed=2)
PREFILL_2K_D128_BF16 = Workload("prefill2k_d128_bf16", "bf16", 1, 16, 16, 2048, 2048, 128, True, None, seed=2)
GQA_1K_D128 = Workload("gqa1k_d128_f16", "f16", 1, 32, 8, 1024, 1024, 128, False, None, seed=3)
DECODE = Workload("decode_skv1152_f16", "f16", 8, 32, 8, 1, 1152, 128, False, None, seed=4)
TAIL100 = Workload("tail100_mask_f16", "f16", 4, 8, 8, 100, 100, 64, False, "bool_keep0.8_rows5pct", seed=5)
# long-context decode (split-KV): the decode shape with a 32K-key cache
DECODE_32K = Workload("decode_skv32k_f16", "f16", 8, 32, 8, 1, 32768, 128, False, None, seed=6)

ALL = [TINY, PREFILL_1K_D64, PREFILL_2K_D128, PREFILL_2K_D128_BF16, GQA_1K_D128, DECODE, TAIL100, DECODE_32K]
BY_NAME = {w.name: w for w in ALL}


def draw_qkv(gen: torch.Generator, B, Hq, Hkv, Sq, Skv, D, dtype, Dv=None):
    """q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv], N(0,1) in fp32 then cast."""
    Dv = D if Dv is None else Dv
    q = torch.randn((B, Hq, Sq, D), generator=gen, dtype=torch.float32).to(dtype)
    k = torch.randn((B, Hkv, Skv, D), generator=gen, dtype=torch.float32).to(dtype)
    v = torch.randn((B, Hkv, Skv, Dv), generator=gen, dtype=torch.float32).to(dtype)
    return q, k, v


def draw_bool_mask(gen: torch.Generator, mb, mh, Sq, Skv, keep=0.8, dead_row_frac=0.05):
    """Bool mask [mb, mh, Sq, Skv]: True (keep) with probability ``keep``; then
    round(dead_row_frac * mb*mh*Sq) distinct query rows are set all-False."""
    m = torch.rand((mb, mh, Sq, Skv), generator=gen) < keep
    nrows = mb * mh * Sq
    ndead = int(round(dead_row_frac * nrows))
    if ndead > 0:
        dead = torch.randperm(nrows, generator=gen)[:ndead]
        flat = m.view(nrows, Skv)
        flat[dead] = False
    return m


def make_inputs(w: Workload):
    """(q, k, v, mask) on the CPU for a workload; mask is None without one."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    q, k, v = draw_qkv(gen, w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.torch_dtype)
    mask = None
    if w.mask == "bool_keep0.8_rows5pct":
        mask = draw_bool_mask(gen, w.B, 1, w.Sq, w.Skv, keep=0.8, dead_row_frac=0.05)
    elif w.mask == "additive":
        mask = (torch.randn((w.B, 1, w.Sq, w.Skv), generator=gen) * 2.0).to(w.torch_dtype)
    return q, k, v, mask


def make_custom(seed, B, Hq, Hkv, Sq, Skv, D, dtype="f16", mask=None, Dv=None,
                mask_b=None, mask_h=1, keep=0.8, dead_row_frac=0.05):
    """Inputs for an arbitrary shape (parity sweeps): same recipe as make_inputs."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    td = _DTYPES[dtype]
    q, k, v = draw_qkv(gen, B, Hq, Hkv, Sq, Skv, D, td, Dv)
    mb = B if mask_b is None else mask_b
    m = None
    if mask == "bool":
        m = draw_bool_mask(gen, mb, mask_h, Sq, Skv, keep=keep, dead_row_frac=dead_row_frac)
    elif mask == "additive":
        m = (torch.randn((mb, mask_h, Sq, Skv), generator=gen) * 2.0).to(td)
    return q, k, v, m

"""Seeded synthetic inputs for the DSA indexer decode path.

This module only draws random inputs and lays them out the way the kernels and
the oracle both read them.  It holds none of the method's arithmetic (no
logits, bins, selection or block maths), so the CUDA path and the oracle can
both be fed from it without sharing any computation.

Layouts (all C-contiguous numpy arrays):
  q            uint8  [R][H][D]     FP8 E4M3 codes, R = B * next_n
  kv           uint8  [P][ps][D]    FP8 E4M3 codes of the paged index-K cache
  kscale       f32    [P][ps]       per-token K scale
  weights      f32    [R][H]        per-row head weights
  page_table   int32  [B][maxp]     logical page -> physical page, -1 past the end
  context_lens int32  [B]           keys of the request's last token
  with key_format "mxfp4" also:
  k_codes      uint8  [P][ps][D/2]  E2M1 codes, two per byte (even dimension low)
  k_exp        uint8  [P][ps][D/32] UE8M0 exponents, one per 32 dimensions

The five named workloads follow the pages' shapes (DeepGEMM PR #94 "Producer
cost" cells; SGLang PR #38944 two-level path at bs=8, 128K with 128-slot
pages), with seed 20260000 + index.  Score distributions:
  normal   q, K ~ N(0,1) -> E4M3, kscale ~ U[0.5,1.5], w ~ N(0,1)/sqrt(H)
  mixed    as normal, head weights 16..31 scaled by 20 (fine, unit and saturating bins)
  fine     as normal, all head weights scaled by 0.25 (|logit| < 16)
  unit     as normal, all head weights scaled by 8   (mostly 16 <= |logit| < 223)
  intexact q, K in {-2..2} (mostly 0), kscale in {0.5, 1}, w in {+-0.5, +-1, +-2}:
           every partial sum is exactly representable, so any summation
           order gives the same float (bitwise comparisons are meaningful)
MXFP4 keys (key_format "mxfp4"): uniform E2M1 codes and block exponents
uniform in [125, 129] (scales of 1/4 .. 4, where block maxima of unit-variance
keys put them), drawn after every other input so the FP8 inputs of a seed stay
the same.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

H_DEFAULT = 32
D_DEFAULT = 128
SEED_BASE = 20260000


@dataclass
class Workload:
    name: str
    B: int
    next_n: int
    context_lens: list  # per request
    page_size: int
    dist: str = "normal"
    seed: int = SEED_BASE
    H: int = H_DEFAULT
    D: int = D_DEFAULT
    spare_pages: int = 3  # unreferenced pool pages, so a wrong gather shows
    extra: dict = field(default_factory=dict)
    key_format: str = "fp8"  # or "mxfp4": also draw E2M1 codes + UE8M0 exponents

    @property
    def R(self) -> int:
        return self.B * self.next_n


def _ctx_uniform(B, lo, hi, seed):
    g = torch.Generator().manual_seed(seed + 7)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def named(name: str) -> Workload:
    """The five workloads, by name c0..c4 (plus c3u: config 3, 'unit')."""
    if name == "c0":
        return Workload("c0: B=1 next_n=1 L=8192 ps=64", 1, 1, [8192], 64, "normal", SEED_BASE + 0)
    if name == "c1":
        return Workload("c1: B=8 next_n=1 L~U[16384,32768] ps=64", 8, 1,
                        _ctx_uniform(8, 16384, 32768, SEED_BASE + 1), 64, "normal", SEED_BASE + 1)
    if name == "c2":
        return Workload("c2: B=32 next_n=1 L=131072 ps=64 mixed", 32, 1, [131072] * 32, 64,
                        "mixed", SEED_BASE + 2)
    if name == "c3":
        return Workload("c3: B=16 next_n=4 L=65536(+j) ps=64 fine", 16, 4, [65536 + 3] * 16, 64,
                        "fine", SEED_BASE + 3)
    if name == "c3u":
        return Workload("c3: B=16 next_n=4 L=65536(+j) ps=64 unit", 16, 4, [65536 + 3] * 16, 64,
                        "unit", SEED_BASE + 3)
    if name == "c4":
        return Workload("c4: B=8 next_n=1 L=131072 ps=128 two-level", 8, 1, [131072] * 8, 128,
                        "normal", SEED_BASE + 4)
    raise KeyError(name)


def _randn_e4m3(shape, g, chunk=1 << 24) -> np.ndarray:
    """N(0,1) draws cast to FP8 E4M3 codes, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=g, dtype=torch.float32)
        out[s:e] = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out.reshape(shape)


def _small_int_e4m3(shape, g) -> np.ndarray:
    """Integers in {-2..2} (70% zero) as E4M3 codes; exact in E4M3."""
    n = int(np.prod(shape))
    u = torch.rand(n, generator=g)
    v = torch.zeros(n)
    v[u > 0.70] = 1.0
    v[u > 0.80] = -1.0
    v[u > 0.90] = 2.0
    v[u > 0.95] = -2.0
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(shape)


def generate(w: Workload) -> dict:
    """Draw every input of a workload.  Returns a dict of numpy arrays."""
    g = torch.Generator().manual_seed(w.seed)
    B, nn, ps, H, D = w.B, w.next_n, w.page_size, w.H, w.D
    ctx = np.asarray(w.context_lens, dtype=np.int32)
    assert ctx.shape == (B,)
    pages_per_req = [(int(c) + ps - 1) // ps if c > 0 else 0 for c in ctx]
    maxp = max(1, max(pages_per_req) if pages_per_req else 1)
    P = sum(pages_per_req) + w.spare_pages
    perm = torch.randperm(P, generator=g).numpy().astype(np.int32)
    page_table = np.full((B, maxp), -1, dtype=np.int32)
    off = 0
    for b, npg in enumerate(pages_per_req):
        page_table[b, :npg] = perm[off:off + npg]
        off += npg
    R = B * nn
    if w.dist == "intexact":
        q = _small_int_e4m3((R, H, D), g)
        kv = _small_int_e4m3((P, ps, D), g)
        ks_choice = torch.randint(0, 2, (P, ps), generator=g).numpy()
        kscale = np.where(ks_choice == 0, 0.5, 1.0).astype(np.float32)
        w_choice = torch.randint(0, 6, (R, H), generator=g).numpy()
        table = np.array([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], dtype=np.float32)
        weights = table[w_choice]
    else:
        q = _randn_e4m3((R, H, D), g)
        kv = _randn_e4m3((P, ps, D), g)
        kscale = (torch.rand((P, ps), generator=g) + 0.5).numpy().astype(np.float32)
        weights = (torch.randn((R, H), generator=g) / math.sqrt(H)).numpy().astype(np.float32)
        if w.dist == "mixed":
            weights[:, H // 2:] *= 20.0
        elif w.dist == "fine":
            weights *= 0.25
        elif w.dist == "unit":
            weights *= 8.0
        elif w.dist != "normal":
            raise ValueError(w.dist)
    out = dict(q=np.ascontiguousarray(q), kv=np.ascontiguousarray(kv),
               kscale=np.ascontiguousarray(kscale), weights=np.ascontiguousarray(weights),
               page_table=page_table, context_lens=ctx, next_n=nn, page_size=ps,
               num_pages=P, H=H, D=D)
    if w.key_format == "mxfp4":
        # uniform bytes are uniform pairs of E2M1 codes (drawn packed: a
        # 128K-token cache holds 2^29 codes)
        out["k_codes"] = torch.randint(0, 256, (P, ps, D // 2), generator=g,
                                       dtype=torch.uint8).numpy()
        out["k_exp"] = torch.randint(125, 130, (P, ps, D // 32), generator=g,
                                     dtype=torch.uint8).numpy()
    elif w.key_format != "fp8":
        raise ValueError(w.key_format)
    return out


def random_logits(R, n, seed, dist="normal", stride=None) -> np.ndarray:
    """Free-standing FP32 score rows for select-only tests."""
    g = torch.Generator().manual_seed(seed)
    stride = n if stride is None else stride
    x = torch.randn((R, stride), generator=g)
    if dist == "mixed":
        x[:, ::2] *= 20.0
    elif dist == "ties":
        x = torch.round(x * 4.0) / 4.0
    elif dist == "flat":
        x = torch.zeros((R, stride))
    return x.numpy().astype(np.float32)

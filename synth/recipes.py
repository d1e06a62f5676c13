"""Synthetic workloads: shapes, per-channel scales and seeds of every calibration stream.

A workload is a list of *units* (linear layers W of shape d_in x d_out, y = x W) and of
the calibration *sites* they read: an activation site feeds the input covariance X of
every unit that consumes it (q, k and v share one), a gradient site feeds the output
covariance G of exactly one unit.  Values are drawn by ``synth.philox`` and are a pure
function of (workload seed, block, site, element index), so any row or column range of
any stream can be regenerated independently on the host or on the device.

Distributions:
  * single 256x512 layer: activations N(0, 1/i) on channel i (1-based), gradients
    N(0, i^-1/2), weights N(0, 0.02^2), all float32;
  * transformer blocks: activations unit Gaussian with round(0.01 d) outlier channels at
    20x scale picked by a seeded Fisher-Yates shuffle, gradients N(0, 1e-6), weights
    N(0, 0.02^2), all rounded to bfloat16.

This module holds no arithmetic of the compression method.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

from . import philox

MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h = ((h ^ b) * 0x100000001B3) & MASK64
    return h


def tensor_seed(cfg_seed: int, block: int, kind: str, name: str) -> int:
    return splitmix64(splitmix64(splitmix64(cfg_seed) ^ block) ^ fnv1a64(kind + ":" + name))


@dataclass(frozen=True)
class Site:
    name: str
    d: int
    kind: str            # "act" (feeds X) or "grad" (feeds G)
    block: int = 0


@dataclass(frozen=True)
class Unit:
    name: str
    m: int               # d_in
    n: int               # d_out
    x_site: str
    g_site: str
    block: int = 0
    # A unit may be a block of a larger weight (an attention head): rows [row0, row0 + m)
    # and columns [col0, col0 + n) of the weight `w_name` (w_m x w_n); it then uses the
    # diagonal blocks [x_off, x_off + m) of its input factor and [g_off, g_off + n) of its
    # output factor.  An empty w_name means the unit is the whole weight `name`.
    w_name: str = ""
    w_m: int = 0
    w_n: int = 0
    row0: int = 0
    col0: int = 0
    x_off: int = 0
    g_off: int = 0

    @property
    def weight(self) -> str:
        return self.w_name or self.name

    @property
    def weight_shape(self):
        return (self.w_m, self.w_n) if self.w_name else (self.m, self.n)


@dataclass
class Workload:
    name: str
    n_tokens: int
    dtype: str                       # "f32" or "bf16": storage type of A, Gr and W
    units: List[Unit]
    sites: Dict[str, Site]
    seed: int
    lam: float = 1e-2
    rho: Optional[float] = None      # kept parameter fraction under global allocation
    fixed_rank: Optional[int] = None
    quant: str = "none"              # "none" or "int8_token" (quantisation-aware whitening)
    spectrum: str = "block"          # "powerlaw" (single layer) or "block"
    extra: dict = field(default_factory=dict)

    @property
    def budget(self) -> int:
        if self.rho is None:
            return -1
        return int(np.floor(self.rho * sum(u.m * u.n for u in self.units)))

    def site(self, name: str) -> Site:
        return self.sites[name]


# --------------------------------------------------------------------- scales
def site_std(wl: Workload, site: Site) -> np.ndarray:
    """Per-channel standard deviation (float32) of one calibration stream."""
    d = site.d
    idx = np.arange(1, d + 1, dtype=np.float32)
    if wl.spectrum == "powerlaw":
        if site.kind == "act":
            return (np.float32(1.0) / np.sqrt(idx)).astype(np.float32)
        return (np.float32(1.0) / np.sqrt(np.sqrt(idx))).astype(np.float32)
    if site.kind == "grad":
        return np.full(d, np.float32(1e-3), dtype=np.float32)
    std = np.ones(d, dtype=np.float32)
    std[outlier_channels(wl, site)] = np.float32(20.0)
    return std


def outlier_channels(wl: Workload, site: Site) -> np.ndarray:
    """round(0.01 d) channels from a seeded Fisher-Yates shuffle of 0..d-1."""
    d = site.d
    k = int(round(0.01 * d))
    seed = tensor_seed(wl.seed, site.block, "outlier", site.name)
    r = philox.uniform_u32(np.arange(d, dtype=np.uint64), seed).astype(np.int64)
    perm = np.arange(d, dtype=np.int64)
    for i in range(d - 1, 0, -1):
        j = int(r[i] % (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:k])


def weight_std(wl: Workload) -> np.float32:
    return np.float32(0.02)


def stream_seed(wl: Workload, site: Site) -> int:
    return tensor_seed(wl.seed, site.block, site.kind, site.name)


def weight_seed(wl: Workload, unit: Unit) -> int:
    return tensor_seed(wl.seed, unit.block, "weight", unit.weight)


# ----------------------------------------------------------------- generation
def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return philox.bf16_bits_to_f32(philox.f32_to_bf16_bits(x))
    return x


def gen_stream(wl: Workload, site: Site, t0: int, t1: int, cols=None) -> np.ndarray:
    """Rows t0..t1-1 (tokens) of a calibration stream as float32 values of its storage type.

    ``cols`` restricts to a subset of channels (e.g. to sample single covariance entries).
    """
    std = site_std(wl, site)
    cols = np.arange(site.d, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
    t = np.arange(t0, t1, dtype=np.uint64)[:, None]
    e = t * np.uint64(site.d) + cols.astype(np.uint64)[None, :]
    z = philox.standard_normal(e, stream_seed(wl, site))
    return _finish(z * std[cols][None, :], wl.dtype)


def gen_full_weight(wl: Workload, unit: Unit) -> np.ndarray:
    """The whole weight a unit belongs to (w_m x w_n, or m x n for a whole-matrix unit)."""
    wm, wn = unit.weight_shape
    i = np.arange(wm, dtype=np.uint64)[:, None]
    j = np.arange(wn, dtype=np.uint64)[None, :]
    z = philox.standard_normal(i * np.uint64(wn) + j, weight_seed(wl, unit))
    return _finish(z * weight_std(wl), wl.dtype)


def gen_weight(wl: Workload, unit: Unit) -> np.ndarray:
    """The unit's own block of its weight (m x n)."""
    w = gen_full_weight(wl, unit)
    return np.ascontiguousarray(w[unit.row0:unit.row0 + unit.m, unit.col0:unit.col0 + unit.n])


# ------------------------------------------------------------------ workloads
def single_linear(n_tokens: int = 2048, m: int = 256, n: int = 512, rank: int = 64,
                  seed: int = 1000) -> Workload:
    """W m x n float32, A N x m with channel variance 1/i, Gr N x n with variance i^-1/2."""
    sites = {"in": Site("in", m, "act"), "out": Site("out", n, "grad")}
    units = [Unit("layer", m, n, "in", "out")]
    return Workload("single_linear_%dx%d" % (m, n), n_tokens, "f32", units, sites, seed,
                    fixed_rank=rank, spectrum="powerlaw")


def decoder_blocks(n_blocks: int, d: int, ffn: int, kv: int, n_tokens: int, rho: float,
                   seed: int, name: str, quant: str = "none") -> Workload:
    """Transformer decoder blocks: q, k, v, o, gate, up, down, each W = d_in x d_out."""
    sites: Dict[str, Site] = {}
    units: List[Unit] = []
    for b in range(n_blocks):
        p = "b%d." % b if n_blocks > 1 else ""
        for s, dd in (("attn_in", d), ("o_in", d), ("mlp_in", d), ("down_in", ffn)):
            sites[p + s] = Site(p + s, dd, "act", b)
        shapes = (("q", d, d, "attn_in"), ("k", d, kv, "attn_in"), ("v", d, kv, "attn_in"),
                  ("o", d, d, "o_in"), ("gate", d, ffn, "mlp_in"), ("up", d, ffn, "mlp_in"),
                  ("down", ffn, d, "down_in"))
        for nm, m, n, xs in shapes:
            sites[p + nm + "_out"] = Site(p + nm + "_out", n, "grad", b)
            units.append(Unit(p + nm, m, n, p + xs, p + nm + "_out", b))
    return Workload(name, n_tokens, "bf16", units, sites, seed, rho=rho, quant=quant)


def llama7b_block(n_tokens: int = 131072) -> Workload:
    """One Llama-7B-shaped block, N = 131072 tokens, 50% of the block's parameters kept."""
    return decoder_blocks(1, 4096, 11008, 4096, n_tokens, 0.5, 1001, "llama7b_block")


def llama7b_model(n_tokens: int = 65536, n_blocks: int = 32) -> Workload:
    """32 Llama-7B-shaped blocks (224 matrices), 65536 tokens per layer, 40% kept globally."""
    return decoder_blocks(n_blocks, 4096, 11008, 4096, n_tokens, 0.4, 1002, "llama7b_model")


def llama70b_block(n_tokens: int = 262144) -> Workload:
    """One 70B-shaped block (GQA k/v 8192x1024), N = 262144 tokens, 30% kept."""
    return decoder_blocks(1, 8192, 28672, 1024, n_tokens, 0.3, 1004, "llama70b_block")


def _attn_heads(units: List[Unit], sites: Dict[str, Site], p: str, b: int, d: int, kv: int,
                head: int, x_attn: str, x_o: str) -> None:
    """Per-head units of one attention layer: q, k, v heads are column blocks (full input
    factor, the head's diagonal block of the output factor); o heads are row blocks (the
    head's diagonal block of the input factor, full output factor)."""
    for nm, n_out in (("q", d), ("k", kv), ("v", kv)):
        g = p + nm + "_out"
        sites[g] = Site(g, n_out, "grad", b)
        for h in range(n_out // head):
            units.append(Unit("%s%s.h%d" % (p, nm, h), d, head, x_attn, g, b, w_name=p + nm, w_m=d, w_n=n_out,
                              col0=h * head, g_off=h * head))
    g = p + "o_out"
    sites[g] = Site(g, d, "grad", b)
    for h in range(d // head):
        units.append(Unit("%so.h%d" % (p, h), head, d, x_o, g, b, w_name=p + "o", w_m=d, w_n=d,
                          row0=h * head, x_off=h * head))


def vlm(n_tokens: int = 147456, vit_blocks: int = 24, vit_d: int = 1024, vit_ffn: int = 4096,
        lm_blocks: int = 28, lm_d: int = 3584, lm_ffn: int = 18944, lm_kv: int = 512, head: int = 128,
        rho: float = 0.5, seed: int = 1003, quant: str = "int8_token", name: str = "vlm") -> Workload:
    """A ViT-L-shaped vision tower (whole-matrix units) and a decoder LM with 128-dim attention
    heads as units (GQA k/v), one global allocation pool, INT8 per-token fake-quantised
    activations (quantisation-aware whitening)."""
    sites: Dict[str, Site] = {}
    units: List[Unit] = []
    for b in range(vit_blocks):
        p = "vit.b%d." % b
        for s_, dd in (("attn_in", vit_d), ("o_in", vit_d), ("mlp_in", vit_d), ("fc2_in", vit_ffn)):
            sites[p + s_] = Site(p + s_, dd, "act", b)
        for nm, m, n, xs in (("q", vit_d, vit_d, "attn_in"), ("k", vit_d, vit_d, "attn_in"),
                             ("v", vit_d, vit_d, "attn_in"), ("o", vit_d, vit_d, "o_in"),
                             ("fc1", vit_d, vit_ffn, "mlp_in"), ("fc2", vit_ffn, vit_d, "fc2_in")):
            sites[p + nm + "_out"] = Site(p + nm + "_out", n, "grad", b)
            units.append(Unit(p + nm, m, n, p + xs, p + nm + "_out", b))
    for b in range(lm_blocks):
        bb = vit_blocks + b
        p = "lm.b%d." % b
        for s_, dd in (("attn_in", lm_d), ("o_in", lm_d), ("mlp_in", lm_d), ("down_in", lm_ffn)):
            sites[p + s_] = Site(p + s_, dd, "act", bb)
        _attn_heads(units, sites, p, bb, lm_d, lm_kv, head, p + "attn_in", p + "o_in")
        for nm, m, n, xs in (("gate", lm_d, lm_ffn, "mlp_in"), ("up", lm_d, lm_ffn, "mlp_in"),
                             ("down", lm_ffn, lm_d, "down_in")):
            sites[p + nm + "_out"] = Site(p + nm + "_out", n, "grad", bb)
            units.append(Unit(p + nm, m, n, p + xs, p + nm + "_out", bb))
    return Workload(name, n_tokens, "bf16", units, sites, seed, rho=rho, quant=quant)


def mini_vlm(n_tokens: int = 600, seed: int = 79) -> Workload:
    """A scaled-down VLM (one ViT block, one LM block with two q heads and one k/v head) with
    ragged FFN widths, for parity tests of the per-head path."""
    return vlm(n_tokens=n_tokens, vit_blocks=1, vit_d=192, vit_ffn=320, lm_blocks=1, lm_d=256, lm_ffn=328,
               lm_kv=128, head=128, rho=0.5, seed=seed, name="mini_vlm")


def mini_block(n_tokens: int = 1000, d: int = 320, ffn: int = 704, kv: int = 192,
               rho: float = 0.5, seed: int = 77, quant: str = "none") -> Workload:
    """A scaled-down block with ragged (non tile-multiple) shapes for parity tests."""
    return decoder_blocks(1, d, ffn, kv, n_tokens, rho, seed, "mini_block_%d_%d" % (d, ffn),
                          quant=quant)

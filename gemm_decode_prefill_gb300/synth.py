"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and packs them into the storage
formats; it holds none of the method's arithmetic.  Both sides of every
parity check (the CUDA path and the fp64 oracle) take their inputs from
here, so the bytes they see are identical.

Generator: numpy ``Generator(PCG64(seed))``; tensors are drawn in the order
they are listed in each function.  Distributions:

* q8_row codes: uniform integers in [-127, 127] (int8);
* row scales rs: uniform [1e-3, 1e-2] (float32);
* activations xs / x: N(0, 1) (float32);
* Q2 codes: uniform in {0..3}, packed four per byte, code k of a row in
  byte k/4 at bits 2(k%4) (a uniform random byte is four uniform codes);
* Q2 group scales d: uniform [0.005, 0.05] drawn as float32 and rounded to
  float16 (round to nearest even); the stored f16 bits are the truth.
* MoE: router logits N(0, 1), x N(0, 1), shared-gate weights N(0,1)/sqrt(hidden),
  then per expert (routed experts first, the shared expert last) gate codes +
  rs, up codes + rs, down codes + rs.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _codes8(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(-127, 128, size=shape, dtype=np.int8)


def _scales(g: np.random.Generator, n) -> np.ndarray:
    return g.uniform(1e-3, 1e-2, size=n).astype(np.float32)


def _normal(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(size=shape, dtype=np.float64).astype(np.float32)


def q8_inputs(rows: int, cols: int, seed: int):
    """q int8 [rows][cols], rs f32 [rows], xs f32 [cols]."""
    g = rng(seed)
    q = _codes8(g, (rows, cols))
    rs = _scales(g, rows)
    xs = _normal(g, cols)
    return q, rs, xs


def qmm_inputs(rows: int, cols: int, nb: int, seed: int):
    """q int8 [rows][cols], rs f32 [rows], xs f32 [nb][cols] (row-major)."""
    g = rng(seed)
    q = _codes8(g, (rows, cols))
    rs = _scales(g, rows)
    xs = _normal(g, (nb, cols))
    return q, rs, xs


def q2_inputs(rows: int, cols: int, group: int, seed: int):
    """codes uint8 [rows][cols/4], d f16 bits uint16 [rows][cols/group], x f32 [cols]."""
    assert cols % group == 0 and group in (64, 128)
    g = rng(seed)
    codes = g.integers(0, 256, size=(rows, cols // 4), dtype=np.uint8)
    d = g.uniform(0.005, 0.05, size=(rows, cols // group)).astype(np.float32)
    d_bits = d.astype(np.float16).view(np.uint16)
    x = _normal(g, cols)
    return codes, d_bits, x


@dataclass
class MoeInputs:
    logits: np.ndarray   # [n_exp] f32
    x: np.ndarray        # [hidden] f32
    sgw: np.ndarray      # [hidden] f32
    gq: np.ndarray       # [n_exp+1][inter][hidden] int8
    grs: np.ndarray      # [n_exp+1][inter] f32
    uq: np.ndarray
    urs: np.ndarray
    dq: np.ndarray       # [n_exp+1][hidden][inter] int8
    drs: np.ndarray      # [n_exp+1][hidden] f32


def moe_inputs(n_exp: int, hidden: int, inter: int, seed: int) -> MoeInputs:
    g = rng(seed)
    logits = _normal(g, n_exp)
    x = _normal(g, hidden)
    sgw = (g.standard_normal(size=hidden) / np.sqrt(hidden)).astype(np.float32)
    E = n_exp + 1
    gq = np.empty((E, inter, hidden), np.int8)
    uq = np.empty((E, inter, hidden), np.int8)
    dq = np.empty((E, hidden, inter), np.int8)
    grs = np.empty((E, inter), np.float32)
    urs = np.empty((E, inter), np.float32)
    drs = np.empty((E, hidden), np.float32)
    for e in range(E):
        gq[e] = _codes8(g, (inter, hidden)); grs[e] = _scales(g, inter)
        uq[e] = _codes8(g, (inter, hidden)); urs[e] = _scales(g, inter)
        dq[e] = _codes8(g, (hidden, inter)); drs[e] = _scales(g, hidden)
    return MoeInputs(logits, x, sgw, gq, grs, uq, urs, dq, drs)


def logit_bank(n_exp: int, count: int, seed: int) -> np.ndarray:
    """``count`` router-logit vectors N(0,1), vector i drawn from seed+1+i."""
    return np.stack([_normal(rng(seed + 1 + i), n_exp) for i in range(count)])


# The five workloads, with the sizes and seeds the pages' model shapes give.
WORKLOADS = {
    "q8_gemv_4096x4096": dict(kind="q8", rows=4096, cols=4096, seed=0),
    "q2_gemv_17408x5120": dict(kind="q2", rows=17408, cols=5120, groups=(64, 128), seed=1),
    "q8_lm_head_151936x4096": dict(kind="q8", rows=151936, cols=4096, seed=2),
    "q8_prefill_gemm_17408x5120_nb512": dict(kind="qmm", rows=17408, cols=5120, nb=512, seed=3),
    "moe_decode_h2048_e128_k8": dict(kind="moe", n_exp=128, hidden=2048, inter=768,
                                     top_k=8, renorm=True, seed=4),
}

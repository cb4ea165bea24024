"""Seeded synthetic inputs of the routed-expert block (shared by the tests, the bench and the oracle's callers).

This module only draws random numbers and lays them out; it holds none of the block's arithmetic (no routing, no
grouping, no quantisation, no expert product).  The router logits are made here because the router projection
X . W_r^T sits upstream of the block: it is computed in double on the host and rounded to fp32, and both the CUDA
library and the oracle receive the same fp32 logits.

Generator: numpy's PCG64 (``numpy.random.default_rng(seed)``), draws in a fixed order:
  x [T][H] fp32 N(0,1); W_r [E][H] N(0, sigma_r); (skewed chunk: a permutation of the expert ranks);
  gate/up codes bytes [E][2F][H/4] uniform (so every 2-bit code is uniform on {0..3}); gate/up scales
  U[0.005, 0.02] -> fp16 [E][2F][H/32]; down codes [E][H][F/4]; down scales [E][H][F/32].

Shared expert (``make_shared``): its own generator, PCG64 seeded with 1000 + the chunk's seed, so the routed inputs
above do not change: gate/up codes [2F][H/4], scales, down codes [H][F/4], scales (the distributions of the routed
experts), then the gate row w_sg [H] fp32 N(0, sigma_r).

Router weights (``make_router``): their own generator, PCG64 seeded with 2000 + the chunk's seed: W_r [E][H]
N(0, sigma_r), stored as bf16 (the top 16 bits of the fp32 value, rounded to nearest even).

Weight format (the library's and the oracle's): a 32-weight block has one fp16 scale d and 2-bit codes q,
w = d * (q - 2); codes are packed four to a byte, weight 4j+i in bits 2i..2i+1 of byte j; gate rows [0, F) and up
rows [F, 2F) of an expert's gate/up matrix; every expert of a matrix contiguous, expert-major.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Strength of the Zipf(s = 1.1) per-expert logit bias of the skewed chunk, bias_e = -ALPHA * 1.1 * ln(rank_e).
# Derived by tests/golden/calibrate_zipf.py (bisection, oracle routing) so that the 32 most-routed experts take half
# of the routed pairs; tests/golden/zipf_alpha.json holds the same figure and a test checks that the two agree.
ZIPF_S = 1.1
ZIPF_ALPHA = 0.4353008270263672


@dataclass(frozen=True)
class Config:
    name: str
    T: int
    H: int
    E: int
    K: int
    F: int
    router_sigma: float
    seed: int
    zipf: bool = False

    @property
    def n(self) -> int:
        return self.T * self.K


CONFIGS = {
    "tiny": Config("tiny", 64, 256, 16, 2, 128, 0.05, 0),
    "t1024": Config("t1024", 1024, 2560, 512, 10, 1024, 0.02, 1),
    "t8192": Config("t8192", 8192, 2560, 512, 10, 1024, 0.02, 2),
    "t32768": Config("t32768", 32768, 2560, 512, 10, 1024, 0.02, 3),
    "skew8192": Config("skew8192", 8192, 2560, 512, 10, 1024, 0.02, 4, zipf=True),
}


def _scales(rng, shape) -> np.ndarray:
    return rng.uniform(0.005, 0.02, size=shape).astype(np.float16).view(np.uint16)


def make_weights(rng, E: int, H: int, F: int) -> dict:
    return dict(
        wgu_c=rng.integers(0, 256, size=(E, 2 * F, H // 4), dtype=np.uint8),
        wgu_s=_scales(rng, (E, 2 * F, H // 32)),
        wd_c=rng.integers(0, 256, size=(E, H, F // 4), dtype=np.uint8),
        wd_s=_scales(rng, (E, H, F // 32)),
    )


def make_layer(cfg: Config, zipf_alpha: float | None = None, with_weights: bool = True) -> dict:
    """All inputs of one block call for `cfg`: logits, x and (optionally) the expert weights."""
    rng = np.random.default_rng(cfg.seed)
    T, H, E, K, F = cfg.T, cfg.H, cfg.E, cfg.K, cfg.F
    x = rng.standard_normal((T, H), dtype=np.float32)
    w_r = rng.standard_normal((E, H)) * cfg.router_sigma
    logits = x.astype(np.float64) @ w_r.T
    if cfg.zipf:
        rank = rng.permutation(E).astype(np.float64) + 1.0
        alpha = ZIPF_ALPHA if zipf_alpha is None else zipf_alpha
        logits = logits + (-alpha * ZIPF_S * np.log(rank))[None, :]
    out = dict(name=cfg.name, T=T, H=H, E=E, K=K, F=F, seed=cfg.seed, x=x,
               logits=np.ascontiguousarray(logits.astype(np.float32)))
    if with_weights:
        out.update(make_weights(rng, E, H, F))
    return out


def make_custom(T: int, H: int, E: int, K: int, F: int, seed: int, router_sigma: float = 0.05) -> dict:
    """A chunk of any shape with the tiny chunk's distributions (parity cases with ragged sizes)."""
    return make_layer(Config("custom", T, H, E, K, F, router_sigma, seed))


def make_gu(n: int, F: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """fp32 gate/up rows [n][2F] N(0, scale^2) (input of the SwiGLU + requant step on its own)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, 2 * F), dtype=np.float32) * np.float32(scale)).astype(np.float32)


def make_rows(rows: int, cols: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """fp32 rows N(0, scale^2) (input of the q8 step on its own)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(scale)).astype(np.float32)


def make_dm(n: int, H: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, H), dtype=np.float32)


def make_shared(cfg_or_inp, sigma: float | None = None) -> dict:
    """The shared expert of a chunk: one expert's weights in the routed experts' format and the scalar gate's row.
    Accepts a Config or an input dict made by make_layer / make_custom (uses its T, H, F and seed)."""
    if isinstance(cfg_or_inp, Config):
        H, F, seed, sig = cfg_or_inp.H, cfg_or_inp.F, cfg_or_inp.seed, cfg_or_inp.router_sigma
    else:
        H, F, seed, sig = cfg_or_inp["H"], cfg_or_inp["F"], cfg_or_inp["seed"], 0.02
    if sigma is not None:
        sig = sigma
    rng = np.random.default_rng(1000 + seed)
    w = make_weights(rng, 1, H, F)
    return dict(sgu_c=w["wgu_c"][0], sgu_s=w["wgu_s"][0], sd_c=w["wd_c"][0], sd_s=w["wd_s"][0],
                wsg=(rng.standard_normal(H) * sig).astype(np.float32))


def make_router(cfg_or_inp, sigma: float | None = None) -> np.ndarray:
    """Router weights bf16 bits (uint16) [E][H] for the fused router projection."""
    if isinstance(cfg_or_inp, Config):
        E, H, seed, sig = cfg_or_inp.E, cfg_or_inp.H, cfg_or_inp.seed, cfg_or_inp.router_sigma
    else:
        E, H, seed, sig = cfg_or_inp["E"], cfg_or_inp["H"], cfg_or_inp["seed"], 0.05
    if sigma is not None:
        sig = sigma
    rng = np.random.default_rng(2000 + seed)
    u = (rng.standard_normal((E, H)) * sig).astype(np.float32).view(np.uint32)
    # storage format: keep the top 16 bits, rounded to nearest, ties to even
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

"""Seeded synthetic inputs for the MoE expert-forward workloads.

This module is the only code shared by the CUDA path's tests/benchmark and the
oracle.  It draws random numbers and casts them to the storage types (BF16 via
torch's round-to-nearest-even cast, FP32 logits); it holds none of the
method's arithmetic (no routing, no scaling, no quantisation).

Workloads (shapes and value distributions of the pages' MoE expert layer,
Qwen3-30B-A3B-shaped: hidden 2048, 128 experts, top-8, expert FFN 768):

  tiny      T=256,   d=256,  E=8,   k=2, d_ff=128; x ~ N(0,1) with 2 outlier
            channels x20; W ~ N(0, 0.02); logits ~ N(0,1).
  small     T=4096,  d=1024, E=32,  k=4, d_ff=512; 1% outlier channels x30;
            logits ~ N(0,1) + per-expert bias ~ N(0, 1.5), with the two lowest
            biases set to -30 so that at least two experts receive no token.
  qwen16k   T=16384, d=2048, E=128, k=8, d_ff=768; 0.5% outlier channels x50;
            logits ~ N(0,1) + log p_pi(e), p_r proportional to r^-1.1 over a
            seeded permutation pi of the experts (Zipf(1.1) skew).
  qwen64k   T=65536 (16 x 4096), same shape, logits ~ N(0,1) (uniform routing).

Every array comes from its own PCG64 stream keyed by (seed, stream name,
index), so one expert's weights or one block of tokens can be regenerated
alone, bit for bit, without generating the rest.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

CONFIGS = {
    "tiny": dict(T=256, d=256, E=8, k=2, d_ff=128, outlier_frac=None,
                 outlier_channels=2, outlier_scale=20.0, logits="normal"),
    "small": dict(T=4096, d=1024, E=32, k=4, d_ff=512, outlier_frac=0.01,
                  outlier_channels=None, outlier_scale=30.0, logits="bias",
                  bias_std=1.5, n_forced_empty=2),
    "qwen16k": dict(T=16384, d=2048, E=128, k=8, d_ff=768, outlier_frac=0.005,
                    outlier_channels=None, outlier_scale=50.0, logits="zipf",
                    zipf_s=1.1),
    "qwen64k": dict(T=65536, d=2048, E=128, k=8, d_ff=768, outlier_frac=0.005,
                    outlier_channels=None, outlier_scale=50.0, logits="normal"),
}

WEIGHT_STD = 0.02
TOKEN_BLOCK = 1024  # tokens per independent x / logits stream


def _rng(seed: int, stream: str, index: int = 0) -> np.random.Generator:
    key = zlib.crc32(stream.encode())
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, key, index])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Cast float32 values to BF16 (round to nearest even, torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass
class Layer:
    name: str
    seed: int
    T: int
    d: int
    E: int
    k: int
    d_ff: int
    cfg: dict

    # ---- channel structure (shared by all tokens) ----
    def outlier_channels(self) -> np.ndarray:
        n = self.cfg["outlier_channels"]
        if n is None:
            n = max(1, int(round(self.cfg["outlier_frac"] * self.d)))
        return np.sort(_rng(self.seed, "outlier_channels").choice(self.d, n, replace=False))

    def expert_bias(self) -> np.ndarray:
        kind = self.cfg["logits"]
        E = self.E
        if kind == "normal":
            return np.zeros(E, np.float64)
        if kind == "bias":
            b = _rng(self.seed, "expert_bias").standard_normal(E) * self.cfg["bias_std"]
            low = np.argsort(b, kind="stable")[: self.cfg["n_forced_empty"]]
            b[low] = -30.0
            return b
        if kind == "zipf":
            r = np.arange(1, E + 1, dtype=np.float64)
            p = r ** (-self.cfg["zipf_s"])
            p /= p.sum()
            perm = _rng(self.seed, "zipf_perm").permutation(E)
            return np.log(p[perm])
        raise ValueError(kind)

    # ---- activations and router logits, by token block ----
    def x_block(self, b: int) -> np.ndarray:
        t0, t1 = b * TOKEN_BLOCK, min(self.T, (b + 1) * TOKEN_BLOCK)
        v = _rng(self.seed, "x", b).standard_normal((t1 - t0, self.d), dtype=np.float32)
        ch = self.outlier_channels()
        v[:, ch] *= np.float32(self.cfg["outlier_scale"])
        return to_bf16_bits(v)

    def logits_block(self, b: int) -> np.ndarray:
        t0, t1 = b * TOKEN_BLOCK, min(self.T, (b + 1) * TOKEN_BLOCK)
        v = _rng(self.seed, "logits", b).standard_normal((t1 - t0, self.E))
        v = v + self.expert_bias()[None, :]
        return v.astype(np.float32)

    def n_blocks(self) -> int:
        return (self.T + TOKEN_BLOCK - 1) // TOKEN_BLOCK

    def x(self) -> np.ndarray:
        return np.concatenate([self.x_block(b) for b in range(self.n_blocks())]) \
            if self.T else np.zeros((0, self.d), np.uint16)

    def logits(self) -> np.ndarray:
        return np.concatenate([self.logits_block(b) for b in range(self.n_blocks())]) \
            if self.T else np.zeros((0, self.E), np.float32)

    def x_rows(self, tokens) -> np.ndarray:
        out = np.zeros((len(tokens), self.d), np.uint16)
        cache = {}
        for i, t in enumerate(tokens):
            b = t // TOKEN_BLOCK
            if b not in cache:
                cache[b] = self.x_block(b)
            out[i] = cache[b][t - b * TOKEN_BLOCK]
        return out

    def logits_rows(self, tokens) -> np.ndarray:
        out = np.zeros((len(tokens), self.E), np.float32)
        cache = {}
        for i, t in enumerate(tokens):
            b = t // TOKEN_BLOCK
            if b not in cache:
                cache[b] = self.logits_block(b)
            out[i] = cache[b][t - b * TOKEN_BLOCK]
        return out

    # ---- expert weights, by expert ----
    def w1_expert(self, e: int) -> np.ndarray:
        """W1[e]: [2 d_ff][d] BF16 bits (gate rows then up rows)."""
        v = _rng(self.seed, "w1", e).standard_normal((2 * self.d_ff, self.d), dtype=np.float32)
        return to_bf16_bits(v * np.float32(WEIGHT_STD))

    def w2_expert(self, e: int) -> np.ndarray:
        """W2[e]: [d][d_ff] BF16 bits."""
        v = _rng(self.seed, "w2", e).standard_normal((self.d, self.d_ff), dtype=np.float32)
        return to_bf16_bits(v * np.float32(WEIGHT_STD))

    def w1(self) -> np.ndarray:
        return np.stack([self.w1_expert(e) for e in range(self.E)])

    def w2(self) -> np.ndarray:
        return np.stack([self.w2_expert(e) for e in range(self.E)])

    def grad_out(self) -> np.ndarray:
        """Output gradient ~ N(0, 1e-3) for the forward+backward workload."""
        v = _rng(self.seed, "dy").standard_normal((self.T, self.d), dtype=np.float32)
        return to_bf16_bits(v * np.float32(1e-3))


def layer(name: str, seed: int = 0, **override) -> Layer:
    cfg = dict(CONFIGS[name])
    cfg.update(override)
    return Layer(name=name, seed=seed, T=cfg["T"], d=cfg["d"], E=cfg["E"],
                 k=cfg["k"], d_ff=cfg["d_ff"], cfg=cfg)


def custom(T, d, E, k, d_ff, seed=0, logits="normal", outlier_channels=2,
           outlier_scale=20.0, **kw) -> Layer:
    cfg = dict(T=T, d=d, E=E, k=k, d_ff=d_ff, outlier_frac=None,
               outlier_channels=outlier_channels, outlier_scale=outlier_scale,
               logits=logits)
    cfg.update(kw)
    return Layer(name="custom", seed=seed, T=T, d=d, E=E, k=k, d_ff=d_ff, cfg=cfg)

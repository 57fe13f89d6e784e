"""Seeded synthetic inputs for the Gated DeltaNet layer.

This module only draws random tensors with fixed shapes, dtypes and
distributions; it holds none of the layer's arithmetic. The CUDA path and the
oracle checks both take their inputs from here.

Distributions (a normal's second parameter is its standard deviation):
  q, k, v, z, a, b ~ N(0, 1) in bf16;  A_log = log U[1, 16) fp32;
  dt_bias ~ U[-1, 1) fp32;  conv_w ~ N(0, 0.25) bf16;  norm_w = 1 + 0.1 N(0, 1) bf16;
  recurrent state ~ N(0, 0.1) fp32;  conv tail zero or N(0, 1) bf16.

Workloads (named by what they are):
  tiny_layer       B=1, T=64 (+8 decode, +8 verify tokens), 2 key / 4 value heads, d=32
  decode_batch     B=64 rows, T=1, 16 key / 32 value heads, d=128 (Qwen3.5-9B-like)
  prefill_long     B=1, T=8192 continued in 512-token calls, same head layout
  verify_paths     8 candidate paths x 8 draft tokens from one shared state
  varlen_rows      32 packed rows, lengths U{16..2048} padded to chunk buckets,
                   24 independent layers
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# Chunk buckets of the prefix-cache rows (statecache.py, squad-0.8b: CHUNKS).
CHUNK_BUCKETS = (16, 32, 64, 128, 192, 256, 320, 384, 448, 512, 640, 768, 1024, 1536, 2048)


@dataclass(frozen=True)
class Shape:
    nk: int
    nv: int
    dk: int
    dv: int
    conv_k: int = 4

    @property
    def kd(self) -> int:
        return self.nk * self.dk

    @property
    def vd(self) -> int:
        return self.nv * self.dv

    @property
    def C(self) -> int:
        return 2 * self.kd + self.vd

    @property
    def Kc(self) -> int:
        return self.conv_k - 1


TINY = Shape(nk=2, nv=4, dk=32, dv=32)
QWEN35_9B = Shape(nk=16, nv=32, dk=128, dv=128)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, std=1.0, dtype=torch.bfloat16, device="cpu"):
    return (torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * std).to(dtype)


def _uniform(shape, gen, lo, hi, device="cpu"):
    return torch.rand(shape, generator=gen, dtype=torch.float32, device=device) * (hi - lo) + lo


def weights(shape: Shape, gen, device="cpu") -> dict:
    return {
        "A_log": torch.log(_uniform((shape.nv,), gen, 1.0, 16.0, device)),
        "dt_bias": _uniform((shape.nv,), gen, -1.0, 1.0, device),
        "conv_w": _randn((shape.C, shape.conv_k), gen, 0.25, device=device),
        "norm_w": (1.0 + 0.1 * torch.randn((shape.dv,), generator=gen, device=device)).to(torch.bfloat16),
    }


def activations(shape: Shape, B: int, T: int, gen, device="cpu") -> dict:
    return {
        "q": _randn((B, T, shape.kd), gen, device=device),
        "k": _randn((B, T, shape.kd), gen, device=device),
        "v": _randn((B, T, shape.vd), gen, device=device),
        "z": _randn((B, T, shape.vd), gen, device=device),
        "a": _randn((B, T, shape.nv), gen, device=device),
        "b": _randn((B, T, shape.nv), gen, device=device),
    }


def states(shape: Shape, n: int, gen, tail: str = "randn", device="cpu") -> dict:
    if tail == "zeros":
        conv = torch.zeros((n, shape.Kc, shape.C), dtype=torch.bfloat16, device=device)
    else:
        conv = _randn((n, shape.Kc, shape.C), gen, device=device)
    S = (torch.randn((n, shape.nv, shape.dk, shape.dv), generator=gen, device=device) * 0.1)
    return {"conv_state": conv, "state": S.to(torch.float32)}


def tiny_layer(seed: int = 0) -> dict:
    """B=1, T=64, 2/4 heads, d=32, zero conv tail, all mask ones; 8 more tokens
    for decode steps and 8 for a verify call, drawn after the rest."""
    s = TINY
    g = _gen(seed)
    d = {"shape": s}
    d.update(weights(s, g))
    d["prefill"] = activations(s, 1, 64, g)
    d.update(states(s, 1, g, tail="zeros"))
    d["decode"] = activations(s, 1, 8, g)
    d["verify"] = activations(s, 1, 8, g)
    return d


def decode_batch(seed: int = 1, B: int = 64, shape: Shape = QWEN35_9B, device="cpu") -> dict:
    """One decode step of B rows (T=1) with random state and conv tail."""
    g = _gen(seed, device)
    d = {"shape": shape}
    d.update(weights(shape, g, device))
    d.update(activations(shape, B, 1, g, device))
    d.update(states(shape, B, g, tail="randn", device=device))
    return d


def prefill_long(seed: int = 2, T: int = 8192, shape: Shape = QWEN35_9B, device="cpu") -> dict:
    """One row of T tokens continuing a random saved state and conv tail."""
    g = _gen(seed, device)
    d = {"shape": shape}
    d.update(weights(shape, g, device))
    d.update(activations(shape, 1, T, g, device))
    d.update(states(shape, 1, g, tail="randn", device=device))
    return d


def verify_paths(seed: int = 3, P: int = 8, K: int = 8, shape: Shape = QWEN35_9B, device="cpu") -> dict:
    """P candidate paths of K draft tokens from one shared state, plus an
    accept length per path drawn uniformly from {0..K}."""
    g = _gen(seed, device)
    d = {"shape": shape}
    d.update(weights(shape, g, device))
    d.update(activations(shape, P, K, g, device))
    d.update(states(shape, 1, g, tail="randn", device=device))
    d["accept_len"] = torch.randint(0, K + 1, (P,), generator=g, device=device).to(torch.int32)
    return d


def bucket(n: int) -> int:
    """Smallest chunk bucket holding n tokens (statecache.py: _bucket)."""
    for b in CHUNK_BUCKETS:
        if n <= b:
            return b
    raise ValueError(f"row of {n} tokens exceeds the largest bucket")


def varlen_lengths(seed: int = 4, n_rows: int = 32, lo: int = 16, hi: int = 2048):
    """Real lengths U{lo..hi}, padded lengths (buckets) and packed offsets."""
    g = _gen(seed)
    real = torch.randint(lo, hi + 1, (n_rows,), generator=g).tolist()
    padded = [bucket(n) for n in real]
    cu = [0]
    for p in padded:
        cu.append(cu[-1] + p)
    return real, padded, cu


def varlen_layer(layer: int, seed: int = 4, n_rows: int = 32, shape: Shape = QWEN35_9B,
                 device="cpu") -> dict:
    """Layer `layer` of the varlen stack: its own weights, per-row states and
    packed activations [1, total, ...], with a 0/1 mask marking real tokens."""
    real, padded, cu = varlen_lengths(seed, n_rows)
    g = _gen(seed * 1_000_003 + 7919 * (layer + 1), device)
    d = {"shape": shape, "real": real, "padded": padded,
         "cu_seqlens": torch.tensor(cu, dtype=torch.int32)}
    d.update(weights(shape, g, device))
    d.update(activations(shape, 1, cu[-1], g, device))
    d.update(states(shape, n_rows, g, tail="randn", device=device))
    mask = torch.zeros((1, cu[-1]), dtype=torch.float32)
    for r in range(n_rows):
        mask[0, cu[r]:cu[r] + real[r]] = 1.0
    d["mask"] = mask.to(device)
    return d


def mxfp8(x: torch.Tensor, block: int = 32):
    """MXFP8 encoding of x [..., n] (n a multiple of `block`): e4m3 elements and
    one E8M0 scale byte per block of `block` consecutive values (OCP
    microscaling): the block's scale is 2^(floor(log2 amax) - 8), 8 being the
    largest e4m3 exponent, the elements are x / scale rounded to e4m3 and
    clamped to its largest finite value (448). Returns (elements as uint8,
    scales as uint8), both on x's device. An all-zero block gets scale 2^-127."""
    *lead, n = x.shape
    xb = x.float().reshape(*lead, n // block, block)
    amax = xb.abs().amax(-1, keepdim=True)
    e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 8,
                    torch.full_like(amax, -127.0)).clamp(-127, 127)
    q = (xb / torch.exp2(e)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(*lead, n), (e + 127).to(torch.uint8).reshape(*lead, n // block)

"""Seeded synthetic workloads (Q, K, V) shaped like the pages' Llama-3.1-8B layer.

This module only draws random numbers and plants a direction in them; it holds
none of the method's arithmetic.  Both the CUDA path (through tests and the
benchmark) and the fp64 oracle read the arrays it returns, so both sides see
bit-identical inputs.

Recipe (per seed):
  * Q, K, V are iid N(0, 1) float32 draws from numpy's Philox generator keyed
    by the seed, then rounded once to the working dtype (bf16: round to
    nearest even); the float32 arrays returned hold those rounded values
    exactly.
  * For every kv-head h a unit vector u_h (a normalised N(0, I_d) draw) is
    planted: alpha * u_h is added to every key of 128-token block 0 and of
    ``n_hot`` distinct blocks drawn uniformly from [1, Lk/128), and to every
    query of the q-heads that share kv-head h.  V is left unplanted.
  * The planted values are rounded to the dtype after the addition.

This gives the sink + needle + local-diagonal structure the long-context
configurations describe (nano-vllm pages: RULER/needle workloads on
Llama-3.1-8B, 32 q-heads, 8 kv-heads, head_dim 128).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BLOCK = 128


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    x = np.ascontiguousarray(x, np.float32)
    bits = x.view(np.uint32)
    # add 0x7FFF plus the lowest kept bit, then drop the low half; for finite
    # values the sum stays below 2**32 (the largest is 0xFF807FFF)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    rounded = (bits + (np.uint32(0x7FFF) + lsb)) & np.uint32(0xFFFF0000)
    out = rounded.view(np.float32)
    # NaN/Inf never occur in these draws; keep them out explicitly
    assert np.isfinite(out).all()
    return out


E4M3_MAX = 448.0


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities) to each value, ties to even, saturated to +-448;
    returned as float32 holding those values exactly.

    The spacing of e4m3 values is 2**(floor(log2|x|) - 3) from 2**-6 up and
    2**-9 below it (subnormals); every step here is exact in float64.
    """
    x = np.asarray(x, np.float32).astype(np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                       # a = m * 2**e with m in [0.5, 1)
    ex = np.maximum(np.where(a > 0, e - 1, -6), -6)
    q = np.ldexp(1.0, ex - 3)
    r = np.minimum(np.round(a / q) * q, E4M3_MAX)   # np.round: half to even
    return np.copysign(r, x).astype(np.float32)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """The e4m3 bit patterns (uint8) of e4m3-exact values."""
    x = np.asarray(x, np.float32)
    a = np.abs(x).astype(np.float64)
    _, e = np.frexp(a)
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e - 1 + 7, 0).astype(np.int64)
    mant = np.where(normal, np.round((a / np.ldexp(1.0, e - 1) - 1.0) * 8.0),
                    np.round(a / 2.0 ** -9)).astype(np.int64)
    sign = np.signbit(x).astype(np.int64)
    return ((sign << 7) | (exp_field << 3) | mant).astype(np.uint8)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-exact float32 values, as uint16."""
    x = np.ascontiguousarray(x, np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class Workload:
    q: np.ndarray        # [B, Lq, Hq, d] float32 (dtype-exact values)
    k: np.ndarray        # [B, Lk, Hkv, d]
    v: np.ndarray        # [B, Lk, Hkv, d]
    q_start_pos: int
    dtype: str           # "bf16" or "f32"
    hot_blocks: np.ndarray  # [B, Hkv, n_hot] planted key blocks (besides block 0)


def make_workload(seed: int, B: int, Hq: int, Hkv: int, d: int, Lk: int,
                  q_start_pos: int, alpha: float = 3.0, n_hot: int = 0,
                  dtype: str = "bf16", q_full: bool = False) -> Workload:
    """Draw one workload.

    Keys/values span positions [0, Lk).  Queries span [q_start_pos, Lk) unless
    ``q_full`` is set, in which case they span [0, Lk) (a whole sequence to
    be processed in chunks); q_start_pos is then recorded as 0.
    """
    assert dtype in ("bf16", "f32")
    assert Lk % BLOCK == 0 and q_start_pos % BLOCK == 0 and Hq % Hkv == 0
    rng = np.random.Generator(np.random.Philox(key=seed))
    q0 = 0 if q_full else q_start_pos
    Lq = Lk - q0
    q = rng.standard_normal((B, Lq, Hq, d), dtype=np.float32)
    k = rng.standard_normal((B, Lk, Hkv, d), dtype=np.float32)
    v = rng.standard_normal((B, Lk, Hkv, d), dtype=np.float32)
    nkb = Lk // BLOCK
    n_hot = min(n_hot, nkb - 1)
    hot = np.zeros((B, Hkv, n_hot), np.int64)
    G = Hq // Hkv
    if alpha != 0.0:
        for b in range(B):
            for h in range(Hkv):
                u = rng.standard_normal(d).astype(np.float64)
                u /= np.linalg.norm(u)
                du = (alpha * u).astype(np.float32)
                if n_hot > 0:
                    hot[b, h] = 1 + rng.choice(nkb - 1, size=n_hot, replace=False)
                for blk in [0] + sorted(hot[b, h].tolist()):
                    k[b, blk * BLOCK:(blk + 1) * BLOCK, h, :] += du
                q[b, :, h * G:(h + 1) * G, :] += du
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    return Workload(q, k, v, 0 if q_full else q_start_pos, dtype, hot)


def random_block_mask(seed: int, B: int, Hq: int, nqb: int, nkb: int,
                      q_start_pos: int, density: float) -> np.ndarray:
    """A seeded random causal block mask with the sink and diagonal set.

    Used to drive the block-sparse attention with masks that are independent
    of any estimator.  Entries above the diagonal are left 0.
    """
    rng = np.random.Generator(np.random.Philox(key=seed + 0x5EED))
    m = (rng.random((B, Hq, nqb, nkb)) < density).astype(np.uint8)
    cur = q_start_pos // BLOCK
    for qb in range(nqb):
        m[:, :, qb, cur + qb + 1:] = 0
        m[:, :, qb, cur + qb] = 1
        m[:, :, qb, 0] = 1
    return m


# The workloads the benchmark and the parity tests use, by name.
CONFIGS = {
    # tiny single chunk: 2 q-heads, 1 kv-head, d 64, 1024 tokens, fp32
    "tiny-1k-f32": dict(B=1, Hq=2, Hkv=1, d=64, Lk=1024, q_start_pos=0,
                        alpha=3.0, n_hot=0, dtype="f32", stride=8, threshold=0.9),
    # one 4096-token chunk at 28672 of a 32K context, Llama-3.1-8B heads
    "llama8b-32k-chunk4096": dict(B=1, Hq=32, Hkv=8, d=128, Lk=32768,
                                  q_start_pos=28672, alpha=3.0, n_hot=16,
                                  dtype="bf16", stride=8, threshold=0.95),
    # the last 4096-token chunk of a 128K context, stride 16
    "llama8b-128k-chunk4096": dict(B=1, Hq=32, Hkv=8, d=128, Lk=131072,
                                   q_start_pos=126976, alpha=3.0, n_hot=64,
                                   dtype="bf16", stride=16, threshold=0.9),
    # GPU-only prefill of a whole 32K sequence (q_start_pos 0, one chunk)
    "llama8b-32k-prefill": dict(B=1, Hq=32, Hkv=8, d=128, Lk=32768, q_start_pos=0,
                                alpha=3.0, n_hot=16, dtype="bf16", stride=8,
                                threshold=0.9),
    # a whole 64K sequence processed as 16 chunks of 4096
    "llama8b-64k-chunked": dict(B=1, Hq=32, Hkv=8, d=128, Lk=65536,
                                q_start_pos=0, alpha=3.0, n_hot=32,
                                dtype="bf16", stride=8, threshold=0.95,
                                chunk=4096),
}

# The sparse regime: the same shapes with a stronger planted direction
# (alpha 8: a planted key scores about alpha^2 / sqrt(d) = 5.7 above the rest
# in the estimator's softmax, so the planted blocks hold nearly all of a row's
# mass) and as many planted blocks as give the wanted share of the causal
# blocks.  The selection still comes from the estimator; the densities in the
# names are what the estimator selects on seed 0 (32K: 0.103, 0.312, 0.506;
# 128K: 0.061, 0.101, 0.291, 0.502 of the causal blocks).
for _rho, _n_hot in (("10", 24), ("30", 80), ("50", 134)):
    CONFIGS[f"llama8b-32k-rho{_rho}"] = dict(CONFIGS["llama8b-32k-chunk4096"], alpha=8.0,
                                              n_hot=_n_hot)
for _rho, _n_hot in (("06", 64), ("10", 110), ("30", 330), ("50", 575)):
    CONFIGS[f"llama8b-128k-rho{_rho}"] = dict(CONFIGS["llama8b-128k-chunk4096"], alpha=8.0,
                                               n_hot=_n_hot)
SPARSE_CONFIGS = tuple(n for n in CONFIGS if "-rho" in n)

"""Seeded synthetic inputs for the fused linear cross entropy (FLCE) workloads.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds NO arithmetic of the method itself: it only draws
numbers.  Every tensor is produced by a counter-based generator so the same
bytes come out on any machine and any numpy version:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; constants as in Vigna's public reference code)
  maps a 64-bit counter to a 64-bit output.  Stream ``k`` of seed ``s`` uses
  the counter sequence ``key(s, k) + i``.
* Uniforms on (0, 1) use the top 53 bits: ``((x >> 11) + 0.5) * 2**-53``.
* Normals use the Box-Muller transform on pairs of uniforms.
* bf16 values are produced by rounding to float32 (round-to-nearest-even,
  numpy's cast) and then to bfloat16 (round-to-nearest-even on the bit
  pattern).  They are stored as ``uint16`` bit patterns; ``bf16_to_float32``
  widens them exactly.
* Ignored positions: exactly ``floor(p * N)`` positions, chosen by a seeded
  partial Fisher-Yates shuffle, so the count of valid targets is fixed.
* Zipf(s) targets: P(id = k - 1) proportional to k**-s for k = 1..V, drawn by
  inverse CDF over the cumulative table.

The workload shapes follow the lm_head shapes the pages measure on (Llama
family hidden sizes and vocabularies, the tensor-parallel shard shape of the
DeepSpeed memory profile, and the 256k-vocabulary logits example of the
torchtune blog post).  No dataset is read; these inputs stand in for the
datasets those pages train on.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Optional

import numpy as np

_GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per vectorised block (bounds temporary memory)

IGNORE_INDEX = -100


def _mix_inplace(z: np.ndarray, tmp: np.ndarray) -> None:
    """SplitMix64 output function, in place on a uint64 array (wrap-around)."""
    np.right_shift(z, np.uint64(30), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _MIX1, out=z)
    np.right_shift(z, np.uint64(27), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _MIX2, out=z)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)


def stream_key(seed: int, stream: int) -> np.uint64:
    """64-bit starting key of stream ``stream`` of ``seed``."""
    z = np.array([(seed * 0x100000001 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    np.multiply(z, _GOLDEN_GAMMA, out=z)
    np.add(z, _GOLDEN_GAMMA, out=z)
    _mix_inplace(z, np.empty_like(z))
    return z[0]


def _splitmix_into(z: np.ndarray, tmp: np.ndarray, key: np.uint64, start: int) -> None:
    """z[i] = output number ``start + i`` of the stream with starting key ``key``."""
    z[:] = np.arange(start + 1, start + 1 + z.size, dtype=np.uint64)
    np.multiply(z, _GOLDEN_GAMMA, out=z)
    np.add(z, key, out=z)
    _mix_inplace(z, tmp)


def splitmix64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the given stream (uint64)."""
    z = np.empty(count, dtype=np.uint64)
    _splitmix_into(z, np.empty_like(z), stream_key(seed, stream), start)
    return z


def _to_unit(x: np.ndarray, out: np.ndarray) -> np.ndarray:
    """Top 53 bits of uint64 draws -> doubles on the open interval (0, 1)."""
    np.right_shift(x, np.uint64(11), out=x)
    out[:] = x
    np.add(out, 0.5, out=out)
    np.multiply(out, 2.0 ** -53, out=out)
    return out


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles on the open interval (0, 1)."""
    x = splitmix64(seed, stream, start, count)
    return _to_unit(x, np.empty(count, dtype=np.float64))


def _normals_pairs(key: np.uint64, p0: int, npairs: int) -> np.ndarray:
    """2*npairs standard normals from Box-Muller pairs p0 .. p0+npairs-1.

    Pair p uses draws 2p (radius) and 2p+1 (angle); its two outputs are
    r*cos(theta) and r*sin(theta), in that order.
    """
    z = np.empty(2 * npairs, dtype=np.uint64)
    _splitmix_into(z, np.empty_like(z), key, 2 * p0)
    u = _to_unit(z, np.empty(2 * npairs, dtype=np.float64))
    r = u[0::2].copy()
    th = u[1::2].copy()
    np.log(r, out=r)
    np.multiply(r, -2.0, out=r)
    np.sqrt(r, out=r)
    np.multiply(th, 2.0 * np.pi, out=th)
    out = u  # reuse
    np.cos(th, out=out[0::2])
    np.sin(th, out=out[1::2])
    np.multiply(out[0::2], r, out=out[0::2])
    np.multiply(out[1::2], r, out=out[1::2])
    return out


def _normals_block(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of a stream."""
    p0 = start // 2
    p1 = (start + count + 1) // 2
    out = _normals_pairs(stream_key(seed, stream), p0, p1 - p0)
    off = start - 2 * p0
    return out[off:off + count]


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    t = np.right_shift(b, np.uint32(16))
    np.bitwise_and(t, np.uint32(1), out=t)
    np.add(t, np.uint32(0x7FFF), out=t)
    np.add(b, t, out=b)
    np.right_shift(b, np.uint32(16), out=b)
    return b.astype(np.uint16)


def bf16_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _parallel_blocks(n: int, fn) -> None:
    """Run fn(start, end) over blocks of _CHUNK elements on a thread pool."""
    blocks = [(s, min(n, s + _CHUNK)) for s in range(0, n, _CHUNK)]
    if len(blocks) <= 1:
        for s, e in blocks:
            fn(s, e)
        return
    workers = max(1, min(len(blocks), len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        for f in [ex.submit(fn, s, e) for s, e in blocks]:
            f.result()


def normal_bf16(seed: int, stream: int, shape, std: float) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) draws (float64 draw -> f32 -> bf16)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def work(s, e):
        x = _normals_block(seed, stream, s, e - s)
        np.multiply(x, std, out=x)
        out[s:e] = float32_to_bf16_bits(x.astype(np.float32))

    _parallel_blocks(n, work)
    return out.reshape(shape)


def normal_f32(seed: int, stream: int, shape, std: float) -> np.ndarray:
    """float32 N(0, std^2) draws (for the fp32 logits variant)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def work(s, e):
        x = _normals_block(seed, stream, s, e - s)
        np.multiply(x, std, out=x)
        out[s:e] = x

    _parallel_blocks(n, work)
    return out.reshape(shape)


def uniform_targets(seed: int, stream: int, n: int, vocab: int) -> np.ndarray:
    u = uniform01(seed, stream, 0, n)
    return np.minimum((u * vocab).astype(np.int64), vocab - 1)


def zipf_targets(seed: int, stream: int, n: int, vocab: int, s: float) -> np.ndarray:
    weights = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(weights)
    u = uniform01(seed, stream, 0, n) * cdf[-1]
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, vocab - 1).astype(np.int64)


def ignore_positions(seed: int, stream: int, n: int, frac: float) -> np.ndarray:
    """Exactly floor(frac * n) distinct positions (partial Fisher-Yates)."""
    k = int(np.floor(frac * n + 1e-9))
    if k == 0 or n == 0:
        return np.zeros(0, dtype=np.int64)
    perm = np.arange(n, dtype=np.int64)
    r = splitmix64(seed, stream, 0, k)
    for i in range(k):
        j = i + int(r[i] % np.uint64(n - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:k])


@dataclasses.dataclass
class FlceInputs:
    """One FLCE problem: bf16 bit patterns (uint16) or float16 values, plus int64 targets."""

    hidden: np.ndarray            # [N, H]: uint16 bf16 bits, or float16
    weight: np.ndarray            # [V, H]: same type as hidden
    bias: Optional[np.ndarray]    # [V]: same type, or None
    target: np.ndarray            # int64 [N]
    ignore_index: int = IGNORE_INDEX

    @property
    def shape(self):
        return self.hidden.shape[0], self.hidden.shape[1], self.weight.shape[0]


# Stream ids (fixed forever so stored values stay valid).
_S_HIDDEN, _S_WEIGHT, _S_BIAS, _S_TARGET, _S_IGNORE, _S_LOGITS, _S_GRADOUT = range(1, 8)


def make_flce_inputs(n: int, h: int, v: int, seed: int, *, h_std: float = 1.0,
                     w_std: float = 0.02, bias_std: Optional[float] = None,
                     targets: str = "uniform", zipf_s: float = 1.1,
                     ignore_frac: float = 0.05,
                     ignore_index: int = IGNORE_INDEX, dtype: str = "bf16") -> FlceInputs:
    """dtype "bf16": bf16 bit patterns; "fp16": float16 values (float64 draw ->
    float32 -> float16, round to nearest even); "fp32": float32 values."""
    if dtype == "bf16":
        gen = normal_bf16
    elif dtype == "fp16":
        def gen(sd, st, shape, std):
            return normal_f32(sd, st, shape, std).astype(np.float16)
    elif dtype == "fp32":
        gen = normal_f32
    else:
        raise ValueError(dtype)
    hidden = gen(seed, _S_HIDDEN, (n, h), h_std)
    weight = gen(seed, _S_WEIGHT, (v, h), w_std)
    bias = gen(seed, _S_BIAS, (v,), bias_std) if bias_std is not None else None
    if targets == "uniform":
        t = uniform_targets(seed, _S_TARGET, n, v)
    elif targets == "zipf":
        t = zipf_targets(seed, _S_TARGET, n, v, zipf_s)
    else:
        raise ValueError(targets)
    t[ignore_positions(seed, _S_IGNORE, n, ignore_frac)] = ignore_index
    return FlceInputs(hidden, weight, bias, t, ignore_index)


def make_ce_logits(n: int, v: int, seed: int, *, std: float = 2.0, dtype: str = "bf16",
                   ignore_frac: float = 0.05, ignore_index: int = IGNORE_INDEX):
    """Materialised logits [n, v] ~ N(0, std^2) (bf16 bits, float16 or float32) and targets."""
    if dtype == "bf16":
        logits = normal_bf16(seed, _S_LOGITS, (n, v), std)
    elif dtype == "fp32":
        logits = normal_f32(seed, _S_LOGITS, (n, v), std)
    elif dtype == "fp16":
        logits = normal_f32(seed, _S_LOGITS, (n, v), std).astype(np.float16)
    else:
        raise ValueError(dtype)
    t = uniform_targets(seed, _S_TARGET, n, v)
    t[ignore_positions(seed, _S_IGNORE, n, ignore_frac)] = ignore_index
    return logits, t


def make_grad_out(n: int, seed: int) -> np.ndarray:
    """Per-row upstream gradients for reduction 'none' (uniform in (0.5, 1.5))."""
    return (uniform01(seed, _S_GRADOUT, 0, n) + 0.5).astype(np.float32)


# The five workloads.  Seeds 1001..1005.  "N(0, s)" in their descriptions is
# read with s as the standard deviation.
CONFIGS = {
    "tiny": dict(n=256, h=128, v=1024, seed=1001, ignore_frac=0.10, reduction="mean"),
    "small_v32k": dict(n=1024, h=128, v=32768, seed=1002, ignore_frac=0.05, reduction="mean"),
    "small_v64k": dict(n=1024, h=128, v=65536, seed=1002, ignore_frac=0.05, reduction="mean"),
    "llama32_1b": dict(n=8192, h=2048, v=128256, seed=1003, ignore_frac=0.05, reduction="mean"),
    "llama3_8b": dict(n=16384, h=4096, v=128256, seed=1004, ignore_frac=0.05, reduction="mean"),
    "stress_256k": dict(n=32768, h=4096, v=256000, seed=1005, ignore_frac=0.10, reduction="sum",
                        targets="zipf"),
}
CE_CONFIG = dict(n=1024, v=32768, seed=1002, std=2.0, ignore_frac=0.05)


def config_inputs(name: str, *, with_bias: bool = False) -> FlceInputs:
    c = dict(CONFIGS[name])
    c.pop("reduction")
    if with_bias:
        c["bias_std"] = 0.01
    return make_flce_inputs(**c)

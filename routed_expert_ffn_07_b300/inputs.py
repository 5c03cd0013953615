"""Seeded synthetic inputs for the routed MoE FFN layer.

This module only draws numbers and lays them out in the storage formats the
library reads.  It holds none of the layer's arithmetic (no routing, no
dequantisation, no FFN), so both the CUDA path and the fp64 CPU oracle can be
fed from it without sharing any of the method.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based stream: draw ``i`` of
a stream with key ``k`` is ``mix(k + (i + 1) * GOLDEN)`` where ``mix`` is the
SplitMix64 finaliser.  Stream keys chain ``mix`` over (seed, layer, tensor,
expert), so any single expert of any layer can be produced on its own.  The
device generator in ``csrc/gen.cu`` implements the same definition for the
int4 and scale planes, which are too large (tens of GB) to draw on the host.

Value recipes (shapes from the model on the pages: 48 layers x 512 experts,
top-10 routing, one shared expert; sizes d=2048, f=768):

* activations x ~ N(0, 1), rounded to bf16 (or kept fp32 for the tiny case);
* router weights ~ N(0, 0.02) in fp32;
* int4 expert planes: every nibble is one uniform 4-bit draw, read as a
  two's-complement value in [-8, 7]; 16 nibbles come from one 64-bit draw;
* fp16 group scales: 0.005 + 0.015 * u with u uniform in [0, 1);
* fp32 experts (tiny case): ~ N(0, 0.02);
* popularity prior (skewed decode): bias[e] = -s * ln(rank(e)) with a seeded
  random permutation of ranks 1..E per layer (Zipf with exponent s).

Normals use Box-Muller on two draws: u1 = ((z >> 11) + 1) * 2^-53 in (0, 1],
u2 = (z >> 11) * 2^-53; n0 = r cos(2 pi u2), n1 = r sin(2 pi u2),
r = sqrt(-2 ln u1).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_C_LAYER = 0x9E3779B97F4A7C15
_C_TENSOR = 0xD1B54A32D192ED03
_C_EXPERT = 0x8CB92BA72F3D8DD7

# tensor ids of the streams
T_X = 0
T_ROUTER = 1
T_PRIOR = 2
T_GU_Q = 3
T_GU_S = 4
T_DN_Q = 5
T_DN_S = 6
T_GU_F32 = 7
T_DN_F32 = 8

# base seed of workload c (c = 1..5 for the five workloads used by the tests and the bench)
def workload_seed(c: int) -> int:
    return 0x5EED0000 + int(c)


def mix64(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2^64)."""
    z &= MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z


def stream_key(seed: int, layer: int, tensor: int, expert: int = 0) -> int:
    k = mix64(seed)
    k = mix64(k ^ (((layer + 1) * _C_LAYER) & MASK64))
    k = mix64(k ^ (((tensor + 1) * _C_TENSOR) & MASK64))
    k = mix64(k ^ (((expert + 1) * _C_EXPERT) & MASK64))
    return k


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    z = z ^ (z >> np.uint64(31))
    return z


def draws(key: int, n: int, start: int = 0) -> np.ndarray:
    """Draws start .. start+n-1 of the stream with the given key (uint64)."""
    i = np.arange(start + 1, start + 1 + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * np.uint64(GOLDEN)
        return _mix64_np(z)


def uniform01(z: np.ndarray) -> np.ndarray:
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(key: int, n: int) -> np.ndarray:
    m = (n + 1) // 2
    z = draws(key, 2 * m)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:n]


# ---------------------------------------------------------------- number formats
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + r) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Pack int values in [-8, 7] of shape [rows, cols] into the int4 plane layout.

    Layout: row-major, two values per byte, the even column in the low nibble,
    two's complement.  A 16-byte block holds one group of 32 columns.
    """
    q = np.asarray(q)
    assert q.ndim == 2 and q.shape[1] % 2 == 0
    assert q.min() >= -8 and q.max() <= 7
    n = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return (n[:, 0::2] | (n[:, 1::2] << 4)).astype(np.uint8)


# ---------------------------------------------------------------- tensors
def gen_activations(seed: int, T: int, d: int, dtype: str = "bf16", layer: int = 0) -> np.ndarray:
    """x ~ N(0, 1) of shape [T, d]; bf16 returns uint16 bit patterns, f32 returns float32.

    For the tiny fp32 workload the values are scaled by 0.02 (all tensors ~N(0, 0.02)).
    """
    v = normals(stream_key(seed, layer, T_X), T * d).reshape(T, d)
    if dtype == "bf16":
        return f32_to_bf16_bits(v.astype(np.float32))
    if dtype == "f32":
        return (0.02 * v).astype(np.float32)
    raise ValueError(dtype)


def gen_router(seed: int, layer: int, E: int, d: int) -> np.ndarray:
    return (0.02 * normals(stream_key(seed, layer, T_ROUTER), E * d)).astype(np.float32).reshape(E, d)


def gen_zipf_prior(seed: int, layer: int, E: int, s: float = 1.1) -> np.ndarray:
    """Router bias carrying a Zipf(s) popularity prior: -s * ln(rank), ranks a seeded permutation."""
    z = draws(stream_key(seed, layer, T_PRIOR), E)
    perm = np.arange(E)
    for i in range(E - 1, 0, -1):  # Fisher-Yates
        j = int(z[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    ranks = perm + 1
    return (-s * np.log(ranks.astype(np.float64))).astype(np.float32)


def _int4_plane(key: int, rows: int, cols: int) -> np.ndarray:
    nbytes = rows * cols // 2
    assert nbytes % 8 == 0
    return draws(key, nbytes // 8).view(np.uint8).reshape(rows, cols // 2).copy()


def _scale_plane(key: int, rows: int, groups: int) -> np.ndarray:
    u = uniform01(draws(key, rows * groups))
    s = 0.005 + 0.015 * u
    return s.astype(np.float16).view(np.uint16).reshape(rows, groups)


def expert_key(seed: int, layer: int, tensor: int, e: int) -> int:
    return stream_key(seed, layer, tensor, e)


def gen_expert_int4(seed: int, layer: int, e: int, d: int, f: int) -> dict:
    """One expert in the int4 group-32 format (e == E is the shared expert).

    gu_q: uint8 [2f, d/2]  rows 0..f-1 = gate, f..2f-1 = up
    gu_s: uint16 (fp16 bits) [2f, d/32]
    dn_q: uint8 [d, f/2]
    dn_s: uint16 (fp16 bits) [d, f/32]
    """
    return dict(
        gu_q=_int4_plane(expert_key(seed, layer, T_GU_Q, e), 2 * f, d),
        gu_s=_scale_plane(expert_key(seed, layer, T_GU_S, e), 2 * f, d // 32),
        dn_q=_int4_plane(expert_key(seed, layer, T_DN_Q, e), d, f),
        dn_s=_scale_plane(expert_key(seed, layer, T_DN_S, e), d, f // 32),
    )


def gen_expert_f32(seed: int, layer: int, e: int, d: int, f: int) -> dict:
    """One expert in plain fp32 (tiny workload): gu [2f, d], dn [d, f], ~N(0, 0.02)."""
    gu = (0.02 * normals(expert_key(seed, layer, T_GU_F32, e), 2 * f * d)).astype(np.float32)
    dn = (0.02 * normals(expert_key(seed, layer, T_DN_F32, e), d * f)).astype(np.float32)
    return dict(gu_q=gu.reshape(2 * f, d), gu_s=None, dn_q=dn.reshape(d, f), dn_s=None)


def gen_layer_experts(seed: int, layer: int, E: int, d: int, f: int, wfmt: str, experts=None) -> dict:
    """Stacked planes for the listed experts (all E by default), keyed by expert index."""
    gen = gen_expert_int4 if wfmt == "int4" else gen_expert_f32
    experts = range(E) if experts is None else experts
    return {int(e): gen(seed, layer, int(e), d, f) for e in experts}


def stack_planes(per_expert: dict, E: int) -> dict:
    """Concatenate per-expert planes 0..E-1 into contiguous [E, ...] planes."""
    out = {}
    for name in ("gu_q", "gu_s", "dn_q", "dn_s"):
        if per_expert[0][name] is None:
            out[name] = None
        else:
            out[name] = np.ascontiguousarray(np.stack([per_expert[e][name] for e in range(E)]))
    return out

"""Seeded synthetic e4m3 workloads.

This module only *makes inputs*: it draws seeded random tensors with the
shapes and value laws of the five workloads below and casts them to OCP E4M3
bytes.  It holds none of the coding arithmetic (no histogram, no codebook, no
bit packing), so both the CPU oracle and the CUDA library can be fed from it
without sharing any of the method's code.

Each workload exists twice:

* a NumPy path (``np_*``), exact and reproducible on any host, used for test
  sizes the oracle finishes in seconds;
* a PyTorch path (``dev_*``) with the same law, drawn by a seeded device
  generator, used for the 2^28 / 2^30-byte and batched workloads whose host
  generation would take minutes.  Its values differ from the NumPy path's
  (different random streams) but follow the same law.

Value laws (the pages measure Gemma 2B FFN activations, which are not
available; these synthetic laws stand in for them):

* ``gauss``      x ~ N(0, sigma^2), near-Gaussian like the FFN1 activation
  (Quad Length Codes, section 3, case 1; Single-Stage Huffman, Figure 1).
* ``zero_spike`` 40% exact 0x00, the rest 2*GELU(z), z ~ N(0,1): a zero spike
  like the FFN2 activation (Quad Length Codes, section 3, case 2).
* ``grad``       s_b * t_4 with a per-4096-element block scale s_b log-uniform
  in [2^-4, 2^4]: heavy-tailed, block-scaled, gradient-like.

Every value is drawn in float64, rounded to float32 (round to nearest even),
then cast to E4M3 with round-to-nearest-even and saturation to +-448.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0

# --------------------------------------------------------------------------
# OCP E4M3 (FN variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
# bits, no infinities, 0x7F/0xFF = NaN, largest finite 448 = 0x7E.
# --------------------------------------------------------------------------


def e4m3_from_f32(x: np.ndarray) -> np.ndarray:
    """Cast float32 values to E4M3 bytes: round to nearest even, saturate.

    Finite values beyond +-448 saturate to +-448 (0x7E / 0xFE).  The sign is
    kept for zeros and for values that round to zero (-0.0 -> 0x80).  NaN maps
    to 0x7F with its sign bit.  Works on the float32 bit pattern in integer
    arithmetic so the rounding is exact.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    sign = ((bits >> np.uint32(31)) & np.uint32(1)).astype(np.uint8) << np.uint8(7)
    nan = np.isnan(x)
    a = np.minimum(np.abs(np.where(nan, np.float32(0), x)), np.float32(E4M3_MAX))
    abits = a.view(np.uint32)
    exp = (abits >> np.uint32(23)).astype(np.int32) - 127          # unbiased
    man = (abits & np.uint32(0x7FFFFF)).astype(np.uint32)
    out = np.zeros(x.shape, dtype=np.uint32)

    # normal E4M3 range: |x| >= 2^-6 -> biased exponent 1..15
    norm = exp >= -6
    e = exp[norm]
    m = man[norm]
    code = ((e + 7).astype(np.uint32) << np.uint32(3)) | (m >> np.uint32(20))
    rem = m & np.uint32(0xFFFFF)
    half = np.uint32(0x80000)
    up = (rem > half) | ((rem == half) & ((code & np.uint32(1)) == 1))
    out[norm] = code + up.astype(np.uint32)        # a carry moves into the exponent

    # subnormal E4M3 range: |x| < 2^-6 -> multiples of 2^-9, round half even
    sub = ~norm
    q = np.rint(a[sub].astype(np.float64) * 512.0)   # exact scaling, RNE
    out[sub] = q.astype(np.uint32)                   # 8 -> 0x08 = 2^-6 (normal)

    res = out.astype(np.uint8) | sign
    res[nan] = np.uint8(0x7F) | sign[nan]
    return res


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """Decode E4M3 bytes to float64 (NaN for 0x7F/0xFF)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return s * val


# --------------------------------------------------------------------------
# seeding
# --------------------------------------------------------------------------

def rng(*key: int) -> np.random.Generator:
    """NumPy generator for a tuple key, e.g. rng(1, 0) for workload 1."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def torch_seed(*key: int) -> int:
    """Deterministic 63-bit seed for a torch generator from a tuple key."""
    return int(np.random.SeedSequence(list(key)).generate_state(2, np.uint64)[0] >> np.uint64(1))


_BATCH = 1 << 22   # host generation batch (elements)


def _to_e4m3(x64: np.ndarray) -> np.ndarray:
    return e4m3_from_f32(x64.astype(np.float32))


# --------------------------------------------------------------------------
# NumPy laws
# --------------------------------------------------------------------------

def np_gauss(n: int, key: tuple, sigma: float | None = None) -> tuple[np.ndarray, float]:
    """n bytes of E4M3(N(0, sigma^2)).  sigma=None draws sigma = 2^U(-2,2)
    from the same stream first (log-uniform in [0.25, 4])."""
    g = rng(*key)
    if sigma is None:
        sigma = float(2.0 ** g.uniform(-2.0, 2.0))
    out = np.empty(n, dtype=np.uint8)
    for i in range(0, n, _BATCH):
        k = min(_BATCH, n - i)
        out[i:i + k] = _to_e4m3(sigma * g.standard_normal(k))
    return out, sigma


def _gelu(z: np.ndarray) -> np.ndarray:
    from scipy.special import erf
    return z * 0.5 * (1.0 + erf(z / math.sqrt(2.0)))


def np_zero_spike(n: int, key: tuple, p_zero: float = 0.4) -> np.ndarray:
    """n bytes: Bernoulli(p_zero) exact 0x00, else E4M3(2*GELU(z))."""
    g = rng(*key)
    out = np.empty(n, dtype=np.uint8)
    for i in range(0, n, _BATCH):
        k = min(_BATCH, n - i)
        mask = g.random(k) < p_zero
        z = g.standard_normal(k)
        b = _to_e4m3(2.0 * _gelu(z))
        b[mask] = 0
        out[i:i + k] = b
    return out


def _t4(g: np.random.Generator, k: int) -> np.ndarray:
    # Student t with 4 degrees of freedom: z / sqrt(chi2_4 / 4), where
    # chi2_4 / 2 ~ Gamma(2, 1) = -ln(u1) - ln(u2), u in (0, 1].
    z = g.standard_normal(k)
    u1 = 1.0 - g.random(k)
    u2 = 1.0 - g.random(k)
    return z / np.sqrt(-0.5 * (np.log(u1) + np.log(u2)))


GRAD_BLOCK = 4096


def np_grad(n: int, key: tuple) -> np.ndarray:
    """n bytes of E4M3(s_b * t_4), s_b = 2^U(-4,4) per 4096-element block."""
    g = rng(*key)
    out = np.empty(n, dtype=np.uint8)
    step = (_BATCH // GRAD_BLOCK) * GRAD_BLOCK
    for i in range(0, n, step):
        k = min(step, n - i)
        nb = -(-k // GRAD_BLOCK)
        s = np.repeat(2.0 ** g.uniform(-4.0, 4.0, nb), GRAD_BLOCK)[:k]
        out[i:i + k] = _to_e4m3(s * _t4(g, k))
    return out


# --------------------------------------------------------------------------
# Workload recipes (host)
# --------------------------------------------------------------------------

def qlc_base_tensor(n: int = 1 << 20, key: tuple = (1, 0)) -> np.ndarray:
    """Base-QLC round trip workload: E4M3(N(0,1)), 2^20 bytes."""
    return np_gauss(n, key, sigma=1.0)[0]


def huffman_shards(count: int, n: int = 1 << 22, fresh: bool = False):
    """Single-stage Huffman shards: N(0, sigma_i), sigma_i log-uniform in
    [0.25, 4].  Warm-up shard i uses key (2, i); fresh shard i (2, 100 + i).
    Yields (bytes, sigma)."""
    base = 100 if fresh else 0
    for i in range(count):
        yield np_gauss(n, (2, base + i))


def zero_spike_tensor(n: int = 1 << 28, key: tuple = (3, 0)) -> np.ndarray:
    return np_zero_spike(n, key)


def grad_tensor(n: int = 1 << 30, key: tuple = (4, 0)) -> np.ndarray:
    return np_grad(n, key)


def grad_warmup(i: int, n: int = 1 << 24) -> np.ndarray:
    return np_grad(n, (4, 1 + i))


# --------------------------------------------------------------------------
# Batched message regime: 4096 tensors, sizes log-uniform in [4 KiB, 8 MiB]
# --------------------------------------------------------------------------

def batch_plan(count: int = 4096, key: tuple = (5,), lo_log2: float = 12.0, hi_log2: float = 23.0):
    """Plan of the batched workload: per tensor (size, law, codebook tag).

    size: floor(2^U(lo_log2, hi_log2)) bytes (4 KiB .. 8 MiB by default).
    law: the generator of workload 1, 2 or 3, drawn uniformly:
    0 = gauss N(0,1), 1 = gauss with sigma log-uniform, 2 = zero spike.
    tag: one of the four precomputed codebooks, drawn uniformly and
    independently of the law: 0 = base QLC of N(0,1) warm-up data,
    1 = adapted QLC of zero-spike warm-up data, 2 = Huffman of pooled
    N(0, sigma) shards, 3 = Huffman of zero-spike warm-up data.  A tensor is
    therefore often coded with a codebook fitted to another law (longer codes,
    even expansion), as happens when one codebook serves mixed traffic.
    """
    plan = []
    for i in range(count):
        g = rng(*key, i)
        size = int(math.floor(2.0 ** g.uniform(lo_log2, hi_log2)))
        law = int(g.integers(0, 3))
        tag = int(g.integers(0, 4))
        plan.append((size, law, tag))
    return plan


def np_batch_tensor(size: int, law: int, key: tuple) -> np.ndarray:
    if law == 0:
        return np_gauss(size, key, sigma=1.0)[0]
    if law == 1:
        return np_gauss(size, key)[0]
    return np_zero_spike(size, key)


# --------------------------------------------------------------------------
# BF16 tensors (the exponent escape code of ZipCCL works on BF16 values)
# --------------------------------------------------------------------------

def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Cast float32 values to BF16 bit patterns (uint16): round to nearest
    even on the float32 bits (finite values)."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> np.uint64(16)) & np.uint64(1)
    return ((f + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def np_bf16_gauss(n: int, key: tuple, sigma: float) -> np.ndarray:
    """n BF16 values of N(0, sigma^2) (drawn in float64, rounded to float32,
    then to BF16), as uint16 bit patterns: the near-Gaussian layer data the
    ZipCCL page codes."""
    g = rng(*key)
    out = np.empty(n, dtype=np.uint16)
    for i in range(0, n, _BATCH):
        k = min(_BATCH, n - i)
        out[i:i + k] = bf16_from_f32((sigma * g.standard_normal(k)).astype(np.float32))
    return out


# --------------------------------------------------------------------------
# PyTorch (device) laws: same recipes, device random streams
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def dev_e4m3(x):
    """Device cast float -> E4M3 bytes (RNE, saturate to +-448)."""
    torch = _torch()
    return x.float().clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _dev_gen(device, key):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(torch_seed(*key))
    return g


_DEV_BATCH = 1 << 26


def dev_gauss(n: int, key: tuple, device="cuda", sigma: float | None = None, out=None):
    torch = _torch()
    g = _dev_gen(device, key)
    if sigma is None:
        sigma = float(2.0 ** (torch.rand(1, generator=g, device=device, dtype=torch.float64).item() * 4.0 - 2.0))
    out = torch.empty(n, dtype=torch.uint8, device=device) if out is None else out
    for i in range(0, n, _DEV_BATCH):
        k = min(_DEV_BATCH, n - i)
        z = torch.randn(k, generator=g, device=device, dtype=torch.float64)
        out[i:i + k] = dev_e4m3((sigma * z).float())
    return out, sigma


def dev_zero_spike(n: int, key: tuple, device="cuda", p_zero: float = 0.4, out=None):
    torch = _torch()
    g = _dev_gen(device, key)
    out = torch.empty(n, dtype=torch.uint8, device=device) if out is None else out
    for i in range(0, n, _DEV_BATCH):
        k = min(_DEV_BATCH, n - i)
        mask = torch.rand(k, generator=g, device=device, dtype=torch.float64) < p_zero
        z = torch.randn(k, generator=g, device=device, dtype=torch.float64)
        y = 2.0 * z * 0.5 * (1.0 + torch.erf(z / math.sqrt(2.0)))
        b = dev_e4m3(y.float())
        b[mask] = 0
        out[i:i + k] = b
    return out


def dev_grad(n: int, key: tuple, device="cuda", out=None):
    torch = _torch()
    g = _dev_gen(device, key)
    out = torch.empty(n, dtype=torch.uint8, device=device) if out is None else out
    step = (_DEV_BATCH // GRAD_BLOCK) * GRAD_BLOCK
    for i in range(0, n, step):
        k = min(step, n - i)
        nb = -(-k // GRAD_BLOCK)
        s = torch.exp2(torch.rand(nb, generator=g, device=device, dtype=torch.float64) * 8.0 - 4.0)
        s = s.repeat_interleave(GRAD_BLOCK)[:k]
        z = torch.randn(k, generator=g, device=device, dtype=torch.float64)
        u1 = 1.0 - torch.rand(k, generator=g, device=device, dtype=torch.float64)
        u2 = 1.0 - torch.rand(k, generator=g, device=device, dtype=torch.float64)
        t4 = z / torch.sqrt(-0.5 * (torch.log(u1) + torch.log(u2)))
        out[i:i + k] = dev_e4m3((s * t4).float())
    return out


def dev_batch_tensor(size: int, law: int, key: tuple, device="cuda", out=None):
    if law == 0:
        return dev_gauss(size, key, device, sigma=1.0, out=out)[0]
    if law == 1:
        return dev_gauss(size, key, device, out=out)[0]
    return dev_zero_spike(size, key, device, out=out)


def dev_bf16_gauss(n: int, key: tuple, sigma: float, device="cuda"):
    """Device BF16 values of N(0, sigma^2) (float64 draw -> float32 -> BF16,
    round to nearest even), returned as an int16 tensor of bit patterns."""
    torch = _torch()
    g = _dev_gen(device, key)
    out = torch.empty(n, dtype=torch.int16, device=device)
    for i in range(0, n, _DEV_BATCH):
        k = min(_DEV_BATCH, n - i)
        z = torch.randn(k, generator=g, device=device, dtype=torch.float64)
        out[i:i + k] = (sigma * z).float().to(torch.bfloat16).view(torch.int16)
    return out

"""Pins of the workload generators' E4M3 cast.

The cast is input generation, not the coding method, but every parity case
depends on it, so it is checked against two independent implementations
(ml_dtypes where installed, and PyTorch's float8_e4m3fn cast after the
saturating clamp) and against special values of the OCP 8-bit floating point
specification (E4M3: bias 7, largest finite 448 = 0x7E, smallest subnormal
2^-9 = 0x01, no infinities).
"""
import numpy as np
import pytest
import torch

from workloads import (E4M3_MAX, batch_plan, e4m3_from_f32, e4m3_to_f64, np_gauss,
                       np_grad, np_zero_spike)


def _torch_cast(x):
    xc = np.clip(x, -E4M3_MAX, E4M3_MAX).astype(np.float32)
    return torch.from_numpy(xc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _dense_f32_sample():
    """Every float32 exponent from 2^-17 to 2^9 (both signs) with a strided
    sweep of mantissas, plus the patterns at every rounding boundary."""
    exps = np.arange(110, 137, dtype=np.uint32)
    man = np.arange(0, 1 << 23, 97, dtype=np.uint32)
    # boundary patterns: low 20 bits = 0, half-1, half, half+1, max
    hi = np.arange(0, 8, dtype=np.uint32) << np.uint32(20)
    lows = np.array([0, 0x7FFFF, 0x80000, 0x80001, 0xFFFFF], np.uint32)
    man = np.concatenate([man, (hi[:, None] | lows[None, :]).ravel()])
    bits = (exps[:, None] << np.uint32(23)) | man[None, :]
    bits = bits.ravel()
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    return bits.view(np.float32)


def test_cast_special_values():
    vals = np.array([0.0, -0.0, 448.0, -448.0, 464.0, 1e30, -1e30, 2.0 ** -9, 2.0 ** -10,
                     1.5 * 2.0 ** -10, 2.0 ** -6, 1.0, -1.0, 1.0625, 1.1875, 240.0, -1e-30],
                    np.float32)
    want = [0x00, 0x80, 0x7E, 0xFE, 0x7E, 0x7E, 0xFE, 0x01, 0x00,
            0x01, 0x08, 0x38, 0xB8, 0x38, 0x3A, 0x77, 0x80]
    assert e4m3_from_f32(vals).tolist() == want


def test_cast_matches_torch():
    x = _dense_f32_sample()
    assert (e4m3_from_f32(x) == _torch_cast(x)).all()


def test_cast_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    x = _dense_f32_sample()
    ref = np.clip(x, -E4M3_MAX, E4M3_MAX).astype(ml.float8_e4m3fn).view(np.uint8)
    assert (e4m3_from_f32(x) == ref).all()


def test_every_code_round_trips():
    b = np.arange(256, dtype=np.uint8)
    v = e4m3_to_f64(b)
    ok = ~np.isnan(v)
    assert ok.sum() == 254
    assert (e4m3_from_f32(v[ok].astype(np.float32)) == b[ok]).all()


def test_generators_are_seeded_and_shaped():
    a, s1 = np_gauss(5000, (2, 3))
    b, s2 = np_gauss(5000, (2, 3))
    assert (a == b).all() and s1 == s2 and 0.25 <= s1 <= 4
    z = np_zero_spike(200000, (3, 1))
    frac0 = (z == 0).mean()
    assert 0.40 < frac0 < 0.45         # 40% forced zeros plus GELU underflow
    g = np_grad(3 * 4096, (4, 2))
    assert g.dtype == np.uint8 and g.size == 3 * 4096
    plan = batch_plan(4096)
    assert all(4096 <= s < 8 * 2 ** 20 for s, _, _ in plan)
    assert {law for _, law, _ in plan} == {0, 1, 2} and {t for _, _, t in plan} == {0, 1, 2, 3}
    # laws uniform over 3, tags uniform over 4, drawn independently: every
    # (law, tag) pair occurs about 4096/12 times
    pairs = np.zeros((3, 4), np.int64)
    for _, law, t in plan:
        pairs[law, t] += 1
    assert pairs.min() > 4096 / 12 * 0.75 and pairs.max() < 4096 / 12 * 1.25
    sizes = np.log2([s for s, _, _ in plan])
    assert abs(sizes.mean() - 17.5) < 0.15   # log2 size uniform on [12, 23]

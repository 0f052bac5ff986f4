"""GPU parity of the BF16 exponent escape code (ZipCCL, section 2.B; the
exponent table of section 2.A) against the bit-serial oracle: tables,
exponent histogram, container (offsets, payload, sub-block bits, totals) and
the round trip, at several scales, sizes and chunk shapes; corruption flags."""
import numpy as np
import pytest

import oracle
from workloads import np_bf16_gauss

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402


def _dev(x16):
    return torch.from_numpy(x16.view(np.int16)).cuda()


def _check(xh, top, C, S):
    x = _dev(xh)
    enc = ecc.bf16_escape_encode(x, top, C, S)
    y, st = ecc.bf16_escape_decode(enc, top)
    torch.cuda.synchronize()
    assert int(enc.status.item()) == 0 and int(st.item()) == 0
    ref = oracle.bf16_escape_encode(xh, top, C, S)
    off = enc.chunk_off.cpu().numpy().view(np.uint64)
    assert (off == ref["chunk_off"]).all()
    assert (enc.payload[: int(off[-1])].cpu().numpy() == ref["payload"]).all()
    assert (enc.sub_bits[: ref["sub_bits"].size].cpu().numpy().view(np.uint16) == ref["sub_bits"]).all()
    assert int(enc.total_bits.item()) == ref["total_bits"]
    assert (y[: xh.size].cpu().numpy().view(np.uint16) == xh).all()
    return enc


@pytest.mark.parametrize("sigma", [0.02, 1.0, 37.0])
@pytest.mark.parametrize("C,S", [(1024, 64), (4096, 256), (4096, 1024), (16384, 1024)])
def test_bf16_escape_matches_oracle(sigma, C, S):
    top = ecc.bf16_escape_table_sigma(sigma)
    assert (top == oracle.bf16_top7_from_sigma(sigma)).all()
    for n in (1, 17, C - 1, C, C + 1, 3 * C + 5, (1 << 18) + 3):
        _check(np_bf16_gauss(n, (41, n % 97), sigma), top, C, S)


def test_bf16_every_pattern_and_mismatched_table():
    g = np.random.default_rng(4)
    xh = g.permutation(np.arange(1 << 16, dtype=np.uint32)).astype(np.uint16)
    # every bit pattern (NaNs, infinities, subnormals included), with a table
    # fitted to another scale: most values escape
    _check(xh, ecc.bf16_escape_table_sigma(1.0), 4096, 256)
    _check(xh, ecc.bf16_escape_table_sigma(1e-3), 16384, 64)


def test_bf16_histogram_and_count_table():
    xh = np_bf16_gauss((1 << 20) + 13, (42, 0), 0.5)
    cnt = ecc.bf16_exponent_histogram(_dev(xh))
    torch.cuda.synchronize()
    ch = cnt.cpu().numpy().view(np.uint64)
    assert (ch == oracle.bf16_exponent_counts(xh)).all()
    top = ecc.bf16_escape_table_counts(ch)
    assert (top == oracle.bf16_top7_from_counts(ch)).all()
    enc = _check(xh, top, 4096, 256)
    assert 1 - int(enc.total_bits.item()) / (16.0 * xh.size) > 0.29   # about 31% (16 -> 11 bits)


def test_bf16_corruption_is_flagged():
    xh = np_bf16_gauss(3 * 4096 + 100, (43, 0), 1.0)
    top = ecc.bf16_escape_table_sigma(1.0)
    enc = ecc.bf16_escape_encode(_dev(xh), top, 4096, 256)
    torch.cuda.synchronize()
    g = np.random.default_rng(5)
    used = int(enc.chunk_off[-1].item())
    for trial in range(6):
        pay = enc.payload.clone()
        pos = int(g.integers(0, used))
        pay[pos] ^= torch.tensor(1 << int(g.integers(0, 8)), dtype=torch.uint8, device="cuda")
        bad = ecc.Encoded(pay, enc.chunk_off, enc.sub_bits, enc.total_bits, enc.status, enc.n, enc.C, enc.S)
        y, st = ecc.bf16_escape_decode(bad, top)
        torch.cuda.synchronize()
        # a flipped bit is caught, or changes the output (never silent and equal)
        assert int(st.item()) == ecc.ERR_CORRUPT or not torch.equal(y[: xh.size], _dev(xh))
    off = enc.chunk_off.clone()
    off[1] += 16
    bad = ecc.Encoded(enc.payload, off, enc.sub_bits, enc.total_bits, enc.status, enc.n, enc.C, enc.S)
    _, st = ecc.bf16_escape_decode(bad, top)
    torch.cuda.synchronize()
    assert int(st.item()) == ecc.ERR_CORRUPT
    # 000 followed by a table exponent (127 is in the sigma = 1 table)
    s = "000" + format(127, "08b") + "00000000"
    raw = np.zeros(16, np.uint8)
    raw[:3] = [int((s + "00000")[i:i + 8], 2) for i in range(0, 24, 8)]
    one = ecc.Encoded(torch.from_numpy(raw).cuda(), torch.tensor([0, 16], dtype=torch.int64, device="cuda"),
                      torch.tensor([19], dtype=torch.int16, device="cuda"), enc.total_bits, enc.status, 1, 1024, 64)
    _, st = ecc.bf16_escape_decode(one, top)
    torch.cuda.synchronize()
    assert int(st.item()) == ecc.ERR_CORRUPT


def test_decode_needs_aligned_output():
    """The decoder writes eight values at a time with 16-byte stores: an
    output that is not 16-byte aligned is a host error (nothing launched)."""
    xh = np_bf16_gauss(4096, (9, 3), 0.02)
    top = oracle.bf16_top7_from_sigma(0.02)
    enc = ecc.bf16_escape_encode(_dev(xh), top, 4096, 64)
    out = torch.empty(4096 + 8, dtype=torch.int16, device="cuda")
    with pytest.raises(ecc.EccError):
        ecc.bf16_escape_decode(enc, top, out=out[1:])
    y, st = ecc.bf16_escape_decode(enc, top, out=out[8:])
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (y[:4096].cpu().numpy().view(np.uint16) == xh).all()

"""Canonical Huffman codebook built on the device (the three-stage pipeline:
histogram, codebook, encode in one stream).

The device codebook must be the host builder's, byte for byte, for the same
weights count + add, and its lengths and codes must be the oracle's Huffman
lengths and canonical codes.  The weight sets cover what decides the tree:
random and workload histograms, ties everywhere (equal weights, runs of the
pseudocount alone), one and two coded bytes, the longest tree within the
length cap, one that exceeds it, and inputs that are not a codebook.
"""
import numpy as np
import pytest

import oracle
from workloads import np_gauss, np_zero_spike

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402


def dev_build(count, add=1, max_len=ecc.MAX_CODE_LEN):
    c = torch.from_numpy(np.asarray(count, np.uint64).view(np.int64)).cuda()
    cb, st = ecc.huff_build_device(c, add, max_len)
    torch.cuda.synchronize()
    return cb.cpu().numpy(), int(st.item())


def check_same(count, add=1, max_len=ecc.MAX_CODE_LEN):
    w = np.asarray(count, np.uint64) + np.uint64(add)
    host = ecc.huff_build_canonical(w, max_len)
    dev, st = dev_build(count, add, max_len)
    assert st == ecc.OK
    assert dev.tobytes() == host.tobytes()
    ref = oracle.huffman_codebook(w)
    v = ecc.codebook_view(dev)
    assert (v["len"] == ref["len"]).all()
    coded = ref["len"] > 0
    assert (v["code"][coded] == ref["code"][coded]).all()
    return dev


def fib_counts(n):
    """Fibonacci weights on bytes 0..n-1: the deepest tree n bytes allow."""
    c = np.zeros(256, np.uint64)
    a, b = 1, 1
    for i in range(n):
        c[i] = a
        a, b = b, a + b
    return c


@pytest.mark.parametrize("seed", range(6))
def test_random_histograms(seed):
    g = np.random.default_rng(seed)
    scale = [1, 10, 1000, 1 << 20, 1 << 40, 3][seed]
    c = g.integers(0, scale + 1, 256).astype(np.uint64)
    c[g.random(256) < 0.3] = 0  # absent bytes keep only the pseudocount
    check_same(c, add=1)
    check_same(c, add=0)  # absent bytes get no code


def test_weights_above_2_55():
    """Weight sums of 2^55 and more take the two-word key path."""
    g = np.random.default_rng(55)
    c = g.integers(0, 1 << 55, 256, dtype=np.uint64)
    check_same(c, add=1)
    c[::2] = np.uint64(1 << 54)  # ties among large weights
    c[1::4] = 0
    check_same(c, add=0)
    check_same(c, add=3)


def test_workload_histograms():
    for x in (np_gauss(1 << 20, (3, 1))[0], np_gauss(1 << 20, (3, 2), 1.0)[0], np_zero_spike(1 << 20, (3, 3))):
        check_same(oracle.histogram(x), add=1)


def test_ties():
    check_same(np.zeros(256, np.uint64), add=1)            # 256 equal weights: all length 8
    check_same(np.full(256, 7, np.uint64), add=0)
    c = np.zeros(256, np.uint64)
    c[::3] = 5
    c[1::7] = 5
    check_same(c, add=0)                                   # equal weights, scattered bytes
    check_same(np.arange(256, dtype=np.uint64) % 4, add=1)  # four weight classes, many ties


def test_one_and_two_symbols():
    for b in (0, 37, 255):
        c = np.zeros(256, np.uint64)
        c[b] = 9
        dev = check_same(c, add=0)
        assert int(ecc.codebook_view(dev)["len"][b]) == 1
    c = np.zeros(256, np.uint64)
    c[200], c[3] = 1, 1 << 50
    check_same(c, add=0)


def test_length_cap():
    c = fib_counts(40)  # a 39-bit deepest code
    check_same(c, add=0, max_len=39)
    dev, st = dev_build(c, add=0, max_len=38)
    assert st == ecc.ERR_CODEBOOK
    assert not dev.any()  # no magic word: unusable
    with pytest.raises(ecc.EccError):
        ecc.huff_build_canonical(c, 38)


def test_not_a_codebook():
    dev, st = dev_build(np.zeros(256, np.uint64), add=0)
    assert st == ecc.ERR_ARG and not dev.any()
    c = np.zeros(256, np.uint64)
    c[0] = np.uint64(1 << 63)
    c[1] = np.uint64(1 << 63)
    assert dev_build(c, add=0)[1] == ecc.ERR_ARG  # the sum wraps
    c = np.zeros(256, np.uint64)
    c[5] = np.uint64(2**64 - 1)
    assert dev_build(c, add=1)[1] == ecc.ERR_ARG  # the weight itself wraps


@pytest.mark.parametrize("tensor", ["gauss", "spike"])
def test_three_stage_pipeline(tensor):
    """histogram -> device codebook -> encode -> decode on one stream, against
    the oracle encoding of the same tensor with the oracle's codebook."""
    n = (1 << 20) + 12345
    x = np_gauss(n, (8, 1))[0] if tensor == "gauss" else np_zero_spike(n, (8, 2))
    xd = torch.from_numpy(x).cuda()
    count = ecc.e4m3_histogram(xd)
    cb, st = ecc.huff_build_device(count, 1)
    C, S = 16384, 256
    enc = ecc.ecc_encode(xd, cb, C, S)
    y, dst = ecc.ecc_decode(enc, cb)
    torch.cuda.synchronize()
    assert int(st.item()) == ecc.OK and int(enc.status.item()) == ecc.OK and int(dst.item()) == ecc.OK
    ref = oracle.encode(x, oracle.huffman_codebook(oracle.histogram(x) + np.uint64(1)), C, S)
    off = enc.chunk_off.cpu().numpy().view(np.uint64)
    assert (off == ref["chunk_off"]).all()
    assert (enc.payload[:int(off[-1])].cpu().numpy() == ref["payload"]).all()
    assert (y[:n].cpu().numpy() == x).all()

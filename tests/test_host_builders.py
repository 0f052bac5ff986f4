"""The library's host side (C ABI, no GPU needed) against the oracle.

The codebook builders, the width search and the figures of the CUDA library
are independent implementations; here they must agree with the oracle bit
for bit (tables) or to 1e-9 relative (float64 figures).
"""
import ctypes as ct
import os
import re

import numpy as np
import pytest

import lossless_entropy_coding_gb300 as ecc
import oracle
from lossless_entropy_coding_gb300 import build as ecc_build
from workloads import np_gauss, np_grad, np_zero_spike, qlc_base_tensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    ecc_build.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "ecc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 19
    lib = ct.CDLL(ecc.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name


def test_codebook_layout():
    assert ecc.codebook_bytes() == ecc.CODEBOOK_DTYPE.itemsize


def pmfs():
    g = np.random.default_rng(7)
    ties = np.zeros(256, np.uint64)
    ties[g.choice(256, 40, replace=False)] = 5
    ties[[0, 255]] = 9
    return {
        "gauss": oracle.histogram(qlc_base_tensor()),
        "spike": oracle.histogram(np_zero_spike(1 << 20, (3, 5))),
        "grad": oracle.histogram(np_grad(1 << 20, (4, 5))),
        "uniform": np.full(256, 11, np.uint64),
        "ties": ties,
        "random": g.integers(0, 1 << 40, 256).astype(np.uint64),
        "one": np.eye(256, dtype=np.uint64)[200] * 77,
    }


@pytest.mark.parametrize("name", list(pmfs().keys()))
def test_qlc_tables_match_oracle(name):
    count = pmfs()[name]
    widths = [ecc.BASE_WIDTHS, (0, 1, 1, 4, 4, 4, 4, 8), (8, 0, 0, 0, 0, 0, 0, 0), (2, 2, 4, 4, 5, 5, 6, 7)]
    for w in widths:
        cb = ecc.codebook_view(ecc.qlc_build_tables(count, w))
        ref = oracle.qlc_codebook(count, w)
        assert cb["magic"] == 0x45434342 and cb["family"] == ecc.FAMILY_QLC
        assert (cb["len"] == ref["len"]).all()
        assert (cb["code"] == ref["code"]).all()
        assert (cb["by_rank"] == ref["by_rank"]).all()
        r, _ = oracle.rank(count)
        assert (cb["rank"] == r).all()
        assert cb["max_len"] == ref["len"].max()


@pytest.mark.parametrize("name", ["gauss", "spike", "grad", "ties", "random"])
@pytest.mark.parametrize("full", [False, True])
def test_width_search_matches_oracle(name, full):
    count = pmfs()[name]
    for md in (2, 3, 4):
        w, cost = ecc.qlc_search_widths(count, md, full)
        wr, cr = oracle.qlc_search(count, md, full)
        assert cost == cr and (w == wr).all()


def test_width_search_rejects_impossible():
    with pytest.raises(ecc.EccError):
        ecc.qlc_search_widths(np.ones(256, np.uint64), 0)


@pytest.mark.parametrize("name", list(pmfs().keys()))
def test_huffman_matches_oracle(name):
    weight = pmfs()[name]
    cb = ecc.codebook_view(ecc.huff_build_canonical(weight))
    ref = oracle.huffman_codebook(weight)
    assert cb["family"] == ecc.FAMILY_HUFFMAN
    assert (cb["len"] == ref["len"]).all()
    assert (cb["code"] == ref["code"]).all()
    fixed = oracle.fixed_codebook_weights([weight])
    cb2 = ecc.codebook_view(ecc.huff_build_canonical(fixed))
    assert (cb2["len"] == oracle.huffman_lengths(fixed)).all()


@pytest.mark.parametrize("name", ["gauss", "spike", "grad", "ties", "random"])
@pytest.mark.parametrize("p", [1, 2, 3])
def test_prefix_bits_qlc_matches_oracle(name, p):
    count = pmfs()[name]
    for md in (2, 4):
        w, cost = ecc.gqlc_search_widths(count, p, md)
        ow, ocost = oracle.qlc_search(count, md, prefix_bits=p)
        assert (w == ow).all() and cost == ocost
        cb = ecc.codebook_view(ecc.gqlc_build_tables(count, w, p))
        ref = oracle.qlc_codebook(count, w, prefix_bits=p)
        assert cb["family"] == ecc.FAMILY_QLC and int(cb["prefix_bits"]) == p
        assert (cb["len"] == ref["len"]).all() and (cb["code"] == ref["code"]).all()
    if p == 3:
        assert (ecc.gqlc_build_tables(count, ecc.BASE_WIDTHS, 3) == ecc.qlc_build_tables(count)).all()
    with pytest.raises(ecc.EccError):
        ecc.gqlc_build_tables(count, (8, 8), 4)


@pytest.mark.parametrize("name", list(pmfs().keys()))
def test_limited_huffman_matches_oracle(name):
    weight = pmfs()[name]
    nz = int((weight > 0).sum())
    for L in (8, 10, 11, 14, 20, 48):
        if nz > (1 << L):
            continue
        cb = ecc.codebook_view(ecc.huff_build_limited(weight, L))
        ref = oracle.huffman_limited_codebook(weight, L)
        assert cb["family"] == ecc.FAMILY_HUFFMAN
        assert (cb["len"] == ref["len"]).all(), L
        assert (cb["code"] == ref["code"]).all(), L
        assert int(cb["max_len"]) <= L
    with pytest.raises(ecc.EccError) as ei:
        ecc.huff_build_limited(np.ones(256, np.uint64), 7)
    assert ei.value.code == ecc.ERR_CODEBOOK


@pytest.mark.parametrize("name", list(pmfs().keys()))
def test_escape_code_matches_oracle(name):
    count = pmfs()[name]
    cb = ecc.codebook_view(ecc.escape_build_tables(count))
    ref = oracle.escape_codebook(count)
    assert cb["family"] == ecc.FAMILY_ESCAPE
    assert (cb["len"] == ref["len"]).all()
    assert (cb["code"] == ref["code"]).all()
    assert (cb["by_rank"][:7] == ref["top"]).all()
    assert int(cb["max_len"]) == 11 and int(cb["min_len"]) == 7 and int(cb["n_coded"]) == 256


def test_huffman_length_limit_is_an_error():
    w = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(52):            # Fibonacci weights: depth 50
        w[s] = a
        a, b = b, a + b
    assert oracle.huffman_lengths(w).max() > 48
    with pytest.raises(ecc.EccError) as ei:
        ecc.huff_build_canonical(w, 48)
    assert ei.value.code == ecc.ERR_CODEBOOK
    with pytest.raises(ecc.EccError):
        ecc.huff_build_canonical(np.zeros(256, np.uint64))


def test_derived_decode_table():
    # every 14-bit index resolves to the code that prefixes it, or is 0 when
    # no code of <= 14 bits does
    for cbb in (ecc.qlc_build_tables(pmfs()["gauss"]), ecc.huff_build_canonical(pmfs()["spike"] + 1),
                ecc.escape_build_tables(pmfs()["grad"])):
        cb = ecc.codebook_view(cbb)
        want = np.zeros(1 << 14, np.uint16)
        for b in range(256):
            L = int(cb["len"][b])
            if 0 < L <= 14:
                lo = int(cb["code"][b]) << (14 - L)
                want[lo:lo + (1 << (14 - L))] = b | (L << 8)
        assert (cb["dec"] == want).all()
        # encode entries: the code with its first bit in bit 31 and the
        # multiplier 2^(32 - len); both 0 where the exact path codes the byte
        for b in range(256):
            L = int(cb["len"][b])
            v, q = int(cb["enc_code"][b]), int(cb["enc_mul"][b])
            if 0 < L <= 31:
                assert q == 1 << (32 - L) and v == (int(cb["code"][b]) << (32 - L)) & 0xFFFFFFFF
                assert v >> (32 - L) == int(cb["code"][b])
            else:
                assert v == 0 and q == 0


def test_figures_match_oracle():
    P = pmfs()
    for a in ("gauss", "spike", "grad", "random"):
        h, hr = ecc.entropy_bits(P[a]), oracle.entropy_bits(P[a])
        assert abs(h - hr) <= 1e-9 * abs(hr)
        for b in ("gauss", "uniform", "random"):
            k, kr = ecc.kl_bits(P[a], P[b] + 1), oracle.kl_bits(P[a], P[b] + 1)
            assert abs(k - kr) <= 1e-9 * max(abs(kr), 1e-300)
        cb = ecc.qlc_build_tables(P[a])
        assert ecc.code_bits(P[a], cb) == oracle.code_bits(P[a], oracle.qlc_codebook(P[a])["len"])


def test_sizes():
    for n in (0, 1, 1023, 1024, 1025, 5 * 16384 + 3):
        for C in (1024, 16384):
            assert ecc.num_chunks(n, C) == -(-n // C)
            for L in (11, 48):
                assert ecc.max_encoded_bytes(n, C, L) == oracle.max_encoded_bytes(n, C, L)


def test_new_builders_reject_bad_arguments():
    """Argument checks of the later builders, through the C ABI (no GPU)."""
    lib = ecc.lib()
    cnt = np.ones(256, np.uint64)
    out = np.zeros(ecc.codebook_bytes(), np.uint8)
    w = np.zeros(8, np.uint8)
    cost = np.zeros(1, np.uint64)
    p = lambda a: a.ctypes.data_as(ct.c_void_p)
    assert lib.escape_build_tables(None, p(out)) == ecc.ERR_ARG
    assert lib.escape_build_tables(p(cnt), None) == ecc.ERR_ARG
    assert lib.huff_build_limited(p(cnt), 0, p(out)) == ecc.ERR_ARG
    assert lib.huff_build_limited(p(cnt), 49, p(out)) == ecc.ERR_ARG
    assert lib.huff_build_limited(p(np.zeros(256, np.uint64)), 14, p(out)) == ecc.ERR_ARG
    assert lib.huff_build_limited(p(np.full(256, 1 << 60, np.uint64)), 14, p(out)) == ecc.ERR_ARG  # sum >= 2^62
    assert lib.gqlc_build_tables(p(cnt), 0, p(w), p(out)) == ecc.ERR_ARG
    assert lib.gqlc_build_tables(p(cnt), 4, p(w), p(out)) == ecc.ERR_ARG
    assert lib.gqlc_build_tables(p(cnt), 2, p(w), p(out)) == ecc.ERR_ARG  # 4 areas of 1 rank: < 256
    assert lib.gqlc_search_widths(p(cnt), 2, 0, 0, p(w), p(cost)) == ecc.ERR_ARG
    # the device builder checks its pointers before any CUDA call
    dummy = ct.c_void_p(16)
    assert lib.huff_build_device(dummy, 1, 48, ct.c_void_p(24), dummy, None) == ecc.ERR_ARG  # misaligned
    assert lib.huff_build_device(None, 1, 48, dummy, dummy, None) == ecc.ERR_ARG
    assert lib.huff_build_device(dummy, 1, 0, dummy, dummy, None) == ecc.ERR_ARG


def test_checked_build_compiles_and_exports():
    """The index-checked variant (-DECC_CHECKED) builds for sm_103a and
    exports the same C ABI (its kernels run in tests/test_gpu_checked.py)."""
    path = ecc_build.build(checked=True)
    lib = ct.CDLL(path)
    for name in header_functions():
        assert hasattr(lib, name), name


def test_default_subblock_rule():
    """The sub-block size the binding picks when none is given: C/64 clamped
    to [64, 256] for the base QLC (and when no codebook is named), C/128
    clamped to [64, 128] for codes the decoder reads through its table
    (Huffman, the escape code, a QLC of fewer areas); always a power of two
    dividing C (valid for every chunk size)."""
    counts = np.random.default_rng(3).integers(1, 1000, 256).astype(np.uint64)
    qlc = ecc.qlc_build_tables(counts)
    table_coded = [ecc.huff_build_canonical(counts), ecc.escape_build_tables(counts),
                   ecc.gqlc_build_tables(counts, [4, 4, 7, 8], 2)]
    for k in range(7):
        C = 1024 << k
        for S, d, hi in [(ecc.default_subblock(C), 64, 256), (ecc.default_subblock(C, qlc), 64, 256)] + \
                [(ecc.default_subblock(C, cb), 128, 128) for cb in table_coded]:
            assert S == min(hi, max(64, C // d))
            assert S & (S - 1) == 0 and C % S == 0 and 64 <= S <= min(C, 1024)


def test_bf16_escape_tables_match_oracle():
    """The library's BF16 exponent tables (from sigma and from counts) equal
    the oracle's (ZipCCL, section 2.A)."""
    for sigma in 2.0 ** np.linspace(-20, 10, 61):
        assert (ecc.bf16_escape_table_sigma(sigma) == oracle.bf16_top7_from_sigma(sigma)).all()
    g = np.random.default_rng(12)
    for trial in range(20):
        count = g.integers(0, 5, 256).astype(np.uint64) * g.integers(0, 1000, 256).astype(np.uint64)
        assert (ecc.bf16_escape_table_counts(count) == oracle.bf16_top7_from_counts(count)).all()
    with pytest.raises(ecc.EccError):
        ecc.bf16_escape_table_sigma(0.0)

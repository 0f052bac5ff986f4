"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties an oracle function to something the pages print, to a closed
form, to a textbook result, to an exhaustive search, or to an invariant of
prefix codes, so that a dropped term, a wrong index or a swapped operand in
the oracle fails at least one of them.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.conftest import golden
from workloads import np_gauss, np_grad, np_zero_spike, qlc_base_tensor

C16K, S256 = 16384, 256


def bits_of(code, length):
    return format(int(code), "b").zfill(int(length)) if length else ""


def pack_bits(bitstring):
    """Pack a '0'/'1' string MSB-first into bytes (test-side helper)."""
    pad = (-len(bitstring)) % 8
    s = bitstring + "0" * pad
    return np.array([int(s[i:i + 8], 2) for i in range(0, len(s), 8)], np.uint8)


def prefix_free(codes):
    """Brute force: no codeword is a prefix of another."""
    for a, b in itertools.permutations(codes, 2):
        if b.startswith(a):
            return False
    return True


def kraft(lengths):
    return sum(Fraction(1, 2 ** int(L)) for L in lengths if L > 0)


@pytest.fixture(scope="module")
def gauss_counts():
    return oracle.histogram(qlc_base_tensor())


@pytest.fixture(scope="module")
def spike_counts():
    return oracle.histogram(np_zero_spike(1 << 20, (3, 99)))


# --------------------------------------------------------------- base QLC

def test_base_layout_matches_page():
    start, size, covered = oracle.qlc_layout(oracle.BASE_WIDTHS)
    rows = golden("qlc_base_layout.txt")
    assert covered == 256
    for k, (area, nsym, pre, suf, tot) in enumerate(rows):
        assert int(area) == k + 1
        assert size[k] == int(nsym)
        assert oracle.BASE_WIDTHS[k] == int(suf)
        assert int(pre) + int(suf) == int(tot)
    cb = oracle.qlc_codebook(np.arange(256)[::-1].astype(np.uint64))
    lens = sorted(set(cb["len"].tolist()))
    assert lens == sorted({int(r[4]) for r in rows})


def test_base_codes_golden():
    # counts 256..1 make rank r the byte r, so code(byte r) is code(rank r)
    cb = oracle.qlc_codebook(np.arange(256, 0, -1).astype(np.uint64))
    assert (cb["by_rank"] == np.arange(256)).all()
    for r, word in golden("qlc_base_codes.txt"):
        r = int(r)
        assert bits_of(cb["code"][r], cb["len"][r]) == word


def test_base_kraft_closed_form():
    cb = oracle.qlc_codebook(np.ones(256, np.uint64))
    # 40/64 + 16/128 + 32/256 + 168/2048: prefix-free but not complete
    assert kraft(cb["len"]) == Fraction(40, 64) + Fraction(16, 128) + Fraction(32, 256) + Fraction(168, 2048)
    assert float(kraft(cb["len"])) == 0.95703125


def test_base_has_four_lengths_and_is_prefix_free(gauss_counts):
    cb = oracle.qlc_codebook(gauss_counts)
    assert sorted(set(cb["len"].tolist())) == [6, 7, 8, 11]
    assert prefix_free([bits_of(c, L) for c, L in zip(cb["code"], cb["len"])])


def test_rank_order_and_ties():
    count = np.zeros(256, np.uint64)
    count[[200, 3, 77]] = 5          # a three-way tie at the top
    count[10] = 4
    r, br = oracle.rank(count)
    assert list(br[:4]) == [3, 77, 200, 10]
    assert (r[br] == np.arange(256)).all()
    # zero-count bytes still get ranks, in byte order
    rest = [b for b in range(256) if b not in (3, 77, 200, 10)]
    assert list(br[4:]) == rest


def test_qlc_decode_reads_prefix_then_suffix():
    # hand-assembled stream of ranks 0, 40, 56, 88, 255 under the base code
    words = {int(r): w for r, w in golden("qlc_base_codes.txt")}
    ranks = [0, 40, 56, 88, 255]
    stream = "".join(words[r] for r in ranks)
    payload = pack_bits(stream)
    payload = np.concatenate([payload, np.zeros((-payload.size) % 16, np.uint8)])
    count = np.arange(256, 0, -1).astype(np.uint64)
    cb = oracle.qlc_codebook(count)
    enc = {"payload": payload, "chunk_off": np.array([0, payload.size], np.uint64),
           "sub_bits": np.array([len(stream)], np.uint16), "n": 5, "C": 1024, "S": 64}
    assert list(oracle.decode(enc, cb)) == ranks
    # and the oracle's encoder writes the same bits
    e = oracle.encode(np.array(ranks, np.uint8), cb, 1024, 64)
    assert (e["payload"] == payload).all()
    assert e["total_bits"] == len(stream)


def test_unused_qlc_suffix_is_corrupt():
    cb = oracle.qlc_codebook(np.arange(256, 0, -1).astype(np.uint64))
    # area 8 suffix 168 (first unused one): 111 10101000
    stream = "11110101000"
    payload = pack_bits(stream)
    payload = np.concatenate([payload, np.zeros((-payload.size) % 16, np.uint8)])
    enc = {"payload": payload, "chunk_off": np.array([0, 16], np.uint64),
           "sub_bits": np.array([11], np.uint16), "n": 1, "C": 1024, "S": 64}
    with pytest.raises(oracle.OracleError) as ei:
        oracle.decode(enc, cb)
    assert ei.value.code == oracle.CORRUPT


# --------------------------------------------------------------- Huffman

def test_huffman_textbook_example():
    rows = golden("huffman_textbook.txt")
    w = np.zeros(256, np.uint64)
    want = {}
    for b, wt, L in rows:
        w[int(b)] = int(wt)
        want[int(b)] = int(L)
    ln = oracle.huffman_lengths(w)
    for b, L in want.items():
        assert ln[b] == L
    assert (ln[6:] == 0).all()
    assert oracle.code_bits(w, ln) == 224


def test_huffman_dyadic_and_uniform():
    w = np.zeros(256, np.uint64)
    w[:5] = [8, 4, 2, 1, 1]                    # p = 1/2, 1/4, 1/8, 1/16, 1/16
    assert list(oracle.huffman_lengths(w)[:5]) == [1, 2, 3, 4, 4]
    for k in range(1, 9):                      # 2^k equal weights -> all length k
        w = np.zeros(256, np.uint64)
        w[: 2 ** k] = 7
        ln = oracle.huffman_lengths(w)
        assert (ln[: 2 ** k] == k).all() and (ln[2 ** k:] == 0).all()


def test_huffman_single_and_absent_symbols():
    w = np.zeros(256, np.uint64)
    w[42] = 1000
    ln = oracle.huffman_lengths(w)
    assert ln[42] == 1 and ln.sum() == 1
    cb = oracle.huffman_codebook(w)
    x = np.full(3000, 42, np.uint8)
    e = oracle.encode(x, cb, 1024, 64)
    assert e["total_bits"] == 3000
    assert (oracle.decode(e, cb) == x).all()
    with pytest.raises(oracle.OracleError) as ei:
        oracle.encode(np.array([41], np.uint8), cb, 1024, 64)
    assert ei.value.code == oracle.CODEBOOK


def _brute_force_min_cost(weights):
    """Minimum of sum(w*l) over all length vectors with Kraft sum <= 1, i.e.
    over all prefix codes (Kraft-McMillan)."""
    n = len(weights)
    w = np.array(weights, np.int64)
    best = None
    grid = np.array(list(itertools.product(range(1, n), repeat=n)), np.int64)
    kr = (2.0 ** (-grid)).sum(axis=1)
    ok = kr <= 1.0 + 1e-12
    costs = (grid[ok] * w).sum(axis=1)
    best = int(costs.min())
    return best


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6, 7])
def test_huffman_optimal_against_brute_force(n):
    g = np.random.default_rng(100 + n)
    for trial in range(4):
        wts = g.integers(1, 50, n)
        w = np.zeros(256, np.uint64)
        syms = g.choice(256, n, replace=False)
        w[syms] = wts
        ln = oracle.huffman_lengths(w)
        assert oracle.code_bits(w, ln) == _brute_force_min_cost(list(wts))


def test_huffman_kraft_canonical_and_entropy_bounds(gauss_counts, spike_counts):
    for count in (gauss_counts, spike_counts, np.arange(1, 257).astype(np.uint64)):
        cb = oracle.huffman_codebook(count)
        ln, code = cb["len"], cb["code"]
        assert kraft(ln) == 1                                  # complete code
        words = [bits_of(c, L) for c, L in zip(code, ln) if L]
        assert prefix_free(words)
        # canonical: ordering by (length, byte) equals ordering of the
        # left-aligned code values, and equal-length codes are consecutive
        order = sorted((int(ln[b]), b) for b in range(256) if ln[b])
        vals = [int(code[b]) << (64 - int(ln[b])) for _, b in order]
        assert vals == sorted(vals)
        for (l1, b1), (l2, b2) in zip(order, order[1:]):
            if l1 == l2:
                assert int(code[b2]) == int(code[b1]) + 1
        # source coding theorem: H <= mean length < H + 1
        n = int(count.sum())
        H = oracle.entropy_bits(count)
        mean = oracle.code_bits(count, ln) / n
        assert H <= mean + 1e-12 and mean < H + 1


def test_mean_length_is_entropy_plus_kl(spike_counts):
    # For a complete code, sum p*l = H(P) + D(P || 2^-l): ties code bits,
    # entropy and KL together exactly.
    cb = oracle.huffman_codebook(spike_counts)
    ln = cb["len"].astype(np.int64)
    q = np.where(ln > 0, 2 ** (ln.max() - ln), 0).astype(np.uint64)
    n = int(spike_counts.sum())
    lhs = oracle.code_bits(spike_counts, cb["len"]) / n
    rhs = oracle.entropy_bits(spike_counts) + oracle.kl_bits(spike_counts, q)
    assert abs(lhs - rhs) < 1e-12 * lhs


# --------------------------------------------------------------- figures

def test_entropy_and_kl_closed_forms(gauss_counts):
    assert oracle.entropy_bits(np.full(256, 3, np.uint64)) == pytest.approx(8.0, abs=1e-15)
    one = np.zeros(256, np.uint64)
    one[5] = 9
    assert oracle.entropy_bits(one) == 0.0
    two = np.zeros(256, np.uint64)
    two[[1, 2]] = 11
    assert oracle.entropy_bits(two) == pytest.approx(1.0, abs=1e-15)
    # D(P || P) = 0; D(P || uniform) = 8 - H(P); Gibbs: D >= 0
    assert abs(oracle.kl_bits(gauss_counts, gauss_counts)) < 1e-15
    uni = np.ones(256, np.uint64)
    assert oracle.kl_bits(gauss_counts, uni) == pytest.approx(8.0 - oracle.entropy_bits(gauss_counts), abs=1e-12)
    assert oracle.kl_bits(gauss_counts, np.arange(1, 257).astype(np.uint64)) > 0
    assert oracle.kl_bits(two, one) == float("inf")


# --------------------------------------------------------------- fixed codebook weights

def _golden_shards():
    rows = golden("fixed_codebook_weights.txt")
    weights = {int(r[0]): int(r[1]) for r in rows if r[0] != "shard"}
    shards = [np.array([int(v) for v in r[1:]], np.uint8) for r in rows if r[0] == "shard"]
    return weights, shards


def _shard_counts(shards):
    return [np.bincount(s, minlength=256).astype(np.uint64) for s in shards]


def test_fixed_codebook_weights_worked_example():
    # hand-worked weights of three 8-byte shards (tests/golden): the average
    # PMF times the pooled size, plus one pseudocount per byte value
    weights, shards = _golden_shards()
    expect = np.ones(256, np.uint64)
    for b, w in weights.items():
        expect[b] = w
    got = oracle.fixed_codebook_weights(_shard_counts(shards))
    assert got.dtype == np.uint64 and got.shape == (256,)
    assert (got == expect).all()


def test_fixed_codebook_weights_are_the_average_pmf():
    # Equal-size shards: weight - 1 equals (mean of the shard PMFs) x (total
    # bytes), exactly, for every byte value.  The mean is taken here in
    # rational arithmetic straight from the definition (a PMF per shard, then
    # their average), not by pooling counts.
    g = np.random.default_rng(31)
    shards = [g.integers(0, 256, 4096).astype(np.uint8) for _ in range(5)]
    shards.append(np.full(4096, 7, np.uint8))  # a shard of one repeated byte
    counts = _shard_counts(shards)
    got = oracle.fixed_codebook_weights(counts)
    total = sum(s.size for s in shards)
    for b in range(256):
        mean_pmf = sum(Fraction(int(c[b]), s.size) for c, s in zip(counts, shards)) / len(shards)
        assert Fraction(int(got[b]) - 1) == mean_pmf * total
    # no warm-up data at all: the pseudocount alone, a uniform codebook
    assert (oracle.fixed_codebook_weights([]) == 1).all()


def test_fixed_codebook_weights_catch_planted_slips():
    # the plausible misreadings of the pseudocount and of the averaging give
    # other weights than the worked example, so the two pins above fail on them
    weights, shards = _golden_shards()
    counts = _shard_counts(shards)
    expect = np.ones(256, np.uint64)
    for b, w in weights.items():
        expect[b] = w
    per_shard = sum(c + 1 for c in counts)                             # +1 per shard
    only_absent = np.where(sum(counts) == 0, 1, sum(counts)).astype(np.uint64)  # +1 only to absent bytes
    float_mean = np.floor(sum(c.astype(np.float64) / 8 for c in counts) / 3 * 256 + 1)  # PMFs averaged as floats
    for slip in (per_shard, only_absent, float_mean):
        assert not (np.asarray(slip, np.uint64) == expect).all()
    # and the codebooks differ too: a slip changes the code lengths
    good = oracle.huffman_codebook(expect)["len"]
    assert not (oracle.huffman_codebook(np.asarray(per_shard, np.uint64))["len"] == good).all()


# --------------------------------------------------------------- adapted QLC

def test_search_space_reduction_matches_all_orderings(spike_counts):
    # the search keeps only non-decreasing widths; all 9^8 orderings give the
    # same optimum (exchange argument, checked exhaustively)
    w, cost = oracle.qlc_search(spike_counts)
    w_all, cost_all = oracle.qlc_search(spike_counts, nondecreasing_only=False)
    assert cost == cost_all


def test_adapted_qlc_properties(gauss_counts, spike_counts):
    n = int(spike_counts.sum())
    base = oracle.qlc_codebook(spike_counts)
    base_bits = oracle.code_bits(spike_counts, base["len"])
    w, cost = oracle.qlc_search(spike_counts)
    cb = oracle.qlc_codebook(spike_counts, w)
    assert oracle.code_bits(spike_counts, cb["len"]) == cost
    assert cost <= base_bits                         # base is in the search space
    assert len(set(cb["len"].tolist())) <= 4         # still four lengths at most
    assert prefix_free([bits_of(c, L) for c, L in zip(cb["code"], cb["len"])])
    huff = oracle.huffman_codebook(spike_counts)
    hbits = oracle.code_bits(spike_counts, huff["len"])
    # ordering: Shannon >= Huffman >= adapted QLC >= base QLC (compressibility)
    assert oracle.shannon_compressibility(spike_counts) >= oracle.compressibility(hbits, n)
    assert hbits <= cost <= base_bits
    # on the Gaussian law the base layout is already optimal among 4-length codes
    wg, cg = oracle.qlc_search(gauss_counts)
    assert cg == oracle.code_bits(gauss_counts, oracle.qlc_codebook(gauss_counts)["len"])
    # the strict reading (capacity exactly 256) can only be worse
    ws, cs = oracle.qlc_search(spike_counts, require_full=True)
    assert sum(2 ** int(b) for b in ws) == 256 and cs >= cost


# --------------------------------------------------------------- codec

@pytest.mark.parametrize("C,S", [(1024, 64), (4096, 128), (16384, 256), (65536, 1024)])
def test_round_trip_and_bit_count(C, S, gauss_counts):
    x = np_grad(3 * C + 777, (9, C))                 # several chunks + ragged tail
    count = oracle.histogram(x)
    for cb in (oracle.qlc_codebook(count),
               oracle.qlc_codebook(count, oracle.qlc_search(count)[0]),
               oracle.huffman_codebook(oracle.fixed_codebook_weights([count]))):
        e = oracle.encode(x, cb, C, S)
        assert e["total_bits"] == oracle.code_bits(count, cb["len"])
        assert int(e["sub_bits"].astype(np.int64).sum()) == e["total_bits"]
        assert (np.diff(e["chunk_off"].astype(np.int64)) % 16 == 0).all()
        assert (oracle.decode(e, cb) == x).all()


def test_edge_sizes():
    count = np.arange(256, 0, -1).astype(np.uint64)
    for cb in (oracle.qlc_codebook(count), oracle.huffman_codebook(count)):
        for n in (0, 1, 63, 64, 65, 1023, 1024, 1025):
            x = np.random.default_rng(n).integers(0, 256, n).astype(np.uint8)
            e = oracle.encode(x, cb, 1024, 64)
            assert len(e["chunk_off"]) == -(-n // 1024) + 1
            assert (oracle.decode(e, cb) == x).all()


def test_long_codes_round_trip():
    # Fibonacci weights give the deepest Huffman tree: lengths up to 40 bits
    w = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(41):
        w[s] = a
        a, b = b, a + b
    cb = oracle.huffman_codebook(w)
    assert cb["len"].max() == 40
    x = np.arange(41, dtype=np.uint8).repeat(3)
    e = oracle.encode(x, cb, 1024, 64)
    assert (oracle.decode(e, cb) == x).all()


def test_capacity_error():
    x = np.zeros(5000, np.uint8)
    cb = oracle.qlc_codebook(np.ones(256, np.uint64))
    with pytest.raises(oracle.OracleError) as ei:
        oracle.encode(x, cb, 1024, 64, cap=100)
    assert ei.value.code == oracle.CAPACITY


def test_corruption_is_detected_or_changes_output():
    x = np_gauss(5000, (7, 1), 1.0)[0]
    count = oracle.histogram(x)
    for cb in (oracle.qlc_codebook(count), oracle.huffman_codebook(count)):
        e = oracle.encode(x, cb, 1024, 64)
        g = np.random.default_rng(5)
        for _ in range(20):
            bad = dict(e)
            bad["payload"] = e["payload"].copy()
            bad["payload"][g.integers(0, e["payload"].size)] ^= np.uint8(1 << int(g.integers(0, 8)))
            try:
                y = oracle.decode(bad, cb)
            except oracle.OracleError as err:
                assert err.code == oracle.CORRUPT
            else:
                assert not (y == x).all()


# --------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(spike_counts):
    """Plant typical slips in oracle outputs and check a pin fails."""
    cb = oracle.huffman_codebook(spike_counts)
    ln = cb["len"].copy()
    # a dropped level (one length one too short) breaks Kraft
    i = int(np.argmax(ln))
    ln_bad = ln.copy()
    ln_bad[i] -= 1
    assert kraft(ln_bad) > 1
    # a swapped pair of lengths loses optimality (cost rises)
    j, k = int(np.argmax(spike_counts)), int(np.argmin(np.where(ln > 0, spike_counts, 2**63)))
    ln_sw = ln.copy()
    ln_sw[j], ln_sw[k] = ln[k], ln[j]
    assert oracle.code_bits(spike_counts, ln_sw) > oracle.code_bits(spike_counts, ln)
    # an off-by-one in the rank order changes the QLC cost
    base = oracle.qlc_codebook(spike_counts)
    r, br = oracle.rank(spike_counts)
    ln_q = base["len"].copy()
    a, b = br[39], br[40]                            # last 6-bit rank, first 7-bit rank
    assert spike_counts[a] > spike_counts[b]
    ln_q[a], ln_q[b] = ln_q[b], ln_q[a]
    assert oracle.code_bits(spike_counts, ln_q) > oracle.code_bits(spike_counts, base["len"])
    # an escape code that numbers the top exponents from 0 collides with 000
    esc = oracle.escape_codebook(spike_counts)
    words = [bits_of(c, l) for c, l in zip(esc["code"], esc["len"])]
    for b in range(256):
        if ((b >> 3) & 15) == esc["top"][0]:
            words[b] = "000" + words[b][3:]
    assert not prefix_free(words)


# --------------------------------------------------------------- escape code

def exponent_counts(count):
    """Summed counts of the 16 e4m3 exponent values (bits 6-3), test side."""
    e = np.zeros(16, np.uint64)
    for b in range(256):
        e[(b >> 3) & 15] += np.uint64(count[b])
    return e


def test_escape_code_shape_and_kraft(gauss_counts):
    """ZipCCL section 2.B on e4m3: 7 exponents x 16 (sign, mantissa) values
    at 3 + 4 bits, the other 9 exponents at 3 + 4 + 4 bits.  Kraft sum
    7*16/2^7 + 9*16/2^11 = 121/128, prefix-free."""
    cb = oracle.escape_codebook(gauss_counts)
    ln = cb["len"]
    assert (np.bincount(ln, minlength=12)[[7, 11]] == [112, 144]).all()
    assert kraft(ln) == Fraction(7 * 16, 2 ** 7) + Fraction(9 * 16, 2 ** 11) == Fraction(121, 128)
    assert prefix_free([bits_of(c, l) for c, l in zip(cb["code"], ln)])


def test_escape_code_fields(spike_counts):
    """Top 7 = exponents with the largest summed counts (ties to the smaller
    exponent, checked against a sort); a byte's codeword is its exponent's
    code (rank + 1, or 000 and the exponent) then sign then mantissa."""
    cb = oracle.escape_codebook(spike_counts)
    ec = exponent_counts(spike_counts)
    want = sorted(range(16), key=lambda e: (-int(ec[e]), e))[:7]
    assert list(cb["top"]) == want
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        tail = format(s, "b") + format(m, "03b")
        word = bits_of(cb["code"][b], cb["len"][b])
        if e in want:
            assert word == format(want.index(e) + 1, "03b") + tail
        else:
            assert word == "000" + format(e, "04b") + tail


def test_escape_code_ties_and_round_trip():
    """Equal exponent counts rank by exponent value; round trip and bit count
    7 x (top-7 bytes) + 11 x (others) on a tensor with escapes."""
    count = np.ones(256, np.uint64)                      # all exponents tie
    cb = oracle.escape_codebook(count)
    assert list(cb["top"]) == list(range(7))
    x = np_grad(50000, (21, 1))
    cb = oracle.escape_codebook(oracle.histogram(np_gauss(1 << 16, (21, 2))[0]))
    e = (x >> 3) & 15
    n_top = int(np.isin(e, cb["top"]).sum())
    assert 0 < n_top < x.size
    for C, S in ((1024, 64), (16384, 256)):
        enc = oracle.encode(x, cb, C, S)
        assert enc["total_bits"] == 7 * n_top + 11 * (x.size - n_top)
        assert (oracle.decode(enc, cb) == x).all()


def test_escape_of_a_top_exponent_is_corrupt():
    """000 followed by a top-7 exponent codes nothing (that byte has a short
    code): a stream holding it is corrupt."""
    cb = oracle.escape_codebook(np.ones(256, np.uint64))  # top 7 = exponents 0..6
    stream = "000" + "0011" + "0" + "101"                  # escape of exponent 3
    payload = pack_bits(stream)
    payload = np.concatenate([payload, np.zeros((-payload.size) % 16, np.uint8)])
    enc = {"payload": payload, "chunk_off": np.array([0, 16], np.uint64),
           "sub_bits": np.array([11], np.uint16), "n": 1, "C": 1024, "S": 64}
    with pytest.raises(oracle.OracleError) as ei:
        oracle.decode(enc, cb)
    assert ei.value.code == oracle.CORRUPT
    # the same byte through its short code decodes
    ok = "100" + "0" + "101"                               # exponent 3 has rank 3 -> code 100
    payload = pack_bits(ok)
    payload = np.concatenate([payload, np.zeros((-payload.size) % 16, np.uint8)])
    enc.update(payload=payload, sub_bits=np.array([7], np.uint16))
    assert list(oracle.decode(enc, cb)) == [(3 << 3) | 5]


# --------------------------------------------------------------- length-limited Huffman

def brute_min_cost(w, L):
    """Minimum sum(w x len) over all length vectors in [1, L]^n with Kraft <= 1."""
    best = None
    for ls in itertools.product(range(1, L + 1), repeat=len(w)):
        if sum(Fraction(1, 2 ** l) for l in ls) <= 1:
            c = sum(int(a) * b for a, b in zip(w, ls))
            best = c if best is None or c < best else best
    return best


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6])
def test_limited_huffman_optimal_against_brute_force(n):
    g = np.random.default_rng(100 + n)
    for trial in range(6):
        w = np.zeros(256, np.uint64)
        syms = g.choice(256, n, replace=False)
        w[syms] = g.integers(1, [2, 10, 1000][trial % 3] + 1, n)
        lo = max(1, int(np.ceil(np.log2(n))))
        for L in range(lo, 6):
            ln = oracle.huffman_limited_lengths(w, L)
            assert ln.max() <= L and (ln[w == 0] == 0).all()
            assert oracle.code_bits(w, ln) == brute_min_cost(w[syms], L)


def test_limited_huffman_properties(spike_counts):
    w = spike_counts + np.uint64(1)
    full = oracle.huffman_lengths(w)
    prev = None
    for L in range(8, int(full.max()) + 3):
        ln = oracle.huffman_limited_lengths(w, L)
        assert ln.max() <= L and kraft(ln) == 1
        cost = oracle.code_bits(w, ln)
        assert prev is None or cost <= prev                    # a looser limit never costs more
        prev = cost
        if L >= full.max():
            assert cost == oracle.code_bits(w, full)           # no binding limit: Huffman's cost
    # 2^k equal weights under limit k: every length k
    assert (oracle.huffman_limited_lengths(np.full(256, 3, np.uint64), 8) == 8).all()
    # lone symbol: length 1; more symbols than 2^L: no code
    one = np.zeros(256, np.uint64)
    one[9] = 4
    assert oracle.huffman_limited_lengths(one, 3)[9] == 1
    with pytest.raises(oracle.OracleError) as ei:
        oracle.huffman_limited_lengths(np.ones(256, np.uint64), 7)
    assert ei.value.code == oracle.CODEBOOK


def test_limited_huffman_round_trip():
    x = np_grad(60000, (22, 1))
    w = oracle.histogram(x) + np.uint64(1)
    cb = oracle.huffman_limited_codebook(w, 11)
    assert cb["len"].max() <= 11
    enc = oracle.encode(x, cb, 4096, 64)
    assert (oracle.decode(enc, cb) == x).all()
    assert enc["total_bits"] == oracle.code_bits(oracle.histogram(x), cb["len"])


# --------------------------------------------------------------- QLC with 1-3 prefix bits

def qlc_cost_py(sorted_counts, p, widths):
    """Test-side cost of widths for 2^p areas filled in rank order, and its
    capacity and distinct lengths (non-empty areas)."""
    nxt, cost, lens = 0, 0, set()
    for w in widths:
        take = max(0, min(1 << w, 256 - nxt))
        if take:
            lens.add(p + w)
            cost += int(sorted_counts[nxt:nxt + take].sum()) * (p + w)
        nxt += take
    return cost, sum(1 << w for w in widths), len(lens)


@pytest.mark.parametrize("p", [1, 2])
def test_fewer_prefix_bits_search_against_all_vectors(p, spike_counts, gauss_counts):
    """With 2 or 4 areas every width vector can be tried in the test: the
    oracle's non-decreasing search reaches the optimum over all orderings,
    and returns the lexicographically smallest optimal non-decreasing one."""
    A = 1 << p
    for counts in (spike_counts, gauss_counts):
        sc = np.sort(counts.astype(np.int64))[::-1]
        for md in (2, 4):
            allv = [(qlc_cost_py(sc, p, v), v) for v in itertools.product(range(9), repeat=A)]
            ok = [(c, v) for (c, cap, nd), v in allv if cap >= 256 and nd <= md]
            best = min(c for c, _ in ok)
            nd_ok = sorted(v for c, v in ok if c == best and list(v) == sorted(v))
            w, cost = oracle.qlc_search(counts, md, prefix_bits=p)
            assert cost == best
            assert tuple(int(x) for x in w) == nd_ok[0]


@pytest.mark.parametrize("p", [1, 2, 3])
def test_prefix_bits_codes_kraft_and_round_trip(p, gauss_counts):
    w, _ = oracle.qlc_search(gauss_counts, 4, prefix_bits=p)
    cb = oracle.qlc_codebook(gauss_counts, w, prefix_bits=p)
    start, size, covered = oracle.qlc_layout(w, prefix_bits=p)
    assert covered == 256
    assert kraft(cb["len"]) == sum(Fraction(int(z), 2 ** (p + int(x))) for z, x in zip(size, w))
    assert prefix_free([bits_of(c, l) for c, l in zip(cb["code"], cb["len"])])
    # the code of rank r in area k is k's p-bit prefix then r - start[k]
    r, br = oracle.rank(gauss_counts)
    for b in range(256):
        k = int(np.searchsorted(start, r[b], side="right")) - 1
        while size[k] == 0:
            k -= 1
        assert bits_of(cb["code"][b], cb["len"][b]) == format(k, f"0{p}b") + (
            format(int(r[b] - start[k]), f"0{int(w[k])}b") if w[k] else "")
    x = qlc_base_tensor()[:50000]
    enc = oracle.encode(x, cb, 4096, 64)
    assert (oracle.decode(enc, cb) == x).all()
    if p == 3:
        assert (cb["len"] == oracle.qlc_codebook(gauss_counts, w)["len"]).all()


# --------------------------------------------------------------- BF16 exponent escape code

def _bf16_from_f64(x):
    """Test-side cast float64 -> float32 -> BF16 bit patterns, round to
    nearest even on the float32 bits (finite inputs)."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> np.uint64(16)) & np.uint64(1)
    return ((f + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def test_bf16_escape_golden_stream():
    rows = {r[0]: r[1:] for r in golden("bf16_escape_example.txt")}
    top = np.array([int(v) for v in rows["top"]], np.uint8)
    vals = np.array([int(v, 16) for v in rows["values"]], np.uint16)
    expect = np.array([int(v, 16) for v in rows["bytes"]], np.uint8)
    enc = oracle.bf16_escape_encode(vals, top, 1024, 64)
    assert enc["total_bits"] == int(rows["bits"][0])
    assert (enc["payload"] == expect).all()
    assert list(enc["chunk_off"]) == [0, 16] and list(enc["sub_bits"]) == [41]
    assert (oracle.bf16_escape_decode(enc, top) == vals).all()


@pytest.mark.parametrize("sigma", [1.0, 0.02, 3.7e-3, 0.75, 40.0])
def test_bf16_exponent_probs_match_a_sample(sigma):
    # the closed form against the exponent frequencies of 2^22 draws of
    # N(0, sigma^2) rounded to BF16 (five binomial standard errors)
    g = np.random.default_rng(int(sigma * 1e4) + 7)
    x = _bf16_from_f64(sigma * g.standard_normal(1 << 22))
    freq = oracle.bf16_exponent_counts(x).astype(np.float64) / x.size
    p = oracle.bf16_exponent_probs(sigma)
    assert abs(p.sum() - 1.0) < 1e-12
    tol = 5 * np.sqrt(np.maximum(p, 1e-7) * (1 - p) / x.size) + 1e-7
    assert (np.abs(freq - p) <= tol).all()
    # and the sigma table is the sample's top 7 where the ranks are clear
    top_s, top_c = oracle.bf16_top7_from_sigma(sigma), oracle.bf16_top7_from_counts(oracle.bf16_exponent_counts(x))
    assert set(top_s[:5].tolist()) == set(top_c[:5].tolist())
    assert set(top_s.tolist()) == set(top_c.tolist())


def test_bf16_top7_covers_97_percent():
    # the page: the 7 most frequent exponents hold more than 97% of the data;
    # for a Gaussian that holds at every scale (the top 7 from sigma)
    for sigma in 2.0 ** np.linspace(-14, 6, 97):
        p = oracle.bf16_exponent_probs(sigma)
        top = oracle.bf16_top7_from_sigma(sigma)
        assert len(set(top.tolist())) == 7
        assert p[top].sum() > 0.97
        assert p[top[0]] >= p[top[1]] >= p[top[6]]             # rank order
        assert p[top].sum() >= np.sort(p)[-7:].sum() - 1e-15   # the 7 largest
        assert 0 < p[top].sum() - np.sort(p)[-6:].sum()        # a 7th matters


def test_bf16_escape_closed_form_and_round_trip():
    # 16 -> 11 bits for exponents of the table, 19 bits for the others; every
    # one of the 65536 bit patterns round-trips
    top = oracle.bf16_top7_from_sigma(1.0)
    allv = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    g = np.random.default_rng(3)
    x = allv[g.permutation(allv.size)]
    for C, S in ((1024, 64), (16384, 1024)):
        enc = oracle.bf16_escape_encode(x, top, C, S)
        in_top = np.isin((x >> 7) & 0xFF, top)
        assert enc["total_bits"] == 11 * int(in_top.sum()) + 19 * int((~in_top).sum())
        assert (oracle.bf16_escape_decode(enc, top) == x).all()
    # a Gaussian tensor: about 31% smaller (16 -> 11 bits for > 97% of values)
    v = _bf16_from_f64(0.02 * g.standard_normal(1 << 18))
    enc = oracle.bf16_escape_encode(v, oracle.bf16_top7_from_sigma(0.02), 4096, 256)
    bits = enc["total_bits"] / v.size
    assert 11.0 < bits < 11.0 + 8 * 0.03 and 1 - bits / 16 > 0.29


def test_bf16_escaped_table_exponent_is_corrupt():
    top = oracle.bf16_top7_from_sigma(1.0)
    # 000 followed by exponent 127 (in the table) is not a codeword
    s = "000" + format(127, "08b") + "0" + "0000000"
    buf = np.zeros(16, np.uint8)
    buf[:3] = [int((s + "0" * 5)[i:i + 8], 2) for i in range(0, 24, 8)]
    enc = {"payload": buf, "chunk_off": np.array([0, 16], np.uint64), "sub_bits": np.array([19], np.uint16),
           "n": 1, "C": 1024, "S": 64}
    with pytest.raises(oracle.OracleError):
        oracle.bf16_escape_decode(enc, top)
    enc["payload"] = oracle.bf16_escape_encode(np.array([0x3F80], np.uint16), top, 1024, 64)["payload"]
    enc["sub_bits"] = np.array([11], np.uint16)
    assert oracle.bf16_escape_decode(enc, top)[0] == 0x3F80

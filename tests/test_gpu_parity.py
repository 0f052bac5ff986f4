"""CUDA path against the oracle, through the C ABI.

Payload bytes, chunk offsets, sub-block bit counts and total bits must be
bit-exact to the oracle's container, decoded bytes must equal the input, and
every status word must be ECC_OK -- or the documented error for the planted
fault.  Sizes span several tiles, chunks and a ragged tail, and the full-size
workloads are checked on sampled chunks the oracle encodes one by one.
"""
import numpy as np
import pytest

import oracle
from workloads import (dev_grad, grad_warmup, huffman_shards, np_gauss, np_grad, np_zero_spike,
                       qlc_base_tensor)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def u16(t):
    return t.cpu().numpy().view(np.uint16)


CANARY = 64


def check_against_oracle(x, cbb, ocb, C, S, stream=None):
    """Encode on the GPU, compare with the oracle, decode, compare.  Every
    output buffer is followed by canary bytes that must stay untouched, and
    payload bytes past the used size must keep their fill value."""
    n = x.size
    xd = torch.from_numpy(x).cuda() if n else torch.empty(0, dtype=torch.uint8, device="cuda")
    dcb = ecc.to_device(cbb)
    view = ecc.codebook_view(cbb)
    cap = max(16, ecc.max_encoded_bytes(n, C, int(view["max_len"])))
    nch, nsub = ecc.num_chunks(n, C), -(-n // S)
    payload = torch.full((cap + CANARY,), 0xEE, dtype=torch.uint8, device="cuda")
    chunk_off = torch.full((nch + 1 + CANARY,), 0x1234, dtype=torch.int64, device="cuda")
    sub_bits = torch.full((nsub + CANARY,), 0x5A5A, dtype=torch.int16, device="cuda")
    enc = ecc.ecc_encode(xd, dcb, C, S, out=payload[:cap], chunk_off=chunk_off[:nch + 1],
                         sub_bits=sub_bits[:max(nsub, 1)], stream=stream)
    torch.cuda.synchronize()
    assert int(enc.status.item()) == ecc.OK
    ref = oracle.encode(x, ocb, C, S)
    off = u64(enc.chunk_off)
    assert (off == ref["chunk_off"]).all()
    used = int(off[-1])
    pay = payload.cpu().numpy()
    assert (pay[:used] == ref["payload"]).all()
    assert (pay[used:] == 0xEE).all(), "encoder wrote past its payload"
    assert (chunk_off[nch + 1:].cpu().numpy() == 0x1234).all(), "encoder wrote past chunk_off"
    assert (u16(sub_bits)[:nsub] == ref["sub_bits"]).all()
    assert (u16(sub_bits)[max(nsub, 1):] == 0x5A5A).all(), "encoder wrote past sub_bits"
    assert int(u64(enc.total_bits)[0]) == ref["total_bits"]
    out = torch.full((max(n, 16) + CANARY,), 0xA5, dtype=torch.uint8, device="cuda")
    _, st = ecc.ecc_decode(enc, dcb, out=out[:max(n, 16)], stream=stream)
    torch.cuda.synchronize()
    assert int(st.item()) == ecc.OK
    o = out.cpu().numpy()
    assert (o[:n] == x).all()
    assert (o[max(n, 16):] == 0xA5).all(), "decoder wrote past its output"
    if n < 16:
        assert (o[n:16] == 0xA5).all(), "decoder wrote past n"
    return enc


def codebooks(count):
    """(library bytes, oracle codebook) for base QLC, adapted QLC and the
    fixed Huffman code of one histogram."""
    w, _ = oracle.qlc_search(count)
    weights = oracle.fixed_codebook_weights([count])
    return [
        (ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
        (ecc.qlc_build_tables(count, w), oracle.qlc_codebook(count, w)),
        (ecc.huff_build_canonical(weights), oracle.huffman_codebook(weights)),
    ]


# ------------------------------------------------------------------ histogram

@pytest.mark.parametrize("n,offset", [(1 << 20, 0), (1, 0), (17, 3), (123457, 5), ((1 << 22) + 9, 1),
                                      (4111, 0), (4096 * 2 + 16, 7), (3 * 6 * 152 * 4096 + 4096 * 5 + 3, 2)])
def test_histogram_matches_oracle(n, offset):
    x = np_grad(n + offset, (11, n))
    xd = torch.from_numpy(x).cuda()[offset:]            # misaligned start
    cnt = ecc.e4m3_histogram(xd)
    ecc.e4m3_histogram(xd, cnt)                         # accumulates
    torch.cuda.synchronize()
    want = oracle.histogram(x[offset:]) * np.uint64(2)
    assert (cnt.cpu().numpy().view(np.uint64) == want).all()


def test_histogram_one_byte_value():
    """Every byte equal: all lanes of every counting step hit the same bin."""
    x = np.full((1 << 26) + 5, 0x38, np.uint8)
    cnt = ecc.e4m3_histogram(torch.from_numpy(x).cuda()[1:])
    torch.cuda.synchronize()
    want = np.zeros(256, np.uint64)
    want[0x38] = x.size - 1
    assert (cnt.cpu().numpy().view(np.uint64) == want).all()


def test_histogram_zero_spike():
    x = np_zero_spike(1 << 22, (3, 7))
    cnt = ecc.e4m3_histogram(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert (cnt.cpu().numpy().view(np.uint64) == oracle.histogram(x)).all()


# ------------------------------------------------------------------ workloads

def test_qlc_base_round_trip_workload():
    """2^20 bytes of E4M3(N(0,1)); ranks from this tensor's own histogram,
    computed on the GPU; identity and bits == sum(count x len)."""
    x = qlc_base_tensor()
    cnt = ecc.e4m3_histogram(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    count = cnt.cpu().numpy().view(np.uint64)
    assert (count == oracle.histogram(x)).all()
    cbb = ecc.qlc_build_tables(count)
    enc = check_against_oracle(x, cbb, oracle.qlc_codebook(count), 16384, 256)
    assert int(u64(enc.total_bits)[0]) == oracle.code_bits(count, oracle.qlc_codebook(count)["len"])


def test_single_stage_huffman_workload():
    """Fixed codebook from warm-up shards (pooled counts + 1), applied to
    fresh shards of the same sigma law; 16 KiB chunks."""
    warm = [oracle.histogram(x) for x, _ in huffman_shards(4, 1 << 20)]
    weights = oracle.fixed_codebook_weights(warm)
    cbb = ecc.huff_build_canonical(weights)
    ocb = oracle.huffman_codebook(weights)
    for x, sigma in huffman_shards(2, 1 << 22, fresh=True):
        check_against_oracle(x, cbb, ocb, 16384, 256)


def test_zero_spike_workload():
    x = np_zero_spike((1 << 22) + 4321, (3, 0))
    count = oracle.histogram(x)
    for cbb, ocb in codebooks(count):
        check_against_oracle(x, cbb, ocb, 16384, 256)


@pytest.mark.parametrize("C", [4096, 16384, 65536])
def test_grad_workload_chunk_sweep(C):
    warm = [oracle.histogram(grad_warmup(i, 1 << 20)) for i in range(2)]
    pooled = oracle.fixed_codebook_weights(warm)
    x = np_grad((1 << 22) + 77, (4, 0))
    S = ecc.default_subblock(C)
    for cbb, ocb in [(ecc.qlc_build_tables(pooled), oracle.qlc_codebook(pooled)),
                     (ecc.huff_build_canonical(pooled), oracle.huffman_codebook(pooled))]:
        check_against_oracle(x, cbb, ocb, C, S)


@pytest.mark.parametrize("C,S", [(1024, 64), (1024, 1024), (2048, 64), (4096, 128), (8192, 512), (65536, 64)])
def test_chunk_and_subblock_shapes(C, S):
    x = np_gauss(5 * C + 333, (12, C), 1.0)[0]
    count = oracle.histogram(x)
    for cbb, ocb in codebooks(count)[::2]:
        check_against_oracle(x, cbb, ocb, C, S)


@pytest.mark.parametrize("C,S", [(65536, 256), (65536, 128), (65536, 512), (65536, 1024), (32768, 64),
                                 (16384, 64)])
def test_decode_in_pieces(C, S):
    """A chunk of more sub-blocks than one warp stages (32 x streams per
    lane, at most 16384 symbols) is decoded in pieces, one warp each.  Last
    chunks end inside the first piece, on a piece boundary and inside a later
    piece (with a partial sub-block); uniform bytes under a Huffman code fitted
    to a Gaussian give pieces too long for the stage (decoded 32 sub-blocks at
    a time, or from global memory)."""
    x = np_gauss(3 * C, (15, C), 1.0)[0]
    count = oracle.histogram(x)
    books = [(ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
             (ecc.huff_build_canonical(count + np.uint64(1)), oracle.huffman_codebook(count + np.uint64(1)))]
    g = np.random.default_rng(C + S)
    for n in (C - 1, 2 * C + C // 2, 2 * C + C // 4 + 5, 2 * C + 3 * C // 4 + S // 2 + 1):
        y = x[:n].copy()
        for cbb, ocb in books:
            check_against_oracle(y, cbb, ocb, C, S)
    u = g.integers(0, 256, 2 * C + 3 * C // 4 + 7).astype(np.uint8)
    check_against_oracle(u, *books[1], C, S)


@pytest.mark.parametrize("C,S", [(1024, 64), (1024, 1024), (2048, 128), (4096, 64), (4096, 1024), (8192, 256)])
def test_encode_in_groups(C, S):
    """Chunks smaller than 16384 symbols are encoded in groups of
    consecutive chunks (one look-back word and one output offset a group):
    tensors ending in a group's first chunk, on a group boundary, one chunk
    short of it and in a partial chunk of a partial group; a rare-byte mix so
    that some segments take the one-by-one and exact paths."""
    seg = max(min(C, 2048), S, 512)    # a group: 8 segments of this many symbols
    G = 8 // (C // seg)                 # chunks a group
    x = np_gauss(5 * 16384, (17, C), 1.0)[0]
    g = np.random.default_rng(C + S)
    m = g.random(x.size) < 0.02
    x[m] = g.integers(0, 256, int(m.sum()))
    count = oracle.histogram(x)
    books = [(ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
             (ecc.huff_build_canonical(count + np.uint64(1)), oracle.huffman_codebook(count + np.uint64(1)))]
    for n in (C // 2 + 3, 2 * G * C, (3 * G - 1) * C, 3 * G * C + 2 * C + 77):
        for cbb, ocb in books:
            check_against_oracle(x[:n].copy(), cbb, ocb, C, S)


@pytest.mark.parametrize("C,S", [(32768, 64), (32768, 1024), (65536, 256), (65536, 1024)])
def test_encode_split_chunks(C, S):
    """Chunks of more than 16384 symbols are coded in units of 16384 symbols
    on different CTAs: each unit starts at the bit where the chunk's earlier
    units end, and the word two units share is handed from one to the next.
    Tensors ending inside a unit, on a unit boundary and one symbol past it;
    a chunk of rare bytes whose units outgrow the stage (the whole chunk is
    left to the deferred pass) between ordinary chunks, and ending inside
    that chunk."""
    x = np_gauss(3 * C, (18, C), 1.0)[0]
    count = oracle.histogram(x)
    w = count + np.uint64(1)
    books = [(ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
             (ecc.huff_build_canonical(w), oracle.huffman_codebook(w))]
    for n in (16384 + 5, 16384, 16385, C + 3 * 16384 - 1, 2 * C + 16384 + 1, 3 * C):
        for cbb, ocb in books:
            check_against_oracle(x[:n].copy(), cbb, ocb, C, S)
    rare = np.argsort(w)[:8].astype(np.uint8)        # the longest Huffman codes
    y = x.copy()
    y[C:2 * C] = np.random.default_rng(C).choice(rare, C)
    assert ecc.codebook_view(books[1][0])["len"][rare].astype(int).min() > 11
    check_against_oracle(y, *books[1], C, S)
    check_against_oracle(y[:C + 777].copy(), *books[1], C, S)
    # one unit of rare bytes: the chunk's first unit, or its last
    for lo in (C, 2 * C - 16384):
        z = x.copy()
        z[lo:lo + 16384] = np.random.default_rng(lo).choice(rare, 16384)
        check_against_oracle(z, *books[1], C, S)


def test_corrupt_pieces_are_flagged():
    """Pieces of a 64 KiB chunk: a sub-block count raised in one piece, or
    moved from one piece to the next, is corrupt (the streams no longer end
    where their counts say)."""
    x = np_gauss(3 * 65536, (16, 0), 1.0)[0]
    count = oracle.histogram(x)
    for cbb in (ecc.qlc_build_tables(count), ecc.huff_build_canonical(count + 1)):
        dcb = ecc.to_device(cbb)
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), dcb, 65536, 256)
        torch.cuda.synchronize()
        assert int(enc.status.item()) == ecc.OK
        for j, d in ((70, 1), (255, -1), (300, 3)):
            sb = enc.sub_bits.clone()
            sb[j] += d
            out, st = ecc.ecc_decode(ecc.Encoded(enc.payload, enc.chunk_off, sb, enc.total_bits, enc.status,
                                                 enc.n, enc.C, enc.S), dcb)
            torch.cuda.synchronize()
            assert int(st.item()) == ecc.ERR_CORRUPT, (j, d)
        sb = enc.sub_bits.clone()
        sb[63] -= 2
        sb[64] += 2
        out, st = ecc.ecc_decode(ecc.Encoded(enc.payload, enc.chunk_off, sb, enc.total_bits, enc.status,
                                             enc.n, enc.C, enc.S), dcb)
        torch.cuda.synchronize()
        assert int(st.item()) == ecc.ERR_CORRUPT


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 63, 64, 65, 4095, 4096, 4097, 16383, 16385])
def test_edge_sizes(n):
    x = np.random.default_rng(n).integers(0, 256, n).astype(np.uint8)
    count = np.arange(256, 0, -1).astype(np.uint64)
    for cbb, ocb in [(ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
                     (ecc.huff_build_canonical(count), oracle.huffman_codebook(count))]:
        check_against_oracle(x, cbb, ocb, 1024 if n < 5000 else 4096, 64)


def test_single_symbol_tensor():
    x = np.full(70000, 0x38, np.uint8)
    w = np.zeros(256, np.uint64)
    w[0x38] = 5
    check_against_oracle(x, ecc.huff_build_canonical(w), oracle.huffman_codebook(w), 16384, 256)
    count = oracle.histogram(x)
    check_against_oracle(x, ecc.qlc_build_tables(count), oracle.qlc_codebook(count), 16384, 256)


def test_all_256_symbols_and_worst_case_qlc():
    # every byte present, and a chunk of only the rarest (11-bit) ranks
    x = np.concatenate([np.arange(256, dtype=np.uint8).repeat(40), np.full(20000, 255, np.uint8)])
    count = np.arange(256, 0, -1).astype(np.uint64)
    check_against_oracle(x, ecc.qlc_build_tables(count), oracle.qlc_codebook(count), 16384, 256)


@pytest.mark.parametrize("book", ["huffman", "qlc_adapted"])
def test_runs_of_a_short_code(book):
    """92% of the bytes are one value (a 1-bit Huffman code, a 3-bit adapted
    QLC code): many 16-symbol groups take less than a 32-bit word, so
    several coding lanes end inside one word, also across the rounds of a
    warp's segment -- every bit of such shared words must survive."""
    g = np.random.default_rng(17)
    n = (1 << 21) + 4099
    x = np.zeros(n, np.uint8)
    m = g.random(n) < 0.08
    x[m] = g.integers(1, 256, int(m.sum()))
    count = oracle.histogram(x)
    if book == "huffman":
        cbb, ocb = ecc.huff_build_canonical(count + np.uint64(1)), oracle.huffman_codebook(count + np.uint64(1))
    else:
        w, _ = oracle.qlc_search(count)
        cbb, ocb = ecc.qlc_build_tables(count, w), oracle.qlc_codebook(count, w)
    for C, S in ((16384, 256), (4096, 1024), (1024, 64)):
        check_against_oracle(x, cbb, ocb, C, S)


def test_long_codes_take_the_slow_paths():
    # Fibonacci weights: codes up to 40 bits; a tensor of the rare symbols
    # expands ~5x, past the encoder's staging buffer and the decoder's
    w = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(41):
        w[s] = a
        a, b = b, a + b
    cbb, ocb = ecc.huff_build_canonical(w), oracle.huffman_codebook(w)
    assert ecc.codebook_view(cbb)["max_len"] == 40
    g = np.random.default_rng(3)
    rare = g.integers(0, 12, 40000).astype(np.uint8)          # lengths 29..40
    mixed = g.choice(41, 50000, p=w[:41] / w[:41].sum()).astype(np.uint8)
    for x in (rare, mixed, np.concatenate([mixed, rare])):
        check_against_oracle(x, cbb, ocb, 4096, 64)


def test_pairs_past_32_bits_with_codes_of_at_most_31():
    """Fibonacci weights on 30 bytes: codes of 1..29 bits.  Rare bytes drawn
    often enough that many 16-symbol groups hold a pair longer than 32 bits
    (the table's pair join fails) while every single code fits 31 bits: such
    groups are coded one code at a time from the table."""
    w = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(30):
        w[s] = a
        a, b = b, a + b
    cbb, ocb = ecc.huff_build_canonical(w), oracle.huffman_codebook(w)
    assert ecc.codebook_view(cbb)["max_len"] == 29
    g = np.random.default_rng(29)
    p = 0.93 * (w[:30] / w[:30].sum()) + 0.07 / 30
    x = g.choice(30, (1 << 20) + 333, p=p / p.sum()).astype(np.uint8)
    L = ocb["len"][x].astype(np.int64)
    pairs = L[: (x.size // 2) * 2].reshape(-1, 2).sum(axis=1)
    assert (pairs > 32).mean() > 0.002
    for C, S in ((16384, 256), (4096, 64), (1024, 64)):
        check_against_oracle(x, cbb, ocb, C, S)


# ------------------------------------------------------------------ errors

@pytest.mark.parametrize("C", [4096, 16384, 65536])
def test_capacity_error_reports_needed_size(C):
    """A payload buffer too small: ECC_ERR_CAPACITY, chunk_off still holds
    the sizes the payload needs, and no byte past out_cap is written (the
    buffer is a view of a larger one whose tail is a canary), whether the
    buffer is far too small or 16 bytes short."""
    x = np_gauss(3 * 65536 + 12345, (13, 0), 1.0)[0]
    count = oracle.histogram(x)
    cbb = ecc.qlc_build_tables(count)
    dcb = ecc.to_device(cbb)
    ref = oracle.encode(x, oracle.qlc_codebook(count), C, 256)
    need = int(ref["chunk_off"][-1])
    for cap in (4096, need - 16):
        big = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), dcb, C, 256, out=big[:cap])
        torch.cuda.synchronize()
        assert int(enc.status.item()) == ecc.ERR_CAPACITY, cap
        assert (u64(enc.chunk_off) == ref["chunk_off"]).all()
        assert bool((big[cap:] == 0xA5).all()), cap


@pytest.mark.parametrize("n,where", [(20, 12), (40000, 20000), (1 << 20, (1 << 20) - 5)])
def test_uncoded_byte_is_a_codebook_error(n, where):
    """A byte the codebook does not code is reported, whether it falls in a
    partial last group, in the middle of full groups, or near the end."""
    w = np.zeros(256, np.uint64)
    w[:10] = 1
    x = (np.arange(n) % 10).astype(np.uint8)
    x[where] = 200
    for C in (1024, 16384, 65536):
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), ecc.to_device(ecc.huff_build_canonical(w)), C, 64)
        torch.cuda.synchronize()
        assert int(enc.status.item()) == ecc.ERR_CODEBOOK


def test_unit_of_uncoded_bytes_is_a_codebook_error():
    """A whole unit of 16384 bytes the codebook does not code (zero bits:
    the unit shares its one word with both neighbours) inside a chunk of
    65536 symbols, or as a whole chunk of 16384: reported, and the other
    chunks are still placed as the oracle places them."""
    w = np.zeros(256, np.uint64)
    w[:10] = 1
    x = (np.arange(4 * 65536 + 77) % 10).astype(np.uint8)
    x[65536 + 16384:65536 + 32768] = 200
    cbb = ecc.huff_build_canonical(w)
    for C in (16384, 65536):
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), ecc.to_device(cbb), C, 64)
        torch.cuda.synchronize()
        assert int(enc.status.item()) == ecc.ERR_CODEBOOK
        y = x.copy()
        y[65536 + 16384:65536 + 32768] = 0
        ref = oracle.encode(y, oracle.huffman_codebook(w), C, 64)
        off = u64(enc.chunk_off)
        lens = np.diff(off)
        rl = np.diff(ref["chunk_off"])
        bad = (65536 + 16384) // C
        # chunks without the uncoded bytes keep their sizes
        keep = [c for c in range(lens.size) if not (bad <= c < bad + max(1, 16384 // C))]
        assert (lens[keep] == rl[keep]).all()


def test_bad_codebook_magic():
    cbb = ecc.qlc_build_tables(np.ones(256, np.uint64)).copy()
    cbb[:4] = 0
    x = np.zeros(5000, np.uint8)
    enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), ecc.to_device(cbb), 1024, 64)
    torch.cuda.synchronize()
    assert int(enc.status.item()) == ecc.ERR_CODEBOOK


def test_corrupt_streams_are_flagged():
    x = np_gauss(200000, (14, 0), 1.0)[0]
    count = oracle.histogram(x)
    for cbb in (ecc.qlc_build_tables(count), ecc.huff_build_canonical(count + 1)):
        dcb = ecc.to_device(cbb)
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), dcb, 16384, 256)
        torch.cuda.synchronize()
        used = int(u64(enc.chunk_off)[-1])
        g = np.random.default_rng(1)
        for _ in range(10):                     # bit flips in the payload
            bad = ecc.Encoded(enc.payload.clone(), enc.chunk_off, enc.sub_bits, enc.total_bits, enc.status,
                              enc.n, enc.C, enc.S)
            pos = int(g.integers(0, used))
            bad.payload[pos] ^= int(1 << int(g.integers(0, 8)))
            out, st = ecc.ecc_decode(bad, dcb)
            torch.cuda.synchronize()
            assert int(st.item()) == ecc.ERR_CORRUPT or not torch.equal(out[:x.size].cpu(), torch.from_numpy(x))
        # offsets past the payload, and a wrong sub-block count
        off = enc.chunk_off.clone()
        off[3] = int(used) + 4096
        out, st = ecc.ecc_decode(ecc.Encoded(enc.payload, off, enc.sub_bits, enc.total_bits, enc.status,
                                             enc.n, enc.C, enc.S), dcb)
        torch.cuda.synchronize()
        assert int(st.item()) == ecc.ERR_CORRUPT
        sb = enc.sub_bits.clone()
        sb[5] += 1
        out, st = ecc.ecc_decode(ecc.Encoded(enc.payload, enc.chunk_off, sb, enc.total_bits, enc.status,
                                             enc.n, enc.C, enc.S), dcb)
        torch.cuda.synchronize()
        assert int(st.item()) == ecc.ERR_CORRUPT


def test_qlc_code_of_an_empty_area_is_corrupt():
    """Widths (8, 0, ..., 0): area 0 holds every rank, areas 1..7 are empty,
    so a code whose 3-bit prefix is not 000 is no code; planting one in a
    sub-block must flag the stream, in every decoder path."""
    g = np.random.default_rng(23)
    x = g.integers(0, 256, 1 << 16).astype(np.uint8)
    count = oracle.histogram(x)
    cbb = ecc.qlc_build_tables(count, (8, 0, 0, 0, 0, 0, 0, 0))
    ocb = oracle.qlc_codebook(count, (8, 0, 0, 0, 0, 0, 0, 0))
    check_against_oracle(x, cbb, ocb, 16384, 256)
    dcb = ecc.to_device(cbb)
    for C, S in ((16384, 256), (4096, 64), (1024, 1024)):
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), dcb, C, S, max_len=11)
        torch.cuda.synchronize()
        off = u64(enc.chunk_off)
        bad = ecc.Encoded(enc.payload.clone(), enc.chunk_off, enc.sub_bits, enc.total_bits, enc.status,
                          enc.n, enc.C, enc.S)
        bad.payload[int(off[2])] |= 0x80  # chunk 2, sub-block 0: its first code now has prefix 1xx
        out, st = ecc.ecc_decode(bad, dcb)
        torch.cuda.synchronize()
        assert int(st.item()) == ecc.ERR_CORRUPT


@pytest.mark.parametrize("law", ["gauss", "spike", "grad"])
def test_escape_code_workloads(law):
    """The ZipCCL-style escape code (7- and 11-bit codes from the e4m3
    exponent) through the same encoder and the table decoder, with the
    codebook fixed from a warm-up tensor of the same law, so that the tensor
    coded also holds escaped exponents."""
    n = (1 << 20) + 777
    if law == "gauss":
        warm, x = np_gauss(1 << 18, (31, 1))[0], np_gauss(n, (31, 2))[0]
    elif law == "spike":
        warm, x = np_zero_spike(1 << 18, (31, 3)), np_zero_spike(n, (31, 4))
    else:
        warm, x = np_grad(1 << 18, (31, 5)), np_grad(n, (31, 6))
    count = oracle.histogram(warm)
    cbb, ocb = ecc.escape_build_tables(count), oracle.escape_codebook(count)
    assert not np.isin((x >> 3) & 15, ocb["top"]).all()
    for C, S in ((16384, 256), (4096, 64), (1024, 1024)):
        check_against_oracle(x, cbb, ocb, C, S)


@pytest.mark.parametrize("L", [11, 14])
def test_limited_huffman_workloads(L):
    """Length-limited canonical Huffman (package-merge) through the same
    encoder and the table decoder: with L = 14 every code resolves from the
    first-level table."""
    n = (1 << 20) + 4099
    for warm, x in ((np_grad(1 << 20, (32, 1)), np_grad(n, (32, 2))),
                    (np_zero_spike(1 << 18, (32, 3)), np_zero_spike(n, (32, 4)))):
        w = oracle.histogram(warm) + np.uint64(1)
        cbb, ocb = ecc.huff_build_limited(w, L), oracle.huffman_limited_codebook(w, L)
        assert int(ecc.codebook_view(cbb)["max_len"]) <= L
        for C, S in ((16384, 256), (4096, 64)):
            check_against_oracle(x, cbb, ocb, C, S)


@pytest.mark.parametrize("p", [1, 2])
def test_prefix_bits_qlc_workloads(p):
    """QLC with 2 or 4 areas (searched widths, at most 4 lengths) through the
    same encoder and the table decoder."""
    n = (1 << 20) + 12345
    for warm, x in ((np_grad(1 << 20, (33, 1)), np_grad(n, (33, 2))),
                    (np_zero_spike(1 << 18, (33, 3)), np_zero_spike(n, (33, 4)))):
        count = oracle.histogram(warm)
        w, _ = oracle.qlc_search(count, 4, prefix_bits=p)
        cbb, ocb = ecc.gqlc_build_tables(count, w, p), oracle.qlc_codebook(count, w, prefix_bits=p)
        for C, S in ((16384, 256), (4096, 64)):
            check_against_oracle(x, cbb, ocb, C, S)


def test_escape_of_a_top_exponent_is_corrupt():
    """000 followed by a top-7 exponent is no codeword: planting one at the
    start of a sub-block flags the stream."""
    g = np.random.default_rng(41)
    x = g.integers(0, 256, 1 << 16).astype(np.uint8)
    count = np.ones(256, np.uint64)                        # top 7 = exponents 0..6
    cbb, ocb = ecc.escape_build_tables(count), oracle.escape_codebook(count)
    check_against_oracle(x, cbb, ocb, 16384, 256)
    dcb = ecc.to_device(cbb)
    for C, S in ((16384, 256), (4096, 64)):
        enc = ecc.ecc_encode(torch.from_numpy(x).cuda(), dcb, C, S, max_len=11)
        torch.cuda.synchronize()
        off = u64(enc.chunk_off)
        bad = ecc.Encoded(enc.payload.clone(), enc.chunk_off, enc.sub_bits, enc.total_bits, enc.status,
                          enc.n, enc.C, enc.S)
        bad.payload[int(off[1])] = 0b00000110              # chunk 1 starts 000 0011 0..: escape of exponent 3
        out, st = ecc.ecc_decode(bad, dcb)
        torch.cuda.synchronize()
        assert int(st.item()) == ecc.ERR_CORRUPT


def test_bounded_wait_times_out():
    """The look-back wait gives up and reports ECC_ERR_TIMEOUT when no
    predecessor ever publishes (nothing here sets the flags)."""
    flags = torch.zeros(64, dtype=torch.int64, device="cuda")
    prefix = torch.zeros(1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ecc.ecc_selftest_wait(flags, 40, 123, 20_000_000, prefix, status)      # 20 ms limit
    torch.cuda.synchronize()
    assert int(status.item()) == ecc.ERR_TIMEOUT
    # with every predecessor published it returns their sum, no timeout
    def word(state, value):                  # (state << 62) | value as int64
        return int(np.array([(state << 62) | value], np.uint64).view(np.int64)[0])
    flags[:40] = word(1, 16)
    flags[0] = word(2, 16)
    ecc.ecc_selftest_wait(flags, 40, 123, 20_000_000, prefix, status)
    torch.cuda.synchronize()
    assert int(status.item()) == ecc.OK and int(prefix.item()) == 40 * 16
    assert int(flags[40].item()) == word(2, 40 * 16 + 123)


def test_host_argument_errors():
    x = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    dcb = ecc.to_device(ecc.qlc_build_tables(np.ones(256, np.uint64)))
    with pytest.raises(ecc.EccError):
        ecc.ecc_encode(x, dcb, 3000, 64)                 # C not a power of two
    with pytest.raises(ecc.EccError):
        ecc.ecc_encode(x, dcb, 1024, 2048)               # S > C
    with pytest.raises(ecc.EccError):
        ecc.ecc_encode(x[1:], dcb, 1024, 64)             # misaligned input


# ------------------------------------------------------------------ batched

def test_batched_matches_single():
    g = np.random.default_rng(21)
    base_counts = oracle.histogram(qlc_base_tensor())
    spike_counts = oracle.histogram(np_zero_spike(1 << 20, (3, 1)))
    cbs = [ecc.qlc_build_tables(base_counts), ecc.qlc_build_tables(spike_counts, oracle.qlc_search(spike_counts)[0]),
           ecc.huff_build_canonical(base_counts + 1), ecc.huff_build_canonical(spike_counts + 1)]
    ocbs = [oracle.qlc_codebook(base_counts), oracle.qlc_codebook(spike_counts, oracle.qlc_search(spike_counts)[0]),
            oracle.huffman_codebook(base_counts + 1), oracle.huffman_codebook(spike_counts + 1)]
    dcbs = [ecc.to_device(c) for c in cbs]
    xs, items, refs = [], [], []
    for i in range(48):
        size = int(2 ** g.uniform(10, 17)) if i else 0
        law = int(g.integers(0, 3))
        x = (np_gauss(size, (5, i), 1.0)[0] if law == 0 else np_gauss(size, (5, i))[0] if law == 1
             else np_zero_spike(size, (5, i)))
        tag = int(g.integers(0, 4))
        C = [1024, 4096, 16384][i % 3]
        S = ecc.default_subblock(C)
        xd = torch.from_numpy(x).cuda() if size else torch.empty(16, dtype=torch.uint8, device="cuda")
        cap = max(16, ecc.max_encoded_bytes(size, C, int(ecc.codebook_view(cbs[tag])["max_len"])))
        it = {"in": xd, "out": torch.empty(cap, dtype=torch.uint8, device="cuda"), "n": size, "cap": cap,
              "chunk_off": torch.empty(ecc.num_chunks(size, C) + 1, dtype=torch.int64, device="cuda"),
              "sub_bits": torch.empty(max(1, ecc.num_subblocks(size, S)), dtype=torch.int16, device="cuda"),
              "total_bits": torch.empty(1, dtype=torch.int64, device="cuda"), "cb": dcbs[tag],
              "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
              "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": C, "S": S}
        items.append(it)
        xs.append(x)
        refs.append(oracle.encode(x, ocbs[tag], C, S))
    descs = ecc.make_descs(items)
    ws = torch.empty(ecc.batched_workspace_bytes(descs), dtype=torch.uint8, device="cuda")
    t0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    ecc.ecc_encode_batched(descs, ws, t0)
    torch.cuda.synchronize()
    for it, x, ref in zip(items, xs, refs):
        assert int(it["status"].item()) == ecc.OK
        off = u64(it["chunk_off"])
        assert (off == ref["chunk_off"]).all()
        assert (it["out"][:int(off[-1])].cpu().numpy() == ref["payload"]).all()
        assert (u16(it["sub_bits"])[:ref["sub_bits"].size] == ref["sub_bits"]).all()
        assert int(u64(it["total_bits"])[0]) == ref["total_bits"]
        if x.size:
            assert int(it["t_done_ns"].item()) >= int(t0.item()) > 0
    # decode: payload -> fresh output buffers
    ditems = []
    for it, x in zip(items, xs):
        ditems.append({"in": it["out"], "out": torch.empty(max(16, x.size), dtype=torch.uint8, device="cuda"),
                       "n": x.size, "cap": it["cap"], "chunk_off": it["chunk_off"], "sub_bits": it["sub_bits"],
                       "total_bits": None, "cb": it["cb"], "status": torch.full((1,), 99, dtype=torch.int32,
                                                                                  device="cuda"),
                       "t_done_ns": None, "C": it["C"], "S": it["S"]})
    ddescs = ecc.make_descs(ditems)
    ws2 = torch.empty(ecc.batched_workspace_bytes(ddescs), dtype=torch.uint8, device="cuda")
    ecc.ecc_decode_batched(ddescs, ws2)
    torch.cuda.synchronize()
    for it, x in zip(ditems, xs):
        assert int(it["status"].item()) == ecc.OK
        assert (it["out"][:x.size].cpu().numpy() == x).all()


# ------------------------------------------------------------------ full size

@pytest.mark.parametrize("C", [16384, 4096, 65536])
def test_gradient_gib_sampled_parity(C):
    """The 2^30-byte gradient-like tensor in the benchmark's launch setup, at
    each chunk size of its sweep (4 KiB: groups of chunks a unit; 64 KiB: a
    chunk in four units): sampled chunks bit-exact to the oracle, offsets
    consistent, GPU counts equal to the oracle's, total bits == sum(count x
    len), and a lossless round trip on the device."""
    n = 1 << 30
    x = dev_grad(n, (4, 0))
    warm = [oracle.histogram(grad_warmup(i, 1 << 22)) for i in range(2)]
    pooled = oracle.fixed_codebook_weights(warm)
    cnt = ecc.e4m3_histogram(x)
    xh = x.cpu().numpy()
    count = oracle.histogram(xh)
    torch.cuda.synchronize()
    assert (cnt.cpu().numpy().view(np.uint64) == count).all()
    g = np.random.default_rng(99)
    for cbb, ocb in [(ecc.qlc_build_tables(pooled), oracle.qlc_codebook(pooled)),
                     (ecc.huff_build_canonical(pooled), oracle.huffman_codebook(pooled))]:
        dcb = ecc.to_device(cbb)
        S = ecc.default_subblock(C, cbb)  # the benchmark's size for this codebook
        enc = ecc.ecc_encode(x, dcb, C, S, max_len=int(ecc.codebook_view(cbb)["max_len"]))
        out, st = ecc.ecc_decode(enc, dcb)
        torch.cuda.synchronize()
        assert int(enc.status.item()) == ecc.OK and int(st.item()) == ecc.OK
        assert torch.equal(out[:n], x)
        assert int(u64(enc.total_bits)[0]) == oracle.code_bits(count, ocb["len"])
        off = u64(enc.chunk_off)
        sub = u16(enc.sub_bits)
        nch = n // C
        for c in sorted(set(g.integers(0, nch, 12).tolist()) | {0, nch - 1}):
            ref = oracle.encode(xh[c * C:(c + 1) * C], ocb, C, S)
            got = enc.payload[int(off[c]):int(off[c + 1])].cpu().numpy()
            assert int(off[c + 1] - off[c]) == int(ref["chunk_off"][1])
            assert (got == ref["payload"]).all()
            assert (sub[c * (C // S):(c + 1) * (C // S)] == ref["sub_bits"]).all()
        del enc, out
        torch.cuda.empty_cache()

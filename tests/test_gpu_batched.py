"""Many-tensor (batched) encode and decode against the oracle.

Each tensor of a batch is an independent container: its payload, offsets,
sub-block bits and total must equal the oracle's encoding of that tensor
alone, whatever the other tensors, their codebooks and container sizes.
The cases cover every decoder variant the batch's container sizes select
(1, 2 or 4 sub-block streams per lane), the single-slot encoder that
64 KiB chunks need, codebooks interleaved in the caller's order (the call
regroups them), empty tensors, and a tensor with a broken codebook.
"""
import numpy as np
import pytest

import oracle
from workloads import np_gauss, np_zero_spike, qlc_base_tensor

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def u16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def books():
    base = oracle.histogram(qlc_base_tensor())
    spike = oracle.histogram(np_zero_spike(1 << 20, (3, 1)))
    w, _ = oracle.qlc_search(spike)
    host = [ecc.qlc_build_tables(base), ecc.qlc_build_tables(spike, w),
            ecc.huff_build_canonical(base + np.uint64(1)), ecc.huff_build_canonical(spike + np.uint64(1))]
    ocb = [oracle.qlc_codebook(base), oracle.qlc_codebook(spike, w),
           oracle.huffman_codebook(base + np.uint64(1)), oracle.huffman_codebook(spike + np.uint64(1))]
    return host, [ecc.to_device(h) for h in host], ocb


def tensor(size, law, key):
    if law == 0:
        return np_gauss(size, key, 1.0)[0]
    if law == 1:
        return np_gauss(size, key)[0]
    return np_zero_spike(size, key)


def run_batch(books, spec, broken=(), data=None):
    """spec: list of (size, law, tag, C, S).  Tensors listed in `broken` get a
    copy of their codebook with a wrong magic word; data (optional) gives
    the tensors themselves."""
    host, dcbs, ocbs = books
    items, xs, tags = [], [], []
    for i, (size, law, tag, C, S) in enumerate(spec):
        x = data[i] if data is not None else tensor(size, law, (41, i))
        cb = dcbs[tag]
        if i in broken:
            bad = host[tag].copy()
            bad[:4] = 0  # the magic word leads the codebook
            cb = ecc.to_device(bad)
        cap = max(16, ecc.max_encoded_bytes(size, C, int(ecc.codebook_view(host[tag])["max_len"])))
        items.append({"in": torch.from_numpy(x).cuda() if size else torch.empty(16, dtype=torch.uint8, device="cuda"),
                      "out": torch.zeros(cap, dtype=torch.uint8, device="cuda"), "n": size, "cap": cap,
                      "chunk_off": torch.zeros(ecc.num_chunks(size, C) + 1, dtype=torch.int64, device="cuda"),
                      "sub_bits": torch.zeros(max(1, ecc.num_subblocks(size, S)), dtype=torch.int16, device="cuda"),
                      "total_bits": torch.empty(1, dtype=torch.int64, device="cuda"), "cb": cb,
                      "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                      "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": C, "S": S})
        xs.append(x)
        tags.append(tag)
    descs = ecc.make_descs(items)
    ws = torch.empty(ecc.batched_workspace_bytes(descs), dtype=torch.uint8, device="cuda")
    t0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    ecc.ecc_encode_batched(descs, ws, t0)
    torch.cuda.synchronize()
    for i, (it, x, tag) in enumerate(zip(items, xs, tags)):
        if i in broken:
            assert int(it["status"].item()) == ecc.ERR_CODEBOOK
            continue
        assert int(it["status"].item()) == ecc.OK, i
        ref = oracle.encode(x, ocbs[tag], it["C"], it["S"])
        off = u64(it["chunk_off"])
        assert (off == ref["chunk_off"]).all(), i
        assert (it["out"][:int(off[-1])].cpu().numpy() == ref["payload"]).all(), i
        assert (u16(it["sub_bits"])[:ref["sub_bits"].size] == ref["sub_bits"]).all(), i
        assert int(u64(it["total_bits"])[0]) == ref["total_bits"], i
        if x.size:
            assert int(it["t_done_ns"].item()) >= int(t0.item()) > 0
    ditems = []
    for i, (it, x) in enumerate(zip(items, xs)):
        ditems.append({"in": it["out"], "out": torch.zeros(max(16, x.size), dtype=torch.uint8, device="cuda"),
                       "n": x.size, "cap": it["cap"], "chunk_off": it["chunk_off"], "sub_bits": it["sub_bits"],
                       "total_bits": None, "cb": it["cb"],
                       "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                       "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": it["C"], "S": it["S"]})
    ddescs = ecc.make_descs(ditems)
    ws2 = torch.empty(ecc.batched_workspace_bytes(ddescs), dtype=torch.uint8, device="cuda")
    t1 = torch.zeros(1, dtype=torch.int64, device="cuda")
    ecc.ecc_decode_batched(ddescs, ws2, t1)
    torch.cuda.synchronize()
    for i, (it, x) in enumerate(zip(ditems, xs)):
        if i in broken:
            assert int(it["status"].item()) == ecc.ERR_CODEBOOK
            continue
        assert int(it["status"].item()) == ecc.OK, i
        assert (it["out"][:x.size].cpu().numpy() == x).all(), i
        if x.size:
            assert int(it["t_done_ns"].item()) >= int(t1.item()) > 0


def spec_of(n, C, S, seed, lo=10.0, hi=17.0, empty=()):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        size = 0 if i in empty else int(2 ** g.uniform(lo, hi))
        out.append((size, int(g.integers(0, 3)), int(g.integers(0, 4)), C, S))
    return out


@pytest.mark.parametrize("C,S", [(16384, 256), (16384, 128), (4096, 64), (1024, 64)])
def test_batched_uniform_sizes(books, C, S):
    """All tensors with one (C, S): streams per lane 2, 4, 2 and 1; codebooks
    interleaved, so the call's regrouping and run padding are exercised."""
    run_batch(books, spec_of(40, C, S, seed=C + S, empty=(3, 17)))


def test_batched_mixed_sizes(books):
    g = np.random.default_rng(77)
    spec = []
    for i in range(36):
        C = [1024, 2048, 8192, 16384, 32768][i % 5]
        S = [64, 128, 256, 512, 1024][int(g.integers(0, 5))]
        S = min(S, C)
        spec.append((int(2 ** g.uniform(8, 18)), int(g.integers(0, 3)), int(g.integers(0, 4)), C, S))
    run_batch(books, spec)


def test_batched_64k_chunks(books):
    """C = 64 KiB takes the single-slot encoder (two stage slots do not fit)."""
    spec = [(int(s), i % 3, i % 4, 65536, 1024) for i, s in enumerate([70000, 1 << 18, 5, 65536, 200000, 0, 131073])]
    run_batch(books, spec)


def test_batched_broken_codebook(books):
    """One tensor's codebook has a wrong magic word: that tensor alone reports
    ECC_ERR_CODEBOOK, every other tensor is still exact."""
    run_batch(books, spec_of(12, 16384, 256, seed=5), broken=(4,))


def test_batched_one_codebook_many_small(books):
    """Hundreds of small tensors sharing one codebook (a message-sized batch)."""
    spec = [(int(s), 0, 0, 4096, 64) for s in np.random.default_rng(9).integers(1, 20000, 300)]
    run_batch(books, spec)


def test_batched_long_codes(books):
    """N(0, 1) tensors coded with the zero-spike Huffman code (about 12.4 bits
    a symbol, more than a chunk's stage holds at 16 KiB chunks) beside tensors
    with short codes: their chunks are sized and placed by the encoder and
    coded by the deferred pass, and the look-back runs across them."""
    g = np.random.default_rng(23)
    spec = []
    for i in range(24):
        size = int(g.integers(1, 5 * 16384))
        spec.append((size, 0, 3 if i % 2 == 0 else int(g.integers(0, 3)), 16384, 256 if i % 3 else 128))
    run_batch(books, spec)


def test_batched_codes_past_the_second_stage():
    """Fibonacci weights: codes of up to 40 bits.  Chunks of the rarest bytes
    average about 34 bits a symbol, more than the second pass's stages hold
    (32 bits a symbol): its storer warp codes them; chunks of about 20 bits a
    symbol are staged by the second pass; chunks of the common bytes by the
    first."""
    w = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(41):
        w[s] = a
        a, b = b, a + b
    host = [ecc.huff_build_canonical(w)]
    fib = (host, [ecc.to_device(host[0])], [oracle.huffman_codebook(w)])
    g = np.random.default_rng(31)
    rare = g.integers(0, 12, 3 * 16384 + 77).astype(np.uint8)       # lengths 29..40
    middle = g.integers(16, 24, 2 * 16384 + 5).astype(np.uint8)     # lengths 17..24
    common = g.choice(41, 3 * 16384, p=w[:41] / w[:41].sum()).astype(np.uint8)
    data = [common, rare, middle, np.concatenate([middle[:20000], rare[:30000]]), common[:5000]]
    run_batch(fib, [(x.size, 0, 0, 16384, 256) for x in data], data=data)

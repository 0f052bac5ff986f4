"""The index-checked build (-DECC_CHECKED) on small cases at every chunk and
sub-block edge.

In that build the kernels test their shared- and global-memory indices
(encoder regions and payload words, decoder stage reads and output stores),
skip an access out of range and report ECC_ERR_CHECK.  This is the stand-in
for a memory checker: every case must finish with ECC_OK and outputs
bit-exact to the oracle, i.e. no index ever left its buffer.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
from workloads import np_gauss, np_zero_spike

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def eck():
    """A second binding instance over the index-checked library."""
    from lossless_entropy_coding_gb300 import build as ecc_build
    path = ecc_build.build(checked=True)
    spec = importlib.util.spec_from_file_location(
        "ecc_checked", os.path.join(ROOT, "lossless_entropy_coding_gb300", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules["ecc_checked"] = mod  # dataclasses look their module up there
    spec.loader.exec_module(mod)
    mod.LIB_PATH = path
    assert os.path.basename(path) == "libecc_gb300_checked.so"
    return mod


def books(e):
    g = np.random.default_rng(61)
    warm = np.concatenate([np_gauss(1 << 16, (61, 1))[0], g.integers(0, 256, 4096).astype(np.uint8)])
    count = oracle.histogram(warm)
    w2, _ = oracle.qlc_search(count, 4, prefix_bits=2)
    fib = np.zeros(256, np.uint64)
    a, b = 1, 1
    for s in range(40):
        fib[s] = a
        a, b = b, a + b
    return [
        ("qlc", e.qlc_build_tables(count), oracle.qlc_codebook(count)),
        ("huffman", e.huff_build_canonical(count + np.uint64(1)), oracle.huffman_codebook(count + np.uint64(1))),
        ("escape", e.escape_build_tables(count), oracle.escape_codebook(count)),
        ("limited11", e.huff_build_limited(count + np.uint64(1), 11),
         oracle.huffman_limited_codebook(count + np.uint64(1), 11)),
        ("qlc4areas", e.gqlc_build_tables(count, w2, 2), oracle.qlc_codebook(count, w2, prefix_bits=2)),
        ("fibonacci", e.huff_build_canonical(fib), oracle.huffman_codebook(fib)),
    ]


def tensor(n, name, key):
    g = np.random.default_rng(key)
    if name == "fibonacci":  # codes of 1..39 bits: fast, one-by-one and exact paths
        w = np.array([1.0 / 1.6 ** s for s in range(40)])
        return g.choice(40, n, p=w / w.sum()).astype(np.uint8)
    x = np_zero_spike(n, (62, key)) if key % 2 else np_gauss(n, (62, key))[0]
    m = g.random(n) < 0.05
    x[m] = g.integers(0, 256, int(m.sum()))  # rare bytes: long codes and escapes
    return x


def round_trip(e, x, cbb, ocb, C, S):
    n = x.size
    xd = torch.from_numpy(x).cuda()
    dcb = e.to_device(cbb)
    max_len = int(e.codebook_view(cbb)["max_len"])
    enc = e.ecc_encode(xd, dcb, C, S, max_len=max_len)
    y, st = e.ecc_decode(enc, dcb)
    torch.cuda.synchronize()
    assert int(enc.status.item()) == e.OK, ("encode", int(enc.status.item()))
    assert int(st.item()) == e.OK, ("decode", int(st.item()))
    ref = oracle.encode(x, ocb, C, S)
    off = enc.chunk_off.cpu().numpy().view(np.uint64)
    assert (off == ref["chunk_off"]).all()
    assert (enc.payload[:int(off[-1])].cpu().numpy() == ref["payload"]).all()
    assert (y[:n].cpu().numpy() == x).all()


@pytest.mark.parametrize("C,S", [(1024, 64), (4096, 64), (4096, 128), (16384, 256), (16384, 1024),
                                 (65536, 1024), (65536, 256), (32768, 64)])
def test_checked_edges(eck, C, S):
    for name, cbb, ocb in books(eck):
        for k, n in enumerate((1, 17, C - 1, C, C + 1, 3 * C + 5)):
            round_trip(eck, tensor(n, name, 7 * k + C % 97), cbb, ocb, C, S)


def test_checked_batched(eck):
    bk = books(eck)
    g = np.random.default_rng(63)
    items, xs = [], []
    for i in range(24):
        name, cbb, ocb = bk[i % len(bk)]
        C = [1024, 4096, 16384][i % 3]
        S = min(C, [64, 128, 256][i % 3])
        n = int(g.integers(0, 3 * C))
        x = tensor(n, name, 100 + i)
        cap = max(16, eck.max_encoded_bytes(n, C, int(eck.codebook_view(cbb)["max_len"])))
        items.append({"in": torch.from_numpy(x).cuda() if n else torch.empty(16, dtype=torch.uint8, device="cuda"),
                      "out": torch.zeros(cap, dtype=torch.uint8, device="cuda"), "n": n, "cap": cap,
                      "chunk_off": torch.zeros(eck.num_chunks(n, C) + 1, dtype=torch.int64, device="cuda"),
                      "sub_bits": torch.zeros(max(1, eck.num_subblocks(n, S)), dtype=torch.int16, device="cuda"),
                      "total_bits": torch.empty(1, dtype=torch.int64, device="cuda"), "cb": eck.to_device(cbb),
                      "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                      "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": C, "S": S})
        xs.append((x, ocb))
    descs = eck.make_descs(items)
    ws = torch.empty(eck.batched_workspace_bytes(descs), dtype=torch.uint8, device="cuda")
    eck.ecc_encode_batched(descs, ws)
    torch.cuda.synchronize()
    dit = []
    for it, (x, ocb) in zip(items, xs):
        assert int(it["status"].item()) == eck.OK
        ref = oracle.encode(x, ocb, it["C"], it["S"])
        off = it["chunk_off"].cpu().numpy().view(np.uint64)
        assert (off == ref["chunk_off"]).all()
        assert (it["out"][:int(off[-1])].cpu().numpy() == ref["payload"]).all()
        dit.append({"in": it["out"], "out": torch.zeros(max(16, x.size), dtype=torch.uint8, device="cuda"),
                    "n": x.size, "cap": it["cap"], "chunk_off": it["chunk_off"], "sub_bits": it["sub_bits"],
                    "total_bits": None, "cb": it["cb"], "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                    "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": it["C"], "S": it["S"]})
    ddescs = eck.make_descs(dit)
    ws2 = torch.empty(eck.batched_workspace_bytes(ddescs), dtype=torch.uint8, device="cuda")
    eck.ecc_decode_batched(ddescs, ws2)
    torch.cuda.synchronize()
    for it, (x, _) in zip(dit, xs):
        assert int(it["status"].item()) == eck.OK
        assert (it["out"][:x.size].cpu().numpy() == x).all()

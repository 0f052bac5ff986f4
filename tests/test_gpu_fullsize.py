"""Full-size workloads on the GPU, checked on sampled outputs.

Each workload runs at its full size in the launch configuration the
benchmark uses (16 KiB chunks, default sub-blocks, persistent kernels).  The
oracle encodes sampled chunks one by one (a chunk is a container of its own:
same payload bytes, same sub-block bits); everything else is checked through
properties that hold at any size: lossless round trip on the device, device
histogram == oracle histogram, total bits == sum(count x length), offsets
consistent, and the orderings the pages state between the codes.
"""
import numpy as np
import pytest

import oracle
from workloads import (batch_plan, dev_batch_tensor, dev_gauss, dev_zero_spike, np_gauss, np_zero_spike)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402

C = 16384


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def device_counts(x):
    c = ecc.e4m3_histogram(x)
    torch.cuda.synchronize()
    return c.cpu().numpy().view(np.uint64).copy()


def sampled_parity(x_host, enc, ocb, S, chunks):
    off = u64(enc.chunk_off)
    sub = enc.sub_bits.cpu().numpy().view(np.uint16)
    n = x_host.size
    for c in chunks:
        lo, hi = c * C, min(n, (c + 1) * C)
        ref = oracle.encode(x_host[lo:hi], ocb, C, S)
        got = enc.payload[int(off[c]):int(off[c + 1])].cpu().numpy()
        assert int(off[c + 1] - off[c]) == int(ref["chunk_off"][1])
        assert (got == ref["payload"]).all()
        s0 = lo // S
        assert (sub[s0:s0 + ref["sub_bits"].size] == ref["sub_bits"]).all()


def round_trip(x, cbb, S):
    dcb = ecc.to_device(cbb)
    enc = ecc.ecc_encode(x, dcb, C, S, max_len=int(ecc.codebook_view(cbb)["max_len"]))
    out, st = ecc.ecc_decode(enc, dcb)
    torch.cuda.synchronize()
    assert int(enc.status.item()) == ecc.OK and int(st.item()) == ecc.OK
    assert torch.equal(out[:x.numel()], x)
    return enc


def test_zero_spike_full_size():
    """2^28 bytes, 40% zeros + 2*GELU(z): adapted QLC (width search on the
    device histogram) against base QLC and the Huffman code of the same
    PMF."""
    n = 1 << 28
    x = dev_zero_spike(n, (3, 0))
    xh = x.cpu().numpy()
    count = device_counts(x)
    assert (count == oracle.histogram(xh)).all()
    w, cost = ecc.qlc_search_widths(count)
    wo, costo = oracle.qlc_search(count)
    assert (w == wo).all() and cost == costo
    books = [("qlc_base", ecc.qlc_build_tables(count), oracle.qlc_codebook(count)),
             ("qlc_adapted", ecc.qlc_build_tables(count, w), oracle.qlc_codebook(count, w)),
             ("huffman", ecc.huff_build_canonical(count + np.uint64(1)),
              oracle.huffman_codebook(count + np.uint64(1)))]
    bits = {}
    g = np.random.default_rng(3)
    for name, cbb, ocb in books:
        S = ecc.default_subblock(C, cbb)  # each codebook at the size the benchmark codes it with
        enc = round_trip(x, cbb, S)
        bits[name] = int(u64(enc.total_bits)[0])
        assert bits[name] == oracle.code_bits(count, ocb["len"])
        nch = n // C
        sampled_parity(xh, enc, ocb, S, sorted(set(g.integers(0, nch, 6).tolist()) | {0, nch - 1}))
        del enc
    # the ordering the pages report: Huffman >= adapted QLC >= base QLC
    assert bits["huffman"] <= bits["qlc_adapted"] <= bits["qlc_base"]
    shannon = oracle.shannon_compressibility(count)
    assert shannon >= oracle.compressibility(bits["huffman"], n)


def test_single_stage_huffman_full_size():
    """16 warm-up shards of 2^22 bytes -> pooled counts + 1 -> one canonical
    Huffman codebook, applied to 64 fresh shards; per shard the fixed code,
    the shard's own Huffman code and the Shannon bound, and D(shard || avg)."""
    n = 1 << 22
    pooled = torch.zeros(256, dtype=torch.int64, device="cuda")
    for i in range(16):
        x, _ = dev_gauss(n, (2, i))
        ecc.e4m3_histogram(x, pooled)
    torch.cuda.synchronize()
    pooled = pooled.cpu().numpy().view(np.uint64).copy()
    weights = pooled + np.uint64(1)
    cbb = ecc.huff_build_canonical(weights)
    ocb = oracle.huffman_codebook(weights)
    dcb = ecc.to_device(cbb)
    max_len = int(ecc.codebook_view(cbb)["max_len"])
    S = ecc.default_subblock(C, cbb)
    g = np.random.default_rng(2)
    for i in range(64):
        x, sigma = dev_gauss(n, (2, 100 + i))
        enc = ecc.ecc_encode(x, dcb, C, S, max_len=max_len)
        out, st = ecc.ecc_decode(enc, dcb)
        count = device_counts(x)
        assert int(enc.status.item()) == ecc.OK and int(st.item()) == ecc.OK
        assert torch.equal(out[:n], x)
        fixed_bits = int(u64(enc.total_bits)[0])
        assert fixed_bits == oracle.code_bits(count, ocb["len"])
        if i % 8 == 0:
            xh = x.cpu().numpy()
            assert (count == oracle.histogram(xh)).all()
            sampled_parity(xh, enc, ocb, S, [int(g.integers(0, n // C))])
        own = ecc.huff_build_canonical(count)          # per-shard Huffman (exact counts)
        own_bits = ecc.code_bits(count, own)
        assert own_bits == oracle.code_bits(count, oracle.huffman_lengths(count))
        # Shannon >= per-shard Huffman >= fixed codebook (compressibility)
        H = ecc.entropy_bits(count)
        assert abs(H - oracle.entropy_bits(count)) <= 1e-9 * H
        assert H * n <= own_bits * (1 + 1e-12) and own_bits <= fixed_bits
        kl = ecc.kl_bits(count, weights)
        assert kl >= 0 and abs(kl - oracle.kl_bits(count, weights)) <= 1e-9 * max(kl, 1e-12)
        # the fixed code costs exactly cross-entropy-like excess: bits/n - H
        # stays within the KL to the codebook distribution plus one bit
        assert fixed_bits / n - H <= kl + 1.0
        del enc, out


def test_batched_full_size():
    """4096 tensors, sizes log-uniform in [4 KiB, 8 MiB], each from one of
    three laws and tagged with one of four codebooks; one batched encode and
    one batched decode launch."""
    plan = batch_plan(4096)
    # the four codebooks, from warm-up data of each law
    g1 = np_gauss(1 << 22, (5, 1001), 1.0)[0]
    g3 = np_zero_spike(1 << 22, (5, 1003))
    c1, c3 = oracle.histogram(g1), oracle.histogram(g3)
    w3, _ = oracle.qlc_search(c3)
    c2 = np.zeros(256, np.uint64)
    for i in range(4):
        c2 += oracle.histogram(np_gauss(1 << 20, (5, 2000 + i))[0])
    books = [(ecc.qlc_build_tables(c1), oracle.qlc_codebook(c1)),
             (ecc.qlc_build_tables(c3, w3), oracle.qlc_codebook(c3, w3)),
             (ecc.huff_build_canonical(c2 + np.uint64(1)), oracle.huffman_codebook(c2 + np.uint64(1))),
             (ecc.huff_build_canonical(c3 + np.uint64(1)), oracle.huffman_codebook(c3 + np.uint64(1)))]
    dcbs = [ecc.to_device(b) for b, _ in books]
    max_len = [int(ecc.codebook_view(b)["max_len"]) for b, _ in books]
    Sb = [ecc.default_subblock(C, b) for b, _ in books]
    total = sum(s for s, _, _ in plan)
    xin = torch.empty(total + 16 * len(plan), dtype=torch.uint8, device="cuda")
    items, views, off = [], [], 0
    for i, (size, law, tag) in enumerate(plan):
        x = xin[off:off + size]
        dev_batch_tensor(size, law, (5, i), out=x)
        cap = ecc.max_encoded_bytes(size, C, max_len[tag])
        items.append({"in": x, "out": torch.empty(cap, dtype=torch.uint8, device="cuda"), "n": size, "cap": cap,
                      "chunk_off": torch.empty(ecc.num_chunks(size, C) + 1, dtype=torch.int64, device="cuda"),
                      "sub_bits": torch.empty(ecc.num_subblocks(size, Sb[tag]), dtype=torch.int16, device="cuda"),
                      "total_bits": torch.empty(1, dtype=torch.int64, device="cuda"), "cb": dcbs[tag],
                      "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                      "t_done_ns": torch.zeros(1, dtype=torch.int64, device="cuda"), "C": C, "S": Sb[tag]})
        views.append(tag)
        off += (size + 15) // 16 * 16
    descs = ecc.make_descs(items)
    ws = torch.empty(ecc.batched_workspace_bytes(descs), dtype=torch.uint8, device="cuda")
    t0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    ecc.ecc_encode_batched(descs, ws, t0)
    ditems = []
    for it in items:
        ditems.append(dict(it, **{"in": it["out"], "out": torch.empty(it["n"], dtype=torch.uint8, device="cuda"),
                                  "cap": it["cap"], "total_bits": None,
                                  "status": torch.full((1,), 99, dtype=torch.int32, device="cuda"),
                                  "t_done_ns": None}))
    ddescs = ecc.make_descs(ditems)
    ws2 = torch.empty(ecc.batched_workspace_bytes(ddescs), dtype=torch.uint8, device="cuda")
    ecc.ecc_decode_batched(ddescs, ws2)
    torch.cuda.synchronize()
    st_enc = torch.cat([it["status"] for it in items]).cpu().numpy()
    st_dec = torch.cat([it["status"] for it in ditems]).cpu().numpy()
    assert (st_enc == 0).all() and (st_dec == 0).all()
    for it, dit in zip(items, ditems):
        assert torch.equal(dit["out"], it["in"])
    stamps = torch.cat([it["t_done_ns"] for it in items]).cpu().numpy()
    assert (stamps >= int(t0.item())).all()
    # exact bits and sampled oracle parity
    g = np.random.default_rng(5)
    for i in sorted(set(g.integers(0, len(plan), 24).tolist())):
        it, tag = items[i], views[i]
        xh = it["in"].cpu().numpy()
        ocb = books[tag][1]
        assert int(u64(it["total_bits"])[0]) == oracle.code_bits(oracle.histogram(xh), ocb["len"])
        nch = ecc.num_chunks(it["n"], C)
        enc = ecc.Encoded(it["out"], it["chunk_off"], it["sub_bits"], it["total_bits"], it["status"],
                          it["n"], C, it["S"])
        sampled_parity(xh, enc, ocb, it["S"], sorted({0, nch - 1, int(g.integers(0, nch))}))

"""ecc_encode_static -- the encode entry point that allocates nothing.

Some callers cannot allocate device memory on their call path: latency-
critical communication code (cudaMalloc can synchronise the whole device)
and code inside a framework whose allocator owns all device memory.  For
them ecc_encode_static keeps its scratch (ticket and look-back words) in a
file-scope device array of the library.  Here it is called through the C ABI
and must produce exactly what ecc_encode produces, on two calls in a row
(the second call reuses the array the first one left behind).
"""
import ctypes as ct

import numpy as np
import pytest

import oracle
from workloads import np_gauss, np_grad, np_zero_spike

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import lossless_entropy_coding_gb300 as ecc  # noqa: E402


def _encode_static_c_abi(x, dcb, C, S, cap):
    """Direct ctypes call of ecc_encode_static (no workspace argument)."""
    dev = x.device
    n = x.numel()
    out = torch.zeros(cap, dtype=torch.uint8, device=dev)
    off = torch.zeros(ecc.num_chunks(n, C) + 1, dtype=torch.int64, device=dev)
    sub = torch.zeros(max(1, ecc.num_subblocks(n, S)), dtype=torch.int16, device=dev)
    tot = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.full((1,), 77, dtype=torch.int32, device=dev)
    rc = ecc.lib().ecc_encode_static(ct.c_void_p(x.data_ptr()), n, ct.c_void_p(dcb.data_ptr()), C, S,
                                     ct.c_void_p(out.data_ptr()), cap, ct.c_void_p(off.data_ptr()),
                                     ct.c_void_p(sub.data_ptr()), ct.c_void_p(tot.data_ptr()),
                                     ct.c_void_p(st.data_ptr()),
                                     ct.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out, off, sub, tot, st


def _same_as_workspace_encode(x, cbb, C, S):
    dcb = ecc.to_device(cbb)
    max_len = int(ecc.codebook_view(cbb)["max_len"])
    cap = ecc.max_encoded_bytes(x.numel(), C, max_len)
    rc, out, off, sub, tot, st = _encode_static_c_abi(x, dcb, C, S, cap)
    ref = ecc.ecc_encode(x, dcb, C, S, max_len=max_len)
    torch.cuda.synchronize()
    assert rc == ecc.OK
    assert int(st.item()) == ecc.OK and int(ref.status.item()) == ecc.OK
    assert torch.equal(off, ref.chunk_off)
    used = int(off[-1].item())
    assert torch.equal(out[:used], ref.payload[:used])
    assert torch.equal(sub, ref.sub_bits[:sub.numel()])
    assert int(tot.item()) == int(ref.total_bits.item())
    return used


def test_static_encode_matches_workspace_encode_twice():
    x1 = torch.from_numpy(np_gauss((1 << 22) + 4097, (31, 1), 1.0)[0]).cuda()
    x2 = torch.from_numpy(np_zero_spike((1 << 21) + 333, (31, 2))).cuda()
    c1 = ecc.e4m3_histogram(x1).cpu().numpy().view(np.uint64)
    c2 = ecc.e4m3_histogram(x2).cpu().numpy().view(np.uint64)
    # two calls in a row, different sizes and codebooks: the second call must
    # not see the first call's look-back words
    u1 = _same_as_workspace_encode(x1, ecc.qlc_build_tables(c1), 16384, 256)
    u2 = _same_as_workspace_encode(x2, ecc.huff_build_canonical(c2 + np.uint64(1)), 4096, 64)
    assert u1 > 0 and u2 > 0


def test_static_encode_matches_oracle():
    """Against the bit-serial oracle: the container (offsets, payload,
    sub-block bits, total) of a gradient-like tensor with a Huffman code."""
    xh = np_grad((1 << 20) + 77, (31, 3))
    count = oracle.histogram(xh)
    weights = oracle.fixed_codebook_weights([count])
    cbb, ocb = ecc.huff_build_canonical(weights), oracle.huffman_codebook(weights)
    x = torch.from_numpy(xh).cuda()
    dcb = ecc.to_device(cbb)
    C, S = 16384, 256
    rc, out, off, sub, tot, st = _encode_static_c_abi(
        x, dcb, C, S, ecc.max_encoded_bytes(x.numel(), C, int(ecc.codebook_view(cbb)["max_len"])))
    torch.cuda.synchronize()
    assert rc == ecc.OK and int(st.item()) == ecc.OK
    ref = oracle.encode(xh, ocb, C, S)
    o = off.cpu().numpy().view(np.uint64)
    assert (o == ref["chunk_off"]).all()
    assert (out[: int(o[-1])].cpu().numpy() == ref["payload"]).all()
    assert (sub.cpu().numpy().view(np.uint16) == ref["sub_bits"]).all()
    assert int(tot.item()) == ref["total_bits"]


def test_static_encode_large_chunks_and_python_wrapper():
    """Chunks of 65536 symbols are coded in units of 16384 symbols, whose
    words (one per unit, after the chunks' words) also live in the static
    array; the Python wrapper
    ecc.ecc_encode_static is called twice in a row and must equal
    ecc_encode."""
    xh = np_grad((1 << 22) + 1234, (31, 4))
    x = torch.from_numpy(xh).cuda()
    count = ecc.e4m3_histogram(x).cpu().numpy().view(np.uint64)
    for cbb in (ecc.qlc_build_tables(count), ecc.huff_build_canonical(count + np.uint64(1))):
        _same_as_workspace_encode(x, cbb, 65536, 256)
        dcb = ecc.to_device(cbb)
        max_len = int(ecc.codebook_view(cbb)["max_len"])
        ref = ecc.ecc_encode(x, dcb, 65536, 1024, max_len=max_len)
        for _ in range(2):
            got = ecc.ecc_encode_static(x, dcb, 65536, 1024, max_len=max_len)
            torch.cuda.synchronize()
            assert int(got.status.item()) == ecc.OK and int(ref.status.item()) == ecc.OK
            assert torch.equal(got.chunk_off, ref.chunk_off)
            used = int(ref.chunk_off[-1].item())
            assert torch.equal(got.payload[:used], ref.payload[:used])
            assert torch.equal(got.sub_bits, ref.sub_bits)
            assert int(got.total_bits.item()) == int(ref.total_bits.item())


def test_static_encode_rejects_too_many_chunks():
    C = 1024
    n = (ecc.STATIC_MAX_CHUNKS + 1) * C
    x = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dcb = ecc.to_device(ecc.qlc_build_tables(np.ones(256, np.uint64)))
    rc, *_ = _encode_static_c_abi(x, dcb, C, 64, 16)
    assert rc == ecc.ERR_ARG

"""Python binding of libecc_gb300: lossless fixed-codebook coding of e4m3
byte tensors on GB300 (Quad Length Codes and single-stage canonical Huffman).

Argument marshalling only.  Every entry point has the name of the C function
it calls (see include/ecc.h for the contract); PyTorch supplies device memory
and the current CUDA stream.  All coding work runs in the library's CUDA
kernels or its host codebook builders -- there is no other code path: if the
shared library has not been built, importing the binding still works but
every call raises.
"""
from __future__ import annotations

import ctypes as ct
import os
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libecc_gb300.so")

OK, ERR_ARG, ERR_CAPACITY, ERR_CORRUPT, ERR_CODEBOOK, ERR_TIMEOUT, ERR_CUDA, ERR_CHECK = range(8)
FAMILY_QLC, FAMILY_HUFFMAN, FAMILY_ESCAPE = 1, 2, 3
MAX_CODE_LEN = 48
BASE_WIDTHS = (3, 3, 3, 3, 3, 4, 5, 8)

# Layout of ecc_codebook (C struct in include/ecc.h), naturally aligned.
CODEBOOK_DTYPE = np.dtype([
    ("magic", "<u4"), ("family", "<u4"), ("max_len", "<u4"), ("min_len", "<u4"),
    ("n_coded", "<u4"), ("prefix_bits", "<u4"), ("reserved", "<u4", (2,)),
    ("code", "<u8", (256,)), ("first", "<u8", (64,)),
    ("enc_code", "<u4", (256,)), ("enc_mul", "<u4", (256,)), ("area", "<u4", (8,)), ("dec", "<u2", (16384,)),
    ("count", "<u2", (64,)), ("index", "<u2", (64,)),
    ("area_start", "<u2", (8,)), ("area_size", "<u2", (8,)),
    ("width", "u1", (8,)), ("len", "u1", (256,)), ("rank", "u1", (256,)),
    ("by_rank", "u1", (256,)), ("sorted", "u1", (256,)),
], align=True)


class EccError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_status_name(code)} ({code})")
        self.code = code


class _Desc(ct.Structure):
    _fields_ = [("in_", ct.c_void_p), ("out", ct.c_void_p), ("n", ct.c_uint64), ("cap", ct.c_uint64),
                ("chunk_off", ct.c_void_p), ("sub_bits", ct.c_void_p), ("total_bits", ct.c_void_p),
                ("cb", ct.c_void_p), ("status", ct.c_void_p), ("t_done_ns", ct.c_void_p),
                ("C", ct.c_uint32), ("S", ct.c_uint32)]


_lock = threading.Lock()
_lib = None


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libecc_gb300 is not built ({LIB_PATH} missing): run "
                               "`python -m lossless_entropy_coding_gb300.build`")
        lib = ct.CDLL(LIB_PATH)
        P, Z, U32, U64, I32, D = ct.c_void_p, ct.c_size_t, ct.c_uint32, ct.c_uint64, ct.c_int32, ct.c_double
        sig = {
            "ecc_codebook_bytes": (Z, []),
            "qlc_build_tables": (I32, [P, P, P]),
            "qlc_search_widths": (I32, [P, U32, U32, P, P]),
            "huff_build_canonical": (I32, [P, U32, P]),
            "escape_build_tables": (I32, [P, P]),
            "gqlc_build_tables": (I32, [P, U32, P, P]),
            "gqlc_search_widths": (I32, [P, U32, U32, U32, P, P]),
            "huff_build_limited": (I32, [P, U32, P]),
            "ecc_entropy_bits": (D, [P]),
            "ecc_kl_bits": (D, [P, P]),
            "ecc_code_bits": (I32, [P, P, P]),
            "ecc_num_chunks": (Z, [Z, U32]),
            "ecc_num_subblocks": (Z, [Z, U32]),
            "ecc_max_encoded_bytes": (Z, [Z, U32, U32]),
            "ecc_encode_workspace_bytes": (Z, [Z, U32]),
            "e4m3_histogram": (I32, [P, Z, P, P]),
            "huff_build_device": (I32, [P, U64, U32, P, P, P]),
            "ecc_encode": (I32, [P, Z, P, U32, U32, P, Z, P, P, P, P, Z, P, P]),
            "ecc_decode": (I32, [P, Z, P, P, Z, U32, U32, P, P, P, P]),
            "ecc_batched_workspace_bytes": (Z, [P, U32]),
            "ecc_encode_batched": (I32, [P, U32, P, Z, P, P]),
            "ecc_decode_batched": (I32, [P, U32, P, Z, P, P]),
            "ecc_selftest_wait": (I32, [P, U64, U64, U64, P, P, P]),
            "ecc_encode_static": (I32, [P, Z, P, U32, U32, P, Z, P, P, P, P, P]),
            "ecc_status_string": (ct.c_char_p, [I32]),
            "bf16_escape_table_sigma": (I32, [ct.c_double, P]),
            "bf16_escape_table_counts": (I32, [P, P]),
            "bf16_exponent_histogram": (I32, [P, Z, P, P]),
            "bf16_escape_max_encoded_bytes": (Z, [Z, U32]),
            "bf16_escape_encode": (I32, [P, Z, P, U32, U32, P, Z, P, P, P, P, Z, P, P]),
            "bf16_escape_decode": (I32, [P, Z, P, P, Z, U32, U32, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    return _load()


def _status_name(code: int) -> str:
    try:
        return _load().ecc_status_string(code).decode()
    except Exception:  # library missing: fall back to the number
        return "status"


def _check(code: int, what: str):
    if code != OK:
        raise EccError(code, what)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ct.c_void_p)


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a).astype(np.uint64, copy=False))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a).astype(np.uint8, copy=False))


# ------------------------------------------------------------------ host builders

def codebook_bytes() -> int:
    return int(_load().ecc_codebook_bytes())


def qlc_build_tables(count, width=BASE_WIDTHS) -> np.ndarray:
    """Host QLC codebook (raw ecc_codebook bytes)."""
    count, width = _u64(count), _u8(width)
    out = np.zeros(codebook_bytes(), np.uint8)
    _check(_load().qlc_build_tables(_np_ptr(count), _np_ptr(width), _np_ptr(out)), "qlc_build_tables")
    return out


def qlc_search_widths(count, max_distinct: int = 4, require_full: bool = False):
    count = _u64(count)
    w = np.zeros(8, np.uint8)
    cost = np.zeros(1, np.uint64)
    _check(_load().qlc_search_widths(_np_ptr(count), max_distinct, int(bool(require_full)), _np_ptr(w),
                                     _np_ptr(cost)), "qlc_search_widths")
    return w, int(cost[0])


def huff_build_canonical(weight, max_len: int = MAX_CODE_LEN) -> np.ndarray:
    """Host canonical Huffman codebook (raw ecc_codebook bytes)."""
    weight = _u64(weight)
    out = np.zeros(codebook_bytes(), np.uint8)
    _check(_load().huff_build_canonical(_np_ptr(weight), max_len, _np_ptr(out)), "huff_build_canonical")
    return out


def codebook_view(cb: np.ndarray):
    """Structured view of raw codebook bytes (fields of ecc_codebook)."""
    return np.frombuffer(np.ascontiguousarray(cb, np.uint8).tobytes(), CODEBOOK_DTYPE)[0]


def entropy_bits(count) -> float:
    return float(_load().ecc_entropy_bits(_np_ptr(_u64(count))))


def kl_bits(p_count, q_count) -> float:
    return float(_load().ecc_kl_bits(_np_ptr(_u64(p_count)), _np_ptr(_u64(q_count))))


def code_bits(count, cb: np.ndarray) -> int:
    out = np.zeros(1, np.uint64)
    cbb = _u8(cb)
    _check(_load().ecc_code_bits(_np_ptr(_u64(count)), _np_ptr(cbb), _np_ptr(out)), "ecc_code_bits")
    return int(out[0])


def num_chunks(n: int, C: int) -> int:
    return int(_load().ecc_num_chunks(n, C))


def num_subblocks(n: int, S: int) -> int:
    return int(_load().ecc_num_subblocks(n, S))


def max_encoded_bytes(n: int, C: int, max_len: int) -> int:
    return int(_load().ecc_max_encoded_bytes(n, C, max_len))


def encode_workspace_bytes(n: int, C: int) -> int:
    return int(_load().ecc_encode_workspace_bytes(n, C))


def _register_path(cb) -> bool:
    """Whether the decoder reads codes of codebook cb through its prefix
    register path (QLC with a 3-bit prefix and codes of at most 11 bits)
    rather than through its first-level table.  cb: host codebook bytes, a
    device codebook made by to_device, or None (taken as the register
    path)."""
    if cb is None:
        return True
    tag = getattr(cb, "_ecc_register_path", None)
    if tag is not None:
        return bool(tag)
    if not isinstance(cb, np.ndarray):  # a device tensor of unknown origin
        return True
    v = codebook_view(cb)
    return int(v["family"]) == FAMILY_QLC and int(v["prefix_bits"]) == 3 and int(v["max_len"]) <= 11


def default_subblock(C: int, cb=None) -> int:
    """Sub-block size used when none is given.

    A QLC codebook the decoder reads through its prefix registers (or no
    codebook given): C/64, clamped to [64, 256].  Any other codebook (Huffman,
    the escape code, a length-limited Huffman or a QLC of fewer areas):
    C/128, clamped to [64, 128].  Its decoder waits on dependent table
    lookups, and sub-blocks of 128 symbols give each lane two independent
    streams at the same number of warps (1 GiB gradient tensor, Huffman
    decode: 1.14 -> 1.03 ms at 16 KiB chunks, 1.15 -> 1.04 ms at 64 KiB,
    for 1/64 byte a symbol more of sub-block counts); the QLC decoder is
    issue-bound and gains nothing.  Larger sub-blocks cost the decoder
    occupancy: a warp stages 32 sub-blocks or more, so with S > 256 fewer
    warps fit an SM."""
    if _register_path(cb):
        return int(min(256, max(64, C // 64)))
    return int(min(128, max(64, C // 128)))


# ------------------------------------------------------------------ device calls

def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ct.c_void_p(s.cuda_stream)


def _dptr(t):
    return ct.c_void_p(t.data_ptr()) if t is not None else ct.c_void_p(0)


def gqlc_build_tables(count, width, prefix_bits: int) -> np.ndarray:
    """Host QLC codebook with 2^prefix_bits areas (raw ecc_codebook bytes)."""
    count = _u64(count)
    w = np.zeros(8, np.uint8)
    w[:len(width)] = _u8(width)
    out = np.zeros(codebook_bytes(), np.uint8)
    _check(_load().gqlc_build_tables(_np_ptr(count), int(prefix_bits), _np_ptr(w), _np_ptr(out)),
           "gqlc_build_tables")
    return out


def gqlc_search_widths(count, prefix_bits: int, max_distinct: int = 4, require_full: bool = False):
    """Best widths of the 2^prefix_bits areas; returns (width, cost_bits)."""
    count = _u64(count)
    w = np.zeros(8, np.uint8)
    cost = np.zeros(1, np.uint64)
    _check(_load().gqlc_search_widths(_np_ptr(count), int(prefix_bits), int(max_distinct), int(bool(require_full)),
                                      _np_ptr(w), _np_ptr(cost)), "gqlc_search_widths")
    return w[:1 << prefix_bits].copy(), int(cost[0])


def huff_build_limited(weight, max_len: int) -> np.ndarray:
    """Host canonical Huffman codebook with lengths of at most max_len
    (package-merge; raw ecc_codebook bytes)."""
    weight = _u64(weight)
    out = np.zeros(codebook_bytes(), np.uint8)
    _check(_load().huff_build_limited(_np_ptr(weight), int(max_len), _np_ptr(out)), "huff_build_limited")
    return out


def escape_build_tables(count) -> np.ndarray:
    """Host escape-code codebook (raw ecc_codebook bytes): top-7 e4m3
    exponents in 3 bits, others 000 + exponent, sign and mantissa kept."""
    count = _u64(count)
    out = np.zeros(codebook_bytes(), np.uint8)
    _check(_load().escape_build_tables(_np_ptr(count), _np_ptr(out)), "escape_build_tables")
    return out


def to_device(cb: np.ndarray, device="cuda"):
    """Copy raw codebook bytes to a device tensor (what the kernels read).
    The tensor remembers which decoder path the codebook takes, for
    default_subblock."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(cb, np.uint8)).to(device)
    t._ecc_register_path = _register_path(cb)
    return t


def e4m3_histogram(x, count=None, stream=None):
    """Add the byte histogram of device tensor x to count (int64[256] on the
    device, zero-initialised when not given) and return count."""
    torch = _torch()
    if count is None:
        count = torch.zeros(256, dtype=torch.int64, device=x.device)
    _check(_load().e4m3_histogram(_dptr(x), x.numel(), _dptr(count), _stream_ptr(stream)), "e4m3_histogram")
    return count


def huff_build_device(count, add: int = 1, max_len: int = MAX_CODE_LEN, out=None, status=None, stream=None):
    """Build the canonical Huffman codebook of weights count + add on the
    device (count: int64[256] device tensor, e.g. from e4m3_histogram).
    Returns (codebook uint8 device tensor, status int32[1] device tensor);
    nothing is synchronised, read status after the stream reaches the call."""
    torch = _torch()
    dev = count.device
    if out is None:
        out = torch.empty(codebook_bytes(), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_load().huff_build_device(_dptr(count), int(add), int(max_len), _dptr(out), _dptr(status),
                                     _stream_ptr(stream)), "huff_build_device")
    return out, status


@dataclass
class Encoded:
    """Device tensors of one encoded container (payload holds out_cap bytes;
    the used part is payload[:chunk_off[-1]])."""
    payload: object
    chunk_off: object
    sub_bits: object
    total_bits: object
    status: object
    n: int
    C: int
    S: int


def ecc_encode(x, dev_cb, C: int = 16384, S: int | None = None, max_len: int = MAX_CODE_LEN, out=None,
               chunk_off=None, sub_bits=None, total_bits=None, ws=None, status=None, stream=None) -> Encoded:
    """Encode device bytes x with device codebook dev_cb (no synchronisation;
    read .status after the stream reaches this point)."""
    torch = _torch()
    dev = x.device
    n = x.numel()
    S = default_subblock(C, dev_cb) if S is None else S
    if out is None:
        out = torch.empty(max(16, max_encoded_bytes(n, C, max_len)), dtype=torch.uint8, device=dev)
    nch = num_chunks(n, C)
    if chunk_off is None:
        chunk_off = torch.empty(nch + 1, dtype=torch.int64, device=dev)
    if sub_bits is None:
        sub_bits = torch.empty(max(1, num_subblocks(n, S)), dtype=torch.int16, device=dev)
    if total_bits is None:
        total_bits = torch.empty(1, dtype=torch.int64, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.empty(encode_workspace_bytes(n, C), dtype=torch.uint8, device=dev)
    _check(_load().ecc_encode(_dptr(x), n, _dptr(dev_cb), C, S, _dptr(out), out.numel(), _dptr(chunk_off),
                              _dptr(sub_bits), _dptr(total_bits), _dptr(ws), ws.numel(), _dptr(status),
                              _stream_ptr(stream)), "ecc_encode")
    return Encoded(out, chunk_off, sub_bits, total_bits, status, n, C, S)


def ecc_decode(enc: Encoded, dev_cb, out=None, status=None, stream=None):
    """Decode a container into device bytes (returns (out, status))."""
    torch = _torch()
    dev = enc.payload.device
    if out is None:
        out = torch.empty(max(16, enc.n), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_load().ecc_decode(_dptr(enc.payload), enc.payload.numel(), _dptr(enc.chunk_off), _dptr(enc.sub_bits),
                              enc.n, enc.C, enc.S, _dptr(dev_cb), _dptr(out), _dptr(status), _stream_ptr(stream)),
           "ecc_decode")
    return out, status


def make_descs(items) -> ct.Array:
    """ecc_desc array from dicts with keys in, out, n, cap, chunk_off,
    sub_bits, total_bits, cb, status, t_done_ns, C, S (tensors or None)."""
    arr = (_Desc * len(items))()
    for d, it in zip(arr, items):
        d.in_ = it["in"].data_ptr()
        d.out = it["out"].data_ptr()
        d.n = int(it["n"])
        d.cap = int(it["cap"])
        d.chunk_off = it["chunk_off"].data_ptr()
        d.sub_bits = it["sub_bits"].data_ptr()
        d.total_bits = it["total_bits"].data_ptr() if it.get("total_bits") is not None else 0
        d.cb = it["cb"].data_ptr()
        d.status = it["status"].data_ptr()
        d.t_done_ns = it["t_done_ns"].data_ptr() if it.get("t_done_ns") is not None else 0
        d.C = int(it["C"])
        d.S = int(it["S"])
    return arr


def batched_workspace_bytes(descs) -> int:
    return int(_load().ecc_batched_workspace_bytes(ct.cast(descs, ct.c_void_p), len(descs)))


def ecc_encode_batched(descs, ws, t_start=None, stream=None):
    _check(_load().ecc_encode_batched(ct.cast(descs, ct.c_void_p), len(descs), _dptr(ws), ws.numel(),
                                      _dptr(t_start), _stream_ptr(stream)), "ecc_encode_batched")


def ecc_decode_batched(descs, ws, t_start=None, stream=None):
    _check(_load().ecc_decode_batched(ct.cast(descs, ct.c_void_p), len(descs), _dptr(ws), ws.numel(),
                                      _dptr(t_start), _stream_ptr(stream)), "ecc_decode_batched")


def ecc_selftest_wait(flags, chunk: int, aggregate: int, timeout_ns: int, prefix, status, stream=None):
    _check(_load().ecc_selftest_wait(_dptr(flags), chunk, aggregate, timeout_ns, _dptr(prefix), _dptr(status),
                                     _stream_ptr(stream)), "ecc_selftest_wait")


STATIC_MAX_CHUNKS = 65536


def ecc_encode_static(x, dev_cb, C: int = 16384, S: int | None = None, max_len: int = MAX_CODE_LEN, out=None,
                      chunk_off=None, sub_bits=None, total_bits=None, status=None, stream=None) -> Encoded:
    """ecc_encode with the library's built-in scratch array instead of a
    caller workspace (for callers that cannot allocate device memory on
    their call path).  Calls that may overlap on the GPU must be ordered by
    the caller: they share the scratch array."""
    torch = _torch()
    dev = x.device
    n = x.numel()
    S = default_subblock(C, dev_cb) if S is None else S
    if out is None:
        out = torch.empty(max(16, max_encoded_bytes(n, C, max_len)), dtype=torch.uint8, device=dev)
    if chunk_off is None:
        chunk_off = torch.empty(num_chunks(n, C) + 1, dtype=torch.int64, device=dev)
    if sub_bits is None:
        sub_bits = torch.empty(max(1, num_subblocks(n, S)), dtype=torch.int16, device=dev)
    if total_bits is None:
        total_bits = torch.empty(1, dtype=torch.int64, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_load().ecc_encode_static(_dptr(x), n, _dptr(dev_cb), C, S, _dptr(out), out.numel(), _dptr(chunk_off),
                                     _dptr(sub_bits), _dptr(total_bits), _dptr(status), _stream_ptr(stream)),
           "ecc_encode_static")
    return Encoded(out, chunk_off, sub_bits, total_bits, status, n, C, S)


# ---------------------------------------------------------------- BF16 exponent escape code

def bf16_escape_table_sigma(sigma: float) -> np.ndarray:
    """The 7-exponent table of N(0, sigma^2) in BF16 (uint8[7], rank order)."""
    top = np.zeros(7, np.uint8)
    _check(_load().bf16_escape_table_sigma(float(sigma), _np_ptr(top)), "bf16_escape_table_sigma")
    return top


def bf16_escape_table_counts(count) -> np.ndarray:
    """The 7 most frequent exponent fields of a count vector (uint8[7])."""
    count = _u64(count)
    top = np.zeros(7, np.uint8)
    _check(_load().bf16_escape_table_counts(_np_ptr(count), _np_ptr(top)), "bf16_escape_table_counts")
    return top


def bf16_exponent_histogram(x, count=None, stream=None):
    """Device exponent-field counts of BF16 values (x: uint16/int16/bfloat16
    device tensor), added to count (int64[256], allocated if None)."""
    torch = _torch()
    if count is None:
        count = torch.zeros(256, dtype=torch.int64, device=x.device)
    _check(_load().bf16_exponent_histogram(_dptr(x), x.numel(), _dptr(count), _stream_ptr(stream)),
           "bf16_exponent_histogram")
    return count


def bf16_escape_max_encoded_bytes(n: int, C: int) -> int:
    return int(_load().bf16_escape_max_encoded_bytes(n, C))


def bf16_escape_encode(x, top7, C: int = 4096, S: int | None = None, out=None, chunk_off=None, sub_bits=None,
                       total_bits=None, ws=None, status=None, stream=None) -> Encoded:
    """Encode device BF16 values (2-byte elements) with the escape code and
    the host table top7."""
    torch = _torch()
    dev = x.device
    n = x.numel()
    S = default_subblock(C) if S is None else S
    top7 = np.ascontiguousarray(top7, dtype=np.uint8)
    if out is None:
        out = torch.empty(max(16, bf16_escape_max_encoded_bytes(n, C)), dtype=torch.uint8, device=dev)
    if chunk_off is None:
        chunk_off = torch.empty(num_chunks(n, C) + 1, dtype=torch.int64, device=dev)
    if sub_bits is None:
        sub_bits = torch.empty(max(1, num_subblocks(n, S)), dtype=torch.int16, device=dev)
    if total_bits is None:
        total_bits = torch.empty(1, dtype=torch.int64, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.empty(encode_workspace_bytes(n, C), dtype=torch.uint8, device=dev)
    _check(_load().bf16_escape_encode(_dptr(x), n, _np_ptr(top7), C, S, _dptr(out), out.numel(), _dptr(chunk_off),
                                      _dptr(sub_bits), _dptr(total_bits), _dptr(ws), ws.numel(), _dptr(status),
                                      _stream_ptr(stream)), "bf16_escape_encode")
    return Encoded(out, chunk_off, sub_bits, total_bits, status, n, C, S)


def bf16_escape_decode(enc: Encoded, top7, out=None, status=None, stream=None):
    """Decode a BF16 escape-code container (returns (values int16, status))."""
    torch = _torch()
    dev = enc.payload.device
    top7 = np.ascontiguousarray(top7, dtype=np.uint8)
    if out is None:
        out = torch.empty(max(8, enc.n), dtype=torch.int16, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_load().bf16_escape_decode(_dptr(enc.payload), enc.payload.numel(), _dptr(enc.chunk_off),
                                      _dptr(enc.sub_bits), enc.n, enc.C, enc.S, _np_ptr(top7), _dptr(out),
                                      _dptr(status), _stream_ptr(stream)), "bf16_escape_decode")
    return out, status

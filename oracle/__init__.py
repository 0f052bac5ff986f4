"""Oracle for fixed-codebook lossless coding of e4m3 byte tensors.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  It wraps ``ecc_oracle.c`` -- a plain, bit-serial C implementation
that shares no code with the CUDA library -- with NumPy marshalling, and adds
the few float64 figures that are one-liners on top of it.

Every function cites the page passage it follows (see the header of
``ecc_oracle.c`` for the page list and for the readings taken where the pages
are silent).

Parity status: the QLC tables, Huffman lengths, canonical codes, codec and
figures are pinned by the tests in ``tests/test_oracle_pins.py``.  The
container layout (chunk padding, offsets, sub-block bit counts) is this
library's own format: the pages fix nothing about it, so beyond round-trip
and bit-count invariants it is "parity unpinned".
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ecc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libecc_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ARG, CAPACITY, CORRUPT, CODEBOOK = 0, 1, 2, 3, 4


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, libm)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ct.CDLL(build())
        P = ct.c_void_p
        U64, U32, I32 = ct.c_uint64, ct.c_uint32, ct.c_int
        sig = {
            "eo_histogram": (None, [P, U64, P]),
            "eo_rank": (None, [P, P, P]),
            "eo_qlc_layout": (I32, [P, P, P]),
            "eo_qlc_codebook": (I32, [P, P, P, P, P]),
            "eo_qlc_search": (I32, [P, I32, I32, I32, P, P]),
            "eo_huffman_lengths": (I32, [P, P]),
            "eo_canonical_codes": (I32, [P, P]),
            "eo_encode": (I32, [P, U64, P, P, U32, U32, P, U64, P, P, P]),
            "eo_decode_qlc": (I32, [P, U64, P, P, U64, U32, U32, P, P, P]),
            "eo_decode_huffman": (I32, [P, U64, P, P, U64, U32, U32, P, P]),
            "eo_escape_codebook": (I32, [P, P, P, P]),
            "eo_gqlc_layout": (I32, [I32, P, P, P]),
            "eo_gqlc_codebook": (I32, [P, I32, P, P, P, P]),
            "eo_gqlc_search": (I32, [P, I32, I32, I32, I32, P, P]),
            "eo_decode_gqlc": (I32, [P, U64, P, P, U64, U32, U32, I32, P, P, P]),
            "eo_huffman_limited": (I32, [P, I32, P]),
            "eo_decode_escape": (I32, [P, U64, P, P, U64, U32, U32, P, P]),
            "eo_entropy_bits": (ct.c_double, [P]),
            "eo_kl_bits": (ct.c_double, [P, P]),
            "eo_code_bits": (U64, [P, P]),
            "eo_bf16_exponent_counts": (I32, [P, U64, P]),
            "eo_bf16_top7_from_counts": (I32, [P, P]),
            "eo_bf16_exponent_probs": (I32, [ct.c_double, P]),
            "eo_bf16_top7_from_sigma": (I32, [ct.c_double, P]),
            "eo_bf16_escape_encode": (I32, [P, U64, P, U32, U32, P, U64, P, P, P]),
            "eo_bf16_escape_decode": (I32, [P, U64, P, P, U64, U32, U32, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ct.c_void_p)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint64)


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


# ---------------------------------------------------------------- statistics

def histogram(x) -> np.ndarray:
    """count[b] = number of bytes equal to b (Single-Stage Huffman,
    Methodology step 1)."""
    x = _u8(x)
    out = np.zeros(256, np.uint64)
    _load().eo_histogram(_p(x), x.size, _p(out))
    return out


def fixed_codebook_weights(counts) -> np.ndarray:
    """Weights of the single-stage codebook: the pooled counts of the warm-up
    batches plus a pseudocount of one per byte.  With equal-size batches the
    pooled counts are the average PMF times the total (Single-Stage Huffman,
    TL;DR and Methodology step 2); the pseudocount gives every byte a code."""
    w = np.ones(256, np.uint64)
    for c in counts:
        w += _u64(c)
    return w


# ---------------------------------------------------------------- QLC

def rank(count):
    """(rank, by_rank): bytes sorted by count descending, ties by byte value
    (Quad Length Codes, section 2, LUT paragraph)."""
    count = _u64(count)
    r = np.zeros(256, np.uint8)
    br = np.zeros(256, np.uint8)
    _load().eo_rank(_p(count), _p(r), _p(br))
    return r, br


BASE_WIDTHS = (3, 3, 3, 3, 3, 4, 5, 8)


def qlc_layout(width, prefix_bits: int = 3):
    """(start, size, covered) of the 2^prefix_bits areas filled in rank order."""
    w = np.zeros(8, np.uint8)
    w[:len(width)] = _u8(width)
    start = np.zeros(8, np.int32)
    size = np.zeros(8, np.int32)
    covered = _load().eo_gqlc_layout(int(prefix_bits), _p(w), _p(start), _p(size))
    A = 1 << prefix_bits
    return start[:A], size[:A], covered


def qlc_codebook(count, width=BASE_WIDTHS, prefix_bits: int = 3) -> dict:
    """Per-byte QLC code (len, code) plus by_rank, for the widths of the
    2^prefix_bits areas (the page's code: 3 prefix bits, 8 areas)."""
    count = _u64(count)
    w = np.zeros(8, np.uint8)
    w[:len(width)] = _u8(width)
    ln = np.zeros(256, np.uint8)
    code = np.zeros(256, np.uint64)
    br = np.zeros(256, np.uint8)
    _check(_load().eo_gqlc_codebook(_p(count), int(prefix_bits), _p(w), _p(ln), _p(code), _p(br)), "qlc_codebook")
    return {"family": "qlc", "prefix_bits": int(prefix_bits), "width": w[:1 << prefix_bits].copy(), "len": ln,
            "code": code, "by_rank": br}


def qlc_search(count, max_distinct=4, require_full=False, nondecreasing_only=True, prefix_bits: int = 3):
    """Adapted-QLC widths of the 2^prefix_bits areas by exhaustive search;
    returns (width, cost_bits)."""
    count = _u64(count)
    w = np.zeros(8, np.uint8)
    cost = np.zeros(1, np.uint64)
    _check(_load().eo_gqlc_search(_p(count), int(prefix_bits), int(max_distinct), int(bool(require_full)),
                                  int(bool(nondecreasing_only)), _p(w), _p(cost)), "qlc_search")
    return w[:1 << prefix_bits].copy(), int(cost[0])


# ---------------------------------------------------------------- Huffman

def huffman_lengths(weight) -> np.ndarray:
    weight = _u64(weight)
    ln = np.zeros(256, np.uint8)
    _check(_load().eo_huffman_lengths(_p(weight), _p(ln)), "huffman_lengths")
    return ln


def canonical_codes(length) -> np.ndarray:
    ln = _u8(length)
    code = np.zeros(256, np.uint64)
    _check(_load().eo_canonical_codes(_p(ln), _p(code)), "canonical_codes")
    return code


def huffman_codebook(weight) -> dict:
    """Canonical Huffman code of a weight vector (Single-Stage Huffman,
    Methodology step 3)."""
    ln = huffman_lengths(weight)
    return {"family": "huffman", "len": ln, "code": canonical_codes(ln)}


def huffman_limited_lengths(weight, max_len: int) -> np.ndarray:
    """Optimal code lengths of at most max_len bits (package-merge)."""
    weight = _u64(weight)
    ln = np.zeros(256, np.uint8)
    _check(_load().eo_huffman_limited(_p(weight), int(max_len), _p(ln)), "huffman_limited")
    return ln


def huffman_limited_codebook(weight, max_len: int) -> dict:
    """Canonical code of the length-limited Huffman lengths."""
    ln = huffman_limited_lengths(weight, max_len)
    return {"family": "huffman", "len": ln, "code": canonical_codes(ln)}


# ---------------------------------------------------------------- escape code

def escape_codebook(count) -> dict:
    """ZipCCL-style escape code on the e4m3 exponent field (ZipCCL, section
    2.B): the 7 most frequent exponents (summed counts, ties to the smaller)
    coded 001..111, others 000 + the 4-bit exponent; sign and mantissa as
    they are."""
    count = _u64(count)
    ln = np.zeros(256, np.uint8)
    code = np.zeros(256, np.uint64)
    top = np.zeros(7, np.uint8)
    _check(_load().eo_escape_codebook(_p(count), _p(ln), _p(code), _p(top)), "escape_codebook")
    return {"family": "escape", "len": ln, "code": code, "top": top}


# ---------------------------------------------------------------- codec

def max_encoded_bytes(n: int, C: int, max_len: int) -> int:
    """Upper bound of the container payload: every symbol at max_len bits,
    each chunk padded to 16 bytes."""
    full, tail = divmod(n, C)
    per = lambda L: (L * max_len + 7) // 8 // 1
    tot = full * ((per(C) + 15) // 16 * 16)
    if tail:
        tot += (per(tail) + 15) // 16 * 16
    return tot


def encode(x, cb: dict, C: int, S: int, cap: int | None = None) -> dict:
    """Bit-serial encode into the chunked container."""
    x = _u8(x)
    n = x.size
    ln = _u8(cb["len"])
    code = _u64(cb["code"])
    if cap is None:
        cap = max_encoded_bytes(n, C, int(ln.max()) if n else 1)
    out = np.zeros(max(cap, 1), np.uint8)
    n_chunks = -(-n // C)
    chunk_off = np.zeros(n_chunks + 1, np.uint64)
    sub_bits = np.zeros(max(-(-n // S), 1), np.uint16)
    total = np.zeros(1, np.uint64)
    _check(_load().eo_encode(_p(x), n, _p(ln), _p(code), C, S, _p(out), cap,
                             _p(chunk_off), _p(sub_bits), _p(total)), "encode")
    used = int(chunk_off[-1])
    return {"payload": out[:used].copy(), "chunk_off": chunk_off,
            "sub_bits": sub_bits[:-(-n // S)].copy(), "total_bits": int(total[0]),
            "n": n, "C": C, "S": S}


def decode(enc: dict, cb: dict) -> np.ndarray:
    """Bit-serial decode of a container produced by encode()."""
    payload = _u8(enc["payload"])
    n, C, S = enc["n"], enc["C"], enc["S"]
    chunk_off = _u64(enc["chunk_off"])
    sub_bits = np.ascontiguousarray(enc["sub_bits"], dtype=np.uint16)
    if sub_bits.size == 0:
        sub_bits = np.zeros(1, np.uint16)
    out = np.zeros(max(n, 1), np.uint8)
    buf = payload if payload.size else np.zeros(1, np.uint8)
    lib = _load()
    if cb["family"] == "qlc":
        w = np.zeros(8, np.uint8)
        w[:len(cb["width"])] = _u8(cb["width"])
        rc = lib.eo_decode_gqlc(_p(buf), payload.size, _p(chunk_off), _p(sub_bits), n, C, S,
                                int(cb.get("prefix_bits", 3)), _p(w), _p(_u8(cb["by_rank"])), _p(out))
    elif cb["family"] == "escape":
        rc = lib.eo_decode_escape(_p(buf), payload.size, _p(chunk_off), _p(sub_bits), n, C, S,
                                  _p(_u8(cb["top"])), _p(out))
    else:
        rc = lib.eo_decode_huffman(_p(buf), payload.size, _p(chunk_off), _p(sub_bits), n, C, S,
                                   _p(_u8(cb["len"])), _p(out))
    _check(rc, "decode")
    return out[:n]


# ---------------------------------------------------------------- figures

def entropy_bits(count) -> float:
    """Shannon entropy H = -sum p log2 p, bits per symbol."""
    return float(_load().eo_entropy_bits(_p(_u64(count))))


def kl_bits(p_count, q_count) -> float:
    """D(P || Q) in bits (Single-Stage Huffman, Figure 3)."""
    return float(_load().eo_kl_bits(_p(_u64(p_count)), _p(_u64(q_count))))


def code_bits(count, length) -> int:
    """Total payload bits sum(count x length) of a codebook on a histogram."""
    v = int(_load().eo_code_bits(_p(_u64(count)), _p(_u8(length))))
    if v == (1 << 64) - 1:
        raise OracleError(CODEBOOK, "code_bits: a counted byte has no code")
    return v


def compressibility(bits: int, n: int) -> float:
    """1 - mean code length / 8: the fraction of the 8-bit container saved
    (the pages quote it in percent, e.g. 15.9% for FFN1 Huffman)."""
    return 1.0 - bits / (8.0 * n)


def shannon_compressibility(count) -> float:
    return 1.0 - entropy_bits(count) / 8.0


# ---------------------------------------------------------------- BF16 escape code

def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def bf16_exponent_counts(x) -> np.ndarray:
    """count[e] = number of BF16 values (uint16 bit patterns) whose exponent
    field (bits 14-7) is e."""
    x = _u16(x)
    out = np.zeros(256, np.uint64)
    _check(_load().eo_bf16_exponent_counts(_p(x), x.size, _p(out)), "bf16_exponent_counts")
    return out


def bf16_top7_from_counts(count) -> np.ndarray:
    """The 7 most frequent exponents, in rank order (ZipCCL, section 2.A;
    count descending, ties to the smaller exponent)."""
    count = _u64(count)
    top = np.zeros(7, np.uint8)
    _check(_load().eo_bf16_top7_from_counts(_p(count), _p(top)), "bf16_top7_from_counts")
    return top


def bf16_exponent_probs(sigma: float) -> np.ndarray:
    """P(exponent field = e) for N(0, sigma^2) rounded to BF16 (ZipCCL,
    section 2.A: the exponent table follows from sigma)."""
    out = np.zeros(256, np.float64)
    _check(_load().eo_bf16_exponent_probs(float(sigma), _p(out)), "bf16_exponent_probs")
    return out


def bf16_top7_from_sigma(sigma: float) -> np.ndarray:
    """The 7 most probable exponents of N(0, sigma^2) in BF16, in rank order
    (ties to the smaller exponent)."""
    top = np.zeros(7, np.uint8)
    _check(_load().eo_bf16_top7_from_sigma(float(sigma), _p(top)), "bf16_top7_from_sigma")
    return top


def bf16_escape_encode(x, top, C: int, S: int, cap: int | None = None) -> dict:
    """Bit-serial encode of BF16 values (uint16 bit patterns) with the
    exponent escape code (ZipCCL, section 2.B) into the chunked container."""
    x = _u16(x)
    top = _u8(top)
    n = x.size
    if cap is None:
        full, tail = divmod(n, C)
        cap = full * ((C * 19 + 7) // 8 + 15) // 16 * 16 + (((tail * 19 + 7) // 8 + 15) // 16 * 16 if tail else 0)
    out = np.zeros(max(cap, 1), np.uint8)
    n_chunks = -(-n // C)
    chunk_off = np.zeros(n_chunks + 1, np.uint64)
    sub_bits = np.zeros(max(-(-n // S), 1), np.uint16)
    total = np.zeros(1, np.uint64)
    _check(_load().eo_bf16_escape_encode(_p(x), n, _p(top), C, S, _p(out), cap, _p(chunk_off), _p(sub_bits),
                                         _p(total)), "bf16_escape_encode")
    used = int(chunk_off[-1])
    return {"payload": out[:used].copy(), "chunk_off": chunk_off, "sub_bits": sub_bits[:-(-n // S)].copy(),
            "total_bits": int(total[0]), "n": n, "C": C, "S": S}


def bf16_escape_decode(enc: dict, top) -> np.ndarray:
    """Bit-serial decode of a container produced by bf16_escape_encode()."""
    payload = _u8(enc["payload"])
    n, C, S = enc["n"], enc["C"], enc["S"]
    chunk_off = _u64(enc["chunk_off"])
    sub_bits = np.ascontiguousarray(enc["sub_bits"], dtype=np.uint16)
    if sub_bits.size == 0:
        sub_bits = np.zeros(1, np.uint16)
    out = np.zeros(max(n, 1), np.uint16)
    buf = payload if payload.size else np.zeros(1, np.uint8)
    _check(_load().eo_bf16_escape_decode(_p(buf), payload.size, _p(chunk_off), _p(sub_bits), n, C, S,
                                         _p(_u8(top)), _p(out)), "bf16_escape_decode")
    return out[:n]

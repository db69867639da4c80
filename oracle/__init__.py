"""FP64 CPU oracle for single-token GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``gqa_decode_attention_sm_gb300``) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``gqa_oracle.c`` (plain C, FP64, POSIX threads); this
module only compiles it and marshals numpy arrays through ctypes.  What it
computes, and the pages it restates:

* "FlashInfer sm110_gqa_decode" article, sections "Input contract" and
  "Convenience API": q [batch,32,128], kv [batch,2,8,capacity,128] (K plane 0,
  V plane 1), int32 lengths in [1, capacity]; softmax scale q_scale/sqrt(128);
  query heads 4g..4g+3 read KV head g (the grouped view: 8 groups of 4 consecutive heads).
* "FP8 KV cache port on Jetson AGX Thor" blog, section 1 (patches 1 and 2):
  e4m3 cache bytes are reinterpreted, not converted; scores are multiplied by
  k_scale and the normalised output by v_scale.
* "Qwen3-VL official BF16 on Jetson Orin (SM87)" docs, "INT8 KV cache
  (kv_mode)": int8 codes, a bf16 scale for each (position, KV head) row.
* "FreeToken-Kai on Turing" notes, change 7: every key of the range scored
  first, then one ordinary softmax over all of them.

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, invariants, exhaustive format tables and torch's float64
``scaled_dot_product_attention``; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, E4M3, I8 = 0, 1, 2, 3
HQ, HKV, D = 32, 8, 128

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gqa.so")
_lib = None
_lock = threading.Lock()

_ERRORS = {1: "invalid argument", 2: "a length is outside [1, capacity]", 3: "out of memory"}


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-std=c11", "-Wall", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) and return the ctypes handle."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib):
    lib.orc_decode_f16.restype = ctypes.c_double
    lib.orc_decode_f16.argtypes = [ctypes.c_uint16]
    lib.orc_decode_bf16.restype = ctypes.c_double
    lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.orc_decode_e4m3.restype = ctypes.c_double
    lib.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.orc_round_f16.restype = ctypes.c_uint16
    lib.orc_round_f16.argtypes = [ctypes.c_double]
    lib.orc_round_bf16.restype = ctypes.c_uint16
    lib.orc_round_bf16.argtypes = [ctypes.c_double]
    p = ctypes.c_void_p
    lib.orc_norm_rope.restype = None
    lib.orc_norm_rope.argtypes = [p, p, ctypes.c_int, ctypes.c_double, ctypes.c_double, p]
    lib.orc_decode_array.restype = None
    lib.orc_decode_array.argtypes = [p, ctypes.c_int, ctypes.c_size_t, p]
    lib.orc_round_array.restype = None
    lib.orc_round_array.argtypes = [p, ctypes.c_size_t, ctypes.c_int, p]
    lib.orc_gqa_decode.restype = ctypes.c_int
    lib.orc_gqa_decode.argtypes = [p, ctypes.c_int, p, ctypes.c_int, p, p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_double, p, ctypes.c_int, p, p, ctypes.c_int,
                                   ctypes.c_int]
    return lib


def decode(bits: np.ndarray, fmt: int, lib=None) -> np.ndarray:
    """Decode raw bit patterns (uint16 for f16/bf16, uint8 for e4m3) to float64."""
    lib = lib or load()
    flat = np.asarray(bits).ravel()
    flat = np.ascontiguousarray(flat.view(np.uint8) if fmt == I8 and flat.dtype == np.int8 else flat,
                                dtype=np.uint8 if fmt in (E4M3, I8) else np.uint16)
    out = np.empty(flat.size, dtype=np.float64)
    lib.orc_decode_array(flat.ctypes.data, fmt, flat.size, out.ctypes.data)
    return out.reshape(np.shape(bits))


def round_to(x: np.ndarray, fmt: int, lib=None) -> np.ndarray:
    """Round float64 values to f16/bf16 bits, nearest-even, in one step."""
    lib = lib or load()
    assert fmt in (F16, BF16)
    flat = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
    out = np.empty(flat.size, dtype=np.uint16)
    lib.orc_round_array(flat.ctypes.data, flat.size, fmt, out.ctypes.data)
    return out.reshape(np.shape(x))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def gqa_decode(q_bits: np.ndarray, q_fmt: int, kv_bits: np.ndarray, kv_fmt: int,
               lens: np.ndarray, q_scale: float = 1.0, k_scale: float = 1.0,
               v_scale: float = 1.0, rows=None, out_fmt: int | None = None,
               threads: int | None = None, lib=None, kv_scales: np.ndarray | None = None):
    """Oracle attention output.

    q_bits    uint16 [B,32,128] (f16 or bf16 bit patterns), or [B,T,32,128] for a
              verify window of T query tokens (query j attends slots [0, L-T+j])
    kv_bits   uint16 [B,2,8,C,128] (f16/bf16), uint8 (e4m3 bytes) or int8 codes (I8)
    kv_scales bf16 bit patterns (uint16) [B,2,8,C], required for I8
    lens      int32 [B]
    rows      optional iterable of (b*T + j)*32 + h; default all rows in order
    Returns (out_f64 [n_rows,128], out_bits uint16 [n_rows,128]).
    """
    lib = lib or load()
    q_bits = np.ascontiguousarray(q_bits)
    kv_bits = np.ascontiguousarray(kv_bits)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    B = q_bits.shape[0]
    T = 1 if q_bits.ndim == 3 else q_bits.shape[1]
    assert q_bits.shape in ((B, HQ, D), (B, T, HQ, D)) and q_bits.dtype == np.uint16
    assert kv_bits.ndim == 5 and kv_bits.shape[:3] == (B, 2, HKV) and kv_bits.shape[4] == D
    if kv_fmt == I8:
        kv_bits = kv_bits.view(np.int8)
        assert kv_scales is not None
        kv_scales = np.ascontiguousarray(kv_scales).view(np.uint16)
        assert kv_scales.shape == kv_bits.shape[:4]
    else:
        assert kv_bits.dtype == (np.uint8 if kv_fmt == E4M3 else np.uint16)
    assert lens.shape == (B,)
    C = kv_bits.shape[3]
    if out_fmt is None:
        out_fmt = q_fmt
    if rows is None:
        rows_arr = np.arange(B * T * HQ, dtype=np.int32)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int32))
    n = int(rows_arr.size)
    out = np.zeros((n, D), dtype=np.float64)
    bits = np.zeros((n, D), dtype=np.uint16)
    st = lib.orc_gqa_decode(q_bits.ctypes.data, q_fmt, kv_bits.ctypes.data, kv_fmt,
                            kv_scales.ctypes.data if kv_fmt == I8 else None,
                            lens.ctypes.data, B, C, T, float(q_scale), float(k_scale),
                            float(v_scale), rows_arr.ctypes.data, n, out.ctypes.data,
                            bits.ctypes.data, out_fmt, threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle: {_ERRORS.get(st, st)}")
    return out, bits


def gather_pages(pages: np.ndarray, block_table: np.ndarray, lens: np.ndarray) -> np.ndarray:
    """A paged cache gathered into one contiguous prefix matrix per batch row.

    pages [num_pages, 2, 8, page_size, 128] (bits), or an int8 cache's row-scale
    pool [num_pages, 2, 8, page_size]; block_table int [B, max_pages]: slot t of
    row b is row t % page_size of page block_table[b, t // page_size].  Only the
    pages that hold slots below each length are gathered; the rest of the
    returned [B, 2, 8, max_pages * page_size(, 128)] array is zero.
    (The "FreeToken-Kai on Turing" notes, change 7: a paged cache's prefix is
    first copied into one contiguous key matrix.)
    """
    B, max_pages = block_table.shape
    ps = pages.shape[3]
    out = np.zeros((B, 2, HKV, max_pages * ps) + tuple(pages.shape[4:]), dtype=pages.dtype)
    for b in range(B):
        for j in range(-(-int(lens[b]) // ps)):
            out[b, :, :, j * ps:(j + 1) * ps] = pages[int(block_table[b, j])]
    return out


def norm_rope(x: np.ndarray, w: np.ndarray, pos: int, eps: float, theta: float, lib=None) -> np.ndarray:
    """RMS norm (weight w) then rotate-half RoPE at position pos, FP64; x, w [128]."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    z = np.empty(D, dtype=np.float64)
    lib.orc_norm_rope(x.ctypes.data, w.ctypes.data, int(pos), float(eps), float(theta), z.ctypes.data)
    return z


def append_kv(q_proj, k_proj, v_proj, q_norm_w, k_norm_w, positions, eps, theta, lib=None):
    """The appended token in FP64: q_out [B,32,128], k_new [B,8,128], v_new [B,8,128].

    Inputs are FP64 values (decode the bf16/fp16 bits first)."""
    B = q_proj.shape[0]
    qo = np.empty((B, HQ, D))
    ko = np.empty((B, HKV, D))
    for b in range(B):
        for h in range(HQ):
            qo[b, h] = norm_rope(q_proj[b, h], q_norm_w, positions[b], eps, theta, lib)
        for g in range(HKV):
            ko[b, g] = norm_rope(k_proj[b, g], k_norm_w, positions[b], eps, theta, lib)
    return qo, ko, np.array(v_proj, dtype=np.float64)

"""fp64 CPU oracle for multi-LoRA shrink/expand (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library and
its binding) never imports, calls or links it, and it shares no code with
that path: the arithmetic lives in ``lora_oracle.c`` (plain loops in fp64),
and this module only compiles it with the host C compiler and marshals
numpy arrays into it.

The definition it follows is restated at the top of ``lora_oracle.c`` with
its sources: "[V1] LoRA - Add triton kernels for V1" (vLLM PR 13096,
"Why do we need a new set of kernels"), "[Tracking] Multi-LoRA Serving"
(MLC-LLM, Overview) and "[Kernel] LoRA - Enable CUDAGraphs for V1" (vLLM
PR 14626, the pad region and the static max_num_tokens buffers).

Pins: every function here is checked against something other than itself
by ``tests/test_oracle_pins.py`` (a textbook stable sort and numpy's stable
argsort, brute force over all permutations of tiny mappings, dense numpy
matmuls for one-adapter batches, associativity of shrink then expand,
exact small-integer cases, a hand-worked example under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

STATUS_BAD_LORA_ID = 1
STATUS_BAD_NUM_TOKENS = 2


def build(force: bool = False) -> str:
    """Compile lora_oracle.c into a shared library (OpenMP when available)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                "-std=c11", _SRC, "-o", tmp]
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                           capture_output=True, text=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_prepare_metadata.restype = ctypes.c_uint32
        lib.oracle_prepare_metadata.argtypes = [p, i64, i64, i64, p, p, p]
        lib.oracle_shrink.restype = None
        lib.oracle_shrink.argtypes = [p, i64, i64, p, i64, i64, ctypes.c_double, p, p, i64, i64,
                                      p, i64, ctypes.c_int, ctypes.c_int]
        lib.oracle_expand.restype = None
        lib.oracle_expand.argtypes = [p, p, p, i64, i64, p, i64, p, i64, i64, p, i64,
                                      ctypes.c_int, ctypes.c_int]
        lib.oracle_decode_bits.restype = None
        lib.oracle_decode_bits.argtypes = [p, i64, ctypes.c_int, p]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP runtime uses by default (1 without OpenMP)."""
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def prepare_metadata(token_lora_mapping: np.ndarray, num_tokens: int, max_loras: int):
    """Stable grouping of tokens 0..n-1 by LoRA id.

    Returns ``(sorted_token_ids[T_max], num_tokens_per_lora[L+1],
    lora_token_start_loc[L+2], status)``; bin L holds the tokens with no
    adapter (-1 or an out-of-range id, the latter also setting status bit 1).
    """
    m = _c(token_lora_mapping, np.int32)
    t_max = m.shape[0]
    sorted_ids = np.empty(t_max, np.int32)
    counts = np.empty(max_loras + 1, np.int32)
    starts = np.empty(max_loras + 2, np.int32)
    status = _load().oracle_prepare_metadata(_ptr(m), int(num_tokens), t_max, int(max_loras),
                                             _ptr(sorted_ids), _ptr(counts), _ptr(starts))
    return sorted_ids, counts, starts, int(status)


def shrink(x_bits: np.ndarray, lora_a_bits, scale: float, token_lora_mapping: np.ndarray,
           num_tokens: int, max_loras: int, u_init: np.ndarray | None = None,
           num_threads: int = 0, lora_scales=None, f16: bool = False) -> np.ndarray:
    """u[s][t][r] = c(m[t]) * sum_h x[t][h] A_s[m[t]][r][h] in fp64, with
    c(l) = scale, or scale * lora_scales[l] when per-adapter factors are given.

    ``x_bits``: uint16 bf16 bits ``[T_max, H]`` (fp16 bits when ``f16``);
    ``lora_a_bits``: list of S uint16 arrays ``[L, R, H]`` of the same type.
    Rows of tokens without an adapter (and rows t >= n) keep ``u_init`` (NaN
    when not given).
    """
    x = _c(x_bits, np.uint16)
    t_max, hidden = x.shape
    a_list = [_c(a, np.uint16) for a in lora_a_bits]
    num_slices = len(a_list)
    rank = a_list[0].shape[1]
    for a in a_list:
        if a.shape != (max_loras, rank, hidden):
            raise ValueError("lora_a shape mismatch")
    m = _c(token_lora_mapping, np.int32)
    if not 0 <= num_tokens <= t_max or m.shape != (t_max,):
        raise ValueError("num_tokens / mapping size out of range")
    if u_init is None:
        u = np.full((num_slices, t_max, rank), np.nan, np.float64)
    else:
        u = np.array(u_init, dtype=np.float64, copy=True, order="C")
    ptrs = (ctypes.c_void_p * num_slices)(*[_ptr(a) for a in a_list])
    ls = None
    if lora_scales is not None:
        ls = _c(np.asarray(lora_scales, dtype=np.float64), np.float64)
        if ls.shape != (max_loras,):
            raise ValueError("lora_scales must have max_loras entries")
    _load().oracle_shrink(_ptr(x), hidden, hidden, ctypes.addressof(ptrs), num_slices, rank,
                          float(scale), None if ls is None else _ptr(ls), _ptr(m),
                          int(num_tokens), int(max_loras), _ptr(u), t_max, int(bool(f16)),
                          int(num_threads) or max_threads())
    return u


def expand(u: np.ndarray, lora_b_bits, y_bits: np.ndarray, token_lora_mapping: np.ndarray,
           num_tokens: int, max_loras: int, num_threads: int = 0,
           f16: bool = False) -> np.ndarray:
    """y[t][off_s + j] + sum_r u[s][t][r] B_s[m[t]][r][j], returned in fp64.

    ``u``: float array ``[S, T_max, R]`` (converted to fp64); ``lora_b_bits``:
    list of S uint16 arrays ``[L, R, N_s]``; ``y_bits``: uint16 ``[T_max, W]``
    with ``W >= sum N_s``; B and y hold bf16 bits, or fp16 bits when ``f16``.
    Every element of the result is written.
    """
    uu = np.ascontiguousarray(u, dtype=np.float64)
    b_list = [_c(b, np.uint16) for b in lora_b_bits]
    num_slices = len(b_list)
    rank = b_list[0].shape[1]
    widths = np.array([b.shape[2] for b in b_list], np.int64)
    y = _c(y_bits, np.uint16)
    t_max, row = y.shape
    if widths.sum() > row or uu.shape != (num_slices, t_max, rank):
        raise ValueError("expand shape mismatch")
    for b in b_list:
        if b.shape[:2] != (max_loras, rank):
            raise ValueError("lora_b shape mismatch")
    m = _c(token_lora_mapping, np.int32)
    if not 0 <= num_tokens <= t_max or m.shape != (t_max,):
        raise ValueError("num_tokens / mapping size out of range")
    out = np.empty((t_max, row), np.float64)
    ptrs = (ctypes.c_void_p * num_slices)(*[_ptr(b) for b in b_list])
    _load().oracle_expand(_ptr(uu), ctypes.addressof(ptrs), _ptr(widths), num_slices, rank,
                          _ptr(y), row, _ptr(m), int(num_tokens), int(max_loras), _ptr(out),
                          t_max, int(bool(f16)), int(num_threads) or max_threads())
    return out


def decode_bits(bits: np.ndarray, f16: bool = False) -> np.ndarray:
    """The oracle's own decoding of 16-bit input words (bf16, or fp16 when
    ``f16``) to float64, as its shrink and expand read them."""
    b = _c(np.asarray(bits, dtype=np.uint16), np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_decode_bits(_ptr(b), b.size, int(bool(f16)), _ptr(out))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64 (a widening, no rounding)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

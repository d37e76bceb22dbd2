"""CPU oracle for the fused GPTQ W4A16 linear layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never
touches it, and it never touches the product library: the arithmetic lives in
``gptq_oracle.c`` (plain C, fp64) and this module only marshals numpy arrays
into it and composes its steps in the order the method defines them:

1. unpack the 4-bit codes of qweight and qzeros (GPTQ-v1 storage: eight codes
   per int32, lowest nibble first; "GPTQ's 'Exllama Kernel Not Installed'
   Warning", section "Why the kernel is missing");
2. map each row to its group, through g_idx when given ("Implementation:
   Predibase Lorax GPTQ Exllama V1", section "I/O Contract": None or trivial
   indices mean no act-order);
3. dequantize  w = s * (q - (z + 1))  exactly, then round once to fp16;
4. y_ref = x . w16 + bias in fp64 (the fallback's route to the same answer,
   "What the fallback actually does" on the first page), and y_exact with the
   unrounded weights.

Every function is pinned by the ``-m "not gpu"`` tests in ``tests/`` against
values that do not come from this oracle (numpy's float16 cast, hand-packed
words, closed forms, brute force, invariants).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gptq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build", platform.machine())
_LIB_PATH = os.path.join(_BUILD_DIR, "libgptq_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags, no target tuning)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_half_to_double_array.argtypes = [P, ctypes.c_size_t, P]
        lib.oracle_double_to_half_array.argtypes = [P, ctypes.c_size_t, P]
        lib.oracle_unpack_qweight.argtypes = [P, I, I, P]
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double_array.argtypes = [P, ctypes.c_size_t, P]
        lib.oracle_f32_to_double.argtypes = [ctypes.c_uint32]
        lib.oracle_f32_to_double.restype = ctypes.c_double
        lib.oracle_f32_to_double_array.argtypes = [P, ctypes.c_size_t, P]
        lib.oracle_unpack_qzeros.argtypes = [P, I, I, P]
        lib.oracle_unpack_qweight8.argtypes = [P, I, I, P]
        lib.oracle_unpack_qzeros8.argtypes = [P, I, I, P]
        lib.oracle_row_groups.argtypes = [P, I, I, P]
        lib.oracle_row_groups.restype = I
        lib.oracle_dequant.argtypes = [P, P, P, P, I, I, P, P, I]
        lib.oracle_linear_f64.argtypes = [P, P, P, I, I, I, P, I]
        lib.oracle_pack.argtypes = [P, P, P, P, I, I, I, I, P, P]
        lib.oracle_pack.restype = I
        lib.oracle_linear_f64.restype = I
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ fp16

def half_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float64, from the binary16 definition."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_half_to_double_array(_ptr(b), b.size, _ptr(out))
    return out


def f64_to_half_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> fp16 bit patterns, one round-to-nearest-even."""
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_double_to_half_array(_ptr(a), a.size, _ptr(out))
    return out


# ---------------------------------------------------------------- steps

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_bf16_to_double_array(_ptr(b), b.size, _ptr(out))
    return out


def f32_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """fp32 bit patterns (uint32) -> exact fp64 values, from the binary32 definition."""
    b = _c(bits, np.uint32)
    out = np.empty(b.shape, np.float64)
    _load().oracle_f32_to_double_array(_ptr(b), b.size, _ptr(out))
    return out


def unpack_qweight(qweight: np.ndarray, K: int, N: int) -> np.ndarray:
    qw = _c(qweight, np.int32)
    assert qw.shape == (K // 8, N)
    q = np.empty((K, N), np.uint8)
    _load().oracle_unpack_qweight(_ptr(qw), K, N, _ptr(q))
    return q


def unpack_qzeros(qzeros: np.ndarray, G: int, N: int) -> np.ndarray:
    qz = _c(qzeros, np.int32)
    assert qz.shape == (G, N // 8)
    z = np.empty((G, N), np.uint8)
    _load().oracle_unpack_qzeros(_ptr(qz), G, N, _ptr(z))
    return z


def unpack_qweight8(qweight: np.ndarray, K: int, N: int) -> np.ndarray:
    """8-bit codes: qweight [K/4, N], four per word along K, lowest byte first."""
    qw = _c(qweight, np.int32)
    assert qw.shape == (K // 4, N)
    q = np.empty((K, N), np.uint8)
    _load().oracle_unpack_qweight8(_ptr(qw), K, N, _ptr(q))
    return q


def unpack_qzeros8(qzeros: np.ndarray, G: int, N: int) -> np.ndarray:
    qz = _c(qzeros, np.int32)
    assert qz.shape == (G, N // 4)
    z = np.empty((G, N), np.uint8)
    _load().oracle_unpack_qzeros8(_ptr(qz), G, N, _ptr(z))
    return z


def row_groups(g_idx, K: int, groupsize: int):
    """Group of every row, and G.  Raises ValueError on an invalid index."""
    gi = None if g_idx is None else _c(g_idx, np.int32)
    gr = np.empty(K, np.int32)
    G = _load().oracle_row_groups(_ptr(gi), K, groupsize, _ptr(gr))
    if G < 0:
        raise ValueError("invalid groupsize or g_idx entry outside [0, G)")
    return gr, G


def dequant(q, z, scales_bits, gr, K: int, N: int, want_f64: bool = True, zero_offset: int = 1):
    """w16 (fp16 bits) and, if asked, the exact fp64 weights.  zero_offset:
    1 for GPTQ checkpoints (effective zero = stored + 1), 0 for GPTQ_V2."""
    qa, za = _c(q, np.uint8), _c(z, np.uint8)
    sb, ga = _c(scales_bits, np.uint16), _c(gr, np.int32)
    w16 = np.empty((K, N), np.uint16)
    w64 = np.empty((K, N), np.float64) if want_f64 else None
    _load().oracle_dequant(_ptr(qa), _ptr(za), _ptr(sb), _ptr(ga), K, N,
                           _ptr(w16), _ptr(w64), int(zero_offset))
    return w16, w64


def linear_f64(x64: np.ndarray, w64: np.ndarray, bias64=None, nthreads: int | None = None):
    """y = x . w + bias in fp64, each output summed over ascending k."""
    x = _c(x64, np.float64)
    w = _c(w64, np.float64)
    M, K = x.shape
    K2, N = w.shape
    assert K == K2
    b = None if bias64 is None else _c(bias64, np.float64)
    y = np.empty((M, N), np.float64)
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    _load().oracle_linear_f64(_ptr(x), _ptr(w), _ptr(b), M, K, N, _ptr(y), nt)
    return y


def pack(w16, scales_bits, zeros, g_idx, K: int, N: int, groupsize: int, zero_offset: int = 1):
    """Float weights w16 [K, N] (fp16 bits) with the quantizer's scales [G, N]
    (fp16 bits) and effective zero points [G, N] (int; None: symmetric, 8)
    -> (qweight [K/8, N], qzeros [G, N/8]) int32, GPTQ (zero_offset 1) or
    GPTQ_V2 (0) storage."""
    wa, sb = _c(w16, np.uint16), _c(scales_bits, np.uint16)
    za = None if zeros is None else _c(zeros, np.int32)
    gi = None if g_idx is None else _c(g_idx, np.int32)
    G = 1 if groupsize == -1 else K // groupsize
    qw = np.zeros((K // 8, N), np.int32)
    qz = np.zeros((G, N // 8), np.int32)
    r = _load().oracle_pack(_ptr(wa), _ptr(sb), _ptr(za), _ptr(gi), K, N, groupsize, int(zero_offset),
                            _ptr(qw), _ptr(qz))
    if r < 0:
        raise ValueError("invalid groupsize or g_idx")
    return qw, qz


# ------------------------------------------------------------ composed

@dataclass
class Dequantized:
    q: np.ndarray        # uint8 [K, N], original row order
    z: np.ndarray        # uint8 [G, N]
    gr: np.ndarray       # int32 [K]
    G: int
    w16: np.ndarray      # uint16 fp16 bits [K, N]
    w64: np.ndarray      # float64 [K, N], exact s * (q - z - zero_offset)


def dequantize_layer(qweight, qzeros, scales, g_idx, K: int, N: int, groupsize: int,
                     zero_offset: int = 1, bits: int = 4) -> Dequantized:
    """Steps 1-3: unpack, group map, dequantize.  scales: fp16 array or its
    bits.  zero_offset 1: GPTQ (v1) checkpoints, 0: GPTQ_V2.  bits: 4 or 8."""
    gr, G = row_groups(g_idx, K, groupsize)
    q = unpack_qweight(qweight, K, N) if bits == 4 else unpack_qweight8(qweight, K, N)
    z = unpack_qzeros(qzeros, G, N) if bits == 4 else unpack_qzeros8(qzeros, G, N)
    sb = np.ascontiguousarray(scales).view(np.uint16) if np.asarray(scales).dtype != np.uint16 else scales
    w16, w64 = dequant(q, z, sb, gr, K, N, zero_offset=zero_offset)
    return Dequantized(q, z, gr, G, w16, w64)


def _bits(a):
    a = np.ascontiguousarray(a)
    return a if a.dtype == np.uint16 else a.view(np.uint16)


def reference_output(x_fp16, dq: Dequantized, bias_fp16=None, nthreads=None, exact: bool = False):
    """Step 4: y_ref = x . w16 + bias (or y_exact with the fp64 weights)."""
    x64 = half_bits_to_f64(_bits(x_fp16))
    w = dq.w64 if exact else half_bits_to_f64(dq.w16)
    b64 = None if bias_fp16 is None else half_bits_to_f64(_bits(bias_fp16))
    return linear_f64(x64, w, b64, nthreads)


def reference_output_bf16(x_bf16_bits, dq: Dequantized, bias_fp16=None, nthreads=None):
    """y_ref = x . w16 + bias with bf16 activations (bit patterns)."""
    x64 = bf16_bits_to_f64(x_bf16_bits)
    b64 = None if bias_fp16 is None else half_bits_to_f64(_bits(bias_fp16))
    return linear_f64(x64, half_bits_to_f64(dq.w16), b64, nthreads)


def reference_output_f32(x_f32_bits, dq: Dequantized, bias_fp16=None, nthreads=None):
    """y_ref = x . w16 + bias with fp32 activations (bit patterns, uint32)."""
    x64 = f32_bits_to_f64(x_f32_bits)
    b64 = None if bias_fp16 is None else half_bits_to_f64(_bits(bias_fp16))
    return linear_f64(x64, half_bits_to_f64(dq.w16), b64, nthreads)


def tolerance_rows_f32(x_f32_bits, w16_bits, y_ref: np.ndarray, K: int) -> np.ndarray:
    """tolerance() for fp32 activations and outputs, with max|x| taken per
    row of x:  1e-2 sqrt(K) max|x[m]| max|w| / 64 + 2e-3 |y_ref|.  An fp32
    output adds no rounding of its own, so the relative term is the stated
    one; the per-row max keeps rows scaled far below the others as strict."""
    xa = np.abs(f32_bits_to_f64(x_f32_bits))
    xmax = xa.max(axis=1, keepdims=True) if xa.size else np.zeros((y_ref.shape[0], 1))
    wmax = float(np.max(np.abs(half_bits_to_f64(_bits(w16_bits))))) if np.size(w16_bits) else 0.0
    return 1e-2 * np.sqrt(K) * xmax * wmax / 64.0 + 2e-3 * np.abs(y_ref)


def tolerance_rows_bf16(x_bf16_bits, w16_bits, y_ref: np.ndarray, K: int) -> np.ndarray:
    """tolerance() for bf16 outputs, with max|x| taken per row of x:
    1e-2 sqrt(K) max|x[m]| max|w| / 64 + (2e-3 + 2^-8) |y_ref|.  The stated
    bound is for fp16 outputs; rounding once to bf16 (an 8-bit significand)
    alone can move a value by 2^-8 of itself, so that is added to the
    relative term."""
    xa = np.abs(bf16_bits_to_f64(x_bf16_bits))
    xmax = xa.max(axis=1, keepdims=True) if xa.size else np.zeros((y_ref.shape[0], 1))
    wmax = float(np.max(np.abs(half_bits_to_f64(_bits(w16_bits))))) if np.size(w16_bits) else 0.0
    return 1e-2 * np.sqrt(K) * xmax * wmax / 64.0 + (2e-3 + 2.0 ** -8) * np.abs(y_ref)


def tolerance(x_fp16, w16_bits, y_ref: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound  1e-2 sqrt(K) max|x| max|w| / 64 + 2e-3 |y_ref|,
    with max|x| over the whole x and max|w| over the whole w16."""
    xmax = float(np.max(np.abs(half_bits_to_f64(_bits(x_fp16))))) if np.size(x_fp16) else 0.0
    wmax = float(np.max(np.abs(half_bits_to_f64(_bits(w16_bits))))) if np.size(w16_bits) else 0.0
    return 1e-2 * np.sqrt(K) * xmax * wmax / 64.0 + 2e-3 * np.abs(y_ref)


def linear_layer(qweight, qzeros, scales, g_idx, bias, x, K, N, groupsize, nthreads=None, zero_offset: int = 1):
    """The whole oracle: returns (Dequantized, y_ref, y_exact, tol)."""
    dq = dequantize_layer(qweight, qzeros, scales, g_idx, K, N, groupsize, zero_offset)
    y_ref = reference_output(x, dq, bias, nthreads)
    y_exact = reference_output(x, dq, bias, nthreads, exact=True)
    tol = tolerance(x, dq.w16, y_ref, K)
    return dq, y_ref, y_exact, tol

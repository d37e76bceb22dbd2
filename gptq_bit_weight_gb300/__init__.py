"""Python binding of the GB300 fused GPTQ W4A16 linear layer.

The functions here carry the C names of ``include/gptq_q4.h`` and do nothing
but marshal arguments: every step of the computation runs in the CUDA
library ``libgptq_q4.so`` built in-tree by ``gptq_bit_weight_gb300.build``.
Importing this package without that library raises ImportError: there is no
fallback route.  PyTorch is used only to own device memory and streams
(``Q4Matrix``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgptq_q4.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"the CUDA library {LIB_PATH} is not built; run "
        "`python -c 'import __graft_entry__ as g; g.build()'` (or "
        "`python gptq_bit_weight_gb300/build.py`) first")

_lib = ctypes.CDLL(LIB_PATH)

GPTQ_Q4_OK = 0
GPTQ_Q4_INVALID_ARGUMENT = -1
GPTQ_Q4_UNSUPPORTED = -2
GPTQ_Q4_CUDA_ERROR = -3
GPTQ_Q4_OUT_OF_MEMORY = -4
GPTQ_Q4_DEVICE_FAULT = -5
GPTQ_Q4_PATH_AUTO = 0
GPTQ_Q4_PATH_DECODE = 1
GPTQ_Q4_PATH_PREFILL = 2
GPTQ_Q4_PATH_DECODE_MMA = 3
GPTQ_Q4_PATH_DECODE_TC = 4
GPTQ_Q4_PATH_DECODE_RING = 5
GPTQ_Q4_PATH_DECODE_STREAM = 6
GPTQ_Q4_FORMAT_GPTQ = 0
GPTQ_Q4_FORMAT_GPTQ_V2 = 1
GPTQ_Q4_DTYPE_FP16 = 0
GPTQ_Q4_DTYPE_BF16 = 1
GPTQ_Q4_DTYPE_FP32 = 2

EXPORTED = [
    "gptq_q4_make", "gptq_q4_set_bias", "gptq_q4_reserve", "gptq_q4_matmul", "gptq_q4_dequant",
    "gptq_q4_debug_unpack", "gptq_q4_matmul_unfused", "gptq_q4_gemm_f16", "gptq_q4_set_path",
    "gptq_q4_set_prefill_min_m", "gptq_q4_info", "gptq_q4_device_error", "gptq_q4_free",
    "gptq_q4_last_status", "gptq_q4_last_error", "gptq_q4_launch_count", "gptq_q4_matmul_noalloc",
    "gptq_q4_set_format", "gptq_q4_debug_wait_probe", "gptq_q4_debug_prefill_plan", "gptq_q4_debug_dispatch", "gptq_q4_make_fused", "gptq_q4_pack",
    "gptq_q4_make8", "gptq_q4_set_act_dtype",
]

_P = ctypes.c_void_p
_I = ctypes.c_int


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_sig("gptq_q4_make", _P, _P, _P, _P, _P, _I, _I, _I)
_sig("gptq_q4_make8", _P, _P, _P, _P, _P, _I, _I, _I)
_sig("gptq_q4_set_bias", _I, _P, _P)
_sig("gptq_q4_reserve", _I, _P, _I)
_sig("gptq_q4_matmul", _I, _P, _P, _I, _P, _P)
_sig("gptq_q4_dequant", _I, _P, _P, _P)
_sig("gptq_q4_debug_unpack", _I, _P, _P, _P, _P)
_sig("gptq_q4_matmul_unfused", _I, _P, _P, _I, _P, _P, _P)
_sig("gptq_q4_gemm_f16", _I, _P, _P, _P, _I, _I, _I, _P, _P)
_sig("gptq_q4_set_path", _I, _P, _I)
_sig("gptq_q4_set_prefill_min_m", _I, _P, _I)
_sig("gptq_q4_set_format", _I, _P, _I)
_sig("gptq_q4_set_act_dtype", _I, _P, _I)
_sig("gptq_q4_make_fused", _P, _I, _P, _P, _P, _P, _I, _P, _I)
_sig("gptq_q4_pack", _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P)
_sig("gptq_q4_debug_wait_probe", _I, _P, ctypes.c_uint, _P)
_sig("gptq_q4_debug_prefill_plan", _I, _I, _I, _I, _I, _P)
_sig("gptq_q4_debug_dispatch", _I, _I, _I, _I, _I, _I, _I, _P)
_sig("gptq_q4_info", _I, _P, _P, _P, _P, _P, _P, _P)
_sig("gptq_q4_device_error", _I, _P)
_sig("gptq_q4_free", None, _P)
_sig("gptq_q4_last_status", _I)
_sig("gptq_q4_last_error", ctypes.c_char_p)
_sig("gptq_q4_launch_count", ctypes.c_uint64)
_sig("gptq_q4_matmul_noalloc", _I, _P, _P, _I, _P, _P)

GPTQ_Q4_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class GPTQ4Error(RuntimeError):
    """A non-zero status from the library, with its message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"gptq_q4 status {status}: {message}")
        self.status = status
        self.message = message


def _check(rc: int) -> int:
    if rc != GPTQ_Q4_OK:
        raise GPTQ4Error(rc, gptq_q4_last_error())
    return rc


# ------------------------------------------------------------------ raw C names

def gptq_q4_make(qweight: int, qzeros: int, scales: int, g_idx: int | None, K: int, N: int, groupsize: int) -> int:
    h = _lib.gptq_q4_make(qweight, qzeros, scales, g_idx or None, K, N, groupsize)
    if not h:
        raise GPTQ4Error(gptq_q4_last_status(), gptq_q4_last_error())
    return h


def gptq_q4_make8(qweight: int, qzeros: int, scales: int, g_idx: int | None, K: int, N: int, groupsize: int) -> int:
    """An 8-bit GPTQ layer: qweight [K/4][N], qzeros [G][N/4] (device pointers)."""
    h = _lib.gptq_q4_make8(qweight, qzeros, scales, g_idx or None, K, N, groupsize)
    if not h:
        raise GPTQ4Error(gptq_q4_last_status(), gptq_q4_last_error())
    return h


def gptq_q4_make_fused(qweights, qzeros, scales, g_idx: int | None, K: int, Ns, groupsize: int) -> int:
    """Sequences of device pointers (one per part) and the parts' widths."""
    n = len(Ns)
    arr = lambda seq: (ctypes.c_void_p * n)(*seq)
    widths = (ctypes.c_int * n)(*Ns)
    h = _lib.gptq_q4_make_fused(n, arr(qweights), arr(qzeros), arr(scales), g_idx or None, K, widths, groupsize)
    if not h:
        raise GPTQ4Error(gptq_q4_last_status(), gptq_q4_last_error())
    return h


def gptq_q4_pack(w: int, scales: int, zeros: int | None, g_idx: int | None, K: int, N: int, groupsize: int,
                 fmt: int, qweight: int, qzeros: int, stream: int) -> int:
    return _check(_lib.gptq_q4_pack(w, scales, zeros or None, g_idx or None, K, N, groupsize, fmt, qweight, qzeros,
                                    stream or None))


def pack(w, scales, zeros=None, g_idx=None, groupsize: int = 128, fmt: int = 0):
    """Torch CUDA tensors in: w [K, N] fp16, scales [G, N] fp16, zeros [G, N]
    int (effective zero points) or None, g_idx [K] or None.  Returns
    (qweight [K/8, N], qzeros [G, N/8]) int32 checkpoint tensors."""
    import torch
    K, N = w.shape
    G = 1 if groupsize == -1 else K // groupsize
    w = w.to(torch.float16).contiguous()
    scales = scales.to(torch.float16).contiguous()
    zeros = None if zeros is None else zeros.to(torch.int32).contiguous()
    g_idx = None if g_idx is None else g_idx.to(torch.int32).contiguous()
    qweight = torch.empty((K // 8, N), dtype=torch.int32, device=w.device)
    qzeros = torch.empty((G, N // 8), dtype=torch.int32, device=w.device)
    gptq_q4_pack(w.data_ptr(), scales.data_ptr(), None if zeros is None else zeros.data_ptr(),
                 None if g_idx is None else g_idx.data_ptr(), K, N, groupsize, fmt, qweight.data_ptr(),
                 qzeros.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return qweight, qzeros


def gptq_q4_set_bias(h: int, bias: int | None) -> int:
    return _check(_lib.gptq_q4_set_bias(h, bias or None))


def gptq_q4_reserve(h: int, max_m: int) -> int:
    return _check(_lib.gptq_q4_reserve(h, max_m))


def gptq_q4_matmul(h: int, x: int, M: int, out: int, stream: int) -> int:
    return _check(_lib.gptq_q4_matmul(h, x or None, M, out or None, stream or None))


def gptq_q4_dequant(h: int, temp_dq: int, stream: int) -> int:
    return _check(_lib.gptq_q4_dequant(h, temp_dq, stream or None))


def gptq_q4_debug_unpack(h: int, q: int | None, z: int | None, stream: int) -> int:
    return _check(_lib.gptq_q4_debug_unpack(h, q or None, z or None, stream or None))


def gptq_q4_matmul_unfused(h: int, x: int, M: int, temp_dq: int, out: int, stream: int) -> int:
    return _check(_lib.gptq_q4_matmul_unfused(h, x or None, M, temp_dq or None, out or None, stream or None))


def gptq_q4_gemm_f16(a: int, b: int, bias: int | None, M: int, K: int, N: int, out: int, stream: int) -> int:
    return _check(_lib.gptq_q4_gemm_f16(a or None, b or None, bias or None, M, K, N, out or None, stream or None))


def gptq_q4_set_path(h: int, path: int) -> int:
    return _check(_lib.gptq_q4_set_path(h, path))


def gptq_q4_set_prefill_min_m(h: int, min_m: int) -> int:
    return _check(_lib.gptq_q4_set_prefill_min_m(h, min_m))


def gptq_q4_set_format(h: int, fmt: int) -> int:
    return _check(_lib.gptq_q4_set_format(h, fmt))


def gptq_q4_set_act_dtype(h: int, dtype: int) -> int:
    return _check(_lib.gptq_q4_set_act_dtype(h, dtype))


def gptq_q4_debug_wait_probe(status: int, limit_us: int, stream: int) -> int:
    return _check(_lib.gptq_q4_debug_wait_probe(status, limit_us, stream or None))


KERNELS = ("prefill", "decode_reg", "decode_stream", "decode_ring", "decode_tc")


def gptq_q4_debug_dispatch(M: int, K: int, N: int, groupsize: int, path: int, sms: int) -> str:
    k = ctypes.c_int()
    _check(_lib.gptq_q4_debug_dispatch(M, K, N, groupsize, path, sms, ctypes.byref(k)))
    return KERNELS[k.value]


def gptq_q4_debug_prefill_plan(M: int, K: int, N: int, sms: int) -> dict:
    out = (ctypes.c_int * 7)()
    _check(_lib.gptq_q4_debug_prefill_plan(M, K, N, sms, out))
    return {"bm": out[0], "bn": out[1], "stream_k": out[2], "grid": out[3], "max_pieces": out[4],
            "piece0_finishes": out[5], "stage_rows": out[6]}


def gptq_q4_info(h: int) -> dict:
    K, N, gs, G, act = (ctypes.c_int() for _ in range(5))
    nb = ctypes.c_size_t()
    _check(_lib.gptq_q4_info(h, ctypes.byref(K), ctypes.byref(N), ctypes.byref(gs), ctypes.byref(G),
                             ctypes.byref(act), ctypes.byref(nb)))
    return {"K": K.value, "N": N.value, "groupsize": gs.value, "G": G.value, "act_order": bool(act.value),
            "device_bytes": nb.value}


def gptq_q4_device_error(h: int) -> int:
    return _check(_lib.gptq_q4_device_error(h))


def gptq_q4_free(h: int | None) -> None:
    if h:
        _lib.gptq_q4_free(h)


def gptq_q4_last_status() -> int:
    return _lib.gptq_q4_last_status()


def gptq_q4_last_error() -> str:
    msg = _lib.gptq_q4_last_error()
    return msg.decode() if msg else ""


def gptq_q4_launch_count() -> int:
    return int(_lib.gptq_q4_launch_count())


def gptq_q4_matmul_noalloc(h: int, x: int, M: int, out: int, stream: int) -> int:
    """gptq_q4_matmul's decode path with its scratch in the library's fixed
    device array: allocates nothing (see include/gptq_q4.h)."""
    return _check(_lib.gptq_q4_matmul_noalloc(h, x or None, M, out or None, stream or None))


# --------------------------------------------------------- torch marshalling

class Q4Matrix:
    """A handle built from torch CUDA tensors (the Q4Matrix / q4_matmul pair
    of the Lorax ExLlama v1 layer).  Only moves pointers and shapes; the
    library does the work and copies what it keeps."""

    def __init__(self, qweight, qzeros, scales, g_idx=None, bias=None, groupsize: int = 128, bits: int = 4):
        import torch
        assert qweight.is_cuda and qweight.dtype == torch.int32 and qweight.dim() == 2
        assert bits in (4, 8)
        K = qweight.shape[0] * (32 // bits)
        N = qweight.shape[1]
        qweight, qzeros, scales = qweight.contiguous(), qzeros.contiguous(), scales.contiguous()
        assert scales.dtype == torch.float16
        g_idx = None if g_idx is None else g_idx.to(torch.int32).contiguous()
        torch.cuda.current_stream().synchronize()
        self.K, self.N, self.groupsize, self.bits = K, N, groupsize, bits
        self.device = qweight.device
        make = gptq_q4_make if bits == 4 else gptq_q4_make8
        self.handle = make(qweight.data_ptr(), qzeros.data_ptr(), scales.data_ptr(),
                           None if g_idx is None else g_idx.data_ptr(), K, N, groupsize)
        if bias is not None:
            b = bias.to(torch.float16).contiguous()
            gptq_q4_set_bias(self.handle, b.data_ptr())

    @classmethod
    def fused(cls, parts, g_idx=None, biases=None, groupsize: int = 128):
        """One handle over projections that read the same input (e.g. Q, K, V),
        concatenated along N; parts = [(qweight, qzeros, scales), ...] torch
        CUDA tensors.  matmul returns [.., sum N_i]; part i is the column range
        [sum_{j<i} N_j, + N_i)."""
        import torch
        self = cls.__new__(cls)
        parts = [(q.contiguous(), z.contiguous(), s.contiguous()) for q, z, s in parts]
        K = parts[0][0].shape[0] * 8
        Ns = [q.shape[1] for q, _, _ in parts]
        g_idx = None if g_idx is None else g_idx.to(torch.int32).contiguous()
        torch.cuda.current_stream().synchronize()
        self.K, self.N, self.groupsize = K, sum(Ns), groupsize
        self.device = parts[0][0].device
        self.parts = Ns
        self.handle = gptq_q4_make_fused([q.data_ptr() for q, _, _ in parts], [z.data_ptr() for _, z, _ in parts],
                                         [s.data_ptr() for _, _, s in parts],
                                         None if g_idx is None else g_idx.data_ptr(), K, Ns, groupsize)
        if biases is not None:
            b = torch.cat([bb.to(torch.float16) for bb in biases]).contiguous()
            gptq_q4_set_bias(self.handle, b.data_ptr())
        return self

    def info(self) -> dict:
        return gptq_q4_info(self.handle)

    def reserve(self, max_m: int) -> None:
        gptq_q4_reserve(self.handle, max_m)

    def set_path(self, path: int) -> None:
        gptq_q4_set_path(self.handle, path)

    def set_prefill_min_m(self, m: int) -> None:
        gptq_q4_set_prefill_min_m(self.handle, m)

    def set_format(self, fmt: int) -> None:
        gptq_q4_set_format(self.handle, fmt)

    def set_act_dtype(self, dtype) -> None:
        """torch.float16 (default), torch.bfloat16 or torch.float32: the type of x and y."""
        import torch
        code = {torch.float16: GPTQ_Q4_DTYPE_FP16, torch.bfloat16: GPTQ_Q4_DTYPE_BF16,
                torch.float32: GPTQ_Q4_DTYPE_FP32}[dtype]
        gptq_q4_set_act_dtype(self.handle, code)
        self.act_dtype = dtype

    def _act_dtype(self):
        import torch
        return getattr(self, "act_dtype", torch.float16)

    def matmul(self, x, out=None):
        import torch
        dt = self._act_dtype()
        shape = x.shape
        x2 = x.reshape(-1, self.K)
        if x2.dtype != dt or not x2.is_contiguous():
            x2 = x2.to(dt).contiguous()
        M = x2.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=dt, device=x2.device)
        gptq_q4_matmul(self.handle, x2.data_ptr(), M, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        return out.reshape(*shape[:-1], self.N)

    __call__ = matmul

    def matmul_unfused(self, x, temp_dq=None):
        import torch
        dt = self._act_dtype()
        x2 = x.reshape(-1, self.K).to(dt).contiguous()
        M = x2.shape[0]
        if temp_dq is None:
            temp_dq = torch.empty((self.K, self.N), dtype=torch.float16, device=x2.device)
        out = torch.empty((M, self.N), dtype=dt, device=x2.device)
        gptq_q4_matmul_unfused(self.handle, x2.data_ptr(), M, temp_dq.data_ptr(), out.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
        return out

    def dequant(self, out=None):
        import torch
        if out is None:
            out = torch.empty((self.K, self.N), dtype=torch.float16, device=self.device)
        gptq_q4_dequant(self.handle, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        return out

    def debug_unpack(self):
        import torch
        G = gptq_q4_info(self.handle)["G"]
        q = torch.empty((self.K, self.N), dtype=torch.uint8, device=self.device)
        z = torch.empty((G, self.N), dtype=torch.uint8, device=self.device)
        gptq_q4_debug_unpack(self.handle, q.data_ptr(), z.data_ptr(), torch.cuda.current_stream().cuda_stream)
        return q, z

    def device_error(self) -> None:
        gptq_q4_device_error(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            gptq_q4_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gemm_f16(a, b, bias=None):
    """out = a . b + bias on the tcgen05 GEMM (torch tensors in, out)."""
    import torch
    M, K = a.shape
    N = b.shape[1]
    out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    gptq_q4_gemm_f16(a.data_ptr(), b.data_ptr(), None if bias is None else bias.data_ptr(), M, K, N,
                     out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out

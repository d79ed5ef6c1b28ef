"""ctypes binding of libqlora_nf4.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; PyTorch only supplies
device memory (``torch.empty``) and the current stream.  There is no fallback:
if the library is missing or the device is not sm_103, calls raise.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqlora_nf4.so")

QLORA_OK = 0
QLORA_ERR_INVALID_ARGUMENT = 1
QLORA_ERR_UNSUPPORTED = 2
QLORA_ERR_CUDA = 3
QLORA_ERR_TIMEOUT = 4
QLORA_ERR_NONFINITE = 5

DTYPE_F32 = 0
DTYPE_BF16 = 1

ACCUM_DX = 1
ACCUM_DA = 2
ACCUM_DB = 4

ADAMW_PREFETCH = 1

# every symbol include/qlora_nf4.h declares
EXPORTS = (
    "qlora_nf4_quantize_workspace_bytes",
    "qlora_nf4_quantize",
    "qlora_nf4_quantize_noalloc",
    "qlora_nf4_dequantize",
    "qlora_nf4_merge",
    "qlora_lowrank_update",
    "qlora_linear_fwd_workspace_bytes",
    "qlora_linear_fwd",
    "qlora_linear_bwd_workspace_bytes",
    "qlora_linear_bwd",
    "qlora_dropout_mask",
    "qlora_linear_fwd_dropout",
    "qlora_linear_bwd_dropout",
    "qlora_linear_fwd_grouped_workspace_bytes",
    "qlora_linear_fwd_grouped",
    "qlora_adamw_step",
    "qlora_silu_mul_fwd",
    "qlora_silu_mul_bwd",
    "qlora_get_status",
    "qlora_strerror",
    "qlora_last_error",
    "qlora_set_wait_limit_ns",
    "qlora_selftest_wait_timeout",
    "qlora_device_sm_count",
    "qlora_copy_many",
    "qlora_launch_count",
    "qlora_profile_enable",
    "qlora_profile_collect",
    "qlora_profile_name",
    "qlora_profile_total_ms",
    "qlora_profile_calls",
    "qlora_profile_reset",
)


class QloraError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


class _Weight(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("absmax_q", ctypes.c_void_p),
        ("absmax_step", ctypes.c_void_p),
        ("absmax_mean", ctypes.c_void_p),
        ("n", ctypes.c_int64),
        ("k", ctypes.c_int64),
    ]


class _Problem(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p),
        ("m", ctypes.c_int64),
        ("w", ctypes.POINTER(_Weight)),
        ("lora_a", ctypes.c_void_p),
        ("lora_b", ctypes.c_void_p),
        ("r", ctypes.c_int),
        ("alpha", ctypes.c_float),
        ("y", ctypes.c_void_p),
        ("t_save", ctypes.c_void_p),
    ]


class _Copy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class _AdamwTensor(ctypes.Structure):
    _fields_ = [
        ("master", ctypes.c_void_p),
        ("param", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("exp_avg", ctypes.c_void_p),
        ("exp_avg_sq", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
    ]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)
_PW = ctypes.POINTER(_Weight)
_PP = ctypes.POINTER(_Problem)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libqlora_nf4.so not built (run __graft_entry__.build() or "
                           "python -m bit_quantized_fine_nf4_b300.build_lib)")
    lib = ctypes.CDLL(p)
    c_int, c_float = ctypes.c_int, ctypes.c_float
    sig = {
        "qlora_nf4_quantize_workspace_bytes": (c_int, [_I64, _I64, _PSZ]),
        "qlora_nf4_quantize": (c_int, [_P, c_int, _I64, _I64, _PW, _P, _SZ, _P]),
        "qlora_nf4_quantize_noalloc": (c_int, [_P, c_int, _I64, _I64, _PW, _P]),
        "qlora_nf4_dequantize": (c_int, [_PW, _P, _P]),
        "qlora_nf4_merge": (c_int, [_PW, _P, _P, c_int, c_float, _P, _P]),
        "qlora_lowrank_update": (c_int, [_P, c_int, _I64, _I64, _PW, _P, _P, c_int, c_float, _P, _P]),
        "qlora_linear_fwd_workspace_bytes": (c_int, [_I64, _I64, _I64, c_int, _PSZ]),
        "qlora_linear_fwd": (c_int, [_P, _I64, _PW, _P, _P, c_int, c_float, _P, _P, _P, _SZ, _P]),
        "qlora_linear_bwd_workspace_bytes": (c_int, [_I64, _I64, _I64, c_int, _PSZ]),
        "qlora_linear_bwd": (c_int, [_P, _P, _I64, _PW, _P, _P, c_int, c_float, _P, _P, _P, _P, c_int, _P, _SZ,
                                     _P]),
        "qlora_dropout_mask": (c_int, [ctypes.c_uint64, ctypes.c_uint64, _I64, _I64, c_float, _P, _P]),
        "qlora_linear_fwd_dropout": (c_int, [_P, _I64, _PW, _P, _P, c_int, c_float, _P, c_float, _P, _P, _P, _P, _SZ,
                                             _P]),
        "qlora_linear_bwd_dropout": (c_int, [_P, _P, _I64, _PW, _P, _P, c_int, c_float, _P, c_float, _P, _P, _P, _P,
                                             c_int, _P, _SZ, _P]),
        "qlora_linear_fwd_grouped_workspace_bytes": (c_int, [_PP, c_int, _PSZ]),
        "qlora_linear_fwd_grouped": (c_int, [_PP, c_int, _P, _SZ, _P]),
        "qlora_adamw_step": (c_int, [ctypes.POINTER(_AdamwTensor), c_int, c_float, c_float, c_float, c_float,
                                     c_float, _I64, c_int, _P]),
        "qlora_silu_mul_fwd": (c_int, [_P, _P, _P, _I64, _P]),
        "qlora_silu_mul_bwd": (c_int, [_P, _P, _P, _P, _P, _I64, _P]),
        "qlora_get_status": (c_int, [_P]),
        "qlora_strerror": (ctypes.c_char_p, [c_int]),
        "qlora_last_error": (ctypes.c_char_p, []),
        "qlora_set_wait_limit_ns": (c_int, [ctypes.c_uint64]),
        "qlora_selftest_wait_timeout": (c_int, [ctypes.c_uint64, _P]),
        "qlora_device_sm_count": (c_int, []),
        "qlora_copy_many": (c_int, [ctypes.POINTER(_Copy), c_int, _P]),
        "qlora_launch_count": (ctypes.c_ulonglong, []),
        "qlora_profile_enable": (c_int, [c_int]),
        "qlora_profile_collect": (c_int, []),
        "qlora_profile_name": (ctypes.c_char_p, [c_int]),
        "qlora_profile_total_ms": (ctypes.c_double, [c_int]),
        "qlora_profile_calls": (ctypes.c_longlong, [c_int]),
        "qlora_profile_reset": (c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != QLORA_OK:
        lib = load()
        raise QloraError(rc, "%s: %s" % (lib.qlora_strerror(rc).decode(), lib.qlora_last_error().decode()))


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class NF4Weight:
    """Device record of a quantised [n, k] weight (see include/qlora_nf4.h)."""

    codes: torch.Tensor        # uint8 [n*k/2]
    absmax_q: torch.Tensor     # int8 [n*k/64]
    absmax_step: torch.Tensor  # float32 [ceil(n*k/64/256)]
    absmax_mean: torch.Tensor  # float32 [1]
    n: int
    k: int

    @staticmethod
    def empty(n: int, k: int, device="cuda") -> "NF4Weight":
        n_a = n * k // 64
        return NF4Weight(
            codes=torch.empty(n * k // 2, dtype=torch.uint8, device=device),
            absmax_q=torch.empty(n_a, dtype=torch.int8, device=device),
            absmax_step=torch.empty((n_a + 255) // 256, dtype=torch.float32, device=device),
            absmax_mean=torch.empty(1, dtype=torch.float32, device=device),
            n=n, k=k)

    def c_struct(self) -> _Weight:
        return _Weight(_ptr(self.codes), _ptr(self.absmax_q), _ptr(self.absmax_step), _ptr(self.absmax_mean),
                       self.n, self.k)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.codes, self.absmax_q, self.absmax_step, self.absmax_mean))


def _ws(nbytes: int, device, workspace: torch.Tensor | None):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small: need %d bytes" % nbytes)
        return workspace, workspace.numel() * workspace.element_size()
    n = max(nbytes, 256)
    return torch.empty(n, dtype=torch.uint8, device=device), n


def quantize_workspace_bytes(n: int, k: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().qlora_nf4_quantize_workspace_bytes(n, k, ctypes.byref(b)))
    return b.value


def quantize(w: torch.Tensor, out: NF4Weight | None = None, workspace=None, stream=None) -> NF4Weight:
    """NF4 + double-quant record of a float32 / bfloat16 [n, k] weight."""
    lib = load()
    n, k = w.shape
    if out is None:
        out = NF4Weight.empty(n, k, w.device)
    dtype = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}.get(w.dtype)
    if dtype is None:
        raise ValueError("weight must be float32 or bfloat16")
    ws, wsb = _ws(quantize_workspace_bytes(n, k), w.device, workspace)
    rec = out.c_struct()
    _check(lib.qlora_nf4_quantize(_ptr(w), dtype, n, k, ctypes.byref(rec), _ptr(ws), wsb, _stream(stream)))
    return out


def quantize_noalloc(w: torch.Tensor, out: NF4Weight | None = None, stream=None) -> NF4Weight:
    """qlora_nf4_quantize_noalloc: same result as quantize(), scratch from the library's fixed
    device array instead of a workspace (n*k <= 2^26; calls must not overlap on the GPU)."""
    lib = load()
    n, k = w.shape
    if out is None:
        out = NF4Weight.empty(n, k, w.device)
    dtype = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}.get(w.dtype)
    if dtype is None:
        raise ValueError("weight must be float32 or bfloat16")
    rec = out.c_struct()
    _check(lib.qlora_nf4_quantize_noalloc(_ptr(w), dtype, n, k, ctypes.byref(rec), _stream(stream)))
    return out


def dequantize(rec: NF4Weight, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    lib = load()
    if out is None:
        out = torch.empty((rec.n, rec.k), dtype=torch.bfloat16, device=rec.codes.device)
    c = rec.c_struct()
    _check(lib.qlora_nf4_dequantize(ctypes.byref(c), _ptr(out), _stream(stream)))
    return out


def merge(rec: NF4Weight, lora_a: torch.Tensor, lora_b: torch.Tensor, alpha: float, out: torch.Tensor | None = None,
          stream=None) -> torch.Tensor:
    """bf16 [n, k] = bf16(deq(W) + (alpha/r) B A): the merged weight for export (qlora_nf4_merge)."""
    lib = load()
    if out is None:
        out = torch.empty((rec.n, rec.k), dtype=torch.bfloat16, device=rec.codes.device)
    c = rec.c_struct()
    _check(lib.qlora_nf4_merge(ctypes.byref(c), _ptr(lora_a), _ptr(lora_b), lora_a.shape[0], float(alpha), _ptr(out),
                               _stream(stream)))
    return out


def lowrank_update(w: torch.Tensor, sub: NF4Weight | None = None, lora_a: torch.Tensor | None = None,
                   lora_b: torch.Tensor | None = None, coef: float = 0.0, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """float32 [n, k] = (W - deq(sub)) + coef B A (qlora_lowrank_update); sub and the LoRA pair are optional."""
    lib = load()
    n, k = w.shape
    dtype = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}.get(w.dtype)
    if dtype is None:
        raise ValueError("weight must be float32 or bfloat16")
    if out is None:
        out = torch.empty((n, k), dtype=torch.float32, device=w.device)
    r = 0 if lora_a is None else lora_a.shape[0]
    cs = ctypes.byref(sub.c_struct()) if sub is not None else None
    _check(lib.qlora_lowrank_update(_ptr(w), dtype, n, k, cs, _ptr(lora_a), _ptr(lora_b), r, float(coef), _ptr(out),
                                    _stream(stream)))
    return out


def fwd_workspace_bytes(m: int, n: int, k: int, r: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().qlora_linear_fwd_workspace_bytes(m, n, k, r, ctypes.byref(b)))
    return b.value


def bwd_workspace_bytes(m: int, n: int, k: int, r: int) -> int:
    b = ctypes.c_size_t(0)
    _check(load().qlora_linear_bwd_workspace_bytes(m, n, k, r, ctypes.byref(b)))
    return b.value


def linear_fwd(x: torch.Tensor, rec: NF4Weight, lora_a: torch.Tensor, lora_b: torch.Tensor, alpha: float,
               y: torch.Tensor | None = None, t_save: torch.Tensor | None = None, workspace=None, stream=None):
    """Y = X deq(W)^T + (alpha/r) (X A^T) B^T.  Returns (y bf16 [m, n], t_save f32 [m, r])."""
    lib = load()
    m = x.shape[0]
    r = lora_a.shape[0]
    dev = x.device
    if y is None:
        y = torch.empty((m, rec.n), dtype=torch.bfloat16, device=dev)
    if t_save is None:
        t_save = torch.empty((m, r), dtype=torch.float32, device=dev)
    ws, wsb = _ws(fwd_workspace_bytes(m, rec.n, rec.k, r), dev, workspace)
    c = rec.c_struct()
    _check(lib.qlora_linear_fwd(_ptr(x), m, ctypes.byref(c), _ptr(lora_a), _ptr(lora_b), r, float(alpha),
                                _ptr(y), _ptr(t_save), _ptr(ws), wsb, _stream(stream)))
    return y, t_save


def linear_bwd(dy: torch.Tensor, x: torch.Tensor, rec: NF4Weight, lora_a: torch.Tensor, lora_b: torch.Tensor,
               alpha: float, t_save: torch.Tensor, dx: torch.Tensor | None = None, da: torch.Tensor | None = None,
               db: torch.Tensor | None = None, flags: int = 0, workspace=None, stream=None):
    """Returns (dx bf16 [m, k], da f32 [r, k], db f32 [n, r]); no gradient for W."""
    lib = load()
    m = x.shape[0]
    r = lora_a.shape[0]
    dev = x.device
    if dx is None:
        dx = torch.empty((m, rec.k), dtype=torch.bfloat16, device=dev)
    if da is None:
        da = torch.empty((r, rec.k), dtype=torch.float32, device=dev)
    if db is None:
        db = torch.empty((rec.n, r), dtype=torch.float32, device=dev)
    ws, wsb = _ws(bwd_workspace_bytes(m, rec.n, rec.k, r), dev, workspace)
    c = rec.c_struct()
    _check(lib.qlora_linear_bwd(_ptr(dy), _ptr(x), m, ctypes.byref(c), _ptr(lora_a), _ptr(lora_b), r, float(alpha),
                                _ptr(t_save), _ptr(dx), _ptr(da), _ptr(db), int(flags), _ptr(ws), wsb,
                                _stream(stream)))
    return dx, da, db


def dropout_mask(seed: int, offset: int, m: int, k: int, p: float, out: torch.Tensor | None = None,
                 device="cuda", stream=None) -> torch.Tensor:
    """uint8 [m, k/8] keep bits of LoRA dropout (qlora_dropout_mask)."""
    if out is None:
        out = torch.empty((m, k // 8), dtype=torch.uint8, device=device)
    _check(load().qlora_dropout_mask(int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), m, k, float(p),
                                     _ptr(out) if m else None, _stream(stream)))
    return out


def linear_fwd_dropout(x: torch.Tensor, rec: NF4Weight, lora_a: torch.Tensor, lora_b: torch.Tensor, alpha: float,
                       mask: torch.Tensor, p: float, y=None, t_save=None, x_drop=None, workspace=None, stream=None):
    """Forward with dropout on the LoRA input.  Returns (y, t_save, x_drop)."""
    lib = load()
    m = x.shape[0]
    r = lora_a.shape[0]
    dev = x.device
    if y is None:
        y = torch.empty((m, rec.n), dtype=torch.bfloat16, device=dev)
    if t_save is None:
        t_save = torch.empty((m, r), dtype=torch.float32, device=dev)
    if x_drop is None:
        x_drop = torch.empty_like(x)
    ws, wsb = _ws(fwd_workspace_bytes(m, rec.n, rec.k, r), dev, workspace)
    c = rec.c_struct()
    _check(lib.qlora_linear_fwd_dropout(_ptr(x), m, ctypes.byref(c), _ptr(lora_a), _ptr(lora_b), r, float(alpha),
                                        _ptr(mask), float(p), _ptr(x_drop), _ptr(y), _ptr(t_save), _ptr(ws), wsb,
                                        _stream(stream)))
    return y, t_save, x_drop


def linear_bwd_dropout(dy: torch.Tensor, x_drop: torch.Tensor, rec: NF4Weight, lora_a: torch.Tensor,
                       lora_b: torch.Tensor, alpha: float, mask: torch.Tensor, p: float, t_save: torch.Tensor,
                       dx=None, da=None, db=None, flags: int = 0, workspace=None, stream=None):
    """Backward of linear_fwd_dropout.  Returns (dx, da, db)."""
    lib = load()
    m = x_drop.shape[0]
    r = lora_a.shape[0]
    dev = x_drop.device
    if dx is None:
        dx = torch.empty((m, rec.k), dtype=torch.bfloat16, device=dev)
    if da is None:
        da = torch.empty((r, rec.k), dtype=torch.float32, device=dev)
    if db is None:
        db = torch.empty((rec.n, r), dtype=torch.float32, device=dev)
    ws, wsb = _ws(bwd_workspace_bytes(m, rec.n, rec.k, r), dev, workspace)
    c = rec.c_struct()
    _check(lib.qlora_linear_bwd_dropout(_ptr(dy), _ptr(x_drop), m, ctypes.byref(c), _ptr(lora_a), _ptr(lora_b), r,
                                        float(alpha), _ptr(mask), float(p), _ptr(t_save), _ptr(dx), _ptr(da), _ptr(db),
                                        int(flags), _ptr(ws), wsb, _stream(stream)))
    return dx, da, db


class GroupedForward:
    """A prepared list of small-token problems for qlora_linear_fwd_grouped.

    ``problems``: sequence of (x [m, k] bf16, NF4Weight, A [r, k], B [n, r], alpha, y [m, n] bf16 or None,
    t_save [m, r] f32 or None).  The ctypes array and the workspace are built once; ``run()`` is one call.
    """

    def __init__(self, problems, workspace=None):
        lib = load()
        self._keep = []
        n = len(problems)
        self.arr = (_Problem * max(n, 1))()
        self.ys = []
        for i, (x, rec, a, b, alpha, y, t_save) in enumerate(problems):
            if y is None:
                y = torch.empty((x.shape[0], rec.n), dtype=torch.bfloat16, device=x.device)
            w = rec.c_struct()
            self._keep.append(w)
            self.arr[i] = _Problem(_ptr(x), x.shape[0], ctypes.pointer(w), _ptr(a), _ptr(b), a.shape[0],
                                   float(alpha), _ptr(y), _ptr(t_save) if t_save is not None else None)
            self.ys.append(y)
        self.count = n
        b_ = ctypes.c_size_t(0)
        _check(lib.qlora_linear_fwd_grouped_workspace_bytes(self.arr, n, ctypes.byref(b_)))
        dev = problems[0][0].device if n else "cuda"
        if workspace is None:  # the grouped call's workspace starts zero-filled (its counters)
            workspace = torch.zeros(max(b_.value, 256), dtype=torch.uint8, device=dev)
        self.ws, self.wsb = _ws(b_.value, dev, workspace)

    def run(self, stream=None):
        _check(load().qlora_linear_fwd_grouped(self.arr, self.count, _ptr(self.ws), self.wsb, _stream(stream)))
        return self.ys


def linear_fwd_grouped(problems, workspace=None, stream=None):
    """One qlora_linear_fwd_grouped call; returns the list of y tensors."""
    return GroupedForward(problems, workspace).run(stream)


def _addr(x) -> int | None:
    """Device address of a tensor, or an integer address as given (e.g. managed memory)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "ptr"):
        return int(x.ptr)
    return _ptr(x)


class AdamwStep:
    """A prepared tensor list for qlora_adamw_step: the ctypes array is built once (the list of
    dicts with keys ``master``, ``param`` (bf16 copy or None), ``grad``, ``exp_avg``,
    ``exp_avg_sq`` and, when the entries are raw addresses or ManagedBuffer objects, ``numel``),
    so that ``run()`` per optimizer step is a single call."""

    def __init__(self, tensors):
        self.count = len(tensors)
        self.arr = (_AdamwTensor * max(self.count, 1))()
        self._keep = list(tensors)
        for i, t in enumerate(tensors):
            numel = t.get("numel")
            if numel is None:
                numel = t["grad"].numel()
            self.arr[i] = _AdamwTensor(_addr(t["master"]), _addr(t.get("param")), _addr(t["grad"]),
                                       _addr(t["exp_avg"]), _addr(t["exp_avg_sq"]), int(numel))

    def run(self, lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0,
            step: int = 1, prefetch: bool = False, stream=None) -> None:
        _check(load().qlora_adamw_step(self.arr, self.count, float(lr), float(beta1), float(beta2), float(eps),
                                       float(weight_decay), int(step), ADAMW_PREFETCH if prefetch else 0,
                                       _stream(stream)))


def adamw_step(tensors, lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
               weight_decay: float = 0.0, step: int = 1, prefetch: bool = False, stream=None) -> None:
    """One AdamW step (qlora_adamw_step) on a list of dicts (see AdamwStep).  All tensors of the
    list go in one launch per 240 tensors."""
    AdamwStep(tensors).run(lr, beta1, beta2, eps, weight_decay, step, prefetch, stream)


class ManagedBuffer:
    """Memory from cudaMallocManaged: one address valid on the GPU and the host, paged
    between them by the driver (where the paged optimizer keeps its state).  Allocated by
    the caller through the CUDA runtime, never by the library."""

    _rt = None

    @classmethod
    def _runtime(cls):
        if cls._rt is None:
            here = os.path.dirname(torch.__file__)
            cands = [os.path.join(here, "..", "nvidia", "cu13", "lib", "libcudart.so.13"), "libcudart.so.13",
                     "/usr/local/cuda/lib64/libcudart.so"]
            err = None
            for c in cands:
                try:
                    cls._rt = ctypes.CDLL(c)
                    break
                except OSError as e:
                    err = e
            if cls._rt is None:
                raise RuntimeError("CUDA runtime library not found: %s" % err)
            cls._rt.cudaMallocManaged.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
            cls._rt.cudaFree.argtypes = [ctypes.c_void_p]
            cls._rt.cudaDeviceSynchronize.argtypes = []
        return cls._rt

    def __init__(self, nbytes: int):
        rt = self._runtime()
        p = ctypes.c_void_p()
        rc = rt.cudaMallocManaged(ctypes.byref(p), ctypes.c_size_t(max(int(nbytes), 16)), 1)  # cudaMemAttachGlobal
        if rc != 0:
            raise RuntimeError("cudaMallocManaged failed (%d)" % rc)
        self.ptr = p.value
        self.nbytes = int(nbytes)

    def host_view(self, ctype, count: int):
        """A numpy view of the buffer on the host (synchronise the device before reading)."""
        import numpy as np
        return np.ctypeslib.as_array((ctype * count).from_address(self.ptr))

    def free(self) -> None:
        if self.ptr:
            self._runtime().cudaFree(ctypes.c_void_p(self.ptr))
            self.ptr = 0


def silu_mul_fwd(g: torch.Tensor, u: torch.Tensor, h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    lib = load()
    if h is None:
        h = torch.empty_like(g)
    _check(lib.qlora_silu_mul_fwd(_ptr(g), _ptr(u), _ptr(h), g.numel(), _stream(stream)))
    return h


def silu_mul_bwd(dh: torch.Tensor, g: torch.Tensor, u: torch.Tensor, dg=None, du=None, stream=None):
    lib = load()
    if dg is None:
        dg = torch.empty_like(g)
    if du is None:
        du = torch.empty_like(u)
    _check(lib.qlora_silu_mul_bwd(_ptr(dh), _ptr(g), _ptr(u), _ptr(dg), _ptr(du), g.numel(), _stream(stream)))
    return dg, du


def get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the latched device status code."""
    return load().qlora_get_status(_stream(stream))


def check_status(stream=None) -> None:
    _check(get_status(stream))


def set_wait_limit_ns(ns: int) -> None:
    _check(load().qlora_set_wait_limit_ns(int(ns)))


def selftest_wait_timeout(wait_ns: int, stream=None) -> None:
    _check(load().qlora_selftest_wait_timeout(int(wait_ns), _stream(stream)))


def device_sm_count() -> int:
    return load().qlora_device_sm_count()


def copy_many(pairs, stream=None) -> None:
    """Copy each (dst, src) pair of equally sized contiguous tensors (device, or pinned host)
    in stream order, the pieces spread over the library's copy streams (qlora_copy_many)."""
    arr = (_Copy * max(1, len(pairs)))()
    for i, (dst, src) in enumerate(pairs):
        if not (dst.is_contiguous() and src.is_contiguous()):
            raise ValueError("copy_many: tensors must be contiguous")
        nb = dst.numel() * dst.element_size()
        if nb != src.numel() * src.element_size():
            raise ValueError("copy_many: pair %d has %d and %d bytes" % (i, nb, src.numel() * src.element_size()))
        arr[i] = _Copy(dst.data_ptr(), src.data_ptr(), nb)
    _check(load().qlora_copy_many(arr, len(pairs), _stream(stream)))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().qlora_launch_count())


def profile_enable(on: bool) -> None:
    _check(load().qlora_profile_enable(1 if on else 0))


def profile_reset() -> None:
    _check(load().qlora_profile_reset())


def profile_read() -> dict:
    """{launcher name: (total ms, calls)} of the launches recorded while profiling was on."""
    lib = load()
    n = lib.qlora_profile_collect()
    out = {}
    for i in range(n):
        calls = int(lib.qlora_profile_calls(i))
        if calls:
            out[lib.qlora_profile_name(i).decode()] = (float(lib.qlora_profile_total_ms(i)), calls)
    return out

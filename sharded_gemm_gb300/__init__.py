"""Python binding of libtp.so, the sharded-GEMM C ABI (include/tp_api.h).

Argument marshalling only: every function here checks that the tensors it
is given can be described to the C ABI (device, dtype, row-major strides),
passes their device pointers and sizes, and enqueues the call on the current
torch CUDA stream.  All arithmetic runs in the library's CUDA kernels.  There
is no fallback: if libtp.so is missing or fails to load, every call raises.

Function names are the C names.  Tensors are torch CUDA tensors; bf16 / f16 /
f32 map to TP_BF16 / TP_F16 / TP_F32.  4-bit codes are int32 tensors holding
the uint32 words (8 codes per word, element k at bits 4*(k % 8)); scales and
quantization biases are float16.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtp.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "tp_api.h")

TP_OK, TP_ERR_INVALID_ARG, TP_ERR_NOT_DIVISIBLE, TP_ERR_ALIGNMENT = 0, -1, -2, -3
TP_ERR_UNSUPPORTED, TP_ERR_CUDA, TP_ERR_TIMEOUT = -4, -5, -6
TP_F32, TP_BF16, TP_F16 = 0, 1, 2
TP_POLICY_AUTO, TP_POLICY_SIMT, TP_POLICY_SINGLE_SM = 0, 1, 2

_lib = None


class TPError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("tp error %d: %s" % (code, msg))
        self.code = code
        self.msg = msg


_rec = threading.local()  # set while prepare() marshals a call


class _Recording:
    """Stands in for the library while prepare() runs an entry point: the one
    call the entry point makes is recorded instead of executed."""

    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("tp_") or name in ("tp_last_error",):
            return getattr(self.real, name)
        fn = getattr(self.real, name)

        def record(*args):
            self.calls.append((fn, args))
            return TP_OK
        return record


def lib() -> ctypes.CDLL:
    """The loaded libtp.so (raises RuntimeError if it has not been built)."""
    r = getattr(_rec, "active", None)
    if r is not None:
        return r
    return _load()


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libtp.so is not built (%s); run `python -m sharded_gemm_gb300.build`"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        vpp = ctypes.POINTER(ctypes.c_void_p)
        sig = {
            "tp_version": ([], i32),
            "tp_last_error": ([], ctypes.c_char_p),
            "tp_launch_count": ([], i64),
            "tp_query_status": ([vp, ctypes.POINTER(ctypes.c_int)], i32),
            "tp_set_policy": ([i32], i32),
            "tp_set_wait_limit_ns": ([i64], i32),
            "tp_shutdown": ([], i32),
            "tp_shard_weight": ([vp, i64, i64, i32, i32, i32, i32, vpp, vp], i32),
            "tp_all_to_sharded": ([i32, vp, i64, i64, i64, vpp, i64, vpp, i32, vpp, i64, i32, vp], i32),
            "tp_sharded_to_all": ([i32, vpp, i64, i64, i64, vpp, i64, vp, i32, vp, i64, i32, vp], i32),
            "tp_gated_all_to_sharded": ([i32, vp, i64, i64, i64, vpp, vpp, i64, vpp, vpp, i32, vpp, i64, i32, vp],
                                        i32),
            "tp_sharded_to_sharded": ([i32, vpp, i64, i64, i64, vpp, i64, vp, i32, vpp, i64, i32, vp], i32),
            "tp_gathered_to_sharded": ([i32, vpp, i64, i64, i64, vpp, i64, vpp, i32, vpp, i64, i32, vp], i32),
            "tp_summa": ([i32, vpp, vpp, vpp, i64, i64, i64, i32, vp], i32),
            "tp_summa_linear": ([i32, vpp, vpp, vpp, vpp, i64, i64, i64, i32, vp], i32),
            "tp_summa_abt": ([i32, vpp, vpp, vpp, i64, i64, i64, i32, vp], i32),
            "tp_summa_atb": ([i32, vpp, vpp, vpp, i64, i64, i64, i32, vp], i32),
            "tp_all_to_sharded_dx": ([i32, vpp, i64, i64, i64, vpp, i64, i32, vp, i64, i32, vp], i32),
            "tp_sharded_to_all_dx": ([i32, vp, i64, i64, i64, vpp, i64, i32, vpp, i64, i32, vp], i32),
            "tp_sharded_dw": ([i32, vpp, i64, vpp, i64, i64, i64, i64, i32, vpp, i64, i32, vp], i32),
            "tp_bias_grad": ([i32, i32, vpp, i64, i64, i64, i32, vpp, vp], i32),
            "tp_mx_quantize": ([vp, i64, i64, vp, vp, vp], i32),
            "tp_mx_all_to_sharded": ([i32, vp, i64, i64, vpp, vpp, i64, vpp, vpp, i64, i32, vp], i32),
            "tp_mx_sharded_to_all": ([i32, vpp, i64, i64, vpp, vpp, i64, vp, vp, i64, i32, vp], i32),
            "tp_q4_quantize": ([vp, i64, i64, i32, vp, vp, vp, vp], i32),
            "tp_q4_all_to_sharded": ([i32, vp, i64, i64, vpp, vpp, vpp, i32, i64, vpp, vpp, i64, i32, vp], i32),
            "tp_q4_sharded_to_all": ([i32, vpp, i64, i64, vpp, vpp, vpp, i32, i64, vp, vp, i64, i32, vp], i32),
            "tp_debug_wait_timeout": ([i64, vp], i32),
            "tp_debug_prep_alone": ([i32], i32),
            "tp_set_trace": ([vp, i64], i32),
            "tp_q4_sharded_to_all_noalloc": ([i32, vpp, i64, i64, vpp, vpp, vpp, i32, i64, vp, vp, i64, i32, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


class Prepared:
    """One entry-point call, checked and marshalled once, replayed by
    ``__call__(stream)`` through the C ABI with the same arguments.

    It holds the device pointers of the tensors it was prepared with (and a
    reference to each, so they stay allocated); the caller must not resize or
    reallocate them.  Replaying costs one ctypes call, about what the C ABI
    itself costs, instead of the per-call argument checks and array building
    of the eager functions.  ``result`` is what the eager call returned (the
    output tensors)."""

    def __init__(self, fn, args, keep, result):
        self.fn = fn
        self.args = list(args)
        self.keep = keep
        self.result = result

    def __call__(self, stream=None):
        self.args[-1] = _stream(stream)
        _check(self.fn(*self.args))
        return self.result


def prepare(entry, *args, **kwargs) -> Prepared:
    """Prepares ``entry(*args, **kwargs)`` (one of this module's entry points
    that takes a ``stream`` argument) for replay; nothing is launched here."""
    if getattr(_rec, "active", None) is not None:
        raise RuntimeError("prepare() calls do not nest")
    rec = _Recording(_load())
    _rec.active = rec
    try:
        result = entry(*args, **kwargs)
    finally:
        _rec.active = None
    if len(rec.calls) != 1:
        raise ValueError("%s made %d library calls; prepare() takes entry points that make one"
                         % (getattr(entry, "__name__", entry), len(rec.calls)))
    fn, cargs = rec.calls[0]
    return Prepared(fn, cargs, (args, kwargs), result)


def declared_functions() -> list[str]:
    """Names of the functions include/tp_api.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", text)))


def _check(rc: int) -> None:
    if rc != TP_OK:
        raise TPError(rc, lib().tp_last_error().decode())


# ------------------------------------------------------------------ marshalling
def _torch():
    import torch
    return torch


def _dt(t) -> int:
    torch = _torch()
    m = {torch.float32: TP_F32, torch.bfloat16: TP_BF16, torch.float16: TP_F16}
    if t.dtype not in m:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return m[t.dtype]


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t


def _rowmajor(t, name):
    _cuda(t, name)
    if t.dim() != 2 or (t.numel() > 0 and t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("%s must be 2-D with unit column stride" % name)
    return t


def _contig(t, name):
    _cuda(t, name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _common_ld(ts, name):
    lds = {t.stride(0) if t.shape[0] > 1 else None for t in ts} - {None}
    if len(lds) > 1:
        raise ValueError("%s: all shards must share one row stride" % name)
    return lds.pop() if lds else ts[0].shape[1]


# ------------------------------------------------------------------ API
def tp_version() -> int:
    return lib().tp_version()


def tp_launch_count() -> int:
    """Kernels launched by the library from this thread so far (monotonic)."""
    return lib().tp_launch_count()


def tp_last_error() -> str:
    return lib().tp_last_error().decode()


def tp_set_policy(policy: int) -> None:
    _check(lib().tp_set_policy(policy))


def tp_set_wait_limit_ns(ns: int) -> None:
    _check(lib().tp_set_wait_limit_ns(ns))


def tp_shutdown() -> None:
    _check(lib().tp_shutdown())


def tp_set_trace(buf=None) -> None:
    """Start (buf: zeroed CUDA uint8/int64 tensor) or stop (None) role tracing."""
    if buf is None:
        _check(lib().tp_set_trace(None, 0))
    else:
        _check(lib().tp_set_trace(buf.data_ptr(), buf.numel() * buf.element_size()))


def decode_trace(buf) -> dict:
    """{event: {stage sequence: ns}} of a trace buffer (non-zero entries)."""
    import numpy as np
    w = buf.detach().cpu().numpy().view(np.uint64)
    out = {}
    for e in range(32):
        row = w[16 + e * 1024:16 + (e + 1) * 1024]
        nz = np.nonzero(row)[0]
        if len(nz):
            out[e] = {int(i): int(row[i]) for i in nz}
    return out


def tp_query_status(stream=None) -> int:
    v = ctypes.c_int(0)
    _check(lib().tp_query_status(_stream(stream), ctypes.byref(v)))
    return v.value


def tp_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().tp_debug_wait_timeout(limit_ns, _stream(stream)))


def tp_debug_prep_alone(on: bool) -> None:
    _check(lib().tp_debug_prep_alone(1 if on else 0))


def tp_shard_weight(w, axis: int, segments: int, N: int, shards=None, stream=None):
    """a1: the N rank slices of ``w`` along ``axis`` (bit-exact).

    ``w`` is 2-D (axis 0, 1 or -1) or 1-D (a bias; axis 0 or -1)."""
    torch = _torch()
    _contig(w, "w")
    if w.dim() == 1:
        if axis not in (0, -1):
            raise ValueError("a 1-D array can only be sharded along axis 0")
        w2, ax = w.reshape(-1, 1), 0
    elif w.dim() == 2:
        if axis not in (0, 1, -1):
            raise ValueError("axis must be 0, 1 or -1")
        w2, ax = w, (0 if axis == 0 else 1)
    else:
        raise ValueError("w must be 1-D or 2-D")
    rows, cols = w2.shape
    if shards is None:
        L = rows if ax == 0 else cols
        shp = (rows // N, cols) if ax == 0 else (rows, cols // N)
        if L % (segments * N) != 0:
            shp = (1, 1)  # the library reports the divisibility error
        shards = [torch.empty(shp, dtype=w.dtype, device=w.device) for _ in range(N)]
    for i, t in enumerate(shards):
        _contig(t, "shards[%d]" % i)
    pp, keep = _ptrs(shards)
    _check(lib().tp_shard_weight(w2.data_ptr(), rows, cols, w.element_size(), ax, segments, N, pp,
                                 _stream(stream)))
    return [t.reshape(-1) for t in shards] if w.dim() == 1 else shards


def tp_all_to_sharded(x, w, bias=None, out=None, out_dtype=None, stream=None):
    """a2/a4: y[r] = x @ w[r].T + bias[r] for every shard r; returns y list.

    ``out`` may be views of one gathered (T, O) buffer (column offset r*O/N)."""
    torch = _torch()
    _rowmajor(x, "x")
    N = len(w)
    T, K = x.shape
    On = w[0].shape[0]
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    if out is None:
        out = [torch.empty((T, On), dtype=out_dtype or x.dtype, device=x.device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    wp, k1 = _ptrs(w)
    yp, k2 = _ptrs(out)
    bp, k3 = (None, None)
    if bias is not None:
        for i, t in enumerate(bias):
            _contig(t, "bias[%d]" % i)
        bp, k3 = _ptrs(bias)
    ldx = x.stride(0) if T > 1 else K
    _check(lib().tp_all_to_sharded(N, x.data_ptr(), T, K, ldx, wp, On * N, bp, _dt(x), yp,
                                   _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_gated_all_to_sharded(x, w1, w3, b1=None, b3=None, out=None, out_dtype=None, stream=None):
    """f2: h[r] = silu(x @ w1[r].T + b1[r]) * (x @ w3[r].T + b3[r]); returns h list."""
    torch = _torch()
    _rowmajor(x, "x")
    N = len(w1)
    if len(w3) != N:
        raise ValueError("w1 and w3 need the same number of shards")
    T, K = x.shape
    Fn = w1[0].shape[0]
    for i, t in enumerate(list(w1) + list(w3)):
        _contig(t, "weight shard %d" % i)
    if out is None:
        out = [torch.empty((T, Fn), dtype=out_dtype or x.dtype, device=x.device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    keep = []

    def ptrs_or_none(ts, name):
        if ts is None:
            return None
        for i, t in enumerate(ts):
            _contig(t, "%s[%d]" % (name, i))
        p, k = _ptrs(ts)
        keep.append(k)
        return p
    w1p, w3p = ptrs_or_none(w1, "w1"), ptrs_or_none(w3, "w3")
    b1p, b3p = ptrs_or_none(b1, "b1"), ptrs_or_none(b3, "b3")
    yp, k_out = _ptrs(out)
    ldx = x.stride(0) if T > 1 else K
    _check(lib().tp_gated_all_to_sharded(N, x.data_ptr(), T, K, ldx, w1p, w3p, Fn * N, b1p, b3p, _dt(x),
                                         yp, _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_sharded_to_all(x, w, bias=None, out=None, out_dtype=None, stream=None):
    """a3: y = sum_r x[r] @ w[r].T (ascending r) + bias; returns y."""
    torch = _torch()
    N = len(x)
    for i, t in enumerate(x):
        _rowmajor(t, "x[%d]" % i)
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    T, Kn = x[0].shape
    O = w[0].shape[0]
    if out is None:
        out = torch.empty((T, O), dtype=out_dtype or torch.float32, device=x[0].device)
    _rowmajor(out, "out")
    if bias is not None:
        _contig(bias, "bias")
    xp, k1 = _ptrs(x)
    wp, k2 = _ptrs(w)
    ldx = _common_ld(x, "x")
    ldy = out.stride(0) if T > 1 else O
    _check(lib().tp_sharded_to_all(N, xp, T, Kn * N, ldx, wp, O,
                                   None if bias is None else bias.data_ptr(), _dt(x[0]),
                                   out.data_ptr(), ldy, _dt(out), _stream(stream)))
    return out


def tp_sharded_to_sharded(x, w, bias=None, out=None, out_dtype=None, stream=None):
    """f1: y[c] = (sum_r x[r] @ w[r][c*O/N:(c+1)*O/N].T, ascending r) + bias[c block].

    The reduce-scatter form of tp_sharded_to_all: rank c keeps only column
    block c of the sum.  ``out`` may be views of one (T, O) buffer (column
    offset c*O/N), which then holds the all-reduced output."""
    torch = _torch()
    N = len(x)
    for i, t in enumerate(x):
        _rowmajor(t, "x[%d]" % i)
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    T, Kn = x[0].shape
    O = w[0].shape[0]
    if out is None:
        out = [torch.empty((T, O // N), dtype=out_dtype or torch.float32, device=x[0].device)
               for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    if bias is not None:
        _contig(bias, "bias")
    xp, k1 = _ptrs(x)
    wp, k2 = _ptrs(w)
    yp, k3 = _ptrs(out)
    _check(lib().tp_sharded_to_sharded(N, xp, T, Kn * N, _common_ld(x, "x"), wp, O,
                                       None if bias is None else bias.data_ptr(), _dt(x[0]), yp,
                                       _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_gathered_to_sharded(x, w, bias=None, out=None, out_dtype=None, stream=None):
    """f1: y[r] = cat(x, dim=1) @ w[r].T + bias[r], without materialising the
    gathered input; x[q] is column block q of the input."""
    torch = _torch()
    N = len(x)
    for i, t in enumerate(x):
        _rowmajor(t, "x[%d]" % i)
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    T, Kn = x[0].shape
    On = w[0].shape[0]
    if out is None:
        out = [torch.empty((T, On), dtype=out_dtype or x[0].dtype, device=x[0].device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    bp, k4 = (None, None)
    if bias is not None:
        for i, t in enumerate(bias):
            _contig(t, "bias[%d]" % i)
        bp, k4 = _ptrs(bias)
    xp, k1 = _ptrs(x)
    wp, k2 = _ptrs(w)
    yp, k3 = _ptrs(out)
    _check(lib().tp_gathered_to_sharded(N, xp, T, Kn * N, _common_ld(x, "x"), wp, On * N, bp,
                                        _dt(x[0]), yp, _common_ld(out, "out"), _dt(out[0]),
                                        _stream(stream)))
    return out


def tp_summa(q: int, X, A, Y=None, stream=None):
    """a5: Y_ij = sum_t X_it A_tj on a q x q grid (blocks indexed i*q+j)."""
    torch = _torch()
    for i, t in enumerate(list(X) + list(A)):
        _contig(t, "block %d" % i)
    bm, bk = X[0].shape
    bn = A[0].shape[1]
    if Y is None:
        Y = [torch.empty((bm, bn), dtype=torch.float32, device=X[0].device) for _ in range(q * q)]
    for i, t in enumerate(Y):
        _contig(t, "Y[%d]" % i)
    xp, k1 = _ptrs(X)
    ap, k2 = _ptrs(A)
    yp, k3 = _ptrs(Y)
    _check(lib().tp_summa(q, xp, ap, yp, bm * q, bk * q, bn * q, _dt(X[0]), _stream(stream)))
    return Y


def tp_q4_quantize(w, group_size: int = 64, stream=None):
    """a6: (codes int32 (rows, K/8), scales f16, qbias f16) of a float32 weight."""
    torch = _torch()
    _contig(w, "w")
    rows, K = w.shape
    wq = torch.empty((rows, max(K // 8, 1)), dtype=torch.int32, device=w.device)
    sc = torch.empty((rows, max(K // group_size, 1)), dtype=torch.float16, device=w.device)
    qb = torch.empty_like(sc)
    _check(lib().tp_q4_quantize(w.data_ptr(), rows, K, group_size, wq.data_ptr(), sc.data_ptr(),
                                qb.data_ptr(), _stream(stream)))
    return wq, sc, qb


def tp_q4_all_to_sharded(x, wq, scales, qbias, bias=None, out=None, out_dtype=None,
                         group_size: int = 64, stream=None):
    """a7 column-parallel: y[r] = x @ What[r].T + bias[r]."""
    torch = _torch()
    _contig(x, "x")
    N = len(wq)
    T, K = x.shape
    On = wq[0].shape[0]
    for lst, nm in ((wq, "wq"), (scales, "scales"), (qbias, "qbias")):
        for i, t in enumerate(lst):
            _contig(t, "%s[%d]" % (nm, i))
    if out is None:
        out = [torch.empty((T, On), dtype=out_dtype or torch.bfloat16, device=x.device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    qp, k1 = _ptrs(wq)
    sp, k2 = _ptrs(scales)
    bq, k3 = _ptrs(qbias)
    yp, k4 = _ptrs(out)
    bp, k5 = (None, None)
    if bias is not None:
        bp, k5 = _ptrs(bias)
    _check(lib().tp_q4_all_to_sharded(N, x.data_ptr(), T, K, qp, sp, bq, group_size, On * N, bp, yp,
                                      _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_q4_sharded_to_all(x, wq, scales, qbias, bias=None, out=None, out_dtype=None,
                         group_size: int = 64, stream=None):
    """a7 row-parallel: y = sum_r x[r] @ What[r].T (ascending r) + bias."""
    torch = _torch()
    N = len(x)
    for lst, nm in ((x, "x"), (wq, "wq"), (scales, "scales"), (qbias, "qbias")):
        for i, t in enumerate(lst):
            _contig(t, "%s[%d]" % (nm, i))
    T, Kn = x[0].shape
    O = wq[0].shape[0]
    if out is None:
        out = torch.empty((T, O), dtype=out_dtype or torch.float32, device=x[0].device)
    _rowmajor(out, "out")
    xp, k1 = _ptrs(x)
    qp, k2 = _ptrs(wq)
    sp, k3 = _ptrs(scales)
    bq, k4 = _ptrs(qbias)
    ldy = out.stride(0) if T > 1 else O
    _check(lib().tp_q4_sharded_to_all(N, xp, T, Kn * N, qp, sp, bq, group_size, O,
                                      None if bias is None else bias.data_ptr(), out.data_ptr(), ldy,
                                      _dt(out), _stream(stream)))
    return out


def tp_q4_sharded_to_all_noalloc(x, wq, scales, qbias, bias=None, out=None, group_size: int = 64,
                                 stream=None):
    """a7 row-parallel without any device allocation inside the library call:
    the split workspace is a fixed array inside libtp.so.  ``out`` must be
    given (allocating it is the caller's business)."""
    if out is None:
        raise ValueError("out must be provided")
    N = len(x)
    for lst, nm in ((x, "x"), (wq, "wq"), (scales, "scales"), (qbias, "qbias")):
        for i, t in enumerate(lst):
            _contig(t, "%s[%d]" % (nm, i))
    T, Kn = x[0].shape
    O = wq[0].shape[0]
    _rowmajor(out, "out")
    xp, k1 = _ptrs(x)
    qp, k2 = _ptrs(wq)
    sp, k3 = _ptrs(scales)
    bq, k4 = _ptrs(qbias)
    ldy = out.stride(0) if T > 1 else O
    _check(lib().tp_q4_sharded_to_all_noalloc(N, xp, T, Kn * N, qp, sp, bq, group_size, O,
                                              None if bias is None else bias.data_ptr(),
                                              out.data_ptr(), ldy, _dt(out), _stream(stream)))
    return out


# ------------------------------------------------------------------ backward (f3)
def _summa_blocks(Xs, name):
    for i, t in enumerate(Xs):
        _contig(t, "%s[%d]" % (name, i))
    return _ptrs(Xs)


def tp_summa_linear(q: int, X, A, bias=None, Y=None, stream=None):
    """Y_ij = sum_t X_it A_tj + bias[j] on a q x q grid (blocks indexed i*q+j)."""
    torch = _torch()
    bm, bk = X[0].shape
    bn = A[0].shape[1]
    if Y is None:
        Y = [torch.empty((bm, bn), dtype=torch.float32, device=X[0].device) for _ in range(q * q)]
    xp, k1 = _summa_blocks(X, "X")
    ap, k2 = _summa_blocks(A, "A")
    yp, k3 = _summa_blocks(Y, "Y")
    bp, k4 = _summa_blocks(bias, "bias") if bias is not None else (None, None)
    _check(lib().tp_summa_linear(q, xp, ap, bp, yp, bm * q, bk * q, bn * q, _dt(X[0]), _stream(stream)))
    return Y


def tp_summa_abt(q: int, A, B, C=None, stream=None):
    """C_ij = sum_t A_it B_jt^T: A blocks (M/q, K/q), B blocks (N/q, K/q)."""
    torch = _torch()
    bm, bk = A[0].shape
    bn = B[0].shape[0]
    if C is None:
        C = [torch.empty((bm, bn), dtype=torch.float32, device=A[0].device) for _ in range(q * q)]
    ap, k1 = _summa_blocks(A, "A")
    bp, k2 = _summa_blocks(B, "B")
    cp, k3 = _summa_blocks(C, "C")
    _check(lib().tp_summa_abt(q, ap, bp, cp, bm * q, bk * q, bn * q, _dt(A[0]), _stream(stream)))
    return C


def tp_summa_atb(q: int, A, B, C=None, stream=None):
    """C_ij = sum_t A_ti^T B_tj: A blocks (K/q, M/q), B blocks (K/q, N/q)."""
    torch = _torch()
    bk, bm = A[0].shape
    bn = B[0].shape[1]
    if C is None:
        C = [torch.empty((bm, bn), dtype=torch.float32, device=A[0].device) for _ in range(q * q)]
    ap, k1 = _summa_blocks(A, "A")
    bp, k2 = _summa_blocks(B, "B")
    cp, k3 = _summa_blocks(C, "C")
    _check(lib().tp_summa_atb(q, ap, bp, cp, bm * q, bk * q, bn * q, _dt(A[0]), _stream(stream)))
    return C


def tp_all_to_sharded_dx(dy, w, out=None, out_dtype=None, stream=None):
    """Input gradient of the column-parallel layer: sum_r dy[r] @ w[r] (ascending r)."""
    torch = _torch()
    N = len(dy)
    for i, t in enumerate(dy):
        _rowmajor(t, "dy[%d]" % i)
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    T, On = dy[0].shape
    K = w[0].shape[1]
    if out is None:
        out = torch.empty((T, K), dtype=out_dtype or torch.float32, device=dy[0].device)
    _rowmajor(out, "out")
    dp, k1 = _ptrs(dy)
    wp, k2 = _ptrs(w)
    _check(lib().tp_all_to_sharded_dx(N, dp, T, On * N, _common_ld(dy, "dy"), wp, K, _dt(dy[0]),
                                      out.data_ptr(), out.stride(0) if T > 1 else K, _dt(out), _stream(stream)))
    return out


def tp_sharded_to_all_dx(dy, w, out=None, out_dtype=None, stream=None):
    """Input gradient of the row-parallel layer: dx[r] = dy @ w[r]."""
    torch = _torch()
    _rowmajor(dy, "dy")
    N = len(w)
    for i, t in enumerate(w):
        _contig(t, "w[%d]" % i)
    T, O = dy.shape
    Kn = w[0].shape[1]
    if out is None:
        out = [torch.empty((T, Kn), dtype=out_dtype or dy.dtype, device=dy.device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    wp, k1 = _ptrs(w)
    yp, k2 = _ptrs(out)
    _check(lib().tp_sharded_to_all_dx(N, dy.data_ptr(), T, O, dy.stride(0) if T > 1 else O, wp, Kn * N,
                                      _dt(dy), yp, _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_sharded_dw(dy, x, out=None, out_dtype=None, stream=None):
    """Weight gradients dw[r] = dy[r].T @ x[r] (lists of equal length N)."""
    torch = _torch()
    N = len(dy)
    if len(x) != N:
        raise ValueError("dy and x need the same number of shards")
    for i, t in enumerate(list(dy) + list(x)):
        _rowmajor(t, "operand %d" % i)
    T, O = dy[0].shape
    K = x[0].shape[1]
    if out is None:
        out = [torch.empty((O, K), dtype=out_dtype or torch.float32, device=dy[0].device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    dp, k1 = _ptrs(dy)
    xp, k2 = _ptrs(x)
    yp, k3 = _ptrs(out)
    _check(lib().tp_sharded_dw(N, dp, _common_ld(dy, "dy"), xp, _common_ld(x, "x"), T, O, K, _dt(dy[0]), yp,
                               _common_ld(out, "out"), _dt(out[0]), _stream(stream)))
    return out


def tp_bias_grad(dy, nin: int = 1, out=None, stream=None):
    """Float32 column sums: out[o] = sum over dy[o*nin .. o*nin+nin-1] of their row sums."""
    torch = _torch()
    n = len(dy)
    if n % nin:
        raise ValueError("len(dy) must be a multiple of nin")
    nout = n // nin
    for i, t in enumerate(dy):
        _rowmajor(t, "dy[%d]" % i)
    rows, cols = dy[0].shape
    if out is None:
        out = [torch.empty((cols,), dtype=torch.float32, device=dy[0].device) for _ in range(nout)]
    for i, t in enumerate(out):
        _contig(t, "out[%d]" % i)
    dp, k1 = _ptrs(dy)
    op, k2 = _ptrs(out)
    _check(lib().tp_bias_grad(nout, nin, dp, rows, cols, _common_ld(dy, "dy"), _dt(dy[0]), op, _stream(stream)))
    return out


# ------------------------------------------------------------------ mxfp8 (f4)
def tp_mx_quantize(w, stream=None):
    """MXFP8-quantize a float32 (rows, K) CUDA tensor: returns (codes uint8
    (rows, K), scales uint8 (rows, K/32))."""
    torch = _torch()
    _contig(w, "w")
    if w.dtype != torch.float32:
        raise TypeError("w must be float32")
    rows, K = w.shape
    codes = torch.empty((rows, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=w.device)
    _check(lib().tp_mx_quantize(w.data_ptr(), rows, K, codes.data_ptr(), scales.data_ptr(), _stream(stream)))
    return codes, scales


def tp_mx_all_to_sharded(x, codes, scales, bias=None, out=None, out_dtype=None, stream=None):
    """y[r] = x @ W_hat_r.T (+ bias[r]) with MXFP8 weight shards; returns y list."""
    torch = _torch()
    _contig(x, "x")
    N = len(codes)
    T, K = x.shape
    On = codes[0].shape[0]
    for i, t in enumerate(list(codes) + list(scales)):
        _contig(t, "weight %d" % i)
    if out is None:
        out = [torch.empty((T, On), dtype=out_dtype or x.dtype, device=x.device) for _ in range(N)]
    for i, t in enumerate(out):
        _rowmajor(t, "out[%d]" % i)
    cp, k1 = _ptrs(codes)
    sp, k2 = _ptrs(scales)
    yp, k3 = _ptrs(out)
    bp, k4 = (None, None)
    if bias is not None:
        for i, t in enumerate(bias):
            _contig(t, "bias[%d]" % i)
        bp, k4 = _ptrs(bias)
    _check(lib().tp_mx_all_to_sharded(N, x.data_ptr(), T, K, cp, sp, On * N, bp, yp, _common_ld(out, "out"),
                                      _dt(out[0]), _stream(stream)))
    return out


def tp_mx_sharded_to_all(x, codes, scales, bias=None, out=None, out_dtype=None, stream=None):
    """y = sum_r x[r] @ W_hat_r.T (ascending r) (+ bias) with MXFP8 weight shards."""
    torch = _torch()
    N = len(x)
    for i, t in enumerate(list(x) + list(codes) + list(scales)):
        _contig(t, "operand %d" % i)
    T, Kn = x[0].shape
    O = codes[0].shape[0]
    if out is None:
        out = torch.empty((T, O), dtype=out_dtype or torch.float32, device=x[0].device)
    _rowmajor(out, "out")
    if bias is not None:
        _contig(bias, "bias")
    xp, k1 = _ptrs(x)
    cp, k2 = _ptrs(codes)
    sp, k3 = _ptrs(scales)
    _check(lib().tp_mx_sharded_to_all(N, xp, T, Kn * N, cp, sp, O, None if bias is None else bias.data_ptr(),
                                      out.data_ptr(), out.stride(0) if T > 1 else O, _dt(out), _stream(stream)))
    return out

"""ctypes binding of libmxq.so, the sm_103a MX quantized-training library.

Argument marshalling only: every operation runs in the CUDA library.  torch
is used to allocate device memory and to name the current stream.  If the
library has not been built, every call raises -- there is no CPU fallback.

Low-level functions keep the C names (``mxq_quantize`` ...) and take raw
pointers; the tensor-level helpers follow the names of the method's
statement: ``mx_quantize``, ``hadamard_mx_quantize``, ``mx_quantize_dual``,
``mx_quantize_ablation``, ``mx_dequantize``, ``mx_gemm``, ``mx_gemm_quantize``.
"""

from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MXQ_BOUNDS_CHECKED=1 selects the bounds-checked build of the same library
# (every kernel checks the global indices it computes and reports
# MXQ_ERR_BOUNDS through mxq_check instead of accessing out of range)
BOUNDS_CHECKED = os.environ.get("MXQ_BOUNDS_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "_lib", "libmxq_debug.so" if BOUNDS_CHECKED else "libmxq.so")

E4M3, E2M1, E5M2 = 0, 1, 2
ROWWISE, COLWISE_T = 0, 1
SCALES_ROWMAJOR, SCALES_TC = 0, 1
SCALE_LAYOUTS = {"rowmajor": SCALES_ROWMAJOR, "tc": SCALES_TC,
                 SCALES_ROWMAJOR: SCALES_ROWMAJOR, SCALES_TC: SCALES_TC}
OUT_F32, OUT_BF16 = 0, 1
FMTS = {"e4m3": E4M3, "e2m1": E2M1, "e5m2": E5M2, E4M3: E4M3, E2M1: E2M1, E5M2: E5M2}
AXES = {"row": ROWWISE, "col": COLWISE_T, ROWWISE: ROWWISE, COLWISE_T: COLWISE_T}

STATUS = {0: "MXQ_OK", 1: "MXQ_ERR_ARG", 2: "MXQ_ERR_ALIGN", 3: "MXQ_ERR_UNSUPPORTED",
          4: "MXQ_ERR_CUDA", 5: "MXQ_ERR_TIMEOUT", 6: "MXQ_ERR_WORKSPACE",
          7: "MXQ_ERR_BOUNDS"}

# C signatures: (name, restype, argtypes)
_I64, _P, _I, _SZ, _U64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
SIGNATURES = [
    ("mxq_version", ctypes.c_int, []),
    ("mxq_status_str", ctypes.c_char_p, [_I]),
    ("mxq_quantize", _I, [_P, _I64, _I64, _I, _I, _P, _P, _P]),
    ("mxq_hadamard_quantize", _I, [_P, _I64, _I64, _I, _I, _P, _P, _P]),
    ("mxq_quantize_dual", _I, [_P, _I64, _I64, _I, _I, _P, _P, _I, _I, _P, _P, _P]),
    ("mxq_quantize_ex", _I, [_P, _I64, _I64, _I, _I, _I, _P, _P, _I, _P]),
    ("mxq_quantize_dual_ex", _I, [_P, _I64, _I64, _I, _I, _P, _P, _I, _I, _P, _P, _I, _P]),
    ("mxq_scales_tc_bytes", _SZ, [_I64, _I64]),
    ("mxq_gemm_ex", _I, [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _I, _P, _SZ, _P]),
    ("mxq_quantize_ablation", _I, [_P, _I64, _I64, _I, _I, _I, ctypes.c_uint32, _I, _U64, _P, _P, _P]),
    ("mxq_dequantize", _I, [_P, _P, _I64, _I64, _I, _I, _P, _I, _P]),
    ("mxq_gemm", _I, [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _P, _SZ, _P]),
    ("mxq_gemm_quantize", _I, [_P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P, _P, _SZ, _P]),
    ("mxq_gemm_quantize_ex", _I, [_P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _P, _P, _I, _P, _SZ,
                                  _P]),
    ("mxq_gemm_workspace_size", _SZ, [_I64, _I64, _I64, _I]),
    ("mxq_gemm_noalloc", _I, [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _P]),
    ("mxq_gemm_grouped", _I, [_P, _I, _I, _P]),
    ("mxq_check", _I, [_P]),
    ("mxq_set_wait_timeout_ns", None, [_U64]),
    ("mxq_debug_expire_wait", _I, [_U64, _P]),
]

class GemmProblem(ctypes.Structure):
    """mxq_gemm_problem of the C header (field order and types as declared)."""
    _fields_ = [("A", ctypes.c_void_p), ("sA", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("sB", ctypes.c_void_p), ("C", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("out_dtype", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


class MXQError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"libmxq.so is not built ({LIB_PATH} missing); run "
                        "precision_mx_quantize_gb300.build.build() first")
                handle = ctypes.CDLL(LIB_PATH)
                for name, res, args in SIGNATURES:
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device=None) -> int:
    """The raw handle of the current CUDA stream of `device` (default: the
    current device).  Uses torch's raw-handle accessor when it has one, which
    skips building a Stream object on every call."""
    if _raw_stream is not None:
        if device is None:
            idx = torch.cuda.current_device()
        elif isinstance(device, int):
            idx = device
        else:
            idx = device.index if device.index is not None else torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _ok(status: int, where: str):
    if status != 0:
        raise MXQError(status, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


# ---- raw C-ABI calls (pointers and sizes) ------------------------------------

def mxq_quantize(x, rows, cols, layout, fmt, codes, scales, stream):
    return lib().mxq_quantize(x, rows, cols, layout, fmt, codes, scales, stream)


def mxq_hadamard_quantize(x, rows, cols, layout, fmt, codes, scales, stream):
    return lib().mxq_hadamard_quantize(x, rows, cols, layout, fmt, codes, scales, stream)


def mxq_quantize_dual(x, rows, cols, fmt_r, had_r, codes_r, scales_r, fmt_c, had_c, codes_c,
                      scales_c, stream):
    return lib().mxq_quantize_dual(x, rows, cols, fmt_r, had_r, codes_r, scales_r, fmt_c, had_c,
                                   codes_c, scales_c, stream)


def mxq_quantize_ex(x, rows, cols, layout, fmt, hadamard, codes, scales, scale_layout, stream):
    return lib().mxq_quantize_ex(x, rows, cols, layout, fmt, hadamard, codes, scales, scale_layout,
                                 stream)


def mxq_quantize_dual_ex(x, rows, cols, fmt_r, had_r, codes_r, scales_r, fmt_c, had_c, codes_c,
                         scales_c, scale_layout, stream):
    return lib().mxq_quantize_dual_ex(x, rows, cols, fmt_r, had_r, codes_r, scales_r, fmt_c,
                                      had_c, codes_c, scales_c, scale_layout, stream)


def mxq_scales_tc_bytes(lines, blocked):
    return lib().mxq_scales_tc_bytes(lines, blocked)


def mxq_gemm_ex(A, sA, B, sB, fmt, M, N, K, C, out_dtype, scale_layout, workspace, ws_bytes,
                stream):
    return lib().mxq_gemm_ex(A, sA, B, sB, fmt, M, N, K, C, out_dtype, scale_layout, workspace,
                             ws_bytes, stream)


def mxq_quantize_ablation(x, rows, cols, layout, fmt, hadamard, sign_mask, stochastic, seed, codes,
                          scales, stream):
    return lib().mxq_quantize_ablation(x, rows, cols, layout, fmt, hadamard, sign_mask, stochastic,
                                       seed, codes, scales, stream)


def mxq_dequantize(codes, scales, rows, cols, layout, fmt, out, out_dtype, stream):
    return lib().mxq_dequantize(codes, scales, rows, cols, layout, fmt, out, out_dtype, stream)


def mxq_gemm(A, sA, B, sB, fmt, M, N, K, C, out_dtype, workspace, ws_bytes, stream):
    return lib().mxq_gemm(A, sA, B, sB, fmt, M, N, K, C, out_dtype, workspace, ws_bytes, stream)


def mxq_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt, codes, scales, workspace, ws_bytes,
                      stream):
    return lib().mxq_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt, codes, scales, workspace,
                                   ws_bytes, stream)


def mxq_gemm_quantize_ex(A, sA, B, sB, fmt, M, N, K, scale_layout, out_fmt, codes, scales,
                         out_scale_layout, workspace, ws_bytes, stream):
    return lib().mxq_gemm_quantize_ex(A, sA, B, sB, fmt, M, N, K, scale_layout, out_fmt, codes,
                                      scales, out_scale_layout, workspace, ws_bytes, stream)


def mxq_gemm_noalloc(A, sA, B, sB, fmt, M, N, K, C, out_dtype, stream):
    """mxq_gemm with the library's fixed internal scratch (for callers that cannot allocate)."""
    return lib().mxq_gemm_noalloc(A, sA, B, sB, fmt, M, N, K, C, out_dtype, stream)


def mxq_gemm_grouped(problems, count, fmt, stream):
    """problems: address of `count` GemmProblem structures in host memory."""
    return lib().mxq_gemm_grouped(problems, count, fmt, stream)


def mxq_gemm_workspace_size(M, N, K, fmt):
    return lib().mxq_gemm_workspace_size(M, N, K, fmt)


def mxq_check(stream=None):
    return lib().mxq_check(stream)


def check(device=None):
    """Synchronize the current stream and raise on any recorded device error."""
    _ok(mxq_check(_stream(device)), "mxq_check")


def set_wait_timeout_ns(ns: int):
    lib().mxq_set_wait_timeout_ns(int(ns))


# ---- tensor-level helpers -----------------------------------------------------

def code_shape(rows: int, cols: int, axis, fmt):
    """(codes shape, scales shape) for a [rows, cols] tensor."""
    ax, f = AXES[axis], FMTS[fmt]
    r, c = (rows, cols) if ax == ROWWISE else (cols, rows)
    return (r, c // 2 if f == E2M1 else c), (r, c // 32)


# The kernels get raw pointers and sizes: a host tensor, or a buffer shorter
# than the sizes imply, would be read or written past its end on the GPU.
# These checks run before every launch (explicit raises, not asserts, so
# that they survive python -O).

def _on_gpu(t):
    return t.is_cuda


def _need(t, name, dtype, numel, dev=None):
    """Raise unless t is a contiguous CUDA tensor of `dtype` (None: any) with
    at least `numel` elements, on device index `dev` when given.  Cheap on
    the success path (the binding runs it on every call): one combined test,
    and the detailed checks only to word the error."""
    try:
        if ((dtype is None or t.dtype is dtype) and t.numel() >= numel and t.is_contiguous()
                and _on_gpu(t) and (dev is None or t.get_device() == dev)):
            return
    except AttributeError:
        pass
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype is not dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; {numel} are needed")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not _on_gpu(t):
        raise ValueError(f"{name} must be on a CUDA device (the library has no CPU path)")
    if dev is not None and t.get_device() != dev:
        raise ValueError(f"{name} is on device {t.get_device()}, the inputs on {dev}")


def _need_input(x):
    """x: a contiguous 2-D bf16 CUDA tensor."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a 2-D torch.Tensor [rows, cols]")
    _need(x, "x", torch.bfloat16, 0)


@functools.lru_cache(maxsize=4096)
def _buffer_sizes(rows, cols, axis, fmt, scale_layout):
    """(code bytes, scale bytes) of a [rows, cols] tensor quantized along
    `axis`, with its scales in `scale_layout`."""
    cs, _ = code_shape(rows, cols, axis, fmt)
    lines, blocked = (rows, cols) if AXES[axis] == ROWWISE else (cols, rows)
    if SCALE_LAYOUTS[scale_layout] == SCALES_TC:
        n = int(mxq_scales_tc_bytes(lines, blocked))
        if n == 0:
            raise ValueError(f"no tensor-core scale layout for {lines} lines x {blocked}")
    else:
        n = lines * (blocked // 32)
    return cs[0] * cs[1], n


def _need_codes(codes, scales, rows, cols, axis, fmt, scale_layout, dev, tag=""):
    """The code and scale buffers of a [rows, cols] tensor quantized along `axis`."""
    nc, ns = _buffer_sizes(int(rows), int(cols), axis, fmt, scale_layout)
    _need(codes, "codes" + tag, torch.uint8, nc, dev)
    _need(scales, "scales" + tag, torch.uint8, ns, dev)


def _out_code(out_dtype):
    if out_dtype is torch.float32:
        return OUT_F32
    if out_dtype is torch.bfloat16:
        return OUT_BF16
    raise ValueError(f"out_dtype must be torch.float32 or torch.bfloat16, got {out_dtype}")


def _need_operands(A, sA, B, sB, fmt, M, N, K, scale_layout):
    """GEMM operands: K-major codes of A [M, K] and B [N, K] and their scales.
    Returns the device index of A."""
    _need(A, "A", torch.uint8, 0)
    dev = A.get_device()
    _need_codes(A, sA, M, K, "row", fmt, scale_layout, dev, "_A")
    _need_codes(B, sB, N, K, "row", fmt, scale_layout, dev, "_B")
    return dev


def _alloc_codes(x, axis, fmt, scale_layout="rowmajor"):
    cs, ss = code_shape(x.shape[0], x.shape[1], axis, fmt)
    if SCALE_LAYOUTS[scale_layout] == SCALES_TC:
        lines, blocked = (x.shape[0], x.shape[1]) if AXES[axis] == ROWWISE else (x.shape[1], x.shape[0])
        n = mxq_scales_tc_bytes(lines, blocked)
        if n == 0:
            raise ValueError(f"no tensor-core scale layout for {lines} lines x {blocked}")
        ss = (n,)
    return (torch.empty(cs, dtype=torch.uint8, device=x.device),
            torch.empty(ss, dtype=torch.uint8, device=x.device))


def mx_quantize(x: torch.Tensor, axis="row", fmt="e4m3", out=None, scale_layout="rowmajor"):
    """MX-quantize a contiguous bf16 CUDA tensor [rows, cols]; returns (codes, scales).

    scale_layout "tc": scales in the tensor cores' chunk layout (a flat byte
    tensor), which mx_gemm(..., scale_layout="tc") reads in place."""
    _need_input(x)
    codes, scales = out if out is not None else _alloc_codes(x, axis, fmt, scale_layout)
    R, C = x.shape
    dev = x.get_device()
    _need_codes(codes, scales, R, C, axis, fmt, scale_layout, dev)
    if SCALE_LAYOUTS[scale_layout] == SCALES_ROWMAJOR:
        _ok(mxq_quantize(x.data_ptr(), R, C, AXES[axis], FMTS[fmt], codes.data_ptr(),
                         scales.data_ptr(), _stream(dev)), "mxq_quantize")
    else:
        _ok(mxq_quantize_ex(x.data_ptr(), R, C, AXES[axis], FMTS[fmt], 0, codes.data_ptr(),
                            scales.data_ptr(), SCALES_TC, _stream(dev)), "mxq_quantize_ex")
    return codes, scales


def hadamard_mx_quantize(x: torch.Tensor, axis="col", fmt="e2m1", out=None,
                         scale_layout="rowmajor"):
    """Fixed 32-point Hadamard rotation of each block, then MX quantization."""
    _need_input(x)
    codes, scales = out if out is not None else _alloc_codes(x, axis, fmt, scale_layout)
    R, C = x.shape
    dev = x.get_device()
    _need_codes(codes, scales, R, C, axis, fmt, scale_layout, dev)
    if SCALE_LAYOUTS[scale_layout] == SCALES_ROWMAJOR:
        _ok(mxq_hadamard_quantize(x.data_ptr(), R, C, AXES[axis], FMTS[fmt], codes.data_ptr(),
                                  scales.data_ptr(), _stream(dev)), "mxq_hadamard_quantize")
    else:
        _ok(mxq_quantize_ex(x.data_ptr(), R, C, AXES[axis], FMTS[fmt], 1, codes.data_ptr(),
                            scales.data_ptr(), SCALES_TC, _stream(dev)), "mxq_quantize_ex")
    return codes, scales


def mx_quantize_dual(x: torch.Tensor, fmt_r="e4m3", had_r=False, fmt_c="e2m1", had_c=True,
                     out=None, scale_layout="rowmajor"):
    """One pass producing the row-wise and the column-wise (transposed) outputs."""
    _need_input(x)
    if out is None:
        cr, sr = _alloc_codes(x, "row", fmt_r, scale_layout)
        cc, sc = _alloc_codes(x, "col", fmt_c, scale_layout)
    else:
        cr, sr, cc, sc = out
    _need_codes(cr, sr, x.shape[0], x.shape[1], "row", fmt_r, scale_layout, x.get_device(), "_r")
    _need_codes(cc, sc, x.shape[0], x.shape[1], "col", fmt_c, scale_layout, x.get_device(), "_c")
    if SCALE_LAYOUTS[scale_layout] == SCALES_ROWMAJOR:
        _ok(mxq_quantize_dual(x.data_ptr(), x.shape[0], x.shape[1], FMTS[fmt_r], int(had_r),
                              cr.data_ptr(), sr.data_ptr(), FMTS[fmt_c], int(had_c), cc.data_ptr(),
                              sc.data_ptr(), _stream(x.device)), "mxq_quantize_dual")
    else:
        _ok(mxq_quantize_dual_ex(x.data_ptr(), x.shape[0], x.shape[1], FMTS[fmt_r], int(had_r),
                                 cr.data_ptr(), sr.data_ptr(), FMTS[fmt_c], int(had_c),
                                 cc.data_ptr(), sc.data_ptr(), SCALES_TC, _stream(x.device)),
            "mxq_quantize_dual_ex")
    return cr, sr, cc, sc


def mx_quantize_ablation(x: torch.Tensor, axis="col", fmt="e2m1", hadamard=True, sign_mask=0,
                         stochastic=False, seed=0, out=None):
    """MX quantization with a random-sign Hadamard rotation (sign_mask) and/or
    stochastic rounding (Philox bits keyed by seed); the ablation of the
    deterministic path."""
    _need_input(x)
    codes, scales = out if out is not None else _alloc_codes(x, axis, fmt)
    _need_codes(codes, scales, x.shape[0], x.shape[1], axis, fmt, "rowmajor", x.get_device())
    _ok(mxq_quantize_ablation(x.data_ptr(), x.shape[0], x.shape[1], AXES[axis], FMTS[fmt],
                              int(hadamard), int(sign_mask) & 0xFFFFFFFF, int(stochastic),
                              int(seed) & 0xFFFFFFFFFFFFFFFF, codes.data_ptr(), scales.data_ptr(),
                              _stream(x.device)), "mxq_quantize_ablation")
    return codes, scales


def mx_dequantize(codes, scales, rows, cols, axis="row", fmt="e4m3", out_dtype=torch.float32,
                  out=None):
    """Dequantize codes written by mx_quantize back to a [rows, cols] tensor."""
    od = _out_code(out_dtype)
    _need(codes, "codes", torch.uint8, 0)
    dev = codes.get_device()
    _need_codes(codes, scales, rows, cols, axis, fmt, "rowmajor", dev)
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype, device=codes.device)
    _need(out, "out", out_dtype, rows * cols, dev)
    _ok(mxq_dequantize(codes.data_ptr(), scales.data_ptr(), rows, cols, AXES[axis], FMTS[fmt],
                       out.data_ptr(), od, _stream(dev)), "mxq_dequantize")
    return out


def gemm_workspace(M, N, K, fmt, device):
    n = mxq_gemm_workspace_size(M, N, K, FMTS[fmt])
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


def mx_gemm(A, sA, B, sB, fmt, M, N, K, out_dtype=torch.float32, out=None, workspace=None,
            scale_layout="rowmajor"):
    """C[M, N] = dec(A) @ dec(B)^T on the tensor cores (A, B K-major MX codes).

    scale_layout "tc": sA, sB in the tensor cores' chunk layout (no workspace)."""
    od = _out_code(out_dtype)
    dev = _need_operands(A, sA, B, sB, fmt, M, N, K, scale_layout)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    _need(out, "out", out_dtype, M * N, dev)
    if SCALE_LAYOUTS[scale_layout] == SCALES_TC:
        _ok(mxq_gemm_ex(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), FMTS[fmt], M, N,
                        K, out.data_ptr(), od, SCALES_TC, None, 0, _stream(A.device)),
            "mxq_gemm_ex")
        return out
    if workspace is None:
        workspace = gemm_workspace(M, N, K, fmt, A.device)
    _need(workspace, "workspace", torch.uint8, 0, dev)   # its size is checked by the library
    _ok(mxq_gemm(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), FMTS[fmt], M, N, K,
                 out.data_ptr(), od, workspace.data_ptr(), workspace.numel(),
                 _stream(A.device)), "mxq_gemm")
    return out


def mx_gemm_grouped(problems, fmt, out_dtype=torch.float32):
    """Independent GEMMs of one format in one launch (see mxq_gemm_grouped).

    problems: list of (A, sA, B, sB, M, N, K) or (A, sA, B, sB, M, N, K, out),
    with the scales in the tensor cores' chunk layout (as returned by the
    quantizers with scale_layout="tc").  Returns the list of outputs C, each
    bitwise what mx_gemm(..., scale_layout="tc") would return."""
    if not 1 <= len(problems) <= 8:
        raise ValueError("mx_gemm_grouped takes 1 to 8 problems")
    od = _out_code(out_dtype)
    arr = (GemmProblem * len(problems))()
    outs = []
    dev = None
    for i, pr in enumerate(problems):
        A, sA, B, sB, M, N, K = pr[:7]
        d = _need_operands(A, sA, B, sB, fmt, M, N, K, "tc")
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError(f"problem {i} is on device {d}, problem 0 on {dev}")
        out = pr[7] if len(pr) > 7 else torch.empty((M, N), dtype=out_dtype, device=A.device)
        _need(out, f"out[{i}]", out_dtype, M * N, dev)
        arr[i] = GemmProblem(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(),
                             out.data_ptr(), M, N, K, od)
        outs.append(out)
    _ok(mxq_gemm_grouped(ctypes.addressof(arr), len(problems), FMTS[fmt], _stream(dev)),
        "mxq_gemm_grouped")
    return outs


def mx_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt="e4m3", out=None, workspace=None,
                     scale_layout="rowmajor", out_scale_layout="rowmajor"):
    """dec(A) @ dec(B)^T with the epilogue writing row-wise MX codes of the
    fp32 product (blocks of 32 along N); returns (codes, scales)."""
    in_tc = SCALE_LAYOUTS[scale_layout] == SCALES_TC
    out_tc = SCALE_LAYOUTS[out_scale_layout] == SCALES_TC
    dev = _need_operands(A, sA, B, sB, fmt, M, N, K, scale_layout)
    if out is None:
        cs, ss = code_shape(M, N, "row", out_fmt)
        if out_tc:
            ss = (mxq_scales_tc_bytes(M, N),)
        out = (torch.empty(cs, dtype=torch.uint8, device=A.device),
               torch.empty(ss, dtype=torch.uint8, device=A.device))
    codes, scales = out
    _need_codes(codes, scales, M, N, "row", out_fmt, out_scale_layout, dev, "_out")
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 0, dev)
    if not in_tc and not out_tc:
        if workspace is None:
            workspace = gemm_workspace(M, N, K, fmt, A.device)
        _ok(mxq_gemm_quantize(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), FMTS[fmt], M,
                              N, K, FMTS[out_fmt], codes.data_ptr(), scales.data_ptr(),
                              workspace.data_ptr(), workspace.numel(), _stream(A.device)),
            "mxq_gemm_quantize")
        return codes, scales
    if not in_tc and workspace is None:
        workspace = gemm_workspace(M, N, K, fmt, A.device)
    ws_ptr, ws_n = (None, 0) if in_tc else (workspace.data_ptr(), workspace.numel())
    _ok(mxq_gemm_quantize_ex(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), FMTS[fmt], M,
                             N, K, SCALE_LAYOUTS[scale_layout], FMTS[out_fmt], codes.data_ptr(),
                             scales.data_ptr(), SCALE_LAYOUTS[out_scale_layout], ws_ptr, ws_n,
                             _stream(A.device)), "mxq_gemm_quantize_ex")
    return codes, scales

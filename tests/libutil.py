"""Shared test helpers: locate/build the CUDA library, move data for the oracle."""

import os

import numpy as np
import torch

from precision_mx_quantize_gb300 import build as _build
from precision_mx_quantize_gb300 import mxq


def _stale() -> bool:
    libs = (mxq.LIB_PATH, _build.LIB, _build.LIB_DEBUG)
    if not all(os.path.exists(p) for p in libs):
        return True
    built = min(os.path.getmtime(p) for p in libs)
    srcs = _build.sources() + [os.path.join(_build.CSRC, f) for f in os.listdir(_build.CSRC)
                               if f.endswith((".cuh", ".h"))]
    srcs += [os.path.join(_build.INCLUDE, f) for f in os.listdir(_build.INCLUDE)]
    return any(os.path.getmtime(f) > built for f in srcs)


def ensure_built():
    """Build the library if it is missing or older than any of its sources."""
    if _stale():
        _build.build()
    return mxq.lib()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_to_f32_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy()


def header_symbols():
    import re
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = set()
    inc = os.path.join(here, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"\b(mxq_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def header_prototypes():
    """{function name: [parameter declarations]} of the functions the headers
    declare (comments stripped; a prototype is a name, a parenthesised
    parameter list and a semicolon)."""
    import re
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    inc = os.path.join(here, "include")
    out = {}
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(inc, f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        for m in re.finditer(r"\b(mxq_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
            params = m.group(2).strip()
            out[m.group(1)] = [] if params in ("", "void") else [
                " ".join(q.split()) for q in params.split(",")]
    return out

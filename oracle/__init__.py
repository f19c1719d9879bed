"""fp64 CPU oracle of one MoE-layer forward (route, dispatch, SwiGLU FFN, combine).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the bench's
CPU-baseline leg are the only callers. The product path never imports this
package; the C library below shares no code with the CUDA kernels.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64); this module only
compiles it with gcc, loads it with ctypes and marshals numpy arrays.
Sources followed: Cui et al., "Fine-grained Computation-Communication Overlap
via Tile-level Signaling and Scheduling for MoE", section 2.1 (the five steps
of the MoE forward); Xian et al., "X-Stage ...", section 2.2 (the two-layer
SwiGLU expert FFN and the router-weighted combine).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc_moe.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no CUDA involved)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i, l = ctypes.c_int, ctypes.c_long
    lib.orc_route.argtypes = [i, i, i, i, P, P, P, P, P, P, P, P, i]
    lib.orc_dispatch.argtypes = [i, i, i, P, P, P, P, P]
    lib.orc_ffn_rows.argtypes = [i, i, i, l, P, P, P, P, P, P, P, i, i]
    lib.orc_combine.argtypes = [i, i, i, P, P, P, P]
    lib.orc_layer_tokens.argtypes = [i, i, i, i, i, P, P, P, P, P, P, l, P, P, i, i]
    for f in (lib.orc_route, lib.orc_dispatch, lib.orc_ffn_rows, lib.orc_combine,
              lib.orc_layer_tokens):
        f.restype = ctypes.c_int
    return lib


_override = None


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _bind(build())
    return _lib


class use_library:
    """Context manager: route every oracle call to another build of moe_oracle.c
    (the tests use it to check that a planted mistake is caught by the pins)."""

    def __init__(self, path: str):
        self.lib = _bind(path)

    def __enter__(self):
        global _override
        self._prev = _override
        _override = self.lib
        return self

    def __exit__(self, *exc):
        global _override
        _override = self._prev
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (test use only)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    src, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else os.cpu_count() or 1)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (code {rc})")


@dataclass
class Route:
    idx: np.ndarray        # [T, k] int32, selected experts in descending-logit order
    gate: np.ndarray       # [T, k] float64, softmax over the selected logits
    z32: np.ndarray | None  # [T, E] float32 logits (selection precision)
    z64: np.ndarray | None  # [T, E] float64 logits
    fp_sensitive: np.ndarray  # [T] bool: fp64 logits would select differently


def route(x_bits, wr_bits, bias, k: int, keep_logits: bool = False, nthreads: int | None = None) -> Route:
    """Router: logits, top-k (descending, ties to lower index), softmax over the selection."""
    x = _u16(x_bits)
    wr = _u16(wr_bits)
    T, d = x.shape
    E = wr.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    z32 = np.empty((T, E), np.float32) if keep_logits else None
    z64 = np.empty((T, E), np.float64) if keep_logits else None
    sens = np.zeros(T, np.uint8)
    rc = _load().orc_route(T, d, E, k, _p(x), _p(wr), _p(b), _p(idx), _p(gate), _p(z32), _p(z64),
                           _p(sens), nthreads or default_threads())
    _check(rc, "route")
    return Route(idx, gate, z32, z64, sens.astype(bool))


@dataclass
class Dispatch:
    counts: np.ndarray       # [E] int32
    offsets: np.ndarray      # [E+1] int32
    row_of_slot: np.ndarray  # [T*k] int32
    slot_of_row: np.ndarray  # [T*k] int32


def dispatch(topk_idx, E: int) -> Dispatch:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    ros = np.empty(T * k, np.int32)
    sor = np.empty(T * k, np.int32)
    _check(_load().orc_dispatch(T, k, E, _p(idx), _p(counts), _p(offsets), _p(ros), _p(sor)),
           "dispatch")
    return Dispatch(counts, offsets, ros, sor)


def ffn_rows(xin_bits, expert_of_row, w1_bits, w3_bits, w2_bits, E: int, keep_h: bool = False,
             identity: bool = False, nthreads: int | None = None):
    """Per-row expert FFN: returns (h [n,F] fp64 or None, y [n,d] fp64)."""
    xin = _u16(xin_bits)
    n, d = xin.shape
    er = np.ascontiguousarray(expert_of_row, dtype=np.int32)
    if identity:
        F = 1
        w1 = w3 = w2 = None
    else:
        w1, w3, w2 = _u16(w1_bits), _u16(w3_bits), _u16(w2_bits)
        F = w1.shape[1]
    h = np.empty((n, F), np.float64) if (keep_h and not identity) else None
    y = np.empty((n, d), np.float64)
    rc = _load().orc_ffn_rows(d, F, E, n, _p(er), _p(xin), _p(w1), _p(w3), _p(w2), _p(h), _p(y),
                              1 if identity else 0, nthreads or default_threads())
    _check(rc, "ffn_rows")
    return h, y


def combine(y_rows, gate, row_of_slot) -> np.ndarray:
    y = np.ascontiguousarray(y_rows, dtype=np.float64)
    g = np.ascontiguousarray(gate, dtype=np.float64)
    T, k = g.shape
    d = y.shape[1]
    ros = np.ascontiguousarray(row_of_slot, dtype=np.int32)
    out = np.empty((T, d), np.float64)
    _check(_load().orc_combine(T, k, d, _p(y), _p(g), _p(ros), _p(out)), "combine")
    return out


def layer_tokens(x_bits, topk_idx, gate, w1_bits, w3_bits, w2_bits, tokens, E: int,
                 identity: bool = False, nthreads: int | None = None) -> np.ndarray:
    """out[t] = sum_j gate[t,j] * FFN_{idx[t,j]}(x[t]) for the listed tokens (fp64)."""
    x = _u16(x_bits)
    T, d = x.shape
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    g = np.ascontiguousarray(gate, dtype=np.float64)
    k = idx.shape[1]
    toks = np.ascontiguousarray(tokens, dtype=np.int32)
    if identity:
        F, w1, w3, w2 = 1, None, None, None
    else:
        w1, w3, w2 = _u16(w1_bits), _u16(w3_bits), _u16(w2_bits)
        F = w1.shape[1]
    out = np.empty((len(toks), d), np.float64)
    rc = _load().orc_layer_tokens(T, d, E, k, F, _p(x), _p(idx), _p(g), _p(w1), _p(w3), _p(w2),
                                  len(toks), _p(toks), _p(out), 1 if identity else 0,
                                  nthreads or default_threads())
    _check(rc, "layer_tokens")
    return out


def layer(x_bits, wr_bits, bias, k, w1_bits, w3_bits, w2_bits, nthreads: int | None = None):
    """The whole layer for every token: returns (Route, Dispatch, out [T,d] fp64)."""
    r = route(x_bits, wr_bits, bias, k, nthreads=nthreads)
    E = wr_bits.shape[0]
    disp = dispatch(r.idx, E)
    T = x_bits.shape[0]
    out = layer_tokens(x_bits, r.idx, r.gate, w1_bits, w3_bits, w2_bits,
                       np.arange(T, dtype=np.int32), E, nthreads=nthreads)
    return r, disp, out

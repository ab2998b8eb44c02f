"""Plain FP64 CPU oracle of Fused-Softmax quantized attention.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it;
the library under ``matrix_core_softmax_gb300`` never does and shares no code
with it.  The arithmetic lives in ``fsa_oracle.c`` (plain C, double precision,
one thread per slice of rows); this module only compiles it with gcc and
marshals numpy arrays.

Every function cites the passage it follows in ``fsa_oracle.c``.  Pins that
tie it to the pages and to mathematics live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

# Element formats (indices used by the C code)
E4M3, E2M3, E2M1 = 0, 1, 2
# Attention formats: element format of Q/K/V and of P
FORMATS = {
    "mxfp8": (E4M3, E4M3),
    "mxfp6": (E2M3, E2M3),
    "mxfp4": (E2M1, E2M3),  # the MXFP4 variant keeps six-bit P
}


def build(force: bool = False) -> str:
    """Compile fsa_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("qkv_fmt", ctypes.c_int),
        ("p_fmt", ctypes.c_int),
        ("exp_mode", ctypes.c_int),
        ("max_mode", ctypes.c_int),
        ("l_from_unquantized", ctypes.c_int),
        ("tile", ctypes.c_int),
        ("threshold", ctypes.c_double),
        ("sm_scale", ctypes.c_double),
        ("gate_mode", ctypes.c_int),
        ("efq_tau", ctypes.c_double),
        ("efq_h", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.ora_decode_elem.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.ora_decode_elem.restype = ctypes.c_double
            lib.ora_encode_elem.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.ora_encode_elem.restype = ctypes.c_int
            lib.ora_mx_scale_exp.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.ora_mx_scale_exp.restype = ctypes.c_int
            lib.ora_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.ora_bf16_to_double.restype = ctypes.c_double
            lib.ora_double_to_bf16.argtypes = [ctypes.c_double]
            lib.ora_double_to_bf16.restype = ctypes.c_uint16
            lib.ora_schraudolph_y.argtypes = [ctypes.c_double]
            lib.ora_schraudolph_y.restype = ctypes.c_double
            lib.ora_schraudolph_code.argtypes = [ctypes.c_double]
            lib.ora_schraudolph_code.restype = ctypes.c_int
            lib.ora_mx_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, P, P]
            lib.ora_mx_quantize.restype = ctypes.c_int
            lib.ora_attention.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.POINTER(_Params), P, ctypes.c_int64, ctypes.c_int,
                                          P, P, P, P, P, P, ctypes.POINTER(ctypes.c_int64)]
            lib.ora_attention.restype = ctypes.c_int
            lib.ora_attention_qk.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int, ctypes.POINTER(_Params), P, ctypes.c_int64,
                                             ctypes.c_int, P, P, P, P, P, P,
                                             ctypes.POINTER(ctypes.c_int64)]
            lib.ora_attention_qk.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- codecs --
def decode_elem(fmt: int, code: int) -> float:
    return _load().ora_decode_elem(fmt, int(code))


def encode_elem(fmt: int, v: float) -> int:
    return _load().ora_encode_elem(fmt, float(v))


def mx_scale_exp(fmt: int, amax: float) -> int:
    return _load().ora_mx_scale_exp(fmt, float(amax))


def bf16_to_double(b: int) -> float:
    return _load().ora_bf16_to_double(int(b))


def double_to_bf16(v: float) -> int:
    return _load().ora_double_to_bf16(float(v))


def schraudolph_y(x: float) -> float:
    return _load().ora_schraudolph_y(float(x))


def schraudolph_code(y: float) -> int:
    return _load().ora_schraudolph_code(float(y))


def mx_quantize(x_bits: np.ndarray, block_axis: int, fmt: int):
    """MX-quantize bf16 bit patterns x[batch][rows][cols] (uint16).

    Returns (codes, scales) laid out as in ``fsa_oracle.c:ora_mx_quantize``.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if x.ndim == 2:
        x = x[None]
    batch, rows, cols = x.shape
    if block_axis == 1:
        codes = np.zeros((batch, rows, cols), np.uint8)
        scales = np.zeros((batch, rows, (cols + 31) // 32), np.uint8)
    else:
        codes = np.zeros((batch, cols, rows), np.uint8)
        scales = np.zeros((batch, cols, (rows + 31) // 32), np.uint8)
    rc = _load().ora_mx_quantize(_ptr(x), batch, rows, cols, block_axis, fmt,
                                 _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError(f"ora_mx_quantize failed ({rc})")
    return codes, scales


# ------------------------------------------------------------- attention --
MODES = ("fused", "conventional", "exact", "exact_frozen", "operands_only", "efq", "online")


# EFQ affine rule parameters, calibrated offline by oracle/efq_calibrate.py
# (tests/golden/efq_calibration.txt)
EFQ_TAU, EFQ_H = -2.44, 0.61


def attention(q_bits, k_bits, v_bits, *, fmt: str | None = "mxfp8", mode: str = "fused",
              threshold: float = 8.0, tile: int = 128, sm_scale: float = 0.0,
              rows=None, threads: int | None = None, want_bits: bool = False,
              want_margins: bool = False, gate: str = "fp32", efq_tau: float | None = None,
              efq_h: float | None = None, p_elem: str | None = None):
    """Oracle attention on bf16 bit patterns q[BH][Sq][D], k/v[BH][Sk][D]
    (uint16; Sq = Sk for self-attention).

    mode:
      "fused"         -- the method: MX Q/K/V, frozen reference + gate,
                         Schraudolph code, two-stage MX P, l from the same P.
      "conventional"  -- conventional softmax on the same quantized operands:
                         MX Q/K/V, exact row max, exact exp, MX P, l from the
                         unquantized P.
      "operands_only" -- MX Q/K/V, exact softmax, P not quantized.
      "exact"         -- FP64 softmax attention on the bf16 inputs.
      "exact_frozen"  -- the method's frozen reference and gate with exact exp
                         and no quantization (equals "exact" for any theta).
      "efq"           -- EFQ-Softmax: MX Q/K/V (fmt, normally "mxfp4"), online
                         attention with the running row max, E2M1 P codes
                         generated directly from the shifted scores with the
                         affine rule (efq_tau, efq_h; defaults EFQ_TAU, EFQ_H),
                         l from the same P.
      "online"        -- online attention with the running max and exact exp,
                         no quantization (equals "exact").
    rows: optional global query-row indices bh*Sq+i; outputs follow that order.
    p_elem: optional P element format overriding the format's own ("e4m3",
    "e2m3", "e2m1"), e.g. MXFP4 with E2M1 P for the conventional baseline of
    the EFQ comparison.
    gate: "fp32" (tile max - m > theta) or "shortcut" (the tile's largest P
    block scale under the frozen reference exceeds the scale of theta's code;
    fused mode only).
    Returns a dict with "out" (float64 [n][D]), "out_bf16" (uint16),
    "m", "l", "rollback_count" and optionally "bits" / "margins" [n][n_t].
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    if q.ndim == 4:
        q = q.reshape(-1, q.shape[-2], q.shape[-1])
        k = k.reshape(-1, k.shape[-2], k.shape[-1])
        v = v.reshape(-1, v.shape[-2], v.shape[-1])
    BH, Sq, D = q.shape
    S = k.shape[1]          # keys
    if k.shape != (BH, S, D) or v.shape != (BH, S, D):
        raise ValueError("k and v must be [BH][Sk][D] with q's BH and D")
    qkv_fmt, p_fmt = FORMATS[fmt] if fmt is not None else (-1, -1)
    p = _Params()
    p.tile, p.threshold, p.sm_scale = tile, float(threshold), float(sm_scale)
    if gate not in ("fp32", "shortcut"):
        raise ValueError(gate)
    p.gate_mode = 1 if gate == "shortcut" else 0
    p.efq_tau = EFQ_TAU if efq_tau is None else float(efq_tau)
    p.efq_h = EFQ_H if efq_h is None else float(efq_h)
    if mode == "fused":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = qkv_fmt, p_fmt, 1, 0, 0
    elif mode == "conventional":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = qkv_fmt, p_fmt, 0, 1, 1
    elif mode == "operands_only":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = qkv_fmt, -1, 0, 1, 1
    elif mode == "exact":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = -1, -1, 0, 1, 1
    elif mode == "exact_frozen":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = -1, -1, 0, 0, 1
    elif mode == "efq":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = qkv_fmt, -1, 2, 2, 0
    elif mode == "online":
        p.qkv_fmt, p.p_fmt, p.exp_mode, p.max_mode, p.l_from_unquantized = -1, -1, 0, 2, 1
    else:
        raise ValueError(mode)
    if p_elem is not None:
        p.p_fmt = {"e4m3": 0, "e2m3": 1, "e2m1": 2}[p_elem]
    if rows is None:
        rows_arr = None
        n = BH * Sq
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    n_t = (S + tile - 1) // tile
    out = np.empty((n, D), np.float64)
    out_bf16 = np.empty((n, D), np.uint16)
    bits = np.zeros((n, n_t), np.uint8) if want_bits else None
    margins = np.full((n, n_t), np.nan) if want_margins else None
    row_m = np.empty(n, np.float64)
    row_l = np.empty(n, np.float64)
    cnt = ctypes.c_int64(0)
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    rc = _load().ora_attention_qk(_ptr(q), _ptr(k), _ptr(v), BH, Sq, S, D, ctypes.byref(p),
                                  _ptr(rows_arr), n, int(threads), _ptr(out), _ptr(out_bf16),
                                  _ptr(bits), _ptr(margins), _ptr(row_m), _ptr(row_l),
                                  ctypes.byref(cnt))
    if rc != 0:
        raise ValueError(f"ora_attention failed ({rc})")
    res = {"out": out, "out_bf16": out_bf16, "m": row_m, "l": row_l,
           "rollback_count": int(cnt.value)}
    if want_bits:
        res["bits"] = bits
    if want_margins:
        res["margins"] = margins
    return res


def rel_l2(a, b) -> float:
    """Global relative error ||a - b||_F / ||b||_F."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def sm_default(D: int) -> float:
    return 1.0 / math.sqrt(D)

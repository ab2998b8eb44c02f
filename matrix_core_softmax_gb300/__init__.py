"""Python binding of libfsa.so, the GB300 Fused-Softmax MX attention library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/fsa.h``.  PyTorch supplies
device memory and streams.  There is no fallback: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfsa.so")

FSA_MXFP8, FSA_MXFP6, FSA_MXFP4, FSA_MXFP4_EFQ = 0, 1, 2, 3
FORMATS = {"mxfp8": FSA_MXFP8, "mxfp6": FSA_MXFP6, "mxfp4": FSA_MXFP4, "mxfp4_efq": FSA_MXFP4_EFQ}
ELEM_E4M3, ELEM_E2M3, ELEM_E2M1 = 0, 1, 2
DEBUG_SKIP_KV_ARRIVE = 0x1

STATUS = {0: "FSA_OK", 1: "FSA_ERR_INVALID_ARGUMENT", 2: "FSA_ERR_UNSUPPORTED",
          3: "FSA_ERR_CUDA", 4: "FSA_ERR_OUT_OF_MEMORY", 5: "FSA_ERR_TIMEOUT"}

# every symbol include/fsa.h declares
EXPORTS = ("fsa_quantize_mx", "fsa_attention_fwd", "fsa_attention_fwd_ex",
           "fsa_attention_prepare", "fsa_attention_run", "fsa_attention_workspace_size", "fsa_bf16_attention_fwd", "fsa_get_device_error",
           "fsa_status_string", "fsa_release_workspace", "fsa_attention_fwd_noalloc",
           "fsa_cross_attention_fwd", "fsa_cross_attention_workspace_size",
           "fsa_cross_attention_prepare", "fsa_cross_attention_run",
           "fsa_attention_fwd_host", "fsa_cross_attention_fwd_host", "fsa_mma_rate_probe")


class FsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [
        ("sm_scale", ctypes.c_float),
        ("rollback_bits", ctypes.c_void_p),
        ("rollback_count", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64),
        ("wait_timeout_ms", ctypes.c_int),
        ("debug_flags", ctypes.c_int),
        ("efq_tau", ctypes.c_float),
        ("efq_h", ctypes.c_float),
        ("host_inputs_ready", ctypes.c_int),
        ("gate_mode", ctypes.c_int),
    ]

GATE_MODES = {"fp32": 0, "shortcut": 1}


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libfsa.so (built by ``matrix_core_softmax_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise OSError(f"libfsa.so not built ({p}); run matrix_core_softmax_gb300/build.py")
            lib = ctypes.CDLL(p)
            V, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.fsa_quantize_mx.argtypes = [V, I64, I64, I64, I, I, V, V, V]
            lib.fsa_quantize_mx.restype = I
            lib.fsa_attention_fwd.argtypes = [V, V, V, V, I, I, I, I, I, F, V]
            lib.fsa_attention_fwd.restype = I
            lib.fsa_attention_fwd_ex.argtypes = [V, V, V, V, I, I, I, I, I, F,
                                                 ctypes.POINTER(Options), V]
            lib.fsa_attention_fwd_ex.restype = I
            lib.fsa_attention_prepare.argtypes = [V, V, V, I, I, I, I, I, V, ctypes.c_uint64, V]
            lib.fsa_attention_prepare.restype = I
            lib.fsa_attention_run.argtypes = [V, ctypes.c_uint64, V, I, I, I, I, I, F,
                                              ctypes.POINTER(Options), V]
            lib.fsa_attention_run.restype = I
            lib.fsa_attention_workspace_size.argtypes = [I, I, I, I, I]
            lib.fsa_attention_workspace_size.restype = ctypes.c_uint64
            lib.fsa_cross_attention_fwd.argtypes = [V, V, V, V, I, I, I, I, I, I, F,
                                                    ctypes.POINTER(Options), V]
            lib.fsa_cross_attention_fwd.restype = I
            lib.fsa_cross_attention_workspace_size.argtypes = [I, I, I, I, I, I]
            lib.fsa_cross_attention_workspace_size.restype = ctypes.c_uint64
            lib.fsa_cross_attention_prepare.argtypes = [V, V, V, I, I, I, I, I, I, V,
                                                        ctypes.c_uint64, V]
            lib.fsa_cross_attention_prepare.restype = I
            lib.fsa_cross_attention_run.argtypes = [V, ctypes.c_uint64, V, I, I, I, I, I, I, F,
                                                    ctypes.POINTER(Options), V]
            lib.fsa_cross_attention_run.restype = I
            lib.fsa_attention_fwd_host.argtypes = [V, V, V, V, I, I, I, I, I, F,
                                                   ctypes.POINTER(Options), V]
            lib.fsa_attention_fwd_host.restype = I
            lib.fsa_cross_attention_fwd_host.argtypes = [V, V, V, V, I, I, I, I, I, I, F,
                                                         ctypes.POINTER(Options), V]
            lib.fsa_cross_attention_fwd_host.restype = I
            lib.fsa_attention_fwd_noalloc.argtypes = [V, V, V, V, I, I, I, I, I, F, V]
            lib.fsa_attention_fwd_noalloc.restype = I
            lib.fsa_bf16_attention_fwd.argtypes = [V, V, V, V, I, I, I, I, V]
            lib.fsa_bf16_attention_fwd.restype = I
            lib.fsa_mma_rate_probe.argtypes = [I, I, I, ctypes.POINTER(ctypes.c_double), V]
            lib.fsa_mma_rate_probe.restype = I
            lib.fsa_get_device_error.argtypes = [V]
            lib.fsa_get_device_error.restype = I
            lib.fsa_status_string.argtypes = [I]
            lib.fsa_status_string.restype = ctypes.c_char_p
            lib.fsa_release_workspace.argtypes = []
            lib.fsa_release_workspace.restype = None
            _lib = lib
    return _lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str):
    if status != 0:
        raise FsaError(status, what)


def _bhsd(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B, H, S, D]")


def quantize_mx(x: torch.Tensor, block_axis: int, elem: int, stream=None):
    """MX-quantize x [batch, rows, cols] (bf16, CUDA).  Returns (codes, scales)
    in the layouts documented for fsa_quantize_mx."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 tensor")
    x3 = x if x.dim() == 3 else x.reshape(1, *x.shape[-2:])
    b, r, c = x3.shape
    if block_axis == 1:
        codes = torch.empty((b, r, c), dtype=torch.uint8, device=x.device)
        scales = torch.empty((b, r, (c + 31) // 32), dtype=torch.uint8, device=x.device)
    else:
        codes = torch.empty((b, c, r), dtype=torch.uint8, device=x.device)
        scales = torch.empty((b, c, (r + 31) // 32), dtype=torch.uint8, device=x.device)
    _check(load().fsa_quantize_mx(_ptr(x3), b, r, c, block_axis, elem, _ptr(codes), _ptr(scales),
                                  _stream(stream)), "fsa_quantize_mx")
    return codes, scales


def workspace_size(B: int, H: int, S: int, D: int, fmt: str = "mxfp8") -> int:
    return int(load().fsa_attention_workspace_size(B, H, S, D, FORMATS[fmt]))


def attention_fwd(q, k, v, fmt: str = "mxfp8", threshold: float = 8.0, *, out=None,
                  sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                  workspace=None, wait_timeout_ms: int = 0, efq_tau: float = 0.0, efq_h: float = 0.0, debug_flags: int = 0, gate: str = "fp32", stream=None):
    """Fused-Softmax MX attention forward (fsa_attention_fwd_ex).

    q, k, v: contiguous CUDA bf16 [B, H, S, D].  rollback_bits: optional uint8
    CUDA tensor [B*H*S, ceil(S/128)]; rollback_count: optional int64 CUDA
    tensor [1] to which the number of gate firings is added."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, S, D = q.shape
    o = torch.empty_like(q) if out is None else out
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    if workspace is not None:
        opt.workspace = workspace.data_ptr()
        opt.workspace_bytes = workspace.numel() * workspace.element_size()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.wait_timeout_ms = wait_timeout_ms
    opt.debug_flags = debug_flags
    _check(load().fsa_attention_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S, D,
                                       FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                       _stream(stream)), "fsa_attention_fwd_ex")
    return o


def cross_attention_fwd(q, k, v, fmt: str = "mxfp8", threshold: float = 8.0, *, out=None,
                        sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                        workspace=None, wait_timeout_ms: int = 0, efq_tau: float = 0.0, efq_h: float = 0.0, gate: str = "fp32", stream=None):
    """fsa_cross_attention_fwd: q contiguous CUDA bf16 [B, H, Sq, D], k and v
    [B, H, Sk, D]; returns o [B, H, Sq, D].  rollback_bits: optional uint8
    CUDA tensor [B*H*Sq, ceil(Sk/128)]."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if k.shape != (B, H, Sk, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Sk, D] with q's B, H and D")
    o = torch.empty_like(q) if out is None else out
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    if workspace is not None:
        opt.workspace = workspace.data_ptr()
        opt.workspace_bytes = workspace.numel() * workspace.element_size()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.wait_timeout_ms = wait_timeout_ms
    _check(load().fsa_cross_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Sq, Sk, D,
                                          FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                          _stream(stream)), "fsa_cross_attention_fwd")
    return o


def _host_bhsd(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.is_cuda or t.dim() != 4 \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host (CPU) bf16 tensor [B, H, S, D]")


def cross_attention_fwd_host(q, k, v, fmt: str = "mxfp8", threshold: float = 8.0, *, out=None,
                             sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                             efq_tau: float = 0.0, efq_h: float = 0.0, host_inputs_ready: bool = False,
                             gate: str = "fp32", stream=None):
    """fsa_cross_attention_fwd_host: q, k, v contiguous HOST bf16 tensors
    ([B, H, Sq, D] and [B, H, Sk, D]; pinned memory lets the copies overlap
    the computation); returns the host output o [B, H, Sq, D] (or fills
    `out`).  Asynchronous on `stream`: synchronise it before reading o.
    rollback_bits / rollback_count, when given, are CUDA tensors.
    host_inputs_ready: q, k, v are final now (no earlier work on `stream`
    writes them), so their copy-in need not wait for that work."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _host_bhsd(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    if k.shape != (B, H, Sk, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Sk, D] with q's B, H and D")
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=q.is_pinned()) if out is None else out
    _host_bhsd(o, "out")
    if o.shape != q.shape:
        raise ValueError("out must have q's shape")
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.host_inputs_ready = int(bool(host_inputs_ready))
    _check(load().fsa_cross_attention_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Sq, Sk, D,
                                               FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                               _stream(stream)), "fsa_cross_attention_fwd_host")
    return o


def attention_fwd_host(q, k, v, fmt: str = "mxfp8", threshold: float = 8.0, *, out=None,
                       sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                       efq_tau: float = 0.0, efq_h: float = 0.0, host_inputs_ready: bool = False,
                       gate: str = "fp32", stream=None):
    """fsa_attention_fwd_host: self-attention on contiguous HOST bf16 tensors
    [B, H, S, D]; see cross_attention_fwd_host."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _host_bhsd(t, n)
    B, H, S, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have one shape [B, H, S, D]")
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=q.is_pinned()) if out is None else out
    _host_bhsd(o, "out")
    if o.shape != q.shape:
        raise ValueError("out must have q's shape")
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.host_inputs_ready = int(bool(host_inputs_ready))
    _check(load().fsa_attention_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S, D,
                                         FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                         _stream(stream)), "fsa_attention_fwd_host")
    return o


def cross_workspace_size(B: int, H: int, Sq: int, Sk: int, D: int, fmt: str = "mxfp8") -> int:
    return int(load().fsa_cross_attention_workspace_size(B, H, Sq, Sk, D, FORMATS[fmt]))


def new_cross_workspace(B: int, H: int, Sq: int, Sk: int, D: int, fmt: str = "mxfp8", device="cuda"):
    """A device workspace tensor sized for cross_attention_prepare / _run."""
    return torch.empty(cross_workspace_size(B, H, Sq, Sk, D, fmt), dtype=torch.uint8, device=device)


def cross_attention_prepare(q, k, v, workspace, fmt: str = "mxfp8", stream=None):
    """First half of cross_attention_fwd: MX-quantize q, k, v into `workspace`."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    _check(load().fsa_cross_attention_prepare(_ptr(q), _ptr(k), _ptr(v), B, H, Sq, Sk, D,
                                              FORMATS[fmt], _ptr(workspace), workspace.numel(),
                                              _stream(stream)), "fsa_cross_attention_prepare")


def cross_attention_run(workspace, out, Sk: int, fmt: str = "mxfp8", threshold: float = 8.0, *,
                        sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                        wait_timeout_ms: int = 0, efq_tau: float = 0.0, efq_h: float = 0.0, gate: str = "fp32", stream=None):
    """Second half of cross_attention_fwd: `out` [B, H, Sq, D] fixes B, H, Sq and D;
    Sk is the key length given to cross_attention_prepare."""
    _bhsd(out, "out")
    B, H, Sq, D = out.shape
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.wait_timeout_ms = wait_timeout_ms
    _check(load().fsa_cross_attention_run(_ptr(workspace), workspace.numel(), _ptr(out), B, H, Sq,
                                          Sk, D, FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                          _stream(stream)), "fsa_cross_attention_run")
    return out


def new_workspace(B: int, H: int, S: int, D: int, fmt: str = "mxfp8", device="cuda"):
    """A device workspace tensor sized for attention_prepare / attention_run."""
    return torch.empty(workspace_size(B, H, S, D, fmt), dtype=torch.uint8, device=device)


def attention_prepare(q, k, v, workspace, fmt: str = "mxfp8", stream=None):
    """First half of attention_fwd: MX-quantize q, k, v into `workspace`."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, S, D = q.shape
    _check(load().fsa_attention_prepare(_ptr(q), _ptr(k), _ptr(v), B, H, S, D, FORMATS[fmt],
                                        _ptr(workspace), workspace.numel(), _stream(stream)),
           "fsa_attention_prepare")


def attention_run(workspace, out, fmt: str = "mxfp8", threshold: float = 8.0, *,
                  sm_scale: float = 0.0, rollback_bits=None, rollback_count=None,
                  wait_timeout_ms: int = 0, efq_tau: float = 0.0, efq_h: float = 0.0, gate: str = "fp32", stream=None):
    """Second half of attention_fwd: the fused kernel on a prepared workspace;
    `out` is the bf16 [B, H, S, D] output and fixes the shape."""
    _bhsd(out, "out")
    B, H, S, D = out.shape
    opt = Options()
    opt.sm_scale = sm_scale
    opt.rollback_bits = None if rollback_bits is None else rollback_bits.data_ptr()
    opt.rollback_count = None if rollback_count is None else rollback_count.data_ptr()
    opt.efq_tau, opt.efq_h = efq_tau, efq_h
    opt.gate_mode = GATE_MODES[gate]
    opt.wait_timeout_ms = wait_timeout_ms
    _check(load().fsa_attention_run(_ptr(workspace), workspace.numel(), _ptr(out), B, H, S, D,
                                    FORMATS[fmt], float(threshold), ctypes.byref(opt),
                                    _stream(stream)), "fsa_attention_run")
    return out


def attention_fwd_noalloc(q, k, v, fmt: str = "mxfp8", threshold: float = 8.0, *, out=None,
                          stream=None):
    """fsa_attention_fwd_noalloc: the fused attention with the library's fixed
    64 MiB scratch array instead of an allocated workspace (see include/fsa.h)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, S, D = q.shape
    o = torch.empty_like(q) if out is None else out
    _check(load().fsa_attention_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S, D,
                                            FORMATS[fmt], float(threshold), _stream(stream)),
           "fsa_attention_fwd_noalloc")
    return o


def bf16_attention_fwd(q, k, v, *, out=None, stream=None):
    """Conventional BF16 flash attention (fsa_bf16_attention_fwd)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bhsd(t, n)
    B, H, S, D = q.shape
    o = torch.empty_like(q) if out is None else out
    _check(load().fsa_bf16_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S, D,
                                         _stream(stream)), "fsa_bf16_attention_fwd")
    return o


# kinds of fsa_mma_rate_probe
PROBE_KINDS = {"mxf8f6f4_e4m3": 0, "mxf8f6f4_e2m3": 1, "mxf4_e2m1": 2, "attention_tile_e4m3": 3,
               "f16_bf16": 4}


def mma_rate_probe(kind: str, ctas: int, iters: int, stream=None) -> float:
    """fsa_mma_rate_probe: launches the tensor-core rate probe on the stream
    (the caller times it) and returns the launch's floating-point operations."""
    fl = ctypes.c_double(0.0)
    _check(load().fsa_mma_rate_probe(PROBE_KINDS[kind], int(ctas), int(iters), ctypes.byref(fl),
                                     _stream(stream)), "fsa_mma_rate_probe")
    return fl.value


def get_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(load().fsa_get_device_error(_stream(stream)))


def status_string(s: int) -> str:
    return load().fsa_status_string(int(s)).decode()


def release_workspace():
    load().fsa_release_workspace()

"""Python binding of the ``vaedec`` C ABI (``include/vaedec.h``).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch is used by callers for device memory and streams; this module
accepts ``torch`` tensors for device buffers and numpy arrays for host weights.
If the shared library has not been built, :func:`load_library` raises -- there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

from .build import lib_path

__all__ = ["Decoder", "VaedecError", "load_library", "EXPORTED_SYMBOLS", "STATUS_NAMES", "inject_fault",
           "band_axis", "BAND_AXES", "band_attention", "band_attention_work_bytes", "groupnorm_noalloc",
           "plan_workspace",
           "set_wait_limit"]

FAMILY = {"kl2d": 1, "wan3d": 2}
DTYPE = {"fp32": 1, "bf16": 2}
MAX_STAGES = 6
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "OOM", 4: "CUDA", 5: "TIMEOUT", 6: "STOPPED"}

EXPORTED_SYMBOLS = (
    "vaedec_create", "vaedec_destroy", "vaedec_output_shape", "vaedec_workspace_bytes",
    "vaedec_decode", "vaedec_decode_host", "vaedec_sync", "vaedec_last_error",
    "vaedec_launch_count", "vaedec_profile_enable", "vaedec_profile_read",
    "vaedec_debug_num_ops", "vaedec_debug_op_desc", "vaedec_debug_run_until",
    "vaedec_groupnorm_noalloc", "vaedec_debug_inject_fault", "vaedec_debug_set_wait_limit",
    "vaedec_debug_wait_probe", "vaedec_band_axis", "vaedec_decode_bands",
    "vaedec_band_attention_work_bytes", "vaedec_band_attention", "vaedec_plan_workspace",
)


class VaedecError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Tensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("data", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("ndim", ctypes.c_int), ("shape", ctypes.c_int64 * 5)]


class _Config(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int), ("dtype", ctypes.c_int),
                ("latent_channels", ctypes.c_int), ("mid_channels", ctypes.c_int),
                ("out_channels", ctypes.c_int), ("n_stages", ctypes.c_int),
                ("stage_channels", ctypes.c_int * MAX_STAGES),
                ("stage_resnets", ctypes.c_int * MAX_STAGES),
                ("stage_upsample", ctypes.c_int * MAX_STAGES),
                ("stage_up_channels", ctypes.c_int * MAX_STAGES),
                ("norm_groups", ctypes.c_int), ("eps", ctypes.c_float),
                ("max_latent", ctypes.c_int64 * 4),
                ("latent_patch", ctypes.c_int), ("latent_bn_eps", ctypes.c_float)]


_LIB: Optional[ctypes.CDLL] = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the built library (raises if it is missing)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"vaedec library not built ({p} missing): run "
                           "`python -m row_band_layerwise_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, i64p, i = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int
    lib.vaedec_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Tensor), i, ctypes.POINTER(vp)]
    lib.vaedec_destroy.argtypes = [vp]
    lib.vaedec_destroy.restype = None
    lib.vaedec_output_shape.argtypes = [vp, i64p, i, i64p]
    lib.vaedec_workspace_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    lib.vaedec_decode.argtypes = [vp, vp, i64p, i, vp, i, vp]
    lib.vaedec_decode_host.argtypes = [vp, vp, i64p, i, vp, i, vp]
    lib.vaedec_sync.argtypes = [vp, vp]
    lib.vaedec_last_error.restype = ctypes.c_char_p
    lib.vaedec_last_error.argtypes = []
    lib.vaedec_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
    lib.vaedec_profile_enable.argtypes = [vp, i]
    lib.vaedec_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i, ctypes.POINTER(i)]
    lib.vaedec_debug_num_ops.argtypes = [vp, i64p, i, i, ctypes.POINTER(i)]
    lib.vaedec_debug_op_desc.argtypes = [vp, i64p, i, i, i, ctypes.c_char_p, i]
    lib.vaedec_debug_run_until.argtypes = [vp, vp, i64p, i, i, i, vp, ctypes.c_size_t, vp, ctypes.c_size_t,
                                           vp, ctypes.c_size_t, vp]
    lib.vaedec_groupnorm_noalloc.argtypes = [i, i, vp, vp, i, i, i, i, i, vp, vp, ctypes.c_float, i, vp]
    lib.vaedec_debug_inject_fault.argtypes = [i, i]
    lib.vaedec_debug_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.vaedec_debug_wait_probe.argtypes = [vp, vp]
    lib.vaedec_band_axis.argtypes = [i64p, i, i, i, ctypes.POINTER(i)]
    lib.vaedec_decode_bands.argtypes = [vp, vp, i64p, i, vp, i, i, vp]
    lib.vaedec_band_attention_work_bytes.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.vaedec_band_attention.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp, ctypes.c_size_t, vp, vp]
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.vaedec_plan_workspace.argtypes = [ctypes.POINTER(_Config), szp, szp, szp]
    for name in EXPORTED_SYMBOLS:
        if name not in ("vaedec_destroy", "vaedec_last_error"):
            getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _LIB = lib
    return lib


def _check(lib, status: int) -> None:
    if status != 0:
        raise VaedecError(status, lib.vaedec_last_error().decode(errors="replace"))


def _shape_arg(shape: Sequence[int]):
    return (ctypes.c_int64 * len(shape))(*[int(s) for s in shape])


def make_config(arch, dtype: str, max_latent: Sequence[int]) -> _Config:
    """Fill a ``vaedec_config`` from an architecture description.

    ``arch`` needs the attributes family, latent_channels, mid_channels,
    out_channels, stage_channels, stage_resnets, stage_upsample,
    stage_up_channels, norm_groups and eps, and optionally latent_patch and latent_bn_eps (the
    AutoencoderKLFlux2 latent front-end); ``max_latent`` is (B, T, H, W) in the decode input's units.
    """
    c = _Config()
    c.family = FAMILY[arch.family]
    c.dtype = DTYPE[dtype]
    c.latent_channels = arch.latent_channels
    c.mid_channels = arch.mid_channels
    c.out_channels = arch.out_channels
    n = len(arch.stage_channels)
    if n > MAX_STAGES:
        raise ValueError("too many stages")
    c.n_stages = n
    for s in range(n):
        c.stage_channels[s] = arch.stage_channels[s]
        c.stage_resnets[s] = arch.stage_resnets[s]
        c.stage_upsample[s] = arch.stage_upsample[s]
        c.stage_up_channels[s] = arch.stage_up_channels[s]
    c.norm_groups = arch.norm_groups
    c.eps = arch.eps
    for k in range(4):
        c.max_latent[k] = int(max_latent[k])
    c.latent_patch = int(getattr(arch, "latent_patch", 1))
    c.latent_bn_eps = float(getattr(arch, "latent_bn_eps", 0.0))
    return c


FAULT_KINDS = {"off": 0, "alloc": 1, "launch": 2}


def inject_fault(kind: str, nth: int = 1) -> None:
    """Make the nth device allocation of a create fail ("alloc"), or stop a decode at its nth
    kernel launch ("launch"), once; "off" clears a pending fault.  Process-wide, for tests."""
    lib = load_library()
    _check(lib, lib.vaedec_debug_inject_fault(FAULT_KINDS[kind], int(nth)))


def set_wait_limit(ns: int) -> None:
    """Set the limit of the kernels' bounded waits in nanoseconds (0 restores the default)."""
    lib = load_library()
    _check(lib, lib.vaedec_debug_set_wait_limit(int(ns)))


BAND_AXES = {"height": 0, "width": 1, "auto": 2}


def band_axis(latent_shape, n_bands: int, axis: str = "auto") -> str:
    """The axis ("height" or "width") a decode of ``latent_shape`` in ``n_bands`` bands is split
    along for the requested ``axis`` (vaedec_band_axis: auto takes the longer latent axis that can
    hold every band, width on ties).  Host only."""
    lib = load_library()
    out = ctypes.c_int(-1)
    _check(lib, lib.vaedec_band_axis(_shape_arg(latent_shape), len(latent_shape), int(n_bands),
                                     BAND_AXES[axis], ctypes.byref(out)))
    return "height" if out.value == 0 else "width"


def groupnorm_noalloc(x, y, groups: int, gamma, beta, eps: float, silu: bool, stream=None) -> None:
    """GroupNorm (+SiLU) of a channels-last [B, rows, W, C] device tensor into ``y`` without
    any device allocation (scratch lives in a fixed array inside the library).

    ``gamma``/``beta`` are fp32 device tensors of C values.  Asynchronous on ``stream``.
    """
    lib = load_library()
    torch = _torch()
    dt = {torch.float32: DTYPE["fp32"], torch.bfloat16: DTYPE["bf16"]}
    if x.dim() != 4:
        raise ValueError("x must be a channels-last [B, rows, W, C] tensor")
    dev = torch.device("cuda", torch.cuda.current_device())
    for name, t in (("x", x), ("y", y), ("gamma", gamma), ("beta", beta)):
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be a CUDA tensor on the current device {dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if tuple(y.shape) != tuple(x.shape):
        raise ValueError("y must have the shape of x")
    if x.dtype not in dt or y.dtype not in dt:
        raise ValueError("x and y must be float32 or bfloat16")
    B, rows, W, C = (int(v) for v in x.shape)
    for name, t in (("gamma", gamma), ("beta", beta)):
        if t.dtype != torch.float32 or t.numel() != C:
            raise ValueError(f"{name} must be float32 with C = {C} values")
    st = torch.cuda.current_stream() if stream is None else stream
    _check(lib, lib.vaedec_groupnorm_noalloc(dt[x.dtype], dt[y.dtype], x.data_ptr(), y.data_ptr(), B, rows, W, C,
                                             int(groups), gamma.data_ptr(), beta.data_ptr(), float(eps),
                                             1 if silu else 0, int(st.cuda_stream)))


def plan_workspace(arch, dtype: str, max_latent: Sequence[int]) -> dict:
    """Workspace a decoder for ``arch`` / ``dtype`` / ``max_latent`` (B, T, H, W) would own, planned
    on the host without a GPU: {"bytes": total, "arena": activation arena, "peak_live": the largest
    sum of activations alive at once}."""
    lib = load_library()
    cfg = make_config(arch, dtype, max_latent)
    b, a, p = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib, lib.vaedec_plan_workspace(ctypes.byref(cfg), ctypes.byref(b), ctypes.byref(a), ctypes.byref(p)))
    return {"bytes": int(b.value), "arena": int(a.value), "peak_live": int(p.value)}


def band_attention_work_bytes(F: int, grid_h: int, grid_w: int, C: int) -> int:
    """Device scratch bytes ``band_attention`` needs for these sizes (0: none)."""
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib, lib.vaedec_band_attention_work_bytes(int(F), int(grid_h), int(grid_w), int(C), ctypes.byref(n)))
    return int(n.value)


def band_attention(q, k, vt, out, grid_h: int, grid_w: int, n_bands: int, work, status, stream=None) -> None:
    """softmax(Q K^T / sqrt(C)) V per frame with band-local queries, on the fused attention kernel.

    ``q``/``k``/``out``: bf16 device tensors [F, ntok, C]; ``vt``: bf16 [F, C, ntok];
    ``work``: a device tensor of at least ``band_attention_work_bytes`` bytes, or None when that is 0;
    ``status``: an int32 device tensor the kernel ORs a timeout bit into.  Asynchronous on ``stream``.
    """
    lib = load_library()
    torch = _torch()
    # the kernel reads and writes through raw pointers: every extent is checked here first
    if q.dim() != 3:
        raise ValueError("q must be [F, ntok, C]")
    F, ntok, C = (int(v) for v in q.shape)
    if ntok != int(grid_h) * int(grid_w):
        raise ValueError(f"q has {ntok} tokens per frame, the grid {grid_h} x {grid_w} has {int(grid_h) * int(grid_w)}")
    dev = q.device
    for name, t, shape in (("q", q, (F, ntok, C)), ("k", k, (F, ntok, C)), ("vt", vt, (F, C, ntok)),
                           ("out", out, (F, ntok, C))):
        if not t.is_cuda or t.device != dev or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor on {dev}")
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if not status.is_cuda or status.device != dev or status.dtype != torch.int32 or status.numel() < 1:
        raise ValueError(f"status must be an int32 tensor on {dev}")
    need = band_attention_work_bytes(F, grid_h, grid_w, C)
    if work is not None:
        if not work.is_cuda or work.device != dev or not work.is_contiguous():
            raise ValueError(f"work must be a contiguous tensor on {dev}")
    wb = work.numel() * work.element_size() if work is not None else 0
    if wb < need:
        raise ValueError(f"work holds {wb} bytes, the key splits need {need}")
    st = torch.cuda.current_stream() if stream is None else stream
    wp = work.data_ptr() if work is not None else None
    _check(lib, lib.vaedec_band_attention(q.data_ptr(), k.data_ptr(), vt.data_ptr(), out.data_ptr(), F, int(grid_h),
                                          int(grid_w), C, int(n_bands), wp, wb, status.data_ptr(),
                                          int(st.cuda_stream)))


def _torch():
    import torch
    return torch


class Decoder:
    """One decoder handle: device weights plus workspace sized for ``max_latent``."""

    def __init__(self, arch, weights: Dict[str, np.ndarray], dtype: str,
                 max_latent: Sequence[int], lib_file: Optional[str] = None):
        self.lib = load_library(lib_file)
        self.arch = arch
        self.dtype = dtype
        self.family = arch.family
        cfg = make_config(arch, dtype, max_latent)
        keep = []
        arr = (_Tensor * len(weights))()
        for i, (name, w) in enumerate(weights.items()):
            a = np.ascontiguousarray(w, dtype=np.float32)
            keep.append(a)
            arr[i].name = name.encode()
            arr[i].data = a.ctypes.data
            arr[i].dtype = DTYPE["fp32"]
            arr[i].ndim = a.ndim
            for k in range(a.ndim):
                arr[i].shape[k] = a.shape[k]
        handle = ctypes.c_void_p()
        _check(self.lib, self.lib.vaedec_create(ctypes.byref(cfg), arr, len(weights), ctypes.byref(handle)))
        self._h = handle
        self.device = _torch().cuda.current_device()   # the device the handle's memory lives on
        del keep

    # ------------------------------------------------------------------ basics
    def close(self) -> None:
        if getattr(self, "_h", None):
            self.lib.vaedec_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def torch_dtype(self):
        torch = _torch()
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def output_shape(self, latent_shape: Sequence[int]) -> Tuple[int, ...]:
        n = len(latent_shape)
        out = (ctypes.c_int64 * n)()
        _check(self.lib, self.lib.vaedec_output_shape(self._h, _shape_arg(latent_shape), n, out))
        return tuple(int(v) for v in out)

    def workspace_bytes(self) -> int:
        v = ctypes.c_size_t()
        _check(self.lib, self.lib.vaedec_workspace_bytes(self._h, ctypes.byref(v)))
        return int(v.value)

    @staticmethod
    def _stream_ptr(stream) -> int:
        torch = _torch()
        if stream is None:
            stream = torch.cuda.current_stream()
        return int(stream.cuda_stream)

    # ------------------------------------------------------------------ decode
    def decode(self, latent, n_bands: int, out=None, stream=None, axis: str = "height"):
        """Decode a device latent (torch tensor, channels-first, model dtype) on ``stream``, split
        into ``n_bands`` bands along ``axis`` ("height", "width" or "auto"; see band_axis)."""
        torch = _torch()
        if not latent.is_cuda or latent.dtype != self.torch_dtype or not latent.is_contiguous():
            raise ValueError("latent must be a contiguous CUDA tensor in the model dtype")
        if latent.device.index != self.device:
            raise ValueError(f"latent is on {latent.device}, the decoder on cuda:{self.device}")
        oshape = self.output_shape(latent.shape)
        if out is None:
            out = torch.empty(oshape, dtype=self.torch_dtype, device=latent.device)
        elif (not out.is_cuda or out.device != latent.device or tuple(out.shape) != oshape or
              out.dtype != self.torch_dtype or not out.is_contiguous()):
            raise ValueError(f"out must be a contiguous {self.torch_dtype} tensor of shape {oshape} on {latent.device}")
        if axis == "height":
            _check(self.lib, self.lib.vaedec_decode(self._h, latent.data_ptr(), _shape_arg(latent.shape),
                                                    latent.dim(), out.data_ptr(), int(n_bands),
                                                    self._stream_ptr(stream)))
        else:
            _check(self.lib, self.lib.vaedec_decode_bands(self._h, latent.data_ptr(), _shape_arg(latent.shape),
                                                          latent.dim(), out.data_ptr(), int(n_bands),
                                                          BAND_AXES[axis], self._stream_ptr(stream)))
        return out

    def decode_host(self, latent_host, out_host, n_bands: int, stream=None):
        """Host buffers in, host buffers out (copies inside the call; synchronous)."""
        for name, t in (("latent_host", latent_host), ("out_host", out_host)):
            if t.is_cuda or t.dtype != self.torch_dtype or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor of dtype {self.torch_dtype}")
        oshape = self.output_shape(latent_host.shape)
        if tuple(out_host.shape) != oshape:
            raise ValueError(f"out_host has shape {tuple(out_host.shape)}, expected {oshape}")
        _check(self.lib, self.lib.vaedec_decode_host(self._h, latent_host.data_ptr(),
                                                     _shape_arg(latent_host.shape), latent_host.dim(),
                                                     out_host.data_ptr(), int(n_bands),
                                                     self._stream_ptr(stream)))
        return out_host

    def sync(self, stream=None) -> None:
        _check(self.lib, self.lib.vaedec_sync(self._h, self._stream_ptr(stream)))

    def wait_probe(self, stream=None) -> None:
        """Enqueue a kernel whose bounded wait runs out (see vaedec_debug_wait_probe)."""
        _check(self.lib, self.lib.vaedec_debug_wait_probe(self._h, self._stream_ptr(stream)))

    def launch_count(self) -> int:
        n = ctypes.c_uint64()
        _check(self.lib, self.lib.vaedec_launch_count(self._h, ctypes.byref(n)))
        return int(n.value)

    def profile(self, enable: bool) -> None:
        _check(self.lib, self.lib.vaedec_profile_enable(self._h, 1 if enable else 0))

    def profile_read(self, max_ops: int = 4096):
        """Per-op device milliseconds of the last profiled decode."""
        buf = (ctypes.c_float * max_ops)()
        n = ctypes.c_int()
        _check(self.lib, self.lib.vaedec_profile_read(self._h, buf, max_ops, ctypes.byref(n)))
        return [float(buf[i]) for i in range(min(n.value, max_ops))]

    # ------------------------------------------------------------------ inspection
    def num_ops(self, latent_shape: Sequence[int], n_bands: int) -> int:
        n = ctypes.c_int()
        _check(self.lib, self.lib.vaedec_debug_num_ops(self._h, _shape_arg(latent_shape), len(latent_shape),
                                                       int(n_bands), ctypes.byref(n)))
        return n.value

    def op_desc(self, latent_shape: Sequence[int], n_bands: int, op: int) -> Dict[str, str]:
        buf = ctypes.create_string_buffer(1024)
        _check(self.lib, self.lib.vaedec_debug_op_desc(self._h, _shape_arg(latent_shape), len(latent_shape),
                                                       int(n_bands), int(op), buf, 1024))
        return dict(kv.split("=", 1) for kv in buf.value.decode().split())

    def ops(self, latent_shape: Sequence[int], n_bands: int) -> Iterable[Dict[str, str]]:
        return [self.op_desc(latent_shape, n_bands, i) for i in range(self.num_ops(latent_shape, n_bands))]

    def run_until(self, latent, n_bands: int, op: int, dst_in=None, dst_aux=None, dst_out=None, stream=None):
        """Run ops [0, op] and copy that op's input / aux / output activations into the given device tensors."""
        if not latent.is_cuda or latent.dtype != self.torch_dtype or not latent.is_contiguous():
            raise ValueError("latent must be a contiguous CUDA tensor in the model dtype")
        if latent.device.index != self.device:
            raise ValueError(f"latent is on {latent.device}, the decoder on cuda:{self.device}")

        def ptr_size(t):
            if t is None:
                return (0, 0)
            if not t.is_cuda or t.device != latent.device or not t.is_contiguous():
                raise ValueError(f"debug buffers must be contiguous tensors on {latent.device}")
            return (t.data_ptr(), t.numel() * t.element_size())
        pi, si = ptr_size(dst_in)
        pa, sa = ptr_size(dst_aux)
        po, so = ptr_size(dst_out)
        _check(self.lib, self.lib.vaedec_debug_run_until(
            self._h, latent.data_ptr(), _shape_arg(latent.shape), latent.dim(), int(n_bands), int(op),
            pi or None, si, pa or None, sa, po or None, so, self._stream_ptr(stream)))

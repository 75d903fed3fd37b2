"""ctypes binding of ``libbwgemm.so`` (C ABI in ``include/bwgemm.h``).

Argument marshalling only: torch tensors are turned into device pointers,
element strides and the current CUDA stream, and every call goes straight to
the library, whose sm_103a kernels do all the arithmetic.  If the library
cannot be loaded the calls raise; there is no host-side fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

BF16 = 0
FP16 = 1

SCHEDULE_AUTO = 0
SCHEDULE_TILES = 1
SCHEDULE_STREAM_K = 2
SCHEDULE_CLC = 3

STATUS_NAMES = {
    0: "BWGEMM_OK",
    1: "BWGEMM_ERR_INVALID_ARG",
    2: "BWGEMM_ERR_ALIGNMENT",
    3: "BWGEMM_ERR_UNSUPPORTED",
    4: "BWGEMM_ERR_NO_DEVICE",
    5: "BWGEMM_ERR_CUDA",
    6: "BWGEMM_ERR_TIMEOUT",
    7: "BWGEMM_ERR_WORKSPACE",
}

# every symbol include/bwgemm.h declares
EXPORTED = [
    "bwgemm_default_options", "bwgemm_create_plan", "bwgemm_destroy", "bwgemm_run",
    "bwgemm_run_host", "bwgemm_get_status", "bwgemm_last_device_status", "bwgemm_check_args",
    "bwgemm_select_config", "bwgemm_plan_last_config", "bwgemm_plan_launch_count",
    "bwgemm_status_string", "bwgemm_version", "bwgemm_run_splitk_noalloc",
    "bwgemm_plan_read_trace", "bwgemm_tune", "bwgemm_plan_tuned_count",
    "bwgemm_probe_tensor_rate", "bwgemm_noalloc_scratch", "bwgemm_bench_load_path",
]

# layouts of bwgemm_bench_load_path
LOAD_PATH_LAYOUTS = {0: "128B swizzle", 1: "no swizzle, plain rows (same copies)",
                     2: "no swizzle, interleaved core matrices (8 copies per tile)",
                     3: "128B swizzle, one 256-row copy per K block",
                     4: "128B swizzle, A multicast in halves across two CTAs",
                     5: "128B swizzle, two K blocks (256-byte row pieces) per copy",
                     6: "128B swizzle, 64 KiB stages, A multicast in halves across two CTAs",
                     7: "128B swizzle, 64 KiB stages, no multicast"}

# timeline slots of bwgemm_plan_read_trace
(TRACE_ENTRY, TRACE_READY, TRACE_FIRST_LOAD, TRACE_LAST_LOAD, TRACE_EPI_DONE, TRACE_EXIT, TRACE_SETUP,
 TRACE_UNIT_KNOWN) = range(8)
TRACE_UNIT0 = 8
TRACE_UNITS = 14


class BwgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, f"status {status}")
        super().__init__(f"{what}: {name}" if what else name)


class PlanOptions(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("tile_n", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("raster_group", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32),
        ("stall_kblock", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64),
        ("workspace_bytes", ctypes.c_uint64),
        ("schedule", ctypes.c_int32),
        ("pdl_off", ctypes.c_int32),
        ("trace", ctypes.c_int32),
        ("prefetch", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32),
        ("multicast", ctypes.c_int32),
        ("copy_kblocks", ctypes.c_int32),
        ("cluster_split", ctypes.c_int32),
        ("tuned_table", ctypes.c_int32),
        ("skinny", ctypes.c_int32),
        ("wholek", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]


class Config(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("tile_m", ctypes.c_int32),
        ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("raster_group", ctypes.c_int32),
        ("num_tiles", ctypes.c_int32),
        ("num_units", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("schedule", ctypes.c_int32),
        ("dp_tiles", ctypes.c_int32),
        ("sk_tiles", ctypes.c_int32),
        ("workers", ctypes.c_int32),
        ("split_scatter", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32),
        ("multicast", ctypes.c_int32),
        ("copy_kblocks", ctypes.c_int32),
        ("prefetch_kblocks", ctypes.c_int32),
        ("prefetch_b", ctypes.c_int32),
        ("cluster_split", ctypes.c_int32),
        ("tuned", ctypes.c_int32),
        ("skinny", ctypes.c_int32),
        ("wholek", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    here = os.path.dirname(os.path.abspath(__file__))
    return os.environ.get("BWGEMM_LIBRARY", os.path.join(here, "_build", "libbwgemm.so"))


def load_library(build_if_missing: bool = False):
    """Load ``libbwgemm.so`` (building it first when asked and missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise BwgemmError(4, f"{path} not built (run __graft_entry__.build())")
            from . import build as _build
            path = _build.build()
        lib = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int32
        st = ctypes.c_int
        lib.bwgemm_default_options.argtypes = [ctypes.POINTER(PlanOptions)]
        lib.bwgemm_default_options.restype = None
        lib.bwgemm_create_plan.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.POINTER(PlanOptions)]
        lib.bwgemm_create_plan.restype = st
        lib.bwgemm_destroy.argtypes = [vp]
        lib.bwgemm_destroy.restype = st
        gemm_args = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_int, vp]
        lib.bwgemm_run.argtypes = gemm_args
        lib.bwgemm_run.restype = st
        lib.bwgemm_run_host.argtypes = gemm_args
        lib.bwgemm_run_host.restype = st
        lib.bwgemm_run_splitk_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                                  ctypes.c_int, i32, vp]
        lib.bwgemm_run_splitk_noalloc.restype = st
        lib.bwgemm_noalloc_scratch.argtypes = [i32, i32, i64, i64, i64, i32,
                                               ctypes.POINTER(ctypes.c_uint64),
                                               ctypes.POINTER(ctypes.c_uint64)]
        lib.bwgemm_noalloc_scratch.restype = st
        lib.bwgemm_get_status.argtypes = [vp, vp]
        lib.bwgemm_get_status.restype = st
        lib.bwgemm_last_device_status.argtypes = [vp]
        lib.bwgemm_last_device_status.restype = ctypes.c_uint32
        lib.bwgemm_check_args.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.bwgemm_check_args.restype = st
        lib.bwgemm_select_config.argtypes = [i32, i32, i32, i64, i64, i64, ctypes.c_int,
                                             ctypes.POINTER(PlanOptions), ctypes.POINTER(Config)]
        lib.bwgemm_select_config.restype = st
        lib.bwgemm_plan_last_config.argtypes = [vp, ctypes.POINTER(Config)]
        lib.bwgemm_plan_last_config.restype = st
        lib.bwgemm_plan_read_trace.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64), i64,
                                               ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.bwgemm_plan_read_trace.restype = st
        lib.bwgemm_plan_launch_count.argtypes = [vp]
        lib.bwgemm_plan_launch_count.restype = ctypes.c_uint64
        lib.bwgemm_tune.argtypes = gemm_args + [i32, ctypes.POINTER(Config)]
        lib.bwgemm_tune.restype = st
        lib.bwgemm_plan_tuned_count.argtypes = [vp]
        lib.bwgemm_plan_tuned_count.restype = i32
        lib.bwgemm_status_string.argtypes = [ctypes.c_int]
        lib.bwgemm_status_string.restype = ctypes.c_char_p
        lib.bwgemm_version.argtypes = []
        lib.bwgemm_version.restype = i32
        lib.bwgemm_probe_tensor_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                                 ctypes.POINTER(i32)]
        lib.bwgemm_probe_tensor_rate.restype = st
        lib.bwgemm_bench_load_path.argtypes = [ctypes.c_int, i32, i32, i32, i32, i32,
                                               ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(ctypes.c_double)]
        lib.bwgemm_bench_load_path.restype = st
        _lib = lib
        return lib


def make_options(**kw) -> PlanOptions:
    lib = load_library()
    o = PlanOptions()
    lib.bwgemm_default_options(ctypes.byref(o))
    for k, v in kw.items():
        if v is None:
            continue
        if not hasattr(o, k) or k == "reserved":
            raise TypeError(f"unknown plan option {k!r}")
        setattr(o, k, v)
    return o


_torch_mod = None
_dtype_codes: dict = {}


def _torch():
    """The torch module, imported once (the per-call path looks it up here)."""
    global _torch_mod
    if _torch_mod is None:
        import torch
        _torch_mod = torch
        _dtype_codes.update({torch.bfloat16: BF16, torch.float16: FP16})
    return _torch_mod


def _dtype_code(t) -> int:
    _torch()
    code = _dtype_codes.get(t.dtype)
    if code is None:
        raise TypeError(f"bwgemm takes bfloat16 or float16 tensors, got {t.dtype}")
    return code


def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("operands must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("operands must be K-major / row-major (unit stride along the last dim)")
    return int(t.stride(0)) if t.shape[0] > 1 else max(int(t.shape[1]), 1)


def select_config(num_sms: int, M: int, N: int, K: int, dtype: int = BF16, max_pairs: int = 0,
                  max_quads: int = 0, **opts) -> dict:
    """Host-only: the configuration a plan would choose (no GPU needed)."""
    lib = load_library()
    o = make_options(**opts)
    cfg = Config()
    rc = lib.bwgemm_select_config(num_sms, max_pairs, max_quads, M, N, K, dtype, ctypes.byref(o),
                                  ctypes.byref(cfg))
    if rc != 0:
        raise BwgemmError(rc, "bwgemm_select_config")
    return cfg.as_dict()


def probe_tensor_rate(device: int = 0):
    """(FLOP per SM clock of one SM's tensor pipe, SM count), measured on `device`
    by bwgemm_probe_tensor_rate."""
    lib = load_library()
    rate = ctypes.c_double(0.0)
    sms = ctypes.c_int32(0)
    rc = lib.bwgemm_probe_tensor_rate(int(device), ctypes.byref(rate), ctypes.byref(sms))
    if rc != 0:
        raise BwgemmError(rc, "bwgemm_probe_tensor_rate")
    return rate.value, sms.value


def bench_load_path(layout: int, source: int = 0, ctas: int = 0, stages: int = 6, kblocks: int = 4096,
                    device: int = 0):
    """(GB/s landed by all CTAs, milliseconds) of bwgemm_bench_load_path."""
    lib = load_library()
    gbs = ctypes.c_double(0.0)
    ms = ctypes.c_double(0.0)
    rc = lib.bwgemm_bench_load_path(int(device), int(layout), int(source), int(ctas), int(stages),
                                    int(kblocks), ctypes.byref(gbs), ctypes.byref(ms))
    if rc != 0:
        raise BwgemmError(rc, "bwgemm_bench_load_path")
    return gbs.value, ms.value


def check_args(A_ptr, B_ptr, C_ptr, M, N, K, lda, ldb, ldc, dtype=BF16) -> int:
    """Host-only: the status bwgemm_run would return for these arguments."""
    return int(load_library().bwgemm_check_args(A_ptr, B_ptr, C_ptr, M, N, K, lda, ldb, ldc, dtype))


class Plan:
    """A bwgemm plan on one CUDA device (see ``bwgemm_create_plan``)."""

    def __init__(self, device: int | None = None, **opts):
        import torch
        self.lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        self.options = make_options(**opts)
        h = ctypes.c_void_p()
        rc = self.lib.bwgemm_create_plan(ctypes.byref(h), self.device, ctypes.byref(self.options))
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_create_plan")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.bwgemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _check_device(self, *tensors):
        # the library refuses operands that are not memory of the plan's
        # device as well; this names the tensor
        for name, t in zip(("A", "B", "out"), tensors):
            if t.device.type != "cuda" or t.device.index != self.device:
                raise ValueError(f"{name} is on {t.device}, the plan on cuda:{self.device}")

    @staticmethod
    def _stream_handle(stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return ctypes.c_void_p(int(stream.cuda_stream))

    def run_raw(self, A_ptr: int, B_ptr: int, C_ptr: int, M: int, N: int, K: int, lda: int,
                ldb: int, ldc: int, dtype: int, stream_ptr: int | None) -> int:
        """Direct call of ``bwgemm_run`` with raw pointers; returns the status code."""
        return int(self.lib.bwgemm_run(self.handle, A_ptr, B_ptr, C_ptr, M, N, K, lda, ldb, ldc,
                                       dtype, stream_ptr))

    def gemm(self, A, B, out=None, stream=None):
        """``out = A @ B.T`` for CUDA bf16/fp16 tensors A (M x K) and B (N x K)."""
        torch = _torch()
        dt = _dtype_code(A)
        if B.dtype != A.dtype:
            raise TypeError("A and B must have the same dtype")
        dev = self.device
        # get_device(): the CUDA device index, -1 for host tensors
        if A.get_device() != dev or B.get_device() != dev:
            if not (A.is_cuda and B.is_cuda):
                raise ValueError("A and B must be CUDA tensors (bwgemm has no host path)")
            self._check_device(A, B)
        M, K = A.shape
        N, Kb = B.shape
        if Kb != K:
            raise ValueError(f"K mismatch: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
        if out is None:
            out = torch.empty((M, N), dtype=A.dtype, device=A.device)
        elif out.dtype != A.dtype or out.shape != (M, N) or out.get_device() != dev:
            if out.dtype != A.dtype or tuple(out.shape) != (M, N) or not out.is_cuda:
                raise ValueError("out must be an M x N CUDA tensor of the operands' dtype")
            self._check_device(A, B, out)
        s = (torch.cuda.current_stream(dev) if stream is None else stream).cuda_stream
        rc = self.lib.bwgemm_run(self.handle, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                                 _ld(A), _ld(B), _ld(out), dt, s)
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_run")
        return out

    def gemm_host(self, A, B, out=None, stream=None):
        """``bwgemm_run_host``: A, B, out are CPU tensors (pinned for speed)."""
        import torch
        dt = _dtype_code(A)
        M, K = A.shape
        N, _ = B.shape
        if out is None:
            out = torch.empty((M, N), dtype=A.dtype)
        rc = self.lib.bwgemm_run_host(self.handle, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N,
                                      K, _ld(A), _ld(B), _ld(out), dt, self._stream_handle(stream))
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_run_host")
        return out

    def status(self, stream=None) -> int:
        """``bwgemm_get_status``: synchronises the stream, returns and clears the status."""
        return int(self.lib.bwgemm_get_status(self.handle, self._stream_handle(stream)))

    def last_device_status(self) -> int:
        return int(self.lib.bwgemm_last_device_status(self.handle))

    def last_config(self) -> dict:
        cfg = Config()
        rc = self.lib.bwgemm_plan_last_config(self.handle, ctypes.byref(cfg))
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_plan_last_config")
        return cfg.as_dict()

    def launch_count(self) -> int:
        return int(self.lib.bwgemm_plan_launch_count(self.handle))

    def tune(self, A, B, out=None, iters: int = 10, stream=None) -> dict:
        """``bwgemm_tune``: time the candidate configurations on A, B, out and
        keep the fastest for this shape; returns its configuration.  `out`
        holds the product afterwards."""
        import torch
        dt = _dtype_code(A)
        if B.dtype != A.dtype or not (A.is_cuda and B.is_cuda):
            raise ValueError("A and B must be CUDA tensors of one dtype")
        M, K = A.shape
        N, _ = B.shape
        if out is None:
            out = torch.empty((M, N), dtype=A.dtype, device=A.device)
        self._check_device(A, B, out)
        cfg = Config()
        rc = self.lib.bwgemm_tune(self.handle, A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                                  _ld(A), _ld(B), _ld(out), dt, self._stream_handle(stream), int(iters),
                                  ctypes.byref(cfg))
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_tune")
        return cfg.as_dict()

    def tuned_count(self) -> int:
        return int(self.lib.bwgemm_plan_tuned_count(self.handle))

    def read_trace(self):
        """Timeline of the last launch (plan created with trace=1): a
        (ctas, slots) numpy uint64 array of %globaltimer stamps in ns."""
        import numpy as np
        cap = 1 << 16
        buf = (ctypes.c_uint64 * cap)()
        ctas, slots = ctypes.c_int32(), ctypes.c_int32()
        rc = self.lib.bwgemm_plan_read_trace(self.handle, buf, cap, ctypes.byref(ctas),
                                             ctypes.byref(slots))
        if rc != 0:
            raise BwgemmError(rc, "bwgemm_plan_read_trace")
        n = ctas.value * slots.value
        return np.ctypeslib.as_array(buf)[:n].copy().reshape(ctas.value, slots.value)


_plans: dict = {}


def gemm(A, B, out=None, stream=None):
    """``A @ B.T`` with a cached default plan per device."""
    dev = A.device.index if A.device.index is not None else 0
    plan = _plans.get(dev)
    if plan is None:
        plan = _plans[dev] = Plan(dev)
    return plan.gemm(A, B, out=out, stream=stream)

"""ctypes binding of libmoonep.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but check the tensors' dtype, device, size and contiguity, take their
device pointers and the current CUDA stream, and raise on a non-zero status.
All arithmetic runs in the library's CUDA kernels; there is no fallback: if
the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoonep.so")

OK = 0
ERR_ARG, ERR_ALIGN, ERR_SLOTS, ERR_SHAPE, ERR_CUDA, ERR_SCRATCH = 1, 2, 3, 4, 5, 6
ERR_ROUTING, ERR_INTERNAL, ERR_TIMEOUT = 0x100, 0x200, 0x400
CNT_FILLS, CNT_MTILES, CNT_OCCUPIED, CNT_REDUCE = 0, 1, 2, 3
CNT_REMOTE_ENTRIES, CNT_REMOTE_PAIRS, CNT_GROUPS = 4, 5, 6
GEMM_SCRATCH_BYTES = 512 << 10  # MOONEP_GEMM_SCRATCH_BYTES: the workspace's last bytes


class MoonepError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status:#x} ({status_string(status)})")


class moonep_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("R", "E", "B", "K", "S", "H", "Hp", "mode", "policy",
                                               "gemm_rows")]

    @property
    def L(self):
        return self.E // self.R

    @property
    def C(self):
        return self.S * self.K

    @property
    def N(self):
        return self.R * self.S * self.K


_SIZE_FIELDS = ("total_bytes", "status", "counters", "counts", "T", "load", "keep", "gidx",
                "fills", "slot_expert", "n_recv", "src", "cu_seqlens", "dst", "inverse",
                "pieces", "occupied", "reduce", "mtiles")
_LAYOUT_FIELDS = _SIZE_FIELDS + ("route", "groups")  # total size, then every table offset


class moonep_plan_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _SIZE_FIELDS] + [
        ("nchunk", ctypes.c_int32), ("max_mtiles", ctypes.c_int32), ("route", ctypes.c_size_t),
        ("groups", ctypes.c_size_t)]


class moonep_plan_view(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("cu_seqlens", "dst", "inverse", "slot_expert",
                                                 "status")]


_lib = None


def library() -> ctypes.CDLL:
    """Load libmoonep.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoonep.so not built ({LIB_PATH}); run "
                          "perfectly_balanced_token_gb300.build.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P, D = ctypes.c_void_p, ctypes.POINTER(moonep_dims)
    sig = {
        "moonep_plan_workspace_bytes": [D, ctypes.POINTER(ctypes.c_size_t)],
        "moonep_get_plan_layout": [D, ctypes.POINTER(moonep_plan_layout)],
        "moonep_plan_views": [D, P, ctypes.POINTER(moonep_plan_view)],
        "moonep_plan": [D, P, P, P],
        "moonep_prefetch_weights": [D, P, P, P, P],
        "moonep_dispatch": [D, P, P, P, P],
        "moonep_dispatch_send_once": [D, P, P, P, P, P, P],
        "moonep_grouped_gemm": [D, P, P, P, P, P, P],
        "moonep_combine": [D, P, P, P, P, P],
        "moonep_reduce_grad": [D, P, P, P, P],
        "moonep_read_status": [D, P, ctypes.POINTER(ctypes.c_int32), P],
        "moonep_plan_export": [D, P, P, P],
        "moonep_plan_noalloc": [D, P, P, P],
        "moonep_combine_backward": [D, P, P, P, P, P, P, P],
        "moonep_grouped_gemm_dx": [D, P, P, P, P, P, P],
        "moonep_grouped_gemm_dw": [D, P, P, P, P, P, P],
        "moonep_dispatch_backward": [D, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.moonep_status_string.argtypes = [ctypes.c_int]
    lib.moonep_status_string.restype = ctypes.c_char_p
    lib.moonep_selftest_bounded_wait.argtypes = [P, ctypes.c_uint32, P, P]
    lib.moonep_selftest_bounded_wait.restype = ctypes.c_int
    lib.moonep_launch_count.argtypes = []
    lib.moonep_launch_count.restype = ctypes.c_uint64
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return library().moonep_status_string(int(status)).decode()
    except ImportError:
        return "library not loaded"


def dims(R, E, B, K, S, H, Hp, mode=0, policy=0, gemm_rows=0) -> moonep_dims:
    """gemm_rows: 0 lets each plan choose the GEMM work-tile height; 128 or 256 fixes it."""
    return moonep_dims(R, E, B, K, S, H, Hp, mode, policy, gemm_rows)


def _check(rc: int, what: str):
    if rc != OK:
        raise MoonepError(rc, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype, numel, name, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return ctypes.c_void_p(t.data_ptr())


def moonep_plan_workspace_bytes(d: moonep_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(library().moonep_plan_workspace_bytes(ctypes.byref(d), ctypes.byref(n)),
           "moonep_plan_workspace_bytes")
    return n.value


def moonep_get_plan_layout(d: moonep_dims) -> moonep_plan_layout:
    out = moonep_plan_layout()
    _check(library().moonep_get_plan_layout(ctypes.byref(d), ctypes.byref(out)),
           "moonep_get_plan_layout")
    return out


def moonep_plan_views(d: moonep_dims, plan_ws) -> dict:
    """Device addresses of cu_seqlens, dst, inverse, slot_expert and the status
    word inside plan_ws (a CUDA uint8 tensor of the workspace size, or its
    device address as an int); host only."""
    addr = plan_ws if isinstance(plan_ws, int) else _ws(d, plan_ws)
    out = moonep_plan_view()
    _check(library().moonep_plan_views(ctypes.byref(d), addr, ctypes.byref(out)),
           "moonep_plan_views")
    return {n: getattr(out, n) for n, _ in moonep_plan_view._fields_}


def _ws(d, ws):
    return _ptr(ws, torch.uint8, moonep_plan_workspace_bytes(d), "plan_ws")


def moonep_plan(d, topk_idx, plan_ws, stream=None):
    _check(library().moonep_plan(ctypes.byref(d), _ptr(topk_idx, torch.int32, d.N, "topk_idx"),
                                 _ws(d, plan_ws), _stream(stream)), "moonep_plan")


def moonep_plan_noalloc(d, topk_idx, plan_ws, stream=None):
    """moonep_plan with the planner's scratch in the library's static device
    array (nothing allocated); same outputs in plan_ws."""
    _check(library().moonep_plan_noalloc(ctypes.byref(d),
                                         _ptr(topk_idx, torch.int32, d.N, "topk_idx"),
                                         _ws(d, plan_ws), _stream(stream)), "moonep_plan_noalloc")


def moonep_prefetch_weights(d, plan_ws, w_home, w_slot, stream=None):
    hh = d.H * d.Hp
    _check(library().moonep_prefetch_weights(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(w_home, torch.bfloat16, d.E * hh, "w_home"),
        _ptr(w_slot, torch.bfloat16, d.R * d.B * hh, "w_slot", allow_none=d.B == 0),
        _stream(stream)), "moonep_prefetch_weights")


def moonep_dispatch(d, plan_ws, x, recv, stream=None):
    _check(library().moonep_dispatch(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(x, torch.bfloat16, d.R * d.S * d.H, "x"),
        _ptr(recv, torch.bfloat16, d.N * d.H, "recv"), _stream(stream)), "moonep_dispatch")


def moonep_dispatch_send_once(d, plan_ws, x, gates, recv, recv_weight, stream=None):
    _check(library().moonep_dispatch_send_once(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(x, torch.bfloat16, d.R * d.S * d.H, "x"),
        _ptr(gates, torch.float32, d.N, "gates"), _ptr(recv, torch.bfloat16, d.N * d.H, "recv"),
        _ptr(recv_weight, torch.float32, d.N, "recv_weight"), _stream(stream)),
        "moonep_dispatch_send_once")


def moonep_grouped_gemm(d, plan_ws, recv, w_home, w_slot, y, stream=None):
    hh = d.H * d.Hp
    _check(library().moonep_grouped_gemm(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(recv, torch.bfloat16, d.N * d.H, "recv"),
        _ptr(w_home, torch.bfloat16, d.E * hh, "w_home"),
        _ptr(w_slot, torch.bfloat16, d.R * d.B * hh, "w_slot", allow_none=d.B == 0),
        _ptr(y, torch.bfloat16, d.N * d.Hp, "y"), _stream(stream)), "moonep_grouped_gemm")


def moonep_combine(d, plan_ws, y, gates, out, stream=None):
    _check(library().moonep_combine(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(y, torch.bfloat16, d.N * d.Hp, "y"),
        _ptr(gates, torch.float32, d.N, "gates"),
        _ptr(out, torch.bfloat16, d.R * d.S * d.Hp, "out"), _stream(stream)), "moonep_combine")


def moonep_reduce_grad(d, plan_ws, g_home, g_slot, stream=None):
    hh = d.H * d.Hp
    _check(library().moonep_reduce_grad(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(g_home, torch.float32, d.E * hh, "g_home"),
        _ptr(g_slot, torch.float32, d.R * d.B * hh, "g_slot", allow_none=d.B == 0),
        _stream(stream)), "moonep_reduce_grad")


def moonep_combine_backward(d, plan_ws, y, gates, d_out, d_y, d_gates, stream=None):
    _check(library().moonep_combine_backward(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(y, torch.bfloat16, d.N * d.Hp, "y"),
        _ptr(gates, torch.float32, d.N, "gates"),
        _ptr(d_out, torch.bfloat16, d.R * d.S * d.Hp, "d_out"),
        _ptr(d_y, torch.bfloat16, d.N * d.Hp, "d_y"), _ptr(d_gates, torch.float32, d.N, "d_gates"),
        _stream(stream)), "moonep_combine_backward")


def moonep_grouped_gemm_dx(d, plan_ws, d_y, w_home, w_slot, d_recv, stream=None):
    hh = d.H * d.Hp
    _check(library().moonep_grouped_gemm_dx(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(d_y, torch.bfloat16, d.N * d.Hp, "d_y"),
        _ptr(w_home, torch.bfloat16, d.E * hh, "w_home"),
        _ptr(w_slot, torch.bfloat16, d.R * d.B * hh, "w_slot", allow_none=d.B == 0),
        _ptr(d_recv, torch.bfloat16, d.N * d.H, "d_recv"), _stream(stream)), "moonep_grouped_gemm_dx")


def moonep_grouped_gemm_dw(d, plan_ws, recv, d_y, g_home, g_slot, stream=None):
    hh = d.H * d.Hp
    _check(library().moonep_grouped_gemm_dw(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(recv, torch.bfloat16, d.N * d.H, "recv"),
        _ptr(d_y, torch.bfloat16, d.N * d.Hp, "d_y"),
        _ptr(g_home, torch.float32, d.E * hh, "g_home"),
        _ptr(g_slot, torch.float32, d.R * d.B * hh, "g_slot", allow_none=d.B == 0),
        _stream(stream)), "moonep_grouped_gemm_dw")


def moonep_dispatch_backward(d, plan_ws, d_recv, d_x, stream=None):
    _check(library().moonep_dispatch_backward(
        ctypes.byref(d), _ws(d, plan_ws), _ptr(d_recv, torch.bfloat16, d.N * d.H, "d_recv"),
        _ptr(d_x, torch.bfloat16, d.R * d.S * d.H, "d_x"), _stream(stream)),
        "moonep_dispatch_backward")


def moonep_read_status(d, plan_ws, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(library().moonep_read_status(ctypes.byref(d), _ws(d, plan_ws), ctypes.byref(st),
                                        _stream(stream)), "moonep_read_status")
    return st.value


def moonep_selftest_bounded_wait(dev_status, limit_us: int, dev_elapsed_us, stream=None):
    _check(library().moonep_selftest_bounded_wait(
        _ptr(dev_status, torch.int32, 1, "dev_status"), ctypes.c_uint32(limit_us),
        _ptr(dev_elapsed_us, torch.int32, 1, "dev_elapsed_us"), _stream(stream)),
        "moonep_selftest_bounded_wait")


def moonep_launch_count() -> int:
    return int(library().moonep_launch_count())


class PlanWorkspace:
    """A device workspace for one set of dims, with typed views of its tables."""

    def __init__(self, d: moonep_dims, device="cuda"):
        self.dims = d
        self.layout = moonep_get_plan_layout(d)
        self.buf = torch.zeros(self.layout.total_bytes, dtype=torch.uint8, device=device)

    def view(self, name: str, shape) -> torch.Tensor:
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        return self.buf[off:off + 4 * n].view(torch.int32).view(*shape)

    def tables(self) -> dict:
        """Host copies of the plan tables (synchronises)."""
        d = self.dims
        v = {
            "status": self.view("status", (1,)),
            "counters": self.view("counters", (8,)),
            "T": self.view("T", (d.E,)),
            "load": self.view("load", (d.R,)),
            "keep": self.view("keep", (d.E,)),
            "gidx": self.view("gidx", (d.R, d.S, d.K)),
            "fills": self.view("fills", (max(d.R - 1, 1), 3)),
            "slot_expert": self.view("slot_expert", (d.R, d.B)),
            "n_recv": self.view("n_recv", (d.R,)),
            "src": self.view("src", (d.R,)),
            "cu_seqlens": self.view("cu_seqlens", (d.R, d.E + d.B + 1)),
            "dst": self.view("dst", (d.R, d.S, d.K)),
            "inverse": self.view("inverse", (d.N,)),
            "route": self.view("route", (d.R, d.S, d.K)),
        }
        return {k: t.cpu().numpy() for k, t in v.items()}

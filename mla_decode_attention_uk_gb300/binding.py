"""ctypes binding of libmla_decode.so: argument marshalling only.

Every function here forwards to the C ABI in include/mla_decode.h with device
pointers taken from torch tensors and the current torch CUDA stream.  There is
no fallback: if the shared library cannot be loaded, importing the binding
raises.
"""
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL", 4: "CUDA_ERROR",
          5: "DEVICE_BOUNDS", 6: "TIMEOUT"}

ENTRY_POINTS = (
    "mla_decode_workspace_size", "mla_decode_workspace_size_ex", "mla_decode_plan",
    "mla_decode_plan_ex", "mla_decode_run", "mla_decode_absorb", "mla_decode_attend",
    "mla_decode_combine", "mla_decode_up_project", "mla_decode_check", "mla_decode_status_string",
    "mla_decode_workspace_offsets", "mla_decode_kernels_per_run",
    "mla_decode_run_static_scratch", "mla_decode_selftest_wait_timeout",
    "mla_decode_run_fp8w", "mla_decode_absorb_fp8w", "mla_decode_up_project_fp8w")


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "q_len", "num_heads", "qk_nope", "qk_rope", "kv_lora", "v_head", "page_size",
        "num_pages", "max_pages_per_seq")]


class MlaDecodeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s (%d) %s" % (where, STATUS.get(code, "?"), code,
                                                   lib().mla_decode_status_string(code).decode()))


_lib = None


def lib():
    """Load (building first if sources are newer) the CUDA library; raises if unavailable."""
    global _lib
    if _lib is None:
        if not _build.up_to_date():
            _build.build()
        L = ctypes.CDLL(LIB_PATH)
        P, D, S = ctypes.c_void_p, ctypes.POINTER(Dims), ctypes.c_size_t
        sz = ctypes.POINTER(ctypes.c_size_t)
        i32 = ctypes.c_int32
        L.mla_decode_workspace_size.argtypes = [D, sz]
        L.mla_decode_workspace_size_ex.argtypes = [D, i32, sz]
        L.mla_decode_plan.argtypes = [D, P, P, S, P]
        L.mla_decode_plan_ex.argtypes = [D, P, i32, P, S, P]
        L.mla_decode_run.argtypes = [D, P, P, P, P, P, P, ctypes.c_float, P, P, P, S, P]
        L.mla_decode_absorb.argtypes = [D, P, P, P, S, P]
        L.mla_decode_attend.argtypes = [D, P, P, P, ctypes.c_float, P, P, S, P]
        L.mla_decode_combine.argtypes = [D, ctypes.c_float, P, P, S, P]
        L.mla_decode_up_project.argtypes = [D, P, P, P, S, P]
        L.mla_decode_check.argtypes = [P, P]
        L.mla_decode_status_string.argtypes = [ctypes.c_int]
        L.mla_decode_status_string.restype = ctypes.c_char_p
        L.mla_decode_workspace_offsets.argtypes = [D, i32, ctypes.POINTER(ctypes.c_int64), i32]
        L.mla_decode_run_static_scratch.argtypes = [D, P, P, P, P, P, P, ctypes.c_float, P, P, P]
        L.mla_decode_selftest_wait_timeout.argtypes = [P, P]
        L.mla_decode_kernels_per_run.argtypes = [D, i32, ctypes.POINTER(ctypes.c_int32)]
        L.mla_decode_run_fp8w.argtypes = [D, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, S, P]
        L.mla_decode_absorb_fp8w.argtypes = [D, P, P, P, P, S, P]
        L.mla_decode_up_project_fp8w.argtypes = [D, P, P, P, P, S, P]
        for n in ENTRY_POINTS:
            if n != "mla_decode_status_string":
                getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def dims_for(q, cache, block_table) -> Dims:
    B, T, H, dq = q.shape
    return Dims(B, T, H, 128, dq - 128, cache.shape[2] - (dq - 128), 128, cache.shape[1],
                cache.shape[0], block_table.shape[1])


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(code, where):
    if code != 0:
        raise MlaDecodeError(code, where)


def workspace_size(d: Dims, num_ranges: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _ok(lib().mla_decode_workspace_size_ex(ctypes.byref(d), num_ranges, ctypes.byref(n)),
        "mla_decode_workspace_size_ex")
    return n.value


def workspace_offsets(d: Dims, num_ranges: int = 0):
    arr = (ctypes.c_int64 * 4)()
    _ok(lib().mla_decode_workspace_offsets(ctypes.byref(d), num_ranges, arr, 4),
        "mla_decode_workspace_offsets")
    return dict(qlat=arr[0], qlo=arr[1], olat=arr[2], header=arr[3])


def kernels_per_run(d: Dims, fp8_weights: bool = False) -> int:
    """Kernels one whole run enqueues on the current device (plan not counted)."""
    n = ctypes.c_int32(0)
    _ok(lib().mla_decode_kernels_per_run(ctypes.byref(d), int(fp8_weights), ctypes.byref(n)),
        "mla_decode_kernels_per_run")
    return n.value


class MlaDecode:
    """Owns a device workspace for one set of dims; plan() once per decode step,
    run() once per layer.  All tensors must be CUDA, contiguous."""

    def __init__(self, d: Dims, device=None, num_ranges: int = 0):
        self.dims = d
        self.num_ranges = num_ranges
        self.ws_bytes = workspace_size(d, num_ranges)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8,
                                     device=device or torch.device("cuda"))

    def plan(self, seq_lens):
        _ok(lib().mla_decode_plan_ex(ctypes.byref(self.dims), _ptr(seq_lens), self.num_ranges,
                                     _ptr(self.workspace), self.ws_bytes, _stream()),
            "mla_decode_plan_ex")

    def run(self, q, cache, block_table, seq_lens, w_uk, w_uv, scale, out, lse):
        _ok(lib().mla_decode_run(ctypes.byref(self.dims), _ptr(q), _ptr(cache), _ptr(block_table),
                                 _ptr(seq_lens), _ptr(w_uk), _ptr(w_uv), float(scale), _ptr(out),
                                 _ptr(lse), _ptr(self.workspace), self.ws_bytes, _stream()),
            "mla_decode_run")

    def run_fp8w(self, q, cache, block_table, seq_lens, w_uk8, w_uk_scale, w_uv8, w_uv_scale,
                 scale, out, lse):
        _ok(lib().mla_decode_run_fp8w(ctypes.byref(self.dims), _ptr(q), _ptr(cache),
                                      _ptr(block_table), _ptr(seq_lens), _ptr(w_uk8),
                                      _ptr(w_uk_scale), _ptr(w_uv8), _ptr(w_uv_scale),
                                      float(scale), _ptr(out), _ptr(lse), _ptr(self.workspace),
                                      self.ws_bytes, _stream()),
            "mla_decode_run_fp8w")

    def absorb_fp8w(self, q, w_uk8, w_uk_scale):
        _ok(lib().mla_decode_absorb_fp8w(ctypes.byref(self.dims), _ptr(q), _ptr(w_uk8),
                                         _ptr(w_uk_scale), _ptr(self.workspace), self.ws_bytes,
                                         _stream()),
            "mla_decode_absorb_fp8w")

    def up_project_fp8w(self, w_uv8, w_uv_scale, out):
        _ok(lib().mla_decode_up_project_fp8w(ctypes.byref(self.dims), _ptr(w_uv8),
                                             _ptr(w_uv_scale), _ptr(out), _ptr(self.workspace),
                                             self.ws_bytes, _stream()),
            "mla_decode_up_project_fp8w")

    def absorb(self, q, w_uk):
        _ok(lib().mla_decode_absorb(ctypes.byref(self.dims), _ptr(q), _ptr(w_uk),
                                    _ptr(self.workspace), self.ws_bytes, _stream()),
            "mla_decode_absorb")

    def attend(self, cache, block_table, seq_lens, scale, lse):
        _ok(lib().mla_decode_attend(ctypes.byref(self.dims), _ptr(cache), _ptr(block_table),
                                    _ptr(seq_lens), float(scale), _ptr(lse), _ptr(self.workspace),
                                    self.ws_bytes, _stream()),
            "mla_decode_attend")

    def combine(self, scale, lse):
        _ok(lib().mla_decode_combine(ctypes.byref(self.dims), float(scale), _ptr(lse),
                                     _ptr(self.workspace), self.ws_bytes, _stream()),
            "mla_decode_combine")

    def up_project(self, w_uv, out):
        _ok(lib().mla_decode_up_project(ctypes.byref(self.dims), _ptr(w_uv), _ptr(out),
                                        _ptr(self.workspace), self.ws_bytes, _stream()),
            "mla_decode_up_project")

    def check(self) -> int:
        """Synchronise the stream; return the device status code (0 = OK)."""
        return lib().mla_decode_check(_ptr(self.workspace), _stream())

    # -- views of intermediates (tests / profiling)
    def _view(self, key, cols, dtype=torch.bfloat16):
        off = workspace_offsets(self.dims, self.num_ranges)[key]
        rows = self.dims.batch * self.dims.q_len * self.dims.num_heads
        n = rows * cols * torch.empty(0, dtype=dtype).element_size()
        return self.workspace[off:off + n].view(dtype).view(rows, cols)

    def q_lat(self):
        return self._view("qlat", 576)

    def q_lo(self):
        """The residual q_lat - bf16(q_lat), times 2^10, as raw E4M3 bytes."""
        return self._view("qlo", 512, torch.uint8)

    def o_lat(self):
        return self._view("olat", 512)

    def plan_header(self):
        off = workspace_offsets(self.dims, self.num_ranges)["header"]
        return self.workspace[off:off + 16].view(torch.int32).tolist()


def decode(q, cache, block_table, seq_lens, w_uk, w_uv, scale, num_ranges: int = 0):
    """One-shot convenience: plan + run, returns (out bf16 [B,T,H,128], lse fp32 [B,T,H])."""
    d = dims_for(q, cache, block_table)
    m = MlaDecode(d, q.device, num_ranges)
    out = torch.empty(q.shape[0], q.shape[1], q.shape[2], 128, dtype=torch.bfloat16,
                      device=q.device)
    lse = torch.empty(q.shape[0], q.shape[1], q.shape[2], dtype=torch.float32, device=q.device)
    m.plan(seq_lens)
    m.run(q, cache, block_table, seq_lens, w_uk, w_uv, scale, out, lse)
    return out, lse

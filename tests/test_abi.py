"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point declared in include/mla_decode.h, and rejects bad arguments
before touching the device."""
import ctypes
import math
import os
import re

import pytest

from mla_decode_attention_uk_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int)\s+(mla_decode_\w+)\s*\(", src,
                                 flags=re.M)))


def test_header_declares_the_boundary():
    fns = declared_functions()
    for must in ("mla_decode_workspace_size", "mla_decode_plan", "mla_decode_run",
                 "mla_decode_check", "mla_decode_status_string"):
        assert must in fns


def test_library_exports_every_declared_symbol():
    L = binding.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(binding.ENTRY_POINTS)


def test_library_links_no_torch_and_no_cuda_driver_at_load():
    # dlopen works on a machine without a GPU driver: the runtime is static and
    # the driver is resolved lazily.
    with open(binding.LIB_PATH, "rb") as f:
        head = f.read()
    assert b"libtorch" not in head and b"libc10" not in head


def test_status_strings():
    L = binding.lib()
    for code in range(7):
        s = L.mla_decode_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.mla_decode_status_string(99).decode() == "unknown status"
    # Bad dims or a null count fail before any device query (no GPU here).
    n = ctypes.c_int32(-1)
    assert L.mla_decode_kernels_per_run(None, 0, ctypes.byref(n)) == 1
    assert L.mla_decode_kernels_per_run(ctypes.byref(good_dims()), 0, None) == 1
    assert n.value == -1


def good_dims(**kw):
    d = dict(batch=2, q_len=1, num_heads=16, qk_nope=128, qk_rope=64, kv_lora=512, v_head=128,
             page_size=64, num_pages=4, max_pages_per_seq=2)
    d.update(kw)
    return binding.Dims(**d)


@pytest.mark.parametrize("field,value,code", [
    ("qk_nope", 64, 2), ("qk_rope", 32, 2), ("kv_lora", 256, 2), ("v_head", 64, 2),
    ("page_size", 16, 2), ("q_len", 9, 2), ("q_len", 0, 2), ("num_heads", 8, 2),
    ("num_heads", 24, 2), ("num_heads", 256, 2), ("batch", 0, 1), ("num_pages", 0, 1),
    ("max_pages_per_seq", 0, 1),
])
def test_bad_dims_rejected_on_host(field, value, code):
    L = binding.lib()
    n = ctypes.c_size_t(0)
    d = good_dims(**{field: value})
    assert L.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code
    assert L.mla_decode_plan(ctypes.byref(d), None, None, 0, None) == code


def test_null_pointers_rejected_before_any_launch():
    L = binding.lib()
    d = good_dims()
    fake = ctypes.c_void_p(4096)
    assert L.mla_decode_workspace_size(None, None) == 1
    assert L.mla_decode_workspace_size(ctypes.byref(d), None) == 1
    assert L.mla_decode_plan(ctypes.byref(d), None, fake, 1 << 20, None) == 1
    assert L.mla_decode_plan(ctypes.byref(d), fake, None, 1 << 20, None) == 1
    assert L.mla_decode_run(ctypes.byref(d), None, fake, fake, fake, fake, fake,
                            ctypes.c_float(0.07), fake, fake, fake, 1 << 20, None) == 1
    assert L.mla_decode_absorb(ctypes.byref(d), fake, None, fake, 1 << 20, None) == 1
    assert L.mla_decode_attend(ctypes.byref(d), fake, None, fake, ctypes.c_float(0.07), fake,
                               fake, 1 << 20, None) == 1
    assert L.mla_decode_combine(ctypes.byref(d), ctypes.c_float(0.07), None, fake, 1 << 20,
                                None) == 1
    assert L.mla_decode_up_project(ctypes.byref(d), fake, None, fake, 1 << 20, None) == 1
    assert L.mla_decode_check(None, None) == 1
    assert L.mla_decode_selftest_wait_timeout(None, None) == 1
    assert L.mla_decode_selftest_wait_timeout(ctypes.c_void_p(4098), None) == 1


def test_misaligned_pointers_rejected():
    L = binding.lib()
    d = good_dims()
    ok, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 2)
    assert L.mla_decode_absorb(ctypes.byref(d), bad, ok, ok, 1 << 30, None) == 1
    assert L.mla_decode_absorb(ctypes.byref(d), ok, ok, bad, 1 << 30, None) == 1
    assert L.mla_decode_up_project(ctypes.byref(d), ok, bad, ok, 1 << 30, None) == 1


def test_workspace_too_small_rejected_before_launch():
    L = binding.lib()
    d = good_dims()
    ok = ctypes.c_void_p(4096)
    assert L.mla_decode_absorb(ctypes.byref(d), ok, ok, ok, 64, None) == 3
    assert L.mla_decode_combine(ctypes.byref(d), ctypes.c_float(0.07), ok, ok, 64, None) == 3


def test_run_checks_every_argument_before_the_first_launch():
    # A bad argument of a late step (the up-projection's weight, an output)
    # must be reported before the absorb step is enqueued.  Without a GPU an
    # enqueue attempt fails with CUDA_ERROR (4), so INVALID_ARG (1) shows that
    # the check came first.
    L = binding.lib()
    d = good_dims()
    ok, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 2)
    sc = ctypes.c_float(0.07)
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ok, ok, None, sc, ok, ok, ok,
                            1 << 30, None) == 1
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ok, ok, bad, sc, ok, ok, ok,
                            1 << 30, None) == 1
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ok, ok, ok, sc, bad, ok, ok,
                            1 << 30, None) == 1
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ctypes.c_void_p(4097), ok, ok, sc, ok,
                            ok, ok, 1 << 30, None) == 1
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ok, ok, ok, sc, ok, ok, ok, 64,
                            None) == 3
    # FP8 weights: codes and both block-scale arrays.
    args = [ok, ok, ok, ok, ok, ok, ok, ok, sc, ok, ok, ok]
    for i, v in ((6, None), (7, None), (7, ctypes.c_void_p(4097)), (6, bad)):
        a = list(args)
        a[i] = v
        assert L.mla_decode_run_fp8w(ctypes.byref(d), *a, 1 << 30, None) == 1, i


def test_fp8_step_calls_check_their_scales():
    L = binding.lib()
    d = good_dims()
    ok = ctypes.c_void_p(4096)
    assert L.mla_decode_absorb_fp8w(ctypes.byref(d), ok, ok, None, ok, 1 << 30, None) == 1
    assert L.mla_decode_absorb_fp8w(ctypes.byref(d), ok, None, ok, ok, 1 << 30, None) == 1
    assert L.mla_decode_up_project_fp8w(ctypes.byref(d), ok, ctypes.c_void_p(4098), ok, ok,
                                        1 << 30, None) == 1
    assert L.mla_decode_up_project_fp8w(ctypes.byref(d), ok, ok, ok, ok, 64, None) == 3



@pytest.mark.parametrize("B,T,H,R", [(2, 1, 16, 5), (64, 1, 16, 152), (256, 2, 128, 38),
                                     (64, 8, 128, 9), (5000, 1, 16, 152), (1, 1, 48, 1)])
def test_workspace_layout_holds_the_documented_buffers(B, T, H, R):
    # With an explicit range count the sizing needs no device.  The header
    # documents q_lat bf16 [B*T*H, 576], q_lo E4M3 bytes [B*T*H, 512] and
    # o_lat bf16 [B*T*H, 512];
    # the split partials (two slots per range: fp32 lse [T*H] and bf16 o
    # [T*H, 512] each) come after them.
    L = binding.lib()
    d = good_dims(batch=B, q_len=T, num_heads=H)
    n = ctypes.c_size_t(0)
    assert L.mla_decode_workspace_size_ex(ctypes.byref(d), R, ctypes.byref(n)) == 0
    off = (ctypes.c_int64 * 4)()
    assert L.mla_decode_workspace_offsets(ctypes.byref(d), R, off, 4) == 0
    q_lat, q_lo, o_lat, header = off
    rows = B * T * H
    assert all(o % 16 == 0 for o in off)
    assert header + 16 <= q_lat  # plan header (four int32) before the buffers
    assert q_lat + rows * 576 * 2 <= q_lo
    assert q_lo + rows * 512 <= o_lat
    partials = 2 * R * T * H * (512 * 2 + 4)
    assert o_lat + rows * 512 * 2 + partials <= n.value
    # Each extra range adds two partial slots (and its range bounds): at least
    # the two bf16 [T*H, 512] outputs; the small arrays may fit in the 256-byte
    # rounding of their regions.
    n2 = ctypes.c_size_t(0)
    assert L.mla_decode_workspace_size_ex(ctypes.byref(d), R + 1, ctypes.byref(n2)) == 0
    grow = n2.value - n.value
    assert 2 * T * H * 512 * 2 <= grow <= 2 * T * H * (512 * 2 + 4) + 4 * 256
    # Without a device the default range count cannot be known.
    assert L.mla_decode_workspace_size_ex(ctypes.byref(d), -1, ctypes.byref(n2)) == 1
    assert L.mla_decode_workspace_size_ex(ctypes.byref(d), 65537, ctypes.byref(n2)) == 1


BAD_SCALES = [0.0, -0.07, float("nan"), float("inf"), -float("inf"), -0.0]


@pytest.mark.parametrize("scale", BAD_SCALES)
def test_softmax_scale_must_be_finite_and_positive(scale):
    # The attention step takes its running maximum over unscaled scores, which
    # is the maximum of the scaled ones only for a positive scale: every call
    # that takes the scale rejects the others on the host, before any launch
    # (without a GPU an enqueue attempt would return CUDA_ERROR instead).
    L = binding.lib()
    d = good_dims()
    ok = ctypes.c_void_p(4096)
    sc = ctypes.c_float(scale)
    assert L.mla_decode_run(ctypes.byref(d), ok, ok, ok, ok, ok, ok, sc, ok, ok, ok,
                            1 << 30, None) == 1
    assert L.mla_decode_run_fp8w(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, ok, sc, ok, ok,
                                 ok, 1 << 30, None) == 1
    assert L.mla_decode_attend(ctypes.byref(d), ok, ok, ok, sc, ok, ok, 1 << 30, None) == 1
    assert L.mla_decode_combine(ctypes.byref(d), sc, ok, ok, 1 << 30, None) == 1
    assert L.mla_decode_run_static_scratch(ctypes.byref(d), ok, ok, ok, ok, ok, ok, sc, ok, ok,
                                           None) == 1


def test_smallest_positive_scale_passes_the_check():
    # A tiny but positive, finite scale is valid: the call gets past the
    # argument check (and, without a GPU, fails only when it reaches the device).
    L = binding.lib()
    d = good_dims()
    ok = ctypes.c_void_p(4096)
    sc = ctypes.c_float(math.ldexp(1.0, -149))
    assert L.mla_decode_combine(ctypes.byref(d), sc, ok, ok, 64, None) == 3


def test_static_scratch_checks_every_argument_before_anything_else():
    # The workspace-free call rejects bad arguments before it sizes its scratch
    # or enqueues the planner on the shared array.  Without a GPU, sizing would
    # return CUDA_ERROR (4): INVALID_ARG / UNSUPPORTED show the check ran first.
    L = binding.lib()
    d = good_dims()
    ok, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 2)
    sc = ctypes.c_float(0.07)
    args = [ok, ok, ok, ok, ok, ok, sc, ok, ok]
    for i, v in ((0, None), (0, bad), (1, bad), (2, ctypes.c_void_p(4097)), (3, None),
                 (4, bad), (5, None), (7, bad), (8, ctypes.c_void_p(4098))):
        a = list(args)
        a[i] = v
        assert L.mla_decode_run_static_scratch(ctypes.byref(d), *a, None) == 1, i
    bad_dims = good_dims(kv_lora=256)
    assert L.mla_decode_run_static_scratch(ctypes.byref(bad_dims), *args, None) == 2
    assert L.mla_decode_run_static_scratch(None, *args, None) == 1

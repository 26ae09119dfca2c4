"""fp64 CPU oracle for weight-absorbed MLA decode (TEST INFRASTRUCTURE).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The computation is the plain definition of MLA decode attention without
materialised absorbed weights (vLLM PR #14770 "[Attention] MLA get rid of
materialization", PR description): q_nope is mapped into latent space with
W_UK, every head attends to the shared paged latent cache, and the latent
output is mapped back with W_UV.  See mla_oracle.c for the step list.

Inputs are torch CPU tensors in bf16 (q, cache, w_uk, w_uv) and int32
(block_table, seq_lens); bf16 values are widened to fp64 exactly in C.
"""
import ctypes
import math

import numpy as np
import torch

from . import build as _build

_lib = None


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "q_len", "num_heads", "qk_nope", "qk_rope", "kv_lora", "v_head",
        "page_size", "num_pages", "max_pages_per_seq")]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        L.mla_oracle_decode.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, P, ctypes.c_double,
                                        ctypes.c_int64, P, P, P, P]
        L.mla_oracle_partial.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, ctypes.c_double,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, P, P]
        L.mla_oracle_combine.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P]
        L.mla_oracle_up_project.argtypes = [ctypes.POINTER(Dims), P, ctypes.c_int, P, P]
        L.mla_oracle_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def threads() -> int:
    return lib().mla_oracle_threads()


def _bits(x: torch.Tensor) -> torch.Tensor:
    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return x.contiguous().view(torch.int16)


def _i32(x: torch.Tensor) -> torch.Tensor:
    assert x.dtype == torch.int32 and x.device.type == "cpu"
    return x.contiguous()


def dims_of(q, cache, block_table, w_uk, w_uv) -> Dims:
    B, T, H, dq = q.shape
    num_pages, page, dc = cache.shape
    nope, lora = w_uk.shape[1], w_uk.shape[2]
    return Dims(B, T, H, nope, dq - nope, lora, w_uv.shape[2], page, num_pages,
                block_table.shape[1])


def decode(q, cache, block_table, seq_lens, w_uk, w_uv, scale, rows=None, want_olat=False):
    """Run the oracle.  Returns (out [n, v], lse [n], o_lat [n, lora] or None) in fp64,
    n = B*T*H (row order (b, t, h)) or len(rows) for a selection of flat row ids."""
    d = dims_of(q, cache, block_table, w_uk, w_uv)
    qb, cb, wk, wv = _bits(q), _bits(cache), _bits(w_uk), _bits(w_uv)
    bt, sl = _i32(block_table), _i32(seq_lens)
    if rows is None:
        n, sel_ptr, sel = d.batch * d.q_len * d.num_heads, None, None
    else:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n, sel_ptr = sel.shape[0], sel.ctypes.data
    out = np.empty((n, d.v_head), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    olat = np.empty((n, d.kv_lora), dtype=np.float64) if want_olat else None
    rc = lib().mla_oracle_decode(ctypes.byref(d), qb.data_ptr(), cb.data_ptr(), bt.data_ptr(),
                                 sl.data_ptr(), wk.data_ptr(), wv.data_ptr(), float(scale), n,
                                 sel_ptr, out.ctypes.data, lse.ctypes.data,
                                 olat.ctypes.data if want_olat else None)
    if rc != 0:
        raise ValueError("oracle rejected inputs (code %d)" % rc)
    return out, lse, olat


def partial(q, cache, block_table, seq_lens, w_uk, scale, b, t, h, k0, k1):
    """Latent output normalised over keys [k0, k1) of row (b, t, h) and that range's LSE."""
    d = dims_of(q, cache, block_table, w_uk, torch.empty(w_uk.shape[0], w_uk.shape[2], 1))
    o = np.empty((d.kv_lora,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = lib().mla_oracle_partial(ctypes.byref(d), _bits(q).data_ptr(), _bits(cache).data_ptr(),
                                  _i32(block_table).data_ptr(), _i32(seq_lens).data_ptr(),
                                  _bits(w_uk).data_ptr(), float(scale), b, t, h, k0, k1,
                                  o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected inputs (code %d)" % rc)
    return o, float(lse[0])


def combine(lse_parts, o_parts):
    """LSE merge of split partials: returns (lse, o)."""
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    n, dim = op.shape
    o = np.empty((dim,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = lib().mla_oracle_combine(n, dim, lp.ctypes.data, op.ctypes.data, lse.ctypes.data,
                                  o.ctypes.data)
    if rc != 0:
        raise ValueError("oracle combine rejected inputs (code %d)" % rc)
    return float(lse[0]), o


def up_project(w_uv, h, o_lat):
    """out = o_lat . W_UV[h] for one row."""
    H, lora, v = w_uv.shape
    d = Dims(1, 1, H, 0, 0, lora, v, 1, 1, 1)
    ol = np.ascontiguousarray(np.asarray(o_lat, dtype=np.float64))
    out = np.empty((v,), dtype=np.float64)
    rc = lib().mla_oracle_up_project(ctypes.byref(d), _bits(w_uv).data_ptr(), h, ol.ctypes.data,
                                     out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle up_project rejected inputs (code %d)" % rc)
    return out


def default_scale(qk_nope=128, qk_rope=64):
    return 1.0 / math.sqrt(qk_nope + qk_rope)


# ---------------------------------------------------------------------------
# FP8 weights.  vLLM PR #14770 (PR description): without an FP8 bmm the
# matrices involved in the bmm are decompressed to bf16 and the bmm runs in
# bf16.  The decompression follows the FP8 E4M3 encoding and one fp32 scale per
# 128 x 128 block (k, m) of each head's matrix; the decompressed weight is the
# fp32 product rounded to the nearest bf16 (ties to even).  The bf16 oracle
# above then applies unchanged.

def e4m3_to_float(codes):
    """Values of FP8 E4M3 codes (uint8 array), the E4M3 encoding of the OCP
    8-bit floating-point formats: sign bit, 4-bit exponent with bias 7, 3-bit
    mantissa; exponent 0 is subnormal (m/8 * 2^-6); no infinities; S.1111.111
    is NaN.  Returns float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = sign * (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def dequant_fp8_weight(w8, scale):
    """bf16 weight [H, K, M] from E4M3 codes w8 (uint8 [H, K, M]) and fp32 block
    scales [H, K/128, M/128]: bf16(fp32(value) * fp32(scale)).  The
    decompression to bf16 that vLLM PR #14770 "[Attention] MLA get rid of
    materialization" (PR description) applies to FP8 weights, since the
    absorbed form has no FP8 bmm; the block-scale layout is this library's
    reading of "FP8 weights"."""
    w8 = torch.as_tensor(w8)
    H, K, M = w8.shape
    vals = torch.from_numpy(e4m3_to_float(w8.numpy()).astype(np.float32))  # exact in fp32
    s = scale.to(torch.float32).repeat_interleave(128, 1).repeat_interleave(128, 2)
    assert s.shape == (H, K, M)
    return (vals * s).to(torch.bfloat16)  # fp32 product, then round to nearest even


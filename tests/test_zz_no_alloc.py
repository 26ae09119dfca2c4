"""The workspace-free entry point (mla_decode_run_static_scratch).

It exists for callers that cannot allocate device memory (an operator inside
an engine whose pool owns the GPU, code under a capture mode that forbids
allocations): it runs the same plan and decode kernels on a fixed scratch array
in static device memory.  This file is collected last on purpose, so a failure
here never hides the rest of the suite; it also passes when run alone.
"""
import ctypes

import pytest
import torch

from mla_decode_attention_uk_gb300 import binding
from mla_decode_attention_uk_gb300.inputs import make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def _static_call(g, out, lse, scale=None):
    d = binding.dims_for(g.q, g.cache, g.block_table)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return binding.lib().mla_decode_run_static_scratch(
        ctypes.byref(d), p(g.q), p(g.cache), p(g.block_table), p(g.seq_lens), p(g.w_uk),
        p(g.w_uv), ctypes.c_float(g.scale if scale is None else scale), p(out), p(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _outputs_like(g):
    B, T, H = g.q.shape[:3]
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device=g.q.device)
    lse = torch.full((B, T, H), float("nan"), dtype=torch.float32, device=g.q.device)
    return out, lse


def _fill_scratch_with_another_batch(dev):
    # A different, larger batch (32 query rows per sequence, long sequences cut
    # into many splits) leaves its plan, partial slots and intermediates in the
    # shared array; the next call must not depend on any of it.
    other = make_inputs(8, [3000, 64, 2500, 777, 4096, 1, 1500, 333], 1, 32, seed=79).to(dev)
    out, lse = _outputs_like(other)
    assert _static_call(other, out, lse) == 0
    return other


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_static_scratch_equals_workspace_entry_point_bitwise(case):
    inp = workload_inputs("tiny") if case == "tiny" else \
        make_inputs(5, [3, 64, 65, 700, 1500], 2, 16, seed=77)
    dev = torch.device("cuda")
    g = inp.to(dev)
    # Same default plan and the same kernels as the workspace entry point, so
    # the results must be identical bit for bit.
    ref_out, ref_lse = binding.decode(g.q, g.cache, g.block_table, g.seq_lens, g.w_uk, g.w_uv,
                                      g.scale)
    _fill_scratch_with_another_batch(dev)
    for _ in range(2):  # two calls in a row on the shared array
        out, lse = _outputs_like(g)
        assert _static_call(g, out, lse) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_static_scratch_rejects_oversized_batches():
    # 128 sequences x 128 heads needs far more than the fixed scratch.
    inp = make_inputs(128, [64] * 128, 1, 128, seed=78)
    g = inp.to(torch.device("cuda"))
    out, lse = _outputs_like(g)
    assert _static_call(g, out, lse) == 3  # MLA_DECODE_WORKSPACE_TOO_SMALL, nothing enqueued
    assert torch.isnan(out.float()).all()


def test_static_scratch_rejects_a_bad_scale_without_touching_outputs():
    inp = workload_inputs("tiny")
    g = inp.to(torch.device("cuda"))
    out, lse = _outputs_like(g)
    assert _static_call(g, out, lse, scale=-1.0) == 1
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()

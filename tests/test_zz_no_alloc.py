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

from parity_util import LSE_MAX, OUT_MAX, OUT_MEAN

pytestmark = pytest.mark.gpu


def _static_call(g, out, lse):
    d = binding.dims_for(g.q, g.cache, g.block_table)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return binding.lib().mla_decode_run_static_scratch(
        ctypes.byref(d), p(g.q), p(g.cache), p(g.block_table), p(g.seq_lens), p(g.w_uk),
        p(g.w_uv), ctypes.c_float(g.scale), p(out), p(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_static_scratch_matches_workspace_entry_point_twice(case):
    inp = workload_inputs("tiny") if case == "tiny" else \
        make_inputs(5, [3, 64, 65, 700, 1500], 2, 16, seed=77)
    dev = torch.device("cuda")
    g = inp.to(dev)
    ref_out, ref_lse = binding.decode(g.q, g.cache, g.block_table, g.seq_lens, g.w_uk, g.w_uv,
                                      g.scale)
    torch.cuda.synchronize()
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _static_call(g, out, lse) == 0
        torch.cuda.synchronize()
        do = (out.double() - ref_out.double()).abs()
        dl = (lse.double() - ref_lse.double()).abs()
        assert torch.isfinite(do).all() and torch.isfinite(dl).all()
        assert do.max().item() <= OUT_MAX and do.mean().item() <= OUT_MEAN
        assert dl.max().item() <= LSE_MAX


def test_static_scratch_rejects_oversized_batches():
    # 128 sequences x 128 heads needs far more than the fixed scratch.
    inp = make_inputs(128, [64] * 128, 1, 128, seed=78)
    g = inp.to(torch.device("cuda"))
    out = torch.empty(128, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(128, 1, 128, dtype=torch.float32, device="cuda")
    assert _static_call(g, out, lse) == 3  # MLA_DECODE_WORKSPACE_TOO_SMALL, nothing enqueued

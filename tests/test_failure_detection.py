"""Failure detection on the GPU without a fault: a bounded device-side wait on
a barrier that nothing completes gives up, records TIMEOUT in the status word,
and the context stays usable for the next decode."""
import ctypes
import time

import pytest
import torch

from mla_decode_attention_uk_gb300 import binding
from mla_decode_attention_uk_gb300.inputs import workload_inputs

from parity_util import assert_parity, compare, run_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    rc = binding.lib().mla_decode_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()),
                                                        binding._stream())
    assert rc == 0
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert int(status.item()) == 6, binding.STATUS.get(int(status.item()))
    assert 1.0 < waited < 30.0
    inp = workload_inputs("tiny")
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "decode after a timed-out wait")

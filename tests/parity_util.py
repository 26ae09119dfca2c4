"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle at the stated tolerances."""
import numpy as np
import torch

import oracle
from mla_decode_attention_uk_gb300 import binding

# Tolerances: max |d out| <= 2e-2, mean |d out| <= 2e-3, max |d lse| <= 1e-3.
OUT_MAX, OUT_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def run_gpu(inp, num_ranges=0, check_status=True):
    dev = torch.device("cuda")
    g = inp.to(dev)
    d = binding.dims_for(g.q, g.cache, g.block_table)
    m = binding.MlaDecode(d, dev, num_ranges)
    B, T, H = g.q.shape[:3]
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, T, H), float("nan"), dtype=torch.float32, device=dev)
    m.plan(g.seq_lens)
    m.run(g.q, g.cache, g.block_table, g.seq_lens, g.w_uk, g.w_uv, g.scale, out, lse)
    st = m.check()
    if check_status:
        assert st == 0, "device status %d (%s)" % (st, binding.STATUS.get(st))
    return out.cpu(), lse.cpu(), m


def compare(inp, out, lse, rows=None):
    """Compare GPU out/lse with the oracle on all rows (rows=None) or a sample."""
    o_ref, l_ref, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                    inp.w_uv, inp.scale, rows=rows)
    o = out.double().reshape(-1, 128).numpy()
    l = lse.double().reshape(-1).numpy()
    if rows is not None:
        o, l = o[rows], l[rows]
    do = np.abs(o - o_ref)
    dl = np.abs(l - l_ref)
    stats = dict(out_max=float(do.max()), out_mean=float(do.mean()), lse_max=float(dl.max()),
                 n_rows=len(l_ref))
    return stats


def assert_parity(stats, what=""):
    assert np.isfinite(stats["out_max"]) and np.isfinite(stats["lse_max"]), (what, stats)
    assert stats["out_max"] <= OUT_MAX, (what, stats)
    assert stats["out_mean"] <= OUT_MEAN, (what, stats)
    assert stats["lse_max"] <= LSE_MAX, (what, stats)

"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: max |d out| <= 2e-2, mean |d out| <= 2e-3, max |d lse| <= 1e-3.
Every case compares every output row, the full-size workloads included (the
oracle is threaded over query rows; the largest, draft_q8, is about 2e8
row-keys)."""
import math
import random

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_uk_gb300 import binding
from mla_decode_attention_uk_gb300.inputs import make_inputs, quantize_fp8_blockwise, workload_inputs

from parity_util import assert_parity, compare, run_gpu

pytestmark = pytest.mark.gpu


def q_lo_values(m):
    """The residual the absorb step stores (E4M3 codes of q_lo * 2^10), decoded
    with PyTorch's float8_e4m3fn."""
    return m.q_lo().cpu().view(torch.float8_e4m3fn).float() * 2.0 ** -10


def test_absorb_bmm_matches_fp32_matmul():
    inp = make_inputs(3, [70, 5, 300], 2, 32, seed=41)
    dev = torch.device("cuda")
    g = inp.to(dev)
    d = binding.dims_for(g.q, g.cache, g.block_table)
    m = binding.MlaDecode(d, dev)
    m.absorb(g.q, g.w_uk)
    torch.cuda.synchronize()
    hi = m.q_lat().float().cpu()
    lo = q_lo_values(m)
    ref = torch.einsum("bthk,hkl->bthl", inp.q[..., :128].double(), inp.w_uk.double())
    ref = ref.reshape(-1, 512)
    got = hi[:, :512].double() + lo.double()
    # hi + lo carries ~13 significant bits: the E4M3 rounding of the residual
    # is at most 2^-4 of a residual that is itself at most 2^-9 of the value
    # (plus E4M3's subnormal step 2^-9 at the 2^10 scale); fp32 accumulation
    # over K = 128 adds far less.
    assert ((got - ref).abs() <= ref.abs() * 2.0 ** -13 + 2.0 ** -19 + 2e-6).all()
    assert torch.equal(hi[:, 512:], inp.q[..., 128:].reshape(-1, 64).float())
    # hi is the bf16 rounding of the fp32 product, lo the E4M3 rounding of the rest
    assert (hi[:, :512].double() - ref).abs().max().item() <= ref.abs().max().item() * 2 ** -8


@pytest.mark.parametrize("B,T,H", [(200, 2, 16), (130, 2, 128), (256, 1, 32), (64, 2, 16),
                                   (129, 1, 48)])
def test_absorb_bmm_large_token_counts_matches_fp64(B, T, H):
    # 128-token tiles of the untransposed absorb kernel: 400 and 260 tokens
    # leave a ragged last tile, 256 is two full ones, 128 exactly one, and 129
    # a last tile of one token (the tensor stores clip the other 127 rows);
    # 16 to 128 heads, so the persistent grid has fewer units than SMs
    # (128 tokens x 16 heads: 64 units) or several per SM (129 x 48: 384).
    # Same bound as the small case above.
    g = torch.Generator().manual_seed(40 + B + H)
    lens = torch.randint(T, 200, (B,), generator=g).tolist()
    inp = make_inputs(B, lens, T, H, seed=42 + H)
    dev = torch.device("cuda")
    gd = inp.to(dev)
    m = binding.MlaDecode(binding.dims_for(gd.q, gd.cache, gd.block_table), dev)
    m.absorb(gd.q, gd.w_uk)
    torch.cuda.synchronize()
    hi = m.q_lat().float().cpu()
    lo = q_lo_values(m)
    ref = torch.einsum("bthk,hkl->bthl", inp.q[..., :128].double(), inp.w_uk.double())
    ref = ref.reshape(-1, 512)
    got = hi[:, :512].double() + lo.double()
    assert ((got - ref).abs() <= ref.abs() * 2.0 ** -13 + 2.0 ** -19 + 2e-6).all()
    assert torch.equal(hi[:, 512:], inp.q[..., 128:].reshape(-1, 64).float())
    assert (hi[:, :512].double() - ref).abs().max().item() <= ref.abs().max().item() * 2 ** -8
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "absorb B=%d T=%d H=%d" % (B, T, H))


def test_tiny_workload_all_rows():
    inp = workload_inputs("tiny")
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "tiny")


# 48/80 heads leave a partial last tile; 96 x 2 rows make three tiles; 112 x 2
# rows make four with a 32-row last tile.  128 x 6, 112 x 8 and 128 x 8 rows
# make 12, 14 and 16 tiles, which do not divide 152 SMs: CTA groups then hold
# 4, 2 and 8 tiles and each takes several (range, tile set) tasks.
@pytest.mark.parametrize("H,T", [(16, 1), (32, 1), (64, 1), (128, 1), (16, 2), (64, 2), (128, 2),
                                 (48, 1), (80, 1), (96, 2), (112, 2),
                                 (16, 4), (128, 3), (64, 8), (128, 8), (128, 6), (112, 8)])
def test_ragged_lengths_all_rows(H, T):
    lens = [T, 1 + T, 63, 64, 65, 127, 128, 129, 200, 511, 700]
    inp = make_inputs(len(lens), lens, T, H, seed=100 + H + T)
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "H=%d T=%d" % (H, T))


def default_ranges_expected(T, H, sms):
    """The attention step's default work-range count: one per CTA group of
    all a sequence's 64-row tiles when those groups fill the SMs to within 3 %;
    otherwise groups of gcd(tiles, SMs) tiles, and the fewest ranges that deal
    every group the same number of (range, tile set) tasks."""
    tiles = -(-T * H // 64)
    idle = sms % tiles
    tpg = math.gcd(tiles, sms) if 100 * idle >= 3 * sms else tiles
    groups, sets = sms // tpg, tiles // tpg
    return groups // math.gcd(groups, sets)


@pytest.mark.parametrize("T,H", [(1, 16), (1, 128), (2, 128), (6, 128), (7, 128), (8, 128),
                                 (8, 112), (3, 128)])
def test_default_range_count(T, H):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    inp = make_inputs(3, [T + 100, T + 700, T + 2000], T, H, seed=44)
    out, lse, m = run_gpu(inp)
    assert m.plan_header()[0] == default_ranges_expected(T, H, sms)
    assert_parity(compare(inp, out, lse), "default ranges T=%d H=%d" % (T, H))


@pytest.mark.parametrize("num_ranges", [1, 3, 7, 64, 300, 1000])
def test_split_counts(num_ranges):
    lens = [5, 700, 64, 1300, 2, 333]
    inp = make_inputs(len(lens), lens, 2, 16, seed=7)
    out, lse, m = run_gpu(inp, num_ranges=num_ranges)
    hdr = m.plan_header()
    assert hdr[0] == num_ranges
    assert_parity(compare(inp, out, lse), "R=%d" % num_ranges)


@pytest.mark.parametrize("num_ranges", [1, 7, 40])
def test_split_counts_long_drafts(num_ranges):
    # q_len 8: query t of the draft sees keys [0, L - 8 + t]
    lens = [8, 9, 600, 1500, 77]
    inp = make_inputs(len(lens), lens, 8, 32, seed=17)
    out, lse, _ = run_gpu(inp, num_ranges=num_ranges)
    assert_parity(compare(inp, out, lse), "T=8 R=%d" % num_ranges)


@pytest.mark.parametrize("T", [1, 2])
def test_many_short_sequences_plan_in_global_memory(T):
    # More sequences than the planner keeps in shared memory (4096): its cost
    # prefix and per-range searches run from global memory.  Lengths up to
    # 130 tokens, page boundaries included; 16 heads.
    g = torch.Generator().manual_seed(71 + T)
    B = 5000
    lens = torch.randint(T, 131, (B,), generator=g).tolist()
    lens[:6] = [T, 63, 64, 65, 128, 130]
    inp = make_inputs(B, lens, T, 16, seed=72 + T)
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "B=%d T=%d" % (B, T))


def test_one_very_long_sequence_split_over_every_range():
    # One sequence of 131072 tokens (2048 pages): every work range takes a
    # piece of it, so the combine merges more than 32 splits per row.
    inp = make_inputs(1, [131072], 1, 16, seed=73)
    out, lse, m = run_gpu(inp)
    assert m.plan_header()[0] > 32
    assert_parity(compare(inp, out, lse), "L=131072")


def test_split_counts_h128():
    lens = [900, 2000, 70]
    inp = make_inputs(len(lens), lens, 1, 128, seed=8)
    for R in (2, 41):
        out, lse, _ = run_gpu(inp, num_ranges=R)
        assert_parity(compare(inp, out, lse), "R=%d" % R)


def test_deterministic_for_a_fixed_plan():
    inp = make_inputs(4, [100, 1000, 64, 2000], 1, 64, seed=9)
    o1, l1, _ = run_gpu(inp, num_ranges=5)
    o2, l2, _ = run_gpu(inp, num_ranges=5)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_one_plan_serves_consecutive_runs_bitwise():
    # The plan is built once per decode step and reused by every layer: runs
    # back to back on one plan (the absorb step of a run overlapping the end of
    # the previous run) must give identical results.
    inp = make_inputs(4, [100, 3000, 64, 777], 1, 128, seed=15)
    dev = torch.device("cuda")
    g = inp.to(dev)
    d = binding.dims_for(g.q, g.cache, g.block_table)
    m = binding.MlaDecode(d, dev)
    outs = [torch.empty(4, 1, 128, 128, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    lses = [torch.empty(4, 1, 128, dtype=torch.float32, device=dev) for _ in range(3)]
    m.plan(g.seq_lens)
    for o, l in zip(outs, lses):
        m.run(g.q, g.cache, g.block_table, g.seq_lens, g.w_uk, g.w_uv, g.scale, o, l)
    assert m.check() == 0
    for o, l in zip(outs[1:], lses[1:]):
        assert torch.equal(o, outs[0]) and torch.equal(l, lses[0])
    assert_parity(compare(inp, outs[0].cpu(), lses[0].cpu()), "plan reused")


# Small batches: mla_decode_run merges the splits inside the up-projection
# (three kernels, see mla_decode_kernels_per_run); the step calls run the
# combine and the up-projection apart.  Both must agree bit for bit, for each
# merge variant (mostly unsplit rows: R < B; a few splits; many splits), for
# ragged last token tiles, and at the largest one-wave size (64 tokens x 16
# heads, 4 tiles each of 16 heads).
@pytest.mark.parametrize("B,T,H,R", [(3, 2, 64, 5), (3, 2, 64, 1), (3, 1, 128, 40),
                                     (10, 2, 32, 4), (64, 1, 16, 0), (8, 1, 128, 0),
                                     (5, 8, 48, 30)])
def test_step_calls_equal_run_bitwise(B, T, H, R):
    g0 = torch.Generator().manual_seed(16 + B + R)
    lens = torch.randint(1, 3000, (B,), generator=g0).tolist()
    inp = make_inputs(B, lens, T, H, seed=16)
    dev = torch.device("cuda")
    g = inp.to(dev)
    d = binding.dims_for(g.q, g.cache, g.block_table)
    m = binding.MlaDecode(d, dev, R)
    o1 = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    m.plan(g.seq_lens)
    m.run(g.q, g.cache, g.block_table, g.seq_lens, g.w_uk, g.w_uv, g.scale, o1, l1)
    m.plan(g.seq_lens)
    m.absorb(g.q, g.w_uk)
    m.attend(g.cache, g.block_table, g.seq_lens, g.scale, l2)
    m.combine(g.scale, l2)
    m.up_project(g.w_uv, o2)
    assert m.check() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert_parity(compare(inp, o1.cpu(), l1.cpu()), "run B=%d T=%d H=%d R=%d" % (B, T, H, R))


def test_kernels_per_run():
    # Fused combine + up-projection for small one-wave batches, bf16 or FP8
    # weights alike.
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def count(B, T, H, fp8=False):
        d = binding.Dims(batch=B, q_len=T, num_heads=H, qk_nope=128, qk_rope=64, kv_lora=512,
                         v_head=128, page_size=64, num_pages=4, max_pages_per_seq=2)
        return binding.kernels_per_run(d, fp8)

    assert count(64, 1, 16) == 3 and count(8, 1, 128) == 3
    assert count(8, 1, 128, fp8=True) == 3 and count(128, 1, 128, fp8=True) == 4
    assert count(128, 1, 128) == 4 and count(64, 2, 16) == 4
    assert count(112, 1, 32) == (3 if 7 * 32 <= sms else 4)
    assert count(48, 1, 48) == (3 if 3 * 48 <= sms else 4)


@pytest.mark.parametrize("R", [0, 400])
def test_large_run_matches_step_calls(R):
    # 160 tokens x 128 heads: 256 (128-token tile, head) units, more than the
    # SMs, so mla_decode_run merges split sequences only in the combine and
    # corrects the other rows in its up-projection, while the step calls keep
    # the combine for every row.  out must agree bit for bit (same o_lat, same
    # products), lse up to the summation order of the correction; both match
    # the oracle on every row.  R = 400 ranges (default: one per SM group)
    # cuts sequences into many splits and makes the split-only combine's grid
    # stride over more ranges than it was sized for.
    g = torch.Generator().manual_seed(91 + R)
    lens = torch.randint(1, 2500, (160,), generator=g).tolist()
    inp = make_inputs(160, lens, 1, 128, seed=92)
    dev = torch.device("cuda")
    gd = inp.to(dev)
    m = binding.MlaDecode(binding.dims_for(gd.q, gd.cache, gd.block_table), dev, R)
    o1 = torch.empty(160, 1, 128, 128, dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(160, 1, 128, dtype=torch.float32, device=dev)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    m.plan(gd.seq_lens)
    m.run(gd.q, gd.cache, gd.block_table, gd.seq_lens, gd.w_uk, gd.w_uv, gd.scale, o1, l1)
    m.plan(gd.seq_lens)
    m.absorb(gd.q, gd.w_uk)
    m.attend(gd.cache, gd.block_table, gd.seq_lens, gd.scale, l2)
    m.combine(gd.scale, l2)
    m.up_project(gd.w_uv, o2)
    assert m.check() == 0
    assert torch.equal(o1, o2)
    assert (l1 - l2).abs().max().item() <= 1e-6
    assert_parity(compare(inp, o1.cpu(), l1.cpu()), "large run R=%d" % R)


def test_large_run_ragged_split_blocks():
    # 400 tokens x 48 heads: 4 token tiles x 48 heads = 192 units of 128
    # tokens x one head, more than the SMs, so the large-run path.  300 ranges make
    # the split-only combine use 32-row blocks, and 48 rows per sequence
    # leave a 16-row last block.  out bit for bit as the step calls, lse up
    # to the summation order of the correction, every row against the oracle.
    g = torch.Generator().manual_seed(93)
    lens = torch.randint(1, 300, (400,), generator=g).tolist()
    inp = make_inputs(400, lens, 1, 48, seed=94)
    dev = torch.device("cuda")
    gd = inp.to(dev)
    m = binding.MlaDecode(binding.dims_for(gd.q, gd.cache, gd.block_table), dev, 300)
    o1 = torch.empty(400, 1, 48, 128, dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(400, 1, 48, dtype=torch.float32, device=dev)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    m.plan(gd.seq_lens)
    m.run(gd.q, gd.cache, gd.block_table, gd.seq_lens, gd.w_uk, gd.w_uv, gd.scale, o1, l1)
    m.plan(gd.seq_lens)
    m.absorb(gd.q, gd.w_uk)
    m.attend(gd.cache, gd.block_table, gd.seq_lens, gd.scale, l2)
    m.combine(gd.scale, l2)
    m.up_project(gd.w_uv, o2)
    assert m.check() == 0
    assert torch.equal(o1, o2)
    assert (l1 - l2).abs().max().item() <= 1e-6
    assert_parity(compare(inp, o1.cpu(), l1.cpu()), "large run, ragged 32-row split blocks")


def test_page_permutation_same_schedule_bitwise():
    inp = make_inputs(3, [130, 640, 77], 1, 32, seed=10)
    o1, l1, _ = run_gpu(inp)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(inp.cache.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    inp.cache = inp.cache[perm].contiguous()
    valid = inp.block_table >= 0
    inp.block_table[valid] = inv[inp.block_table[valid].long()].to(torch.int32)
    o2, l2, _ = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_unreferenced_nan_pages_do_not_leak():
    inp = make_inputs(3, [100, 31, 64], 1, 16, seed=11, spare_pages=4)
    out, lse, _ = run_gpu(inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert_parity(compare(inp, out, lse), "nan spare")


def test_single_key_closed_form():
    inp = make_inputs(2, [1, 1], 1, 16, seed=12)
    out, lse, _ = run_gpu(inp)
    assert_parity(compare(inp, out, lse), "L=1")


def test_bad_block_table_entry_sets_status_without_fault():
    inp = make_inputs(2, [100, 100], 1, 16, seed=13)
    inp.block_table[1, 1] = inp.cache.shape[0] + 5
    out, lse, m = run_gpu(inp, check_status=False)
    assert m.check() == 5
    # the other sequence is still right
    st = compare(inp.__class__(inp.q[:1].clone(), inp.cache, inp.block_table[:1].clone(),
                               inp.seq_lens[:1].clone(), inp.w_uk, inp.w_uv, inp.scale),
                 out[:1], lse[:1])
    assert_parity(st, "valid sequence next to a bad one")


def test_seq_len_beyond_block_table_sets_status():
    inp = make_inputs(2, [100, 100], 1, 16, seed=14)
    inp.seq_lens[0] = inp.block_table.shape[1] * 64 + 1
    _, _, m = run_gpu(inp, check_status=False)
    assert m.check() == 5


def _late_pages_score_higher(inp, step, seed=0):
    """Add (page index in the sequence) * step * u to every key's k_pe columns,
    u one fixed random direction.  For a row whose q_pe has a positive
    component along u, later pages then score higher as a whole: the running
    max grows page after page and the online softmax must rescale its
    accumulator, while scores within a page keep their spread (the attention
    stays spread over many keys, so outputs stay O(1)).  Latent (value)
    columns are untouched."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(64, generator=g, dtype=torch.float64) / 8.0
    cache = inp.cache.clone()
    for b in range(inp.block_table.shape[0]):
        n = (int(inp.seq_lens[b]) + 63) // 64
        for i in range(n):
            pg = int(inp.block_table[b, i])
            cache[pg, :, 512:] = (cache[pg, :, 512:].double() + step * i * u).to(torch.bfloat16)
    inp.cache = cache
    return inp


@pytest.mark.parametrize("H,T,R", [(16, 1, 1), (16, 1, 3), (16, 2, 1), (32, 1, 2), (64, 1, 1),
                                   (128, 1, 3), (128, 2, 1)])
def test_late_pages_force_rescale(H, T, R):
    lens = [700, 2500, 130]
    inp = _late_pages_score_higher(make_inputs(len(lens), lens, T, H, seed=300 + H + T), 8.0)
    # The case needs rescales: for some row of sequence 1 a late page's LSE
    # exceeds the first page's by more than the 8-bit (log2) rescale threshold
    # plus ln 64 (the most a page's LSE can exceed its max score).
    need = 0
    for h in range(H):
        args = (inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk, inp.scale, 1, 0, h)
        _, l_first = oracle.partial(*args, 0, 64)
        _, l_late = oracle.partial(*args, 2432, 2496)
        need += l_late - l_first > 8 * math.log(2) + math.log(64)
    assert need >= max(1, H // 8)
    out, lse, _ = run_gpu(inp, num_ranges=R)
    assert_parity(compare(inp, out, lse), "H=%d T=%d R=%d" % (H, T, R))


@pytest.mark.parametrize("name", ["tp_shard", "full_head", "long", "mixed_spec", "draft_q8"])
def test_full_size_workloads_all_rows(name):
    # The bench's workloads at full size, in the launch configuration it times
    # (default plan), every query row against the oracle.
    inp = workload_inputs(name)
    out, lse, _ = run_gpu(inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    stats = compare(inp, out, lse)
    assert stats["n_rows"] == out.shape[0] * out.shape[1] * out.shape[2]
    print(name, stats)
    assert_parity(stats, name)


@pytest.mark.parametrize("B,T,H", [(3, 1, 16), (20, 1, 64), (64, 1, 16), (40, 2, 128),
                                   (100, 2, 16), (72, 8, 32)])
def test_fp8_weights_equal_bf16_run_on_decompressed_weights(B, T, H):
    # 16-, 32-, 64- and 128-token bmm tiles, up to five 128-token tiles per
    # head with a ragged last one (576 tokens).  The kernels decompress each
    # FP8 weight tile to bf16 as they load it; the result must equal, bit for
    # bit, the bf16 path given the weights the oracle decompresses, and match
    # the oracle.
    g = torch.Generator().manual_seed(60 + H + B)
    lens = torch.randint(T, 900 if B * T <= 256 else 300, (B,), generator=g).tolist()
    inp = make_inputs(B, lens, T, H, seed=61 + H)
    uk8, uk_s = quantize_fp8_blockwise(inp.w_uk)
    uv8, uv_s = quantize_fp8_blockwise(inp.w_uv)
    inp.w_uk = oracle.dequant_fp8_weight(uk8, uk_s)
    inp.w_uv = oracle.dequant_fp8_weight(uv8, uv_s)
    dev = torch.device("cuda")
    gd = inp.to(dev)
    d = binding.dims_for(gd.q, gd.cache, gd.block_table)
    m = binding.MlaDecode(d, dev)
    o8 = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    l8 = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    ob, lb = torch.empty_like(o8), torch.empty_like(l8)
    m.plan(gd.seq_lens)
    m.run_fp8w(gd.q, gd.cache, gd.block_table, gd.seq_lens, uk8.to(dev), uk_s.to(dev),
               uv8.to(dev), uv_s.to(dev), gd.scale, o8, l8)
    m.run(gd.q, gd.cache, gd.block_table, gd.seq_lens, gd.w_uk, gd.w_uv, gd.scale, ob, lb)
    assert m.check() == 0
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    assert_parity(compare(inp, o8.cpu(), l8.cpu()), "fp8 weights B=%d T=%d H=%d" % (B, T, H))


@pytest.mark.parametrize("name", ["tp_shard", "mixed_spec"])
def test_full_size_fp8_weights_all_rows(name):
    # The bench's FP8 configuration at full size: 64-token tiles (tp_shard)
    # and four 128-token tiles per head (mixed_spec), every row.
    inp = workload_inputs(name)
    uk8, uk_s = quantize_fp8_blockwise(inp.w_uk)
    uv8, uv_s = quantize_fp8_blockwise(inp.w_uv)
    inp.w_uk = oracle.dequant_fp8_weight(uk8, uk_s)
    inp.w_uv = oracle.dequant_fp8_weight(uv8, uv_s)
    dev = torch.device("cuda")
    gd = inp.to(dev)
    B, T, H = inp.q.shape[:3]
    d = binding.dims_for(gd.q, gd.cache, gd.block_table)
    m = binding.MlaDecode(d, dev)
    out = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, T, H, dtype=torch.float32, device=dev)
    m.plan(gd.seq_lens)
    m.run_fp8w(gd.q, gd.cache, gd.block_table, gd.seq_lens, uk8.to(dev), uk_s.to(dev),
               uv8.to(dev), uv_s.to(dev), gd.scale, out, lse)
    assert m.check() == 0
    assert_parity(compare(inp, out.cpu(), lse.cpu()), "fp8 weights " + name)


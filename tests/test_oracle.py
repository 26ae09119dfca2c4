"""Pins for the fp64 oracle, each against something other than the oracle itself.

* the explicit, non-absorbed formulation (decompress K = C W_UK^T and
  V = C W_UV per head, ordinary multi-head attention with the RoPE part
  concatenated) -- the algebra that weight absorption regroups (vLLM PR #14770
  "[Attention] MLA get rid of materialization", PR description);
* torch's scaled_dot_product_attention in fp64 on that explicit K/V;
* closed forms (one key; identical keys; zero query; constant latent rows);
* invariants (page permutation, NaN in unreferenced pages, split + LSE combine,
  the causal query pair);
* a pure-Python brute force at reduced dims and a hand-derived example;
* planted mistakes in a copy of the oracle source must fail these pins.
"""
import ctypes
import json
import math
import os
import random
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_uk_gb300.inputs import make_inputs, workload_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def explicit_numpy(inp):
    """Non-absorbed MLA decode in numpy fp64: per head, K_h = [C_lat W_UK[h]^T || k_pe],
    V_h = C_lat W_UV[h]; softmax(scale q K_h^T) V_h.  Returns out [B*T*H, v], lse [B*T*H]."""
    q = inp.q.double().numpy()
    cache = inp.cache.double().numpy()
    wuk = inp.w_uk.double().numpy()
    wuv = inp.w_uv.double().numpy()
    B, T, H, dq = q.shape
    nope = wuk.shape[1]
    lora = wuk.shape[2]
    P = cache.shape[1]
    outs, lses = [], []
    for b in range(B):
        L = int(inp.seq_lens[b])
        pages = inp.block_table[b, :(L + P - 1) // P].numpy()
        C = cache[pages].reshape(-1, cache.shape[2])[:L]
        for t in range(T):
            n = L - T + t + 1
            for h in range(H):
                K = np.concatenate([C[:n, :lora] @ wuk[h].T, C[:n, lora:]], axis=1)
                V = C[:n, :lora] @ wuv[h]
                s = inp.scale * (K @ q[b, t, h])
                m = s.max()
                lse = m + math.log(np.exp(s - m).sum())
                outs.append(np.exp(s - lse) @ V)
                lses.append(lse)
    return np.stack(outs), np.array(lses)


def rand_case(seed, B, lens, T, H, spare=0):
    return make_inputs(B, lens, T, H, seed, spare_pages=spare)


# ---------------------------------------------------------------------------
def test_tiny_workload_matches_explicit_form():
    inp = workload_inputs("tiny")
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    eo, el = explicit_numpy(inp)
    np.testing.assert_allclose(out, eo, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, el, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_random_small_matches_explicit_form(seed):
    r = random.Random(seed)
    B = r.randint(1, 3)
    T = r.choice([1, 2])
    lens = [r.randint(T, 300) for _ in range(B)]
    inp = rand_case(100 + seed, B, lens, T, 4)
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    eo, el = explicit_numpy(inp)
    np.testing.assert_allclose(out, eo, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, el, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T", [2, 4, 8])
def test_matches_torch_sdpa_fp64_with_causal_block(T):
    inp = rand_case(7 + T, 2, [70, 130], T, 3)
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    q = inp.q.double()
    cache = inp.cache.double()
    got = out.reshape(2, T, 3, -1)
    for b in range(2):
        L = int(inp.seq_lens[b])
        pages = inp.block_table[b, :(L + 63) // 64].long()
        C = cache[pages].reshape(-1, 576)[:L]
        for h in range(3):
            K = torch.cat([C[:, :512] @ inp.w_uk[h].double().T, C[:, 512:]], 1)
            V = C[:, :512] @ inp.w_uv[h].double()
            # query t of the block does not see the block's later new tokens
            mask = torch.ones(T, L, dtype=torch.bool)
            for t in range(T):
                mask[t, L - T + t + 1:] = False
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b, :, h][None, None], K[None, None], V[None, None], attn_mask=mask[None, None],
                scale=inp.scale)[0, 0]
            np.testing.assert_allclose(got[b, :, h], ref.numpy(), rtol=1e-10, atol=1e-12)
            s = inp.scale * (q[b, :, h] @ K.T)
            s = s.masked_fill(~mask, float("-inf"))
            np.testing.assert_allclose(lse.reshape(2, T, 3)[b, :, h],
                                       torch.logsumexp(s, dim=1).numpy(), rtol=1e-12)


# ---------------------------------------------------------------------------
def test_closed_form_single_key():
    inp = rand_case(11, 1, [1], 1, 2)
    out, lse, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                   inp.w_uv, inp.scale, want_olat=True)
    c0 = inp.cache[int(inp.block_table[0, 0]), 0].double()
    for h in range(2):
        qn, qp = inp.q[0, 0, h, :128].double(), inp.q[0, 0, h, 128:].double()
        # score written with the key decompressed (W_UK applied to c), not to q
        s0 = inp.scale * (qn @ (inp.w_uk[h].double() @ c0[:512]) + qp @ c0[512:])
        assert lse[h] == pytest.approx(float(s0), rel=1e-12, abs=1e-12)
        np.testing.assert_allclose(olat[h], c0[:512].numpy(), rtol=0, atol=1e-15)
        np.testing.assert_allclose(out[h], (c0[:512] @ inp.w_uv[h].double()).numpy(), rtol=1e-12)


def test_closed_form_identical_keys():
    L = 150
    inp = rand_case(12, 1, [L], 1, 2)
    row = inp.cache[0, 0].clone()
    inp.cache[:] = row
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    c = row.double()
    for h in range(2):
        qn, qp = inp.q[0, 0, h, :128].double(), inp.q[0, 0, h, 128:].double()
        s = inp.scale * (qn @ (inp.w_uk[h].double() @ c[:512]) + qp @ c[512:])
        assert lse[h] == pytest.approx(float(s) + math.log(L), rel=1e-12)
        np.testing.assert_allclose(out[h], (c[:512] @ inp.w_uv[h].double()).numpy(), rtol=1e-11,
                                   atol=1e-13)


def test_closed_form_zero_query():
    inp = rand_case(13, 2, [33, 200], 1, 2)
    inp.q.zero_()
    out, lse, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                   inp.w_uv, inp.scale, want_olat=True)
    cache = inp.cache.double()
    for b, L in enumerate([33, 200]):
        pages = inp.block_table[b, :(L + 63) // 64].long()
        C = cache[pages].reshape(-1, 576)[:L, :512]
        mean = C.mean(0)
        for h in range(2):
            i = b * 2 + h
            assert lse[i] == pytest.approx(math.log(L), rel=1e-14)
            np.testing.assert_allclose(olat[i], mean.numpy(), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(out[i], (mean @ inp.w_uv[h].double()).numpy(), rtol=1e-11,
                                       atol=1e-13)


def test_softmax_weights_sum_to_one():
    # With every latent entry equal to 1, o_lat = sum_j p_j for every dim.
    inp = rand_case(14, 2, [64, 321], 2, 3)
    inp.cache[:, :, :512] = 1.0
    _, _, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                               inp.w_uv, inp.scale, want_olat=True)
    np.testing.assert_allclose(olat, 1.0, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
def test_page_permutation_invariance_bitwise():
    inp = rand_case(15, 3, [65, 128, 257], 1, 4)
    base = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk, inp.w_uv,
                         inp.scale)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(inp.cache.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    cache2 = inp.cache[perm].contiguous()       # physical page i now holds old page perm[i]
    bt2 = inp.block_table.clone()
    valid = bt2 >= 0
    bt2[valid] = inv[bt2[valid].long()].to(torch.int32)
    other = oracle.decode(inp.q, cache2, bt2, inp.seq_lens, inp.w_uk, inp.w_uv, inp.scale)
    assert np.array_equal(base[0], other[0]) and np.array_equal(base[1], other[1])


def test_unreferenced_nan_pages_are_never_read():
    inp = rand_case(16, 2, [100, 31], 1, 2, spare=3)
    assert torch.isnan(inp.cache[-1].float()).all()
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    clean = inp.cache[:inp.used_pages].contiguous()
    out2, lse2, _ = oracle.decode(inp.q, clean, inp.block_table, inp.seq_lens, inp.w_uk, inp.w_uv,
                                  inp.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("k", [1, 2, 3, 7])
def test_split_and_lse_combine_equal_unsplit(k):
    L = 203
    inp = rand_case(17, 1, [L], 1, 2)
    out, lse, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                   inp.w_uv, inp.scale, want_olat=True)
    r = random.Random(k)
    cuts = sorted(r.sample(range(1, L), k - 1))  # ranges end mid-page in general
    bounds = [0] + cuts + [L]
    for h in range(2):
        parts = [oracle.partial(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.scale, 0, 0, h, bounds[i], bounds[i + 1]) for i in range(k)]
        lse_c, o_c = oracle.combine([p[1] for p in parts], np.stack([p[0] for p in parts]))
        assert lse_c == pytest.approx(lse[h], rel=1e-13, abs=1e-13)
        np.testing.assert_allclose(o_c, olat[h], rtol=1e-12, atol=1e-14)
        # the merged latent output, mapped back by W_UV, is the unsplit out
        up = oracle.up_project(inp.w_uv, h, o_c)
        np.testing.assert_allclose(up, out[h], rtol=1e-11, atol=1e-13)


def _up_project_rows(up_fn, inp, olat):
    B, T, H = inp.q.shape[:3]
    return np.stack([up_fn(inp.w_uv, r % H, olat[r]) for r in range(B * T * H)])


@pytest.mark.parametrize("seed", range(3))
def test_up_project_matches_explicit_value_projection(seed):
    """mla_oracle_up_project (o_lat . W_UV[h]) against the non-absorbed form,
    which decompresses V_h = C_lat W_UV[h] first and then takes the softmax
    average of V_h's rows: the other association of the same product (vLLM PR
    #14770, PR description).  Each row must use its own head's W_UV."""
    r = random.Random(100 + seed)
    T = r.choice([1, 2])
    B, H = r.randint(1, 3), 3
    lens = [r.randint(T, 200) for _ in range(B)]
    inp = rand_case(300 + seed, B, lens, T, H)
    out, _, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                 inp.w_uv, inp.scale, want_olat=True)
    up = _up_project_rows(oracle.up_project, inp, olat)
    eo, _ = explicit_numpy(inp)
    np.testing.assert_allclose(up, eo, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(up, out, rtol=1e-12, atol=1e-14)


def test_causal_pair_first_query_equals_single_query_on_shorter_sequence():
    L = 129
    inp2 = rand_case(18, 1, [L], 2, 3)
    out2, lse2, _ = oracle.decode(inp2.q, inp2.cache, inp2.block_table, inp2.seq_lens, inp2.w_uk,
                                  inp2.w_uv, inp2.scale)
    q1 = inp2.q[:, :1].contiguous()
    out1, lse1, _ = oracle.decode(q1, inp2.cache, inp2.block_table,
                                  torch.tensor([L - 1], dtype=torch.int32), inp2.w_uk, inp2.w_uv,
                                  inp2.scale)
    assert np.array_equal(out2.reshape(2, 3, -1)[0], out1.reshape(3, -1))
    assert np.array_equal(lse2.reshape(2, 3)[0], lse1)


def test_row_selection_matches_full_run():
    inp = rand_case(19, 2, [90, 40], 2, 3)
    out, lse, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                                inp.w_uv, inp.scale)
    rows = [0, 5, 11, 7]
    o2, l2, _ = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                              inp.w_uv, inp.scale, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


def test_rejects_bad_block_table_and_seq_len():
    inp = rand_case(20, 1, [70], 1, 1)
    bt = inp.block_table.clone()
    bt[0, 1] = inp.cache.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(inp.q, inp.cache, bt, inp.seq_lens, inp.w_uk, inp.w_uv, inp.scale)
    with pytest.raises(ValueError):
        oracle.decode(inp.q, inp.cache, inp.block_table, torch.tensor([0], dtype=torch.int32),
                      inp.w_uk, inp.w_uv, inp.scale)


# ---------------------------------------------------------------------------
def _small_dims_case(seed, nope=2, rope=1, lora=3, v=2, page=2, B=2, T=2, H=2, lens=(5, 3)):
    g = torch.Generator().manual_seed(seed)
    rnd = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    npages = [(L + page - 1) // page for L in lens]
    P = sum(npages)
    cache = rnd(P, page, lora + rope)
    perm = torch.randperm(P, generator=g).to(torch.int32)
    bt = torch.full((B, max(npages)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return dict(q=rnd(B, T, H, nope + rope), cache=cache, bt=bt,
                sl=torch.tensor(list(lens), dtype=torch.int32), wuk=rnd(H, nope, lora),
                wuv=rnd(H, lora, v), scale=0.7, dims=(nope, rope, lora, v, page, B, T, H))


def brute_force_python(c):
    """Pure-Python loops over lists of floats (no numpy), straight from the definition."""
    nope, rope, lora, v, page, B, T, H = c["dims"]
    q, cache = c["q"].double().tolist(), c["cache"].double().tolist()
    wuk, wuv = c["wuk"].double().tolist(), c["wuv"].double().tolist()
    bt, sl = c["bt"].tolist(), c["sl"].tolist()
    outs, lses = [], []
    for b in range(B):
        for t in range(T):
            for h in range(H):
                qv = q[b][t][h]
                ql = [sum(qv[k] * wuk[h][k][l] for k in range(nope)) for l in range(lora)]
                ql += qv[nope:]
                n = sl[b] - T + t + 1
                keys = [cache[bt[b][j // page]][j % page] for j in range(n)]
                s = [c["scale"] * sum(a * x for a, x in zip(ql, key)) for key in keys]
                m = max(s)
                lse = m + math.log(sum(math.exp(x - m) for x in s))
                p = [math.exp(x - lse) for x in s]
                o = [sum(p[j] * keys[j][l] for j in range(n)) for l in range(lora)]
                outs.append([sum(o[l] * wuv[h][l][k] for l in range(lora)) for k in range(v)])
                lses.append(lse)
    return np.array(outs), np.array(lses)


def oracle_small(c, lib=None):
    nope, rope, lora, v, page, B, T, H = c["dims"]
    L = lib or oracle.lib()
    d = oracle.Dims(B, T, H, nope, rope, lora, v, page, c["cache"].shape[0], c["bt"].shape[1])
    out = np.empty((B * T * H, v))
    lse = np.empty((B * T * H,))
    bits = lambda x: x.contiguous().view(torch.int16)
    qb, cb, wk, wv = bits(c["q"]), bits(c["cache"]), bits(c["wuk"]), bits(c["wuv"])
    rc = L.mla_oracle_decode(ctypes.byref(d), qb.data_ptr(), cb.data_ptr(), c["bt"].data_ptr(),
                             c["sl"].data_ptr(), wk.data_ptr(), wv.data_ptr(), c["scale"], 0, None,
                             out.ctypes.data, lse.ctypes.data, None)
    assert rc == 0
    return out, lse


@pytest.mark.parametrize("seed", range(4))
def test_pure_python_brute_force_reduced_dims(seed):
    c = _small_dims_case(seed, lens=(5 + seed, 2 + seed))
    bo, bl = brute_force_python(c)
    oo, ol = oracle_small(c)
    np.testing.assert_allclose(oo, bo, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ol, bl, rtol=1e-12, atol=1e-14)


def test_hand_derived_golden_example():
    with open(os.path.join(HERE, "golden", "hand_small_dims.json")) as f:
        gd = json.load(f)
    dm = gd["dims"]
    c = dict(q=torch.tensor(gd["q"]).to(torch.bfloat16),
             cache=torch.tensor(gd["cache_pages"]).to(torch.bfloat16),
             bt=torch.tensor(gd["block_table"], dtype=torch.int32),
             sl=torch.tensor(gd["seq_lens"], dtype=torch.int32),
             wuk=torch.tensor(gd["w_uk"]).to(torch.bfloat16),
             wuv=torch.tensor(gd["w_uv"]).to(torch.bfloat16), scale=gd["scale"],
             dims=(dm["nope"], dm["rope"], dm["lora"], dm["v"], dm["page"], dm["batch"],
                   dm["q_len"], dm["heads"]))
    out, lse = oracle_small(c)
    e = math.e
    assert lse[0] == pytest.approx(math.log(e + 2 * e * e), rel=1e-15)
    assert out[0, 0] == pytest.approx((1 + 4 * e) / (1 + 2 * e), rel=1e-14)


# ---------------------------------------------------------------------------
MUTANTS = {
    "w_uk_transposed": ("wk[(int64_t)k * dl + l]", "wk[(int64_t)l * dn + k]"),
    "rope_dropped": ("for (int k = 0; k < dc; ++k) acc += ql[k]", "for (int k = 0; k < dl; ++k) acc += ql[k]"),
    "causal_mask_dropped": ("const int n = L - T + t + 1;", "const int n = L;"),
    "causal_off_by_one": ("const int n = L - T + t + 1;", "const int n = L - T + t;"),
    "page_row_swapped": ("((int64_t)pg * P + (j % P)) * dc;\n    double acc", "((int64_t)pg * P + (P - 1 - j % P)) * dc;\n    double acc"),
    "w_uv_transposed": ("wv[(int64_t)l * dv + v]);\n    out_row", "wv[(int64_t)v * dl + l]);\n    out_row"),
    "scale_missing": ("s[j] = scale * acc;", "s[j] = acc;"),
    "lse_without_max": ("const double lse = m + log(sum);\n\n  /* step 5", "const double lse = log(sum);\n\n  /* step 5"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, mutant_dir):
    """A plausible mistake planted in a copy of the oracle must break the explicit-form pin."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new, 1)
    d = mutant_dir / name
    d.mkdir()
    (d / "mla_oracle.c").write_text(mutated)
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.h"), d / "mla_oracle.h")
    so = d / "libm.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(d / "mla_oracle.c"), "-lm"], check=True)
    L = ctypes.CDLL(str(so))
    L.mla_oracle_decode.argtypes = oracle.lib().mla_oracle_decode.argtypes
    inp = rand_case(21, 2, [70, 129], 2, 2)
    d_ = oracle.dims_of(inp.q, inp.cache, inp.block_table, inp.w_uk, inp.w_uv)
    n = 2 * 2 * 2
    out = np.empty((n, 128))
    lse = np.empty((n,))
    bits = lambda x: x.contiguous().view(torch.int16)
    rc = L.mla_oracle_decode(ctypes.byref(d_), bits(inp.q).data_ptr(), bits(inp.cache).data_ptr(),
                             inp.block_table.data_ptr(), inp.seq_lens.data_ptr(),
                             bits(inp.w_uk).data_ptr(), bits(inp.w_uv).data_ptr(), inp.scale, 0,
                             None, out.ctypes.data, lse.ctypes.data, None)
    eo, el = explicit_numpy(inp)
    caught = rc != 0 or not (np.allclose(out, eo, rtol=1e-9, atol=1e-11)
                             and np.allclose(lse, el, rtol=1e-11, atol=1e-11))
    assert caught, "planted mistake %s went unnoticed" % name


UP_PROJECT_MUTANTS = {
    "up_project_w_uv_transposed": ("acc += o_lat[l] * bf16_to_double(wv[(int64_t)l * dv + v]);",
                                   "acc += o_lat[l] * bf16_to_double(wv[(int64_t)v * dl + l]);"),
    "up_project_last_latent_dropped": ("for (int l = 0; l < dl; ++l) acc += o_lat[l]",
                                       "for (int l = 0; l < dl - 1; ++l) acc += o_lat[l]"),
    "up_project_head_ignored": ("const uint16_t* wv = w_uv + (int64_t)h * dl * dv;\n  for (int v = 0; v < dv; ++v) {\n    double acc = 0.0;\n    for (int l = 0; l < dl; ++l) acc += o_lat[l]",
                                "const uint16_t* wv = w_uv;\n  for (int v = 0; v < dv; ++v) {\n    double acc = 0.0;\n    for (int l = 0; l < dl; ++l) acc += o_lat[l]"),
}


@pytest.mark.parametrize("name", sorted(UP_PROJECT_MUTANTS))
def test_planted_mistake_in_up_project_fails_its_pin(name, mutant_dir):
    """A mistake planted in mla_oracle_up_project must break the explicit-form pin."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    old, new = UP_PROJECT_MUTANTS[name]
    assert src.count(old) == 1, name
    d = mutant_dir / name
    d.mkdir()
    (d / "mla_oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.h"), d / "mla_oracle.h")
    so = d / "libm.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(d / "mla_oracle.c"), "-lm"], check=True)
    L = ctypes.CDLL(str(so))
    L.mla_oracle_up_project.argtypes = oracle.lib().mla_oracle_up_project.argtypes

    def mutated_up(w_uv, h, o_lat):
        H, lora, v = w_uv.shape
        dm = oracle.Dims(1, 1, H, 0, 0, lora, v, 1, 1, 1)
        ol = np.ascontiguousarray(o_lat, dtype=np.float64)
        res = np.empty((v,))
        assert L.mla_oracle_up_project(ctypes.byref(dm), w_uv.contiguous().view(torch.int16).data_ptr(),
                                       h, ol.ctypes.data, res.ctypes.data) == 0
        return res

    inp = rand_case(22, 2, [70, 129], 2, 3)
    _, _, olat = oracle.decode(inp.q, inp.cache, inp.block_table, inp.seq_lens, inp.w_uk,
                               inp.w_uv, inp.scale, want_olat=True)
    up = _up_project_rows(mutated_up, inp, olat)
    eo, _ = explicit_numpy(inp)
    assert not np.allclose(up, eo, rtol=1e-9, atol=1e-11), "planted mistake %s went unnoticed" % name


# ---------------------------------------------------------------------------
# FP8 weights: E4M3 decoding and the bf16 decompression rule.

def test_e4m3_decoding_matches_torch_float8_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


def test_e4m3_known_values():
    v = oracle.e4m3_to_float(np.array([0x00, 0x38, 0x40, 0x7E, 0x01, 0x08, 0xB8, 0x80, 0x7F, 0xFF],
                                      dtype=np.uint8))
    assert list(v[:7]) == [0.0, 1.0, 2.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0]
    assert v[7] == 0.0 and np.signbit(v[7])
    assert np.isnan(v[8]) and np.isnan(v[9])


def test_fp8_dequant_rounds_to_nearest_even_bf16_and_uses_block_scales():
    # Code 0x38 is 1.0.  With scale 1 + 2^-8 the product lies exactly halfway
    # between the bf16 neighbours 1 and 1 + 2^-7: ties go to the even one, 1.
    # With 1 + 3 * 2^-8 it lies halfway between 1 + 2^-7 and 1 + 2^-6: 1 + 2^-6.
    w8 = torch.full((1, 128, 256), 0x38, dtype=torch.uint8)
    scale = torch.tensor([[[1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]]], dtype=torch.float32)
    d = oracle.dequant_fp8_weight(w8, scale).double()
    assert torch.all(d[0, :, :128] == 1.0) and torch.all(d[0, :, 128:] == 1 + 2.0 ** -6)
    # Each 128 x 128 block takes its own scale.
    w8 = torch.full((2, 256, 128), 0x38, dtype=torch.uint8)
    scale = torch.tensor([[[2.0], [4.0]], [[8.0], [0.5]]], dtype=torch.float32)
    d = oracle.dequant_fp8_weight(w8, scale).double()
    assert torch.all(d[0, :128] == 2.0) and torch.all(d[0, 128:] == 4.0)
    assert torch.all(d[1, :128] == 8.0) and torch.all(d[1, 128:] == 0.5)


def test_fp8_test_weights_round_trip_within_e4m3_precision():
    # The FP8 test inputs: per-block scale = amax / 448, codes rounded to the
    # nearest E4M3 value.  Decompressed, each weight is within half an E4M3
    # step of the original (relative 2^-4 for normal values, 2^-10 of the
    # scale in the subnormal range, plus the bf16 rounding), and each block's
    # largest magnitude maps to code 448.
    from mla_decode_attention_uk_gb300.inputs import make_inputs, quantize_fp8_blockwise
    inp = make_inputs(1, [5], 1, 16, seed=91)
    for w in (inp.w_uk, inp.w_uv):
        codes, scale = quantize_fp8_blockwise(w)
        d = oracle.dequant_fp8_weight(codes, scale).double()
        H, K, M = w.shape
        s = scale.double().repeat_interleave(128, 1).repeat_interleave(128, 2)
        err = (d - w.double()).abs()
        bound = torch.maximum(w.double().abs() * 2.0 ** -4, s * 2.0 ** -10) * 1.01 + \
            d.abs() * 2.0 ** -8
        assert torch.all(err <= bound)
        vals = torch.from_numpy(oracle.e4m3_to_float(codes.numpy()))
        blockmax = vals.abs().reshape(H, K // 128, 128, M // 128, 128).amax(dim=(2, 4))
        assert torch.all(blockmax == 448.0)

"""Seeded synthetic inputs for MLA decode (shared by tests, benchmark and smoke).

This module draws random numbers and lays them out; it holds none of the
attention arithmetic.  Recipe (one torch CPU generator per workload, seeded):

* draw order: seq_lens (when random) -> q -> W_UK -> W_UV -> latent cache ->
  page permutation;
* q [B, T, H, 192] ~ N(0, 1); W_UK [H, 128, 512] ~ N(0, 1/sqrt(128));
  W_UV [H, 512, 128] ~ N(0, 1/sqrt(512)) (std = 1/sqrt(fan_in), fan_in = the
  contracted dim); latent cache [num_pages, 64, 576] ~ N(0, 1) including the
  unused tail rows of partial pages;  all drawn in fp32 and rounded to bf16;
* num_pages = sum_b ceil(L_b / 64), assigned to (b, logical page) in order by
  one randperm(num_pages); block_table entries past a sequence's pages are -1;
* optional spare pages (appended, never referenced) are filled with NaN so a
  stray read shows up in the output;
* softmax scale = 1/sqrt(128 + 64).

Sequence lengths count the q_len new tokens (query t of T sees keys
[0, L - T + t]).
"""
import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

QK_NOPE, QK_ROPE, KV_LORA, V_HEAD, PAGE = 128, 64, 512, 128, 64


@dataclass
class Workload:
    name: str
    batch: int
    q_len: int
    heads: int
    seed: int
    lens: tuple  # ("list", [..]) | ("const", L) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    note: str = ""


WORKLOADS = {
    "tiny": Workload("tiny", 2, 1, 16, 1001, ("list", [17, 80]),
                     "oracle smoke: B=2, L={17,80}, H=16"),
    "tp_shard": Workload("tp_shard", 64, 1, 16, 1002, ("const", 4096),
                         "TP-shard decode: B=64, L=4096, H=16 (memory-bound)"),
    "full_head": Workload("full_head", 128, 1, 128, 1003, ("uniform", 1000, 10000),
                          "full-head decode: B=128, L~U[1000,10000], H=128"),
    "long": Workload("long", 8, 1, 128, 1004, ("const", 32768),
                     "long-context decode: B=8, L=32768, H=128"),
    "mixed_spec": Workload("mixed_spec", 256, 2, 128, 1005, ("lognormal", 800, 1.0, 32, 30000),
                           "mixed batch, q_len=2 causal pair: B=256, L~LogN(ln 800, 1) in [32,30000], H=128"),
    "draft_q8": Workload("draft_q8", 64, 8, 128, 1006, ("lognormal", 2000, 1.0, 64, 30000),
                         "speculative drafts, q_len=8 causal block: B=64, L~LogN(ln 2000, 1) in [64,30000], H=128"),
}


def draw_seq_lens(w: Workload, g: torch.Generator) -> List[int]:
    kind = w.lens[0]
    if kind == "list":
        return list(w.lens[1])
    if kind == "const":
        return [w.lens[1]] * w.batch
    if kind == "uniform":
        lo, hi = w.lens[1], w.lens[2]
        return torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()
    if kind == "lognormal":
        median, sigma, lo, hi = w.lens[1:]
        z = torch.randn(w.batch, generator=g, dtype=torch.float64)
        vals = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
        return [int(v) for v in vals.tolist()]
    raise ValueError(kind)


@dataclass
class Inputs:
    q: torch.Tensor            # [B, T, H, 192] bf16
    cache: torch.Tensor        # [num_pages, 64, 576] bf16
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    w_uk: torch.Tensor         # [H, 128, 512] bf16
    w_uv: torch.Tensor         # [H, 512, 128] bf16
    scale: float
    used_pages: int = 0
    meta: dict = field(default_factory=dict)

    def to(self, device):
        return Inputs(self.q.to(device), self.cache.to(device), self.block_table.to(device),
                      self.seq_lens.to(device), self.w_uk.to(device), self.w_uv.to(device),
                      self.scale, self.used_pages, dict(self.meta))

    @property
    def sum_len(self) -> int:
        return int(self.seq_lens.sum().item())


def _randn_bf16(shape, g, std=1.0, chunk=1 << 26):
    """N(0, std) drawn in fp32 chunk by chunk and rounded to bf16 (bounded temp memory)."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def make_inputs(batch: int, seq_lens: List[int], q_len: int, heads: int, seed: int,
                spare_pages: int = 0, g: Optional[torch.Generator] = None,
                max_pages_per_seq: Optional[int] = None) -> Inputs:
    if g is None:
        g = torch.Generator().manual_seed(seed)
    assert len(seq_lens) == batch
    q = _randn_bf16((batch, q_len, heads, QK_NOPE + QK_ROPE), g)
    w_uk = _randn_bf16((heads, QK_NOPE, KV_LORA), g, 1.0 / math.sqrt(QK_NOPE))
    w_uv = _randn_bf16((heads, KV_LORA, V_HEAD), g, 1.0 / math.sqrt(KV_LORA))
    pages_per = [(L + PAGE - 1) // PAGE for L in seq_lens]
    used = sum(pages_per)
    cache = _randn_bf16((used + spare_pages, PAGE, KV_LORA + QK_ROPE), g)
    if spare_pages:
        cache[used:] = float("nan")
    perm = torch.randperm(used, generator=g).to(torch.int32) if used else torch.empty(0, dtype=torch.int32)
    mp = max(pages_per) if pages_per else 1
    if max_pages_per_seq is not None:
        assert max_pages_per_seq >= mp
        mp = max_pages_per_seq
    block_table = torch.full((batch, max(mp, 1)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = perm[off:off + n]
        off += n
    return Inputs(q, cache, block_table, torch.tensor(seq_lens, dtype=torch.int32), w_uk, w_uv,
                  1.0 / math.sqrt(QK_NOPE + QK_ROPE), used)


def workload_inputs(name: str, spare_pages: int = 0) -> Inputs:
    w = WORKLOADS[name]
    g = torch.Generator().manual_seed(w.seed)
    lens = draw_seq_lens(w, g)
    inp = make_inputs(w.batch, lens, w.q_len, w.heads, w.seed, spare_pages=spare_pages, g=g)
    inp.meta = {"workload": w.name, "note": w.note, "seed": w.seed}
    return inp


def workload_seq_lens(name: str) -> List[int]:
    w = WORKLOADS[name]
    g = torch.Generator().manual_seed(w.seed)
    return draw_seq_lens(w, g)


def quantize_fp8_blockwise(w):
    """FP8 E4M3 weights with one fp32 scale per 128 x 128 block of each head's
    [K, M] matrix: scale = block amax / 448, codes = E4M3(w / scale).  Input
    preparation for the FP8-weight path (the decompression is the method's
    step and lives in the kernels and the oracle).  Returns (uint8 [H, K, M],
    fp32 [H, K/128, M/128])."""
    H, K, M = w.shape
    wf = w.to(torch.float32).reshape(H, K // 128, 128, M // 128, 128)
    amax = wf.abs().amax(dim=(2, 4))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (wf / scale[:, :, None, :, None]).reshape(H, K, M)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.contiguous()


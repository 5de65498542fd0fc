"""Seeded synthetic inputs for paged-E4M3 verification attention.

This module only draws numbers and lays them out; it holds none of the attention arithmetic.
Both the CUDA path and the CPU oracle are fed from it.

Shapes follow "[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Test Plan
(q8 / Hq6 / Hkv1 / D256 per rank, FP16 activations, E4M3 KV, sixteen distinct layer KV
allocations), and the capacity boundary of "[Perf] Reduce DFlash2 long-context verification
decay", Purpose (service capacity 262144; boundary window 261888 input tokens).

Recipe, per layer (seed = seed_base + 10 * layer + tensor id, seed_base = 1000 * config for
configs 0-3 and 5, 40000 + 1000 * q_len + 200 * context index for the tail sweep and
60000 + 1000 * batch for the batched whole-model config; tensor ids: 0 Q,
1 K, 2 V, 3 block-table permutation, 4 boost mask, 5 fill of unused pool bytes):
  * Q ~ N(0, 1) in FP32, rounded to FP16.
  * K, V ~ N(0, 1) in FP32 over the N logical tokens; optionally a seeded fraction of K tokens is
    multiplied by a boost factor (a peaked softmax). Each tensor gets one FP32 scale
    amax(|x|) / 448 and is encoded as E4M3FN codes of x / scale (round to nearest even,
    saturated to +-448) with torch's float8_e4m3fn cast.
  * The physical page of each logical page is a seeded random injective map into the pool; table
    entries past the used pages hold an out-of-range sentinel, and unused pool bytes (including
    the tail slots of the last page) hold seeded random codes, NaN codes included, so that a read
    outside the context shows up.
Inputs can be drawn on any torch device; CPU and CUDA draws differ (different generators), so a
test draws once and hands the same tensors to both sides.
"""
from __future__ import annotations

import dataclasses
import math

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    context: tuple  # N per sequence (counts the q_len drafted tokens)
    q_len: int = 8
    num_q_heads: int = 6
    num_kv_heads: int = 1
    head_dim: int = 256
    page_size: int = 16
    pool_factor: float = 1.0  # physical pages = ceil(pool_factor * logical pages)
    boost_frac: float = 0.0
    boost_factor: float = 1.0
    seed_base: int = 0
    max_context: int = 0  # block-table row covers this many tokens (0: max(context))

    @property
    def batch(self) -> int:
        return len(self.context)

    @property
    def max_ctx(self) -> int:
        return self.max_context or max(self.context)

    @property
    def max_pages_per_seq(self) -> int:
        return max(1, math.ceil(self.max_ctx / self.page_size))

    @property
    def logical_pages(self) -> int:
        return sum(math.ceil(n / self.page_size) for n in self.context)

    @property
    def num_pages(self) -> int:
        return max(1, math.ceil(self.pool_factor * self.logical_pages))

    def kv_bytes_per_layer(self) -> int:
        """Bytes of K plus V the N logical tokens occupy (one code per element)."""
        return 2 * sum(self.context) * self.num_kv_heads * self.head_dim


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def encode_e4m3(x: torch.Tensor):
    """Per-tensor scale amax/448 and E4M3FN codes (uint8) of x/scale; library cast, RNE."""
    amax = x.abs().max().to(torch.float32)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (x.to(torch.float32) / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.reshape(1)


def make_layer(w: Workload, layer: int, device="cpu") -> dict:
    """Inputs of one layer: q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale."""
    dev = torch.device(device)
    seed = w.seed_base + 10 * layer
    B, q_len, Hq, Hkv, D, P = (w.batch, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                               w.page_size)
    q = torch.randn((B, q_len, Hq, D), generator=_gen(dev, seed + 0), device=dev,
                    dtype=torch.float32).to(torch.float16)
    total = sum(w.context)
    k = torch.randn((total, Hkv, D), generator=_gen(dev, seed + 1), device=dev,
                    dtype=torch.float32)
    v = torch.randn((total, Hkv, D), generator=_gen(dev, seed + 2), device=dev,
                    dtype=torch.float32)
    if w.boost_frac > 0 and total > 0:
        u = torch.rand((total,), generator=_gen(dev, seed + 4), device=dev)
        k = torch.where((u < w.boost_frac)[:, None, None], k * w.boost_factor, k)
    if total > 0:
        k_codes, k_scale = encode_e4m3(k)
        v_codes, v_scale = encode_e4m3(v)
    else:
        k_codes = v_codes = torch.empty((0, Hkv, D), dtype=torch.uint8, device=dev)
        k_scale = v_scale = torch.ones((1,), dtype=torch.float32, device=dev)
    num_pages = w.num_pages
    fill = torch.randint(0, 256, (2, num_pages, P, Hkv, D), generator=_gen(dev, seed + 5),
                         device=dev, dtype=torch.int32).to(torch.uint8)
    k_pool, v_pool = fill[0].contiguous(), fill[1].contiguous()
    perm = torch.randperm(num_pages, generator=_gen(dev, seed + 3), device=dev)
    block_table = torch.full((B, w.max_pages_per_seq), num_pages + 7, dtype=torch.int32,
                             device=dev)
    used = 0
    tok0 = 0
    for b, n in enumerate(w.context):
        npg = math.ceil(n / P)
        phys = perm[used:used + npg]
        used += npg
        block_table[b, :npg] = phys.to(torch.int32)
        if n == 0:
            continue
        full = (n // P) * P
        if full:
            kk = k_codes[tok0:tok0 + full].reshape(full // P, P, Hkv, D)
            vv = v_codes[tok0:tok0 + full].reshape(full // P, P, Hkv, D)
            k_pool[phys[:full // P]] = kk
            v_pool[phys[:full // P]] = vv
        if n > full:
            last = phys[full // P]
            k_pool[last, :n - full] = k_codes[tok0 + full:tok0 + n]
            v_pool[last, :n - full] = v_codes[tok0 + full:tok0 + n]
        tok0 += n
    context_lens = torch.tensor(list(w.context), dtype=torch.int32, device=dev)
    return dict(q=q, k_pool=k_pool, v_pool=v_pool, block_table=block_table,
                context_lens=context_lens, k_scale=k_scale.to(torch.float32),
                v_scale=v_scale.to(torch.float32))


# The five synthetic workloads (context lengths and structure as described in the module doc).
def config0() -> Workload:
    """1 layer, N=1024, page 16, block table a permutation of 64 pages."""
    return Workload("c0_q8_ctx1024_p16", layers=1, context=(1024,), seed_base=0)


def config1() -> Workload:
    """16 layers, N=32768, page 16, pool twice the logical pages (injective random map)."""
    return Workload("c1_q8_ctx32768_p16", layers=16, context=(32768,), pool_factor=2.0,
                    seed_base=1000)


def config2() -> Workload:
    """16 layers, N=131072, page 64, 5% of K tokens boosted x4 (peaked softmax)."""
    return Workload("c2_q8_ctx131072_p64_boost", layers=16, context=(131072,), page_size=64,
                    boost_frac=0.05, boost_factor=4.0, seed_base=2000)


def config3() -> Workload:
    """16 layers, N=261888 (capacity boundary window), page 16, 16368 shuffled pages."""
    return Workload("c3_q8_ctx261888_p16", layers=16, context=(261888,), seed_base=3000)


def config4(q_len: int, context: int) -> Workload:
    """Tail-shape sweep point: q_len in 1..8 (longer drafted blocks, up to 16, take the same
    recipe), N in {4096, 65536, 262144}, 16 layers, page 16."""
    return Workload(f"c4_q{q_len}_ctx{context}_p16", layers=16, context=(context,), q_len=q_len,
                    seed_base=40000 + 1000 * q_len + 200 * _ctx_index(context))


def config5() -> Workload:
    """Whole-model head count on one GPU (Hq 24, Hkv 4: the four-way tensor-parallel shard of
    q8 / Hq6 / Hkv1 un-sharded), N=261888, page 16, 16 layers."""
    return Workload("c5_q8_hq24_hkv4_ctx261888_p16", layers=16, context=(261888,),
                    num_q_heads=24, num_kv_heads=4, seed_base=5000)


def config6(batch: int, context: int) -> Workload:
    """A batch of `batch` sequences with whole-model heads (Hq 24, Hkv 4), 16 layers, page 16;
    ragged lengths from `context` down to about half of it in equal steps (multiples of 16)."""
    step = context // (2 * batch) // 16 * 16
    lens = tuple(context - i * step for i in range(batch))
    return Workload(f"c6_b{batch}_q8_hq24_hkv4_ctx{context}_p16", layers=16, context=lens,
                    num_q_heads=24, num_kv_heads=4, seed_base=60000 + 1000 * batch)


TAIL_QLENS = tuple(range(1, 9))
TAIL_CONTEXTS = (4096, 65536, 262144)


def _ctx_index(context: int) -> int:
    return TAIL_CONTEXTS.index(context) if context in TAIL_CONTEXTS else len(TAIL_CONTEXTS)


def all_configs():
    out = [config0(), config1(), config2(), config3()]
    out += [config4(qq, n) for qq in TAIL_QLENS for n in TAIL_CONTEXTS]
    return out

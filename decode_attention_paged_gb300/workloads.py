"""Seeded synthetic inputs for paged MLA decode.

This module only draws random inputs: it holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Every tensor is made on the CPU with ``torch.Generator`` (seeds: q = 1,
k_cache = 2, block_table = 3, seqlens = 4, plus an optional offset), values
~N(0, 1) rounded to bf16, pages of 64 tokens, one KV head of 576 dims whose
first 512 dims are also V.  The shapes are those of the decode workloads the
FlashMLA pages discuss ("[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成
GPU 吞吐", sec. 3 tensor shapes; FlashMLA deep dive, "如何在仓库中验证与复现":
h_q = 128, h_kv = 1, d = 576, dv = 512, block size 64); the benchmark script
they name is not available, so these synthetic workloads stand in for it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

D_QK = 576
D_V = 512
PAGE = 64
SCALE = D_QK ** -0.5


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor            # [b, s_q, h_q, 576] bf16
    k_cache: torch.Tensor      # [num_pages, 64, 1, 576] bf16
    block_table: torch.Tensor  # [b, max_blocks] int32
    cache_seqlens: torch.Tensor  # [b] int32
    softmax_scale: float
    causal: bool

    @property
    def b(self) -> int:
        return self.q.shape[0]

    @property
    def s_q(self) -> int:
        return self.q.shape[1]

    @property
    def h_q(self) -> int:
        return self.q.shape[2]

    def to(self, device) -> "Workload":
        return dataclasses.replace(
            self, q=self.q.to(device), k_cache=self.k_cache.to(device),
            block_table=self.block_table.to(device), cache_seqlens=self.cache_seqlens.to(device))


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, seed: int) -> torch.Tensor:
    # Drawn in chunks of pages so that the peak fp32 footprint stays small.
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    g = _gen(seed)
    step = 1 << 24
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        flat[s:e] = torch.randn(e - s, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def make(name: str, b: int, s_q: int, h_q: int, seqlens: Sequence[int], num_pages: int,
         max_blocks: Optional[int] = None, causal: bool = False, seed_offset: int = 0,
         block_table: Optional[torch.Tensor] = None, scale: float = SCALE,
         d: int = D_QK) -> Workload:
    """Generic workload: block_table = randperm(num_pages)[:b*max_blocks].view(b, max_blocks)
    unless given; q and cache rows of d dims (576 unless given)."""
    seqlens = torch.tensor(list(seqlens), dtype=torch.int32)
    assert seqlens.numel() == b
    need = max(1, max((int(x) + PAGE - 1) // PAGE for x in seqlens.tolist()) if b else 1)
    if max_blocks is None:
        max_blocks = need
    assert max_blocks >= need
    if block_table is None:
        assert num_pages >= b * max_blocks, "page pool too small for a permutation"
        perm = torch.randperm(num_pages, generator=_gen(3 + seed_offset)).to(torch.int32)
        block_table = perm[: b * max_blocks].view(b, max_blocks).contiguous()
    q = _randn_bf16((b, s_q, h_q, d), 1 + seed_offset)
    k_cache = _randn_bf16((num_pages, PAGE, 1, d), 2 + seed_offset)
    return Workload(name, q, k_cache, block_table.to(torch.int32), seqlens, scale, causal)


def tiny(seed_offset: int = 0) -> Workload:
    """batch 1, s_q 1, h_q 16, 4 pages, identity block table, L = 256, non-causal."""
    bt = torch.arange(4, dtype=torch.int32).view(1, 4)
    return make("tiny b1 s_q1 h_q16 L256", 1, 1, 16, [256], 4, 4, block_table=bt,
                seed_offset=seed_offset)


def memory_bound(seed_offset: int = 0) -> Workload:
    """batch 64, s_q 1, h_q 16, every L = 4096, 4096 pages permuted."""
    return make("memory-bound b64 s_q1 h_q16 L4096", 64, 1, 16, [4096] * 64, 4096, 64,
                seed_offset=seed_offset)


def compute_bound(seed_offset: int = 0) -> Workload:
    """batch 64, s_q 1, h_q 128, L ~ U[1, 8192] (seed 4), 64*128 pages permuted."""
    L = torch.randint(1, 8193, (64,), generator=_gen(4 + seed_offset), dtype=torch.int64).tolist()
    return make("compute-bound b64 s_q1 h_q128 L~U[1,8192]", 64, 1, 128, L, 64 * 128, 128,
                seed_offset=seed_offset)


def mtp(seed_offset: int = 0) -> Workload:
    """batch 128, s_q 2, h_q 128, causal within the 2 query tokens, L = 4096."""
    return make("MTP b128 s_q2 h_q128 causal L4096", 128, 2, 128, [4096] * 128, 8192, 64,
                causal=True, seed_offset=seed_offset)


def long_ragged(seed_offset: int = 0) -> Workload:
    """batch 8, s_q 1, h_q 64, L = 1 .. 65536, 8192 pages, 1024 blocks per row."""
    L = [1, 64, 1000, 8191, 16384, 32768, 49152, 65536]
    return make("long ragged b8 s_q1 h_q64 L<=65536", 8, 1, 64, L, 8192, 1024,
                seed_offset=seed_offset)


CONFIGS = {
    "tiny": tiny,
    "memory_bound": memory_bound,
    "compute_bound": compute_bound,
    "mtp": mtp,
    "long_ragged": long_ragged,
}
CONFIG_ORDER = ["tiny", "memory_bound", "compute_bound", "mtp", "long_ragged"]


def random_case(seed: int, b: int, s_q: int, h_q: int, seqlens: Sequence[int], causal: bool,
                extra_pages: int = 3, d: int = D_QK) -> Workload:
    """A small random case whose pool has a few pages no sequence references
    (rows of d dims; softmax_scale d^-0.5)."""
    need = max(1, max((int(x) + PAGE - 1) // PAGE for x in seqlens))
    return make(f"random seed{seed}", b, s_q, h_q, seqlens, b * need + extra_pages, need,
                causal=causal, seed_offset=10 * seed, d=d,
                scale=SCALE if d == D_QK else d ** -0.5)


def flops(seqlens: Sequence[int], s_q: int, h_q: int, causal: bool) -> int:
    """Algorithmic FLOPs: 2*(576+512) per (query row, visible key)."""
    total = 0
    for L in seqlens:
        L = int(L)
        for s in range(s_q):
            vis = max(0, min(L, L - s_q + s + 1)) if causal else L
            total += vis * h_q
    return total * 2 * (D_QK + D_V)


def hbm_bytes(seqlens: Sequence[int], s_q: int, h_q: int) -> int:
    """Algorithmic bytes: every cached token once (1152 B), q in, out and lse out."""
    rows = len(seqlens) * s_q * h_q
    return sum(int(L) for L in seqlens) * D_QK * 2 + rows * (D_QK * 2 + D_V * 2 + 4)


def unit_work(seqlens: Sequence[int], s_q: int, h_q: int, causal: bool, units) -> tuple:
    """(bytes, FLOPs) of a sample of (request, row) units, row = s * h_q + h:
    each row's share of its request's cached tokens (1152 B per token, spread
    evenly over the request's s_q * h_q rows), its q / out / lse bytes, and
    2 * (576 + 512) FLOPs per visible key.  Summed over every unit of a
    workload this is hbm_bytes and flops."""
    R = s_q * h_q
    nbytes = 0.0
    nflops = 0
    for i, rho in units:
        L = int(seqlens[int(i)])
        s = int(rho) // h_q
        vis = max(0, min(L, L - s_q + s + 1)) if causal else L
        nbytes += L * D_QK * 2 / R + (D_QK * 2 + D_V * 2 + 4)
        nflops += vis * 2 * (D_QK + D_V)
    return nbytes, nflops


# ---------------------------------------------------------------- sparse decode
# Sparse decode ("[DeepSeek-3] FlashMLA", sec. 11): every query token attends
# to its own list of topk cache positions, index = physical page * 64 + offset.
# The selector that makes the lists is outside the path; here each list is
# topk distinct tokens of the request's own context, drawn at random (seeded,
# in random order), optionally with some slots turned into padding (-1).

@dataclasses.dataclass
class SparseWorkload:
    name: str
    q: torch.Tensor        # [b, s_q, h_q, 576] bf16
    k_cache: torch.Tensor  # [num_pages, 64, 1, 576] bf16
    indices: torch.Tensor  # [b, s_q, topk] int32
    softmax_scale: float

    @property
    def b(self) -> int:
        return self.q.shape[0]

    @property
    def s_q(self) -> int:
        return self.q.shape[1]

    @property
    def h_q(self) -> int:
        return self.q.shape[2]

    @property
    def topk(self) -> int:
        return self.indices.shape[2]

    @property
    def num_tokens(self) -> int:
        return self.k_cache.shape[0] * PAGE

    def to(self, device) -> "SparseWorkload":
        return dataclasses.replace(self, q=self.q.to(device), k_cache=self.k_cache.to(device),
                                   indices=self.indices.to(device))


def make_sparse(name: str, b: int, s_q: int, h_q: int, topk: int, context: int,
                pad_frac: float = 0.0, extra_pages: int = 0, seed_offset: int = 0,
                scale: float = SCALE) -> SparseWorkload:
    """Request i owns `context` tokens on ceil(context / 64) pages of a random
    permutation of the pool (seed 3); list (i, s) holds min(topk, context)
    distinct tokens of that context in random order (seed 5), the rest of its
    topk slots -1; then a fraction pad_frac of all slots is set to -1 (seed 6)."""
    npg = (context + PAGE - 1) // PAGE
    num_pages = b * npg + extra_pages
    perm = torch.randperm(num_pages, generator=_gen(3 + seed_offset)).to(torch.int64)
    bt = perm[: b * npg].view(b, npg)
    g = _gen(5 + seed_offset)
    k = min(topk, context)
    idx = torch.full((b, s_q, topk), -1, dtype=torch.int64)
    for i in range(b):
        for s in range(s_q):
            t = torch.randperm(context, generator=g)[:k]
            idx[i, s, :k] = bt[i, t // PAGE] * PAGE + t % PAGE
    if pad_frac > 0:
        drop = torch.rand((b, s_q, topk), generator=_gen(6 + seed_offset)) < pad_frac
        idx[drop] = -1
    q = _randn_bf16((b, s_q, h_q, D_QK), 1 + seed_offset)
    k_cache = _randn_bf16((num_pages, PAGE, 1, D_QK), 2 + seed_offset)
    return SparseWorkload(name, q, k_cache, idx.to(torch.int32).contiguous(), scale)


def sparse(seed_offset: int = 0) -> SparseWorkload:
    """batch 128, s_q 2, h_q 128, topk 2048 of a 4096-token context per request."""
    return make_sparse("sparse b128 s_q2 h_q128 topk2048 ctx4096", 128, 2, 128, 2048, 4096,
                       seed_offset=seed_offset)


def random_sparse_case(seed: int, b: int, s_q: int, h_q: int, topk: int, context: int,
                       pad_frac: float = 0.0) -> SparseWorkload:
    return make_sparse(f"sparse seed{seed}", b, s_q, h_q, topk, context, pad_frac,
                       extra_pages=3, seed_offset=10 * seed)


def sparse_flops(indices: torch.Tensor, h_q: int) -> int:
    """Algorithmic FLOPs: 2*(576+512) per (query row, listed key); padding adds none."""
    return int((indices >= 0).sum().item()) * h_q * 2 * (D_QK + D_V)


def sparse_hbm_bytes(indices: torch.Tensor, h_q: int) -> int:
    """Algorithmic bytes: each listed key row once per list (1152 B), q in, out and lse out."""
    b, s_q, _ = indices.shape
    rows = b * s_q * h_q
    return int((indices >= 0).sum().item()) * D_QK * 2 + rows * (D_QK * 2 + D_V * 2 + 4)


# ------------------------------------------------------------ FP8 KV cache
# FP8 cache layout ("[DeepSeek-3] FlashMLA", sec. 12): 656 bytes per token,
# 512 float8_e4m3 latent values, 4 fp32 scales (one per 128 latent values),
# then the 64 RoPE values in bf16.  The decode path only reads this layout;
# writing it is the cache writer's job, done here with torch's own float8
# conversion so that synthetic FP8 caches can be drawn.
FP8_ROW_BYTES = 656
E4M3_MAX = 448.0


def fp8_cache(k_cache: torch.Tensor) -> torch.Tensor:
    """[pages, 64, 1, 576] bf16 -> [pages, 64, 1, 656] uint8: per 128-value tile
    scale = amax / 448, latent = e4m3(x / scale), RoPE copied."""
    assert k_cache.dtype == torch.bfloat16 and k_cache.shape[-1] == D_QK
    lead = k_cache.shape[:-1]
    x = k_cache[..., :512].float().reshape(*lead, 4, 128)
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q8 = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    out = torch.empty(*lead, FP8_ROW_BYTES, dtype=torch.uint8)
    out[..., :512] = q8.reshape(*lead, 512).view(torch.uint8)
    out[..., 512:528] = scale.reshape(*lead, 4).contiguous().view(torch.uint8)
    out[..., 528:] = k_cache[..., 512:].contiguous().view(torch.uint8)
    return out


@dataclasses.dataclass
class Fp8Workload:
    """A decode workload whose cache is stored in the FP8 layout."""
    name: str
    q: torch.Tensor            # [b, s_q, h_q, 576] bf16
    k_cache: torch.Tensor      # [num_pages, 64, 1, 656] uint8
    block_table: torch.Tensor  # [b, max_blocks] int32
    cache_seqlens: torch.Tensor
    softmax_scale: float
    causal: bool

    @property
    def b(self) -> int:
        return self.q.shape[0]

    @property
    def s_q(self) -> int:
        return self.q.shape[1]

    @property
    def h_q(self) -> int:
        return self.q.shape[2]

    def to(self, device) -> "Fp8Workload":
        return dataclasses.replace(
            self, q=self.q.to(device), k_cache=self.k_cache.to(device),
            block_table=self.block_table.to(device), cache_seqlens=self.cache_seqlens.to(device))


def as_fp8(w: Workload) -> Fp8Workload:
    return Fp8Workload(w.name + " fp8", w.q, fp8_cache(w.k_cache), w.block_table,
                       w.cache_seqlens, w.softmax_scale, w.causal)


def memory_bound_fp8(seed_offset: int = 0) -> Fp8Workload:
    """The memory-bound workload with its cache in the FP8 layout."""
    return as_fp8(memory_bound(seed_offset))


def fp8_hbm_bytes(seqlens: Sequence[int], s_q: int, h_q: int) -> int:
    """Algorithmic bytes with the FP8 cache: 656 B per cached token read once,
    plus q in, out and lse out."""
    rows = len(seqlens) * s_q * h_q
    return sum(int(L) for L in seqlens) * FP8_ROW_BYTES + rows * (D_QK * 2 + D_V * 2 + 4)


# ------------------------------------------------------------ h_kv > 1
@dataclasses.dataclass
class HeadsWorkload:
    """Decode with several cache heads: k_cache [pages, 64, h_kv, 576]."""
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    softmax_scale: float
    causal: bool

    @property
    def b(self) -> int:
        return self.q.shape[0]

    @property
    def s_q(self) -> int:
        return self.q.shape[1]

    @property
    def h_q(self) -> int:
        return self.q.shape[2]

    @property
    def h_kv(self) -> int:
        return self.k_cache.shape[2]

    def to(self, device) -> "HeadsWorkload":
        return dataclasses.replace(
            self, q=self.q.to(device), k_cache=self.k_cache.to(device),
            block_table=self.block_table.to(device), cache_seqlens=self.cache_seqlens.to(device))


def gqa(seed_offset: int = 0) -> HeadsWorkload:
    """batch 32, s_q 1, h_q 64, h_kv 4 (groups of 16 heads), every L = 4096,
    2048 pages permuted: 604 MB of cache."""
    b, h_q, h_kv, L = 32, 64, 4, 4096
    nb = L // PAGE
    perm = torch.randperm(b * nb, generator=_gen(3 + seed_offset)).to(torch.int32)
    bt = perm.view(b, nb).contiguous()
    q = _randn_bf16((b, 1, h_q, D_QK), 1 + seed_offset)
    kc = _randn_bf16((b * nb, PAGE, h_kv, D_QK), 2 + seed_offset)
    return HeadsWorkload("GQA b32 s_q1 h_q64 h_kv4 L4096", q, kc, bt,
                         torch.full((b,), L, dtype=torch.int32), SCALE, False)


def heads_hbm_bytes(seqlens: Sequence[int], s_q: int, h_q: int, h_kv: int) -> int:
    """Algorithmic bytes with h_kv cache heads: 1152 B per cached token and head."""
    rows = len(seqlens) * s_q * h_q
    return sum(int(L) for L in seqlens) * h_kv * D_QK * 2 + rows * (D_QK * 2 + D_V * 2 + 4)

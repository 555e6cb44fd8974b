"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and builds index structures (cu_seqlens,
block tables); it holds none of the attention arithmetic.  Every tensor is
drawn on the CPU from ``torch.Generator().manual_seed(seed)`` as float32
N(0, 1) in the order q, k, v (then the cache) and rounded to bfloat16, so the
oracle (which upcasts the same bf16 tensors exactly) and the GPU kernels see
identical numbers.

The workloads follow the shapes the pages run the attention backends on:
diffusion-transformer self- and cross-attention (vllm-omni ``flash_attn.py``,
dense and packed routes), packed prefill of several documents, and paged
decode over a ``(2, num_blocks, 128, Hkv, D)`` cache (vllm-ascend
``attention_v1.py``, ``forward_paged_attention``).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 128  # the only paged block size (``AscendAttentionBackend.get_supported_block_size``)
HEAD_SIZES = (64, 96, 128, 192, 256)  # ``FlashAttentionBackend.get_supported_head_sizes``


def randn_bf16(gen: torch.Generator, *shape: int) -> torch.Tensor:
    """N(0,1) float32 draw from ``gen``, rounded to bf16 (CPU tensor)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def randn_bf16_chunked(gen: torch.Generator, shape, chunk_rows: int = 64) -> torch.Tensor:
    """Like ``randn_bf16`` for very large tensors: draws along dim 0 in chunks
    so the float32 staging buffer stays small.  Same stream of numbers for a
    given (seed, shape, chunk_rows)."""
    out = torch.empty(*shape, dtype=torch.bfloat16)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        out[r0:r1] = torch.randn(r1 - r0, *shape[1:], generator=gen, dtype=torch.float32)
    return out


def default_scale(head_dim: int) -> float:
    """1/sqrt(head_size) (vllm-omni ``fastvideo_vsa.py``: ``head_size ** -0.5``)."""
    return 1.0 / math.sqrt(head_dim)


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


@dataclass
class Dense:
    """Fixed-length batch: q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D]."""
    name: str
    B: int
    Sq: int
    Sk: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    seed: int
    scale: float = 0.0

    def __post_init__(self):
        if not self.scale:
            self.scale = default_scale(self.D)

    def make(self):
        g = torch.Generator().manual_seed(self.seed)
        q = randn_bf16(g, self.B, self.Sq, self.Hq, self.D)
        k = randn_bf16(g, self.B, self.Sk, self.Hkv, self.D)
        v = randn_bf16(g, self.B, self.Sk, self.Hkv, self.D)
        return q, k, v

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask lets through, per (batch, head)."""
        if not self.causal:
            return self.Sq * self.Sk
        off = self.Sk - self.Sq
        return sum(max(0, min(self.Sk, i + off + 1)) for i in range(self.Sq))

    def flops(self) -> float:
        """4*D per visible score: 2*D for q.k and 2*D for p.v."""
        return 4.0 * self.D * self.B * self.Hq * self.visible_pairs()


@dataclass
class Varlen:
    """Packed documents: q [Tq, Hq, D], k/v [Tk, Hkv, D], cu_seqlens int32."""
    name: str
    lens_q: list
    lens_k: list
    Hq: int
    Hkv: int
    D: int
    causal: bool
    seed: int
    scale: float = 0.0

    def __post_init__(self):
        if not self.scale:
            self.scale = default_scale(self.D)

    @property
    def Tq(self):
        return int(sum(self.lens_q))

    @property
    def Tk(self):
        return int(sum(self.lens_k))

    def make(self):
        g = torch.Generator().manual_seed(self.seed)
        q = randn_bf16(g, self.Tq, self.Hq, self.D)
        k = randn_bf16(g, self.Tk, self.Hkv, self.D)
        v = randn_bf16(g, self.Tk, self.Hkv, self.D)
        return q, k, v, cu_from_lengths(self.lens_q), cu_from_lengths(self.lens_k)

    def visible_pairs(self) -> int:
        total = 0
        for lq, lk in zip(self.lens_q, self.lens_k):
            if not self.causal:
                total += lq * lk
            else:
                off = lk - lq
                # rows i in [0, lq): visible keys min(lk, max(0, i + off + 1))
                total += sum(max(0, min(lk, i + off + 1)) for i in range(lq))
        return total

    def flops(self) -> float:
        return 4.0 * self.D * self.Hq * self.visible_pairs()


@dataclass
class Paged:
    """Paged-KV decode: q [S, Hq, D], cache [2, nb, 128, Hkv, D] bf16,
    block_table [S, max_blocks] int32 (unused entries -1), seq_lens [S] int32.
    Physical blocks are a seeded random permutation, handed out to the
    sequences in consecutive slices."""
    name: str
    seq_lens: list
    Hq: int
    Hkv: int
    D: int
    seed: int
    max_blocks_per_seq: int = 0
    scale: float = 0.0
    block_size: int = BLOCK_SIZE
    extra_blocks: int = 0  # spare physical blocks nobody points at

    def __post_init__(self):
        if not self.scale:
            self.scale = default_scale(self.D)
        need = max([-(-n // self.block_size) for n in self.seq_lens] + [1])
        if not self.max_blocks_per_seq:
            self.max_blocks_per_seq = need
        if self.max_blocks_per_seq < need:
            raise ValueError("max_blocks_per_seq too small for the longest sequence")

    @property
    def num_blocks(self) -> int:
        return sum(-(-n // self.block_size) for n in self.seq_lens) + self.extra_blocks

    def block_table(self) -> torch.Tensor:
        g = torch.Generator().manual_seed(self.seed)
        perm = torch.randperm(self.num_blocks, generator=g).to(torch.int32)
        bt = torch.full((len(self.seq_lens), self.max_blocks_per_seq), -1, dtype=torch.int32)
        at = 0
        for s, n in enumerate(self.seq_lens):
            nblk = -(-n // self.block_size)
            bt[s, :nblk] = perm[at:at + nblk]
            at += nblk
        return bt

    def make(self, chunk_rows: int = 64):
        """Returns q, kv_cache, block_table, seq_lens (CPU tensors)."""
        bt = self.block_table()
        g = torch.Generator().manual_seed(self.seed + 1000)
        q = randn_bf16(g, len(self.seq_lens), self.Hq, self.D)
        cache = randn_bf16_chunked(
            g, (2 * self.num_blocks, self.block_size, self.Hkv, self.D), chunk_rows
        ).view(2, self.num_blocks, self.block_size, self.Hkv, self.D)
        return q, cache, bt, torch.tensor(self.seq_lens, dtype=torch.int32)

    def context_tokens(self) -> int:
        return int(sum(self.seq_lens))

    def algorithmic_bytes(self, out_bytes_per_elem: int = 4, with_lse: bool = True) -> int:
        """Bytes one decode call must move at minimum: every context token's K
        and V row for every KV head (read once, shared by the GQA group), the
        block-table entries in use, seq_lens, q, and the outputs."""
        s = len(self.seq_lens)
        kv = 2 * self.context_tokens() * self.Hkv * self.D * 2
        bt = 4 * sum(-(-n // self.block_size) for n in self.seq_lens) + 4 * s
        q = s * self.Hq * self.D * 2
        out = s * self.Hq * self.D * out_bytes_per_elem + (4 * s * self.Hq if with_lse else 0)
        return kv + bt + q + out

    def flops(self) -> float:
        return 4.0 * self.D * self.Hq * self.context_tokens()


@dataclass
class CacheWrite:
    """New tokens' K/V [T, Hkv, D] bf16 written into a paged cache
    [2, nb, block_size, Hkv, D] through slot_mapping [T] int32.  Each
    document's tokens take consecutive slots of its blocks; the physical
    blocks are a seeded random permutation (as in ``Paged``)."""
    name: str
    lens: list
    Hkv: int
    D: int
    seed: int
    block_size: int = BLOCK_SIZE

    @property
    def tokens(self) -> int:
        return int(sum(self.lens))

    @property
    def num_blocks(self) -> int:
        return sum(-(-n // self.block_size) for n in self.lens)

    def make(self, chunk_rows: int = 256):
        """Returns key, value, slot_mapping (CPU tensors) and the cache shape."""
        g = torch.Generator().manual_seed(self.seed)
        perm = torch.randperm(self.num_blocks, generator=g)
        slots, at = [], 0
        for n in self.lens:
            nblk = -(-n // self.block_size)
            blocks = perm[at:at + nblk]
            t = torch.arange(n)
            slots.append(blocks[t // self.block_size] * self.block_size + t % self.block_size)
            at += nblk
        key = randn_bf16_chunked(g, (self.tokens, self.Hkv, self.D), chunk_rows)
        value = randn_bf16_chunked(g, (self.tokens, self.Hkv, self.D), chunk_rows)
        return key, value, torch.cat(slots).to(torch.int32), (2, self.num_blocks, self.block_size, self.Hkv, self.D)

    def algorithmic_bytes(self) -> int:
        """K and V read once and written once, plus the slot list."""
        return 2 * 2 * self.tokens * self.Hkv * self.D * 2 + 4 * self.tokens


def prefill_kv_write() -> CacheWrite:
    """The K/V of the packed causal GQA workload (8 documents, 8 KV heads,
    D=128) stored into a paged cache, as a prefill step does before decode."""
    lens = doc_lengths_capped(2, 8, 512, 8192, 32768)
    return CacheWrite("kv_write_8docs_kv8_d128", lens, 8, 128, seed=13)


@dataclass
class PagedPrefill:
    """q_len new query tokens per sequence (the last of its context) against
    a paged cache: the context (cache, block table) is the ``Paged`` one of
    the same sizes and seed; q [sum q_len, Hq, D] packed by cu_seqlens_q."""
    name: str
    seq_lens: list
    q_lens: list
    Hq: int
    Hkv: int
    D: int
    seed: int
    causal: bool = True

    def paged(self) -> Paged:
        return Paged(self.name, self.seq_lens, self.Hq, self.Hkv, self.D, seed=self.seed)

    @property
    def scale(self) -> float:
        return default_scale(self.D)

    def make(self, chunk_rows: int = 256):
        """Returns q, kv_cache, block_table, seq_lens, cu_seqlens_q (CPU tensors)."""
        _, cache, bt, sl = self.paged().make(chunk_rows)
        q = randn_bf16(torch.Generator().manual_seed(self.seed + 2000), sum(self.q_lens), self.Hq, self.D)
        return q, cache, bt, sl, cu_from_lengths(self.q_lens)

    def visible_pairs(self) -> int:
        total = 0
        for lk, lq in zip(self.seq_lens, self.q_lens):
            if not self.causal:
                total += lq * lk
            else:  # query i sees keys j <= i + lk - lq
                total += sum(max(0, min(lk, i + lk - lq + 1)) for i in range(lq))
        return total

    def flops(self) -> float:
        return 4.0 * self.D * self.Hq * self.visible_pairs()


def chunked_prefill() -> PagedPrefill:
    """16 sequences with contexts U[2048, 32768] (seed 14) whose last 512
    tokens are a new prefill chunk, 32 query / 8 KV heads, D=128, causal."""
    g = torch.Generator().manual_seed(14)
    lens = _uniform_int(g, 2048, 32768, 16)
    return PagedPrefill("chunked_prefill_16seq_q512_h32kv8_d128", lens, [512] * 16, 32, 8, 128, seed=14)


def spec_decode() -> PagedPrefill:
    """64 sequences with contexts U[1024, 32768] (seed 3, as the decode
    workload) verifying 16 draft tokens each, 32 query / 8 KV heads, D=128."""
    g = torch.Generator().manual_seed(3)
    lens = _uniform_int(g, 1024, 32768, 64)
    return PagedPrefill("spec_decode_64seq_q16_h32kv8_d128", lens, [16] * 64, 32, 8, 128, seed=3)


@dataclass
class Masked:
    """Padded batch q/k/v [B, S, H, D] with a [B, S] padding mask keeping the
    first lens[b] tokens of row b (the structural padding at the end of a
    packed video-latent batch)."""
    name: str
    lens: list
    S: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    seed: int

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def scale(self) -> float:
        return default_scale(self.D)

    def make(self):
        g = torch.Generator().manual_seed(self.seed)
        q = randn_bf16(g, self.B, self.S, self.Hq, self.D)
        k = randn_bf16(g, self.B, self.S, self.Hkv, self.D)
        v = randn_bf16(g, self.B, self.S, self.Hkv, self.D)
        mask = torch.zeros(self.B, self.S, dtype=torch.uint8)
        for b, n in enumerate(self.lens):
            mask[b, :n] = 1
        return q, k, v, mask

    def flops(self) -> float:
        pairs = sum((n * (n + 1)) // 2 if self.causal else n * n for n in self.lens)
        return 4.0 * self.D * self.Hq * pairs


def masked_dit() -> Masked:
    """The DiT self-attention shape, B=2, S=4096, 24 heads, D=128, with the
    second row padded after 3072 tokens."""
    return Masked("masked_dit_b2_s4096_h24_d128_len4096_3072", [4096, 3072], 4096, 24, 24, 128, False, seed=15)


@dataclass
class Vsa:
    """One sequence for block-sparse video attention: prefix segments, then a
    T x H x W video latent grid; q [S, Hq, D], k / v [S, Hkv, D]; each video
    query block keeps its topk best video key blocks plus the prefix."""
    name: str
    prefix: list
    video: tuple
    Hq: int
    Hkv: int
    D: int
    topk: int
    seed: int

    @property
    def tokens(self) -> int:
        return sum(self.prefix) + self.video[0] * self.video[1] * self.video[2]

    @property
    def scale(self) -> float:
        return default_scale(self.D)

    def make(self):
        g = torch.Generator().manual_seed(self.seed)
        q = randn_bf16(g, self.tokens, self.Hq, self.D)
        k = randn_bf16(g, self.tokens, self.Hkv, self.D)
        v = randn_bf16(g, self.tokens, self.Hkv, self.D)
        return q, k, v


def vsa_video(frames: int = 21) -> Vsa:
    """A 512-token prefix and a 21 x 45 x 80 video latent grid (76112 tokens,
    1448 blocks), 40 heads, D=128, the page's default topk of 64 blocks.
    ``frames`` shortens the grid's T axis (smaller profiling captures)."""
    return Vsa(f"vsa_p512_t{frames}h45w80_h40_d128_top64", [512], (frames, 45, 80), 40, 40, 128, 64, seed=16)

def _uniform_int(gen: torch.Generator, lo: int, hi: int, n: int) -> list:
    """n integers uniform in [lo, hi] (inclusive)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def doc_lengths_capped(seed: int, n: int, lo: int, hi: int, cap: int) -> list:
    """n lengths uniform in [lo, hi], re-drawn as a whole until their sum <= cap."""
    g = torch.Generator().manual_seed(seed)
    while True:
        lens = _uniform_int(g, lo, hi, n)
        if sum(lens) <= cap:
            return lens


# ---------------------------------------------------------------------------
# The five workloads (parity cases and bench lines) and small variants.
# ---------------------------------------------------------------------------

def tiny_varlen() -> Varlen:
    """2 documents of 37 and 91 tokens, 4 heads, D=64, non-causal, seed 0."""
    return Varlen("tiny_varlen_37_91_h4_d64", [37, 91], [37, 91], 4, 4, 64, False, seed=0)


def dit_self() -> Dense:
    """Diffusion-transformer self-attention: B=2, S=4096, 24 heads, D=128."""
    return Dense("dit_self_b2_s4096_h24_d128", 2, 4096, 4096, 24, 24, 128, False, seed=1)


def varlen_causal_gqa() -> Varlen:
    """8 packed documents, lengths U[512, 8192] capped at 32768 tokens in
    total (seed 2), 32 query / 8 KV heads, D=128, causal, tensors seed 12."""
    lens = doc_lengths_capped(2, 8, 512, 8192, 32768)
    return Varlen("varlen_causal_gqa_8docs_h32kv8_d128", lens, lens, 32, 8, 128, True, seed=12)


def paged_decode() -> Paged:
    """64 sequences, context lengths U[1024, 32768] (seed 3), 32 query /
    8 KV heads, D=128, block size 128."""
    g = torch.Generator().manual_seed(3)
    lens = _uniform_int(g, 1024, 32768, 64)
    return Paged("paged_decode_64seq_h32kv8_d128", lens, 32, 8, 128, seed=3,
                 max_blocks_per_seq=-(-32768 // BLOCK_SIZE))


def cross_attn() -> Dense:
    """16384 video-latent queries attend 512 text tokens, 40 heads, D=128."""
    return Dense("cross_sq16384_sk512_h40_d128", 1, 16384, 512, 40, 40, 128, False, seed=4)


def head_sweep(d: int) -> Dense:
    """Dense self-attention, S=8192, 16 heads, head_dim d in {64, 96, 192, 256}."""
    return Dense(f"self_s8192_h16_d{d}", 1, 8192, 8192, 16, 16, d, False, seed=5)


def all_workloads():
    return [tiny_varlen(), dit_self(), varlen_causal_gqa(), paged_decode(), cross_attn()] + [
        head_sweep(d) for d in (64, 96, 192, 256)
    ]

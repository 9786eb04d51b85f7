"""Seeded synthetic decode workloads.

Structure (context lengths, physical block placement, prefix-sharing groups)
is drawn with ``numpy.random.Generator(PCG64(seed))``; values (Q, K, V, new
K/V) with a ``torch.Generator`` seeded the same way on the device the tensors
live on.  Integer ranges are inclusive.

Pool layout is ``[num_blocks, num_kv_heads, block_size, head_dim]`` for both K
and V; a block table row lists physical block ids in logical order and pads
unused entries with -1 (or with an out-of-range poison id when asked).

The workloads follow the decode shapes named on the pages' subject: a
Llama-3-8B-shaped layer (32 query heads / 8 KV heads, head_dim 128), a
Llama-3-70B-shaped layer (64 / 8, head_dim 128), a 70B-style multi-head layer
(64 / 64) at 32K context, and parallel sampling that shares a prompt's
blocks across 8 samples per group (PagedAttention page, "Copy-on-Write
Memory Sharing").
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    seed: int
    ctx_fixed: Optional[tuple] = None      # explicit per-sequence lengths
    ctx_range: Optional[tuple] = None      # inclusive uniform range
    ctx_append: int = 0                    # tokens appended this step, included in the length
    pool_blocks: Optional[int] = None      # explicit pool size
    pool_factor: float = 1.1               # else pool = ceil(factor * blocks in use)
    description: str = ""

    @property
    def max_context_len(self) -> int:
        if self.ctx_fixed is not None:
            return max(self.ctx_fixed) + self.ctx_append
        return self.ctx_range[1] + self.ctx_append

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-self.max_context_len // self.block_size))


CONFIGS = {
    "tiny": DecodeConfig(
        name="tiny", num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64,
        block_size=16, dtype="fp16", seed=1001, ctx_fixed=(17, 33, 64, 100),
        pool_blocks=64,
        description="4 seqs, ctx {17,33,64,100}, 8 q = 8 kv heads, d 64, block 16, pool 64"),
    "llama3_8b_b64": DecodeConfig(
        name="llama3_8b_b64", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
        block_size=16, dtype="bf16", seed=1002, ctx_range=(512, 4096), ctx_append=1,
        description="Llama-3-8B-shaped layer: batch 64, 32/8 heads, d 128, block 16, "
                    "ctx U[512,4096] + 1 appended token"),
    "llama3_70b_b256": DecodeConfig(
        name="llama3_70b_b256", num_seqs=256, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, dtype="bf16", seed=1003, ctx_range=(1024, 8192),
        description="Llama-3-70B-shaped layer: batch 256, 64/8 heads, d 128, block 16, "
                    "ctx U[1024,8192] (the newest token included), pool 1.1x"),
    "long_mha_32k": DecodeConfig(
        name="long_mha_32k", num_seqs=32, num_q_heads=64, num_kv_heads=64, head_dim=128,
        block_size=16, dtype="bf16", seed=1004, ctx_fixed=(32768,) * 32,
        pool_blocks=65536,
        description="70B-style MHA layer: batch 32, 64/64 heads, d 128, block 16, ctx 32768"),
}


@dataclass
class DecodeCase:
    cfg: DecodeConfig
    context_lens: np.ndarray           # int32 [N]
    block_tables: np.ndarray           # int32 [N, MB], -1 (or poison) past the last block
    num_blocks: int
    scale: float
    q: Optional[torch.Tensor] = None       # [N, Hq, d]
    k_pool: Optional[torch.Tensor] = None  # [NB, Hkv, B, d]
    v_pool: Optional[torch.Tensor] = None
    k_new: Optional[torch.Tensor] = None   # [N, Hkv, d]: the newest token of each sequence
    v_new: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)


def _torch_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_values(shape, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    """Standard-normal values in the storage dtype (drawn in fp32, rounded
    once), generated in slices along the first dimension so large pools do
    not need an fp32 copy of their own size."""
    out = torch.empty(shape, dtype=DTYPES[dtype], device=device)
    if out.numel() == 0:
        return out
    rows = out.shape[0]
    per_row = out.numel() // rows
    step = max(1, (1 << 27) // max(per_row, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(out.shape[1:]), generator=gen, device=device,
                                 dtype=torch.float32)
    return out


def _context_lens(cfg: DecodeConfig, rng: np.random.Generator) -> np.ndarray:
    if cfg.ctx_fixed is not None:
        base = np.asarray(cfg.ctx_fixed, dtype=np.int64)
        assert base.size == cfg.num_seqs
    else:
        lo, hi = cfg.ctx_range
        base = rng.integers(lo, hi, size=cfg.num_seqs, endpoint=True)
    return (base + cfg.ctx_append).astype(np.int32)


def make_decode_case(cfg: DecodeConfig, device="cpu", seed: Optional[int] = None,
                     values: bool = True, poison_unused: bool = False,
                     num_seqs: Optional[int] = None) -> DecodeCase:
    """Build one decode workload.

    Placement: the pool's block ids are shuffled once (seeded) and handed out
    in that order, sequence by sequence, so each sequence's blocks are
    scattered through the pool.

    ``poison_unused`` fills table entries past each sequence's last block
    with an out-of-range id and every pool slot that no sequence uses (free
    blocks, and the slots past the end of each last block) with NaN, so a
    kernel that reads past the context shows up in its output.
    ``num_seqs`` truncates the batch (same structure for the first rows).
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = _context_lens(cfg, rng)
    if num_seqs is not None:
        ctx = ctx[:num_seqs]
    n = ctx.size
    B = cfg.block_size
    nblk = (ctx.astype(np.int64) + B - 1) // B
    used = int(nblk.sum())
    if cfg.pool_blocks is not None and num_seqs is None:
        nb = cfg.pool_blocks
    else:
        nb = max(int(math.ceil(cfg.pool_factor * used)), used, 1)
    assert nb >= used
    perm = rng.permutation(nb).astype(np.int32)
    mb = cfg.max_blocks_per_seq
    tables = np.full((n, mb), -1, dtype=np.int32)
    if poison_unused:
        tables[:] = nb + 7
    pos = 0
    for s in range(n):
        k = int(nblk[s])
        tables[s, :k] = perm[pos:pos + k]
        pos += k
    case = DecodeCase(cfg=cfg, context_lens=ctx, block_tables=tables, num_blocks=nb,
                      scale=float(np.float32(1.0 / math.sqrt(cfg.head_dim))))
    if values:
        g = _torch_gen(seed, device)
        hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
        case.q = make_values((n, hq, d), cfg.dtype, g, device)
        case.k_pool = make_values((nb, hkv, B, d), cfg.dtype, g, device)
        case.v_pool = make_values((nb, hkv, B, d), cfg.dtype, g, device)
        case.k_new = make_values((n, hkv, d), cfg.dtype, g, device)
        case.v_new = make_values((n, hkv, d), cfg.dtype, g, device)
        if poison_unused:
            nan = float("nan")
            live = np.zeros(nb, dtype=bool)
            live[perm[:used]] = True
            dead = torch.from_numpy(~live).to(device)
            case.k_pool[dead] = nan
            case.v_pool[dead] = nan
            for s in range(n):
                k = int(nblk[s])
                fill = int(ctx[s]) - (k - 1) * B
                if fill < B:
                    last = int(tables[s, k - 1])
                    case.k_pool[last, :, fill:, :] = nan
                    case.v_pool[last, :, fill:, :] = nan
    return case


# ---------------------------------------------------------------------------
# Parallel sampling with a shared prompt
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class SamplingConfig:
    name: str = "parallel_sampling"
    groups: int = 64
    samples: int = 8
    prompt_len: int = 2032
    tail_range: tuple = (0, 256)
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    block_size: int = 32
    dtype: str = "bf16"
    seed: int = 1005
    pool_factor: float = 1.1
    description: str = ("parallel sampling: 64 prompt groups x 8 samples, 2032-token shared "
                        "prompt (64 blocks of 32, last one half full), divergent tail "
                        "U[0,256] + 1 new token per sample, 32/8 heads, d 128")

    @property
    def num_seqs(self) -> int:
        return self.groups * self.samples

    @property
    def max_context_len(self) -> int:
        return self.prompt_len + self.tail_range[1] + 1

    @property
    def max_blocks_per_seq(self) -> int:
        return -(-self.max_context_len // self.block_size)


SAMPLING = SamplingConfig()

# The block-aligned reading of the same workload: a 2048-token prompt fills its
# 64 blocks, so the samples' first writes open fresh blocks and nothing is
# copied on write.
SAMPLING_ALIGNED = SamplingConfig(
    name="parallel_sampling_aligned", prompt_len=2048, seed=1006,
    description=("parallel sampling, block-aligned prompt: 64 prompt groups x 8 samples, 2048-token "
                 "shared prompt (64 full blocks of 32, no copy-on-write), divergent tail U[0,256] + 1 "
                 "new token per sample, 32/8 heads, d 128"))

SAMPLINGS = {c.name: c for c in (SAMPLING, SAMPLING_ALIGNED)}


@dataclass
class SamplingCase:
    cfg: SamplingConfig
    prompt_blocks: np.ndarray          # int32 [G, nP] shared physical ids
    tails: np.ndarray                  # int32 [G*S] divergent tokens written this step (excl. the new one)
    private_last: np.ndarray           # int32 [G*S] private copy of the last prompt block, -1 = keeps it
    tail_blocks: list                  # per sample: int32 array of blocks past the prompt
    num_blocks: int
    scale: float
    q: Optional[torch.Tensor] = None
    k_pool: Optional[torch.Tensor] = None
    v_pool: Optional[torch.Tensor] = None
    k_new: Optional[torch.Tensor] = None   # [T, Hkv, d], T = sum(tails + 1), sample-major
    v_new: Optional[torch.Tensor] = None


def make_sampling_case(cfg: SamplingConfig = SAMPLING, device="cpu", seed: Optional[int] = None,
                       values: bool = True, groups: Optional[int] = None) -> SamplingCase:
    """Shared-prompt state just before the samples diverge.

    Every sample of a group points at the same prompt blocks.  The last
    prompt block is only partly filled when ``prompt_len`` is not a multiple
    of the block size; a sample that writes past the prompt then needs its
    own copy of it (all but the last sample of a group; the last one is the
    sole owner by then and writes in place).  Extra blocks for each sample's
    tail come from the same shuffled pool order.
    """
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    G = cfg.groups if groups is None else groups
    S, B = cfg.samples, cfg.block_size
    nS = G * S
    lo, hi = cfg.tail_range
    tails = rng.integers(lo, hi, size=nS, endpoint=True).astype(np.int32)
    nP = -(-cfg.prompt_len // B)
    partial = (cfg.prompt_len % B) != 0
    total_len = cfg.prompt_len + tails.astype(np.int64) + 1
    need_blocks = -(-total_len // B)
    n_extra = need_blocks - nP
    n_private = nS - G if partial else 0
    used = G * nP + n_private + int(n_extra.sum())
    nb = max(int(math.ceil(cfg.pool_factor * used)), used)
    perm = rng.permutation(nb).astype(np.int32)
    pos = 0
    prompt_blocks = perm[pos:pos + G * nP].reshape(G, nP).copy()
    pos += G * nP
    private_last = np.full(nS, -1, dtype=np.int32)
    tail_blocks = []
    for i in range(nS):
        if partial and (i % S) != S - 1:
            private_last[i] = perm[pos]
            pos += 1
        k = int(n_extra[i])
        tail_blocks.append(perm[pos:pos + k].copy())
        pos += k
    case = SamplingCase(cfg=cfg, prompt_blocks=prompt_blocks, tails=tails,
                        private_last=private_last, tail_blocks=tail_blocks, num_blocks=nb,
                        scale=float(np.float32(1.0 / math.sqrt(cfg.head_dim))))
    if values:
        g = _torch_gen(seed, device)
        hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
        T = int((tails.astype(np.int64) + 1).sum())
        case.q = make_values((nS, hq, d), cfg.dtype, g, device)
        case.k_pool = make_values((nb, hkv, B, d), cfg.dtype, g, device)
        case.v_pool = make_values((nb, hkv, B, d), cfg.dtype, g, device)
        case.k_new = make_values((T, hkv, d), cfg.dtype, g, device)
        case.v_new = make_values((T, hkv, d), cfg.dtype, g, device)
    return case


def sampling_tables(case: SamplingCase):
    """Block tables and lengths of every sample after the divergent step:
    the group's prompt blocks (the last one replaced by the sample's private
    copy where it has one), then the sample's own tail blocks."""
    cfg = case.cfg
    nS = case.prompt_blocks.shape[0] * cfg.samples
    tables = np.full((nS, cfg.max_blocks_per_seq), -1, dtype=np.int32)
    for i in range(nS):
        row = [int(b) for b in case.prompt_blocks[i // cfg.samples]]
        if case.private_last[i] >= 0:
            row[-1] = int(case.private_last[i])
        row += [int(b) for b in case.tail_blocks[i]]
        tables[i, :len(row)] = row
    ctx = (cfg.prompt_len + case.tails.astype(np.int64) + 1).astype(np.int32)
    return tables, ctx


def make_codes(shape, gen: torch.Generator, device, below: int = 0x50) -> torch.Tensor:
    """Random 8-bit codes: a uniform magnitude byte in [0, below) and a
    random top (sign) bit, as uint8.  Used to fill 8-bit caches directly."""
    mag = torch.randint(0, below, shape, generator=gen, device=device, dtype=torch.int32)
    sign = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32)
    return (mag | (sign << 7)).to(torch.uint8)


def make_int4_pool(num_blocks, num_kv_heads, block_size, head_dim, gen: torch.Generator, device,
                   scale_range=(0.05, 0.4)) -> torch.Tensor:
    """Random contents for a 4-bit pool (uint8 [NB, Hkv, B, d + 8]): each piece
    is B * d random code bytes followed by 2 * B fp32 scales drawn uniformly
    from scale_range.  Any nibble is a valid code, so every piece decodes to
    finite values."""
    NB, Hkv, B, d = num_blocks, num_kv_heads, block_size, head_dim
    pool = torch.empty((NB, Hkv, B * (d + 8)), dtype=torch.uint8, device=device)
    codes = B * d
    step = max(1, (1 << 26) // max(1, Hkv * B * (d + 8)))
    lo, hi = scale_range
    for b0 in range(0, NB, step):
        b1 = min(NB, b0 + step)
        pool[b0:b1, :, :codes] = torch.randint(0, 256, (b1 - b0, Hkv, codes), generator=gen, device=device,
                                               dtype=torch.int32).to(torch.uint8)
        sc = torch.rand((b1 - b0, Hkv, 2 * B), generator=gen, device=device) * (hi - lo) + lo
        pool[b0:b1, :, codes:] = sc.contiguous().view(torch.uint8).view(b1 - b0, Hkv, 8 * B)
    return pool.view(NB, Hkv, B, d + 8)


"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the benchmark and the smoke check.  It holds
none of the attention arithmetic: it draws random numbers, picks context lengths,
allocates physical blocks (the host-side block allocator of a paged cache) and
fills the pool the way a finished prefill would have left it.  Both the CUDA
library and the fp64 oracle are then fed the same bits.

Workloads (shapes from the configurations the library is measured on):

  tiny            3 seqs, context lens {1, 17, 37}, 4 q heads = 4 KV heads,
                  head_dim 64, block_size 16, fp16, 16-block pool
  llama7b_mha     32 seqs, 32 q / 32 KV heads, head_dim 128, fp16,
                  context lens uniform in [512, 4096]
  gqa             64 seqs, 32 q / 8 KV heads, head_dim 128, bf16, context lens
                  lognormal (median 1500, sigma 0.5 -- an assumed spread), cap 8192
  long_split      4 seqs x 32768 tokens, 32 q / 8 KV heads, head_dim 128, bf16,
                  16 split-KV partitions
  prefix_verify   128 seqs sharing a 1024-token prefix (the same 64 physical
                  blocks), private tails of U[64, 2048] tokens, 4 causal query
                  positions per seq, 32 q / 8 KV heads, head_dim 128, fp16
  chunked_prefill 16 seqs, each appending a chunk of 512 new tokens (8192 tokens a
                  step) at the end of a context uniform in [512, 8192], causal;
                  32 q / 8 KV heads, head_dim 128, bf16
  llama7b_mha_fp8, gqa_fp8, chunked_prefill_fp8
                  the same shapes over an FP8 (e4m3) cache with one scale per KV
                  head (K and V separately, drawn in [0.02, 0.05]); q and the new
                  rows stay in the 16-bit type

Every value in q, the pool and the new rows is N(0, 1), rounded to nearest even
into the 16-bit type.  Physical block ids are a seeded random permutation of the
pool.  With ``poison=True`` every slot that holds no token before this step's
append (the slots the append will fill, unused tail slots, free blocks and the
padding block that fills block-table rows past a sequence's length) is NaN, so
that a kernel reading a slot it must not read produces NaN.

Random streams: numpy PCG64, one ``SeedSequence([seed, stream, chunk])`` per
fixed-size chunk of 2^22 values, so the values do not depend on how many threads
generate them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np
import torch

_CHUNK = 1 << 22

# stream tags (arbitrary distinct constants)
_S_LENS, _S_PERM, _S_Q, _S_KNEW, _S_VNEW, _S_KCACHE, _S_VCACHE = 11, 12, 13, 14, 15, 16, 17

TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Config:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                 # "fp16" | "bf16"
    q_len: int = 1             # new (query) tokens per sequence this step
    lens: tuple = ()           # context-length recipe, see _context_lens
    num_splits: int = 1        # split-KV partitions (1 = single pass)
    pool_blocks: int | None = None   # fixed pool size; None = exactly what is needed + spare
    shared_prefix: int = 0     # tokens of a prefix whose blocks all sequences share
    spare_blocks: int = 8      # free (never referenced) blocks added to the pool
    kv_fp8: bool = False       # cache holds FP8 (e4m3) codes with per-KV-head scales

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


CONFIGS: dict[str, Config] = {
    "tiny": Config("tiny", 3, 4, 4, 64, 16, "fp16", lens=("fixed", (1, 17, 37)),
                   pool_blocks=16),
    "llama7b_mha": Config("llama7b_mha", 32, 32, 32, 128, 16, "fp16",
                          lens=("uniform", 512, 4096)),
    "gqa": Config("gqa", 64, 32, 8, 128, 16, "bf16", lens=("lognormal", 1500.0, 0.5, 8192)),
    "long_split": Config("long_split", 4, 32, 8, 128, 16, "bf16",
                         lens=("fixed", (32768,) * 4), num_splits=16),
    "prefix_verify": Config("prefix_verify", 128, 32, 8, 128, 16, "fp16", q_len=4,
                            lens=("prefix", 1024, 64, 2048), shared_prefix=1024),
    "chunked_prefill": Config("chunked_prefill", 16, 32, 8, 128, 16, "bf16", q_len=512,
                              lens=("uniform", 512, 8192)),
    # the same shapes over an FP8 (e4m3) cache, q and new rows in the 16-bit type
    "llama7b_mha_fp8": Config("llama7b_mha_fp8", 32, 32, 32, 128, 16, "fp16",
                              lens=("uniform", 512, 4096), kv_fp8=True),
    "gqa_fp8": Config("gqa_fp8", 64, 32, 8, 128, 16, "bf16",
                      lens=("lognormal", 1500.0, 0.5, 8192), kv_fp8=True),
    "chunked_prefill_fp8": Config("chunked_prefill_fp8", 16, 32, 8, 128, 16, "bf16", q_len=512,
                                  lens=("uniform", 512, 8192), kv_fp8=True),
}


def config(name: str, **overrides) -> Config:
    """A named configuration, optionally with fields replaced (e.g. num_seqs=4)."""
    return replace(CONFIGS[name], **overrides)


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_tensor(shape, dtype: str, seed: int, stream: int) -> torch.Tensor:
    """N(0,1) values rounded to nearest even into fp16/bf16, as a CPU tensor."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=TORCH_DTYPE[dtype])
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = _rng(seed, stream, c).standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = torch.from_numpy(x)      # float32 -> fp16/bf16, round to nearest even

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.view(*shape)


def _context_lens(cfg: Config, seed: int) -> np.ndarray:
    kind = cfg.lens[0]
    rng = _rng(seed, _S_LENS)
    if kind == "fixed":
        lens = np.array(cfg.lens[1], dtype=np.int64)
        if lens.shape[0] != cfg.num_seqs:
            lens = np.resize(lens, cfg.num_seqs)
    elif kind == "uniform":
        lo, hi = cfg.lens[1], cfg.lens[2]
        lens = rng.integers(lo, hi + 1, size=cfg.num_seqs)
    elif kind == "lognormal":
        median, sigma, cap = cfg.lens[1], cfg.lens[2], cfg.lens[3]
        z = rng.standard_normal(cfg.num_seqs)
        lens = np.rint(np.exp(math.log(median) + sigma * z))
        lens = np.clip(lens, 1, cap).astype(np.int64)
    elif kind == "prefix":
        prefix, lo, hi = cfg.lens[1], cfg.lens[2], cfg.lens[3]
        lens = prefix + rng.integers(lo, hi + 1, size=cfg.num_seqs)
    else:
        raise ValueError(f"unknown context-length recipe {cfg.lens}")
    return lens.astype(np.int32)


@dataclass
class Workload:
    cfg: Config
    seed: int
    scale: float                 # 1/sqrt(head_dim), computed in float32
    context_lens: torch.Tensor   # [N] int32, counts this step's new tokens
    block_tables: torch.Tensor   # [N, max_blocks_per_seq] int32
    q: torch.Tensor              # [N, q_len, H_q, D]
    k_new: torch.Tensor          # [N*q_len, H_kv, D]
    v_new: torch.Tensor
    k_cache: torch.Tensor        # [P, H_kv, B, D] state before this step's append
    v_cache: torch.Tensor
    padding_block: int           # block id used for table entries past a sequence's end
    info: dict = field(default_factory=dict)
    k_scale: torch.Tensor | None = None   # [H_kv] float32, FP8 caches only (uint8 codes)
    v_scale: torch.Tensor | None = None

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.to(torch.int64).sum())

    def bits(self, name: str) -> np.ndarray:
        """A 16-bit tensor field as a numpy uint16 bit-pattern array (shares memory);
        FP8 caches come back as their uint8 codes."""
        t = getattr(self, name)
        if t.dtype == torch.uint8:
            return t.numpy()
        return t.view(torch.int16).numpy().view(np.uint16)


def make(cfg: Config | str, seed: int = 0, poison: bool = True, **overrides) -> Workload:
    """Build the seeded workload for ``cfg`` (a Config or a name in CONFIGS)."""
    if isinstance(cfg, str):
        cfg = config(cfg, **overrides)
    elif overrides:
        cfg = replace(cfg, **overrides)
    B, H_kv, D = cfg.block_size, cfg.num_kv_heads, cfg.head_dim
    lens = _context_lens(cfg, seed)
    nblocks = (lens.astype(np.int64) + B - 1) // B
    shared = cfg.shared_prefix // B
    if cfg.shared_prefix % B:
        raise ValueError("a shared prefix must cover whole blocks")
    private = np.maximum(nblocks - shared, 0)
    needed = shared + int(private.sum()) + 1            # + the padding block
    if cfg.pool_blocks is not None:
        pool = cfg.pool_blocks
        if pool < needed:
            raise ValueError(f"pool of {pool} blocks is smaller than the {needed} needed")
    else:
        pool = needed + cfg.spare_blocks
    perm = _rng(seed, _S_PERM).permutation(pool).astype(np.int64)
    # allocation order: shared prefix blocks, then each sequence's private blocks,
    # then the padding block; the rest of the permutation stays free
    shared_ids = perm[:shared]
    cursor = shared
    max_blocks = max(1, int(nblocks.max()) if len(nblocks) else 1)
    tables = np.empty((cfg.num_seqs, max_blocks), dtype=np.int64)
    owned = []
    for i in range(cfg.num_seqs):
        k = int(private[i])
        own = perm[cursor:cursor + k]
        cursor += k
        owned.append(own)
        row = np.concatenate([shared_ids[:min(shared, int(nblocks[i]))], own])
        tables[i, :row.shape[0]] = row
    padding_block = int(perm[cursor])
    for i in range(cfg.num_seqs):
        tables[i, int(nblocks[i]):] = padding_block

    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    n_new = cfg.num_seqs * cfg.q_len
    q = normal_tensor((cfg.num_seqs, cfg.q_len, cfg.num_q_heads, D), cfg.dtype, seed, _S_Q)
    k_new = normal_tensor((n_new, H_kv, D), cfg.dtype, seed, _S_KNEW)
    v_new = normal_tensor((n_new, H_kv, D), cfg.dtype, seed, _S_VNEW)
    k_cache = normal_tensor((pool, H_kv, B, D), cfg.dtype, seed, _S_KCACHE)
    v_cache = normal_tensor((pool, H_kv, B, D), cfg.dtype, seed, _S_VCACHE)
    k_scale = v_scale = None
    if cfg.kv_fp8:
        # FP8 pool: codes of N(0,1) values under a per-head scale drawn in
        # [0.02, 0.05] (|value / scale| stays well inside e4m3's +-448); the codes
        # are made with torch's float8 conversion.
        srng = _rng(seed, _S_PERM + 100)
        k_scale = torch.from_numpy(srng.uniform(0.02, 0.05, H_kv).astype(np.float32))
        v_scale = torch.from_numpy(srng.uniform(0.02, 0.05, H_kv).astype(np.float32))
        k_cache = (k_cache.float() / k_scale[None, :, None, None]).to(torch.float8_e4m3fn)
        v_cache = (v_cache.float() / v_scale[None, :, None, None]).to(torch.float8_e4m3fn)
        k_cache, v_cache = k_cache.view(torch.uint8), v_cache.view(torch.uint8)

    if poison:
        # filled[block] = how many leading slots of the block carry a token written
        # by an earlier step (prefill): positions < context_len - q_len of the
        # sequences owning it.  Everything after them is NaN.
        filled = np.zeros(pool, dtype=np.int64)
        for i in range(cfg.num_seqs):
            old = int(lens[i]) - cfg.q_len
            for j in range(int(nblocks[i])):
                first = j * B
                if first >= old:
                    break
                b = tables[i, j]
                filled[b] = max(filled[b], min(B, old - first))
        nan = 0x7F if cfg.kv_fp8 else float("nan")      # e4m3 NaN code
        empty = torch.from_numpy(np.nonzero(filled == 0)[0])
        k_cache[empty] = nan
        v_cache[empty] = nan
        for b in np.nonzero((filled > 0) & (filled < B))[0]:
            k_cache[int(b), :, int(filled[b]):, :] = nan
            v_cache[int(b), :, int(filled[b]):, :] = nan

    info = {
        "pool_blocks": pool,
        "blocks_in_use": int(needed - 1),
        "unique_tokens": int(cfg.shared_prefix + np.maximum(lens - cfg.shared_prefix, 0).sum())
        if cfg.shared_prefix else int(lens.sum()),
    }
    return Workload(cfg=cfg, seed=seed, scale=scale,
                    context_lens=torch.from_numpy(lens.copy()),
                    block_tables=torch.from_numpy(tables.astype(np.int32)),
                    q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                    padding_block=padding_block, info=info, k_scale=k_scale, v_scale=v_scale)

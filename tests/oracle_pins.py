"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with what the pages or the mathematics fix:

  * IEEE decoding of every fp16 / bf16 bit pattern (numpy / torch conversions);
  * worked examples printed or drawn on the pages (tests/golden/*.txt);
  * library routines that the paged computation reduces to once the blocks are
    gathered (torch scaled_dot_product_attention in float64, with the causal mask
    built by torch.triu exactly as the LLM-Code-Hot-100 listing builds it);
  * closed forms (context length 1 returns V, two tokens give a sigmoid blend,
    scale 0 gives the mean of V, identical V rows return that row);
  * invariants the pages state (paging does not change the result under any
    permutation of physical blocks; online/partitioned softmax gives the same
    result as plain softmax) and algebraic ones (key shift, convex hull, GQA equals
    MHA with duplicated KV heads, a causal query equals a shorter decode).

The same functions run in ``test_oracle.py`` against the real oracle and in
``test_oracle_mutants.py`` against altered copies, each of which must fail at
least one pin.  Run as ``python -m tests.oracle_pins <libpath>`` to check one
compiled copy (exit status = number of failing pins).
"""
from __future__ import annotations

import math
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")

FP16, BF16 = "fp16", "bf16"
_NP = {FP16: np.float16}


# ----------------------------------------------------------------------------- helpers
def _bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values -> 16-bit patterns (round to nearest even), via torch."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    t = t.to(torch.float16 if dtype == FP16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _vals(bits: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == FP16 else torch.bfloat16)
    return t.to(torch.float64).numpy()


def _golden_rows(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _nan_pool(num_blocks, h_kv, block_size, head_dim, dtype):
    nan = 0x7E00 if dtype == FP16 else 0x7FC0
    return np.full((num_blocks, h_kv, block_size, head_dim), nan, dtype=np.uint16)


class Paged:
    """A paged cache filled from logical sequences through the oracle's own
    slot mapping and append (the way a serving engine writes it)."""

    def __init__(self, o, K, V, block_size, dtype, perm_seed=None, spare=3, order=None):
        # K[i], V[i]: uint16 [L_i, H_kv, D]
        self.dtype = dtype
        self.block_size = block_size
        self.lens = np.array([k.shape[0] for k in K], dtype=np.int32)
        h_kv, d = K[0].shape[1], K[0].shape[2]
        nb = [(int(L) + block_size - 1) // block_size for L in self.lens]
        max_blocks = max(1, max(nb))
        pool = sum(nb) + spare
        ids = np.arange(pool)
        if perm_seed is not None:
            ids = np.random.default_rng(perm_seed).permutation(pool)
        if order is not None:
            ids = np.asarray(order)
        self.tables = np.full((len(K), max_blocks), ids[-1], dtype=np.int32)
        cur = 0
        for i, n in enumerate(nb):
            self.tables[i, :n] = ids[cur:cur + n]
            cur += n
        self.k = _nan_pool(pool, h_kv, block_size, d, dtype)
        self.v = _nan_pool(pool, h_kv, block_size, d, dtype)
        for i in range(len(K)):
            L = int(self.lens[i])
            if L == 0:
                continue
            slots = o.slot_mapping(self.tables[i:i + 1], self.lens[i:i + 1], block_size, q_len=L)
            o.append_kv(self.k, self.v, K[i], V[i], slots)

    def decode(self, o, q, scale, q_len=1, lens=None):
        lens = self.lens if lens is None else np.asarray(lens, dtype=np.int32)
        return o.decode(q, self.k, self.v, self.tables, lens, scale, self.dtype, q_len=q_len)


def _rand_case(seed, n_seqs, h_q, h_kv, d, dtype, lens, q_len=1, qscale=1.0):
    rng = np.random.default_rng(seed)
    K = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    V = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    q = _bits(qscale * rng.standard_normal((n_seqs, q_len, h_q, d)), dtype)
    return q, K, V


def _sdpa(q_bits, K_bits, V_bits, scale, dtype, q_len):
    """torch float64 scaled_dot_product_attention on the logical (unpaged) rows."""
    h_q = q_bits.shape[1]
    h_kv = K_bits.shape[1]
    g = h_q // h_kv
    L = K_bits.shape[0]
    q = torch.from_numpy(_vals(q_bits, dtype)).permute(1, 0, 2)          # [H_q, q_len, D]
    k = torch.from_numpy(_vals(K_bits, dtype)).permute(1, 0, 2)          # [H_kv, L, D]
    v = torch.from_numpy(_vals(V_bits, dtype)).permute(1, 0, 2)
    k = k.repeat_interleave(g, dim=0)
    v = v.repeat_interleave(g, dim=0)
    mask = None
    if q_len > 1:
        hidden = torch.triu(torch.ones(q_len, L), diagonal=L - q_len + 1).bool()
        mask = ~hidden
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    return out.permute(1, 0, 2).numpy()                                   # [q_len, H_q, D]


# ----------------------------------------------------------------------------- pins
def pin_fp16_decoding(o):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.decode_bits(bits, FP16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_bf16_decoding(o):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.decode_bits(bits, BF16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_slot_mapping_page_example(o):
    for req, table, pos, want in _golden_rows("slot_mapping_pano_2_2.txt"):
        t = np.array([[int(x) for x in table.split(",")]], dtype=np.int32)
        got = o.slot_mapping(t, np.array([int(pos) + 1], dtype=np.int32), 16, q_len=1)
        assert int(got[0]) == int(want), (req, table, pos, int(got[0]), want)


def pin_slot_mapping_multi_query(o):
    # q_len new tokens are the last q_len positions; a position < 0 maps to -1.
    t = np.array([[1, 3, 5], [2, 4, 6]], dtype=np.int32)
    got = o.slot_mapping(t, np.array([18, 2], dtype=np.int32), 16, q_len=4)
    # seq 0 positions 14..17 -> 30, 31, 48, 49 ; seq 1 positions -2..1 -> -1, -1, 32, 33
    assert got.tolist() == [30, 31, 48, 49, -1, -1, 32, 33], got.tolist()


def pin_append_layout(o):
    # cache layout [num_blocks][num_kv_heads][block_size][head_dim]: writing token
    # slot s, head h, element d lands at ((s//B * H + h) * B + s%B) * D + d.
    H, B, D, P = 3, 16, 8, 6
    kc = np.zeros((P, H, B, D), dtype=np.uint16)
    vc = np.zeros((P, H, B, D), dtype=np.uint16)
    k_new = np.arange(1, 1 + 2 * H * D, dtype=np.uint16).reshape(2, H, D)
    v_new = k_new + 1000
    o.append_kv(kc, vc, k_new, v_new, np.array([52, -1], dtype=np.int64))
    flat_k, flat_v = kc.reshape(-1), vc.reshape(-1)
    changed = np.nonzero(flat_k)[0]
    assert changed.size == H * D
    for h in range(H):
        for d in range(D):
            off = ((3 * H + h) * B + 4) * D + d          # slot 52 = block 3, offset 4
            assert flat_k[off] == k_new[0, h, d] and flat_v[off] == v_new[0, h, d]


def pin_append_only_targets(o):
    rng = np.random.default_rng(1)
    P, H, B, D = 9, 2, 16, 16
    kc = rng.integers(0, 65536, size=(P, H, B, D)).astype(np.uint16)
    vc = rng.integers(0, 65536, size=(P, H, B, D)).astype(np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    slots = np.array([5, 77, -1, 143, 16], dtype=np.int64)
    k_new = rng.integers(0, 65536, size=(5, H, D)).astype(np.uint16)
    v_new = rng.integers(0, 65536, size=(5, H, D)).astype(np.uint16)
    o.append_kv(kc, vc, k_new, v_new, slots)
    touched = np.zeros((P, B), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc[s // B, :, s % B, :], k_new[t])
        assert np.array_equal(vc[s // B, :, s % B, :], v_new[t])
        touched[s // B, s % B] = True
    tk, tv = kc.transpose(0, 2, 1, 3), vc.transpose(0, 2, 1, 3)     # [P, B, H, D]
    assert np.array_equal(tk[~touched], k0.transpose(0, 2, 1, 3)[~touched])
    assert np.array_equal(tv[~touched], v0.transpose(0, 2, 1, 3)[~touched])


def pin_matches_sdpa(o):
    cases = [
        # seed, h_q, h_kv, d, dtype, lens, q_len
        (2, 4, 4, 64, FP16, [1, 17, 37, 16], 1),
        (3, 8, 2, 32, BF16, [5, 33, 64], 1),
        (4, 6, 3, 16, FP16, [9, 20, 40], 4),
        (5, 4, 1, 32, BF16, [4, 31], 2),
        # chunked prefill: many query rows; L == q_len is a plain causal prefill
        (18, 4, 2, 16, FP16, [40, 57, 100], 40),
    ]
    for seed, h_q, h_kv, d, dtype, lens, q_len in cases:
        q, K, V = _rand_case(seed, len(lens), h_q, h_kv, d, dtype, lens, q_len=q_len)
        pc = Paged(o, K, V, 16, dtype, perm_seed=seed)
        scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
        got = pc.decode(o, q, scale, q_len=q_len)
        for i, L in enumerate(lens):
            want = _sdpa(q[i], K[i], V[i], scale, dtype, q_len)
            assert np.abs(got[i] - want).max() < 1e-12, (seed, i)


def pin_paging_invariance(o):
    lens = [3, 16, 29, 50]
    q, K, V = _rand_case(6, 4, 4, 2, 32, FP16, lens)
    scale = 0.17
    ref = Paged(o, K, V, 16, FP16, perm_seed=None).decode(o, q, scale)
    for s in range(4):
        got = Paged(o, K, V, 16, FP16, perm_seed=100 + s).decode(o, q, scale)
        assert np.array_equal(got, ref)


def pin_block_size_invariance(o):
    """The same logical sequences in pools of 8-, 16- and 32-token blocks (random
    physical order) attend to bit-identical results, and equal torch SDPA: the
    block size only changes where the rows live ([PANO] §2.3: block_size is a
    parameter of the pool)."""
    lens = [1, 7, 8, 9, 31, 33, 64, 70]
    q, K, V = _rand_case(61, len(lens), 6, 2, 32, BF16, lens, q_len=1)
    scale = float(np.float32(0.19))   # the oracle takes the scale as a float
    ref = Paged(o, K, V, 16, BF16, perm_seed=3).decode(o, q, scale)
    for bs in (8, 32):
        got = Paged(o, K, V, bs, BF16, perm_seed=4).decode(o, q, scale)
        assert np.array_equal(got, ref), bs
    for i in range(len(lens)):
        assert np.abs(ref[i] - _sdpa(q[i], K[i], V[i], scale, BF16, 1)).max() < 1e-12, i


def pin_context_one_returns_v(o):
    for dtype in (FP16, BF16):
        q, K, V = _rand_case(7, 2, 4, 4, 64, dtype, [1, 1], qscale=3.0)
        got = Paged(o, K, V, 16, dtype, perm_seed=1).decode(o, q, 0.125)
        for i in range(2):
            want = _vals(V[i][0], dtype)                      # [H, D]
            assert np.array_equal(got[i, 0], want)


def pin_two_token_sigmoid(o):
    # softmax over two scores s0, s1 is (1 - sigma, sigma) with sigma = 1/(1+e^(s0-s1))
    q, K, V = _rand_case(8, 1, 2, 2, 16, FP16, [2])
    scale = float(np.float32(0.3))            # the kernel's scale argument is a float
    got = Paged(o, K, V, 16, FP16).decode(o, q, scale)[0, 0]
    qv, kv, vv = _vals(q[0, 0], FP16), _vals(K[0], FP16), _vals(V[0], FP16)
    for h in range(2):
        s0 = scale * float(np.dot(qv[h], kv[0, h]))
        s1 = scale * float(np.dot(qv[h], kv[1, h]))
        sig = 1.0 / (1.0 + math.exp(s0 - s1))
        want = vv[0, h] + sig * (vv[1, h] - vv[0, h])
        assert np.abs(got[h] - want).max() < 1e-13


def pin_scale_zero_mean(o):
    lens = [7, 40]
    q, K, V = _rand_case(9, 2, 2, 2, 32, BF16, lens)
    got = Paged(o, K, V, 16, BF16, perm_seed=3).decode(o, q, 0.0)
    for i in range(2):
        want = _vals(V[i], BF16).mean(axis=0)                 # [H, D]
        assert np.abs(got[i, 0] - want).max() < 1e-13


def pin_identical_rows(o):
    rng = np.random.default_rng(10)
    L = 37
    row = _bits(rng.standard_normal((1, 2, 32)), FP16)
    V = [np.repeat(row, L, axis=0)]
    K = [_bits(rng.standard_normal((L, 2, 32)), FP16)]
    q = _bits(2 * rng.standard_normal((1, 1, 2, 32)), FP16)
    got = Paged(o, K, V, 16, FP16, perm_seed=4).decode(o, q, 0.2)
    want = _vals(row[0], FP16)
    assert np.abs(got[0, 0] - want).max() <= 1e-14 * np.abs(want).max()


def pin_convex_hull(o):
    lens = [5, 23, 61]
    q, K, V = _rand_case(11, 3, 4, 2, 16, BF16, lens, qscale=4.0)
    got = Paged(o, K, V, 16, BF16, perm_seed=5).decode(o, q, 0.25)
    for i, L in enumerate(lens):
        v = _vals(V[i], BF16)                                 # [L, H_kv, D]
        lo = v.min(axis=0).repeat(2, axis=0)                  # [H_q, D] (group 2)
        hi = v.max(axis=0).repeat(2, axis=0)
        assert np.all(got[i, 0] >= lo - 1e-12) and np.all(got[i, 0] <= hi + 1e-12)


def pin_key_shift_invariance(o):
    # keys on a grid of 1/8 plus a shared shift stay exact in fp16; adding the same
    # vector c to every key adds q.c to every score of a row, which softmax ignores.
    rng = np.random.default_rng(12)
    L, H, D = 30, 2, 16
    k0 = rng.integers(-16, 17, size=(L, H, D)) / 8.0
    c = rng.integers(-8, 9, size=(1, H, D)) / 4.0
    v = rng.standard_normal((L, H, D))
    q = rng.integers(-8, 9, size=(1, 1, H, D)) / 4.0
    qb, vb = _bits(q, FP16), _bits(v, FP16)
    a = Paged(o, [_bits(k0, FP16)], [vb], 16, FP16, perm_seed=6).decode(o, qb, 0.25)
    b = Paged(o, [_bits(k0 + c, FP16)], [vb], 16, FP16, perm_seed=7).decode(o, qb, 0.25)
    assert np.abs(a - b).max() < 1e-13


def pin_gqa_mapping_figure(o):
    for hq, hkv, qf, ql, kf, kl in _golden_rows("gqa_heads_anim_1.txt"):
        hq, hkv, qf, ql, kf, kl = map(int, (hq, hkv, qf, ql, kf, kl))
        L, D = 5, 8
        # KV head j holds V rows all equal to j: attention over it returns exactly j
        V = np.broadcast_to(np.arange(hkv, dtype=np.float64)[None, :, None], (L, hkv, D))
        rng = np.random.default_rng(13)
        K = [_bits(rng.standard_normal((L, hkv, D)), FP16)]
        q = _bits(rng.standard_normal((1, 1, hq, D)), FP16)
        got = Paged(o, K, [_bits(V, FP16)], 16, FP16).decode(o, q, 0.3)[0, 0]   # [hq, D]
        assert np.abs(got - np.rint(got)).max() < 1e-12     # each head returns one KV head
        used = np.rint(got[:, 0]).astype(int)
        assert np.all((used[qf:ql + 1] >= kf) & (used[qf:ql + 1] <= kl))
        assert np.array_equal(used, np.arange(hq) // (hq // hkv))   # contiguous groups


def pin_gqa_equals_duplicated_mha(o):
    lens = [12, 35]
    g = 3
    q, K, V = _rand_case(14, 2, 6, 2, 16, FP16, lens)
    gqa = Paged(o, K, V, 16, FP16, perm_seed=8).decode(o, q, 0.2)
    Kd = [np.repeat(k, g, axis=1) for k in K]
    Vd = [np.repeat(v, g, axis=1) for v in V]
    mha = Paged(o, Kd, Vd, 16, FP16, perm_seed=9).decode(o, q, 0.2)
    assert np.array_equal(gqa, mha)


def pin_causal_reduces_to_decode(o):
    lens = [9, 21, 48]
    q_len = 4
    q, K, V = _rand_case(15, 3, 4, 2, 16, BF16, lens, q_len=q_len)
    pc = Paged(o, K, V, 16, BF16, perm_seed=10)
    multi = pc.decode(o, q, 0.25, q_len=q_len)
    for u in range(q_len):
        shorter = pc.lens - q_len + u + 1
        single = pc.decode(o, np.ascontiguousarray(q[:, u:u + 1]), 0.25, q_len=1, lens=shorter)
        assert np.array_equal(multi[:, u], single[:, 0])


def pin_partitions_combine(o):
    lens = [1, 17, 70, 0]
    for q_len in (1, 3):
        q, K, V = _rand_case(16, 4, 4, 2, 16, FP16, lens, q_len=q_len, qscale=3.0)
        pc = Paged(o, K, V, 16, FP16, perm_seed=11)
        full = pc.decode(o, q, 0.3, q_len=q_len).reshape(4, q_len * 4, 16)
        for S in (1, 2, 3, 16, 10):
            m, l, acc = o.decode_partitions(q, pc.k, pc.v, pc.tables, pc.lens, 0.3, FP16, S,
                                            q_len=q_len)
            got = o.combine(m, l, acc)
            assert np.abs(got - full).max() < 1e-12, S
            if S == 1:
                ok = l[:, 0] > 0
                norm = acc[:, 0][ok] / l[:, 0][ok][:, None]
                assert np.abs(norm - full[ok]).max() < 1e-13
            # partitions past the context are empty
            nb = (pc.lens.astype(int) + 15) // 16
            for i in range(4):
                C = -(-nb[i] // S)
                for p in range(S):
                    if p * C >= nb[i]:
                        assert np.all(l[i, p] == 0) and np.all(np.isneginf(m[i, p]))


def pin_empty_context_zero(o):
    q, K, V = _rand_case(17, 2, 2, 2, 16, FP16, [0, 3])
    got = Paged(o, K, V, 16, FP16).decode(o, q, 0.3)
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert not np.any(np.isnan(got))


def pin_copy_blocks_then_diverge(o):
    # copy-on-write: two sequences share their first blocks; the second gets a
    # private copy of the shared last block before appending into it.  Attention of
    # every sequence is unchanged by the copy, and the copy holds the source bytes.
    rng = np.random.default_rng(18)
    H, D = 2, 16
    K = [_bits(rng.standard_normal((40, H, D)), FP16)]
    V = [_bits(rng.standard_normal((40, H, D)), FP16)]
    pc = Paged(o, K, V, 16, FP16, perm_seed=19, spare=4)      # blocks of seq 0: 3
    q = _bits(rng.standard_normal((1, 1, H, D)), FP16)
    before = pc.decode(o, q, 0.25)
    src = int(pc.tables[0, 2])
    free = [b for b in range(pc.k.shape[0]) if b not in set(pc.tables[0].tolist())]
    dst = free[0]
    k0, v0 = pc.k.copy(), pc.v.copy()
    assert o.copy_blocks(pc.k, pc.v, [src, -1], [dst, 0]) == 1   # second pair skipped
    assert np.array_equal(pc.k[dst], pc.k[src]) and np.array_equal(pc.v[dst], pc.v[src])
    changed = np.any(pc.k != k0, axis=(1, 2, 3)) | np.any(pc.v != v0, axis=(1, 2, 3))
    assert set(np.nonzero(changed)[0].tolist()) <= {dst}
    pc.tables[0, 2] = dst                                    # the table now points at the copy
    assert np.array_equal(pc.decode(o, q, 0.25), before)


def _torch_e4m3_values(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def pin_e4m3_decoding(o):
    codes = np.arange(256, dtype=np.uint8)
    got, want = o.decode_e4m3(codes), _torch_e4m3_values(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])


def pin_e4m3_encoding(o):
    # torch rounds to nearest even but turns |x| > 464 into NaN; within +-464 the
    # two must agree bit for bit (ties included), beyond it the oracle saturates.
    f16 = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    rng = np.random.default_rng(31)
    rnd = (rng.standard_normal(200000) * rng.choice([1e-3, 0.05, 1.0, 40.0, 300.0], 200000))
    xs = np.concatenate([f16, rnd.astype(np.float32)])
    fin = np.isfinite(xs) & (np.abs(xs) <= 464.0)
    got = o.encode_e4m3(xs[fin])
    want = torch.from_numpy(xs[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    big = np.array([464.5, 500.0, 1e6, -465.0, -3e38], dtype=np.float32)
    assert o.encode_e4m3(big).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert o.encode_e4m3(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def _fp8_case(o, seed, lens, h_q, h_kv, d, dtype):
    """Logical rows quantised into an FP8 paged cache by the oracle's own append."""
    rng = np.random.default_rng(seed)
    K = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    V = [_bits(rng.standard_normal((L, h_kv, d)), dtype) for L in lens]
    q = _bits(rng.standard_normal((len(lens), 1, h_q, d)), dtype)
    ks = (0.5 + rng.random(h_kv)).astype(np.float32) / 64
    vs = (0.5 + rng.random(h_kv)).astype(np.float32) / 64
    nb = [(L + 15) // 16 for L in lens]
    pool = sum(nb) + 2
    ids = rng.permutation(pool)
    tables = np.full((len(lens), max(nb)), ids[-1], dtype=np.int32)
    cur = 0
    for i, n in enumerate(nb):
        tables[i, :n] = ids[cur:cur + n]
        cur += n
    kc = np.full((pool, h_kv, 16, d), 0x7F, dtype=np.uint8)
    vc = np.full((pool, h_kv, 16, d), 0x7F, dtype=np.uint8)
    cl = np.array(lens, dtype=np.int32)
    for i, L in enumerate(lens):
        slots = o.slot_mapping(tables[i:i + 1], cl[i:i + 1], 16, q_len=L)
        o.append_kv_fp8(kc, vc, K[i], V[i], slots, dtype, ks, vs)
    return q, K, V, kc, vc, ks, vs, tables, cl


def pin_fp8_append_quantises_per_head(o):
    q, K, V, kc, vc, ks, vs, tables, cl = _fp8_case(o, 32, [5, 40], 4, 2, 16, BF16)
    # the stored code of every appended element is e4m3(x / scale[h]) (float division)
    for i, L in enumerate([5, 40]):
        for t in range(L):
            blk, off = tables[i, t // 16], t % 16
            for h in range(2):
                x = _vals(K[i][t, h], BF16).astype(np.float32)
                want = torch.from_numpy(x / ks[h]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(kc[blk, h, off], want)


def pin_fp8_decode_matches_sdpa_on_dequantised(o):
    lens = [1, 17, 60]
    for dtype, h_q in ((FP16, 4), (BF16, 8)):
        q, K, V, kc, vc, ks, vs, tables, cl = _fp8_case(o, 33, lens, h_q, 2, 32, dtype)
        got = o.decode_fp8(q, kc, vc, ks, vs, tables, cl, 0.2, dtype)
        for i, L in enumerate(lens):
            rows_k = np.stack([kc[tables[i, t // 16], :, t % 16] for t in range(L)])   # [L, H, D]
            rows_v = np.stack([vc[tables[i, t // 16], :, t % 16] for t in range(L)])
            kd = _torch_e4m3_values(rows_k) * ks[None, :, None].astype(np.float64)
            vd = _torch_e4m3_values(rows_v) * vs[None, :, None].astype(np.float64)
            g = h_q // 2
            qq = torch.from_numpy(_vals(q[i, 0], dtype))[:, None, :]               # [Hq, 1, D]
            kk = torch.from_numpy(kd).permute(1, 0, 2).repeat_interleave(g, 0)
            vv = torch.from_numpy(vd).permute(1, 0, 2).repeat_interleave(g, 0)
            want = torch.nn.functional.scaled_dot_product_attention(
                qq, kk, vv, scale=float(np.float32(0.2)))[:, 0].numpy()
            assert np.abs(got[i, 0] - want).max() < 1e-12


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]


def main(argv) -> int:
    sys.path.insert(0, os.path.dirname(HERE))
    import oracle as _oracle
    o = _oracle.load(argv[1]) if len(argv) > 1 else _oracle.get()
    failed = 0
    for pin in PINS:
        try:
            pin(o)
        except AssertionError as e:          # a pin that disagrees
            failed += 1
            print(f"FAIL {pin.__name__}: {e}")
        except Exception as e:               # a crash counts as a failure too
            failed += 1
            print(f"ERROR {pin.__name__}: {type(e).__name__}: {e}")
    return failed


if __name__ == "__main__":
    sys.exit(min(main(sys.argv), 100))

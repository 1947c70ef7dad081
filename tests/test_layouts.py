"""Shared-memory and fragment layouts of the decode kernels, checked on the CPU.

TMA writes every K/V tile with the 128-byte swizzle: 16-byte chunk c of row t of a
128-byte-wide sub-tile sits at chunk position c ^ (t % 8).  A warp's 16-byte
shared load is served in 4 phases of 8 lanes and is conflict-free when the 8 lanes
of a phase hit 8 distinct 16-byte bank groups; an ldmatrix reads each 8-row
matrix in one phase.  Each load pattern below restates the index arithmetic of one
path.  The FP8 paths' register-widened fragments are emulated lane by lane on the
operand layouts of mma.sync m16n8k16 and compared with the dense products.
"""
import numpy as np
import pytest


def sw128(rows: int, row: int, chunk: int) -> int:
    """Byte offset of 16-byte chunk `chunk` of token row `row` in a 16-bit tile of
    `rows` rows: 128-column heads are two 64-column sub-tiles."""
    return (chunk >> 3) * (rows * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4)


def sw128_row128(row: int, chunk: int) -> int:
    """The same for an FP8 tile: one 128-byte row per token."""
    return row * 128 + ((chunk ^ (row & 7)) << 4)


def conflict_free(addr_of_lane) -> bool:
    for ph in range(4):
        groups = {(addr_of_lane(l) >> 4) & 7 for l in range(8 * ph, 8 * ph + 8)}
        if len(groups) != 8:
            return False
    return True


@pytest.mark.parametrize("D,K", [(128, 4), (128, 8), (64, 4), (64, 8)])
def test_cuda_core_path_loads(D, K):
    # K lanes share a token, each holding CH chunks; D = 128 rotates a lane's chunk
    # loop by (lane >> shift) % CH
    CH, TPP = D // 8 // K, 32 // K
    rotate, shift = (D == 128 and K in (4, 8)), (2 if K == 8 else 0)
    for p in range(16 // TPP):
        for jj in range(CH):
            def addr(l):
                part, tip = l % K, l // K
                rot = (l >> shift) % CH
                chunk = part * CH + (((jj + rot) % CH) if rotate else jj)
                return sw128(16, p * TPP + tip, chunk)
            assert conflict_free(addr), (D, K, p, jj)


def test_cuda_core_path_needs_its_rotation():
    # without the rotation, D = 128 with 4 lanes per token would conflict
    D, K = 128, 4
    CH = D // 8 // K
    assert not all(conflict_free(lambda l, jj=jj: sw128(16, l // K, (l % K) * CH + jj))
                   for jj in range(CH))


def test_fp8_cuda_core_path_loads():
    K, CH, TPP = 4, 2, 8
    for p in range(2):
        for jj in range(CH):
            assert conflict_free(lambda l: sw128_row128(p * TPP + l // K, (l % K) * CH + jj))


@pytest.mark.parametrize("D", [64, 128])
def test_tensor_core_ldmatrix_rows(D):
    # swapped-operand path: matrix mi of an ldmatrix.x4 takes rows (tokens)
    # ri + 8 (mi & 1) of chunk 2 ks + (mi >> 1) (K) or tokens ri + 8 (mi >> 1) of
    # chunk 2 mt + (mi & 1) (V, transposed); each matrix is one phase
    for ks in range(D // 16):
        k_rows = lambda l: sw128(16, (l & 7) + (((l >> 3) & 1) << 3), 2 * ks + (l >> 4))
        v_rows = lambda l: sw128(16, (l & 7) + ((l >> 4) << 3), 2 * ks + ((l >> 3) & 1))
        assert conflict_free(k_rows) and conflict_free(v_rows)


def test_fp8_tensor_core_path_loads():
    g = lambda l: l >> 2
    c = lambda l: l & 3
    for h in range(2):       # K: tokens g and g + 8, chunks 2c and 2c + 1
        for t8 in (0, 8):
            assert conflict_free(lambda l: sw128_row128(g(l) + t8, 2 * c(l) + h))
    for dt in (0, 1, 8, 9):  # V: tokens 2c, 2c + 1, 2c + 8, 2c + 9, chunk g
        assert conflict_free(lambda l: sw128_row128(2 * c(l) + dt, g(l)))


# ------------------------------------------------------------------ m16n8k16 emulation
def mma(afr, bfr):
    """D = A B from the per-lane fragments: lane (g, c) holds A[g][2c..2c+1],
    A[g+8][2c..], A[g][2c+8..], A[g+8][2c+8..] and B[2c..2c+1][g], B[2c+8..][g]."""
    A, B = np.full((16, 16), np.nan), np.full((16, 8), np.nan)
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        a, b = afr[lane], bfr[lane]
        A[g, 2 * c:2 * c + 2], A[g + 8, 2 * c:2 * c + 2] = a[0], a[1]
        A[g, 2 * c + 8:2 * c + 10], A[g + 8, 2 * c + 8:2 * c + 10] = a[2], a[3]
        B[2 * c:2 * c + 2, g], B[2 * c + 8:2 * c + 10, g] = b[0], b[1]
    assert not np.isnan(A).any() and not np.isnan(B).any()
    return A @ B


def accum(D):
    """Accumulator fragment: lane (g, c) holds D[g][2c], D[g][2c+1], D[g+8][2c],
    D[g+8][2c+1]."""
    return [[D[l >> 2, 2 * (l & 3)], D[l >> 2, 2 * (l & 3) + 1],
             D[(l >> 2) + 8, 2 * (l & 3)], D[(l >> 2) + 8, 2 * (l & 3) + 1]] for l in range(32)]


def byte_perm(a, b, sel):
    """prmt.b32 / __byte_perm: result byte i is byte sel[i] of (b:a)."""
    src = list(a) + list(b)
    return [src[(sel >> (4 * i)) & 0xF] for i in range(4)]


@pytest.fixture
def tile():
    rng = np.random.default_rng(0)
    return (rng.standard_normal((16, 128)), rng.standard_normal((16, 128)),
            rng.standard_normal((8, 128)), rng.random((16, 8)), rng.standard_normal((16, 128)),
            rng.random((16, 16)))


def test_fp8_swapped_path_fragments(tile):
    K, V, q, Pt, _, _ = tile   # K, V [token][dim], q [row][dim], P^T [token][row]
    # S^T = K q^T: lane c's k slots of k-step ks are dims 32c + 4ks .. +3
    ST = np.zeros((16, 8))
    for ks in range(8):
        afr, bfr = [], []
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            d0 = 32 * c + 4 * ks
            w0, w8 = K[g, d0:d0 + 4], K[g + 8, d0:d0 + 4]
            afr.append([w0[0:2], w8[0:2], w0[2:4], w8[2:4]])
            bfr.append([q[g, d0:d0 + 2], q[g, d0 + 2:d0 + 4]])
        ST += mma(afr, bfr)
    np.testing.assert_allclose(ST, K @ q.T, rtol=1e-12, atol=1e-12)
    # O^T += V^T P^T: row g of m-tile b is dim 16g + 2b, row g + 8 is dim 16g + 2b + 1
    OT = np.zeros((128, 8))
    for j in range(4):
        for b, sel in ((2 * j, 0x5140), (2 * j + 1, 0x7362)):
            afr, bfr = [], []
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                s = slice(16 * g + 4 * j, 16 * g + 4 * j + 4)
                p01 = byte_perm(V[2 * c, s], V[2 * c + 1, s], sel)
                p89 = byte_perm(V[2 * c + 8, s], V[2 * c + 9, s], sel)
                afr.append([p01[0:2], p01[2:4], p89[0:2], p89[2:4]])
                bfr.append([Pt[2 * c:2 * c + 2, g], Pt[2 * c + 8:2 * c + 10, g]])
            frag = accum(mma(afr, bfr))
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                for e in range(2):
                    OT[16 * g + 2 * b, 2 * c + e] += frag[lane][e]
                    OT[16 * g + 2 * b + 1, 2 * c + e] += frag[lane][2 + e]
    np.testing.assert_allclose(OT, V.T @ Pt, rtol=1e-12, atol=1e-12)


def test_fp8_sixteen_row_path_fragments(tile):
    K, V, _, _, Q, P = tile    # Q [row][dim], P [row][token]
    for nt in range(2):        # S = Q K^T, tokens nt*8 .. nt*8 + 7 as the n-tile
        S = np.zeros((16, 8))
        for ks in range(8):
            afr, bfr = [], []
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                d0 = 32 * c + 4 * ks
                afr.append([Q[g, d0:d0 + 2], Q[g + 8, d0:d0 + 2],
                            Q[g, d0 + 2:d0 + 4], Q[g + 8, d0 + 2:d0 + 4]])
                k = K[nt * 8 + g, d0:d0 + 4]
                bfr.append([k[0:2], k[2:4]])
            S += mma(afr, bfr)
        np.testing.assert_allclose(S, Q @ K[nt * 8:nt * 8 + 8].T, rtol=1e-12, atol=1e-12)
    # O += P V: column n of n-tile nt is dim 16n + nt
    O = np.zeros((16, 128))
    for j in range(4):
        for t in range(4):
            nt, sel, h = 4 * j + t, (0x5140 if t < 2 else 0x7362), 2 * (t & 1)
            afr, bfr = [], []
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                afr.append([P[g, 2 * c:2 * c + 2], P[g + 8, 2 * c:2 * c + 2],
                            P[g, 2 * c + 8:2 * c + 10], P[g + 8, 2 * c + 8:2 * c + 10]])
                s = slice(16 * g + 4 * j, 16 * g + 4 * j + 4)
                p01 = byte_perm(V[2 * c, s], V[2 * c + 1, s], sel)
                p89 = byte_perm(V[2 * c + 8, s], V[2 * c + 9, s], sel)
                bfr.append([p01[h:h + 2], p89[h:h + 2]])
            frag = accum(mma(afr, bfr))
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                for hr in range(2):
                    O[g + 8 * hr, 32 * c + nt] += frag[lane][2 * hr]
                    O[g + 8 * hr, 32 * c + 16 + nt] += frag[lane][2 * hr + 1]
    np.testing.assert_allclose(O, P @ V, rtol=1e-12, atol=1e-12)


def test_byte_perm_pairs_tokens_per_dim():
    a, b = [10, 11, 12, 13], [20, 21, 22, 23]   # dims 0..3 of two tokens
    assert byte_perm(a, b, 0x5140) == [10, 20, 11, 21]
    assert byte_perm(a, b, 0x7362) == [12, 22, 13, 23]


# ------------------------------------------------------------ many-row (prefill) kernel
@pytest.mark.parametrize("PB", [64])
def test_prefill_epilogue_scratch(PB):
    """The epilogue's transpose: lane l writes its row's CPR chunks at
    l*PB + 16*(c ^ swz(l)); lane l then reads chunk c = l % CPR of row
    RPI*j + l // CPR.  Both directions conflict-free, and every (row, chunk) read
    back is the one written."""
    CPR = PB // 16
    RPI = 32 // CPR

    def swz(r):
        return (r // (8 // CPR)) % CPR

    def waddr(l, c):
        return l * PB + ((c ^ swz(l)) << 4)

    for c in range(CPR):
        assert conflict_free(lambda l: waddr(l, c))
    stored = {waddr(l, c): (l, c) for l in range(32) for c in range(CPR)}
    assert len(stored) == 32 * CPR and max(stored) < 32 * PB
    for j in range(CPR):
        def raddr(l):
            r = RPI * j + l // CPR
            return r * PB + (((l % CPR) ^ swz(r)) << 4)
        assert conflict_free(raddr)
        for l in range(32):
            assert stored[raddr(l)] == (RPI * j + l // CPR, l % CPR)


@pytest.mark.parametrize("CG", [2])
def test_prefill_p_columns_match_the_pv_operand(CG):
    """P_j in tensor memory (CG column groups, one softmax warp each per 32 rows):
    the softmax warp of column group g writes positions
    g*kCols + 2e, +1 of a 128-position chunk into word column g*kCols + e (hi) and
    g*kCols + kCols/2 + e (lo); the P V MMA's K step kk reads positions 16kk..16kk+15
    from 8 word columns at pc = (kk // kSteps)*kCols + (kk % kSteps)*8 (lo at
    + kCols/2).  Every position lands where the MMA reads it, and hi and lo never
    overlap another group's columns."""
    chunk = 128
    kCols = chunk // CG
    kSteps = kCols // 16
    written_hi, written_lo = {}, {}
    for g in range(CG):
        for e in range(kCols // 2):
            for p in (0, 1):
                pos = g * kCols + 2 * e + p
                written_hi[pos] = (g * kCols + e, p)
                written_lo[pos] = (g * kCols + kCols // 2 + e, p)
    cols = [c for c, _ in written_hi.values()] + [c for c, _ in written_lo.values()]
    assert sorted(set(cols)) == list(range(chunk))        # the chunk's 128 columns, each used
    for kk in range(chunk // 16):
        pc = (kk // kSteps) * kCols + (kk % kSteps) * 8
        for i in range(16):                                 # k index inside the step
            pos = 16 * kk + i
            assert written_hi[pos] == (pc + i // 2, i % 2)  # lower k in the low half
            assert written_lo[pos] == (pc + kCols // 2 + i // 2, i % 2)


def test_prefill_fp8_widening_in_place():
    """The many-row kernel over an FP8 cache widens a chunk's codes in place.  Lane l
    of a widening warp handles position r = r0 + 32k + l: it reads the swizzled
    16-byte code chunks 4..7 (dims 64..127) and writes them, widened, to the second
    half of the 16-bit tile layout ([half][128 positions][128 B], chunk c' of a row
    at c' ^ (r % 8)), then reads chunks 0..3 and writes the first half, which lies
    over the codes row.  Simulated byte for byte: every code is read before it is
    overwritten, every fp16 dim lands where the MMA reads it, and each phase's
    loads and stores are conflict-free."""
    chunk = 128
    mem = {}
    for r in range(chunk):
        for c in range(8):
            for b in range(16):
                mem[r * 128 + ((c ^ (r & 7)) << 4) + b] = ("code", r, 16 * c + b)
    for k in range(chunk // 32):
        for h in (1, 0):
            for i in range(4):
                c = 4 * h + i
                assert conflict_free(lambda l: (32 * k + l) * 128 + ((c ^ ((32 * k + l) & 7)) << 4))
            got = {}
            for l in range(32):                          # all loads of the phase first
                r = 32 * k + l
                for i in range(4):
                    c = 4 * h + i
                    a = r * 128 + ((c ^ (r & 7)) << 4)
                    got[(l, i)] = [mem[a + b] for b in range(16)]
                    assert got[(l, i)] == [("code", r, 16 * c + b) for b in range(16)]
            for i in range(4):
                for f in (2 * i, 2 * i + 1):
                    def waddr(l):
                        r = 32 * k + l
                        return h * chunk * 128 + r * 128 + ((f ^ (r & 7)) << 4)
                    assert conflict_free(waddr)
                    for l in range(32):
                        r = 32 * k + l
                        for b in range(8):              # 8 fp16 values = 16 bytes
                            dim = 16 * (4 * h + i) + 8 * (f - 2 * i) + b
                            mem[waddr(l) + 2 * b] = ("fp16", r, dim)
                            mem[waddr(l) + 2 * b + 1] = ("fp16", r, dim)
    # the 16-bit layout: dims 64h + 8f' .. +7 of position r at h*16384 + 128r + ((f' ^ r%8) << 4)
    for r in range(chunk):
        for h in range(2):
            for fp in range(8):
                a = h * chunk * 128 + r * 128 + ((fp ^ (r & 7)) << 4)
                for b in range(8):
                    assert mem[a + 2 * b] == ("fp16", r, 64 * h + 8 * fp + b)


def _tile_walk(tb, te, kvh, num_kv_heads, gw, TW):
    """The tiles cluster warp gw reads, in the decode kernel's order: tile number
    k = gw + TW n, rotated by rot = kvh * ntiles / num_kv_heads."""
    ntiles = te - tb
    if ntiles <= 0:
        return []
    rot = (kvh * ntiles) // num_kv_heads
    n_my = (ntiles - gw + TW - 1) // TW if ntiles - gw > 0 else 0
    out = []
    for n in range(n_my):
        k = gw + TW * n + rot
        if k >= ntiles:
            k -= ntiles
        out.append(tb + k)
    return out


def _reads_new(L, q_len, tb, te, kvh, num_kv_heads, crank, NW, TW):
    """The fused append's test: does CTA crank read a tile holding a new position
    (the inverse of the walk, as the kernel computes it)."""
    ntiles = te - tb
    if ntiles <= 0:
        return False
    rot = (kvh * ntiles) // num_kv_heads
    j1 = min(te, (L + 15) // 16)
    for j in range(max(tb, max(0, L - q_len) // 16), j1):
        k = j - tb - rot
        if k < 0:
            k += ntiles
        if (k % TW) // NW == crank:
            return True
    return False


@pytest.mark.parametrize("NW,csize", [(4, 1), (4, 2), (3, 4), (4, 8)])
def test_fused_append_owner_matches_the_tile_walk(NW, csize):
    """The CTAs that append are exactly those whose warps' walks contain a tile of
    a new position; every tile of the unit is walked by exactly one warp."""
    TW = NW * csize
    rng = np.random.default_rng(3)
    for _ in range(400):
        L = int(rng.integers(0, 700))
        q_len = int(rng.integers(1, 17))
        kvh, H = int(rng.integers(0, 8)), 8
        nb = (L + 15) // 16
        # a partition [tb, te) of the tiles, as the split pass takes them
        tb = int(rng.integers(0, nb + 1))
        te = int(rng.integers(tb, nb + 1))
        walks = [_tile_walk(tb, te, kvh, H, gw, TW) for gw in range(TW)]
        flat = sorted(t for w in walks for t in w)
        assert flat == list(range(tb, te))
        new_tiles = {p // 16 for p in range(max(0, L - q_len), L)}
        for crank in range(csize):
            mine = {t for gw in range(crank * NW, crank * NW + NW) for t in walks[gw]}
            assert _reads_new(L, q_len, tb, te, kvh, H, crank, NW, TW) == bool(mine & new_tiles)

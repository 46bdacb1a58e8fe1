"""The tensor-core GEMVs' index arithmetic, emulated on the CPU (no GPU).

The kernel's GEMVs feed mma.sync m16n8k16 (BF16 in, fp32 accumulate) from
weight stages that a tensor copy lands with the 128-byte swizzle, and read the
products back from per-lane accumulator fragments.  Every index in that chain
(the stage layout, the ldmatrix row addresses, which activation column each
lane loads, which accumulator entries each lane keeps, the shuffles that add a
row's parts, the slot of each partial sum) is restated here from the kernel's
formulas and run on random data with the PTX fragment layouts of ldmatrix.x4
and m16n8k16:

* ldmatrix.x4: lane 8 i + g gives the address of row g of 8 x 8 tile i; tile
  i fills A rows 8 (i & 1) + 0..7, columns 8 (i >> 1) + 0..7;
* B fragment: lane (g = lane / 4, c = lane % 4) holds B[2c][g], B[2c + 1][g]
  in its first register and B[2c + 8][g], B[2c + 9][g] in its second;
* C fragment: the same lane holds C[g][2c], C[g][2c + 1], C[g + 8][2c],
  C[g + 8][2c + 1].

The checks: the swizzled stage is a bijection onto its 32 KB; the eight rows
of every ldmatrix tile fall in distinct 16-byte bank groups (no bank
conflict); and the partial sums, added over the warps as the kernel's
epilogue adds them, equal W (x_hi + x_lo) for every row and token.  The high
and low halves of x are drawn independently, so a dropped, doubled or swapped
half fails.  A dropped term, a wrong part or token index, or a transposed
operand fails the equality; the partial-slot bound is checked for every chunk
the producer can hand over.  The 8-bit expert paths (m16n8k32 with E4M3
operands, x as four E4M3 terms) and the attention's two products on a staged
page (ldmatrix .trans for V, movmatrix for P^T) are checked the same way
further down.
"""
from __future__ import annotations

import numpy as np
import pytest

STAGE_BYTES = 32768
PART_FLOATS = 2048          # one GEMV partial-sum buffer (floats)
WARPS = 8                   # consumer warps
LANES = np.arange(32)


def swizzled_stage(W: np.ndarray, rows_per_box: int) -> np.ndarray:
    """Rows of W as one stage [K / 64 column blocks][rows][64 columns] with the
    128-byte swizzle: the 16-byte chunk c of 128-byte line L sits at chunk
    c ^ (L & 7).  Returns the stage as 2-byte slots holding the values."""
    R, K = W.shape
    r, k = np.meshgrid(np.arange(R), np.arange(K), indexing="ij")
    cb, cin = k // 64, k % 64
    line = cb * rows_per_box + r
    byte = line * 128 + ((cin // 8) ^ (line & 7)) * 16 + (cin % 8) * 2
    slot = (byte // 2).ravel()
    assert len(np.unique(slot)) == slot.size, "two elements in one slot"
    assert byte.max() < STAGE_BYTES
    st = np.full(STAGE_BYTES // 2, np.nan)
    st[slot] = W[r, k].ravel()
    return st


def ldmatrix_x4(stage: np.ndarray, addr: np.ndarray) -> np.ndarray:
    """A (16 x 16) from the 32 lanes' row addresses (bytes); asserts that each
    8 x 8 tile's rows hit eight distinct 16-byte bank groups."""
    A = np.full((16, 16), np.nan)
    for i in range(4):
        a = addr[8 * i:8 * i + 8]
        assert len(set(((a // 16) % 8).tolist())) == 8, "bank conflict"
        for g in range(8):
            A[g + 8 * (i & 1), 8 * (i >> 1):8 * (i >> 1) + 8] = stage[a[g] // 2:a[g] // 2 + 8]
    return A


def b_from_lanes(val) -> np.ndarray:
    """B (16 x 8) assembled from each lane's fragment; val(g, c, hf) returns
    the pair the lane loads for register hf."""
    B = np.zeros((16, 8))
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        for hf in range(2):
            v0, v1 = val(g, c, hf)
            B[2 * c + 8 * hf, g], B[2 * c + 1 + 8 * hf, g] = v0, v1
    return B


def c_lane(C: np.ndarray, lane: int):
    g, c = lane >> 2, lane & 3
    return C[g, 2 * c], C[g, 2 * c + 1], C[g + 8, 2 * c], C[g + 8, 2 * c + 1]


def shfl_xor(v: np.ndarray, m: int) -> np.ndarray:
    return v[LANES ^ m]


def mma_block(NH: int, warp: int, j: int, t: int) -> int:
    """Column block of part j, block t of the warp's share (rows of 2048 NH)."""
    return 4 * warp + 2 * j + t if NH == 1 else 8 * warp + 4 * (j >> 1) + 2 * t + (j & 1)


def a_offsets(NH: int, warp: int):
    """The ldmatrix row addresses of the 8 k-steps: lane row m = (row m % R,
    part m / R), column half kh = lane / 16."""
    R = 8 // NH
    off = np.zeros((8, 32), dtype=np.int64)
    for lane in range(32):
        m, kh = ((lane >> 3) & 1) * 8 + (lane & 7), lane >> 4
        for s in range(8):
            line = mma_block(NH, warp, m // R, s >> 2) * R + m % R
            off[s, lane] = line * 128 + ((((s & 3) * 2 + kh) ^ (line & 7)) << 4)
    return off


@pytest.mark.parametrize("NH", [1, 2])
def test_one_token_rows(NH):
    """gemv_mma: one token, R = 8 / NH rows of 2048 NH columns per stage."""
    rng = np.random.default_rng(10 + NH)
    K, R = 2048 * NH, 8 // NH
    W = rng.standard_normal((R, K))
    xh, xl = rng.standard_normal(K), rng.standard_normal(K)
    st = swizzled_stage(W, R)
    assert not np.isnan(st).any()                      # the stage is full
    part = np.zeros((R, WARPS))
    for warp in range(WARPS):
        aoff = a_offsets(NH, warp)
        C = np.zeros((16, 8))
        for s in range(8):
            def val(g, c, hf, s=s):
                j, lo = g >> 1, g & 1
                if j >= 2 * NH:
                    return 0.0, 0.0
                col = mma_block(NH, warp, j, s >> 2) * 64 + (s & 3) * 16 + 2 * c + hf * 8
                x = xl if lo else xh
                return x[col], x[col + 1]
            C += ldmatrix_x4(st, aoff[s]) @ b_from_lanes(val)
        v = np.zeros(32)
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            c0, c1, c2, c3 = c_lane(C, lane)
            v[lane] = (c0 + c1 if c == g // R else 0.0) + (c2 + c3 if c == (g + 8) // R else 0.0)
        v = v + shfl_xor(v, 1)
        v = v + shfl_xor(v, 2)
        if R == 4:
            v = v + shfl_xor(v, 16)
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            if c == 0 and g < R:
                part[g, warp] = v[lane]
    np.testing.assert_allclose(part.sum(1), W @ (xh + xl), rtol=1e-12, atol=1e-9)


def multi_rows(NH: int, nt: int, rows: int, rng):
    """gemv_mma_multi on one stage: NQ = ceil(nt / TPT) n-tiles, column
    n = 8 q + g of n-tile q holds token q TPT + g / (4 NH), part (g / 2) % P,
    half g % 2; returns part[row][warp][token] for the stage's first `rows`."""
    K, R, TPT = 2048 * NH, 8 // NH, 2 // NH
    NQ = (nt + TPT - 1) // TPT
    W = rng.standard_normal((R, K))
    xh, xl = rng.standard_normal((nt, K)), rng.standard_normal((nt, K))
    st = swizzled_stage(W, R)
    part = np.full((R, WARPS, nt), np.nan)
    for warp in range(WARPS):
        aoff = a_offsets(NH, warp)
        for q in range(NQ):
            C = np.zeros((16, 8))
            for s in range(8):
                def val(g, c, hf, s=s, q=q):
                    tk, j, lo = q * TPT + g // (4 * NH), (g >> 1) & (2 * NH - 1), g & 1
                    if tk >= nt:
                        return 0.0, 0.0
                    col = mma_block(NH, warp, j, s >> 2) * 64 + (s & 3) * 16 + hf * 8 + 2 * c
                    x = xl if lo else xh
                    return x[tk, col], x[tk, col + 1]
                C += ldmatrix_x4(st, aoff[s]) @ b_from_lanes(val)
            v = np.zeros(32)
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                pc = c & (2 * NH - 1)
                c0, c1, c2, c3 = c_lane(C, lane)
                v[lane] = (c0 + c1 if pc == g // R else 0.0) + (c2 + c3 if pc == (g + 8) // R else 0.0)
            v = v + shfl_xor(v, 1)
            if NH == 2:
                v = v + shfl_xor(v, 2)
                v = v + shfl_xor(v, 16)
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                tk = q * TPT + ((c >> 1) if NH == 1 else 0)
                writer = (not (c & 1)) if NH == 1 else (c == 0 and g < R)
                if writer and g < rows and tk < nt:
                    assert np.isnan(part[g, warp, tk]), "two writers of one partial"
                    part[g, warp, tk] = v[lane]
    return part, W, xh + xl


@pytest.mark.parametrize("NH,nt", [(1, 1), (1, 2), (1, 3), (1, 5), (1, 8), (2, 1), (2, 2), (2, 3), (2, 4)])
def test_several_token_rows(NH, nt):
    rng = np.random.default_rng(100 * NH + nt)
    R = 8 // NH
    part, W, x = multi_rows(NH, nt, R, rng)
    assert not np.isnan(part).any()
    np.testing.assert_allclose(part.sum(1), W @ x.T, rtol=1e-12, atol=1e-9)


def test_several_token_ragged_stage_writes_only_its_rows():
    part, W, x = multi_rows(1, 4, 5, np.random.default_rng(3))
    assert np.isnan(part[5:]).all()
    np.testing.assert_allclose(part[:5].sum(1), (W @ x.T)[:5], rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("K,nt", [(128, 1), (256, 3), (768, 4), (768, 7), (768, 16), (1024, 5), (1024, 16)])
def test_down_rows(K, nt):
    """gemv_mma_down: 16 rows of K (a multiple of 128, at most 1024) per stage
    as [K / 64 blocks][16 rows][64], warp w takes columns [w K / 8, (w + 1) K / 8)
    in K / 128 k-steps; column n = 8 q + g of n-tile q holds token 4 q + g / 2,
    half g % 2."""
    rng = np.random.default_rng(K + nt)
    R, ks, NQ = 16, K >> 7, (nt + 3) >> 2
    W = rng.standard_normal((R, K))
    xh, xl = rng.standard_normal((nt, K)), rng.standard_normal((nt, K))
    st = swizzled_stage(W, R)
    part = np.full((R, WARPS, nt), np.nan)
    for warp in range(WARPS):
        col0 = warp * (K >> 3)
        aoff = np.zeros((8, 32), dtype=np.int64)
        for lane in range(32):
            m, kh = ((lane >> 3) & 1) * 8 + (lane & 7), lane >> 4
            for s in range(ks):
                col = col0 + 16 * s + 8 * kh
                line = (col >> 6) * R + m
                aoff[s, lane] = line * 128 + ((((col & 63) >> 3) ^ (line & 7)) << 4)
        for q in range(NQ):
            C = np.zeros((16, 8))
            for s in range(ks):
                def val(g, c, hf, s=s, q=q):
                    tk, lo = 4 * q + (g >> 1), g & 1
                    if tk >= nt:
                        return 0.0, 0.0
                    col = col0 + 16 * s + 8 * hf + 2 * c
                    x = xl if lo else xh
                    return x[tk, col], x[tk, col + 1]
                C += ldmatrix_x4(st, aoff[s]) @ b_from_lanes(val)
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                tk = 4 * q + c
                if tk < nt:
                    c0, c1, c2, c3 = c_lane(C, lane)
                    part[g, warp, tk] = c0 + c1
                    part[g + 8, warp, tk] = c2 + c3
    assert not np.isnan(part).any()
    np.testing.assert_allclose(part.sum(1), W @ (xh + xl).T, rtol=1e-12, atol=1e-9)


def _chunk_rows(K: int, nt: int) -> int:
    """Rows of one dense GEMV chunk: the partial buffer holds rows x segments x
    tokens floats (segments = K / 256), at most 512 rows."""
    nseg = 1 if K < 256 else K // 256
    return min(512, PART_FLOATS // (nseg * max(nt, 1)))


def _mma_multi_rows(K: int, nt: int) -> bool:
    return nt >= 1 and ((K == 2048 and nt <= 8) or (K == 4096 and nt <= 4))


@pytest.mark.parametrize("nt", range(1, 17))
def test_partial_slots_stay_in_the_buffer(nt):
    """Every partial slot ((blk nr + row) W + warp) nt + token a tensor-core
    chunk writes is inside one buffer, for the chunks the producer hands over:
    dense rows (one block of chunk_rows rows), an expert's gate / up rows (two
    blocks of chunk_rows / 2 rows) and its down rows (16-row multiples of at
    most buffer / (W nt) rows)."""
    for K in (2048, 4096):
        if not _mma_multi_rows(K, nt):
            continue
        for nblk, nr in ((1, _chunk_rows(K, nt)), (2, max(1, _chunk_rows(K, nt) // 2))):
            top = ((nblk - 1) * nr + nr - 1) * WARPS + WARPS - 1
            assert top * nt + nt - 1 < PART_FLOATS, (K, nt, nblk, nr)
    cd = max(16, min(512, PART_FLOATS // (WARPS * nt)) // 16 * 16)
    assert ((cd - 1) * WARPS + WARPS - 1) * nt + nt - 1 < PART_FLOATS


# ---------------------------------------------------------------- 8-bit experts
# mma.sync m16n8k32 with E4M3 operands (PTX fragment layout of the 8-bit
# types): lane (g, c) holds A[g][4c..4c+3] (a0), A[g+8][4c..] (a1),
# A[g][16+4c..] (a2), A[g+8][16+4c..] (a3), B[4c..4c+3][g] (b0) and
# B[16+4c..][g] (b1); C as above.  ldmatrix.x4 of b16 tiles hands lane l the
# 4 bytes 4 (l % 4) .. + 3 of row l / 4 of each tile.

def ldmatrix_x4_bytes(stage: np.ndarray, addr: np.ndarray):
    """Per lane, the four 4-byte registers ldmatrix.x4 returns."""
    regs = np.zeros((32, 4, 4))
    for i in range(4):
        a = addr[8 * i:8 * i + 8]
        assert len(set(((a // 16) % 8).tolist())) == 8, "bank conflict"
        for lane in range(32):
            row = a[lane >> 2]
            regs[lane, i] = stage[row + 4 * (lane & 3):row + 4 * (lane & 3) + 4]
    return regs


def a_from_regs(regs) -> np.ndarray:
    A = np.full((16, 32), np.nan)
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        A[g, 4 * c:4 * c + 4] = regs[lane][0]
        A[g + 8, 4 * c:4 * c + 4] = regs[lane][1]
        A[g, 16 + 4 * c:20 + 4 * c] = regs[lane][2]
        A[g + 8, 16 + 4 * c:20 + 4 * c] = regs[lane][3]
    return A


def b_from_words(b0, b1) -> np.ndarray:
    B = np.zeros((32, 8))
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        B[4 * c:4 * c + 4, g] = b0[lane]
        B[16 + 4 * c:20 + 4 * c, g] = b1[lane]
    return B


def term_scales(s0: float, c: int):
    """The lane's scales of its C columns 2 c and 2 c + 1 (terms 2 c, 2 c + 1;
    columns past the four terms carry nothing)."""
    return (s0 * 16.0 ** (-2 * c), s0 * 16.0 ** (-2 * c - 1)) if c < 2 else (0.0, 0.0)


@pytest.mark.parametrize("rows", [16, 11])
def test_e4m3_gate_up_rows(rows):
    """gemv_mma_e4m3: 16 rows of 2048 bytes per stage, copied as rows of 1024
    two-byte words (128-byte block cb of row r is line 16 cb + r, chunk c at
    c ^ (line & 7)); warp w takes columns [256 w, 256 w + 256) in 8 k-steps;
    N column t < 4 is x's term t.  Byte values are stand-ins (the index
    arithmetic does not depend on them)."""
    rng = np.random.default_rng(rows)
    K, s0 = 2048, 0.375
    W = rng.standard_normal((16, K))
    xq = rng.standard_normal((4, K))
    r, k = np.meshgrid(np.arange(16), np.arange(K), indexing="ij")
    line = (k // 128) * 16 + r
    byte = line * 128 + (((k % 128) // 16) ^ (line & 7)) * 16 + k % 16
    assert len(np.unique(byte)) == byte.size and byte.max() < STAGE_BYTES
    st = np.full(STAGE_BYTES, np.nan)
    st[byte.ravel()] = W[r, k].ravel()
    part = np.full((16, WARPS), np.nan)
    for warp in range(WARPS):
        C = np.zeros((16, 8))
        for s in range(8):
            addr = np.zeros(32, dtype=np.int64)
            for lane in range(32):
                rr, ch = ((lane >> 3) & 1) * 8 + (lane & 7), 2 * s + (lane >> 4)
                ln = (2 * warp + (ch >> 3)) * 16 + rr
                addr[lane] = ln * 128 + (((ch & 7) ^ (rr & 7)) << 4)
            b0, b1 = np.zeros((32, 4)), np.zeros((32, 4))
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                k0 = 256 * warp + 32 * s + 4 * c
                if g < 4:
                    b0[lane], b1[lane] = xq[g, k0:k0 + 4], xq[g, k0 + 16:k0 + 20]
            C += a_from_regs(ldmatrix_x4_bytes(st, addr)) @ b_from_words(b0, b1)
        v0, v8 = np.zeros(32), np.zeros(32)
        for lane in range(32):
            sa, sb = term_scales(s0, lane & 3)
            c0, c1, c2, c3 = c_lane(C, lane)
            v0[lane], v8[lane] = sa * c0 + sb * c1, sa * c2 + sb * c3
        v0, v8 = v0 + shfl_xor(v0, 1), v8 + shfl_xor(v8, 1)
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            if c == 0:
                if g < rows:
                    part[g, warp] = v0[lane]
                if g + 8 < rows:
                    part[g + 8, warp] = v8[lane]
    x = sum(s0 * 16.0 ** -t * xq[t] for t in range(4))
    assert np.isnan(part[rows:]).all()
    np.testing.assert_allclose(part[:rows].sum(1), (W @ x)[:rows], rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("H,ncb", [(256, 1), (256, 5), (512, 8), (1024, 3), (2048, 1), (2048, 6), (2048, 8)])
def test_e4m3_down_quads(H, ncb):
    """down_mma_e4m3: a piece's ncb groups of 8 columns arrive as quads; a
    stage holds the quad's rows [hb, hb + rd) (rd = min(H, 1024); group slot j
    at j rd 8 bytes, 8 bytes a row); lane (g, c) takes columns 4 (c & 1) ..
    + 3 of slots c >> 1 and 2 + (c >> 1) in rows h0 + g and h0 + g + 8, the
    two loads of a pair swapped between the slots' lanes; the B words are the
    hidden terms of the same columns.  The 32 lanes' words must fall in
    distinct banks."""
    rng = np.random.default_rng(H + ncb)
    s0, rd, nb = 0.0625, min(H, 1024), H // 128
    Wd = rng.standard_normal((ncb, H, 8))          # group c: [H][8]
    aq = np.zeros((4, 64))
    aq[:, :8 * ncb] = rng.standard_normal((4, 8 * ncb))
    scl = rng.standard_normal(H)
    out = np.full(H, np.nan)
    for warp in range(WARPS):
        acc = np.zeros((16, 16, 8))                  # [block][C]
        for q0 in range(0, ncb, 4):
            nq = min(4, ncb - q0)
            b0, b1 = np.zeros((32, 4)), np.zeros((32, 4))
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                g1, wsel = c >> 1, 4 * (c & 1)
                if g < 4 and g1 < nq:
                    b0[lane] = aq[g, (q0 + g1) * 8 + wsel:(q0 + g1) * 8 + wsel + 4]
                if g < 4 and 2 + g1 < nq:
                    b1[lane] = aq[g, (q0 + 2 + g1) * 8 + wsel:(q0 + 2 + g1) * 8 + wsel + 4]
            B = b_from_words(b0, b1)
            for hb in range(0, H, rd):
                st = np.full(STAGE_BYTES, np.nan)
                for j in range(nq):
                    st[j * rd * 8:(j + 1) * rd * 8] = Wd[q0 + j, hb:hb + rd].ravel()
                blocks = ([(8 * (hb // 1024) + j, 16 * warp + 128 * j) for j in range(8)] if H == 2048 else
                          [(i, 16 * (warp + 8 * i) - hb) for i in range(nb) if hb <= 16 * (warp + 8 * i) < hb + rd])
                for i, r in blocks:
                    regs = np.zeros((32, 4, 4))
                    banks = []
                    for lane in range(32):
                        g, c = lane >> 2, lane & 3
                        g1, wsel = c >> 1, 4 * (c & 1)
                        sl, sh = g1 * rd * 8 + wsel, (2 + g1) * rd * 8 + wsel
                        ra, rb = 8 * (r + g + 8 * g1), 8 * (r + g + 8 - 8 * g1)
                        onl, onh = g1 < nq, 2 + g1 < nq
                        la = st[sl + ra:sl + ra + 4] if onl else np.zeros(4)
                        lb = st[sl + rb:sl + rb + 4] if onl else np.zeros(4)
                        ha = st[sh + ra:sh + ra + 4] if onh else np.zeros(4)
                        hb2 = st[sh + rb:sh + rb + 4] if onh else np.zeros(4)
                        regs[lane] = (lb, la, hb2, ha) if g1 else (la, lb, ha, hb2)
                        banks.append(((sl + ra) // 4) % 32)
                    assert sorted(banks) == list(range(32)), "bank conflict"
                    A = a_from_regs(regs)
                    assert not np.isnan(A).any()
                    acc[i] += A @ B
        for i in range(nb):
            v0, v8 = np.zeros(32), np.zeros(32)
            for lane in range(32):
                sa, sb = term_scales(s0, lane & 3)
                c0, c1, c2, c3 = c_lane(acc[i], lane)
                v0[lane], v8[lane] = sa * c0 + sb * c1, sa * c2 + sb * c3
            v0, v8 = v0 + shfl_xor(v0, 1), v8 + shfl_xor(v8, 1)
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                if c == 0:
                    h = 16 * (warp + 8 * i) + g
                    assert np.isnan(out[h]) and np.isnan(out[h + 8])
                    out[h], out[h + 8] = v0[lane] * scl[h], v8[lane] * scl[h + 8]
    a = sum(s0 * 16.0 ** -t * aq[t] for t in range(4))
    ref = sum(Wd[c] @ a[8 * c:8 * c + 8] for c in range(ncb)) * scl
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-9)


def _e4m3(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at 448."""
    import torch
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32)).to(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def _scale0(mx: float) -> float:
    """The smallest power of two s with mx / s <= 448 (1 for mx = 0)."""
    y = np.float32(mx) / np.float32(448.0)
    if not y > 0:
        return 1.0
    m, e = np.frexp(np.float64(y))               # y = m 2^e, m in [0.5, 1)
    return float(2.0 ** (e - 1) if m == 0.5 else 2.0 ** e)


@pytest.mark.parametrize("kind", ["normal", "outliers", "tiny", "zero"])
def test_four_e4m3_terms_keep_x_to_about_16_bits(kind):
    """The activations' cut into E4M3 terms: s_0 the smallest power of two
    with max|x| / s_0 <= 448, s_t = s_0 16^-t, term t the nearest E4M3 value
    of the remainder / s_t.  No term saturates (|remainder / s_t| <= 448) and
    the four terms give x back to within 2^-16 of max|x| (each term's
    remainder is at most half its largest step)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal(4096).astype(np.float32)
    if kind == "outliers":
        x[rng.integers(0, 4096, 5)] *= 300.0
    elif kind == "tiny":
        x *= np.float32(1e-30)
    elif kind == "zero":
        x[:] = 0.0
    s0 = _scale0(float(np.abs(x).max()))
    r = x.copy()
    rec = np.zeros(4096)
    for t in range(4):
        st = np.float32(s0 * 16.0 ** -t)
        y = r / st
        assert np.abs(y).max() <= 448.0
        q = _e4m3(y)
        rec += np.float64(st) * q
        r = (r - st * q).astype(np.float32)
    bound = 2.0 ** -16 * float(np.abs(x).max())
    assert np.abs(rec - x).max() <= bound


# ------------------------------------------------------------------ attention
# One page of one KV group g, as a warp of the attention item sees it.  The
# page image holds rows = hkv x 16 rows (head-major: row g P + token) of D
# dims as boxes of 64 dims, 128-byte swizzled; the query is staged as [head][D]
# with 16-byte chunk c of row h at c ^ (h & 7).  ldmatrix .trans hands lane l
# the pair (2 (l % 4), l / 4), (2 (l % 4) + 1, l / 4) of each tile as stored;
# movmatrix .trans turns lane l's pair of row l / 4 into the same pair of the
# transposed 8 x 8 block.

PAGE = 16


def kv_off(r: int, c: int, rows: int) -> int:
    return (c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4)


def page_image(KV: np.ndarray) -> np.ndarray:
    """KV [hkv][16][D] as the staged page image, in 2-byte slots."""
    hkv, P, D = KV.shape
    rows = hkv * P
    img = np.full(rows * D, np.nan)
    for g in range(hkv):
        for t in range(P):
            for k in range(D):
                o = kv_off(g * P + t, k >> 3, rows) + (k & 7) * 2
                assert np.isnan(img[o // 2])
                img[o // 2] = KV[g, t, k]
    assert not np.isnan(img).any()
    return img


def ldmatrix_x4_trans(stage: np.ndarray, addr: np.ndarray) -> np.ndarray:
    A = np.full((16, 16), np.nan)
    for i in range(4):
        a = addr[8 * i:8 * i + 8]
        assert len(set(((a // 16) % 8).tolist())) == 8, "bank conflict"
        tile = np.array([stage[a[g] // 2:a[g] // 2 + 8] for g in range(8)])
        A[8 * (i & 1):8 * (i & 1) + 8, 8 * (i >> 1):8 * (i >> 1) + 8] = tile.T
    return A


def movmatrix_trans(pairs: np.ndarray) -> np.ndarray:
    """pairs[lane] = (X[l / 4][2 (l % 4)], X[l / 4][2 (l % 4) + 1]) of an 8 x 8
    block X; returns the same pairs of X^T."""
    X = np.zeros((8, 8))
    for lane in range(32):
        X[lane >> 2, 2 * (lane & 3):2 * (lane & 3) + 2] = pairs[lane]
    out = np.zeros((32, 2))
    for lane in range(32):
        out[lane] = X.T[lane >> 2, 2 * (lane & 3):2 * (lane & 3) + 2]
    return out


def b_from_pairs(b0: np.ndarray, b1: np.ndarray) -> np.ndarray:
    """m16n8k16 B from each lane's two registers (pairs of rows 2c, 2c + 1 and
    2c + 8, 2c + 9 of column g)."""
    B = np.zeros((16, 8))
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        B[2 * c:2 * c + 2, g] = b0[lane]
        B[8 + 2 * c:8 + 2 * c + 2, g] = b1[lane]
    return B


@pytest.mark.parametrize("D,hkv,grp,lo_t,hi_t", [(128, 4, 8, 0, 16), (128, 4, 8, 3, 11), (64, 2, 2, 0, 16),
                                                 (128, 8, 4, 5, 16), (64, 4, 3, 0, 7)])
def test_attention_page_fragments(D, hkv, grp, lo_t, hi_t):
    """S^T = K Q^T (A: the group's K rows by ldmatrix, B: Q^T from the swizzled
    query staging, high and low halves) and O^T = V^T P^T (A: ldmatrix .trans
    of the V rows, B: the score fragments' probabilities transposed by
    movmatrix, high and low halves): every group g, every valid token and
    every head of the group, for both D."""
    rng = np.random.default_rng(D + hkv + grp + lo_t)
    KS, rows, hq = D // 16, hkv * PAGE, hkv * grp
    Kp, Vp = rng.standard_normal((hkv, PAGE, D)), rng.standard_normal((hkv, PAGE, D))
    kimg, vimg = page_image(Kp), page_image(Vp)
    qh, ql = rng.standard_normal((hq, D)), rng.standard_normal((hq, D))
    qhi, qlo = np.full(hq * D, np.nan), np.full(hq * D, np.nan)
    for h in range(hq):
        for k in range(D):
            o = h * D * 2 + (((k >> 3) ^ (h & 7)) << 4) + (k & 7) * 2
            qhi[o // 2], qlo[o // 2] = qh[h, k], ql[h, k]
    ph, pl = rng.standard_normal((PAGE, 8)), rng.standard_normal((PAGE, 8))   # [token][head]
    for g in range(hkv):
        # B fragments of Q^T
        qb = {}
        for s in range(KS):
            for which, img in (("h", qhi), ("l", qlo)):
                regs = np.zeros((2, 32, 2))
                for lane in range(32):
                    gl, cq = lane >> 2, lane & 3
                    qrow = g * grp + gl
                    for hf in range(2):
                        off = qrow * D * 2 + (((2 * s + hf) ^ (qrow & 7)) << 4) + 4 * cq
                        regs[hf, lane] = img[off // 2:off // 2 + 2] if gl < grp else 0.0
                qb[s, which] = b_from_pairs(regs[0], regs[1])
        # S^T = K Q^T
        C = np.zeros((16, 8))
        for s in range(KS):
            addr = np.array([kv_off(g * PAGE + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * s + (lane >> 4), rows)
                             for lane in range(32)])
            A = ldmatrix_x4(kimg, addr)
            C += A @ qb[s, "h"] + A @ qb[s, "l"]
        ref = Kp[g] @ (qh + ql)[g * grp:g * grp + grp].T          # [token][head]
        for lane in range(32):
            gl, cq = lane >> 2, lane & 3
            c0, c1, c2, c3 = c_lane(C, lane)
            for tok, hd, v in ((gl, 2 * cq, c0), (gl, 2 * cq + 1, c1), (gl + 8, 2 * cq, c2), (gl + 8, 2 * cq + 1, c3)):
                if hd < grp:
                    assert abs(v - ref[tok, hd]) < 1e-9, (g, tok, hd)
                else:
                    assert v == 0.0                                  # no padded head carries a score
        # O^T += V^T P^T with the lanes' probabilities (invalid rows give 0)
        pv = {}
        for which, src in (("h", ph), ("l", pl)):
            p01, p23 = np.zeros((32, 2)), np.zeros((32, 2))
            for lane in range(32):
                gl, cq = lane >> 2, lane & 3
                ok0, ok1 = lo_t <= gl < hi_t, lo_t <= gl + 8 < hi_t
                p01[lane] = src[gl, 2 * cq:2 * cq + 2] if ok0 else 0.0
                p23[lane] = src[gl + 8, 2 * cq:2 * cq + 2] if ok1 else 0.0
            pv[which] = b_from_pairs(movmatrix_trans(p01), movmatrix_trans(p23))
        P = np.zeros((PAGE, 8))
        P[lo_t:hi_t] = (ph + pl)[lo_t:hi_t]
        oref = Vp[g].T @ P                                           # [dim][head]
        for s in range(KS):
            addr = np.array([kv_off(g * PAGE + (lane >> 4) * 8 + (lane & 7), 2 * s + ((lane >> 3) & 1), rows)
                             for lane in range(32)])
            A = ldmatrix_x4_trans(vimg, addr)
            O = A @ pv["h"] + A @ pv["l"]
            for lane in range(32):
                gl, cq = lane >> 2, lane & 3
                o0, o1, o2, o3 = c_lane(O, lane)
                for dim, hd, v in ((16 * s + gl, 2 * cq, o0), (16 * s + gl, 2 * cq + 1, o1),
                                   (16 * s + 8 + gl, 2 * cq, o2), (16 * s + 8 + gl, 2 * cq + 1, o3)):
                    assert abs(v - oref[dim, hd]) < 1e-9, (g, s, dim, hd)

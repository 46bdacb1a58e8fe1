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
the producer can hand over.
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

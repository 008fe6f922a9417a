"""A CPU model of how the 4-bit decode projection (gemm_q4r.cu) feeds mma.sync m16n8k16.

Each lane loads two code words per 16-row block and group of 64 columns straight from the
native block layout, turns each pair of codes into one bf16x2 A register, and takes its B
registers from the staged operand row in plain column order.  Rebuilding the 16 x 16 A tile
and the 16 x 8 B tile of every MMA from the per-lane registers, by the fragment layout of the
PTX ISA (row/column of each register element as a function of the lane), must show that
every MMA pairs a weight and an operand value of the same column, that the four MMAs of a
group cover its 64 columns exactly once, and that the fold
    y = s * sum (128 + q) x + (b - 128 s) * sum x
equals the dequantised product.  A planted change of the column order on one side fails.
"""
import numpy as np
import pytest


def native_word(codes8):
    """Eight codes (columns 8i .. 8i+7) as the native word: pair p = (bits 4p.., bits 16+4p..)
    holds columns 2p and 2p + 1."""
    w = 0
    for p in range(4):
        w |= int(codes8[2 * p]) << (4 * p)
        w |= int(codes8[2 * p + 1]) << (16 + 4 * p)
    return w


def unpack_pair(w, p):
    """The kernel's (w >> 4p) & 0x000F000F | 0x43004300, as the two values it encodes."""
    v = ((w >> (4 * p)) & 0x000F000F) | 0x43004300
    lo, hi = v & 0xFFFF, v >> 16
    # bf16 0x4300 | q is 128 + q exactly (ulp 1 at 128)
    return 128 + (lo & 0xF), 128 + (hi & 0xF)


def group_tiles(q16x64, x8x64, swap_b_pairs=False):
    """The 4 MMAs of one 64-column group for a 16-row block: per MMA the (A, B) tiles rebuilt
    from the lanes' registers, plus the column each k index came from on each side."""
    # native words of each row: word i covers columns 8i .. 8i + 7 of the group
    words = [[native_word(q16x64[r, 8 * i:8 * i + 8]) for i in range(8)] for r in range(16)]
    tiles = []
    for j in range(4):
        A = np.zeros((16, 16))
        B = np.zeros((16, 8))
        colA = -np.ones((16, 16), int)
        colB = -np.ones(16, int)
        for lane in range(32):
            g, t = lane >> 2, lane & 3
            jp = j >> 1
            # lane (g, t) holds columns 16t .. 16t+15 of rows g and g+8: words 2t + jp
            wa, wb = words[g][2 * t + jp], words[g + 8][2 * t + jp]
            pp = 2 * (j & 1)
            regs = [(unpack_pair(wa, pp), g, 2 * t), (unpack_pair(wb, pp), g + 8, 2 * t),
                    (unpack_pair(wa, pp + 1), g, 2 * t + 8), (unpack_pair(wb, pp + 1), g + 8, 2 * t + 8)]
            base = 16 * t + 8 * jp + 4 * (j & 1)
            for r, ((v0, v1), row, k0) in enumerate(regs):
                A[row, k0], A[row, k0 + 1] = v0, v1
                c0 = base + (2 if r >= 2 else 0)
                colA[row, k0], colA[row, k0 + 1] = c0, c0 + 1
            # B registers: operand row n = g, columns 16t + 4j' .. (plain order of the row)
            xs = x8x64[g, 16 * t:16 * t + 16]
            b01 = xs[4 * j:4 * j + 2]
            b23 = xs[4 * j + 2:4 * j + 4]
            if swap_b_pairs:
                b01, b23 = b23, b01
            B[2 * t, g], B[2 * t + 1, g] = b01
            B[2 * t + 8, g], B[2 * t + 9, g] = b23
            colB[2 * t], colB[2 * t + 1] = 16 * t + 4 * j, 16 * t + 4 * j + 1
            colB[2 * t + 8], colB[2 * t + 9] = 16 * t + 4 * j + 2, 16 * t + 4 * j + 3
        tiles.append((A, B, colA, colB))
    return tiles


@pytest.mark.parametrize("seed", [0, 1])
def test_fragments_pair_same_columns_and_fold_is_exact(seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, (16, 64))
    x = rng.normal(size=(8, 64))
    s = rng.uniform(0.001, 0.01, 16)
    b = rng.uniform(-0.05, 0.0, 16)
    tiles = group_tiles(q, x)
    seen = np.zeros((16, 64), int)
    acc = np.zeros((16, 8))
    for A, B, colA, colB in tiles:
        for r in range(16):
            assert (colA[r] == colB).all()  # A[r, k] and B[k, :] come from one column
            seen[r, colA[r]] += 1
        acc += A @ B
    assert (seen == 1).all()  # the four MMAs cover the 64 columns once each
    X = x.sum(axis=1)
    y = s[:, None] * acc + (b - 128 * s)[:, None] * X[None, :]
    ref = (s[:, None] * q + b[:, None]) @ x.T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_planted_operand_order_change_is_caught():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, (16, 64))
    x = rng.normal(size=(8, 64))
    acc = sum(A @ B for A, B, _, _ in group_tiles(q, x, swap_b_pairs=True))
    ref = (128 + q) @ x.T
    assert np.abs(acc - ref).max() > 1e-6

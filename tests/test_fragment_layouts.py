"""CPU model of the warp-level fragment layouts the bf16 tensor-core decode
uses (csrc/pa_decode_mma.cuh), checked against plain matrix products.

The PTX lane layouts (as documented for ldmatrix .m8n8.x4 [.trans], movmatrix
.m8n8.trans and mma.m16n8k16 .row.col) are modelled in numpy; the kernel's
address arithmetic -- the 128-byte swizzle of the TMA tiles, the lane -> row /
16-byte chunk choice for the K (non-transposed) and V (transposed) loads, and
the P^T fragment built by transposing the score fragment -- is restated here.
The model must give S = K q^T and O^T = V^T P exactly.
"""
import numpy as np

D, T, H = 256, 16, 8


def sw_off(row, byte):
    """byte offset of (row, byte) in a tile of 16-row x 128-byte boxes with the
    128-byte swizzle (16-byte chunk index XOR row % 8)"""
    return (byte >> 7) * (16 * 128) + row * 128 + ((((byte >> 4) & 7) ^ (row & 7)) << 4) + (byte & 15)


def store(m):
    """a [16][D] 16-bit tile as the TMA writes it: element (t, d) at sw_off(t, 2d)"""
    return {sw_off(t, 2 * d): m[t, d] for t in range(T) for d in range(D)}


def ldsm_x4(sm, addr_of_lane, trans):
    """regs[lane][i] = the (low, high) 16-bit pair lane gets from matrix i"""
    regs = [[None] * 4 for _ in range(32)]
    for i in range(4):
        rows = [addr_of_lane(8 * i + k) for k in range(8)]
        mat = np.array([[sm[rows[k] + 2 * e] for e in range(8)] for k in range(8)])
        if trans:
            mat = mat.T
        for lane in range(32):
            g, c = lane // 4, lane % 4
            regs[lane][i] = (mat[g, 2 * c], mat[g, 2 * c + 1])
    return regs


def mma_16816(a, b, acc):
    """acc[lane] (4 floats) += A (16x16) B (16x8) from the lanes' fragments"""
    am = np.zeros((16, 16))
    bm = np.zeros((16, 8))
    for lane in range(32):
        g, c = lane // 4, lane % 4
        am[g, 2 * c], am[g, 2 * c + 1] = a[lane][0]
        am[g + 8, 2 * c], am[g + 8, 2 * c + 1] = a[lane][1]
        am[g, 2 * c + 8], am[g, 2 * c + 9] = a[lane][2]
        am[g + 8, 2 * c + 8], am[g + 8, 2 * c + 9] = a[lane][3]
        bm[2 * c, g], bm[2 * c + 1, g] = b[lane][0]
        bm[2 * c + 8, g], bm[2 * c + 9, g] = b[lane][1]
    dm = am @ bm
    for lane in range(32):
        g, c = lane // 4, lane % 4
        acc[lane] += np.array([dm[g, 2 * c], dm[g, 2 * c + 1], dm[g + 8, 2 * c], dm[g + 8, 2 * c + 1]])


def movmatrix_trans(vals):
    """vals[lane] = (low, high) of row lane // 4, columns 2 (lane % 4) .. + 1"""
    m = np.zeros((8, 8))
    for lane in range(32):
        m[lane // 4, 2 * (lane % 4)], m[lane // 4, 2 * (lane % 4) + 1] = vals[lane]
    m = m.T
    return [(m[lane // 4, 2 * (lane % 4)], m[lane // 4, 2 * (lane % 4) + 1]) for lane in range(32)]


def test_scores_from_ldmatrix_fragments():
    rng = np.random.default_rng(0)
    K = rng.standard_normal((T, D))
    q = rng.standard_normal((H, D))
    sm = store(K)
    acc = [np.zeros(4) for _ in range(32)]
    for t in range(D // 16):
        # lane l addresses token row (l & 7) + 8 ((l >> 3) & 1), 16-byte chunk l >> 4 of k-step t
        a = ldsm_x4(sm, lambda l: sw_off((l & 7) + ((l >> 3) & 1) * 8, 32 * t + 16 * (l >> 4)), False)
        # q fragment: d = 16 t + 2c (+1) and + 8, column = head l // 4
        b = [((q[l // 4, 16 * t + 2 * (l % 4)], q[l // 4, 16 * t + 2 * (l % 4) + 1]),
              (q[l // 4, 16 * t + 2 * (l % 4) + 8], q[l // 4, 16 * t + 2 * (l % 4) + 9]))
             for l in range(32)]
        mma_16816(a, b, acc)
    S = K @ q.T
    for lane in range(32):
        g, c = lane // 4, lane % 4
        assert np.allclose(acc[lane], [S[g, 2 * c], S[g, 2 * c + 1], S[g + 8, 2 * c], S[g + 8, 2 * c + 1]])


def test_pv_from_transposed_fragments():
    rng = np.random.default_rng(1)
    V = rng.standard_normal((T, D))
    P = rng.random((T, H))
    # the lane holds P[token g | g + 8][heads 2c, 2c + 1] (the score accumulator's layout)
    pr = [(P[l // 4, 2 * (l % 4)], P[l // 4, 2 * (l % 4) + 1], P[l // 4 + 8, 2 * (l % 4)],
           P[l // 4 + 8, 2 * (l % 4) + 1]) for l in range(32)]
    b0 = movmatrix_trans([(p[0], p[1]) for p in pr])
    b1 = movmatrix_trans([(p[2], p[3]) for p in pr])
    sm = store(V)
    O = V.T @ P
    for m in range(D // 16):
        # lane l addresses token row (l & 7) + 8 ((l >> 4) & 1), 16-byte chunk (l >> 3) & 1 of m-tile m
        a = ldsm_x4(sm, lambda l: sw_off((l & 7) + ((l >> 4) & 1) * 8, 32 * m + 16 * ((l >> 3) & 1)), True)
        o = [np.zeros(4) for _ in range(32)]
        mma_16816(a, [(b0[l], b1[l]) for l in range(32)], o)
        for lane in range(32):
            g, c = lane // 4, lane % 4
            d = 16 * m + g
            assert np.allclose(o[lane], [O[d, 2 * c], O[d, 2 * c + 1], O[d + 8, 2 * c], O[d + 8, 2 * c + 1]])


def test_swizzle_is_a_permutation_of_each_row_and_conflict_free():
    """Each token row's 32 chunks land on distinct 16-byte slots, and the 8 rows an
    ldmatrix phase reads for one chunk index fall on 8 distinct bank groups."""
    for row in range(T):
        offs = {sw_off(row, 16 * j) for j in range(2 * D // 16)}
        assert len(offs) == 2 * D // 16
    for j in range(8):
        banks = {(sw_off(r, 16 * j) % 128) // 16 for r in range(8)}
        assert len(banks) == 8

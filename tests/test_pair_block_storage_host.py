"""Upper pair-block storage of the bf16 symmetric matrices A and B, checked on
the host by restating the kernels' index rules (no GPU).

The SYRK products compute, per m_pad x m_pad matrix, the tiles that touch the
upper triangle: the 2-SM form pair tiles (q, tn >= q) whose two CTAs hold
rows 256 q + 128 rank, the 1-SM form tiles (tm, tn >= tm // 2) of 128 rows;
both over 256-wide column tiles. By default they store every chunk of those
tiles and nothing else; with the mirror they also write the transpose of
every tile right of its rows' diagonal pair block. The readers (A*A: both
operands, B*X: its A operand) take each 64-wide K-block left of the operand
rows' diagonal pair block from the transposed block, the rest as rows.

Checked for every tile-row count 1..40, both tilings of the writer and of the
reader: every element a reader loads was written, and with the mirror the
whole matrix is written. Also: in a 2-SM diagonal pair tile of A*A each CTA's
B rows are its own A rows (the loaded-once shortcut), and the K-block runs of
one layout cover [0, k_blocks) in order.
"""

import numpy as np
import pytest

BM, BN, BK = 128, 256, 64


def written(t, form, mirror):
    """Boolean m_pad x m_pad map (in units of 64 x 64 blocks) of what a SYRK
    launch with `form` ('pair' or 'single') writes."""
    m_pad = BM * t
    nb = m_pad // BK
    tiles_n = -(-m_pad // BN)
    w = np.zeros((nb, nb), dtype=bool)

    def tile(tm, tn):
        if tm >= t:                     # a pair's second row past the last tile row
            return
        r0, c0 = tm * BM // BK, tn * BN // BK
        c1 = min(c0 + BN // BK, nb)
        w[r0:r0 + BM // BK, c0:c1] = True
        if mirror and tn > tm // 2:     # right of the rows' diagonal pair block
            w[c0:c1, r0:r0 + BM // BK] = True

    if form == "pair":
        for q in range(-(-t // 2)):
            for tn in range(q, tiles_n):
                for rank in (0, 1):
                    tile(2 * q + rank, tn)
    else:
        for tm in range(t):
            for tn in range(tm // 2, tiles_n):
                tile(tm, tn)
    return w


def runs(kb_ta, kb_tb, kb_n, phase, diag=False):
    """The K-block runs of one operand layout the producer and issuer walk:
    (a_mn, b_mn, kb0, kb1) in order."""
    if phase == "bx":
        return [(True, True, 0, kb_ta), (False, True, kb_ta, kb_n)]
    if diag:
        return [(True, True, 0, kb_ta), (False, False, kb_ta, kb_n)]
    return [(True, True, 0, kb_ta), (False, True, kb_ta, kb_tb), (False, False, kb_tb, kb_n)]


def operand_blocks(rows0, nrows, kb, mn):
    """64 x 64 blocks one operand load touches: rows [rows0, +nrows) of the
    operand at K-block kb, read as rows (K-major) or from the transposed block
    (MN-major: rows kb, columns rows0..)."""
    r = range(rows0 // BK, (rows0 + nrows) // BK)
    return [(kb, i) for i in r] if mn else [(i, kb) for i in r]


def reads(t, form, phase, mirror):
    """Every 64 x 64 block of the symmetric operand(s) a launch reads."""
    m_pad = BM * t
    kb_n = m_pad // BK
    tiles_n = -(-m_pad // BN)
    out = []
    items = []
    if phase == "bx":
        # B*X tiles over the n columns; only the A operand (B) is symmetric
        if form == "pair":
            items = [(2 * q + rank, None) for q in range(-(-t // 2)) for rank in (0, 1)]
        else:
            items = [(tm, None) for tm in range(t)]
    else:
        if form == "pair":
            items = [(2 * q + rank, tn) for q in range(-(-t // 2)) for tn in range(q, tiles_n) for rank in (0, 1)]
        else:
            items = [(tm, tn) for tm in range(t) for tn in range(tm // 2, tiles_n)]
    for tm, tn in items:
        kb_ta = 0 if mirror else (tm // 2) * (2 * BM // BK)
        kb_tb = 0 if (mirror or tn is None) else tn * (BN // BK)
        diag = phase == "a2b" and form == "pair" and tn == tm // 2
        rank = tm % 2
        for a_mn, b_mn, kb0, kb1 in runs(kb_ta, kb_tb, kb_n, phase, diag):
            for kb in range(kb0, kb1):
                if tm < t or form == "pair":
                    # A operand rows (a spare pair half reads TMA's zero fill past m_pad)
                    if tm < t:
                        out += operand_blocks(tm * BM, BM, kb, a_mn)
                if phase == "a2b" and not diag:
                    if form == "pair":
                        n0, nrows = tn * BN + rank * (BN // 2), BN // 2
                    else:
                        n0, nrows = tn * BN, BN
                    n1 = min(n0 + nrows, m_pad)
                    if n1 > n0:
                        out += operand_blocks(n0, n1 - n0, kb, b_mn)
    return out


@pytest.mark.parametrize("t", list(range(1, 41)))
@pytest.mark.parametrize("mirror", [False, True])
def test_every_read_was_written(t, mirror):
    for wform in ("pair", "single"):
        if t < 2 and wform == "pair":
            continue                    # one tile row always runs on single CTAs
        w = written(t, wform, mirror)
        if mirror:
            assert w.all(), (t, wform)  # with the mirror the whole matrix exists
        for rform in ("pair", "single"):
            if t < 2 and rform == "pair":
                continue
            for phase in ("a2b", "bx"):
                for blk in reads(t, rform, phase, mirror):
                    assert w[blk], (t, wform, rform, phase, blk)


@pytest.mark.parametrize("t", list(range(1, 41)))
def test_upper_storage_writes_only_upper_pair_blocks(t):
    # without the mirror nothing below the diagonal pair blocks is written
    for form in ("pair", "single"):
        if t < 2 and form == "pair":
            continue
        w = written(t, form, False)
        nb = w.shape[0]
        for i in range(nb):
            for j in range(nb):
                upper = (j * BK) // BN >= (i * BK) // BN
                assert w[i, j] == upper, (t, form, i, j)


@pytest.mark.parametrize("q,tn", [(0, 0), (3, 3), (7, 7), (2, 5)])
def test_diagonal_pair_tile_b_rows_are_a_rows(q, tn):
    for rank in (0, 1):
        a_rows = (2 * q + rank) * BM
        b_rows = tn * BN + rank * (BN // 2)
        assert (a_rows == b_rows) == (tn == q)


@pytest.mark.parametrize("t", [2, 5, 11, 16, 32])
def test_layout_runs_cover_the_k_blocks_in_order(t):
    kb_n = BM * t // BK
    tiles_n = -(-BM * t // BN)
    for tm in range(t):
        for tn in range(tm // 2, tiles_n):
            for mirror in (False, True):
                kb_ta = 0 if mirror else (tm // 2) * 4
                kb_tb = 0 if mirror else tn * 4
                for phase, diag in (("a2b", False), ("a2b", tn == tm // 2), ("bx", False)):
                    seq = [kb for a, b, k0, k1 in runs(kb_ta, kb_tb, kb_n, phase, diag) for kb in range(k0, k1)]
                    assert seq == list(range(kb_n))
                    # the layout of each K-block matches the per-block rule
                    for a_mn, b_mn, k0, k1 in runs(kb_ta, kb_tb, kb_n, phase, diag):
                        for kb in range(k0, k1):
                            assert a_mn == (kb < kb_ta)
                            if phase == "bx":
                                assert b_mn
                            elif not diag:
                                assert b_mn == (kb < kb_tb)

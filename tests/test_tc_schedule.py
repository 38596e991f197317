"""Host-side checks of the tensor-core kernels' TMEM slot schedules and
operand layouts (no GPU).

Both backward kernels, at d = 128 on SM pairs, cycle four 32-column TMEM
slots by halves of a block (key-major) or chunk (query-major, in both its
two-pass and single-pass forms). The slot
functions below restate KmCfg::w_s_slot / w_dp_slot / w_first and
QmCfg::c_s_slot / c_dp_slot / c_first of csrc/tc_bwd.cu; the tests replay the
MMA issue order of each kernel (the tensor core runs MMAs in issue order)
with the softmax steps between the hand-backs, and check that every MMA and
every softmax reads the (block, half) data it expects, that no slot is
rewritten before its last reader, and that a softmax never touches a slot an
MMA in flight beside it uses. They also check the column maps the kernels'
descriptors assume: the Q sub-tile boxes of the key-major kernel and the K'
row permutation of the query-major kernel.
"""
import pytest


def s_slot(p, h):        # S (S^T) slot of half h of a block / chunk of parity p
    return 3 * h if p == 0 else 3 - h


def dp_slot(p, h):       # dP (dP^T) slot; the two are adjacent, half 0 below
    return 1 - p + h


def first(p):            # the half handed back first
    return p


class Tmem:
    def __init__(self):
        self.slot = [None] * 4

    def write(self, sl, what):
        self.slot[sl] = what

    def expect(self, sl, what):
        assert self.slot[sl] == what, (sl, self.slot[sl], what)


def run_key_major(n_blocks):
    """Key-major issue order: per block m, after the first half f's hand-back
    dV_f(m), dK_f(m), dP^T(m+1); after the second half l's: dK_l(m), S^T of
    the next block's first half, dV_l(m), S^T of its second half."""
    t = Tmem()

    def dp_pair(n):
        p = n & 1
        assert dp_slot(p, 1) == dp_slot(p, 0) + 1
        t.write(dp_slot(p, 0), ("dP", n, 0))
        t.write(dp_slot(p, 1), ("dP", n, 1))

    def s_half(n, h):
        t.write(s_slot(n & 1, h), ("S", n, h))

    def softmax(n, h):   # P^T over S^T, dS^T over dP^T
        p = n & 1
        t.expect(s_slot(p, h), ("S", n, h))
        t.expect(dp_slot(p, h), ("dP", n, h))
        t.write(s_slot(p, h), ("P", n, h))
        t.write(dp_slot(p, h), ("dS", n, h))

    def dv(m, h):
        t.expect(s_slot(m & 1, h), ("P", m, h))

    def dk(m, h):
        t.expect(dp_slot(m & 1, h), ("dS", m, h))

    dp_pair(0)
    s_half(0, first(0))
    s_half(0, first(0) ^ 1)
    for m in range(n_blocks):
        more = m + 1 < n_blocks
        hf = first(m & 1)
        hl = hf ^ 1
        softmax(m, hf)
        # burst F runs beside the second half's softmax: disjoint slots
        burst_f = {s_slot(m & 1, hf), dp_slot(m & 1, hf)}
        if more:
            burst_f |= {dp_slot((m + 1) & 1, 0), dp_slot((m + 1) & 1, 1)}
        assert not burst_f & {s_slot(m & 1, hl), dp_slot(m & 1, hl)}
        dv(m, hf)
        dk(m, hf)
        if more:
            dp_pair(m + 1)
        softmax(m, hl)
        dk(m, hl)
        if more:
            assert first((m + 1) & 1) == hl
            s_half(m + 1, hl)
            # the next block's first softmax runs beside dV_l(m) and its
            # second S^T half
            nxt = {s_slot((m + 1) & 1, hl), dp_slot((m + 1) & 1, hl)}
            assert not nxt & {s_slot(m & 1, hl), s_slot((m + 1) & 1, hf)}
        dv(m, hl)
        if more:
            s_half(m + 1, hf)


def run_query_major(n_chunks):
    """Query-major pass 2: after the first half's hand-back dQ_f(j) and
    dP(j+1); after the second's the next chunk's first S half, dQ_l(j), the
    next chunk's second S half. dS is written over S; the dP slot is free as
    soon as the softmax has read it."""
    t = Tmem()

    def dp_pair(j):
        p = j & 1
        t.write(dp_slot(p, 0), ("dP", j, 0))
        t.write(dp_slot(p, 1), ("dP", j, 1))

    def s_half(j, h):
        t.write(s_slot(j & 1, h), ("S", j, h))

    def softmax(j, h):
        p = j & 1
        t.expect(s_slot(p, h), ("S", j, h))
        t.expect(dp_slot(p, h), ("dP", j, h))
        t.write(s_slot(p, h), ("dS", j, h))
        t.write(dp_slot(p, h), None)          # consumed

    def dq(j, h):
        t.expect(s_slot(j & 1, h), ("dS", j, h))

    dp_pair(0)
    s_half(0, first(0))
    s_half(0, first(0) ^ 1)
    for j in range(n_chunks):
        more = j + 1 < n_chunks
        hf = first(j & 1)
        hl = hf ^ 1
        softmax(j, hf)
        # burst F (dQ_f reads S_f; dP(j+1) rewrites S_f, dP_f) runs beside
        # the second half's softmax
        assert not {s_slot(j & 1, hf), dp_slot(j & 1, hf)} & {s_slot(j & 1, hl), dp_slot(j & 1, hl)}
        if more:
            assert {dp_slot((j + 1) & 1, 0), dp_slot((j + 1) & 1, 1)} == {s_slot(j & 1, hf), dp_slot(j & 1, hf)}
        dq(j, hf)
        if more:
            dp_pair(j + 1)
        softmax(j, hl)
        if more:
            assert t.slot[s_slot((j + 1) & 1, hl)] is None   # the dP slot just read
            s_half(j + 1, hl)
            # the next chunk's first softmax runs beside dQ_l(j) and its second S half
            nxt = {s_slot((j + 1) & 1, hl), dp_slot((j + 1) & 1, hl)}
            assert not nxt & {s_slot(j & 1, hl), s_slot((j + 1) & 1, hf)}
        dq(j, hl)
        if more:
            s_half(j + 1, hf)


def run_query_major_single_pass(n_chunks):
    """Query-major single pass (QmCfg::SP): the softmax writes P over S and
    P dP over dP; after the first half's hand-back W_f(j) (reads the S slot),
    U_f(j) (reads the dP slot), dP(j+1); after the second's U_l(j), the next
    chunk's first S half, W_l(j), the next chunk's second S half."""
    t = Tmem()

    def dp_pair(j):
        p = j & 1
        t.write(dp_slot(p, 0), ("dP", j, 0))
        t.write(dp_slot(p, 1), ("dP", j, 1))

    def s_half(j, h):
        t.write(s_slot(j & 1, h), ("S", j, h))

    def softmax(j, h):
        p = j & 1
        t.expect(s_slot(p, h), ("S", j, h))
        t.expect(dp_slot(p, h), ("dP", j, h))
        t.write(s_slot(p, h), ("P", j, h))
        t.write(dp_slot(p, h), ("PdP", j, h))

    def w(j, h):
        t.expect(s_slot(j & 1, h), ("P", j, h))

    def u(j, h):
        t.expect(dp_slot(j & 1, h), ("PdP", j, h))

    dp_pair(0)
    s_half(0, first(0))
    s_half(0, first(0) ^ 1)
    for j in range(n_chunks):
        more = j + 1 < n_chunks
        hf = first(j & 1)
        hl = hf ^ 1
        softmax(j, hf)
        burst_f = {s_slot(j & 1, hf), dp_slot(j & 1, hf)}
        if more:
            assert {dp_slot((j + 1) & 1, 0), dp_slot((j + 1) & 1, 1)} == burst_f
        assert not burst_f & {s_slot(j & 1, hl), dp_slot(j & 1, hl)}
        w(j, hf)
        u(j, hf)
        if more:
            dp_pair(j + 1)
        softmax(j, hl)
        u(j, hl)
        if more:
            s_half(j + 1, hl)
            nxt = {s_slot((j + 1) & 1, hl), dp_slot((j + 1) & 1, hl)}
            assert not nxt & {s_slot(j & 1, hl), s_slot((j + 1) & 1, hf)}
        w(j, hl)
        if more:
            s_half(j + 1, hf)


@pytest.mark.parametrize("n", range(1, 9))
def test_query_major_single_pass_schedule(n):
    run_query_major_single_pass(n)


def sw128_offset(row, col, rows):
    return (col // 32) * rows * 128 + row * 128 + ((((col % 32) // 4) ^ (row % 8)) * 16) + (col % 4) * 4


def test_single_pass_do_tile_layout():
    """The compute warps store the slab's dO rows (128 rows x 128 floats) as
    four 16 KB panels of 128-byte rows with the 16-byte chunks of row r XORed
    by r % 8: every float lands once inside the 64 KB tile, and the K step ks
    descriptor offset (panel ks / 4, 32 bytes per step inside the row) finds
    column 8 ks of row 0."""
    offs = {sw128_offset(r, c, 128) for r in range(128) for c in range(128)}
    assert len(offs) == 128 * 128 and min(offs) == 0 and max(offs) == 65536 - 4
    assert all(o % 4 == 0 for o in offs)
    for ks in range(16):
        assert sw128_offset(0, 8 * ks, 128) == (ks // 4) * 16384 + (ks % 4) * 32
    # a quarter warp (8 consecutive rows) storing the same 16-byte chunk hits
    # eight distinct 16-byte bank groups
    for c in range(0, 32, 4):
        for r0 in range(0, 128, 8):
            assert len({sw128_offset(r, c, 128) % 128 for r in range(r0, r0 + 8)}) == 8


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
def test_dq_box_rows_match_tmem_rows(G):
    """The query-major epilogue writes TMEM lane r (query r // G of the slab,
    head r % G of the kv group) at sw128_offset(r, col, 128) and adds the
    tile to dQ as one TMA box over dQ's (32 floats, heads, queries, d/32
    panels) view, box (32, G, 128 / G, d/32). TMA lays a box out innermost
    coordinate first in 128-byte rows, swizzled by the row's index modulo 8,
    so element (x, head, query, panel) must be where lane r put it."""
    QR, d = 128 // G, 128
    for r in range(128):
        qi, h = r // G, r % G
        for col in range(0, d, 7):
            panel, x = col // 32, col % 32
            box_row = (panel * QR + qi) * G + h        # 128-byte row of the box
            expect = box_row * 128 + (((x // 4) ^ (box_row % 8)) * 16) + (x % 4) * 4
            assert sw128_offset(r, col, 128) == expect


@pytest.mark.parametrize("n", range(1, 9))
def test_key_major_slot_schedule(n):
    run_key_major(n)


@pytest.mark.parametrize("n", range(1, 9))
def test_query_major_slot_schedule(n):
    run_query_major(n)


def test_slot_functions_cover_the_stage():
    for p in (0, 1):
        used = {s_slot(p, 0), s_slot(p, 1), dp_slot(p, 0), dp_slot(p, 1)}
        assert used == {0, 1, 2, 3}


def test_half_column_maps():
    # S^T / S half h: an N = 32 pair MMA takes B rows [0, 16) from the even
    # CTA's sub-tile h and [16, 32) from the odd one's; sub-tile h of CTA r
    # holds block columns (keys) 32 h + 16 r + [0, 16)
    for h in (0, 1):
        cols = [32 * h + 16 * (c // 16) + c % 16 for c in range(32)]
        assert cols == list(range(32 * h, 32 * h + 32))
    # dV / dK (dQ) K step i of half h reads block columns 32 h + 8 i from
    # panel h of the transposed tile: desc_off(4h + i) = panel (4h+i)/4,
    # byte offset 32 ((4h+i) % 4)
    for h in (0, 1):
        for i in range(4):
            kk = 4 * h + i
            assert (kk // 4) * 32 + (kk % 4) * 8 == 32 * h + 8 * i


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32])
def test_key_major_q_sub_tile_boxes(G):
    """Boxes of (min(G,16) heads, 16/min(G,16) queries) starting at block
    column c0 = 32 h + 16 r land the 16 rows of sub-tile h in block-column
    order (rows query-major, head-minor)."""
    gb = min(G, 16)
    qb = 16 // gb
    QB = 64 // G
    for r in (0, 1):
        for h in (0, 1):
            c0 = 32 * h + 16 * r
            head0, q0 = c0 % G, c0 // G
            assert head0 + gb <= G
            rows = [(q0 + dq) * G + head0 + dh for dq in range(qb) for dh in range(gb)]
            assert rows == list(range(c0, c0 + 16))
            assert q0 + qb <= QB


def kp_source_row(i):
    """K' row i of a 64-row chunk -> the K row it copies (group_transpose)."""
    return 32 * ((i >> 4) & 1) + 16 * (i >> 5) + (i & 15)


def test_k_prime_permutation():
    src = [kp_source_row(i) for i in range(64)]
    assert sorted(src) == list(range(64))
    # CTA r loads K' rows 32 r + [0, 32): rows 16 a + i are keys 32 a + 16 r + i
    for r in (0, 1):
        unit = src[32 * r: 32 * r + 32]
        for a in (0, 1):
            assert unit[16 * a: 16 * a + 16] == list(range(32 * a + 16 * r, 32 * a + 16 * r + 16))
    # pass 1's N = 64 S (rows [0, 32) even, [32, 64) odd): warpgroup wg's
    # keys 32 wg + [0, 32) sit in S columns 16 wg + [0, 16) and 32 + 16 wg + [0, 16)
    s_cols = src
    for wg in (0, 1):
        keys = s_cols[16 * wg: 16 * wg + 16] + s_cols[32 + 16 * wg: 32 + 16 * wg + 16]
        assert keys == list(range(32 * wg, 32 * wg + 32))


@pytest.mark.parametrize("S", [1, 63, 64, 65, 100, 2048, 4097])
def test_transpose_grid_covers_k_prime(S):
    ld = (S + 31) // 32 * 32
    rows_p = (S + 63) // 64 * 64
    assert (ld + 63) // 64 * 64 >= rows_p

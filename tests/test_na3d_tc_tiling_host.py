"""A CPU model of the tensor-core neighbourhood-attention kernel's index
arithmetic (rope_rope3d_apply_gb300/csrc/rope3d_na3d.cu,
rope3d_na3d_tc_kernel), checked without a GPU.

For every CTA (a 2 x 8 x 8 query block) the model walks the kernel's chunks
of the key region with the kernel's own integer formulas (region bounds, rows
per chunk, the row width's multiply-high division) and asserts that:
  - the TMA boxes (the launch-wide width min(W, kw + 7) x rows per chunk)
    start at aligned channel coordinates and non-negative positions, land
    inside their tiles, and every key a mask selects is a grid token of the
    region (never a zero-filled box element);
  - the ranges every tcgen05 MMA reads through its shared-memory descriptors
    (Q, K, P: K-major with the 128-byte swizzle; V: MN-major, column blocks
    kTcN x 128 bytes apart) lie inside their tiles, the MMA shapes are valid
    (M = 128, N a multiple of 16 up to 256) and the tensor-memory columns of
    S and O do not overlap;
  - each query meets each key of its window exactly once through the
    per-thread window masks, and no other key.
It also checks the instruction and shared-memory descriptor encoders against
the field layout they implement. The attention's arithmetic is left to the
GPU tests, which compare the outputs with the float64 oracle."""
from __future__ import annotations

import random

import pytest

TC_M = 128                 # queries per CTA
QT, QH, QW = 2, 8, 8
Q_CB = TC_M * 128          # bytes per column block of Q or P


class Config:
    """The kernel's layout: chunks of up to 112 keys, two-slot rings of K, V
    and P tiles, two S buffers in tensor memory, one CTA per SM; 256 softmax
    threads, two per query row."""

    def __init__(self):
        self.TC_N = 112
        self.THREADS = 256          # softmax threads
        self.CTAS = 1
        self.PARTS = self.THREADS // TC_M
        self.KV_CB = self.TC_N * 128
        self.KV_SLOT = 2 * self.KV_CB
        self.OFF_Q, self.OFF_K = 0, 4 * Q_CB   # two Q buffers (block parity)
        self.OFF_V = self.OFF_K + 2 * self.KV_SLOT
        self.OFF_RED = self.OFF_V + 2 * self.KV_SLOT
        self.SBUFS = 3              # S buffers: b at column b * 128
        self.COL_S = 128
        self.COL_O = 384            # the O buffer
        self.OBUFS = 1
        self.TMEM_COLS = 512


CONFIGS = {"tc": Config()}


def na_start(i, L, k):
    s = max(i - k // 2, 0)
    return L - k if s + k > L else s


def fastdiv_make(d):
    """The kernel's device-side constants (ceil log2, multiplier)."""
    l = (d - 1).bit_length() if d > 1 else 0
    m = ((1 << 32) * ((1 << l) - d)) // d + 1
    return d, m & 0xFFFFFFFF, l


def fdiv(n, f):
    d, m, l = f
    return (((n * m) >> 32) + n) >> l


def sw128(row, c, cb_bytes):
    return (c >> 3) * cb_bytes + row * 128 + (((c & 7) ^ (row & 7)) << 4)


def sdesc(addr, lbo, sbo):
    return ((addr & 0x3FFFF) >> 4) | (((lbo & 0x3FFFF) >> 4) << 16) | \
        (((sbo & 0x3FFFF) >> 4) << 32) | (1 << 46) | (2 << 61)


def idesc(m, n, b_mn):
    return (1 << 4) | (1 << 7) | (1 << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((m >> 4) << 24)


def test_descriptor_encoders():
    # instruction descriptor: D fp32 (bits 4-5), A and B bf16 (7-9, 10-12),
    # B major (16), N >> 3 (17-22), M >> 4 (24-28); everything else zero
    for n in range(16, 257, 16):
        for b_mn in (0, 1):
            d = idesc(128, n, b_mn)
            assert (d >> 4) & 3 == 1 and (d >> 7) & 7 == 1 and (d >> 10) & 7 == 1
            assert (d >> 15) & 1 == 0 and (d >> 16) & 1 == b_mn
            assert (d >> 17) & 0x3F == n // 8 and (d >> 23) & 1 == 0
            assert (d >> 24) & 0x1F == 8 and d >> 29 == 0
            assert d & 0b1111 == 0 and (d >> 6) & 1 == 0 and (d >> 13) & 3 == 0
    # shared-memory descriptor: 14-bit fields of 16-byte units at 0, 16, 32,
    # 0b001 at 46-48, the 128-byte swizzle (2) at 61-63
    for addr in (0, 1024, 0x3FFF0, 139264 + 3 * 16384 + 96):
        for lbo, sbo in ((16, 1024), (80 * 128, 1024), (208 * 128, 1024)):
            d = sdesc(addr, lbo, sbo)
            assert d & 0x3FFF == addr >> 4 and (d >> 16) & 0x3FFF == lbo >> 4
            assert (d >> 32) & 0x3FFF == sbo >> 4 and (d >> 46) & 7 == 1
            assert (d >> 61) == 2 and (d >> 49) & 0xFFF == 0 and (d >> 14) & 3 == 0


def test_device_fastdiv_of_region_widths():
    for d in range(1, 208 + 1):
        f = fastdiv_make(d)
        for n in list(range(0, 300)) + list(range(4096 - 300, 4096)):
            assert fdiv(n, f) == n // d, (n, d)


def test_q_warps_write_every_q_tile_chunk_once():
    """The Q warps: thread rt (0 .. 127) writes 16-byte vector cv = rt % 16 of
    query rows rt / 16 + 8 i (i = 0 .. 15), the query (t, h, w) = (i / 8,
    i % 8, rt / 16) from the block's corner, which is the query the MMA row
    and the softmax thread of that row stand for (row = 64 t + 8 h + w); each
    of the tile's 2048 chunks is written once, inside the 32 KB Q tile, and
    a warp reads two tokens' 256 contiguous bytes."""
    seen = set()
    for rt in range(128):
        cv, qw = rt & 15, rt >> 4
        for i in range(16):
            r = qw + 8 * i
            t, h, w = i >> 3, i & 7, qw
            assert (r >> 6, (r >> 3) & 7, r & 7) == (t, h, w)
            a = sw128(r, cv, Q_CB)
            assert 0 <= a and a + 16 <= 2 * Q_CB and a % 16 == 0
            seen.add(a)
    assert len(seen) == 2048
    for warp in range(4):
        for i in range(16):
            toks = {}
            for lane in range(32):
                rt = 32 * warp + lane
                toks.setdefault(rt >> 4, set()).add(rt & 15)
            assert len(toks) == 2 and all(v == set(range(16)) for v in toks.values())


@pytest.mark.parametrize("cfg", sorted(CONFIGS))
def test_shared_memory_layout(cfg):
    c = CONFIGS[cfg]
    assert all(o % 1024 == 0 for o in (c.OFF_K, c.OFF_V, c.OFF_RED, c.KV_CB, c.KV_SLOT))
    # maxima [chunk parity][parts] and sums [block parity][parts] of 128
    # floats, window masks [3 sets][4 offsets][parts][128] of 8 bytes, two
    # block descriptors (16 bytes + 16 per query row), 36 mbarriers + the TMEM
    # address
    total = (c.OFF_RED + 4 * c.PARTS * TC_M * 4 + 3 * 4 * c.THREADS * 8 + 2 * (16 + TC_M * 16) + 36 * 8 +
             16 + 1024)
    assert c.CTAS * (total + 1024) <= 228 * 1024          # 1 KB reserved per CTA
    assert c.TC_N <= c.COL_S and (c.SBUFS - 1) * c.COL_S + c.TC_N <= c.COL_O
    assert c.SBUFS * c.COL_S <= c.COL_O and c.COL_O + 128 * c.OBUFS <= c.TMEM_COLS


def check_block(cfg, T, H, W, kt, kh, kw, bt, bh, bw, heads=3):
    TC_N, THREADS, PARTS = cfg.TC_N, cfg.THREADS, cfg.PARTS
    KV_CB, OFF_Q, OFF_K, OFF_V = cfg.KV_CB, cfg.OFF_Q, cfg.OFF_K, cfg.OFF_V
    COL_O, COL_S, KV_SLOT, SBUFS = cfg.COL_O, cfg.COL_S, cfg.KV_SLOT, cfg.SBUFS
    t0, h0, w0 = bt * QT, bh * QH, bw * QW
    rt0 = na_start(t0, T, kt)
    rt1 = na_start(min(t0 + 1, T - 1), T, kt) + kt
    rh0 = na_start(h0, H, kh)
    RH = na_start(min(h0 + QH - 1, H - 1), H, kh) + kh - rh0
    rw0 = na_start(w0, W, kw)
    RW = na_start(min(w0 + QW - 1, W - 1), W, kw) + kw - rw0
    # the launch-wide box: rwb columns (the widest region row), chb rows
    rwb = min(W, kw + QW - 1)
    chb = TC_N // rwb
    assert 1 <= RW <= rwb <= TC_N and 1 <= RH and chb >= 1 and chb * rwb <= TC_N
    assert rwb <= 256 and chb <= 256                 # TMA box dimensions
    per_frame = (RH + chb - 1) // chb
    n_chunks = (rt1 - rt0) * per_frame
    rwd = fastdiv_make(rwb)
    # Q tile rows and their offsets
    q_offsets = set()
    for r in range(TC_M):
        for cv in range(16):
            o = sw128(r, cv, Q_CB)
            assert 0 <= o < 2 * Q_CB
            q_offsets.add(o)
    assert len(q_offsets) == TC_M * 16
    seen = {}
    for c in range(n_chunks):
        f = rt0 + c // per_frame
        r0 = (c % per_frame) * chb
        nr = min(chb, RH - r0)
        N = (nr * rwb + 15) & ~15
        assert 16 <= N <= TC_N and N % 16 == 0
        # the TMA boxes: channel coordinate 0 or 64 (0 or 128 bytes), the other
        # coordinates never negative; box element (cc, rr) lands in tile row
        # rr * rwb + cc; coordinates past the grid read zeros
        assert rw0 >= 0 and rh0 + r0 >= 0 and 0 <= f < T
        rows = {}
        for rr in range(chb):
            for cc in range(rwb):
                j = rr * rwb + cc
                assert j < TC_N
                h, w = rh0 + r0 + rr, rw0 + cc
                rows[j] = (f, h, w) if (h < H and w < W) else None
        for j in range(chb * rwb):
            for cv in range(16):
                assert 0 <= sw128(j, cv, KV_CB) < 2 * KV_CB
        # the rows the set-up zeroes (past the box, up to the next multiple
        # of 16) are disjoint from the box's rows and inside each tile, and
        # every MMA row past the box is one of them
        box_rows = rwb * chb
        pad = ((box_rows + 15) & ~15) - box_rows
        zeroed = set(range(box_rows, box_rows + pad))
        assert all(r < TC_N for r in zeroed) and not zeroed & set(range(box_rows))
        assert set(range(box_rows, N)) <= zeroed
        slot = c & 1   # ring slot of the chunk's K and V tiles
        sb = c % SBUFS  # its S buffer
        ks_base, vs_base = OFF_K + slot * KV_SLOT, OFF_V + slot * KV_SLOT
        # S = Q K^T: eight k16 steps; A reads 128 rows of 32 bytes at koff in
        # column block ks / 4, B reads N rows likewise
        for ks in range(8):
            koff = (ks & 3) * 32
            a0 = OFF_Q + (ks >> 2) * Q_CB + koff
            b0 = ks_base + (ks >> 2) * KV_CB + koff
            assert OFF_Q <= a0 and a0 - koff + TC_M * 128 <= OFF_Q + 2 * Q_CB
            assert ks_base <= b0 and b0 - koff + N * 128 <= ks_base + KV_SLOT
        # O += P V: N / 16 k16 steps; A = P from tensor memory (the S buffer's
        # columns 8 s .. 8 s + 7: keys 16 s .. 16 s + 15 as bf16 pairs); V as an
        # MN-major operand: 16 keys (2 groups of 8 rows, SBO = 1024) x 128
        # channels (2 column blocks, LBO = KV_CB)
        for s in range(N // 16):
            pcol = sb * COL_S + 8 * s
            assert sb * COL_S <= pcol and pcol + 8 <= sb * COL_S + TC_N // 2
            va = vs_base + s * 2048
            assert vs_base <= va and va + 1024 + 1024 + KV_CB <= vs_base + KV_SLOT
        # S buffer `sb` holds columns [sb * COL_S, + N), clear of the others and of O
        assert sb * COL_S + N <= (sb + 1) * COL_S <= COL_O
        # the softmax: thread part qq of a row reads columns [qq * 56, + 56) of
        # its S buffer (columns past the chunk's keys masked) and writes the
        # weights of all 56 as 28 bf16 pairs from column qq * 28 (16 + 8 + 4
        # columns): the parts' P columns are disjoint, cover every column the
        # P V MMA reads, and overwrite only S columns [0, 56), which both parts
        # have read before either writes (the row's exchange lies between)
        npart = 56
        assert PARTS == 2 and PARTS * npart == TC_N
        written = []
        for qq in range(PARTS):
            cb0 = qq * npart
            assert cb0 + npart <= COL_S                # inside this S buffer
            col = cb0 // 2
            for width in (16, 8, 4):
                written += range(col, col + width)
                col += width
        assert sorted(written) == list(range(TC_N // 2)) and (N // 16) * 8 <= TC_N // 2
        # the window masks of every query row: a 64-bit mask per thread part,
        # built from the chunk rows its part spans, each in the window
        # contributing columns [clo, chi)
        for row in range(TC_M):
            qt, qh, qw = t0 + (row >> 6), h0 + ((row >> 3) & 7), w0 + (row & 7)
            row_ok = qt < T and qh < H and qw < W
            st_q = na_start(min(qt, T - 1), T, kt)
            ah = na_start(min(qh, H - 1), H, kh) - rh0
            aw = na_start(min(qw, W - 1), W, kw) - rw0
            clo, chi = max(aw, 0), min(aw + kw, RW)
            frame_ok = row_ok and 0 <= f - st_q < kt
            for qq in range(PARTS):
                cb0 = qq * npart
                win = 0
                if frame_ok:
                    rr = fdiv(cb0, rwd)
                    js = rr * rwb - cb0
                    while js < npart and rr < nr:
                        if 0 <= r0 + rr - ah < kh:
                            a, b2 = max(js + clo, 0), min(js + chi, npart)
                            if a < b2:
                                win |= ((1 << 64) - 1 >> (64 - (b2 - a))) << a
                        rr += 1
                        js += rwb
                assert win < (1 << npart)
                assert win >> max(nr * rwb - cb0, 0) == 0     # only the chunk's keys
                for k in range(npart):
                    if win >> k & 1:
                        key = rows[cb0 + k]
                        assert key is not None          # never a zero-filled key
                        meet = (qt, qh, qw) + key
                        seen[meet] = seen.get(meet, 0) + 1
    # every query of the block meets each key of its window once, and no other
    expected = 0
    for qt in range(t0, min(t0 + QT, T)):
        for qh in range(h0, min(h0 + QH, H)):
            for qw in range(w0, min(w0 + QW, W)):
                st, sh, sw_ = na_start(qt, T, kt), na_start(qh, H, kh), na_start(qw, W, kw)
                for tt in range(st, st + kt):
                    for a in range(sh, sh + kh):
                        for b in range(sw_, sw_ + kw):
                            assert seen.get((qt, qh, qw, tt, a, b)) == 1, (qt, qh, qw, tt, a, b)
                expected += kt * kh * kw
    assert sum(seen.values()) == expected
    return expected


def check_grid(cfg, T, H, W, kt, kh, kw, blocks=None):
    nbt, nbh, nbw = (T + QT - 1) // QT, (H + QH - 1) // QH, (W + QW - 1) // QW
    if blocks is None:
        blocks = [(bt, bh, bw) for bt in range(nbt) for bh in range(nbh) for bw in range(nbw)]
    assert sum(check_block(cfg, T, H, W, kt, kh, kw, *blk) for blk in blocks) > 0


def tc_eligible(W, kw, tc_n=112):
    """The host's choice: the tensor-core kernel when a region row fits a chunk."""
    return min(W, kw + QW - 1) <= tc_n


GEOMETRIES = [
    (3, 12, 12, 3, 5, 5), (2, 9, 17, 1, 3, 7), (5, 8, 8, 5, 7, 7), (4, 16, 24, 3, 7, 7),
    (3, 10, 13, 3, 5, 5), (2, 9, 10, 1, 1, 1), (3, 8, 8, 3, 3, 3), (1, 9, 10, 1, 3, 3),
    (2, 20, 70, 1, 3, 67), (3, 17, 9, 3, 17, 9), (2, 5, 90, 1, 1, 73),
    (2, 6, 80, 1, 3, 67), (2, 12, 40, 1, 9, 33), (2, 12, 30, 1, 5, 23), (4, 13, 11, 3, 5, 7),
    (3, 16, 16, 3, 7, 7), (2, 30, 80, 1, 1, 79), (2, 9, 100, 1, 3, 73),
]


@pytest.mark.parametrize("cfg", sorted(CONFIGS))
def test_eligibility_bounds_every_region_row(cfg):
    """min(W, kw + 7) <= kTcN makes every block's region row fit a chunk."""
    TC_N = CONFIGS[cfg].TC_N
    for W in range(1, 240):
        for kw in range(1, W + 1, 2):
            if not tc_eligible(W, kw, TC_N):
                continue
            for w0 in range(0, W, QW):
                rw0 = na_start(w0, W, kw)
                RW = na_start(min(w0 + QW - 1, W - 1), W, kw) + kw - rw0
                assert 1 <= RW <= TC_N


@pytest.mark.parametrize("cfg", sorted(CONFIGS))
@pytest.mark.parametrize("geom", GEOMETRIES, ids=[str(g) for g in GEOMETRIES])
def test_tc_tiling_covers_every_window_once(geom, cfg):
    assert tc_eligible(geom[2], geom[5], CONFIGS[cfg].TC_N)
    check_grid(CONFIGS[cfg], *geom)


@pytest.mark.parametrize("cfg", sorted(CONFIGS))
def test_tc_tiling_of_the_benchmark_geometry(cfg):
    """16 x 64 x 64 tokens, window 3 x 7 x 7: corner, edge and inner blocks of
    the first, a middle and the last frame pair."""
    picks = [0, 1, 4, 7]
    check_grid(CONFIGS[cfg], 16, 64, 64, 3, 7, 7,
               blocks=[(bt, bh, bw) for bt in (0, 4, 7) for bh in picks for bw in picks])


def block_mma_widths(cfg, T, H, W, kt, kh, kw, bt, bh, bw):
    """The MMA widths (keys rounded up to 16) of one query block's chunks, by
    the same region and chunk arithmetic as check_block."""
    t0, h0 = bt * QT, bh * QH
    rt0 = na_start(t0, T, kt)
    rt1 = na_start(min(t0 + 1, T - 1), T, kt) + kt
    rh0 = na_start(h0, H, kh)
    RH = na_start(min(h0 + QH - 1, H - 1), H, kh) + kh - rh0
    rwb = min(W, kw + QW - 1)
    chb = cfg.TC_N // rwb
    per_frame = (RH + chb - 1) // chb
    return [(min(chb, RH - (c % per_frame) * chb) * rwb + 15) & ~15 for c in range((rt1 - rt0) * per_frame)]


@pytest.mark.parametrize("geom", [(16, 64, 64, 3, 7, 7), (5, 13, 27, 3, 5, 7), (3, 9, 40, 1, 3, 33)])
def test_bench_mma_flops_match_the_tiling(geom):
    """bench.py's count of the tensor-core attention's issued MMA work is the
    sum over every query block's chunks of 4 * 128 * 128 * N."""
    import bench

    T, H, W, kt, kh, kw = geom
    cfg = CONFIGS["tc"]
    nbt, nbh, nbw = (T + QT - 1) // QT, (H + QH - 1) // QH, (W + QW - 1) // QW
    want = sum(4 * 128 * 128 * n
               for bt in range(nbt) for bh in range(nbh) for bw in range(nbw)
               for n in block_mma_widths(cfg, T, H, W, kt, kh, kw, bt, bh, bw))
    assert bench.na3d_tc_mma_flops(1, T, H, W, 1, (kt, kh, kw)) == want
    assert bench.na3d_tc_mma_flops(2, T, H, W, 3, (kt, kh, kw)) == 6 * want

"""A CPU model of the neighbourhood-attention kernel's index arithmetic
(rope_rope3d_apply_gb300/csrc/rope3d_na3d.cu, rope3d_na3d_kernel), checked
against the window definition without a GPU.

For every CTA (a 1 x 8 x 8 query block) the model walks the kernel's chunks
of the key region exactly as the kernel computes them (region bounds, rows
per chunk, the strided row order ri, ri + S, ..., column groups), emulates
every thread's copy addresses and key slots, and then every warp's run of
16-key steps and its per-element mask. It asserts that:
  - every global offset a thread copies from is the token the slot stands
    for, and inside the grid;
  - the slots a chunk fills are exactly 0 .. rows x 16 segments - 1 (slots
    past a row's last column hold zeros), and a warp's run lies inside them;
  - a warp needs at most 4 steps per chunk (the compiled step counts);
  - each query of the block meets each key of its window exactly once, and
    no other key.
The model mirrors the kernel's integer formulas; a change to the kernel's
tiling has to change this model too. It carries no arithmetic of the
attention itself (the GPU tests compare the kernel's outputs with the
float64 oracle)."""
from __future__ import annotations

import pytest

KKC = 64      # key slots per chunk
QBH = QBW = 8  # query block


def na_start(i, L, k):
    s = max(i - k // 2, 0)
    return L - k if s + k > L else s


def check_block(T, H, W, kt, kh, kw, qt, bh, bw, heads=3):
    """Emulate CTA (qt, bh, bw) of one (batch, head); returns the number of
    (query, key) meetings."""
    tok = heads * 128                 # elements per token
    grid_row, frame = W * tok, H * W * tok
    h0, w0 = bh * QBH, bw * QBW
    rt0 = na_start(qt, T, kt)
    hl, wl = min(h0 + QBH, H) - 1, min(w0 + QBW, W) - 1
    rh0, rh1 = na_start(h0, H, kh), na_start(hl, H, kh) + kh
    rw0, rw1 = na_start(w0, W, kw), na_start(wl, W, kw) + kw
    RH, RW = rh1 - rh0, rw1 - rw0
    CW = min(RW, KKC)
    CH = min(RH, KKC // (16 * ((CW + 15) // 16)))
    assert CH >= 1
    S, ncc = (RH + CH - 1) // CH, (RW + CW - 1) // CW
    qR, mR = divmod(RH, S)
    seen = {}
    for c in range(kt * S * ncc):
        # chunk c: column group fastest, then ri, then the frame
        ci, rest = c % ncc, c // ncc
        ri, dt = rest % S, rest // S
        t, rb = rt0 + dt, rh0 + ri
        nr = qR + (1 if ri < mR else 0)
        c0 = rw0 + ci * CW
        cw = min(CW, rw1 - c0)
        nseg = (cw + 15) // 16
        sw = 16 * nseg
        assert nr * sw <= KKC
        # the copies: thread (cv, slot0) fills slots slot0 + 8 m
        slots = {}
        wrap = S * grid_row - sw * tok
        for slot0 in range(8):
            i, j = 0, slot0
            off = t * frame + rb * grid_row + (c0 + slot0) * tok
            for m in range(KKC * 16 // 128):
                slot = slot0 + 8 * m
                if i < nr:
                    assert slot == i * sw + j
                    if j < cw:
                        h, w = rb + i * S, c0 + j
                        assert 0 <= h < H and rw0 <= w < rw1 <= W
                        assert off == ((t * H + h) * W + w) * tok
                        slots[slot] = (t, h, w)
                    else:
                        slots[slot] = None          # zero-filled
                j += 8
                off += 8 * tok
                if j >= sw:
                    j -= sw
                    i += 1
                    off += wrap
        assert sorted(slots) == list(range(nr * sw))
        # the warps: rows 2 warp and 2 warp + 1 of the block
        for warp in range(4):
            hq = h0 + 2 * warp
            wh0 = na_start(min(hq, H - 1), H, kh)
            wh1 = na_start(min(hq + 1, H - 1), H, kh)
            bl = wh0 - rh0
            bu = (wh1 + kh if hq < H else wh0) - rh0
            qb, mb = divmod(bl, S)
            qu, mu = divmod(bu, S)
            ilo = qb + (1 if ri < mb else 0)
            ihi = qu + (1 if ri < mu else 0)
            nq = (ihi - ilo) * nseg
            if nq <= 0:
                continue
            assert nq <= 4
            j0 = ilo * 16 * nseg
            assert j0 + 16 * nq <= nr * sw
            for g in range(8):                       # MMA rows g and g + 8
                wq = w0 + g
                ww = na_start(min(wq, W - 1), W, kw)
                valid = [hq < H and wq < W, hq + 1 < H and wq < W]
                hk, seg = rb + ilo * S, 0
                for q in range(nq):
                    for jj in range(seg * 16, seg * 16 + 16):
                        key = slots[j0 + q * 16 + (jj - seg * 16)]
                        col = jj < cw and 0 <= c0 + jj - ww < kw
                        if jj < cw:
                            assert key == (t, hk, c0 + jj)
                        else:
                            assert key is None
                        for r, whr in ((0, wh0), (1, wh1)):
                            if col and valid[r] and 0 <= hk - whr < kh:
                                meet = (hq + r, wq) + key
                                seen[meet] = seen.get(meet, 0) + 1
                    seg += 1
                    if seg == nseg:
                        seg, hk = 0, hk + S
    # every query of the block meets each key of its window once, and no other
    for hh in range(h0, min(h0 + QBH, H)):
        for wq in range(w0, min(w0 + QBW, W)):
            st, sh, sw_ = na_start(qt, T, kt), na_start(hh, H, kh), na_start(wq, W, kw)
            for tt in range(st, st + kt):
                for a in range(sh, sh + kh):
                    for b in range(sw_, sw_ + kw):
                        assert seen.get((hh, wq, tt, a, b)) == 1, (hh, wq, tt, a, b)
    assert sum(seen.values()) == sum(
        kt * kh * kw for hh in range(h0, min(h0 + QBH, H)) for wq in range(w0, min(w0 + QBW, W)))
    return sum(seen.values())


def check_grid(T, H, W, kt, kh, kw, blocks=None):
    nbh, nbw = (H + QBH - 1) // QBH, (W + QBW - 1) // QBW
    if blocks is None:
        blocks = [(qt, bh, bw) for qt in range(T) for bh in range(nbh) for bw in range(nbw)]
    total = sum(check_block(T, H, W, kt, kh, kw, *blk) for blk in blocks)
    assert total > 0


GEOMETRIES = [
    (3, 12, 12, 3, 5, 5), (2, 9, 17, 1, 3, 7), (5, 8, 8, 5, 7, 7), (4, 16, 24, 3, 7, 7),
    (3, 10, 13, 3, 5, 5), (2, 9, 10, 1, 1, 1), (3, 8, 8, 3, 3, 3),
    (2, 20, 70, 1, 3, 67),    # region rows of 74 keys: cut into column groups
    (2, 5, 90, 1, 1, 81),
    (3, 17, 9, 3, 17, 9),     # windows covering the grid
    (2, 6, 80, 1, 3, 67), (2, 12, 40, 1, 9, 33), (2, 12, 30, 1, 5, 23),
]


@pytest.mark.parametrize("geom", GEOMETRIES, ids=[str(g) for g in GEOMETRIES])
def test_tiling_covers_every_window_once(geom):
    check_grid(*geom)


def test_tiling_of_the_benchmark_geometry():
    """16 x 64 x 64 tokens, window 3 x 7 x 7: the corner, edge and interior
    query blocks of the first, second, a middle and the last frame."""
    picks = [0, 1, 4, 7]
    check_grid(16, 64, 64, 3, 7, 7,
               blocks=[(qt, bh, bw) for qt in (0, 1, 8, 15) for bh in picks for bw in picks])

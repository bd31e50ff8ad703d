"""A CPU model of the cast kernels' index arithmetic: bounds, alignment, coverage.

compute-sanitizer is not available on the test machines, so the kernels'
memory accesses are checked here instead: this file restates, for every thread
of every CTA of one launch, the global addresses quantize_kernel (flat and
grouped, with and without dbias, plain and GEMM-ready scales),
quantize_dact_kernel and the dbias reduces compute, with
the same expressions as csrc/quantize.cuh, csrc/dact.cuh, csrc/dbias_reduce.cuh
and csrc/api.cu (persistent tile loop, per-group tile prefix, phase-1 and
phase-2 lane maps, 16- and 8-byte stores, scale and partial-sum rows).  Each
write increments a counter over the output it lands in, after a bounds and
alignment check.  Every output byte must be written exactly once, every
partial-sum entry a reduce reads must have been written, and every TMA box
origin must be in the tensor with a 16-byte aligned inner coordinate.

The model holds no arithmetic of the method (no values are computed); it is
not the oracle.  It is kept in step with the kernels by hand: a change to a
kernel's indexing must be mirrored here.
"""
import numpy as np
import pytest

BM, BN, BOX, THREADS = 128, 128, 64, 256
DBN = 64                     # backward-fusion tile columns
LANES = np.arange(32)


class Plane:
    """Write counters for one output buffer of `size` elements of `width` bytes."""

    def __init__(self, name, size, width=1):
        self.name, self.size, self.width = name, size, width
        self.parts = []
        self._count = None

    def write(self, idx, nbytes=1, align=1):
        idx = np.asarray(idx, np.int64).ravel()
        if idx.size == 0:
            return
        assert idx.min() >= 0 and idx.max() + nbytes <= self.size, (self.name, int(idx.min()), int(idx.max()))
        assert np.all((idx * self.width) % align == 0), (self.name, "misaligned")
        self.parts.append((idx[:, None] + np.arange(nbytes)).ravel())
        self._count = None

    @property
    def count(self):
        if self._count is None:
            allidx = np.concatenate(self.parts) if self.parts else np.zeros(0, np.int64)
            self._count = np.bincount(allidx, minlength=self.size)
        return self._count

    def once(self, mask=None):
        c = self.count if mask is None else self.count[mask]
        assert np.all(c == 1), (self.name, int((c != 1).sum()), np.unique(c))


def swizzled_offset(r, c, C):
    col_tiles = (C + 3) >> 2
    return (((r >> 7) * col_tiles + (c >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3)


def swizzled_bytes(R, C):
    return ((R + 127) // 128 * 128) * ((C + 3) // 4 * 4)


def tile_list(M, N, offsets):
    """The kernel's tiles in order: (row0, row_end, col0, rt, sb, g) per tile index; sb is the
    columnwise scale row of the tile's first 32-row block, g the tile's group (0 when flat)."""
    col_tiles = -(-N // BN)
    if offsets is None:
        row_tiles = -(-M // BM)
        return [(rt * BM, min(rt * BM + BM, M), ct * BN, rt, rt * (BM // 32), 0)
                for rt in range(row_tiles) for ct in range(col_tiles)]
    G = len(offsets) - 1
    gpre, gsb = [0], [0]
    for g in range(G):
        gpre.append(gpre[-1] + -(-(offsets[g + 1] - offsets[g]) // BM) * col_tiles)
        gsb.append(gsb[-1] + -(-(offsets[g + 1] - offsets[g]) // 32))
    tiles = []
    for t in range(gpre[G]):
        lo, hi = 0, G                       # binary search: gpre[lo] <= t < gpre[hi]
        while hi - lo > 1:
            mid = (lo + hi) >> 1
            if gpre[mid] <= t:
                lo = mid
            else:
                hi = mid
        local = t - gpre[lo]
        rtl, ct = local // col_tiles, local % col_tiles
        row0 = offsets[lo] + rtl * BM
        tiles.append((row0, min(row0 + BM, offsets[lo + 1]), ct * BN, gpre[lo] // col_tiles + rtl,
                      gsb[lo] + rtl * (BM // 32), lo))
    return tiles


def scale_col_rows(M, offsets):
    if offsets is None:
        return -(-M // 32)
    return sum(-(-(offsets[g + 1] - offsets[g]) // 32) for g in range(len(offsets) - 1))


def model_quantize(M, N, grid, offsets=None, dbias=False, swz=False, do_row=True, do_col=True, reuse=False):
    rows16 = N % 16 == 0
    Cr = -(-N // 32)
    out_row = Plane("out_row", M * N)
    out_col = Plane("out_col", M * N)
    if swz and offsets is not None:     # one GEMM-ready plane per group, in group order
        tiles_g = sum(-(-(offsets[g + 1] - offsets[g]) // BM) for g in range(len(offsets) - 1))
        scale_row = Plane("scale_row", tiles_g * 128 * ((Cr + 3) // 4 * 4))
        scale_col = Plane("scale_col", tiles_g * 4 * ((N + 127) // 128 * 128))
    elif swz:
        scale_row = Plane("scale_row", swizzled_bytes(M, Cr))
        scale_col = Plane("scale_col", swizzled_bytes(N, -(-M // 32)))
    else:
        scale_row = Plane("scale_row", M * Cr)
        scale_col = Plane("scale_col", scale_col_rows(M, offsets) * N)
    tiles = tile_list(M, N, offsets)
    ws_rows = max([t[3] for t in tiles], default=-1) + 1
    ws = Plane("ws", ws_rows * N, 4)

    # GEMM-ready planes: the kernel addresses one 512-byte plane tile per cast tile (swz_row_tile /
    # swz_col_tile) plus the entry's byte within it; each is checked against the layout's
    # definition on the whole plane (swizzled_offset, after the planes of the groups before)
    def in_tile(r, c):
        return ((r & 31) << 4) | (((r >> 5) & 3) << 2) | c

    def swz_row(tile, r, sc):
        row0, _, col0, rt, _, g = tile
        got = (rt * -(-N // BN) + (col0 >> 7)) * 512 + in_tile(r - row0, sc - (col0 >> 5))
        first = 0 if offsets is None else offsets[g]
        before = rt - (row0 - first) // BM
        want = before * 128 * ((Cr + 3) // 4 * 4) + swizzled_offset(r - first, sc, Cr)
        assert np.array_equal(got, want)
        return got

    def swz_col(tile, gcol, grow):
        row0, _, col0, rt, _, g = tile
        ct, rb = col0 >> 7, (grow - row0) >> 5
        if offsets is None:
            got = (ct * -(-M // BM) + rt) * 512 + in_tile(gcol - col0, rb)
            want = swizzled_offset(gcol, grow >> 5, -(-M // 32))
        else:
            first = offsets[g]
            rtl, tiles_g = (row0 - first) >> 7, -(-(offsets[g + 1] - first) // BM)
            got = ((rt - rtl) * -(-N // BN) + ct * tiles_g + rtl) * 512 + in_tile(gcol - col0, rb)
            want = ((rt - rtl) * 4 * ((N + 127) // 128 * 128) +
                    swizzled_offset(gcol, (grow - first) >> 5, -(-(offsets[g + 1] - first) // 32)))
        assert np.array_equal(got, want)
        return got

    # phase-1 lane map: warp -> (32-row block, box); lane -> (4-column group, 16-row half)
    w1, l1 = np.repeat(np.arange(8), 32), np.tile(LANES, 8)
    rb1, box1, cq1, half1 = w1 >> 1, w1 & 1, l1 & 15, l1 >> 4
    assert np.all(box1 * 16384 + (rb1 * 32 + half1 * 16 + 15) * 128 + 127 < 32768)      # stage bounds
    # phase-2 lane map: warp, task k -> (8-row group, box); lane -> (row in group, 16-column segment)
    w2 = np.repeat(np.arange(8), 4 * 32)
    k2 = np.tile(np.repeat(np.arange(4), 32), 8)
    l2 = np.tile(LANES, 32)
    task = w2 + 8 * k2
    if reuse:   # transcendental activations: warp = (32-row block, box), tasks = its 8-row groups
        rg2, box2 = (w2 >> 1) * 4 + k2, w2 & 1
    else:
        rg2, box2 = task >> 1, task & 1
    rr2, sp2 = l2 >> 2, l2 & 3
    for b in range(grid):
        for t in range(b, len(tiles), grid):
            row0, row_end, col0, rt, sb, g = tiles[t]
            for box in range(2):            # TMA box origins (x must be 16-byte aligned)
                x = col0 + box * BOX
                if x < N:
                    assert (x * 2) % 16 == 0 and 0 <= row0 < M
            # phase 1 of a grouped tile: the warp of (32-row block rb, box) zeroes the block's rows
            # past the group's end in its own box (16-byte chunks c = live*8 + lane, step 32) before
            # its column pass, so the next group's rows (loaded with the tile) count as zeros; the
            # chunks stay inside the warp's own 4 KiB of the stage, and the nonzero rows left are
            # exactly the group's rows of the block
            if offsets is not None:
                for rb in range(4):
                    first = row0 + rb * 32
                    if first >= row_end:
                        continue
                    live = min(32, row_end - first)
                    for box in range(2):
                        chunks = [live * 8 + lane + 32 * j for lane in range(32) for j in range(8)
                                  if live * 8 + lane + 32 * j < 256]
                        byte = box * 16384 + rb * 32 * 128 + np.array(chunks, int) * 16
                        assert np.all((byte >= box * 16384 + rb * 4096) & (byte + 16 <= box * 16384 + rb * 4096 + 4096))
                        zeroed_rows = sorted({first + c // 8 for c in chunks})
                        assert zeroed_rows == list(range(first + live, first + 32))
                        assert len(chunks) == len(set(chunks)) == (32 - live) * 8
            tile = tiles[t]
            grow, gcol = row0 + rb1 * 32, col0 + box1 * BOX + cq1 * 4
            sel = (grow < row_end) & (half1 == 0) & (gcol < N) & do_col
            if swz:
                # one offset per lane, the next three plane rows 16 bytes on (gcol % 4 == 0)
                o = swz_col(tile, gcol[sel], grow[sel])
                for j in range(4):
                    assert np.array_equal(o + 16 * j, swz_col(tile, gcol[sel] + j, grow[sel]))
                    scale_col.write(o + 16 * j)
                # the tile's own plane tiles' padding: warp (rb, box) zeroes the entries of its
                # 32 rows x 2 row blocks past the tile's end or N (all lanes, one row each), and
                # of its 64 columns x 1 column block (lanes < 16, four plane rows each)
                if do_row:
                    r = row0 + rb1 * 32 + l1
                    for j in range(2):
                        bc = col0 + box1 * BOX + j * 32
                        pad = (r >= row_end) | (reuse & (bc >= N))
                        scale_row.write(swz_row(tile, r[pad], bc[pad] >> 5))
                if do_col:
                    pad = (l1 < 16) & ((grow >= row_end) | (gcol >= N))
                    o = swz_col(tile, gcol[pad], grow[pad])
                    for j in range(4):
                        scale_col.write(o + 16 * j)
            else:
                scale_col.write((sb + rb1[sel]) * N + gcol[sel], 4, align=4)
            if dbias:
                gc = col0 + np.arange(BN)
                ws.write(rt * N + gc[gc < N], 1, align=4)
            grow = row0 + rg2 * 8 + rr2
            gcol = col0 + box2 * BOX + sp2 * 16
            ok = (row0 + rg2 * 8 < row_end) & (grow < row_end) & (gcol < N)
            half_seg = gcol + 16 > N
            assert not (rows16 and np.any(ok & half_seg))
            full, part = ok & ~half_seg, ok & half_seg
            for plane, on in ((out_row, do_row), (out_col, do_col)):
                if on:
                    plane.write(grow[full] * N + gcol[full], 16, align=16 if rows16 else 8)
                    plane.write(grow[part] * N + gcol[part], 8, align=8)
            se = ok & (sp2 % 2 == 0)
            if do_row and reuse:    # one byte per (row, block): lanes sp = 0, 2
                scale_row.write(swz_row(tile, grow[se], gcol[se] >> 5) if swz else grow[se] * Cr + (gcol[se] >> 5))
            elif do_row:
                # phase 2 puts row r's block b scale at byte 4r + b of the shared rowsc; after the
                # tile's barrier thread tid < 128 stores row tid's four bytes (blocks past N: not
                # stored, or zero padding of the GEMM-ready plane), one 32-bit store where aligned
                staged = (grow[se] - row0) * 4 + box2[se] * 2 + (sp2[se] >> 1)
                assert len(set(staged.tolist())) == staged.size and staged.max(initial=0) < 4 * BM
                nb = min(4, -(-(N - col0) // 32))
                live = np.arange(row0, row_end)
                want = {4 * (r - row0) + b for r in live for b in range(nb)}
                assert want == set(staged.tolist())         # every stored byte was formed by this tile
                if swz:
                    scale_row.write(swz_row(tile, live, np.full(live.size, col0 >> 5)), 4, align=4)
                elif nb == 4 and Cr % 4 == 0:
                    scale_row.write(live * Cr + (col0 >> 5), 4, align=4)
                else:
                    scale_row.write(live * Cr + (col0 >> 5), nb)
    return dict(out_row=out_row, out_col=out_col, scale_row=scale_row, scale_col=scale_col, ws=ws,
                ws_rows=ws_rows, tiles=tiles)


def check_quantize(M, N, grid, offsets=None, dbias=False, swz=False, do_row=True, do_col=True, reuse=False):
    m = model_quantize(M, N, grid, offsets, dbias, swz, do_row, do_col, reuse)
    for name, on in (("out_row", do_row), ("out_col", do_col)):
        if on:
            m[name].once()
        else:
            assert not m[name].count.any()
    # every scale byte once; a GEMM-ready plane's padding entries included (written by the tiles)
    for name, on in (("scale_row", do_row), ("scale_col", do_col)):
        if on:
            m[name].once()
        else:
            assert not m[name].count.any()
    if dbias:
        # the reduce reads ws[t * N + j] for every tile row t < ws_rows and column j < N
        m["ws"].once()
    return m


FLAT = [(1, 8), (33, 8), (45, 80), (96, 40), (128, 256), (257, 1032), (130, 144), (1000, 2056), (31, 4096),
        (544, 1056), (384, 224)]


@pytest.mark.parametrize("shape", FLAT)
@pytest.mark.parametrize("grid", [1, 7, 304])
def test_flat_cast_writes_every_byte_once(shape, grid):
    M, N = shape
    check_quantize(M, N, grid, dbias=True)


@pytest.mark.parametrize("shape", FLAT)
def test_activated_cast_task_map_writes_every_byte_once(shape):
    """The transcendental activations' phase-2 task map (a warp's tasks in one 32-row block)."""
    check_quantize(*shape, grid=7, reuse=True)
    check_quantize(*shape, grid=7, swz=True, reuse=True)


@pytest.mark.parametrize("shape", [(45, 80), (96, 40), (257, 1032), (130, 144)])
@pytest.mark.parametrize("dirs", [(True, False), (False, True)])
def test_flat_cast_swizzled_single_direction(shape, dirs):
    check_quantize(*shape, grid=5, swz=True, do_row=dirs[0], do_col=dirs[1])
    check_quantize(*shape, grid=5, swz=True)


@pytest.mark.parametrize("N", [24, 40, 96, 160, 1032])
@pytest.mark.parametrize("grid", [3, 304])
def test_grouped_cast_writes_every_byte_once(N, grid):
    sizes = [64, 0, 32, 416, 0, 0, 128, 96, 160, 32]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    m = check_quantize(off[-1], N, grid, offsets=off, dbias=True)
    # no tile straddles two groups; each group's tiles are contiguous in the partial-sum rows
    for row0, row_end, col0, rt, sb, g_tile in m["tiles"]:
        g = max(i for i in range(len(off) - 1) if off[i] <= row0)
        assert row_end <= off[g + 1]


@pytest.mark.parametrize("sizes", [[45, 0, 1, 31, 33, 96, 70, 127, 129, 0, 13], [64, 0, 32, 416, 96]])
def test_grouped_activated_cast_task_map_writes_every_byte_once(sizes):
    """The grouped cast with a transcendental activation: warp-local task map; grouped tiles, or
    with every offset a multiple of 32 the flat tiles (the same bytes)."""
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    sched = None if all(o % 32 == 0 for o in off) else off
    for N in (40, 160):
        check_quantize(off[-1], N, 7, offsets=sched, reuse=True)


def test_grouped_many_groups_and_empty_ones():
    rng = np.random.Generator(np.random.PCG64(5))
    sizes = (32 * rng.choice([0, 1, 3, 4, 5, 17], size=200)).tolist()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    check_quantize(off[-1], 48, 304, offsets=off, dbias=True)


@pytest.mark.parametrize("sizes", [[45, 0, 1, 31, 33, 96, 70, 127, 129, 0, 13], [1] * 40 + [300], [17, 15],
                                   [0, 200, 0]])
@pytest.mark.parametrize("N", [40, 160])
def test_grouped_unaligned_offsets_write_every_byte_once(sizes, N):
    """Groups that are not multiples of 32 rows: each group's columnwise scale rows follow the
    previous group's (sum of ceil(rows/32)), every output byte is written once, and no tile or
    block takes rows of two groups."""
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    m = check_quantize(off[-1], N, 7, offsets=off, dbias=True)
    assert m["scale_col"].count.size == scale_col_rows(off[-1], off) * N
    for row0, row_end, col0, rt, sb, g_tile in m["tiles"]:
        g = max(i for i in range(len(off) - 1) if off[i] <= row0 and off[i + 1] > off[i])
        assert off[g] <= row0 < row_end <= off[g + 1]
        assert sb == sum(-(-(off[h + 1] - off[h]) // 32) for h in range(g)) + (row0 - off[g]) // 32


@pytest.mark.parametrize("sizes", [[45, 0, 1, 31, 33, 96, 70, 127, 129, 0, 13], [64, 0, 32, 416, 96], [300]])
@pytest.mark.parametrize("N", [24, 72, 1032])
@pytest.mark.parametrize("reuse", [False, True])
def test_grouped_swizzled_planes_written_once(sizes, N, reuse):
    """The grouped cast with one GEMM-ready scale plane per group: the tiles' scale writes and their
    padding zeros together cover every byte of both concatenated planes exactly once."""
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    check_quantize(off[-1], N, 5, offsets=off, swz=True, reuse=reuse)


def model_dact(M, N, grid, dbias=True, reuse=False, offsets=None):
    """quantize_dact_kernel (the backward fusion, and with offsets the grouped gated cast)."""
    rows16 = N % 16 == 0
    out_row, out_col = Plane("out_row", M * N), Plane("out_col", M * N)
    scale_row, scale_col = Plane("scale_row", M * -(-N // 32)), Plane("scale_col", scale_col_rows(M, offsets) * N)
    row_tiles, col_tiles = -(-M // BM), -(-N // DBN)
    ws = Plane("ws", row_tiles * N, 4)
    if offsets is None or all(o % 32 == 0 for o in offsets):
        # flat tiles; also the grouped gated cast's when every offset is a multiple of 32
        tiles = [(rt * BM, min(rt * BM + BM, M), ct * DBN, rt, rt * 4, 0) for rt in range(row_tiles)
                 for ct in range(col_tiles)]
    else:   # the grouped schedule with 64-column tiles: tile_list's rows, DBN's columns
        tiles = []
        G = len(offsets) - 1
        gpre, gsb = [0], [0]
        for g in range(G):
            gpre.append(gpre[-1] + -(-(offsets[g + 1] - offsets[g]) // BM) * col_tiles)
            gsb.append(gsb[-1] + -(-(offsets[g + 1] - offsets[g]) // 32))
        for t in range(gpre[G]):
            lo = max(g for g in range(G) if gpre[g] <= t and gpre[g + 1] > gpre[g])
            local = t - gpre[lo]
            rtl, ct = local // col_tiles, local % col_tiles
            r0 = offsets[lo] + rtl * BM
            tiles.append((r0, min(r0 + BM, offsets[lo + 1]), ct * DBN, gpre[lo] // col_tiles + rtl, gsb[lo] + rtl * 4,
                          lo))
    tid = np.arange(THREADS)
    rb1, c1 = tid >> 6, tid & 63                       # one thread per (32-row block, column)
    w2 = np.repeat(np.arange(8), 2 * 32)
    k2 = np.tile(np.repeat(np.arange(2), 32), 8)
    l2 = np.tile(LANES, 16)
    rg2 = 2 * w2 + k2 if reuse else w2 + 8 * k2   # dSReLU .. dQGeLU: one 32-row block per warp
    rr2, sp2 = l2 >> 2, l2 & 3
    for b in range(grid):
        for t in range(b, len(tiles), grid):
            row0, row_end, col0, rt, sb, g = tiles[t]
            assert (col0 * 2) % 16 == 0 and col0 < N and row0 < M
            grow, gcol = row0 + rb1 * 32, col0 + c1
            sel = (grow < row_end) & (gcol < N)
            scale_col.write((sb + rb1[sel]) * N + gcol[sel])
            if dbias:
                gc = col0 + np.arange(DBN)
                ws.write(rt * N + gc[gc < N], 1, align=4)
            grow, gcol = row0 + rg2 * 8 + rr2, col0 + sp2 * 16
            ok = (row0 + rg2 * 8 < row_end) & (grow < row_end) & (gcol < N)
            half_seg = gcol + 16 > N
            full, part = ok & ~half_seg, ok & half_seg
            for plane in (out_row, out_col):
                plane.write(grow[full] * N + gcol[full], 16, align=16 if rows16 else 8)
                plane.write(grow[part] * N + gcol[part], 8, align=8)
            se = ok & (sp2 % 2 == 0)
            scale_row.write(grow[se] * -(-N // 32) + (gcol[se] >> 5))
    for p in (out_row, out_col, scale_row, scale_col) + ((ws,) if dbias else ()):
        p.once()


@pytest.mark.parametrize("sizes", [[45, 0, 1, 31, 33, 96, 70, 127, 129, 0, 13], [64, 0, 32, 416, 96], [17, 15]])
@pytest.mark.parametrize("N", [24, 96, 1032])
def test_grouped_gated_cast_writes_every_byte_once(sizes, N):
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    model_dact(off[-1], N, 7, dbias=False, reuse=True, offsets=off)
    model_dact(off[-1], N, 304, dbias=False, reuse=True, offsets=off)


@pytest.mark.parametrize("shape", [(45, 80), (70, 24), (257, 1032), (130, 144), (256, 64)])
def test_backward_fusion_writes_every_byte_once(shape):
    for reuse in (False, True):
        model_dact(*shape, grid=5, reuse=reuse)
        model_dact(*shape, grid=304, reuse=reuse)


def model_dgated(M, N, grid):
    """quantize_dgated_kernel: da and db side by side in [M, 2N] codes, [M, 2 ceil(N/32)] row scales,
    [ceil(M/32), 2N] column scales; the stage holds three boxes (g, a, b) of 16 KiB."""
    rows16 = N % 16 == 0
    N2, Cn = 2 * N, -(-N // 32)
    out_row, out_col = Plane("out_row", M * N2), Plane("out_col", M * N2)
    scale_row, scale_col = Plane("scale_row", M * 2 * Cn), Plane("scale_col", -(-M // 32) * N2)
    row_tiles, col_tiles = -(-M // BM), -(-N // DBN)
    tiles = [(rt * BM, min(rt * BM + BM, M), ct * DBN) for rt in range(row_tiles) for ct in range(col_tiles)]
    tid = np.arange(THREADS)
    rb1, c1 = tid >> 6, tid & 63
    w2 = np.repeat(np.arange(8), 2 * 32)
    k2 = np.tile(np.repeat(np.arange(2), 32), 8)
    l2 = np.tile(LANES, 16)
    rg2, rr2, sp2 = 2 * w2 + k2, l2 >> 2, l2 & 3
    for b in range(grid):
        for t in range(b, len(tiles), grid):
            row0, row_end, col0 = tiles[t]
            assert (col0 * 2) % 16 == 0 and col0 < N and row0 < M
            # the a and b maps: bases x and x + 2N bytes, pitch 4N bytes, both 16-byte multiples
            assert (2 * N) % 16 == 0 and (4 * N) % 16 == 0
            grow, gcol = row0 + rb1 * 32, col0 + c1
            sel = (grow < row_end) & (gcol < N)
            for out in range(2):
                scale_col.write((grow[sel] >> 5) * N2 + out * N + gcol[sel])
            grow, gcol = row0 + rg2 * 8 + rr2, col0 + sp2 * 16
            # phase 2 rows stay in the box; the b box is the last 16 KiB of the 48 KiB stage
            assert np.all(rg2 * 8 + rr2 < 128) and np.all(2 * 16384 + (rg2 * 8 + rr2) * 128 + 127 < 3 * 16384)
            ok = (row0 + rg2 * 8 < row_end) & (grow < row_end) & (gcol < N)
            half_seg = gcol + 16 > N
            full, part = ok & ~half_seg, ok & half_seg
            for plane in (out_row, out_col):
                for out in range(2):
                    plane.write(grow[full] * N2 + out * N + gcol[full], 16, align=16 if rows16 else 8)
                    plane.write(grow[part] * N2 + out * N + gcol[part], 8, align=8)
            se = ok & (sp2 % 2 == 0)
            for out in range(2):
                scale_row.write(grow[se] * 2 * Cn + out * Cn + (gcol[se] >> 5))
    for p in (out_row, out_col, scale_row, scale_col):
        p.once()


@pytest.mark.parametrize("shape", [(45, 80), (70, 24), (257, 1032), (130, 144), (256, 64), (33, 8)])
def test_gated_backward_writes_every_byte_once(shape):
    model_dgated(*shape, grid=5)
    model_dgated(*shape, grid=304)


def keep_chunk(c, r):
    return c ^ ((c >> 3) << 1) ^ (r & 1)


def model_dgated_keep(M, N, grid):
    """quantize_dgated_keep_kernel (GeGLU, SwiGLU, QGeGLU backward): 64-row x 64-column tiles, da and
    db kept in fp32 in a [2][64][64] area between the phases; the same side-by-side outputs."""
    KR = 64
    rows16 = N % 16 == 0
    N2, Cn = 2 * N, -(-N // 32)
    out_row, out_col = Plane("out_row", M * N2), Plane("out_col", M * N2)
    scale_row, scale_col = Plane("scale_row", M * 2 * Cn), Plane("scale_col", -(-M // 32) * N2)
    row_tiles, col_tiles = -(-M // KR), -(-N // DBN)
    tiles = [(rt * KR, min(rt * KR + KR, M), ct * DBN) for rt in range(row_tiles) for ct in range(col_tiles)]
    # phase 1: warp w, lane l -> rows 32 (w >> 2) + 8 (w & 3) + 4 (l >> 4) + i, column quad l & 15
    w1, l1 = np.repeat(np.arange(8), 32), np.tile(LANES, 8)
    r01 = 32 * (w1 >> 2) + 8 * (w1 & 3) + 4 * (l1 >> 4)
    stage_reads = []
    keep_w = []
    for i in range(4):
        r = r01 + i
        stage_reads.append(r * 128 + ((((l1 & 15) >> 1) ^ (r & 7)) << 4) + (l1 & 1) * 8)
        kc = keep_chunk(l1 & 15, r)
        for out in range(2):
            keep_w.append((out * KR + r) * 16 + kc)
        # 128-bit keep stores: each quarter warp (8 lanes) meets 8 distinct 16-byte bank groups
        for qw in range(0, 256, 8):
            assert len(set((kc[qw:qw + 8] % 8).tolist())) == 8
    stage_reads = np.concatenate(stage_reads)
    assert stage_reads.size == len(set(stage_reads.tolist())) == KR * 128 // 8 and stage_reads.max() + 8 <= 8192
    keep_w = np.concatenate(keep_w)
    assert keep_w.size == len(set(keep_w.tolist())) == 2 * KR * 16          # every kept chunk once
    # phase 2: warp w -> rows 8w + (l >> 2), segment l & 3: chunks 4 sp + j of its row
    w2, l2 = np.repeat(np.arange(8), 32), np.tile(LANES, 8)
    r2, sp2 = 8 * w2 + (l2 >> 2), l2 & 3
    keep_r = []
    for j in range(4):
        kc = keep_chunk(4 * sp2 + j, r2)
        for qw in range(0, 256, 8):
            assert len(set((kc[qw:qw + 8] % 8).tolist())) == 8
        for out in range(2):
            keep_r.append((out * KR + r2) * 16 + kc)
    assert set(np.concatenate(keep_r).tolist()) == set(keep_w.tolist())  # phase 2 reads what phase 1 kept
    # the scale step: thread t -> (output t >> 7, row block (t >> 6) & 1, column t & 63)
    t = np.arange(THREADS)
    so, srb, sc = t >> 7, (t >> 6) & 1, t & 63
    assert len({(int(a), int(b), int(c)) for a, b, c in zip(so, srb, sc)}) == 256
    for b in range(grid):
        for ti in range(b, len(tiles), grid):
            row0, row_end, col0 = tiles[ti]
            assert (col0 * 2) % 16 == 0 and col0 < N and row0 < M
            grow, gcol = row0 + srb * 32, col0 + sc
            sel = (grow < row_end) & (gcol < N)
            scale_col.write((grow[sel] >> 5) * N2 + so[sel] * N + gcol[sel])
            grow, gcol = row0 + r2, col0 + sp2 * 16
            ok = (row0 + 8 * w2 < row_end) & (grow < row_end) & (gcol < N)
            half_seg = gcol + 16 > N
            full, part = ok & ~half_seg, ok & half_seg
            for out in range(2):
                for plane in (out_row, out_col):
                    plane.write(grow[full] * N2 + out * N + gcol[full], 16, align=16 if rows16 else 8)
                    plane.write(grow[part] * N2 + out * N + gcol[part], 8, align=8)
                se = ok & (sp2 % 2 == 0)
                scale_row.write(grow[se] * 2 * Cn + out * Cn + (gcol[se] >> 5))
    for p_ in (out_row, out_col, scale_row, scale_col):
        p_.once()


@pytest.mark.parametrize("shape", [(45, 80), (70, 24), (257, 1032), (130, 144), (256, 64), (33, 8), (64, 8)])
def test_gated_backward_keep_kernel_writes_every_byte_once(shape):
    model_dgated_keep(*shape, grid=5)
    model_dgated_keep(*shape, grid=304)


def grouped_reduce_reads(hdr, N):
    """dbias_reduce_grouped_kernel: the partial rows each (group, column) sums, for one CTA of 32
    columns, following its 16 contiguous warp ranges and the head / tail hand-over."""
    G = len(hdr) - 1
    T = hdr[G]
    sums = {g: [] for g in range(G)}
    for w in range(16):
        a, b = T * w // 16, T * (w + 1) // 16
        for t in range(a, b):
            g = max(i for i in range(G) if hdr[i] <= t)
            sums[g].append(t)
    return sums


@pytest.mark.parametrize("sizes", [[64, 0, 32, 416, 0, 0, 128, 96, 160, 32], [8192], [0, 2080, 0, 0, 32, 4096, 0]])
def test_grouped_reduce_reads_each_partial_row_of_its_group_once(sizes):
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(int).tolist()
    N = 96
    m = model_quantize(off[-1], N, 304, offsets=off, dbias=True)
    col_tiles = -(-N // BN)
    G = len(sizes)
    hdr, acc = [0], 0
    for g in range(G):
        acc += -(-sizes[g] // BM) * col_tiles
        hdr.append(acc // col_tiles)
    sums = grouped_reduce_reads(hdr, N)
    written_rows = {t[3] for t in m["tiles"]}
    for g in range(G):
        assert sorted(sums[g]) == list(range(hdr[g], hdr[g + 1]))
        assert set(sums[g]) <= written_rows

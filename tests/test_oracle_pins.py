"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU needed).

Page tags: [MLSys-TMA] mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA";
[H200-TMA] coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card.
"""
import numpy as np
import pytest

import oracle
import workloads
from conftest import read_golden
from expect import (apply_page_swizzle128, box_none, checksum_reference, inbounds_mask,
                    sector_table, strided_view)


def w1_map(buf, span):
    return oracle.Map(buf, 2, dims=[128, 16], strides=[256], box=[64, 8], span=span)


# ---- [MLSys-TMA] §"TMA 如何写入 swizzled layout": the 16 x 128 fp16 tensor and its 8 x 64 tile --
@pytest.mark.parametrize("start", [(0, 0), (64, 8)])
def test_w1_none_is_plain_slice(start):
    x = workloads.w1_tensor()
    img = oracle.image(w1_map(x, 0), start).view(np.uint16).reshape(8, 64)
    c0, r0 = start
    np.testing.assert_array_equal(img, x[r0:r0 + 8, c0:c0 + 64])


@pytest.mark.parametrize("start", [(0, 0), (64, 8)])
def test_w1_128b_follows_col_xor_row(start):
    """Closed form: physical sector (col XOR row) of image row r holds logical sector col, i.e.
    the eight fp16 values (r0 + r)*128 + c0 + 8*col + e."""
    x = workloads.w1_tensor()
    img = oracle.image(w1_map(x, 128), start).view(np.uint16).reshape(8, 8, 8)
    t = sector_table()
    c0, r0 = start
    for r in range(8):
        for col in range(8):
            want = (r0 + r) * 128 + c0 + 8 * col + np.arange(8)
            np.testing.assert_array_equal(img[r, t[r, col]], want)
            assert t[r, col] == col ^ r
    # spot values: row 1's bytes 16..31 are logical sector 0 of row 1 -> 128..135
    flat = img.reshape(-1)
    if start == (0, 0):
        np.testing.assert_array_equal(flat[64 + 8:64 + 16], np.arange(128, 136))
        np.testing.assert_array_equal(flat[7 * 64:7 * 64 + 8], np.arange(952, 960))


# ---- [MLSys-TMA] §"用 3D TMA 搬运多个 swizzle atoms" ----------------------------------------------
def w2_map(buf, span, group_cols=64, offset=0, groups=4):
    gbytes = group_cols * 2
    return oracle.Map(buf, 2, dims=[group_cols, 16, groups], strides=[512, gbytes],
                      box=[group_cols, 16, 128 // group_cols], span=span, offset=offset)


def test_3d_regroup_is_address_identity():
    """global[row, j] == global3[j // 64, row, j % 64] for every element of the 16 x 256 matrix."""
    x = workloads.w2_tensor()
    m = oracle.Map(x, 2, dims=[64, 16, 4], strides=[512, 128], box=[1, 1, 1])
    for row in range(16):
        for j in range(256):
            v = oracle.image(m, (j % 64, row, j // 64)).view(np.uint16)[0]
            assert v == x[row, j]


@pytest.mark.parametrize("slice_no", [0, 1])
def test_w2_128b_image_is_four_swizzled_atoms(slice_no):
    x = workloads.w2_tensor()
    c0 = 128 * slice_no
    none = oracle.image(w2_map(x, 0), (0, 0, 2 * slice_no)).view(np.uint16)
    g = np.stack([x[:, c0:c0 + 64], x[:, c0 + 64:c0 + 128]])  # (group, row, col)
    np.testing.assert_array_equal(none.reshape(2, 16, 64), g)
    sw = oracle.image(w2_map(x, 128), (0, 0, 2 * slice_no))
    np.testing.assert_array_equal(sw, apply_page_swizzle128(none.view(np.uint8)))
    # per-slice map (base moved by the slice's byte offset, two groups) gives the same image
    per = oracle.Map(x, 2, dims=[64, 16, 2], strides=[512, 128], box=[64, 16, 2], span=128,
                     offset=c0 * 2)
    np.testing.assert_array_equal(oracle.image(per, (0, 0, 0)), sw)


@pytest.mark.parametrize("span,gcols", [(64, 32), (32, 16)])
def test_w2_narrow_swizzles_permute_whole_sectors(span, gcols):
    """64B / 32B (the pages name them without defining them; their pin is the published pattern
    test above): the same 16-byte units as the unswizzled image, each unit moved whole within its
    atom."""
    x = workloads.w2_tensor()
    ng = 128 // gcols
    for start in [(0, 0, 0), (0, 0, ng)]:
        none = oracle.image(w2_map(x, 0, gcols, groups=256 // gcols), start).reshape(-1, 16)
        sw = oracle.image(w2_map(x, span, gcols, groups=256 // gcols), start).reshape(-1, 16)
        atom = 8 * span // 16  # units per 8-row atom
        for a in range(0, none.shape[0], atom):
            got = sorted(map(bytes, sw[a:a + atom]))
            assert got == sorted(map(bytes, none[a:a + atom]))


@pytest.mark.parametrize("span,gcols", [(64, 32), (32, 16)])
def test_narrow_swizzles_spread_a_column_over_eight_bank_sectors(span, gcols):
    """64B / 32B: the pages fix no permutation for them (the published pattern test above pins
    it).  They fix its purpose ([MLSys-TMA] "128-byte swizzle 的分组要求": eight rows reading the same column should
    hit eight distinct bank sectors, and a narrower atom is the fallback when 128 B do not fit),
    and, by the 128B rule of "TMA 如何写入 swizzled layout", that sectors move inside their own
    row by a pattern that depends on row % 8 only.  Checked on the W2 images against the
    unswizzled image: each 16-byte unit stays in its span-byte row, its new place depends on
    (row % 8, column) alone, and any eight consecutive rows put a column in eight distinct bank
    sectors.  Unswizzled rows of this width reach only 16 * 8 / span distinct sectors."""
    x = workloads.w2_tensor()
    ng = 128 // gcols
    units = span // 16
    for start in [(0, 0, 0), (0, 0, ng)]:
        none = oracle.image(w2_map(x, 0, gcols, groups=256 // gcols), start).reshape(-1, units, 16)
        sw = oracle.image(w2_map(x, span, gcols, groups=256 // gcols), start).reshape(-1, units, 16)
        rows = none.shape[0]
        place = np.empty((rows, units), np.int64)
        for r in range(rows):
            for c in range(units):
                hit = [k for k in range(units) if bytes(sw[r, k]) == bytes(none[r, c])]
                assert len(hit) == 1  # the unit is found in its own row, exactly once
                place[r, c] = hit[0]
        for r in range(8, rows):
            np.testing.assert_array_equal(place[r], place[r % 8])
        for r0 in range(rows - 7):
            for c in range(units):
                sectors = {((r * span + place[r, c] * 16) >> 4) & 7 for r in range(r0, r0 + 8)}
                plain = {((r * span + c * 16) >> 4) & 7 for r in range(r0, r0 + 8)}
                assert len(sectors) == 8
                assert len(plain) == 16 * 8 // span


# ---- all three swizzle modes against NVIDIA's published patterns -----------------------------
def test_swizzle_modes_match_the_published_chunk_patterns():
    """orc_swz for 32B, 64B and 128B against the chunk permutations NVIDIA's CUDA documentation
    draws for the three modes (tests/golden/cuda_tma_swizzle_modes.txt, cited there), over four
    repeats of each pattern, byte by byte: a 16-byte chunk moves whole, to the physical chunk the
    table gives for its 128-byte line inside the repeat period.  This is the pin of the 64B and
    32B modes, which the pages name but do not define."""
    rows = read_golden("cuda_tma_swizzle_modes.txt")
    table = {}
    for r in rows:
        mode, period, line, *phys = map(int, r)
        table.setdefault((mode, period), {})[line] = phys
    assert set(table) == {(32, 256), (64, 512), (128, 1024)}
    for (mode, period), lines in table.items():
        assert sorted(lines) == list(range(period // 128))
        for off in range(4 * period):
            line = (off % period) // 128
            chunk, byte = (off % 128) // 16, off % 16
            want = off - off % 128 + lines[line][chunk] * 16 + byte
            assert oracle.swz(off, mode) == want, (mode, off)


# ---- swizzle function invariants ------------------------------------------------------------
@pytest.mark.parametrize("span", [32, 64, 128])
def test_swizzle_is_involution_and_bijection(span):
    block = 8 * span
    for base in (0, block, 7 * block):
        img = [oracle.swz(base + o, span) for o in range(block)]
        assert sorted(img) == list(range(base, base + block))
        assert all(oracle.swz(v, span) == base + o for o, v in enumerate(img))
        assert all((v ^ (base + o)) & ~0x70 == 0 for o, v in enumerate(img))  # only bits 4..6


def test_swizzle_none_is_identity():
    assert all(oracle.swz(o, 0) == o for o in range(4096))


# ---- [MLSys-TMA] §"128-byte swizzle 的分组要求" ----------------------------------------------------
def test_bank_sectors_grouped_vs_ungrouped():
    want = {r[0]: (int(r[1]), int(r[2])) for r in read_golden("mlsys_bank_sectors.txt")}
    for col in range(16):
        for row0 in range(9):
            for grouped in (True, False):
                s = oracle.bank_sectors(col, row0, grouped)
                distinct, hits = want["grouped" if grouped else "ungrouped"]
                assert len(set(s)) == distinct
                assert max(s.count(v) for v in set(s)) == hits
                for k, v in enumerate(s):
                    row = row0 + k
                    if grouped:
                        assert v == (col % 8) ^ (row % 8)
                    else:
                        assert v == (col % 8) ^ ((2 * row + col // 8) % 8)


# ---- [MLSys-TMA] §"如何等待 TMA load 完成" and [H200-TMA] §05 --------------------------------------
def test_expect_tx_tally_of_two_tiles():
    g = {r[0]: r[1:] for r in read_golden("mlsys_expect_tx_tally.txt")}
    a, b, total = int(g["tile_bytes_A"][0]), int(g["tile_bytes_B"][0]), int(g["expect_total"][0])
    assert a + b == total
    m = oracle.Mbar(1)
    m.arrive_expect_tx(total)
    assert (m.pending, m.tx, int(m.test_wait(0))) == tuple(map(int, g["after_arrive_expect_tx"]))
    m.complete_tx(a)
    assert not m.test_wait(0)
    m.complete_tx(b)
    assert m.test_wait(0)
    # after completion the next phase starts: pending arrivals reset to the init count
    assert (m.pending - 1, m.tx, int(m.test_wait(0))) == tuple(map(int, g["after_both_copies"]))
    assert not m.test_wait(1)


def test_arrive_before_expect_completes_early():
    """The card's pitfall: the byte count must be announced before the copy is counted on; a bare
    arrival with nothing expected completes the phase while data is still in flight."""
    m = oracle.Mbar(1)
    m.arrive()
    assert m.test_wait(0)
    m.expect_tx(2048)  # too late: this belongs to the next phase
    assert not m.test_wait(1)


def test_ring_stage_tally_is_32768():
    a, b = workloads.w5b_maps()
    buf = np.zeros(16, np.uint16)
    ma = oracle.Map(buf, 2, a["dims"], a["strides"], a["box"], a["span"])
    mb = oracle.Map(buf, 2, b["dims"], b["strides"], b["box"], b["span"])
    assert ma.box_bytes + mb.box_bytes == 32768
    m = oracle.Mbar(1)
    m.arrive_expect_tx(ma.box_bytes + mb.box_bytes)
    m.complete_tx(ma.box_bytes)
    assert not m.test_wait(0)
    m.complete_tx(mb.box_bytes)
    assert m.test_wait(0)


# ---- brute force on tiny tensors -------------------------------------------------------------
def random_case(rng, span):
    """A tiny map: dim 0 contiguous, dims 1.. stored in a random order with random padding (so
    strides are often non-monotone, like the 3-D regroup), and a start anywhere from 3 before the
    tensor to 3 past its end."""
    rank = int(rng.integers(1, 6))
    esize = int(rng.choice([2, 4])) if span else int(rng.choice([1, 2, 4, 8]))
    dims = [int(rng.integers(1, 6)) for _ in range(rank)]
    box = [int(rng.integers(1, 5)) for _ in range(rank)]
    if span:
        box[0] = span // esize
        dims[0] = int(rng.integers(1, box[0] + 6))
    strides = [esize] * rank
    step = (dims[0] + int(rng.integers(0, 3))) * esize
    for d in rng.permutation(np.arange(1, rank)):
        strides[d] = step
        step *= dims[d] + int(rng.integers(0, 3))
    start = [int(rng.integers(-3, d + 4)) for d in dims]
    return rank, esize, dims, box, strides, step, start


@pytest.mark.parametrize("span", [0, 128, 64, 32])
def test_brute_force_image_and_store(span):
    rng = np.random.default_rng(1000 + span)
    for _ in range(150):
        rank, esize, dims, box, strides, total, start = random_case(rng, span)
        buf = rng.integers(0, 256, size=total + 64, dtype=np.uint16).astype(np.uint8)
        m = oracle.Map(buf, esize, dims, strides[1:], box, span)
        img = oracle.image(m, start)
        view = strided_view(buf, 0, esize, dims, strides[1:])
        none = box_none(view, start, box)
        if span == 0:
            np.testing.assert_array_equal(img, none.reshape(-1).view(np.uint8))
        elif span == 128:
            np.testing.assert_array_equal(img, apply_page_swizzle128(
                np.ascontiguousarray(none).reshape(-1).view(np.uint8)))
        else:  # narrow modes (pinned by the published patterns): same 16-byte units, permuted in each atom
            u_img = img.reshape(-1, 16)
            u_none = np.ascontiguousarray(none).reshape(-1).view(np.uint8).reshape(-1, 16)
            atom = 8 * span // 16
            for a in range(0, u_img.shape[0], atom):
                assert sorted(map(bytes, u_img[a:a + atom])) == sorted(map(bytes,
                                                                           u_none[a:a + atom]))
        # store(image) into a sentinel-filled copy restores exactly the in-bounds elements
        dst = np.full_like(buf, 0xA5)
        md = oracle.Map(dst, esize, dims, strides[1:], box, span)
        oracle.store(md, start, img)
        dview = strided_view(dst, 0, esize, dims, strides[1:])
        sent = np.full(1, 0xA5A5A5A5A5A5A5A5, dtype=np.uint64).view(np.uint8)[:esize]
        sent = sent.view(view.dtype)[0]
        mask = inbounds_mask(dims, start, box)
        got = box_none(dview, start, box)
        np.testing.assert_array_equal(got[mask], none[mask])
        # nothing outside the box's in-bounds elements was written
        touched = np.zeros(view.shape, dtype=bool)
        idx = [np.arange(max(0, start[i]), min(dims[i], start[i] + box[i]))
               for i in reversed(range(rank))]
        if all(len(i) for i in idx):
            touched[np.ix_(*idx)] = True
        assert np.all(dview[~touched] == sent)


def test_box_grid_covers_tensor_once():
    rng = np.random.default_rng(7)
    for _ in range(50):
        rank = int(rng.integers(1, 6))
        dims = [int(rng.integers(1, 9)) for _ in range(rank)]
        box = [int(rng.integers(1, 5)) for _ in range(rank)]
        buf = np.zeros(8, np.uint8)
        m = oracle.Map(buf, 1, dims, [1] * (rank - 1), box)
        count = np.zeros(tuple(reversed(dims)), dtype=np.int64)
        nb = 1
        for d, b in zip(dims, box):
            nb *= -(-d // b)
        assert m.num_boxes == nb
        for b in range(m.num_boxes):
            s = m.box_start(b)
            idx = tuple(slice(s[i], min(dims[i], s[i] + box[i])) for i in reversed(range(rank)))
            count[idx] += 1
        assert np.all(count == 1)


# ---- [Book-TMA] reduce: one IEEE binary32 add per element ---------------------------------------
def test_reduce_add_equals_numpy_float32():
    dst, src = workloads.w5a_tensors(rows=300, cols=200, seed_dst=5, seed_src=6)
    want = (dst + src).astype(np.float32)
    md = oracle.Map(dst, 4, dims=[200, 300], strides=[800], box=[32, 128], span=128)
    ms = oracle.Map(src, 4, dims=[200, 300], strides=[800], box=[32, 128], span=128)
    oracle.tile_reduce_add(md, ms)
    np.testing.assert_array_equal(dst.view(np.uint32), want.view(np.uint32))


# ---- ring consumer checksum --------------------------------------------------------------------
@pytest.mark.parametrize("span", [0, 128])
def test_tile_checksum_matches_numpy(span):
    rng = np.random.default_rng(11)
    rows = workloads.normal_bf16((128, 64), 12)
    none = rows.reshape(-1).view(np.uint8)
    img = none if span == 0 else apply_page_swizzle128(none)
    cs, bits = oracle.tile_checksum(img, 128, 128, span)
    want_cs, want_bits = checksum_reference(rows)
    assert bits == want_bits
    assert np.float32(cs).view(np.uint32) == want_cs.view(np.uint32)
    del rng


def test_stream_checksums_pair_tiles_in_grid_order():
    a, b = workloads.w5b_tensors(m=256, k=192, n=192, seed_a=1, seed_b=2)
    ra, rb = workloads.w5b_maps(m=256, k=192, n=192)
    ma = oracle.Map(a, 2, ra["dims"], ra["strides"], ra["box"], ra["span"])
    mb = oracle.Map(b, 2, rb["dims"], rb["strides"], rb["box"], rb["span"])
    assert ma.num_boxes == mb.num_boxes == 6
    cs_a, cs_b, bits_a, bits_b = oracle.stream_checksums(ma, mb)
    for t in range(6):
        for x, m, cs, bits in ((a, ma, cs_a, bits_a), (b, mb, cs_b, bits_b)):
            c0, r0 = m.box_start(t)
            tile = np.zeros((128, 64), np.uint16)
            part = x[r0:r0 + 128, c0:c0 + 64]
            tile[:part.shape[0], :part.shape[1]] = part
            want_cs, want_bits = checksum_reference(tile)
            assert int(bits[t]) == want_bits
            assert cs[t].view(np.uint32) == want_cs.view(np.uint32)


def test_workload_generators_are_seeded_and_clean():
    np.testing.assert_array_equal(workloads.w3_tensor(64, 64), workloads.w3_tensor(64, 64))
    x = workloads.w2_tensor()
    assert not np.any((x & 0x7C00) == 0x7C00)
    d, s = workloads.w5a_tensors(rows=64, cols=64)
    exact = d.astype(np.float64) + s.astype(np.float64)
    assert not np.any((np.abs(exact) < 2.0 ** -126) & (exact != 0))
    w4 = workloads.w4_tensor(batch=2, rows=5, cols=1000, pitch=1024)
    assert np.all(w4[:, :, 1000:] == workloads.SENTINEL_U16)

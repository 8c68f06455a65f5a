"""Index arithmetic of the shared-memory operand images, checked on the CPU.

The tensor-core kernels place fp16/bf16 elements in 128-byte-swizzled tiles
(K-major: rows of 64 elements per K block, 16-byte chunks XOR-permuted by
row mod 8; MN-major: 64-wide MN atoms, K rows 128 bytes apart, 8-row K groups).
These tests restate the offset formulas the kernels use and check that every
tile is filled exactly once, inside its buffer, and that the shortcuts the
kernels take (fixed per-thread offsets, the seam record's half-size Kbar
planes) agree with the general formulas."""
import itertools


def sw128_off(row, k, rows):
    """K-major SW128: byte offset of 2-byte element (row, k) in a tile of `rows`
    rows and 64-element K blocks."""
    kb, kk = k >> 6, k & 63
    return kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + \
        (((kk >> 3) ^ (row & 7)) << 4) + ((kk & 7) << 1)


def mn_off(mn, k, lbo, sbo):
    """MN-major SW128: byte offset of 2-byte element (mn, k) with MN atoms of 64
    elements `lbo` bytes apart and 8-row K groups `sbo` bytes apart."""
    return (mn >> 6) * lbo + (k >> 3) * sbo + (k & 7) * 128 + \
        ((((mn >> 3) & 7) ^ (k & 7)) << 4) + ((mn & 7) << 1)


def test_k_major_tiles_are_bijective():
    for rows, K in ((128, 128), (16, 128), (64, 64)):
        offs = [sw128_off(r, k, rows) for r in range(rows) for k in range(K)]
        assert sorted(offs) == list(range(0, rows * K * 2, 2))


def test_mn_major_tiles_are_bijective():
    # (MN extent, K extent, lbo, sbo): the build's [64 K][64..128 MN] tiles and the
    # seam record's Kbar image (16 K rows, MN atoms 1 KB apart, K groups 2 KB apart)
    for MN, K, lbo, sbo in ((128, 64, 8192, 1024), (64, 64, 8192, 1024), (128, 16, 1024, 2048)):
        offs = [mn_off(m, k, lbo, sbo) for m in range(MN) for k in range(K)]
        assert sorted(offs) == list(range(0, MN * K * 2, 2))


def test_kbar_image_nonzero_rows_fill_the_first_half():
    """Rows s < 8 of the Kbar image occupy bytes [0, 2048) of a plane and rows
    8..15 (zero) bytes [2048, 4096), so the record stores only the first half;
    the prep kernel's per-lane offset (lane = channels 4L .. 4L+3) agrees."""
    lo = [mn_off(i, s, 1024, 2048) for i in range(128) for s in range(8)]
    hi = [mn_off(i, s, 1024, 2048) for i in range(128) for s in range(8, 16)]
    assert max(lo) < 2048 <= min(hi) and max(hi) < 4096
    for lane, s in itertools.product(range(32), range(8)):
        lane_off = (lane >> 4) * 1024 + s * 128 + ((((lane >> 1) & 7) ^ s) << 4) + (lane & 1) * 8
        assert lane_off == mn_off(4 * lane, s, 1024, 2048)


def test_converter_fixed_offsets_match_the_tile():
    """The compose converter's thread ct handles k = 4 (ct mod 32) .. +3 of rows
    ct / 32 + 2 it; over four consecutive it the swizzle phase takes four values,
    so it keeps four base offsets and adds 1 KB per eight rows."""
    for ct in range(64):
        k4, i0 = ct & 31, ct >> 5
        base = [(k4 >> 4) * 16384 + (i0 + 2 * u) * 128 + ((((k4 & 15) >> 1) ^ (i0 + 2 * u)) << 4)
                + (k4 & 1) * 8 for u in range(4)]
        for m in range(16):
            for u in range(4):
                e = ct + 256 * m + 64 * u
                assert base[u] + 1024 * m == sw128_off(e >> 5, 4 * (e & 31), 128)


def test_seam_record_layout():
    """The chunk record in global memory (W image, the Kbar planes' first
    halves, U~ and the tables) and its shared-memory slot: every piece copied
    lands where the kernel reads it, 16-byte aligned, without overlap."""
    rec = {"w": (0, 8192), "kh": (8192, 2048), "kl": (10240, 2048), "u_t": (12288, 4608)}
    slot = {"w": 0, "kh": 8192, "kl": 8192 + 4096, "u_t": 16384}
    assert sum(n for _, n in rec.values()) == 16896
    spans = sorted((slot[k], slot[k] + rec[k][1]) for k in rec)
    assert all(a % 16 == 0 for a, _ in spans) and all(n % 16 == 0 for _, n in rec.values())
    assert all(spans[i][1] <= spans[i + 1][0] for i in range(len(spans) - 1))
    assert spans[-1][1] <= 20992                       # the slot
    # the zeroed halves of the Kbar planes are exactly what is not copied
    zero = [(8192 + 2048, 8192 + 4096), (12288 + 2048, 12288 + 4096)]
    for a, b in zero:
        assert all(not (a < e and s < b) for s, e in spans)

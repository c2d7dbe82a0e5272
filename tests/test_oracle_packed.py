"""Pins for the packed (tensor-core staging order) MX scale layout (CPU only).

The scatter formulation is checked against the tile-by-tile reshape
formulation, against positions worked out by hand from the layout's
definition, and against invariants (every scale lands exactly once, everything
else is zero, empty segments own no tiles).  Its reading by the tensor cores
is pinned by the GPU GEMM tests that feed it to the GEMM."""

import numpy as np
import pytest

import oracle

SEGMENTS = [
    [1], [128], [129], [0, 5, 0], [1, 130], [127, 128, 129, 0, 300], [0, 0, 1], [513, 7, 256],
]


@pytest.mark.parametrize("seg", SEGMENTS)
@pytest.mark.parametrize("blocks", [1, 4, 5, 7, 12])
def test_two_formulations_agree(seg, blocks):
    rng = np.random.default_rng(sum(seg) + blocks)
    s = rng.integers(0, 256, size=(sum(seg), blocks), dtype=np.uint8)
    a = oracle.pack_scales_mma(s, seg)
    b = oracle.pack_scales_mma_by_tiles(s, seg)
    assert a.shape == b.shape and np.array_equal(a, b)
    assert a.size == oracle.packed_scale_bytes(seg, blocks)


def test_hand_worked_positions():
    # segments of 1 and 130 rows, 5 blocks: tiles [seg0 t0, seg1 t0, seg1 t1] -> RT = 3; KC = 2
    seg, blocks = [1, 130], 5
    s = np.zeros((131, blocks), dtype=np.uint8)
    s[0, 0] = 11            # seg 0 row 0, block 0 -> chunk (0, 0), byte 0
    s[1, 1] = 22            # seg 1 row 0, block 1 -> chunk (0, 1), lane 0, quarter 0, j 1 -> 512 + 1
    s[1 + 33, 2] = 33       # seg 1 row 33 -> lane 1, quarter 1; block 2 -> 512 + 16 + 4 + 2 = 534
    s[1 + 129, 4] = 44      # seg 1 row 129 -> tile 2, row 1; block 4 -> chunk (1, 2): (3 + 2)*512 + 16 = 2576
    s[1 + 127, 3] = 55      # seg 1 row 127 -> lane 31, quarter 3; block 3 -> 512 + 496 + 12 + 3 = 1023
    p = oracle.pack_scales_mma(s, seg)
    assert p.size == 2 * 3 * 512
    expect = {0: 11, 513: 22, 534: 33, 2576: 44, 1023: 55}
    for pos, v in expect.items():
        assert p[pos] == v, pos
    assert np.count_nonzero(p) == len(expect)


def test_every_scale_lands_once_and_the_rest_is_zero():
    seg, blocks = [3, 0, 200, 128, 1], 9
    R = sum(seg)
    s = (np.arange(R * blocks, dtype=np.int64) % 255 + 1).astype(np.uint8).reshape(R, blocks)
    p = oracle.pack_scales_mma(s, seg)
    assert np.count_nonzero(p) == R * blocks
    assert np.array_equal(np.sort(p[p != 0]), np.sort(s.ravel()))
    # tiles: 1 + 0 + 2 + 1 + 1 = 5, chunks: 3
    assert oracle.tile_prefix(seg).tolist() == [0, 1, 1, 3, 4, 5]
    assert p.size == 3 * 5 * 512


def test_uniform_segments_equal_plain_row_tiles():
    # weights: G segments of N rows, N a multiple of 128 -> tile rt holds rows 128*rt .. 128*rt + 127
    G, N, blocks = 3, 256, 8
    rng = np.random.default_rng(5)
    s = rng.integers(0, 256, size=(G * N, blocks), dtype=np.uint8)
    p = oracle.pack_scales_mma(s, [N] * G).reshape(2, G * N // 128, 32, 4, 4)  # kc, rt, lane, quarter, j
    for rt in (0, 3, 5):
        for kc in (0, 1):
            rows = s[rt * 128:(rt + 1) * 128, kc * 4:(kc + 1) * 4]          # [128, 4]
            for lane in (0, 17, 31):
                for qtr in range(4):
                    assert np.array_equal(p[kc, rt, lane, qtr], rows[qtr * 32 + lane])


# ------------------------------------------------------------------ column-wise (k-segmented) operands

KSEG = [[0, 32], [0, 128], [0, 160], [0, 0, 64, 64, 320], [0, 32, 32, 288], [0, 512, 544]]


@pytest.mark.parametrize("poff", KSEG)
@pytest.mark.parametrize("C", [1, 128, 130, 300])
def test_kseg_two_formulations_agree(poff, C):
    rng = np.random.default_rng(C + poff[-1])
    s = rng.integers(0, 256, size=(C, poff[-1] // 32), dtype=np.uint8)
    a = oracle.pack_scales_mma_kseg(s, poff)
    b = oracle.pack_scales_mma_kseg_by_experts(s, poff)
    assert np.array_equal(a, b)
    assert a.size == oracle.kseg_chunk_prefix(poff)[-1] * ((C + 127) // 128) * 512


def test_kseg_hand_worked_positions():
    # two experts of 160 and 32 padded positions, 130 channels: expert 0 has chunks 0 (blocks 0-3)
    # and 1 (block 4), expert 1 chunk 2 (block 0); RT = 2 (channels 0-127, 128-129)
    poff, C = [0, 160, 192], 130
    s = np.zeros((C, 6), dtype=np.uint8)
    s[0, 0] = 11       # kc 0, rt 0, lane 0, quarter 0, j 0          -> byte 0
    s[33, 3] = 22      # kc 0, rt 0, channel 33 -> lane 1, quarter 1, j 3 -> 16 + 4 + 3 = 23
    s[0, 4] = 33       # expert 0 block 4 -> kc 1, j 0: (1*2 + 0)*512 = 1024
    s[129, 5] = 44     # expert 1 block 0 -> kc 2, rt 1, channel 1: (2*2 + 1)*512 + 16 = 2576
    p = oracle.pack_scales_mma_kseg(s, poff)
    assert p.size == 3 * 2 * 512
    for pos, v in {0: 11, 23: 22, 1024: 33, 2576: 44}.items():
        assert p[pos] == v, pos
    assert np.count_nonzero(p) == 4


def test_kseg_uniform_segments_match_the_dgrad_weight_chunks():
    # dgrad weights: G segments of N (N % 128 == 0) -> k-chunk g*N/128 + c, exactly the plain 128-column chunks
    G, N, C = 3, 256, 256
    rng = np.random.default_rng(4)
    s = rng.integers(1, 256, size=(C, G * N // 32), dtype=np.uint8)
    poff = np.arange(G + 1) * N
    p = oracle.pack_scales_mma_kseg(s, poff).reshape(G * N // 128, 2, 32, 4, 4)   # kc, rt, lane, quarter, j
    for kc in (0, 3, 5):
        for rt in (0, 1):
            blk = s[rt * 128:(rt + 1) * 128, kc * 4:(kc + 1) * 4]
            for lane in (0, 9, 31):
                for q in range(4):
                    assert np.array_equal(p[kc, rt, lane, q], blk[q * 32 + lane])

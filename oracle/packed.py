"""MX scales in the tensor-core staging order ("pre-swizzled" scales).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Integrate MXFP4 hipblaslt GEMM support" (ROCm TransformerEngine PR #697),
Takeaways: a GEMM fed plain UE8M0 scales ran at about 0.61x of the one fed
scales already laid out in the matrix engine's blocked order, so that order is
worth producing in the quantizer itself; "Grouped MXFP8 GEMMs with HipKittens"
(PR #661) does the same with its "fused scale packing kernel" commit.
The blocked order here is the one a Blackwell block-scaled MMA reads: the
scale factors of 128 rows x 4 blocks (128 contraction elements) form one
512-byte chunk, which fills four TMEM columns of a 32-lane quarter -- lane l
holds rows l, l+32, l+64, l+96, four block bytes each.

The layout of an operand whose rows are cut into segments (the experts' rows:
the routing splits for activations and gradients, G equal segments of N rows
for forward weights):

* each segment is cut into row tiles of 128, the last one short; tiles are
  numbered across segments in order (``tile_prefix``), RT tiles in all;
* the contraction is cut into chunks of 4 blocks, KC = ceil(blocks / 4);
* chunk (kc, rt) occupies bytes [(kc*RT + rt)*512, +512), and the scale of
  local row i of the tile and block j of the chunk sits at byte
  (i % 32)*16 + (i // 32)*4 + j;
* every byte not covered by a row or block of the operand is zero.

Column-wise (k-segmented) operands -- the dgrad weights and both wgrad
operands, whose contraction is cut into the experts' padded segments -- use
the same chunks with the chunk grid restarting at every segment
(``pack_scales_mma_kseg``).

Parity: ``pack_scales_mma`` (a scatter, one index formula per scale) is pinned
on the CPU against ``pack_scales_mma_by_tiles`` (each chunk built as a
reshaped and transposed 128 x 4 tile) and by invariants; its reading by the
tensor cores is pinned on the GPU, where a GEMM fed these bytes must match the
oracle's plain grouped GEMM.
"""

from __future__ import annotations

import numpy as np

TILE_ROWS = 128
CHUNK_BLOCKS = 4
CHUNK_BYTES = 512


def tile_prefix(seg_rows) -> np.ndarray:
    """[G+1] exclusive prefix of ceil(m_g / 128): the first row tile of each
    segment; entry G is RT."""
    m = np.asarray(seg_rows, dtype=np.int64)
    tiles = (m + TILE_ROWS - 1) // TILE_ROWS
    return np.concatenate([[0], np.cumsum(tiles)]).astype(np.int64)


def packed_scale_bytes(seg_rows, blocks: int) -> int:
    """Bytes of the packed layout: KC * RT * 512."""
    kc = (blocks + CHUNK_BLOCKS - 1) // CHUNK_BLOCKS
    return int(kc * tile_prefix(seg_rows)[-1] * CHUNK_BYTES)


def pack_scales_mma(scale: np.ndarray, seg_rows) -> np.ndarray:
    """Plain scales [R, blocks] (uint8, rows in segment order) -> the packed
    bytes (uint8, ``packed_scale_bytes`` long)."""
    scale = np.asarray(scale, dtype=np.uint8)
    R, KB = scale.shape
    m = np.asarray(seg_rows, dtype=np.int64)
    assert m.sum() == R and (m >= 0).all()
    rtp = tile_prefix(m)
    RT = int(rtp[-1])
    out = np.zeros(packed_scale_bytes(m, KB), dtype=np.uint8)
    if R == 0 or KB == 0:
        return out
    off = np.concatenate([[0], np.cumsum(m)])
    r = np.arange(R, dtype=np.int64)
    g = np.searchsorted(off, r, side="right") - 1      # segment of each row
    i = r - off[g]                                     # row inside its segment
    rt = rtp[g] + i // TILE_ROWS                       # global row tile
    lr = i % TILE_ROWS                                 # row inside the tile
    b = np.arange(KB, dtype=np.int64)
    kc, j = b // CHUNK_BLOCKS, b % CHUNK_BLOCKS
    pos = ((kc[None, :] * RT + rt[:, None]) * CHUNK_BYTES
           + ((lr % 32) * 16 + (lr // 32) * 4)[:, None] + j[None, :])
    out[pos.ravel()] = scale.ravel()
    return out


def pack_scales_mma_by_tiles(scale: np.ndarray, seg_rows) -> np.ndarray:
    """Second formulation of ``pack_scales_mma``: each 128-row tile of a
    segment is zero-padded to 128 rows and 4*KC blocks, and each of its chunks
    is the [128, 4] slice viewed as [4 row quarters, 32 lanes, 4 blocks] and
    transposed to lane-major order."""
    scale = np.asarray(scale, dtype=np.uint8)
    R, KB = scale.shape
    m = np.asarray(seg_rows, dtype=np.int64)
    KC = (KB + CHUNK_BLOCKS - 1) // CHUNK_BLOCKS
    tiles = []
    row = 0
    for mg in m:
        for t0 in range(0, int(mg), TILE_ROWS):
            n = min(TILE_ROWS, int(mg) - t0)
            tile = np.zeros((TILE_ROWS, KC * CHUNK_BLOCKS), dtype=np.uint8)
            tile[:n, :KB] = scale[row + t0: row + t0 + n]
            tiles.append(tile)
        row += int(mg)
    RT = len(tiles)
    out = np.zeros((KC, RT, CHUNK_BYTES), dtype=np.uint8)
    for rt, tile in enumerate(tiles):
        for kc in range(KC):
            sl = tile[:, kc * CHUNK_BLOCKS:(kc + 1) * CHUNK_BLOCKS]     # [128 rows, 4 blocks]
            out[kc, rt] = sl.reshape(4, 32, CHUNK_BLOCKS).transpose(1, 0, 2).ravel()
    return out.ravel()


def kseg_chunk_prefix(pad_offsets) -> np.ndarray:
    """[G+1] exclusive prefix of ceil(p_g / 128) for padded segment lengths
    p_g = poff[g+1] - poff[g]: the first k-chunk of each expert; entry G is
    the operand's k-chunk count."""
    poff = np.asarray(pad_offsets, dtype=np.int64)
    chunks = (np.diff(poff) + TILE_ROWS - 1) // TILE_ROWS
    return np.concatenate([[0], np.cumsum(chunks)]).astype(np.int64)


def pack_scales_mma_kseg(scale: np.ndarray, pad_offsets) -> np.ndarray:
    """Scales of a column-wise (k-segmented) operand -> packed bytes.

    The operand has C rows (channels) and a contraction cut into the experts'
    padded segments [poff_g, poff_{g+1}) (multiples of 32); ``scale`` is its
    plain [C, poff_G / 32] byte array.  The chunk grid restarts at every
    segment: expert g's k-chunks are kseg_chunk_prefix[g] + c, c over
    ceil(p_g / 128) chunks of 4 blocks counted from poff_g; rows are cut into
    128-row tiles (RT = ceil(C / 128)).  Chunk (kc, rt) at (kc*RT + rt)*512,
    channel i of the tile and block j of the chunk at (i%32)*16 + (i//32)*4 + j,
    zero where no channel or block exists (the layout the grouped GEMM reads
    for the dgrad weights and both wgrad operands)."""
    scale = np.asarray(scale, dtype=np.uint8)
    C = scale.shape[0]
    poff = np.asarray(pad_offsets, dtype=np.int64)
    kcp = kseg_chunk_prefix(poff)
    RT = (C + TILE_ROWS - 1) // TILE_ROWS
    out = np.zeros(int(kcp[-1] * RT * CHUNK_BYTES), dtype=np.uint8)
    ch = np.arange(C, dtype=np.int64)
    rt, i = ch // TILE_ROWS, ch % TILE_ROWS
    row_off = (i % 32) * 16 + (i // 32) * 4
    for g in range(poff.shape[0] - 1):
        nb = int((poff[g + 1] - poff[g]) // 32)
        for lb in range(nb):                      # local 32-block of the expert
            kc = kcp[g] + lb // CHUNK_BLOCKS
            pos = (kc * RT + rt) * CHUNK_BYTES + row_off + lb % CHUNK_BLOCKS
            out[pos] = scale[:, poff[g] // 32 + lb]
    return out


def pack_scales_mma_kseg_by_experts(scale: np.ndarray, pad_offsets) -> np.ndarray:
    """Second formulation of ``pack_scales_mma_kseg``: each expert's slice
    [C, p_g / 32] is a row-wise operand of one segment of C rows; its packed
    chunk planes (``pack_scales_mma``) are concatenated in expert order."""
    scale = np.asarray(scale, dtype=np.uint8)
    C = scale.shape[0]
    poff = np.asarray(pad_offsets, dtype=np.int64)
    parts = []
    for g in range(poff.shape[0] - 1):
        sl = scale[:, poff[g] // 32: poff[g + 1] // 32]
        if sl.shape[1]:
            parts.append(pack_scales_mma(sl, [C]))
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.uint8)

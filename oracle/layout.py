"""Reference definition of the prepacked ("interleaved pre-tiled") weight blob.

THIS IS TEST INFRASTRUCTURE (see ``oracle/tf_oracle.py``).  It restates the
blob format element by element so that the C++ ``tf_prepack`` can be checked
byte for byte; it shares no code with it.

The TileFuse pages (section "Methodology", item 2 "Interleaved pre-tiling")
fix two properties of the offline layout: (a) the quantisation metadata
(scales and zero points) is packed *into* the weight tiles, so that everything
a tile needs for its dequantisation is contiguous, and (b) the matrix is
reordered so that the tiles one consumer streams are contiguous, which removes
large strides and keeps the layout valid for dimensions up to 32K.  The tile
shape and element order below are this implementation's GB300 design (the
pages' AIE tile shapes are prior art):

Blob = 64-byte header, then ``NB * KT`` tiles of ``tile_bytes`` each; tile
``(nb, kt)`` sits at byte ``64 + (nb * KT + kt) * tile_bytes`` (n-block major:
the K tiles of one 128-row block are contiguous).  ``NB = ceil(N / 128)``,
``KT = ceil(K / 128)``.

Header (little-endian): u32 magic 0x4B504654 ('TFPK'), u32 version 1,
i32 N, i32 K, i32 bits, i32 group (0 = per channel), i32 tile_n 128,
i32 tile_k 128, i32 NB, i32 KT, i32 tile_bytes, i32 groups_per_tile,
u64 total_bytes, 8 zero bytes.

Tile = weights (128 * 128 * bits / 8 bytes), then scales, then zeros.

Weights: 8 row blocks ``mb`` of 16 rows x 2 K-quads ``h`` of 64 columns; block
``(mb, h)`` starts at byte ``(mb * 2 + h) * 32 * P`` with ``P = 16`` (INT4) or
32 (INT8) bytes per slot.  Slot ``p = 4 gr + t`` (``gr`` in 0..7, ``t`` in
0..3: the lane order of an mma.sync fragment) holds four words ``j = 0..3``;
word j holds eight codes ``i = 0..7``: INT4 code i sits at bits ``4 i`` of the
little-endian uint32 at slot byte ``4 j``; INT8 code i is slot byte
``8 j + i``.  With ``r = i & 3`` and
``e = i >> 2``, code i of word j in slot (gr, t) is the weight at tile
row / column::

    row = mb * 16 + gr + 8 * (r & 1)
    col = h * 64 + 16 * t + 4 * j + 2 * (r >> 1) + e

Scales: bf16 ``[gi][mb][gr][e]`` (``256 * GPT`` bytes) = scale of row
``mb*16 + gr + 8e`` in the group of tile column block ``gi``.  Zeros: INT4 one
byte per ``[gi][mb][gr]`` (low nibble row ``gr``, high nibble row ``gr + 8``);
INT8 one byte per ``[gi][mb][gr][e]``.  ``GPT`` (groups per tile) is
``128 / g`` for g in {32, 64}, else 1; column block gi covers tile columns
``[gi * g, (gi + 1) * g)`` (all 128 when GPT = 1, whose group is
``kt * 128 // g``).

Padding: rows >= N have q = z = 0 and s = 0; columns >= K hold q = z of their
group, or q = z = s = 0 where that group lies entirely beyond K.
"""

from __future__ import annotations

import struct

import numpy as np

MAGIC = 0x4B504654
VERSION = 1
HEADER_BYTES = 64
TILE_N = 128
TILE_K = 128
_HDR = "<IIiiiiiiiiiiQ"


def groups_per_tile(group: int) -> int:
    return TILE_K // group if group in (32, 64) else 1


def tile_bytes(bits: int, group: int) -> int:
    gpt = groups_per_tile(group)
    w = TILE_N * TILE_K * bits // 8
    s = 2 * TILE_N * gpt
    z = (TILE_N // 2 if bits == 4 else TILE_N) * gpt
    return (w + s + z + 15) // 16 * 16


def blob_geometry(N: int, K: int, bits: int, group: int):
    nb = -(-N // TILE_N)
    kt = -(-K // TILE_K)
    tb = tile_bytes(bits, group)
    return nb, kt, tb, HEADER_BYTES + nb * kt * tb


def header(N, K, bits, group) -> bytes:
    nb, kt, tb, total = blob_geometry(N, K, bits, group)
    h = struct.pack(_HDR, MAGIC, VERSION, N, K, bits, group, TILE_N, TILE_K,
                    nb, kt, tb, groups_per_tile(group), total)
    return h + bytes(HEADER_BYTES - len(h))


def code_coordinates():
    """Tile (row, col) of every code of a tile, in blob order (mb, h, p, j, i)."""
    mb, h, p, j, i = np.meshgrid(np.arange(8), np.arange(2), np.arange(32), np.arange(4),
                                 np.arange(8), indexing="ij")
    gr = p // 4
    t = p % 4
    r = i & 3
    e = i >> 2
    row = mb * 16 + gr + 8 * (r & 1)
    col = h * 64 + 16 * t + 4 * j + 2 * (r >> 1) + e
    return row.ravel(), col.ravel()


def _meta_rows():
    """Tile rows of the metadata entries, shape [mb][gr][e]."""
    return (np.arange(8)[:, None, None] * 16 + np.arange(8)[None, :, None]
            + 8 * np.arange(2)[None, None, :])


def prepack(qweight, scales_bits, zeros, N, K, bits, group) -> np.ndarray:
    """Build the blob (uint8 array) from natural-order inputs."""
    from oracle.tf_oracle import unpack

    q = unpack(qweight, bits, K)
    g = K if group == 0 else group
    nb, kt, tb, total = blob_geometry(N, K, bits, group)
    gpt = groups_per_tile(group)
    Np, Kp = nb * TILE_N, kt * TILE_K
    n_groups = K // g
    col = np.arange(Kp)
    # group of every padded column (may point past the last group in the K pad)
    gidx = col // g if gpt > 1 else (col // TILE_K * TILE_K) // g
    width = max(n_groups, int(gidx.max()) + 1)
    s_pad = np.zeros((Np, width), dtype=np.uint16)
    z_pad = np.zeros((Np, width), dtype=np.uint8)
    s_pad[:N, :n_groups] = scales_bits
    z_pad[:N, :n_groups] = zeros
    q_pad = np.zeros((Np, Kp), dtype=np.uint8)
    q_pad[:N, :K] = q
    if Kp > K:
        q_pad[:, K:] = z_pad[:, gidx[K:]]

    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = np.frombuffer(header(N, K, bits, group), dtype=np.uint8)
    row, colt = code_coordinates()
    mrows = _meta_rows()
    wbytes = TILE_N * TILE_K * bits // 8
    zb = (TILE_N // 2) if bits == 4 else TILE_N
    for b in range(nb):
        for t in range(kt):
            base = HEADER_BYTES + (b * kt + t) * tb
            codes = q_pad[b * TILE_N + row, t * TILE_K + colt]
            if bits == 4:
                c = codes.reshape(-1, 8).astype(np.uint32)
                words = np.zeros(c.shape[0], dtype=np.uint32)
                for i in range(8):
                    words |= c[:, i] << np.uint32(4 * i)
                out[base:base + wbytes] = words.astype("<u4").view(np.uint8)
            else:
                out[base:base + wbytes] = codes
            sptr = base + wbytes
            zptr = sptr + 256 * gpt
            for gi in range(gpt):
                grp = gidx[t * TILE_K + gi * (g if gpt > 1 else 0)]
                s = s_pad[b * TILE_N + mrows, grp]
                z = z_pad[b * TILE_N + mrows, grp]
                out[sptr + gi * 256: sptr + (gi + 1) * 256] = s.astype("<u2").view(np.uint8).ravel()
                zz = (z[..., 0] | (z[..., 1] << 4)).astype(np.uint8).ravel() if bits == 4 else z.ravel()
                out[zptr + gi * zb: zptr + (gi + 1) * zb] = zz
    return out


def parse_header(blob) -> dict:
    blob = np.asarray(blob, dtype=np.uint8)
    keys = ("magic", "version", "N", "K", "bits", "group", "tile_n", "tile_k", "NB", "KT",
            "tile_bytes", "groups_per_tile", "total_bytes")
    return dict(zip(keys, struct.unpack(_HDR, blob[:56].tobytes())))


def unprepack(blob: np.ndarray):
    """Inverse of :func:`prepack`: (qweight, scales_bits, zeros, N, K, bits, group)."""
    blob = np.asarray(blob, dtype=np.uint8)
    hd = parse_header(blob)
    assert hd["magic"] == MAGIC and hd["version"] == VERSION
    N, K, bits, group = hd["N"], hd["K"], hd["bits"], hd["group"]
    nb, kt, tb, gpt = hd["NB"], hd["KT"], hd["tile_bytes"], hd["groups_per_tile"]
    g = K if group == 0 else group
    n_groups = K // g
    row, colt = code_coordinates()
    mrows = _meta_rows()
    wbytes = TILE_N * TILE_K * bits // 8
    zb = (TILE_N // 2) if bits == 4 else TILE_N
    q = np.zeros((nb * TILE_N, kt * TILE_K), dtype=np.uint8)
    scales = np.zeros((nb * TILE_N, n_groups), dtype=np.uint16)
    zeros = np.zeros((nb * TILE_N, n_groups), dtype=np.uint8)
    for b in range(nb):
        for t in range(kt):
            base = HEADER_BYTES + (b * kt + t) * tb
            if bits == 4:
                words = blob[base:base + wbytes].view("<u4")
                codes = (words[:, None] >> (4 * np.arange(8, dtype=np.uint32))[None, :]) & 0xF
                codes = codes.astype(np.uint8).ravel()
            else:
                codes = blob[base:base + wbytes]
            q[b * TILE_N + row, t * TILE_K + colt] = codes
            sptr = base + wbytes
            zptr = sptr + 256 * gpt
            for gi in range(gpt):
                c0 = t * TILE_K + gi * (g if gpt > 1 else 0)
                if c0 >= K:
                    continue
                grp = c0 // g
                s = blob[sptr + gi * 256: sptr + (gi + 1) * 256].view("<u2").reshape(8, 8, 2)
                zz = blob[zptr + gi * zb: zptr + (gi + 1) * zb]
                z = np.stack([zz & 0xF, zz >> 4], axis=-1).reshape(8, 8, 2) if bits == 4 \
                    else zz.reshape(8, 8, 2)
                scales[b * TILE_N + mrows, grp] = s
                zeros[b * TILE_N + mrows, grp] = z
    q = q[:N, :K]
    if bits == 4:
        qr = q.reshape(N, K // 8, 8).astype(np.uint32)
        qweight = np.zeros((N, K // 8), dtype=np.uint32)
        for i in range(8):
            qweight |= qr[:, :, i] << np.uint32(4 * i)
    else:
        qweight = q
    return qweight, scales[:N], zeros[:N], N, K, bits, group

"""Reference definition of the prepacked ("interleaved pre-tiled") weight blob.

THIS IS TEST INFRASTRUCTURE (see ``oracle/tf_oracle.py``).  It restates the
blob format element by element so that the C++ ``tf_prepack`` can be checked
byte for byte; it shares no code with it.

The TileFuse pages (section "Methodology", item 2 "Interleaved pre-tiling")
fix two properties of the offline layout: (a) the quantisation metadata
(scales and zero points) is packed *into* the weight tiles, so that everything
a tile needs for its dequantisation is contiguous, and (b) the matrix is
reordered so that the tiles one consumer streams are contiguous, which removes
large strides and keeps the layout valid for dimensions up to 32K.  The unit
shape and element order below are this implementation's GB300 design (the
pages' AIE tile shapes are prior art):

Blob = 64-byte header, then ``S * KT`` units of ``unit_bytes`` each.  A unit
covers one 16-row slab of W (rows ``16 s .. 16 s + 15``) and 128 columns of K
(``128 kt .. 128 kt + 127``).  Unit ``(s, kt)`` sits at byte
``64 + (s * KT + kt) * unit_bytes``: slab-major, so all K units of a slab —
and of any run of whole slabs — are contiguous.  ``S = 8 * ceil(N / 128)``
(rows padded to a multiple of 128, so that eight consecutive slabs form a
128-row tile), ``KT = ceil(K / 128)``.

Header (little-endian): u32 magic 0x4B504654 ('TFPK'), u32 version 2,
i32 N, i32 K, i32 bits, i32 group (0 = per channel), i32 unit_n 16,
i32 unit_k 128, i32 S, i32 KT, i32 unit_bytes, i32 groups_per_unit,
u64 total_bytes, 8 zero bytes.

Unit = codes (16 * 128 * bits / 8 bytes), then scales, then zeros, then zero
padding to a multiple of 16 bytes (INT4) or 32 bytes (INT8).

Codes: 2 K-halves ``h`` of 64 columns; half h starts at byte ``h * 32 * P``
with ``P = 16`` (INT4) or 32 (INT8) bytes per slot.  Slot ``p = 4 gr + t``
(``gr`` in 0..7, ``t`` in 0..3: the lane order of an mma.sync fragment) holds
four words ``j = 0..3``; word j holds eight codes ``i = 0..7``: INT4 code i
sits at bits ``4 i`` of the little-endian uint32 at slot byte ``4 j``; INT8
code i is slot byte ``8 j + i``.  With ``r = i & 3`` and ``e = i >> 2``, code
i of word j in slot (gr, t) is the weight at unit row / column::

    row = gr + 8 * (r & 1)
    col = h * 64 + 16 * t + 4 * j + 2 * (r >> 1) + e

Scales: bf16 ``[gi][gr][e]`` (``32 * GPU`` bytes) = scale of unit row
``gr + 8e`` in the group of unit column block ``gi``.  Zeros: INT4 one byte per
``[gi][gr]`` (low nibble row ``gr``, high nibble row ``gr + 8``; 8 bytes per
gi); INT8 one byte per ``[gi][gr][e]`` (16 bytes per gi).  ``GPU`` (groups per
unit) is ``128 / g`` for g in {32, 64}, else 1; column block gi covers unit
columns ``[gi * g, (gi + 1) * g)`` (all 128 when GPU = 1, whose group is
``kt * 128 // g``).

Padding: rows >= N have q = z = 0 and s = 0; columns >= K hold q = z of their
group, or q = z = s = 0 where that group lies entirely beyond K.
"""

from __future__ import annotations

import struct

import numpy as np

MAGIC = 0x4B504654
VERSION = 2
HEADER_BYTES = 64
UNIT_N = 16
UNIT_K = 128
TILE_N = 128  # rows per 128-row block; S = 8 * ceil(N / 128)
_HDR = "<IIiiiiiiiiiiQ"


def groups_per_unit(group: int) -> int:
    return UNIT_K // group if group in (32, 64) else 1


def unit_bytes(bits: int, group: int) -> int:
    gpu = groups_per_unit(group)
    codes = UNIT_N * UNIT_K * bits // 8
    scales = 2 * UNIT_N * gpu
    zeros = (UNIT_N // 2 if bits == 4 else UNIT_N) * gpu
    align = 16 if bits == 4 else 32
    return (codes + scales + zeros + align - 1) // align * align


def blob_geometry(N: int, K: int, bits: int, group: int):
    """(S, KT, unit_bytes, total_bytes)."""
    s = 8 * -(-N // TILE_N)
    kt = -(-K // UNIT_K)
    ub = unit_bytes(bits, group)
    return s, kt, ub, HEADER_BYTES + s * kt * ub


def header(N, K, bits, group) -> bytes:
    s, kt, ub, total = blob_geometry(N, K, bits, group)
    h = struct.pack(_HDR, MAGIC, VERSION, N, K, bits, group, UNIT_N, UNIT_K,
                    s, kt, ub, groups_per_unit(group), total)
    return h + bytes(HEADER_BYTES - len(h))


def code_coordinates():
    """Unit (row, col) of every code of a unit, in blob order (h, p, j, i)."""
    h, p, j, i = np.meshgrid(np.arange(2), np.arange(32), np.arange(4), np.arange(8), indexing="ij")
    gr = p // 4
    t = p % 4
    r = i & 3
    e = i >> 2
    row = gr + 8 * (r & 1)
    col = h * 64 + 16 * t + 4 * j + 2 * (r >> 1) + e
    return row.ravel(), col.ravel()


def _meta_rows():
    """Unit rows of the metadata entries, shape [gr][e]."""
    return np.arange(8)[:, None] + 8 * np.arange(2)[None, :]


def prepack(qweight, scales_bits, zeros, N, K, bits, group) -> np.ndarray:
    """Build the blob (uint8 array) from natural-order inputs."""
    from oracle.tf_oracle import unpack

    q = unpack(qweight, bits, K)
    g = K if group == 0 else group
    S, KT, ub, total = blob_geometry(N, K, bits, group)
    gpu = groups_per_unit(group)
    Np, Kp = S * UNIT_N, KT * UNIT_K
    n_groups = K // g
    col = np.arange(Kp)
    # group of every padded column (may point past the last group in the K pad)
    gidx = col // g if gpu > 1 else (col // UNIT_K * UNIT_K) // g
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
    row, colu = code_coordinates()
    mrows = _meta_rows()
    cbytes = UNIT_N * UNIT_K * bits // 8
    zb = (UNIT_N // 2) if bits == 4 else UNIT_N
    for s in range(S):
        for t in range(KT):
            base = HEADER_BYTES + (s * KT + t) * ub
            codes = q_pad[s * UNIT_N + row, t * UNIT_K + colu]
            if bits == 4:
                c = codes.reshape(-1, 8).astype(np.uint32)
                words = np.zeros(c.shape[0], dtype=np.uint32)
                for i in range(8):
                    words |= c[:, i] << np.uint32(4 * i)
                out[base:base + cbytes] = words.astype("<u4").view(np.uint8)
            else:
                out[base:base + cbytes] = codes
            sptr = base + cbytes
            zptr = sptr + 32 * gpu
            for gi in range(gpu):
                grp = gidx[t * UNIT_K + gi * (g if gpu > 1 else 0)]
                sv = s_pad[s * UNIT_N + mrows, grp]
                zv = z_pad[s * UNIT_N + mrows, grp]
                out[sptr + gi * 32: sptr + (gi + 1) * 32] = sv.astype("<u2").view(np.uint8).ravel()
                zz = (zv[:, 0] | (zv[:, 1] << 4)).astype(np.uint8) if bits == 4 else zv.ravel()
                out[zptr + gi * zb: zptr + (gi + 1) * zb] = zz
    return out


def parse_header(blob) -> dict:
    blob = np.asarray(blob, dtype=np.uint8)
    keys = ("magic", "version", "N", "K", "bits", "group", "unit_n", "unit_k", "S", "KT",
            "unit_bytes", "groups_per_unit", "total_bytes")
    return dict(zip(keys, struct.unpack(_HDR, blob[:56].tobytes())))


def unprepack(blob: np.ndarray):
    """Inverse of :func:`prepack`: (qweight, scales_bits, zeros, N, K, bits, group)."""
    blob = np.asarray(blob, dtype=np.uint8)
    hd = parse_header(blob)
    assert hd["magic"] == MAGIC and hd["version"] == VERSION
    N, K, bits, group = hd["N"], hd["K"], hd["bits"], hd["group"]
    S, KT, ub, gpu = hd["S"], hd["KT"], hd["unit_bytes"], hd["groups_per_unit"]
    g = K if group == 0 else group
    n_groups = K // g
    row, colu = code_coordinates()
    mrows = _meta_rows()
    cbytes = UNIT_N * UNIT_K * bits // 8
    zb = (UNIT_N // 2) if bits == 4 else UNIT_N
    q = np.zeros((S * UNIT_N, KT * UNIT_K), dtype=np.uint8)
    scales = np.zeros((S * UNIT_N, n_groups), dtype=np.uint16)
    zeros = np.zeros((S * UNIT_N, n_groups), dtype=np.uint8)
    for s in range(S):
        for t in range(KT):
            base = HEADER_BYTES + (s * KT + t) * ub
            if bits == 4:
                words = blob[base:base + cbytes].view("<u4")
                codes = (words[:, None] >> (4 * np.arange(8, dtype=np.uint32))[None, :]) & 0xF
                codes = codes.astype(np.uint8).ravel()
            else:
                codes = blob[base:base + cbytes]
            q[s * UNIT_N + row, t * UNIT_K + colu] = codes
            sptr = base + cbytes
            zptr = sptr + 32 * gpu
            for gi in range(gpu):
                c0 = t * UNIT_K + gi * (g if gpu > 1 else 0)
                if c0 >= K:
                    continue
                grp = c0 // g
                sv = blob[sptr + gi * 32: sptr + (gi + 1) * 32].view("<u2").reshape(8, 2)
                zz = blob[zptr + gi * zb: zptr + (gi + 1) * zb]
                zv = np.stack([zz & 0xF, zz >> 4], axis=-1) if bits == 4 else zz.reshape(8, 2)
                scales[s * UNIT_N + mrows, grp] = sv
                zeros[s * UNIT_N + mrows, grp] = zv
    q = q[:N, :K]
    if bits == 4:
        K8 = (K + 7) // 8 * 8  # the last word's unused nibbles are zero
        qr = np.zeros((N, K8), dtype=np.uint32)
        qr[:, :K] = q
        qr = qr.reshape(N, K8 // 8, 8)
        qweight = np.zeros((N, K8 // 8), dtype=np.uint32)
        for i in range(8):
            qweight |= qr[:, :, i] << np.uint32(4 * i)
    else:
        qweight = q
    return qweight, scales[:N], zeros[:N], N, K, bits, group

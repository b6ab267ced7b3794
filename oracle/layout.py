"""Byte layout of the packed cache, restated for the oracle.

TEST INFRASTRUCTURE (see ckv_oracle.py). The layout is this library's own
storage format; the pages fix only what is stored (int8 q8_0 codes with fp16
block scales for K, 3-bit codes with one fp16 norm for V), not where. It is
written here from its definition, independently of the CUDA packer, so that
the packer's bytes can be compared with the oracle's.

Definition. Each (sequence, kv-head) owns T_cap / 16 tile records; tile t covers
token positions [16 t, 16 t + 16). With b bits per V code (b = 2, 3 or 4; 3 is
the method's TBQ3) a record is 17 D + 2 b D + 32 bytes (D = head_dim; 23 D + 32
at b = 3):

  [0, 16D)      K codes, each stored as the byte q + 128 (offset binary; q in
                [-127, 127]). Element (p, i) (p = position in tile, i = dim) sits at
                ((i // 32) * 32 + L) * 16 + (p // 8) * 8 + (i % 8),
                with lane L = 4 * (p % 8) + (i % 32) // 8.
  [16D, 17D)    K scales, fp16, [16][D/32] row-major: (p, block) at 16D + 2 (p D/32 + block).
  [17D, 17D + 2bD)  V codes, b bits each. Lane L owns a stream of b D/16 bytes. With
                G = D/8, g = i // G, u = i % G, L = 4 g + (p % 8) // 2 and
                pair index pi = 4 (u // 2) + (u % 2) + 2 (p // 8), the code of (p, i)
                occupies stream bits [2b pi + b (p % 2), 2b pi + b (p % 2) + b), least
                significant bit first (stream bit x is bit x % 8 of stream byte x // 8).
                Stream byte s of lane L is stored at 17D + ((s // gr) * 32 + L) * gr + s % gr,
                gr = 16, 8 or 4: the largest of those dividing b D/16.
  [17D + 2bD, +32)  V norms, fp16, one per position: p at 17D + 2bD + 2 p.
                With the block-diagonal rotation (one norm per 128-dim group, G' =
                D / 128 groups) the norm region is 32 G' bytes, group-major: norm
                (p, j) at 17D + 2bD + 2 (16 j + p).
"""
from __future__ import annotations

import numpy as np

TILE = 16


def record_bytes(D: int, bits: int = 3, groups: int = 1) -> int:
    """Bytes of one 16-position record: ``groups`` fp16 V norms per position (1
    for the full transform, D / 128 for the block-diagonal variant)."""
    return 17 * D + 2 * bits * D + 32 * groups


def _granule(D: int, bits: int = 3) -> int:
    per_lane = bits * D // 16
    for gr in (16, 8, 4):
        if per_lane % gr == 0:
            return gr
    raise ValueError("unsupported head_dim")


def k_code_offsets(D: int) -> np.ndarray:
    """[16, D] byte offset of each K code inside a record."""
    p = np.arange(TILE)[:, None]
    i = np.arange(D)[None, :]
    lane = 4 * (p % 8) + (i % 32) // 8
    return ((i // 32) * 32 + lane) * 16 + (p // 8) * 8 + (i % 8)


def k_scale_offsets(D: int) -> np.ndarray:
    """[16, D/32] byte offset of each fp16 K scale inside a record."""
    p = np.arange(TILE)[:, None]
    b = np.arange(D // 32)[None, :]
    return 16 * D + 2 * (p * (D // 32) + b)


def v_code_bits(D: int, bits: int = 3) -> np.ndarray:
    """[16, D, bits] absolute bit index (byte * 8 + bit) of each V code bit inside a record."""
    G = D // 8
    gr = _granule(D, bits)
    p = np.arange(TILE)[:, None]
    i = np.arange(D)[None, :]
    g, u = i // G, i % G
    lane = 4 * g + (p % 8) // 2
    pair = 4 * (u // 2) + (u % 2) + 2 * (p // 8)
    first = 2 * bits * pair + bits * (p % 2)
    sbit = first[..., None] + np.arange(bits)[None, None, :]
    stream_byte = sbit // 8
    byte = 17 * D + ((stream_byte // gr) * 32 + lane[..., None]) * gr + stream_byte % gr
    return byte * 8 + sbit % 8


def v_norm_offsets(D: int, bits: int = 3, groups: int = 1) -> np.ndarray:
    """Byte offset of the norm of position p (and group j): group-major,
    17 D + 2 b D + 2 (16 j + p). Shape [16] for one group, else [16, groups]."""
    p = np.arange(TILE)
    if groups == 1:
        return 17 * D + 2 * bits * D + 2 * p
    j = np.arange(groups)
    return 17 * D + 2 * bits * D + 2 * (TILE * j[None, :] + p[:, None])


def pack_records(qs, d16, codes, n16, capacity: int, bits: int = 3, groups: int = 1) -> np.ndarray:
    """Lay out one (sequence, kv-head) stream of T tokens as capacity/16 records.

    ``qs int8 [T, D]``, ``d16 fp16 [T, D/32]``, ``codes uint8 [T, D]`` (0..2^bits - 1),
    ``n16 fp16 [T]`` (``[T, groups]`` for several norm groups). Positions >= T
    are left zero. Returns uint8 ``[capacity/16, record_bytes(D, bits, groups)]``.
    """
    qs = np.asarray(qs, dtype=np.int8)
    T, D = qs.shape
    if capacity % TILE or T > capacity:
        raise ValueError("capacity must be a multiple of 16 and hold every token")
    n_tiles = capacity // TILE
    out = np.zeros((n_tiles, record_bytes(D, bits, groups)), dtype=np.uint8)
    kofs, sofs = k_code_offsets(D), k_scale_offsets(D)
    vbits, nofs = v_code_bits(D, bits), v_norm_offsets(D, bits, groups).reshape(TILE, groups)
    qs_u8 = qs.view(np.uint8) ^ np.uint8(0x80)
    d16_u8 = np.asarray(d16, dtype=np.float16).view(np.uint8).reshape(T, D // 32, 2)
    n16_u8 = np.asarray(n16, dtype=np.float16).view(np.uint8).reshape(T, groups, 2)
    codes = np.asarray(codes, dtype=np.uint8)
    for t in range(T):
        tile, p = divmod(t, TILE)
        rec = out[tile]
        rec[kofs[p]] = qs_u8[t]
        rec[sofs[p]] = d16_u8[t, :, 0]
        rec[sofs[p] + 1] = d16_u8[t, :, 1]
        rec[nofs[p]] = n16_u8[t, :, 0]
        rec[nofs[p] + 1] = n16_u8[t, :, 1]
        for k in range(bits):
            bit = vbits[p, :, k]
            val = (codes[t] >> k) & 1
            np.bitwise_or.at(rec, bit // 8, (val << (bit % 8)).astype(np.uint8))
    return out


def unpack_records(records, T: int, D: int, bits: int = 3, groups: int = 1):
    """Inverse of :func:`pack_records` for the first T positions."""
    records = np.asarray(records, dtype=np.uint8)
    kofs, sofs = k_code_offsets(D), k_scale_offsets(D)
    vbits, nofs = v_code_bits(D, bits), v_norm_offsets(D, bits, groups).reshape(TILE, groups)
    qs = np.zeros((T, D), dtype=np.int8)
    d16 = np.zeros((T, D // 32), dtype=np.float16)
    codes = np.zeros((T, D), dtype=np.uint8)
    n16 = np.zeros((T, groups), dtype=np.float16)
    for t in range(T):
        tile, p = divmod(t, TILE)
        rec = records[tile]
        qs[t] = (rec[kofs[p]] ^ np.uint8(0x80)).view(np.int8)
        d16[t] = (rec[sofs[p]].astype(np.uint16) | (rec[sofs[p] + 1].astype(np.uint16) << 8)).view(np.float16)
        n16[t] = (rec[nofs[p]].astype(np.uint16) | (rec[nofs[p] + 1].astype(np.uint16) << 8)).view(np.float16)
        c = np.zeros(D, dtype=np.uint8)
        for k in range(bits):
            bit = vbits[p, :, k]
            c |= (((rec[bit // 8] >> (bit % 8)) & 1) << k).astype(np.uint8)
        codes[t] = c
    return qs, d16, codes, (n16[:, 0] if groups == 1 else n16)

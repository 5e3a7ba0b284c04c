"""Q8_0 block format, quantiser and dequantiser (oracle; test infrastructure).

Source: "Core Architecture & The 4-Brick Pipeline", §5 part 2 "Dynamic Q8_0 KV
Cache Compression": keys and values are quantised to symmetric 8-bit blocks;
each block of 32 values costs 32 one-byte codes plus one two-byte fp16 scale,
34 bytes in all (against 64 bytes in fp16, a 46.88 % reduction).

Readings where the page is silent (each listed in the design notes):
  * scale: d = amax / 127 computed in IEEE fp32 (amax = max |x| over the 32
    values of the block), then rounded to fp16 with round-to-nearest-even;
    the fp16 value is what the block stores.
  * codes: q = round(x / d16) with x / d16 an IEEE fp32 division by the
    *stored* fp16 scale, rounded half away from zero, clamped to [-127, 127].
    Dividing by the stored scale makes the round trip |x - d16*q| <= d16/2
    hold against the bytes actually kept.
  * amax == 0 (or a scale that underflows to fp16 zero): d16 = +0, all codes 0.
  * byte layout of one block: fp16 d (little-endian) at offset 0, then the
    32 int8 codes at offsets 2..33.  A head row of 64 values is two blocks,
    68 bytes: channels 0..31 then 32..63.  A wider head row is quantised the
    same way, one block per 32 channels in channel order (head_dim 128: four
    blocks, 136 bytes).
"""

import numpy as np

BLOCK_VALUES = 32          # values per Q8_0 block
BLOCK_BYTES = 34           # 2-byte fp16 scale + 32 int8 codes
ROW_BYTES = 2 * BLOCK_BYTES  # one 64-channel head row = two blocks


def quantize_blocks(x):
    """Quantise fp32 values, grouped in blocks of 32 along the last axis.

    x: float32 array [..., 32*nb].  Returns (d16, q): d16 float16 [..., nb],
    q int8 [..., nb, 32].  Every step is IEEE fp32 (numpy float32 arithmetic),
    so the bytes are uniquely defined.
    """
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % BLOCK_VALUES:
        raise ValueError("last axis must be a multiple of 32")
    xb = x.reshape(*x.shape[:-1], x.shape[-1] // BLOCK_VALUES, BLOCK_VALUES)
    amax = np.max(np.abs(xb), axis=-1)                       # fp32, exact
    d32 = amax / np.float32(127.0)                           # IEEE fp32 division
    d16 = d32.astype(np.float16)                             # round to nearest even
    dd = d16.astype(np.float32)[..., None]                   # the stored scale, exact in fp32
    nz = dd > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(nz, xb / np.where(nz, dd, np.float32(1.0)), np.float32(0.0))  # fp32 quotient
    # round half away from zero; done in fp64 where |r| + 0.5 is exact
    r64 = r.astype(np.float64)
    qf = np.sign(r64) * np.floor(np.abs(r64) + 0.5)
    q = np.clip(qf, -127, 127).astype(np.int8)
    return d16, q


def dequantize_blocks(d16, q):
    """Exact dequantisation d16 * q, in fp64.  Returns [..., nb*32]."""
    v = d16.astype(np.float64)[..., None] * q.astype(np.float64)
    return v.reshape(*v.shape[:-2], v.shape[-2] * v.shape[-1])


def pack_rows(d16, q):
    """Serialise blocks to bytes: [..., nb] scales + [..., nb, 32] codes ->
    uint8 [..., nb*34], each block = fp16 d (little-endian) then 32 codes."""
    lead = d16.shape
    out = np.empty(lead + (BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = d16.astype("<f2").view(np.uint8).reshape(lead + (2,))
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(*lead[:-1], lead[-1] * BLOCK_BYTES)


def unpack_rows(raw, nb=2):
    """Inverse of pack_rows: uint8 [..., nb*34] -> (d16 [..., nb], q [..., nb, 32])."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    blk = raw.reshape(*raw.shape[:-1], nb, BLOCK_BYTES)
    d16 = np.ascontiguousarray(blk[..., 0:2]).view("<f2").reshape(blk.shape[:-1]).astype(np.float16)
    q = np.ascontiguousarray(blk[..., 2:]).view(np.int8)
    return d16, q


def quantize_kv(x):
    """Quantise a K or V tensor as the GPU path stores it.

    x: float32 [B, M, H, D] (token-major, as a projection emits it), D a
    multiple of 32 (64 for the GPU path).
    Returns uint8 [B, H, M, D/32*34]: head-major planes of rows of D/32 blocks
    (68 bytes at D = 64).
    """
    x = np.asarray(x, dtype=np.float32)
    B, M, H, D = x.shape
    if D % BLOCK_VALUES or D == 0:
        raise ValueError("head_dim must be a positive multiple of 32")
    d16, q = quantize_blocks(x)                 # [B,M,H,D/32], [B,M,H,D/32,32]
    rows = pack_rows(d16, q)                    # [B,M,H,D/32*34]
    return np.ascontiguousarray(rows.transpose(0, 2, 1, 3))


def dequantize_kv(raw):
    """uint8 [..., nb*34] rows -> fp64 [..., nb*32] exact dequantised values
    (nb = 2 for the 68-byte rows of head_dim 64)."""
    if raw.shape[-1] % BLOCK_BYTES:
        raise ValueError("row length must be a multiple of 34 bytes")
    d16, q = unpack_rows(raw, nb=raw.shape[-1] // BLOCK_BYTES)
    return dequantize_blocks(d16, q)


def kv_cache_bytes(layers, heads, tokens, head_dim):
    """Bytes of a Q8_0 K+V cache: 2 tensors x layers x heads x tokens x
    (head_dim/32 blocks x 34 bytes)  ("Out-of-Core Flash Streaming ...", §1)."""
    if head_dim % BLOCK_VALUES:
        raise ValueError("head_dim must be a multiple of 32")
    return 2 * layers * heads * tokens * (head_dim // BLOCK_VALUES) * BLOCK_BYTES


def fp16_kv_cache_bytes(layers, heads, tokens, head_dim):
    """Bytes of the same cache held in fp16: 2 x layers x heads x tokens x head_dim x 2."""
    return 2 * layers * heads * tokens * head_dim * 2

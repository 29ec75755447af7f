"""Dequantization of packed block-scaled tensors to BF16 (oracle; test infrastructure only).

Rule (the backward's "dequantize to BF16" step):
    out = bf16_round( bf16(value) * bf16_round(scale) )
with the product taken exactly (float64 holds it: a code value has at most 4
significant bits and a BF16 scale at most 8) and rounded once, to nearest even.

  * FP8 E4M3 with 128x128 float32 ``scale_inv`` blocks: transformers PR #50031,
    `_dequantize_fp8_weight` -- the scale grid is cast to the gradient dtype,
    repeated 128x along both axes, cropped to the weight's shape, and multiplied
    into the weight cast to that dtype.
  * FP8 E4M3 with one float32 ``scale_inv`` per tensor: the same function's
    `block_size is None` branch -- the scale, cast to the gradient dtype, is
    broadcast over the weight without repetition; for a grouped weight [E, N, K]
    there is one scale per expert.
  * FP8 E5M2 with one float32 quantization step per tensor: the gradient of AstrAI
    fp8.py's "hybrid" backward (quantize.py), dequantized by the same rule.
  * MXFP4 (E2M1 codes, two per byte, one E8M0 scale per 32 consecutive elements
    of a row) and NVFP4 (E2M1 codes, one E4M3 scale per 16 consecutive elements
    of a row, one float32 scale per tensor): MSLK PR #393, "Implementation
    Method" ("dequantizes saved packed FP4 inputs to BF16").

Readings taken where the pages say nothing:
  * byte j of a packed FP4 row holds element 2j in bits 0-3 and element 2j+1 in
    bits 4-7;
  * scale arrays are plain row-major, one row of scales per row of data;
  * NVFP4's two scales combine as one float32 product (E4M3 block value times
    the float32 tensor scale, rounded to float32), which is then cast to BF16.

Shapes: every tensor is [batch, rows, cols] with cols the contiguous axis.
"""

import numpy as np

from .formats import (E2M1_TABLE, E4M3_TABLE, E5M2_TABLE, E8M0_TABLE, bf16_bits, bf16_round,
                      fp32_round)

FMT_BF16 = "bf16"
FMT_FP8 = "fp8_e4m3_b128"
FMT_FP8_TENSOR = "fp8_e4m3_tensor"
FMT_E5M2_TENSOR = "fp8_e5m2_tensor"
FMT_MXFP4 = "mxfp4"
FMT_NVFP4 = "nvfp4"

FP8_BLOCK = 128
MX_BLOCK = 32
NV_BLOCK = 16


def unpack_fp4(packed, cols):
    """uint8 [..., cols/2] -> E2M1 codes uint8 [..., cols]; low nibble is the even element."""
    packed = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(packed.shape[:-1] + (cols,), dtype=np.uint8)
    codes[..., 0::2] = packed & 0x0F
    codes[..., 1::2] = packed >> 4
    return codes


def scale_values(fmt, scale, tensor_scale, batch, rows, cols):
    """Per-element scale (float64, before the BF16 cast) as a [batch, rows, cols] array."""
    if fmt == FMT_FP8:
        s = np.asarray(scale, dtype=np.float32).astype(np.float64)
        s = s.reshape(batch, -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK))
        ri = np.arange(rows) // FP8_BLOCK
        ci = np.arange(cols) // FP8_BLOCK
        return s[:, ri][:, :, ci]
    if fmt in (FMT_FP8_TENSOR, FMT_E5M2_TENSOR):
        s = np.asarray(scale, dtype=np.float32).astype(np.float64).reshape(batch, 1, 1)
        return np.broadcast_to(s, (batch, rows, cols))
    if fmt == FMT_MXFP4:
        b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // MX_BLOCK)
        s = E8M0_TABLE[b]
        return s[:, :, np.arange(cols) // MX_BLOCK]
    if fmt == FMT_NVFP4:
        b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // NV_BLOCK)
        ts = np.asarray(tensor_scale, dtype=np.float32).astype(np.float64).reshape(batch, 1, 1)
        s = fp32_round(E4M3_TABLE[b] * ts)  # one float32 product per block
        return s[:, :, np.arange(cols) // NV_BLOCK]
    raise ValueError(f"no scales for format {fmt!r}")


def code_values(fmt, data, batch, rows, cols):
    """Exact values of the stored codes, float64 [batch, rows, cols]."""
    if fmt == FMT_BF16:
        bits = np.asarray(data, dtype=np.uint16).reshape(batch, rows, cols)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if fmt in (FMT_FP8, FMT_FP8_TENSOR):
        return E4M3_TABLE[np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)]
    if fmt == FMT_E5M2_TENSOR:
        return E5M2_TABLE[np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)]
    if fmt in (FMT_MXFP4, FMT_NVFP4):
        packed = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols // 2)
        return E2M1_TABLE[unpack_fp4(packed, cols)]
    raise ValueError(f"unknown format {fmt!r}")


def dequant_values(fmt, data, scale=None, tensor_scale=None, batch=1, rows=None, cols=None):
    """Dequantized tensor as float64 values that are exactly BF16 values."""
    v = code_values(fmt, data, batch, rows, cols)
    if fmt == FMT_BF16:
        return v
    s_bf = bf16_round(scale_values(fmt, scale, tensor_scale, batch, rows, cols))
    v_bf = bf16_round(v)  # exact for every E4M3, E5M2 and E2M1 value
    return bf16_round(v_bf * s_bf)


def dequant_bits(fmt, data, scale=None, tensor_scale=None, batch=1, rows=None, cols=None):
    """Dequantized tensor as BF16 bit patterns (uint16), NaNs canonical."""
    return bf16_bits(dequant_values(fmt, data, scale, tensor_scale, batch, rows, cols))


def dequant_cols(fmt, data, scale, tensor_scale, rows, cols, col_idx, batch_idx=0, batch=1):
    """Dequantize only the columns ``col_idx`` of one batch entry: float64 [rows, len(col_idx)].

    Used to check sampled outputs of full-size problems without decoding the
    whole tensor; it applies exactly the rule of :func:`dequant_values`.
    """
    col_idx = np.asarray(col_idx)
    if fmt == FMT_BF16:
        bits = np.asarray(data, dtype=np.uint16).reshape(batch, rows, cols)[batch_idx][:, col_idx]
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if fmt == FMT_FP8:
        codes = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)[batch_idx][:, col_idx]
        v = E4M3_TABLE[codes]
        s = np.asarray(scale, dtype=np.float32).astype(np.float64)
        s = s.reshape(batch, -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK))[batch_idx]
        s = s[np.arange(rows) // FP8_BLOCK][:, col_idx // FP8_BLOCK]
    elif fmt in (FMT_FP8_TENSOR, FMT_E5M2_TENSOR):
        codes = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)[batch_idx][:, col_idx]
        v = (E4M3_TABLE if fmt == FMT_FP8_TENSOR else E5M2_TABLE)[codes]
        s = float(np.asarray(scale, dtype=np.float32).reshape(batch)[batch_idx])
    elif fmt in (FMT_MXFP4, FMT_NVFP4):
        packed = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols // 2)[batch_idx]
        byte = packed[:, col_idx // 2]
        codes = np.where(col_idx % 2 == 0, byte & 0x0F, byte >> 4).astype(np.uint8)
        v = E2M1_TABLE[codes]
        if fmt == FMT_MXFP4:
            b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // MX_BLOCK)[batch_idx]
            s = E8M0_TABLE[b[:, col_idx // MX_BLOCK]]
        else:
            b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // NV_BLOCK)[batch_idx]
            ts = float(np.asarray(tensor_scale, dtype=np.float32).reshape(batch)[batch_idx])
            s = fp32_round(E4M3_TABLE[b[:, col_idx // NV_BLOCK]] * ts)
    else:
        raise ValueError(f"unknown format {fmt!r}")
    return bf16_round(bf16_round(v) * bf16_round(s))


def dequant_rows(fmt, data, scale, tensor_scale, rows, cols, row_idx, batch_idx=0, batch=1):
    """Dequantize only the rows ``row_idx`` of one batch entry: float64 [len(row_idx), cols]."""
    row_idx = np.asarray(row_idx)
    if fmt == FMT_BF16:
        bits = np.asarray(data, dtype=np.uint16).reshape(batch, rows, cols)[batch_idx][row_idx]
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if fmt == FMT_FP8:
        codes = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)[batch_idx][row_idx]
        v = E4M3_TABLE[codes]
        s = np.asarray(scale, dtype=np.float32).astype(np.float64)
        s = s.reshape(batch, -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK))[batch_idx]
        s = s[row_idx // FP8_BLOCK][:, np.arange(cols) // FP8_BLOCK]
    elif fmt in (FMT_FP8_TENSOR, FMT_E5M2_TENSOR):
        codes = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols)[batch_idx][row_idx]
        v = (E4M3_TABLE if fmt == FMT_FP8_TENSOR else E5M2_TABLE)[codes]
        s = float(np.asarray(scale, dtype=np.float32).reshape(batch)[batch_idx])
    elif fmt in (FMT_MXFP4, FMT_NVFP4):
        packed = np.asarray(data, dtype=np.uint8).reshape(batch, rows, cols // 2)[batch_idx][row_idx]
        v = E2M1_TABLE[unpack_fp4(packed, cols)]
        if fmt == FMT_MXFP4:
            b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // MX_BLOCK)[batch_idx][row_idx]
            s = E8M0_TABLE[b][:, np.arange(cols) // MX_BLOCK]
        else:
            b = np.asarray(scale, dtype=np.uint8).reshape(batch, rows, cols // NV_BLOCK)[batch_idx][row_idx]
            ts = float(np.asarray(tensor_scale, dtype=np.float32).reshape(batch)[batch_idx])
            s = fp32_round(E4M3_TABLE[b] * ts)[:, np.arange(cols) // NV_BLOCK]
    else:
        raise ValueError(f"unknown format {fmt!r}")
    return bf16_round(bf16_round(v) * bf16_round(s))

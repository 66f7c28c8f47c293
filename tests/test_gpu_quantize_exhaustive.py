"""Exhaustive E2M1 encoder parity: every finite fp32 value x with |x| <= 6.

In a 16-channel block whose absolute maximum is exactly 6 the E4M3 scale is
E4M3(6 / 6) = 1 and x / scale = x, so the block's codes are the E2M1 codes of
its values themselves.  Each block here holds one 6.0 and fifteen consecutive
fp32 bit patterns; the sweep walks every pattern from +0 to 6.0 and from -0
to -6.0 (2,172,649,474 values) through the CUDA quantiser and compares the
packed bytes with the oracle's, chunk by chunk.  A second sweep covers the
scale's own rounding and the saturation of x / scale at 6: a block holding
only x (every 256th fp32 pattern from 6 to 2,688 = 6 x 448) and zeros.
The encoder is a threshold ladder on the GPU and a nearest-value search in the
oracle, so a wrong comparison at any midpoint of the grid fails here.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SIX = 0x40C00000          # 6.0f
CHUNK = 15 * (1 << 22)    # values per chunk: whole blocks of fifteen


def _check_rows(cuda, orc, x):
    """x: [n, 512] fp32; the CUDA FP4 main-KV rows equal the oracle's."""
    n = x.shape[0]
    cache = cuda.Cache.contiguous(cuda.FMT_FP4_KV, 1, n)
    cuda.csa2_quantize_kv(torch.from_numpy(x)[None].cuda(), cache)
    got = cache.data.cpu().numpy().reshape(n, 288)
    qc, qs = orc.quant_fp4(x)
    want = orc.kv_rows(qc, qs)
    bad = np.argwhere(got != want)
    if bad.size:
        r, byte = bad[0]
        blk = byte // 8 if byte < 256 else byte - 256
        raise AssertionError(f"row {r} byte {byte}: got {got[r, byte]:#x}, oracle {want[r, byte]:#x}; "
                             f"block values {x[r, 16 * blk:16 * blk + 16].tolist()}")


def _blocks_to_rows(blocks):
    nb = blocks.shape[0]
    pad = (-nb) % 32
    if pad:
        blocks = np.concatenate([blocks, np.zeros((pad, 16), np.float32)])
    return np.ascontiguousarray(blocks.reshape(-1, 512))


def test_every_fp32_up_to_six_in_unit_scale_blocks(cuda, orc):
    orc.set_threads(os.cpu_count() or 1)
    try:
        for sign in (0, 0x80000000):
            for start in range(0, SIX + 1, CHUNK):
                n = min(CHUNK, SIX + 1 - start)
                vals = (np.arange(start, start + n, dtype=np.uint32) | np.uint32(sign)).view(np.float32)
                nb = (n + 14) // 15
                blocks = np.zeros((nb, 16), np.float32)
                blocks[:, 0] = -6.0 if sign else 6.0
                body = blocks[:, 1:].reshape(-1)
                body[:n] = vals
                blocks[:, 1:] = body.reshape(nb, 15)
                _check_rows(cuda, orc, _blocks_to_rows(blocks))
    finally:
        orc.set_threads(1)


def test_scale_rounding_and_saturation_range(cuda, orc):
    hi = np.float32(6.0 * 448.0).view(np.uint32)
    bits = np.arange(SIX, int(hi) + 1, 256, dtype=np.uint32)
    for sign in (0, 0x80000000):
        vals = (bits | np.uint32(sign)).view(np.float32)
        blocks = np.zeros((vals.size, 16), np.float32)
        blocks[:, 3] = vals
        blocks[::2, 9] = vals[::2] * np.float32(0.75)   # a second, smaller value in half the blocks
        _check_rows(cuda, orc, _blocks_to_rows(blocks))

"""Small numpy helpers shared by the tests (dequantisation with numpy bit operations, tensor transfers)."""
import numpy as np


def deq_w(codes, scales, cols):
    """2-bit rows [rows][cols/4] + fp16 scales [rows][cols/32] -> float64 d * (q - 2)."""
    rows = codes.shape[0]
    q = np.stack([(codes >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(rows, cols).astype(np.float64)
    d = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)
    return d * (q - 2.0)


def deq_a(codes, scales):
    """q8 rows [rows][cols] + fp16 scales [rows][cols/32] -> float64 d * q."""
    return codes.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)


def i16(a):
    return np.ascontiguousarray(a).view(np.int16)


def to_slices(codes, scales):
    """q8 rows in the expert products' slice form: per row and per 64 values, the 64 codes, the two fp16 scales of
    the slice's 32-value blocks (little-endian), 12 zero bytes -> uint8 [rows][cols/64][80]."""
    rows, cols = codes.shape
    out = np.zeros((rows, cols // 64, 80), np.uint8)
    out[:, :, :64] = np.ascontiguousarray(codes).view(np.uint8).reshape(rows, cols // 64, 64)
    out[:, :, 64:68] = np.ascontiguousarray(scales).view(np.uint8).reshape(rows, cols // 64, 4)
    return out


def packed_q2(codes, scales):
    """Row-major Q2 matrices [E][rows][cols/4] + [E][rows][cols/32] -> the packed block sequence (uint8)."""
    E, rows, c4 = codes.shape
    cols = c4 * 4
    sc = np.ascontiguousarray(scales).view(np.uint8).reshape(E, rows, cols // 16)
    blocks = []
    for e in range(E):
        for mt in range(rows // 128):
            for kt in range(cols // 64):
                blocks.append(codes[e, mt * 128:(mt + 1) * 128, kt * 16:(kt + 1) * 16].ravel())
                blocks.append(sc[e, mt * 128:(mt + 1) * 128, kt * 4:(kt + 1) * 4].ravel())
    return np.concatenate(blocks)

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


def to_operand(codes, scales):
    """q8 rows [rows][cols] + fp16 scales [rows][cols/32] in the expert products' operand form: hi = fp16(d q),
    lo = d q - hi (both exact from float64), and within each group of 16 values position 2j holds value j and 2j+1
    value j+8 -> float16 [2][rows][cols]."""
    rows, cols = codes.shape
    v = np.asarray(codes).astype(np.float64) * np.repeat(np.asarray(scales).view(np.float16).astype(np.float64), 32,
                                                         axis=1)
    hi = v.astype(np.float16)
    lo = (v - hi.astype(np.float64)).astype(np.float16)
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), v), "the hi/lo split must be exact"
    perm = lambda a: np.ascontiguousarray(a.reshape(rows, cols // 16, 2, 8).transpose(0, 1, 3, 2)).reshape(rows, cols)
    return np.stack([perm(hi), perm(lo)])


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

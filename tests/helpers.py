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

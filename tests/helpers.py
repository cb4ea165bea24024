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


def tile_list(offsets, max_rows):
    """A tile list for the expert products built from grouping offsets (a test input, not an expected value): each
    expert's c rows split into ceil(c / max_rows) near-equal contiguous tiles, experts in id order -> int32 [nt][4]
    rows {expert, first row, rows, 0}."""
    out = []
    for e in range(len(offsets) - 1):
        r0, c = int(offsets[e]), int(offsets[e + 1] - offsets[e])
        nt = -(-c // max_rows)
        for i in range(nt):
            a, b = i * c // nt, (i + 1) * c // nt
            out.append((e, r0 + a, b - a, 0))
    return np.array(out, np.int32).reshape(-1, 4)


def check_tile_list(tiles, offsets, max_rows, max_tiles):
    """What any valid tile list over a grouping must satisfy: every tile lies inside one expert's rows and holds
    1..max_rows of them, tiles come in expert order and walk each expert's rows contiguously, every routed row is in
    exactly one tile, and no expert uses more than ceil(c / max_rows) tiles (so the count never exceeds
    max_tiles)."""
    tiles = np.asarray(tiles).reshape(-1, 4)
    E = len(offsets) - 1
    n = int(offsets[-1])
    assert len(tiles) <= max_tiles
    covered = np.zeros(n, np.int32)
    e_prev, next_row = -1, 0
    for e, r0, rows, pad in tiles.tolist():
        assert 0 <= e < E and 1 <= rows <= max_rows and pad == 0
        assert offsets[e] <= r0 and r0 + rows <= offsets[e + 1]
        if e != e_prev:
            assert e > e_prev and r0 == offsets[e]
            e_prev = e
        else:
            assert r0 == next_row
        next_row = r0 + rows
        covered[r0:r0 + rows] += 1
    assert np.all(covered == 1)
    counts = np.diff(np.asarray(offsets))
    per_e = np.bincount(tiles[:, 0], minlength=E) if len(tiles) else np.zeros(E, np.int64)
    assert np.all(per_e == -(-counts // max_rows))


def q2_columns(codes, scales, cols_idx, cols):
    """Selected columns of one row-major Q2 matrix (codes [rows][cols/4], scales [rows][cols/32]) dequantised to
    float64: -> [rows][len(cols_idx)] of d * (q - 2)."""
    j = np.asarray(cols_idx)
    q = (codes[:, j // 4] >> (2 * (j % 4))) & 3
    d = scales.view(np.float16)[:, j // 32].astype(np.float64)
    return d * (q.astype(np.float64) - 2.0)


def check_h_decisions(hc_g, hs_g, h_o, hc_o, hs_o):
    """The GPU's H codes and scales against the oracle's, where floating point decides the integer: a scale may
    differ only to the adjacent fp16 value and only where the oracle's amax / 127 lies within 1e-5 of the midpoint
    between the two; in blocks whose scales agree a code may differ only by 1 and only where the oracle's h / d lies
    within 1e-3 of the .5 tie between the two codes; at most 1e-4 of the codes may differ at all.  Arrays [..][F]
    (codes, h) and [..][F/32] (scale bits).  Returns (scale flips, code flips) as boolean masks."""
    F = hc_o.shape[-1]
    sflip = hs_g != hs_o
    if sflip.any():
        a = hs_g[sflip].view(np.float16).astype(np.float64)
        b = hs_o[sflip].view(np.float16).astype(np.float64)
        lo, hi = np.minimum(a, b), np.maximum(a, b)
        assert np.all(np.nextafter(lo.astype(np.float16), np.float16(np.inf)).astype(np.float64) == hi), \
            "a scale differs by more than one fp16 step"
        amax = np.abs(h_o.reshape(*h_o.shape[:-1], F // 32, 32)).max(-1)[sflip].astype(np.float64) / 127.0
        assert np.all(np.abs(amax - 0.5 * (lo + hi)) <= 1e-5 * amax), "a scale differs away from an fp16 midpoint"
    same = ~np.repeat(sflip, 32, axis=-1)
    cflip = (hc_g != hc_o) & same
    assert (hc_g != hc_o).sum() <= max(64, int(1e-4 * hc_o.size)), "too many H codes differ"
    if cflip.any():
        d = np.repeat(hs_o.view(np.float16).astype(np.float64), 32, axis=-1)
        assert np.all(np.abs(hc_g[cflip].astype(int) - hc_o[cflip].astype(int)) == 1), "a code differs by more than 1"
        ratio = np.abs(h_o[cflip].astype(np.float64) / d[cflip])
        assert np.all(np.abs(ratio % 1.0 - 0.5) <= 1e-3), "a code differs away from a .5 tie"
    return sflip, cflip


def tie_correction(hc_g, hs_g, hc_o, hs_o, ids, w, wd_c, wd_s):
    """What the valid tie decisions of check_h_decisions add to the block's output: for each (token, k) whose H
    differs, w[t][k] * W_down[e] (dequantised, double) applied to (GPU H - oracle H), with both H dequantised in
    double.  Arrays per token and slot: hc [T][K][F], hs [T][K][F/32], ids / w [T][K].  -> [T][H] float64."""
    T, K, F = hc_o.shape
    H = wd_c.shape[1]
    corr = np.zeros((T, H))
    diff = (hc_g != hc_o) | np.repeat(hs_g != hs_o, 32, axis=-1)
    for t, k in zip(*np.nonzero(diff.any(axis=-1))):
        j = np.nonzero(diff[t, k])[0]
        dg = hc_g[t, k, j].astype(np.float64) * hs_g[t, k, j // 32].view(np.float16).astype(np.float64)
        do = hc_o[t, k, j].astype(np.float64) * hs_o[t, k, j // 32].view(np.float16).astype(np.float64)
        e = int(ids[t, k])
        corr[t] += w[t, k] * (q2_columns(wd_c[e], wd_s[e], j, F) @ (dg - do))
    return corr

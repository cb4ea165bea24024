"""Thin Python binding of libsmoe's C ABI (include/smoe.h): the calls of include/smoe.h, argument marshalling only.

Every step runs in the CUDA kernels of libsmoe.so; this module checks tensor types and shapes, passes raw device
pointers and the current CUDA stream, and raises SmoeError on a non-OK status.  There is no fallback: when the
library is missing or the device is not an sm_103 part, the calls raise.

``SmoeBlock`` holds the intermediate buffers of one chunk size (allocated once with PyTorch) and runs the eight
calls in order; it is what the tests and the benchmark drive.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsmoe.so")

SMOE_OK, SMOE_ERR_ARG, SMOE_ERR_LAUNCH, SMOE_ERR_UNSUPPORTED, SMOE_ERR_RANGE, SMOE_ERR_TIMEOUT, SMOE_ERR_CUDA = range(7)
TILE_ROWS = 192


class SmoeError(RuntimeError):
    def __init__(self, call: str, status: int, text: str):
        super().__init__(f"{call}: status {status} ({text})")
        self.status = status


_lock = threading.Lock()
_lib = None

_SIGS = {
    "smoe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "smoe_last_error_string": ([], ctypes.c_char_p),
    "smoe_device_check": ([], ctypes.c_int),
    "smoe_max_tiles": ([ctypes.c_int64, ctypes.c_int], ctypes.c_int64),
    "smoe_tiles_bytes": ([ctypes.c_int64, ctypes.c_int], ctypes.c_size_t),
    "smoe_group_work_bytes": ([ctypes.c_int64, ctypes.c_int], ctypes.c_size_t),
    "smoe_route_topk": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                         ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_group": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                    ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "smoe_group_noalloc": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                            ctypes.c_void_p], ctypes.c_int),
    "smoe_quantize_q8": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                          ctypes.c_void_p], ctypes.c_int),
    "smoe_pack_q2": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                      ctypes.c_void_p], ctypes.c_int),
    "smoe_pack_q2_bytes": ([ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_size_t),
    "smoe_pack_q2_swiglu": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                             ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_gather_q8": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_gateup": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_gateup_swiglu": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_q8_work_bytes": ([ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_size_t),
    "smoe_experts_gateup_q8": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_down_q8": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                              ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_swiglu_requant": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                             ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_down": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_combine": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                      ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_experts_down_h": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_combine_h": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                        ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_router_topk": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_router_work_bytes": ([ctypes.c_int64, ctypes.c_int], ctypes.c_size_t),
    "smoe_shared_gate": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                          ctypes.c_void_p], ctypes.c_int),
    "smoe_combine_shared": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                            ctypes.c_int),
    "smoe_block_create": ([ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "smoe_block_destroy": ([ctypes.c_void_p], None),
    "smoe_block_run": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                       ctypes.c_int),
    "smoe_block_submit_host": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                               ctypes.c_int),
    "smoe_block_sync": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "smoe_block_status": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)],
                          ctypes.c_int),
}

# every symbol include/smoe.h declares
EXPORTS = tuple(_SIGS)


def load_library(path: str = LIB_PATH):
    """Load libsmoe.so and set the C signatures (no GPU needed to load it)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libsmoe.so is missing at {path}: build it first (__graft_entry__.build() or "
                                   "python quantized_routed_expert_smoe_gb300/build.py); there is no fallback path")
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return load_library().smoe_status_string(status).decode()


def _check(call: str, status: int):
    if status != SMOE_OK:
        text = status_string(status)
        if status in (SMOE_ERR_LAUNCH, SMOE_ERR_CUDA):
            text += ": " + load_library().smoe_last_error_string().decode()
        raise SmoeError(call, status, text)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _as_stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def device_check():
    _check("smoe_device_check", load_library().smoe_device_check())


def max_tiles(n: int, E: int) -> int:
    return int(load_library().smoe_max_tiles(n, E))


def tiles_bytes(n: int, E: int) -> int:
    return int(load_library().smoe_tiles_bytes(n, E))


def group_work_bytes(n: int, E: int) -> int:
    return int(load_library().smoe_group_work_bytes(n, E))


def pack_q2_bytes(E: int, rows: int, cols: int) -> int:
    return int(load_library().smoe_pack_q2_bytes(E, rows, cols))


def _opt(t, dtype, name):
    return ctypes.c_void_p(0) if t is None else _dev(t, dtype, name)


# ------------------------------------------------------------------------------------------------ the calls
def smoe_route_topk(logits, ids, w, stream=None):
    T, E = logits.shape
    K = ids.shape[1]
    _check("smoe_route_topk", load_library().smoe_route_topk(
        _dev(logits, torch.float32, "logits"), T, E, K, _dev(ids, torch.int32, "ids"), _dev(w, torch.float32, "w"),
        _stream(stream)))


def smoe_group(ids, E, counts, offsets, src, slot, tiles, work, stream=None):
    T, K = ids.shape
    _check("smoe_group", load_library().smoe_group(
        _dev(ids, torch.int32, "ids"), T, K, E, _dev(counts, torch.int32, "counts"),
        _dev(offsets, torch.int32, "offsets"), _dev(src, torch.int32, "src"), _dev(slot, torch.int32, "slot"),
        _dev(tiles, torch.int32, "tiles"), tiles.numel() * 4, _dev(work, torch.uint8, "work"), work.numel(),
        _stream(stream)))


def smoe_group_noalloc(ids, E, counts, offsets, src, slot, tiles, stream=None):
    """smoe_group with the library's built-in scratch (for callers that cannot allocate device memory)."""
    T, K = ids.shape
    _check("smoe_group_noalloc", load_library().smoe_group_noalloc(
        _dev(ids, torch.int32, "ids"), T, K, E, _dev(counts, torch.int32, "counts"),
        _dev(offsets, torch.int32, "offsets"), _dev(src, torch.int32, "src"), _dev(slot, torch.int32, "slot"),
        _dev(tiles, torch.int32, "tiles"), tiles.numel() * 4, _stream(stream)))


def smoe_quantize_q8(x, codes, scales, stream=None):
    rows, cols = x.shape
    _check("smoe_quantize_q8", load_library().smoe_quantize_q8(
        _dev(x, torch.float32, "x"), rows, cols, _dev(codes, torch.int8, "codes"),
        _dev(scales, torch.int16, "scales"), _stream(stream)))


def smoe_pack_q2(codes, scales, packed, stream=None):
    """Row-major Q2 weights (codes uint8 [E][rows][cols/4], scales int16 bits [E][rows][cols/32]) -> packed."""
    E, rows, c4 = codes.shape
    _check("smoe_pack_q2", load_library().smoe_pack_q2(
        _dev(codes, torch.uint8, "codes"), _dev(scales, torch.int16, "scales"), E, rows, c4 * 4,
        _dev(packed, torch.uint8, "packed"), _stream(stream)))


def smoe_gather_q8(codes, scales, src, out, stream=None):
    """out = the q8 rows src[r] of (codes int8 [in_rows][cols], scales [in_rows][cols/32]) in operand form, fp16
    [2][n][cols] (n = src.numel())."""
    in_rows, cols = codes.shape
    _check("smoe_gather_q8", load_library().smoe_gather_q8(
        _dev(codes, torch.int8, "codes"), _dev(scales, torch.int16, "scales"), in_rows, cols,
        _dev(src, torch.int32, "src"), src.numel(), _dev(out, torch.float16, "out"), _stream(stream)))


def smoe_experts_gateup(xop, tiles, n, E, wgu, H, F, gu, stream=None):
    _check("smoe_experts_gateup", load_library().smoe_experts_gateup(
        _dev(xop, torch.float16, "xop"), _dev(tiles, torch.int32, "tiles"), n, E, _dev(wgu, torch.uint8, "wgu"), H, F,
        _dev(gu, torch.float32, "gu"), _stream(stream)))


def smoe_pack_q2_swiglu(codes, scales, packed, stream=None):
    """Gate/up Q2 weights (codes uint8 [E][2F][H/4], scales int16 bits [E][2F][H/32]) -> packed for the fused product."""
    E, rows, c4 = codes.shape
    _check("smoe_pack_q2_swiglu", load_library().smoe_pack_q2_swiglu(
        _dev(codes, torch.uint8, "codes"), _dev(scales, torch.int16, "scales"), E, rows // 2, c4 * 4,
        _dev(packed, torch.uint8, "packed"), _stream(stream)))


def smoe_experts_gateup_swiglu(xop, tiles, n, E, wgs, H, F, hc, hs, hop, stream=None):
    _check("smoe_experts_gateup_swiglu", load_library().smoe_experts_gateup_swiglu(
        _dev(xop, torch.float16, "xop"), _dev(tiles, torch.int32, "tiles"), n, E, _dev(wgs, torch.uint8, "wgs"), H, F,
        _dev(hc, torch.int8, "hc"), _dev(hs, torch.int16, "hs"), _dev(hop, torch.float16, "hop"), _stream(stream)))


def experts_q8_work_bytes(n: int, E: int, H: int, F: int) -> int:
    return int(load_library().smoe_experts_q8_work_bytes(n, E, H, F))


def q2_descriptors(experts):
    """A device array of smoe_q2w descriptors (two 64-bit pointers each) for a list of (codes, scales) CUDA tensors,
    one per expert: codes uint8 [rows][cols/4], scales int16 bits [rows][cols/32].  The tensors must stay alive while
    the descriptors are used."""
    ptrs = []
    for c, sc in experts:
        _dev(c, torch.uint8, "codes")
        _dev(sc, torch.int16, "scales")
        ptrs += [c.data_ptr(), sc.data_ptr()]
    dev = experts[0][0].device if experts else torch.device("cuda")
    return torch.tensor(ptrs, dtype=torch.int64).to(dev)


def smoe_experts_gateup_q8(xc, xs, src, tiles, n, E, w_gu, H, F, work, gu, stream=None):
    """gate/up from per-token q8 activations (xc int8 [T][H], xs int16 bits [T][H/32]), src int32 [n] and a device
    array of E weight descriptors (q2_descriptors); work: uint8 scratch of experts_q8_work_bytes(n, E, H, F)."""
    _check("smoe_experts_gateup_q8", load_library().smoe_experts_gateup_q8(
        _dev(xc, torch.int8, "xc"), _dev(xs, torch.int16, "xs"), xc.shape[0], _dev(src, torch.int32, "src"),
        _dev(tiles, torch.int32, "tiles"), n, E, _dev(w_gu, torch.int64, "w_gu"), H, F, _dev(work, torch.uint8, "work"),
        work.numel(), _dev(gu, torch.float32, "gu"), _stream(stream)))


def smoe_experts_down_q8(hc, hs, tiles, n, E, w_d, H, F, work, dm, stream=None):
    """down from planar q8 H (hc int8 [n][F], hs int16 bits [n][F/32]) and a device array of E weight descriptors."""
    _check("smoe_experts_down_q8", load_library().smoe_experts_down_q8(
        _dev(hc, torch.int8, "hc"), _dev(hs, torch.int16, "hs"), _dev(tiles, torch.int32, "tiles"), n, E,
        _dev(w_d, torch.int64, "w_d"), H, F, _dev(work, torch.uint8, "work"), work.numel(),
        _dev(dm, torch.float32, "dm"), _stream(stream)))


def smoe_swiglu_requant(gu, hc, hs, hop=None, stream=None):
    n, twoF = gu.shape
    _check("smoe_swiglu_requant", load_library().smoe_swiglu_requant(
        _dev(gu, torch.float32, "gu"), n, twoF // 2, _dev(hc, torch.int8, "hc"), _dev(hs, torch.int16, "hs"),
        _opt(hop, torch.float16, "hop"), _stream(stream)))


def smoe_experts_down(hop, tiles, n, E, wd, H, F, dm, stream=None):
    _check("smoe_experts_down", load_library().smoe_experts_down(
        _dev(hop, torch.float16, "hop"), _dev(tiles, torch.int32, "tiles"), n, E, _dev(wd, torch.uint8, "wd"), H, F,
        _dev(dm, torch.float32, "dm"), _stream(stream)))


def smoe_combine(dm, slot, w, y, stream=None):
    T, K = w.shape
    H = y.shape[1]
    _check("smoe_combine", load_library().smoe_combine(
        _dev(dm, torch.float32, "dm"), _dev(slot, torch.int32, "slot"), _dev(w, torch.float32, "w"), T, K, H,
        _dev(y, torch.float32, "y"), _stream(stream)))


def smoe_experts_down_h(hop, tiles, n, E, wd, H, F, dm_h, stream=None):
    """smoe_experts_down with the rows stored as fp16 (dm_h torch.float16 [n][H])."""
    _check("smoe_experts_down_h", load_library().smoe_experts_down_h(
        _dev(hop, torch.float16, "hop"), _dev(tiles, torch.int32, "tiles"), n, E, _dev(wd, torch.uint8, "wd"), H, F,
        _dev(dm_h, torch.float16, "dm_h"), _stream(stream)))


def smoe_combine_h(dm_h, slot, w, y, stream=None):
    """smoe_combine from fp16 down rows (dm_h torch.float16 [n][H])."""
    T, K = w.shape
    H = y.shape[1]
    _check("smoe_combine_h", load_library().smoe_combine_h(
        _dev(dm_h, torch.float16, "dm_h"), _dev(slot, torch.int32, "slot"), _dev(w, torch.float32, "w"), T, K, H,
        _dev(y, torch.float32, "y"), _stream(stream)))


def router_work_bytes(T: int, H: int) -> int:
    return int(load_library().smoe_router_work_bytes(T, H))


def smoe_router_topk(x, wr, ids, w, work, stream=None):
    """Router projection (bf16 weights wr [E][H] as int16 bits, activations x fp32 [T][H] split into bf16 hi + lo)
    fused into the top-K: ids int32 [T][K], w fp32 [T][K]; work: uint8 scratch of router_work_bytes(T, H)."""
    T, H = x.shape
    E = wr.shape[0]
    K = ids.shape[1]
    _check("smoe_router_topk", load_library().smoe_router_topk(
        _dev(x, torch.float32, "x"), _dev(wr, torch.int16, "wr"), T, H, E, K, _dev(work, torch.uint8, "work"),
        _dev(ids, torch.int32, "ids"), _dev(w, torch.float32, "w"), _stream(stream)))


def smoe_shared_gate(x, wsg, sg, stream=None):
    """sg [T] = sigmoid(x [T][H] . w_sg [H]) (the shared expert's scalar gate)."""
    T, H = x.shape
    _check("smoe_shared_gate", load_library().smoe_shared_gate(
        _dev(x, torch.float32, "x"), _dev(wsg, torch.float32, "wsg"), T, H, _dev(sg, torch.float32, "sg"),
        _stream(stream)))


def smoe_combine_shared(dm, slot, w, ds, sg, y, stream=None):
    T, K = w.shape
    H = y.shape[1]
    _check("smoe_combine_shared", load_library().smoe_combine_shared(
        _dev(dm, torch.float32, "dm"), _dev(slot, torch.int32, "slot"), _dev(w, torch.float32, "w"), T, K, H,
        _dev(ds, torch.float32, "ds"), _dev(sg, torch.float32, "sg"), _dev(y, torch.float32, "y"), _stream(stream)))


# ------------------------------------------------------------------------------------------------ one block
class SmoeBlock:
    """The routed-expert block for chunks of up to T tokens: weights resident on the device, every intermediate
    buffer allocated once.  run(logits, x) issues the eight calls on the current stream and returns y [T][H].

    shared: optional dict(sgu_c, sgu_s, sd_c, sd_s, wsg) -- a shared expert (gate/up codes [2F][H/4] and scales,
    down codes [H][F/4] and scales, in the routed experts' format) and its scalar gate row w_sg [H]; every token
    takes it and the combine adds sigmoid(x . w_sg) times its row.

    router: optional bf16 router weights (uint16 / int16 bits [E][H]); the block then computes the router projection
    itself (smoe_router_topk) and run() ignores its logits argument.

    fused: run gate/up, SwiGLU and the requantisation as one product (smoe_experts_gateup_swiglu, the gate/up weights
    packed interleaved); GU is then never written.

    narrow_dm: keep the down rows Dm in fp16 (smoe_experts_down_h / smoe_combine_h) instead of fp32, the pages' form;
    not with a shared expert."""

    def __init__(self, T: int, H: int, E: int, K: int, F: int, wgu_c, wgu_s, wd_c, wd_s, device="cuda",
                 shared=None, router=None, fused=False, narrow_dm=False):
        load_library()
        if narrow_dm and shared is not None:
            raise ValueError("narrow_dm: the shared-expert combine reads fp32 down rows")
        device_check()
        self.T, self.H, self.E, self.K, self.F = T, H, E, K, F
        dev = torch.device(device)
        as_t = lambda a, dt: torch.as_tensor(a).to(device=dev, dtype=dt).contiguous()
        # the expert weights, packed once for the expert products (the row-major copies are not kept)
        self.fused = bool(fused)
        self.wgu = pack_weights(wgu_c, wgu_s, dev, swiglu=self.fused)
        self.wd = pack_weights(wd_c, wd_s, dev)
        n = T * K
        self.n = n
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)
        self.ids = e(T, K, dt=torch.int32)
        self.w = e(T, K, dt=torch.float32)
        self.counts = e(E, dt=torch.int32)
        self.offsets = e(E + 1 + 3, dt=torch.int32)  # padded to 16 bytes
        self.src = e(max(n, 4), dt=torch.int32)
        self.slot = e(max(n, 4), dt=torch.int32)
        self.tiles = e(tiles_bytes(n, E) // 4, dt=torch.int32)
        self.work = e(max(group_work_bytes(n, E), 16), dt=torch.uint8)
        self.xc = e(T, H, dt=torch.int8)
        self.xs = e(T, H // 32, dt=torch.int16)
        self.xop = e(2, max(n, 1), H, dt=torch.float16)  # routed rows, operand form (hi, lo)
        self.gu = e(0 if self.fused else n, 2 * F, dt=torch.float32)
        self.hc = e(n, F, dt=torch.int8)
        self.hs = e(n, F // 32, dt=torch.int16)
        self.hop = e(2, max(n, 1), F, dt=torch.float16)
        self.narrow_dm = bool(narrow_dm)
        self.dm = e(n, H, dt=torch.float16 if self.narrow_dm else torch.float32)
        self.y = e(T, H, dt=torch.float32)
        self.router = None
        if router is not None:
            self.router = _as_i16(router, dev)
            self.router_work = e(max(router_work_bytes(T, H), 16), dt=torch.uint8)
        self._side = None  # side stream for the quantisation (created on the first run)
        self.shared = shared is not None
        if self.shared:
            lift = lambda a: a[None] if a.ndim == 2 else a  # one expert: [rows][..] -> [1][rows][..]
            as_np = lambda a: a.cpu().numpy() if isinstance(a, torch.Tensor) else a
            self.swgu = pack_weights(lift(as_np(shared["sgu_c"])), lift(as_np(shared["sgu_s"])), dev)
            self.swd = pack_weights(lift(as_np(shared["sd_c"])), lift(as_np(shared["sd_s"])), dev)
            self.wsg = as_t(shared["wsg"], torch.float32)
            # the shared expert's grouping: E = 1, K = 1, every id 0 -> row r = token r, its tiles; fixed for T
            zeros = torch.zeros(T, 1, dtype=torch.int32, device=dev)
            self.s_counts = e(1 + 3, dt=torch.int32)
            self.s_offsets = e(2 + 2, dt=torch.int32)
            self.s_src = e(max(T, 4), dt=torch.int32)
            self.s_slot = e(max(T, 4), dt=torch.int32)
            self.s_tiles = e(tiles_bytes(T, 1) // 4, dt=torch.int32)
            s_work = e(max(group_work_bytes(T, 1), 16), dt=torch.uint8)
            smoe_group(zeros, 1, self.s_counts[:1], self.s_offsets[:2], self.s_src[:T], self.s_slot[:T],
                       self.s_tiles, s_work)
            self.sxop = e(2, max(T, 1), H, dt=torch.float16)
            self.sgu = e(T, 2 * F, dt=torch.float32)
            self.shc = e(T, F, dt=torch.int8)
            self.shs = e(T, F // 32, dt=torch.int16)
            self.shop = e(2, max(T, 1), F, dt=torch.float16)
            self.ds = e(T, H, dt=torch.float32)
            self.sg = e(max(T, 4), dt=torch.float32)

    def run(self, logits, x, stream=None, out=None):
        """y = the block on (logits [T][E], x [T][H]); into `out` (fp32 [T][H] on the device) when given.

        The q8 quantisation of x depends on neither the routing nor the grouping, so it runs on a side stream beside
        them (forked from and joined back into `stream` with events; the same holds inside a CUDA-graph capture)."""
        y = self.y if out is None else out
        main = _as_stream(stream, x.device)
        if self._side is None:
            self._side = torch.cuda.Stream(device=x.device)
            self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()
        self._fork.record(main)
        self._side.wait_event(self._fork)
        smoe_quantize_q8(x, self.xc, self.xs, self._side)
        self._join.record(self._side)
        if self.router is not None:
            smoe_router_topk(x, self.router, self.ids, self.w, self.router_work, main)
        else:
            smoe_route_topk(logits, self.ids, self.w, main)
        smoe_group(self.ids, self.E, self.counts, self.offsets, self.src[:self.n], self.slot[:self.n], self.tiles,
                   self.work, main)
        main.wait_event(self._join)
        stream = main
        smoe_gather_q8(self.xc, self.xs, self.src[:self.n], self.xop, stream)
        if self.fused:
            smoe_experts_gateup_swiglu(self.xop, self.tiles, self.n, self.E, self.wgu, self.H, self.F, self.hc,
                                       self.hs, self.hop, stream)
        else:
            smoe_experts_gateup(self.xop, self.tiles, self.n, self.E, self.wgu, self.H, self.F, self.gu, stream)
            smoe_swiglu_requant(self.gu, self.hc, self.hs, self.hop, stream)
        if self.narrow_dm:
            smoe_experts_down_h(self.hop, self.tiles, self.n, self.E, self.wd, self.H, self.F, self.dm, stream)
            smoe_combine_h(self.dm, self.slot, self.w, y, stream)
            return y
        smoe_experts_down(self.hop, self.tiles, self.n, self.E, self.wd, self.H, self.F, self.dm, stream)
        if not self.shared:
            smoe_combine(self.dm, self.slot, self.w, y, stream)
            return y
        T = self.T
        smoe_shared_gate(x, self.wsg, self.sg[:T], stream)
        smoe_gather_q8(self.xc, self.xs, self.s_src[:T], self.sxop, stream)
        smoe_experts_gateup(self.sxop, self.s_tiles, T, 1, self.swgu, self.H, self.F, self.sgu, stream)
        smoe_swiglu_requant(self.sgu, self.shc, self.shs, self.shop, stream)
        smoe_experts_down(self.shop, self.s_tiles, T, 1, self.swd, self.H, self.F, self.ds, stream)
        smoe_combine_shared(self.dm, self.slot, self.w, self.ds, self.sg[:T], y, stream)
        return y

    def capture(self, logits, x, out=None):
        """A CUDA graph of one run() on these device inputs (their buffers, read again at every replay): replaying it
        issues the block's kernels without the host's per-launch cost.  run() must have been called once before (the
        libraries' one-time set-up per device is not captured)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(logits, x, out=out)
        return g

    def device_status(self):
        """(group status, kernel status) from the tiles header; reads the device (synchronises)."""
        h = self.tiles[:4].cpu().tolist()
        return h[1], h[3]


class SmoePipeline:
    """A SmoeBlock fed from and into pinned host memory, with the copies overlapped with the compute: step i's inputs
    go to the device (one copy stream) while step i-1 computes, and its output comes back (another copy stream) while
    step i+1 computes; device inputs and outputs are double-buffered.

    start(event): the copies of the first step wait for `event` (e.g. recorded on the compute stream before a timed
    region); submit(h_logits, h_x, h_y) queues one step -- h_y (pinned fp32 [T][H]) holds the result once the step's
    copy back has completed; drain(): the compute stream waits for every queued copy back; synchronize(): the host
    waits for all of it.

    graphs=True: each of the two device buffer sets gets a CUDA graph of the block's run() on it (captured here; the
    block must have run once before), and a step replays its set's graph instead of launching the kernels one by
    one."""

    def __init__(self, block: "SmoeBlock", stream=None, graphs=False):
        self.blk = block
        dev = block.y.device
        T, H, E = block.T, block.H, block.E
        e = lambda *sh: torch.empty(*sh, dtype=torch.float32, device=dev)
        self.d_logits = [e(T, E), e(T, E)]
        self.d_x = [e(T, H), e(T, H)]
        self.d_y = [e(T, H), e(T, H)]
        self.compute = stream if stream is not None else torch.cuda.current_stream(dev)
        self.copy_in = torch.cuda.Stream(device=dev)
        self.copy_out = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event(), torch.cuda.Event()]    # slot b's inputs are on the device
        self.ev_done = [torch.cuda.Event(), torch.cuda.Event()]  # slot b's step has computed
        self.ev_out = [torch.cuda.Event(), torch.cuda.Event()]   # slot b's output is back on the host
        self.i = 0
        self.graphs = None
        if graphs:
            torch.cuda.synchronize(dev)
            self.graphs = [block.capture(self.d_logits[b], self.d_x[b], out=self.d_y[b]) for b in range(2)]

    def start(self, event):
        self.copy_in.wait_event(event)
        self.copy_out.wait_event(event)

    def submit(self, h_logits, h_x, h_y):
        b = self.i & 1
        with torch.cuda.stream(self.copy_in):
            if self.i >= 2:
                self.copy_in.wait_event(self.ev_done[b])  # step i-2 has consumed slot b's inputs
            if h_logits is not None:  # a block that computes its own router projection needs none
                self.d_logits[b].copy_(h_logits, non_blocking=True)
            self.d_x[b].copy_(h_x, non_blocking=True)
            self.ev_in[b].record(self.copy_in)
        self.compute.wait_event(self.ev_in[b])
        if self.i >= 2:
            self.compute.wait_event(self.ev_out[b])  # slot b's previous output is back on the host
        if self.graphs is not None:
            with torch.cuda.stream(self.compute):
                self.graphs[b].replay()
        else:
            self.blk.run(self.d_logits[b], self.d_x[b], stream=self.compute, out=self.d_y[b])
        self.ev_done[b].record(self.compute)
        with torch.cuda.stream(self.copy_out):
            self.copy_out.wait_event(self.ev_done[b])
            h_y.copy_(self.d_y[b], non_blocking=True)
            self.ev_out[b].record(self.copy_out)
        self.i += 1

    def drain(self):
        for k in range(min(self.i, 2)):
            self.compute.wait_event(self.ev_out[k])

    def synchronize(self):
        self.drain()
        self.compute.synchronize()


class NativeBlock:
    """The block as the library's own object (smoe_block_*): its device buffers, streams and CUDA graphs live in
    libsmoe; this class only passes pointers.  run(logits, x, y): one chunk device to device.  submit_host(logits,
    x, y): one chunk from and into host memory (torch CPU tensors, pinned for overlapped copies), queued; sync(): the
    host (and `stream`) wait for every submitted chunk.  The expert weights are packed here once and kept alive as
    long as the block."""

    def __init__(self, T: int, H: int, E: int, K: int, F: int, wgu_c, wgu_s, wd_c, wd_s, device="cuda"):
        load_library()
        device_check()
        self.T, self.H, self.E, self.K, self.F = T, H, E, K, F
        self.wgu = pack_weights(wgu_c, wgu_s, device)
        self.wd = pack_weights(wd_c, wd_s, device)
        torch.cuda.synchronize(self.wgu.device)
        h = ctypes.c_void_p()
        lib = load_library()
        _check("smoe_block_create", lib.smoe_block_create(T, H, E, K, F, self.wgu.data_ptr(), self.wd.data_ptr(),
                                                          ctypes.byref(h)))
        self._h = h

    def _stream(self, stream):
        return _as_stream(stream, self.wgu.device).cuda_stream

    def run(self, logits, x, y, stream=None):
        _check("smoe_block_run", load_library().smoe_block_run(self._h, logits.data_ptr(), x.data_ptr(), y.data_ptr(),
                                                               self._stream(stream)))
        return y

    def submit_host(self, logits, x, y, stream=None):
        for t in (logits, x, y):
            assert t.device.type == "cpu" and t.dtype == torch.float32 and t.is_contiguous()
        assert logits.numel() == self.T * self.E and x.numel() == self.T * self.H and y.numel() == self.T * self.H
        _check("smoe_block_submit_host", load_library().smoe_block_submit_host(
            self._h, logits.data_ptr(), x.data_ptr(), y.data_ptr(), self._stream(stream)))

    def sync(self, stream=None):
        _check("smoe_block_sync", load_library().smoe_block_sync(self._h, self._stream(stream)))

    def device_status(self):
        g, k = ctypes.c_int(), ctypes.c_int()
        _check("smoe_block_status", load_library().smoe_block_status(self._h, ctypes.byref(g), ctypes.byref(k)))
        return g.value, k.value

    def close(self):
        if getattr(self, "_h", None) is not None:
            load_library().smoe_block_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pack_weights(codes, scales, device="cuda", swiglu=False):
    """Row-major Q2 weights (numpy or torch: codes [E][rows][cols/4], scales fp16 bits [E][rows][cols/32]) packed on
    the device for the expert products; swiglu=True packs a gate/up matrix for the fused gate/up + SwiGLU product."""
    dev = torch.device(device)
    c = codes.to(dev).contiguous() if isinstance(codes, torch.Tensor) else torch.from_numpy(codes).to(dev).contiguous()
    s = _as_i16(scales, dev)
    E, rows, c4 = c.shape
    packed = torch.empty(pack_q2_bytes(E, rows, c4 * 4), dtype=torch.uint8, device=dev)
    (smoe_pack_q2_swiglu if swiglu else smoe_pack_q2)(c, s, packed)
    return packed


def _as_i16(a, dev):
    if isinstance(a, torch.Tensor):
        return a.to(dev).view(torch.int16).contiguous()
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

"""GB300-native block-scaled MXFP4 GEMM: C[M,N] (bf16) = MXFP4(A[M,K] bf16) . MXFP4(B[N,K])^T.

Thin Python binding over the C ABI in ``include/mxfp4_gb300.h`` (libmxfp4_gb300.so, built
in-tree for sm_103a). The functions keep the C names and only marshal arguments: PyTorch
provides device memory and the current CUDA stream; every step of the computation runs in
the library's CUDA kernels. There is no CPU fallback: if the library cannot be loaded or
built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "Mxfp4Error", "load_library", "mxfp4_quantize", "mxfp4_prepack_b_size", "mxfp4_prepack_b",
    "mxfp4_gemm_workspace_size", "mxfp4_workspace_init", "mxfp4_gemm", "mxfp4_gemm_host", "mxfp4_gemm_noalloc",
    "mxfp4_gemm_plan", "mxfp4_gemm_plan_model", "mxfp4_device_status", "mxfp4_selftest_timeout", "mxfp4_version",
    "PreparedCall", "prepare_gemm", "prepare_gemm_host", "TokenBlocks", "mxfp4_token_tile", "mxfp4_token_blocks_size",
    "mxfp4_quantize_tokens", "mxfp4_gemm_tokens", "mxfp4_gemm_unpacked",
]

_LOCK = threading.Lock()
_LIB = None
_WS: dict = {}

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_int = ctypes.c_int


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _LIB
        name = lib.mxfp4_status_string(status).decode() if lib is not None else str(status)
        extra = ""
        if lib is not None and name == "MXFP4_ERR_CUDA":
            extra = f" (cudaError {lib.mxfp4_last_cuda_error()})"
        super().__init__(f"{where}: {name}{extra}")
        self.status = status


class _Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("splits", ctypes.c_int), ("m_tile", ctypes.c_int),
                ("flags", ctypes.c_int), ("reserved", ctypes.c_int * 4)]


GEMM_A_READY = 1   # mxfp4_gemm_options.flags: MXFP4_GEMM_A_READY


def load_library() -> ctypes.CDLL:
    """Load (building first if needed) libmxfp4_gb300.so. Raises if that is impossible."""
    global _LIB
    lib = _LIB
    if lib is not None:   # loaded: no lock on the per-call path
        return lib
    with _LOCK:
        if _LIB is None:
            path = _build.LIB_PATH
            if not _build.up_to_date():
                path = _build.build()
            L = ctypes.CDLL(path)
            L.mxfp4_status_string.restype = ctypes.c_char_p
            L.mxfp4_status_string.argtypes = [_int]
            L.mxfp4_last_cuda_error.restype = _int
            L.mxfp4_version.restype = _int
            L.mxfp4_quantize.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _vp]
            L.mxfp4_quantize.restype = _int
            L.mxfp4_prepack_b_size.argtypes = [_i64, _i64]
            L.mxfp4_prepack_b_size.restype = _sz
            L.mxfp4_prepack_b.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp]
            L.mxfp4_prepack_b.restype = _int
            L.mxfp4_gemm_workspace_size.argtypes = [_i64, _i64, _i64]
            L.mxfp4_gemm_workspace_size.restype = _sz
            L.mxfp4_gemm_workspace_size_ex.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_Options)]
            L.mxfp4_gemm_workspace_size_ex.restype = _sz
            L.mxfp4_workspace_init.argtypes = [_vp, _sz, _vp]
            L.mxfp4_workspace_init.restype = _int
            L.mxfp4_gemm.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _sz, _vp]
            L.mxfp4_gemm.restype = _int
            L.mxfp4_gemm_ex.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _sz,
                                        ctypes.POINTER(_Options), _vp]
            L.mxfp4_gemm_ex.restype = _int
            L.mxfp4_gemm_plan.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_Options)] + [ctypes.POINTER(_int)] * 5
            L.mxfp4_gemm_plan.restype = _int
            L.mxfp4_gemm_host.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _sz, _vp]
            L.mxfp4_gemm_host.restype = _int
            L.mxfp4_gemm_noalloc.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
            L.mxfp4_gemm_noalloc.restype = _int
            L.mxfp4_gemm_plan_model.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_Options), _int,
                                                ctypes.POINTER(_int), ctypes.POINTER(_PlanInfo)]
            L.mxfp4_gemm_plan_model.restype = _int
            L.mxfp4_gemm_plan_info.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_Options), ctypes.POINTER(_PlanInfo)]
            L.mxfp4_gemm_plan_info.restype = _int
            L.mxfp4_device_status.argtypes = [_vp]
            L.mxfp4_device_status.restype = _int
            L.mxfp4_selftest_timeout.argtypes = [_int, _vp]
            L.mxfp4_selftest_timeout.restype = _int
            L.mxfp4_token_tile.argtypes = [_i64, _i64, _int]
            L.mxfp4_token_tile.restype = _int
            L.mxfp4_token_blocks_size.argtypes = [_i64, _i64, _int]
            L.mxfp4_token_blocks_size.restype = _sz
            L.mxfp4_quantize_tokens.argtypes = [_vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]
            L.mxfp4_quantize_tokens.restype = _int
            L.mxfp4_gemm_tokens.argtypes = [_vp, _sz, _i64, _i64, _int, _vp, _i64, _vp, _i64, _int, _vp]
            L.mxfp4_gemm_tokens.restype = _int
            L.mxfp4_gemm_unpacked_workspace_size.argtypes = [_i64, _i64, _i64]
            L.mxfp4_gemm_unpacked_workspace_size.restype = _sz
            L.mxfp4_gemm_unpacked.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _i64, _vp, _sz, _vp]
            L.mxfp4_gemm_unpacked.restype = _int
            _pp = ctypes.POINTER(_vp)
            L.mxfp4_call_create.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _sz,
                                            ctypes.POINTER(_Options), _pp]
            L.mxfp4_call_create.restype = _int
            L.mxfp4_call_create_host.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _sz,
                                                 ctypes.c_uint, _pp]
            L.mxfp4_call_create_host.restype = _int
            L.mxfp4_call_run.argtypes = [_vp, _vp]
            L.mxfp4_call_run.restype = _int
            L.mxfp4_call_destroy.argtypes = [_vp]
            L.mxfp4_call_destroy.restype = None
            _LIB = L
    return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        raise Mxfp4Error(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str) -> None:
    """The library plans and launches on the current CUDA device: `t` must live there."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current CUDA device")


def _on(t: torch.Tensor, device: torch.device, name: str) -> None:
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, with the other operands")


def _out_bytes(t: torch.Tensor, shape: tuple, device: torch.device, name: str) -> None:
    """A caller-supplied uint8 output: the kernels write it as one dense [rows, cols] block."""
    if t.device != device or t.dtype != torch.uint8 or tuple(t.shape) != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous uint8 tensor of shape {list(shape)} on {device}")


def _opts(path: int, splits: int, m_tile: int = 0, flags: int = 0):
    return ctypes.byref(_Options(path, splits, m_tile, flags))


def mxfp4_version() -> int:
    return load_library().mxfp4_version()


def mxfp4_quantize(x: torch.Tensor, q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                   stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 [rows, K] (row stride may exceed K, K % 8 == 0) -> (e2m1 uint8 [rows, nblk*16],
    e8m0 uint8 [rows, nblk]) with nblk = ceil(K/32); codes past K are zero."""
    L = load_library()
    _dev(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bf16 tensor with unit column stride")
    rows, K = x.shape
    nblk = (K + 31) // 32
    if q is None:
        q = torch.empty(rows, nblk * 16, dtype=torch.uint8, device=x.device)
    else:
        _out_bytes(q, (rows, nblk * 16), x.device, "q")
    if scales is None:
        scales = torch.empty(rows, nblk, dtype=torch.uint8, device=x.device)
    else:
        _out_bytes(scales, (rows, nblk), x.device, "scales")
    _check(L.mxfp4_quantize(x.data_ptr(), rows, K, x.stride(0), q.data_ptr(), scales.data_ptr(), _stream(stream)),
           "mxfp4_quantize")
    return q, scales


def mxfp4_prepack_b_size(N: int, K: int) -> int:
    return int(load_library().mxfp4_prepack_b_size(N, K))


def mxfp4_prepack_b(bq: torch.Tensor, bs: torch.Tensor, packed: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Pre-quantized B (e2m1 [N, nblk*16], e8m0 [N, nblk], the layout mxfp4_quantize writes) ->
    packed uint8 buffer for mxfp4_gemm with any K in (32*(nblk-1), 32*nblk]."""
    L = load_library()
    _dev(bq, "bq")
    _on(bs, bq.device, "bs")
    N, K = bq.shape[0], bq.shape[1] * 2
    if bs.shape != (N, K // 32) or not bq.is_contiguous() or not bs.is_contiguous():
        raise ValueError("bq [N, nblk*16] and bs [N, nblk] must be contiguous and consistent")
    if bq.element_size() != 1 or bs.element_size() != 1:
        raise ValueError("bq and bs must be byte tensors")
    size = mxfp4_prepack_b_size(N, K)
    if size == 0:
        raise Mxfp4Error(2, "mxfp4_prepack_b_size")
    if packed is None:
        packed = torch.empty(size + 1024, dtype=torch.uint8, device=bq.device)
        off = (-packed.data_ptr()) % 1024
        packed = packed[off:off + size]
    elif packed.device != bq.device or packed.nbytes < size or not packed.is_contiguous():
        raise ValueError(f"packed must be a contiguous buffer of at least {size} bytes on {bq.device}")
    _check(L.mxfp4_prepack_b(bq.data_ptr(), bs.data_ptr(), N, K, packed.data_ptr(), _stream(stream)),
           "mxfp4_prepack_b")
    return packed


class TokenBlocks:
    """A quantized into the GEMM's token-block layout (mxfp4_quantize_tokens): `data` is the
    uint8 buffer (256-byte aligned), M, K and m_tile the layout's parameters, m_tile already
    cut to M (mxfp4_token_tile)."""

    __slots__ = ("data", "M", "K", "m_tile")

    def __init__(self, data: torch.Tensor, M: int, K: int, m_tile: int):
        self.data, self.M, self.K, self.m_tile = data, M, K, m_tile


def mxfp4_token_tile(M: int, K: int, m_tile: int = 0) -> int:
    return int(load_library().mxfp4_token_tile(M, K, m_tile))


def mxfp4_token_blocks_size(M: int, K: int, m_tile: int = 0) -> int:
    return int(load_library().mxfp4_token_blocks_size(M, K, m_tile))


def _aligned_bytes(nbytes: int, align: int, device: torch.device) -> torch.Tensor:
    buf = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % align
    return buf[off:off + nbytes]


def mxfp4_quantize_tokens(a: torch.Tensor, m_tile: int = 0, out: torch.Tensor | None = None,
                          stream=None) -> TokenBlocks:
    """bf16 A [M, K] (row stride may exceed K, K % 8 == 0) -> TokenBlocks for mxfp4_gemm_tokens.
    `out`, if given, is a contiguous uint8 buffer of at least mxfp4_token_blocks_size bytes,
    256-byte aligned, on A's device."""
    L = load_library()
    _dev(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    M, K = a.shape
    mt = mxfp4_token_tile(M, K, m_tile)
    size = mxfp4_token_blocks_size(M, K, m_tile)
    if mt == 0 or size == 0:
        raise ValueError(f"no token-block layout for M={M}, K={K}, m_tile={m_tile}")
    if out is None:
        out = _aligned_bytes(size, 256, a.device)
    elif (out.device != a.device or out.dtype != torch.uint8 or out.nbytes < size or not out.is_contiguous()
          or out.data_ptr() % 256):
        raise ValueError(f"out must be a contiguous 256-byte aligned uint8 buffer of at least {size} bytes on "
                         f"{a.device}")
    _check(L.mxfp4_quantize_tokens(a.data_ptr(), M, K, a.stride(0), mt, out.data_ptr(), out.nbytes, _stream(stream)),
           "mxfp4_quantize_tokens")
    return TokenBlocks(out, M, K, mt)


def mxfp4_gemm_tokens(tokens: TokenBlocks, packed_b: torch.Tensor, N: int, c: torch.Tensor | None = None,
                      splits: int = 0, stream=None) -> torch.Tensor:
    """C [M, N] bf16 = A . MXFP4(B)^T for A already quantized by mxfp4_quantize_tokens."""
    L = load_library()
    data, M, K = tokens.data, tokens.M, tokens.K
    _dev(data, "tokens")
    if M and N:
        _check_packed(packed_b, N, K, data.device)
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=data.device)
    _on(c, data.device, "c")
    if c.dtype != torch.bfloat16 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be a bf16 [M, N] tensor with unit column stride")
    _check(L.mxfp4_gemm_tokens(data.data_ptr(), data.nbytes, M, K, tokens.m_tile, packed_b.data_ptr(), N,
                               c.data_ptr(), c.stride(0), splits, _stream(stream)), "mxfp4_gemm_tokens")
    return c


def mxfp4_gemm_workspace_size(M: int, N: int, K: int, path: int = 0, splits: int = 0, m_tile: int = 0) -> int:
    return int(load_library().mxfp4_gemm_workspace_size_ex(M, N, K, _opts(path, splits, m_tile)))


_WS_NEED: dict = {}


def _ws_need(device: torch.device, M: int, N: int, K: int, path: int = 0, splits: int = 0, m_tile: int = 0) -> int:
    """mxfp4_gemm_workspace_size, remembered per (device, shape, options): the plan depends only on
    those, and the per-call query would otherwise cost a library round trip on every GEMM."""
    key = (device.index, M, N, K, path, splits, m_tile)
    need = _WS_NEED.get(key)
    if need is None:
        need = mxfp4_gemm_workspace_size(M, N, K, path, splits, m_tile) if M and N else 0
        _WS_NEED[key] = need
    return need


_PACKED_NEED: dict = {}


def _check_packed(packed_b: torch.Tensor, N: int, K: int, device: torch.device | None) -> None:
    """The packed weights must cover mxfp4_prepack_b_size(N, K) bytes on the GEMM's device: the
    kernel streams that many bytes, so a smaller buffer would be read past its end. `device`
    None checks only that the buffer is on a CUDA device (the per-step host call)."""
    need = _PACKED_NEED.get((N, K))
    if need is None:
        need = mxfp4_prepack_b_size(N, K)
        _PACKED_NEED[(N, K)] = need
    if need == 0 or packed_b.nbytes < need or not packed_b.is_cuda or (device is not None and packed_b.device != device):
        raise ValueError(f"packed_b must be a CUDA buffer of at least mxfp4_prepack_b_size({N}, {K}) = {need} bytes"
                         " on the device of the other operands")


def mxfp4_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(load_library().mxfp4_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "mxfp4_workspace_init")


def _workspace(device: torch.device, nbytes: int, stream, st: int) -> torch.Tensor | None:
    """A zero-initialised workspace of at least nbytes per (device, stream), grown on demand.
    One per stream: calls sharing a workspace must be ordered, and calls on different streams
    need not be. A workspace used on a stream other than the current one is recorded on it, so
    that growing it never hands its memory to other work while that stream may still use it."""
    if nbytes == 0:
        return None
    dev_index = device.index if device.index is not None else torch.cuda.current_device()
    key = (dev_index, st)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        if st != torch.cuda.current_stream(dev_index).cuda_stream:
            ws.record_stream(torch.cuda.ExternalStream(st, device=device))
        mxfp4_workspace_init(ws, stream)
        _WS[key] = ws
    return ws


def _gemm_call_args(a, packed_b, N, c, workspace, path, splits, stream, m_tile, a_ready=False) -> tuple:
    """(C, the checked arguments of one mxfp4_gemm_ex call in C order)."""
    L = load_library()
    _dev(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    M, K = a.shape
    if M and N:
        _check_packed(packed_b, N, K, a.device)
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _on(c, a.device, "c")
    if c.dtype != torch.bfloat16 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be a bf16 [M, N] tensor with unit column stride")
    st = _stream(stream)
    if workspace is not None:
        _on(workspace, a.device, "workspace")
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
    else:
        dev = a.device
        need = _ws_need(dev, M, N, K, path, splits, m_tile)
        workspace = _workspace(dev, need, stream, st) if need else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    flags = GEMM_A_READY if a_ready else 0
    # NULL: the automatic plan without flags
    opts = _opts(path, splits, m_tile, flags) if (path or splits or m_tile or flags) else None
    return c, (a.data_ptr(), M, K, a.stride(0), packed_b.data_ptr(), N, c.data_ptr(), c.stride(0), ws_ptr, ws_bytes,
               opts, st), workspace


def mxfp4_gemm(a: torch.Tensor, packed_b: torch.Tensor, N: int, c: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, path: int = 0, splits: int = 0,
               stream=None, m_tile: int = 0, a_ready: bool = False) -> torch.Tensor:
    """C [M, N] bf16 = MXFP4(a) . MXFP4(B)^T, `packed_b` from mxfp4_prepack_b. a_ready: the
    caller guarantees MXFP4_GEMM_A_READY (every write to `a` finished before the operation just
    before this call on the stream began to run), so the kernels read A without waiting for it."""
    c, args, _ = _gemm_call_args(a, packed_b, N, c, workspace, path, splits, stream, m_tile, a_ready)
    _check(load_library().mxfp4_gemm_ex(*args), "mxfp4_gemm")
    return c


def _host_call_args(a_host, packed_b, N, c_host, a_dev, c_dev, workspace, stream) -> tuple:
    """The checked arguments of one mxfp4_gemm_host call, in C order."""
    L = load_library()
    # every tensor property is read once: this call sits on the per-step host path
    bf16 = torch.bfloat16
    if a_host.dtype != bf16 or c_host.dtype != bf16 or a_dev.dtype != bf16 or c_dev.dtype != bf16:
        raise ValueError("a_host, c_host, a_dev and c_dev must be bf16 tensors")
    if a_host.is_cuda or c_host.is_cuda or not a_dev.is_cuda or not c_dev.is_cuda:
        raise ValueError("a_host and c_host must be host tensors, a_dev and c_dev CUDA tensors")
    a_shape, c_shape = a_host.shape, c_host.shape
    a_stride, c_stride = a_host.stride(), c_host.stride()
    if len(a_shape) != 2 or len(c_shape) != 2 or a_stride[1] != 1 or c_stride[1] != 1:
        raise ValueError("a_host and c_host must be 2-D with unit column stride")
    M, K = a_shape
    if tuple(c_shape) != (M, N):
        raise ValueError("c_host must be [M, N]")
    if M and N:
        _check_packed(packed_b, N, K, None)
    if a_dev.shape != (M, K) or a_dev.stride() != (K, 1) or c_dev.shape != (M, N) or c_dev.stride() != (N, 1):
        raise ValueError("a_dev must be a packed [M, K] and c_dev a packed [M, N] tensor")
    st = _stream(stream)
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
    else:
        dev = a_dev.device
        need = _ws_need(dev, M, N, K)
        workspace = _workspace(dev, need, stream, st) if need else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return (a_host.data_ptr(), M, K, a_stride[0], packed_b.data_ptr(), N, c_host.data_ptr(), c_stride[0],
            a_dev.data_ptr(), c_dev.data_ptr(), ws_ptr, ws_bytes, st)


def mxfp4_gemm_host(a_host: torch.Tensor, packed_b: torch.Tensor, N: int, c_host: torch.Tensor,
                    a_dev: torch.Tensor, c_dev: torch.Tensor, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """mxfp4_gemm_host: A and C in (preferably pinned) host memory, device staging buffers a_dev
    [M, K] and c_dev [M, N] from the caller; asynchronous on `stream`. Returns c_host."""
    args = _host_call_args(a_host, packed_b, N, c_host, a_dev, c_dev, workspace, stream)
    _check(load_library().mxfp4_gemm_host(*args), "mxfp4_gemm_host")
    return c_host


class PreparedCall:
    """A GEMM call whose buffers stay the same from one call to the next (a serving loop with
    fixed input and output buffers), prepared in the library (mxfp4_call_create*): its checks,
    plan and host-buffer queries are done once, and each call only enqueues its kernels and
    copies on the stream given when it was prepared. The tensors are kept alive by this object;
    the caller must not resize or replace their storage while it is in use. Calling it raises
    Mxfp4Error if the library refuses the run."""

    __slots__ = ("_run", "_handle", "_stream", "_where", "_keep", "_destroy")

    def __init__(self, create, args: tuple, stream: int, where: str, keep: tuple):
        L = load_library()
        handle = ctypes.c_void_p()
        _check(create(*args, ctypes.byref(handle)), where)
        self._run, self._destroy = L.mxfp4_call_run, L.mxfp4_call_destroy
        self._handle, self._stream, self._where, self._keep = handle.value, stream, where, keep

    def __call__(self) -> None:
        st = self._run(self._handle, self._stream)
        if st != 0:
            raise Mxfp4Error(st, self._where)

    def __del__(self):
        handle, self._handle = getattr(self, "_handle", None), None
        if handle:
            self._destroy(handle)


def prepare_gemm(a: torch.Tensor, packed_b: torch.Tensor, N: int, c: torch.Tensor,
                 workspace: torch.Tensor | None = None, path: int = 0, splits: int = 0,
                 stream=None, m_tile: int = 0, a_ready: bool = False) -> PreparedCall:
    """mxfp4_gemm prepared for repeated calls on the same buffers (see PreparedCall); `c` is
    required, the other arguments are those of mxfp4_gemm (a_ready holds for every run)."""
    c, args, ws = _gemm_call_args(a, packed_b, N, c, workspace, path, splits, stream, m_tile, a_ready)
    return PreparedCall(load_library().mxfp4_call_create, args[:-1], args[-1], "mxfp4_call_create",
                        (a, packed_b, c, ws))


def prepare_gemm_host(a_host: torch.Tensor, packed_b: torch.Tensor, N: int, c_host: torch.Tensor,
                      a_dev: torch.Tensor, c_dev: torch.Tensor, workspace: torch.Tensor | None = None,
                      stream=None, a_host_written: bool = False) -> PreparedCall:
    """mxfp4_gemm_host prepared for repeated calls on the same buffers (see PreparedCall); the
    arguments are those of mxfp4_gemm_host. a_host_written: the caller guarantees that a_host is
    written by the host only, never by device work (MXFP4_CALL_A_HOST_WRITTEN), so A crosses the
    link while the work before the call still runs."""
    args = _host_call_args(a_host, packed_b, N, c_host, a_dev, c_dev, workspace, stream)
    keep = (a_host, packed_b, c_host, a_dev, c_dev, workspace)
    flags = 1 if a_host_written else 0
    return PreparedCall(load_library().mxfp4_call_create_host, args[:-1] + (flags,), args[-1],
                        "mxfp4_call_create_host", keep)


def mxfp4_gemm_unpacked(a: torch.Tensor, bq: torch.Tensor, bs: torch.Tensor, c: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """mxfp4_gemm on B as mxfp4_quantize writes it (e2m1 [N, nblk*16], e8m0 [N, nblk], nblk =
    ceil(K/32)): the call writes B's packed image into its workspace, then runs the GEMM
    (mxfp4_gemm_unpacked). `workspace`, if given: a contiguous CUDA byte buffer of at least
    mxfp4_gemm_unpacked_workspace_size bytes starting 1024-byte aligned."""
    L = load_library()
    _dev(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    M, K = a.shape
    _on(bq, a.device, "bq")
    _on(bs, a.device, "bs")
    N = bq.shape[0] if bq.dim() == 2 else -1
    nblk = -(-K // 32)
    if (bq.dim() != 2 or tuple(bq.shape) != (N, nblk * 16) or tuple(bs.shape) != (N, nblk)
            or not bq.is_contiguous() or not bs.is_contiguous() or bq.element_size() != 1 or bs.element_size() != 1):
        raise ValueError("bq [N, ceil(K/32)*16] and bs [N, ceil(K/32)] must be contiguous byte tensors")
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _on(c, a.device, "c")
    if c.dtype != torch.bfloat16 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be a bf16 [M, N] tensor with unit column stride")
    st = _stream(stream)
    need = L.mxfp4_gemm_unpacked_workspace_size(M, N, K) if M and N else 0
    if workspace is None:
        ws = _workspace(a.device, need + 1024, stream, st) if need else None
        workspace = ws[(-ws.data_ptr()) % 1024:][:need] if ws is not None else None
    elif (not workspace.is_cuda or not workspace.is_contiguous() or workspace.device != a.device
          or workspace.nbytes < need):
        raise ValueError(f"workspace must be a contiguous buffer of at least {need} bytes on {a.device}")
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.nbytes if workspace is not None else 0
    _check(L.mxfp4_gemm_unpacked(a.data_ptr(), M, K, a.stride(0), bq.data_ptr(), bs.data_ptr(), N, c.data_ptr(),
                                 c.stride(0), ws_ptr, ws_bytes, st), "mxfp4_gemm_unpacked")
    return c


def mxfp4_gemm_noalloc(a: torch.Tensor, packed_b: torch.Tensor, N: int, c: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """mxfp4_gemm without a workspace: the automatic plan with the library's own fixed scratch
    (for callers that must not allocate device memory; calls on one device must be ordered)."""
    L = load_library()
    _dev(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    M, K = a.shape
    if M and N:
        _check_packed(packed_b, N, K, a.device)
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _on(c, a.device, "c")
    if c.dtype != torch.bfloat16 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be a bf16 [M, N] tensor with unit column stride")
    _check(L.mxfp4_gemm_noalloc(a.data_ptr(), M, K, a.stride(0), packed_b.data_ptr(), N, c.data_ptr(), c.stride(0),
                                _stream(stream)), "mxfp4_gemm_noalloc")
    return c


_PLAN_FIELDS = ("path", "splits", "m_tile", "ctas", "stages", "issuers", "reduction", "recv_dedicated",
                "smem_bytes", "tmem_cols", "scale_stores", "a_early")


class _PlanInfo(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in _PLAN_FIELDS] + [("reserved", ctypes.c_int * 4)]


def mxfp4_gemm_plan(M: int, N: int, K: int, path: int = 0, splits: int = 0, m_tile: int = 0,
                    a_ready: bool = False) -> dict:
    """The plan mxfp4_gemm would run (with a_ready: the plan of a call that declares A ready), as
    a dict of the mxfp4_plan_info fields."""
    L = load_library()
    info = _PlanInfo()
    _check(L.mxfp4_gemm_plan_info(M, N, K, _opts(path, splits, m_tile, GEMM_A_READY if a_ready else 0),
                                  ctypes.byref(info)), "mxfp4_gemm_plan_info")
    return {name: getattr(info, name) for name in _PLAN_FIELDS}


def mxfp4_gemm_plan_model(M: int, N: int, K: int, sm_count: int, cluster_caps=None, path: int = 0,
                          splits: int = 0, m_tile: int = 0, a_ready: bool = False) -> dict:
    """The planner alone for a described device (no GPU needed): `cluster_caps` lists, for cluster
    sizes 1..16, how many clusters can be resident at once (None: no limit)."""
    L = load_library()
    info = _PlanInfo()
    caps = None
    if cluster_caps is not None:
        caps = (ctypes.c_int * 17)(0, *[int(c) for c in cluster_caps])
    _check(L.mxfp4_gemm_plan_model(M, N, K, _opts(path, splits, m_tile, GEMM_A_READY if a_ready else 0), sm_count,
                                   caps, ctypes.byref(info)),
           "mxfp4_gemm_plan_model")
    return {name: getattr(info, name) for name in _PLAN_FIELDS}


def mxfp4_device_status(stream=None) -> int:
    return int(load_library().mxfp4_device_status(_stream(stream)))


def mxfp4_selftest_timeout(limit_us: int, stream=None) -> None:
    _check(load_library().mxfp4_selftest_timeout(limit_us, _stream(stream)), "mxfp4_selftest_timeout")

"""Thin ctypes binding of libgptq_gb300.so, with the C ABI's names.

Argument marshalling only: torch tensors are passed as raw device pointers plus sizes,
every step of the computation runs in the library's CUDA kernels.  A missing or
unloadable library raises ``GptqLibraryError``; there is no other code path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "GPTQ_OK", "GPTQ_ERR_INVALID_ARG", "GPTQ_ERR_UNSUPPORTED", "GPTQ_ERR_NOT_PD",
    "GPTQ_ERR_NONFINITE", "GPTQ_ERR_CUDA", "GPTQ_ERR_TIMEOUT", "GPTQ_ERR_WORKSPACE",
    "GPTQ_F32", "GPTQ_BF16", "GPTQ_OP_HESSIAN", "GPTQ_OP_PREPARE", "GPTQ_OP_QUANTIZE",
    "GPTQ_OP_DEQUANT_MATMUL", "gptq_dequant_matmul", "gptq_dequantize",
    "GptqError", "GptqLibraryError", "lib", "library_path",
    "gptq_workspace_size", "gptq_hessian_accumulate", "gptq_hessian_accumulate_async",
    "gptq_hessian_status", "gptq_hessian_rescale", "gptq_check_wait_timeout", "gptq_set_wait_limit", "gptq_scales_fp16",
    "gptq_prepare", "gptq_quantize_layer",
    "gptq_last_error", "gptq_status_string", "gptq_abi_version",
    "gptq_profile_enable", "gptq_profile_select", "gptq_profile_read", "gptq_profile_reset",
    "gptq_kernel_name",
    "gptq_launch_count", "KERNEL_KINDS", "GPTQ_K_SYRK_TC", "GPTQ_K_DEQUANT_MATMUL",
    "GPTQ_QUANT_STATIC_GROUPS", "gptq_layer_host_size", "gptq_quantize_layer_host",
    "workspace",
]

GPTQ_OK, GPTQ_ERR_INVALID_ARG, GPTQ_ERR_UNSUPPORTED, GPTQ_ERR_NOT_PD = 0, 1, 2, 3
GPTQ_ERR_NONFINITE, GPTQ_ERR_CUDA, GPTQ_ERR_TIMEOUT, GPTQ_ERR_WORKSPACE = 4, 5, 6, 7
GPTQ_F32, GPTQ_BF16 = 0, 1
GPTQ_OP_HESSIAN, GPTQ_OP_PREPARE, GPTQ_OP_QUANTIZE, GPTQ_OP_DEQUANT_MATMUL = 0, 1, 2, 3
KERNEL_KINDS = 24
GPTQ_K_SYRK_TC = 0  # the gptq_kernel_kind of the tensor-core SYRK
GPTQ_K_DEQUANT_MATMUL = 20
GPTQ_QUANT_STATIC_GROUPS = 1


class GptqLibraryError(RuntimeError):
    """The CUDA library is missing or cannot be loaded."""


class GptqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{gptq_status_string(status)}: {message}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None

_c = ctypes
_vp, _sz, _i64, _i32, _f32 = _c.c_void_p, _c.c_size_t, _c.c_int64, _c.c_int32, _c.c_float
_SIGS = {
    "gptq_workspace_size": (_sz, [_c.c_int, _i64, _i32, _i32, _c.c_int, _c.c_int]),
    "gptq_hessian_accumulate": (_c.c_int, [_vp, _c.POINTER(_i64), _vp, _c.c_int, _i64, _i32,
                                           _vp, _sz, _vp]),
    "gptq_hessian_accumulate_noalloc": (_c.c_int, [_vp, _c.POINTER(_i64), _vp, _c.c_int,
                                                   _i64, _i32, _vp]),
    "gptq_hessian_accumulate_async": (_c.c_int, [_vp, _c.POINTER(_i64), _vp, _c.c_int, _i64,
                                                 _i32, _vp, _sz, _vp]),
    "gptq_hessian_status": (_c.c_int, [_vp, _sz, _vp]),
    "gptq_hessian_rescale": (_c.c_int, [_vp, _i32, _i64, _i64, _vp]),
    "gptq_check_wait_timeout": (_c.c_int, [_c.c_uint64, _vp, _sz, _vp]),
    "gptq_set_wait_limit": (_c.c_int, [_c.c_uint64]),
    "gptq_scales_fp16": (_c.c_int, [_vp, _i64, _vp, _vp]),
    "gptq_prepare": (_c.c_int, [_vp, _i32, _f32, _c.c_int, _vp, _vp, _vp, _c.POINTER(_i32),
                                _vp, _sz, _vp]),
    "gptq_quantize_layer": (_c.c_int, [_vp, _c.c_int, _vp, _vp, _vp, _i32, _i32, _c.c_int,
                                       _c.c_int, _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _sz, _vp]),
    "gptq_quantize_layer_ex": (_c.c_int, [_vp, _c.c_int, _vp, _vp, _vp, _i32, _i32, _c.c_int,
                                          _c.c_int, _c.c_int, _c.c_int, _c.c_int, _vp, _vp,
                                          _vp, _vp, _vp, _vp, _sz, _vp]),
    "gptq_layer_host_size": (_sz, [_i64, _i32, _i32, _c.c_int, _c.c_int, _c.c_int, _c.c_int]),
    "gptq_quantize_layer_host": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _vp, _c.c_int, _i32, _i32,
                                            _f32, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                            _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp,
                                            _c.POINTER(_c.c_double), _c.POINTER(_i32), _vp, _sz,
                                            _vp]),
    "gptq_dequant_matmul": (_c.c_int, [_vp, _c.c_int, _i64, _i32, _i32, _c.c_int, _vp, _vp,
                                       _vp, _vp, _i32, _vp, _vp, _sz, _vp]),
    "gptq_dequantize": (_c.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _c.c_int, _i32, _vp,
                                   _c.c_int, _vp, _sz, _vp]),
    "gptq_last_error": (_c.c_char_p, []),
    "gptq_status_string": (_c.c_char_p, [_c.c_int]),
    "gptq_abi_version": (_c.c_int, []),
    "gptq_profile_enable": (None, [_c.c_int]),
    "gptq_profile_select": (None, [_c.c_uint32]),
    "gptq_profile_read": (_c.c_int, [_c.c_int, _c.POINTER(_c.c_double), _c.POINTER(_i64)]),
    "gptq_profile_reset": (None, []),
    "gptq_kernel_name": (_c.c_char_p, [_c.c_int]),
    "gptq_launch_count": (_i64, []),
}


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load (building in-tree if needed) and return the library."""
    global _lib
    if _lib is None:
        try:
            path = _build.ensure_built()
            handle = ctypes.CDLL(path)
        except Exception as e:  # no nvcc, failed build, wrong architecture
            raise GptqLibraryError(f"libgptq_gb300.so unavailable: {e}") from e
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _buf(t: Optional[torch.Tensor], dtype, numel: Optional[int], name: str) -> Optional[int]:
    """Device pointer of a caller buffer, after checking its element type and (when known)
    its number of elements: the library reads raw memory and cannot check either."""
    if t is None:
        return None
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")
    return _ptr(t)


def _ngroups(d: int, group: int) -> Optional[int]:
    """Rows of scales / qzeros for a valid group size (None: left to the library)."""
    if group == -1:
        return 1
    return -(-d // group) if group > 0 else None


def _packed(bits: int, count: int) -> Optional[int]:
    """32-bit words of `count` codes of `bits` bits (None: bits left to the library)."""
    return bits * count // 32 if bits in (2, 3, 4, 8) else None


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int):
    if status != GPTQ_OK:
        raise GptqError(status, gptq_last_error())


def gptq_last_error() -> str:
    return lib().gptq_last_error().decode()


def gptq_status_string(status: int) -> str:
    return lib().gptq_status_string(int(status)).decode()


def gptq_abi_version() -> int:
    return lib().gptq_abi_version()


def gptq_workspace_size(op: int, ntok: int, d_out: int, d_in: int, bits: int = 4,
                        group: int = 128) -> int:
    return int(lib().gptq_workspace_size(op, ntok, d_out, d_in, bits, group))


def workspace(nbytes: int, device) -> torch.Tensor:
    """Caller-owned workspace (torch allocates; the library never does)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GPTQ_BF16
    if t.dtype == torch.float32:
        return GPTQ_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def gptq_hessian_accumulate(H: torch.Tensor, nseen: int, X: torch.Tensor,
                            ws: Optional[torch.Tensor] = None, stream=None) -> int:
    """One hook step on device tensors H [d, d] float32 and X [t, d]; returns the new n."""
    d = H.shape[0]
    if X.dim() != 2 or X.shape[1] != d:
        raise ValueError("X must be [ntok, d_in]")
    pH = _buf(H, torch.float32, d * d, "H")
    if ws is None:
        ws = workspace(gptq_workspace_size(GPTQ_OP_HESSIAN, X.shape[0], 0, d), H.device)
    n = ctypes.c_int64(int(nseen))
    _check(lib().gptq_hessian_accumulate(pH, ctypes.byref(n), _ptr(X) if X.numel() else None,
                                         _dtype_code(X), X.shape[0], d, _ptr(ws), ws.numel(),
                                         _stream(stream)))
    return int(n.value)


def gptq_hessian_accumulate_async(H: torch.Tensor, nseen: int, X: torch.Tensor,
                                  ws: torch.Tensor, stream=None) -> int:
    """Enqueue one hook step without waiting; returns the new n.  Device-side failures
    are reported by gptq_hessian_status on the same workspace."""
    d = H.shape[0]
    if X.dim() != 2 or X.shape[1] != d:
        raise ValueError("X must be [ntok, d_in]")
    pH = _buf(H, torch.float32, d * d, "H")
    n = ctypes.c_int64(int(nseen))
    _check(lib().gptq_hessian_accumulate_async(pH, ctypes.byref(n),
                                               _ptr(X) if X.numel() else None, _dtype_code(X),
                                               X.shape[0], d, _ptr(ws), ws.numel(),
                                               _stream(stream)))
    return int(n.value)


def gptq_hessian_status(ws: torch.Tensor, stream=None) -> None:
    """Synchronise the stream; raise the first failure of the async Hessian steps on ws."""
    _check(lib().gptq_hessian_status(_ptr(ws), ws.numel(), _stream(stream)))


def gptq_hessian_rescale(H: torch.Tensor, n_from: int, n_to: int, stream=None) -> None:
    """H <- H * n_from / n_to on the upper tiles (a partial Hessian's share of a stream of
    n_to tokens)."""
    d = H.shape[0]
    _check(lib().gptq_hessian_rescale(_buf(H, torch.float32, d * d, "H"), d, int(n_from),
                                      int(n_to), _stream(stream)))


def gptq_check_wait_timeout(limit_ns: int, ws: torch.Tensor, stream=None) -> None:
    """Run the library's bounded device wait on an mbarrier nothing arrives on; raises
    GptqError with GPTQ_ERR_TIMEOUT when the wait gives up, as it must."""
    _check(lib().gptq_check_wait_timeout(int(limit_ns), _ptr(ws), ws.numel(), _stream(stream)))


def gptq_set_wait_limit(limit_ns: int) -> None:
    """Limit of the tensor-core kernels' device waits for later calls in this process (0:
    the default, 2 s).  A diagnostic: with a limit of a few nanoseconds the waits run out,
    the kernel drains what it issued and the call raises GptqError(GPTQ_ERR_TIMEOUT)."""
    _check(lib().gptq_set_wait_limit(int(limit_ns)))


def gptq_scales_fp16(scales: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """The checkpoint's fp16 copy of float32 scales (device tensors), rounded to nearest
    even; returns ``out`` (allocated like ``scales`` when not given)."""
    if out is None:
        out = torch.empty(scales.shape, dtype=torch.float16, device=scales.device)
    n = scales.numel()
    ps = _buf(scales, torch.float32, n, "scales")
    po = _buf(out, torch.float16, n, "out")
    _check(lib().gptq_scales_fp16(ps, n, po, _stream(stream)))
    return out


def gptq_prepare(H: torch.Tensor, damp: float, actorder: bool, perm: torch.Tensor,
                 dead: torch.Tensor, Hinv_chol: torch.Tensor, ws: Optional[torch.Tensor] = None,
                 stream=None) -> int:
    """Dead fix, act-order, damping, U; returns info (0, or the failing pivot)."""
    d = H.shape[0]
    ptrs = (_buf(H, torch.float32, d * d, "H"), _buf(perm, torch.int32, d, "perm"),
            _buf(dead, torch.uint8, d, "dead"), _buf(Hinv_chol, torch.float32, d * d, "Hinv_chol"))
    if ws is None:
        ws = workspace(gptq_workspace_size(GPTQ_OP_PREPARE, 0, 0, d), H.device)
    info = ctypes.c_int32(0)
    st = lib().gptq_prepare(ptrs[0], d, float(damp), int(bool(actorder)), ptrs[1], ptrs[2],
                            ptrs[3], ctypes.byref(info), _ptr(ws), ws.numel(),
                            _stream(stream))
    if st != GPTQ_OK:
        err = GptqError(st, gptq_last_error())
        err.info = int(info.value)
        raise err
    return int(info.value)


def gptq_quantize_layer(W: torch.Tensor, Hinv_chol: torch.Tensor, perm: Optional[torch.Tensor],
                        dead: Optional[torch.Tensor], bits: int, group: int, sym: bool,
                        blocksize: int, qweight: torch.Tensor, scales: torch.Tensor,
                        qzeros: torch.Tensor, g_idx: torch.Tensor, loss: torch.Tensor,
                        ws: Optional[torch.Tensor] = None, stream=None,
                        static_groups: bool = False) -> None:
    """The column loop and packing; ``static_groups`` fits the groups in the original
    column order before the loop (gptq_quantize_layer_ex, GPTQ_QUANT_STATIC_GROUPS)."""
    m, d = W.shape
    G = _ngroups(d, group)
    words = _packed(bits, d)
    zwords = _packed(bits, m)
    ptrs = (_buf(Hinv_chol, torch.float32, d * d, "Hinv_chol"),
            _buf(perm, torch.int32, d, "perm"), _buf(dead, torch.uint8, d, "dead"),
            _buf(qweight, torch.int32, None if words is None else words * m, "qweight"),
            _buf(scales, torch.float32, None if G is None else G * m, "scales"),
            _buf(qzeros, torch.int32, None if G is None or zwords is None else G * zwords,
                 "qzeros"),
            _buf(g_idx, torch.int32, d, "g_idx"), _buf(loss, torch.float64, 1, "loss"))
    if ws is None:
        ws = workspace(gptq_workspace_size(GPTQ_OP_QUANTIZE, 0, m, d, bits, group), W.device)
    flags = GPTQ_QUANT_STATIC_GROUPS if static_groups else 0
    _check(lib().gptq_quantize_layer_ex(_ptr(W), _dtype_code(W), ptrs[0], ptrs[1], ptrs[2], m, d,
                                        bits, group, int(bool(sym)), blocksize, flags, *ptrs[3:],
                                        _ptr(ws), ws.numel(), _stream(stream)))


def _hbuf(t: torch.Tensor, dtype, numel: int, name: str) -> int:
    """Host pointer of a caller buffer (a contiguous CPU tensor) after checking its type
    and size."""
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")
    return t.data_ptr()


def gptq_layer_host_size(chunk_tokens: int, d_out: int, d_in: int, bits: int, group: int,
                         xdtype: int, wdtype: int) -> int:
    return int(lib().gptq_layer_host_size(chunk_tokens, d_out, d_in, bits, group, xdtype,
                                          wdtype))


def gptq_quantize_layer_host(X: torch.Tensor, W: torch.Tensor, chunk_tokens: int, damp: float,
                             actorder: bool, bits: int, group: int, sym: bool, blocksize: int,
                             qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor,
                             g_idx: torch.Tensor, perm: torch.Tensor, dev: torch.Tensor,
                             stream=None, static_groups: bool = False):
    """The whole layer from host tensors X [ntok, d_in] and W [d_out, d_in] (page-locked
    for overlapped copies) into host outputs; ``dev`` is the caller's device buffer of
    gptq_layer_host_size bytes.  Returns (loss, info)."""
    if X.dim() != 2 or W.dim() != 2 or X.shape[1] != W.shape[1]:
        raise ValueError("X must be [ntok, d_in] and W [d_out, d_in]")
    m, d = W.shape
    G, words, zwords = _ngroups(d, group), _packed(bits, d), _packed(bits, m)
    if G is None or words is None or zwords is None:
        raise ValueError("unsupported bits or group")
    px = _hbuf(X, X.dtype, X.numel(), "X")
    pw = _hbuf(W, W.dtype, W.numel(), "W")
    outs = (_hbuf(qweight, torch.int32, words * m, "qweight"),
            _hbuf(scales, torch.float32, G * m, "scales"),
            _hbuf(qzeros, torch.int32, G * zwords, "qzeros"),
            _hbuf(g_idx, torch.int32, d, "g_idx"), _hbuf(perm, torch.int32, d, "perm"))
    loss = ctypes.c_double(0.0)
    info = ctypes.c_int32(0)
    flags = GPTQ_QUANT_STATIC_GROUPS if static_groups else 0
    st = lib().gptq_quantize_layer_host(px, _dtype_code(X), X.shape[0], int(chunk_tokens), pw,
                                        _dtype_code(W), m, d, float(damp), int(bool(actorder)),
                                        bits, group, int(bool(sym)), blocksize, flags, *outs,
                                        ctypes.byref(loss), ctypes.byref(info), _ptr(dev),
                                        dev.numel(), _stream(stream))
    if st != GPTQ_OK:
        err = GptqError(st, gptq_last_error())
        err.info = int(info.value)
        raise err
    return float(loss.value), int(info.value)


def _checkpoint_ptrs(qweight, scales, qzeros, g_idx, bits: int, m: int, d: int):
    """Pointers of a packed checkpoint after checking types and sizes (G = rows of scales)."""
    G = scales.shape[0] if scales.dim() == 2 else None
    words, zwords = _packed(bits, d), _packed(bits, m)
    return (_buf(qweight, torch.int32, None if words is None else words * m, "qweight"),
            _buf(scales, torch.float32, None if G is None else G * m, "scales"),
            _buf(qzeros, torch.int32, None if G is None or zwords is None else G * zwords,
                 "qzeros"),
            _buf(g_idx, torch.int32, d, "g_idx"))


def gptq_dequant_matmul(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                        qzeros: torch.Tensor, g_idx: torch.Tensor, bits: int,
                        y: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """y = x W_hat^T from the packed checkpoint (x [n, d_in] bf16 or fp32; y [n, d_out])."""
    if x.dim() != 2:
        raise ValueError("x must be [n, d_in]")
    n, d = x.shape
    m = qweight.shape[1]
    if y is None:
        y = torch.empty(n, m, dtype=torch.float32, device=x.device)
    ptrs = _checkpoint_ptrs(qweight, scales, qzeros, g_idx, bits, m, d)
    py = _buf(y, torch.float32, n * m, "y")
    if ws is None:
        ws = workspace(gptq_workspace_size(GPTQ_OP_DEQUANT_MATMUL, 0, m, d, bits, -1), x.device)
    _check(lib().gptq_dequant_matmul(_ptr(x) if x.numel() else None, _dtype_code(x), n, d, m,
                                     bits, *ptrs, scales.shape[0], py, _ptr(ws),
                                     ws.numel(), _stream(stream)))
    return y


def gptq_dequantize(qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor,
                    g_idx: torch.Tensor, bits: int, dtype=torch.bfloat16,
                    W: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """W_hat [d_out, d_in] (bf16 or fp32) from the packed checkpoint."""
    m = qweight.shape[1]
    d = qweight.shape[0] * 32 // bits
    if W is None:
        W = torch.empty(m, d, dtype=dtype, device=qweight.device)
    ptrs = _checkpoint_ptrs(qweight, scales, qzeros, g_idx, bits, m, d)
    if W.numel() != m * d:
        raise ValueError(f"W must hold {m * d} elements, got {W.numel()}")
    if ws is None:
        ws = workspace(gptq_workspace_size(GPTQ_OP_DEQUANT_MATMUL, 0, m, d, bits, -1),
                       qweight.device)
    _check(lib().gptq_dequantize(*ptrs, m, d, bits, scales.shape[0], _ptr(W), _dtype_code(W),
                                 _ptr(ws), ws.numel(), _stream(stream)))
    return W


def gptq_profile_enable(on: bool) -> None:
    lib().gptq_profile_enable(int(bool(on)))


def gptq_profile_select(kinds) -> None:
    """Trace only the given kernel kinds (an iterable of kinds, or None for all)."""
    mask = 0xFFFFFFFF if kinds is None else sum(1 << int(k) for k in kinds)
    lib().gptq_profile_select(mask)


def gptq_profile_reset() -> None:
    lib().gptq_profile_reset()


def gptq_profile_read(kind: int):
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int64(0)
    if lib().gptq_profile_read(kind, ctypes.byref(ms), ctypes.byref(n)) != 0:
        raise ValueError(kind)
    return float(ms.value), int(n.value)


def gptq_kernel_name(kind: int) -> str:
    return lib().gptq_kernel_name(kind).decode()


def gptq_launch_count() -> int:
    return int(lib().gptq_launch_count())

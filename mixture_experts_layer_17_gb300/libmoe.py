"""ctypes binding of libmoe (include/moe.h), with the same entry-point names.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and the
stream); they must be contiguous and of the dtype the C ABI expects.  A
missing library raises at once: there is no other code path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Tuple

import torch

from .build import LIB_PATH

MOE_BF16, MOE_MXFP8, MOE_FP8_BWD = 0, 1, 2
PRECISIONS = {"bf16": MOE_BF16, "mxfp8": MOE_MXFP8, "fp8_bwd": MOE_FP8_BWD}
MOE_FLAG_SYNC_CHECK = 0x1
MOE_FLAG_TEST_TIMEOUT = 0x2
MOE_FLAG_CTA_PAIRS_OFF = 0x4
MOE_FLAG_CTA_PAIRS_ON = 0x8
MOE_FLAG_RECOMPUTE = 0x10

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
          3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
          6: "MOE_ERR_UNSUPPORTED_DEVICE", 7: "MOE_ERR_NOT_IMPLEMENTED"}

# every symbol include/moe.h declares
EXPORTED = ("moe_workspace_size", "moe_route", "moe_forward", "moe_backward", "moe_gemm_bf16",
            "moe_get_device_status", "moe_status_string", "moe_profile_enable",
            "moe_profile_read", "moe_profile_select", "moe_launch_count", "moe_route_noalloc",
            "moe_gemm_mxfp8",
            "moe_backward_accumulate", "moe_prepared_weights_size", "moe_prepare_weights")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("precision", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("max_sms", ctypes.c_int32),
                ("prepared_weights", ctypes.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_lib: Optional[ctypes.CDLL] = None
_vp, _sz, _i64, _i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libmoe.so (built by __graft_entry__.build()), or the library that
    LIBMOE_PATH names (such as the index-checking debug build); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = os.environ.get("LIBMOE_PATH") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    cfgp = ctypes.POINTER(MoeConfig)
    sig = {
        "moe_workspace_size": [cfgp, ctypes.POINTER(_sz), ctypes.POINTER(_sz), ctypes.POINTER(_sz)],
        "moe_route": [cfgp] + [_vp] * 10 + [_sz, _vp],
        "moe_forward": [cfgp] + [_vp] * 9 + [_sz, _vp],
        "moe_backward": [cfgp] + [_vp] * 13 + [_sz, _vp],
        "moe_backward_accumulate": [cfgp] + [_vp] * 13 + [_sz, _vp],
        "moe_prepared_weights_size": [cfgp, ctypes.POINTER(_sz)],
        "moe_prepare_weights": [cfgp, _vp, _vp, _vp, _vp, _sz, _vp],
        "moe_gemm_bf16": [_i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _vp, _sz, _vp],
        "moe_get_device_status": [_vp, _vp],
        "moe_status_string": [_i32],
        "moe_profile_enable": [_i32],
        "moe_profile_select": [ctypes.c_char_p],
        "moe_profile_read": [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_i64),
                             ctypes.POINTER(ctypes.c_double), _i32],
        "moe_launch_count": [],
        "moe_route_noalloc": [cfgp] + [_vp] * 11 + [_vp],
        "moe_gemm_mxfp8": [_i64, _i64, _i64, _vp, _vp, _vp, _vp, ctypes.POINTER(_sz), _vp],
    }
    for name, argtypes in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = _i32
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_launch_count.restype = _i64
    lib.moe_profile_enable.restype = None
    lib.moe_profile_select.restype = None
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(code: int, where: str) -> None:
    if code != 0:
        raise MoeError(code, where)


def make_config(T: int, H: int, F: int, E: int, top_k: int, precision="bf16",
                flags: int = 0, max_sms: int = 0) -> MoeConfig:
    prec = PRECISIONS[precision] if isinstance(precision, str) else int(precision)
    return MoeConfig(T, H, F, E, top_k, prec, flags, max_sms)


def moe_workspace_size(cfg: MoeConfig) -> Tuple[int, int, int]:
    f, c, b = _sz(), _sz(), _sz()
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(f), ctypes.byref(c),
                                     ctypes.byref(b)), "moe_workspace_size")
    return f.value, c.value, b.value


def moe_route(cfg: MoeConfig, x, W_r, logit_bias, logits, topk_idx, topk_w, counts, offsets,
              perm_token, slot_row, ws, stream=None) -> None:
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    _check(load().moe_route(ctypes.byref(cfg), _ptr(x, bf), _ptr(W_r, bf), _ptr(logit_bias, f32),
                            _ptr(logits, f32), _ptr(topk_idx, i32), _ptr(topk_w, f32),
                            _ptr(counts, i32), _ptr(offsets, i32), _ptr(perm_token, i32),
                            _ptr(slot_row, i32), _ptr(ws), ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_route")


def moe_route_noalloc(cfg: MoeConfig, x, W_r, logit_bias, logits, topk_idx, topk_w, counts,
                      offsets, perm_token, slot_row, device_status=None, stream=None) -> None:
    """moe_route without a workspace: the library's fixed scratch array is used
    instead, for callers that cannot allocate device memory."""
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    _check(load().moe_route_noalloc(ctypes.byref(cfg), _ptr(x, bf), _ptr(W_r, bf),
                                    _ptr(logit_bias, f32), _ptr(logits, f32), _ptr(topk_idx, i32),
                                    _ptr(topk_w, f32), _ptr(counts, i32), _ptr(offsets, i32),
                                    _ptr(perm_token, i32), _ptr(slot_row, i32),
                                    _ptr(device_status, i32), _stream(stream)),
           "moe_route_noalloc")


def moe_forward(cfg: MoeConfig, x, W_r, logit_bias, W_gate, W_up, W_down, y, ctx, ws,
                stream=None) -> None:
    bf = torch.bfloat16
    _check(load().moe_forward(ctypes.byref(cfg), _ptr(x, bf), _ptr(W_r, bf),
                              _ptr(logit_bias, torch.float32), _ptr(W_gate, bf), _ptr(W_up, bf),
                              _ptr(W_down, bf), _ptr(y, bf), _ptr(ctx), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_backward(cfg: MoeConfig, x, W_r, W_gate, W_up, W_down, ctx, dY, dx, dW_r, dW_gate,
                 dW_up, dW_down, ws, stream=None) -> None:
    bf = torch.bfloat16
    _check(load().moe_backward(ctypes.byref(cfg), _ptr(x, bf), _ptr(W_r, bf), _ptr(W_gate, bf),
                               _ptr(W_up, bf), _ptr(W_down, bf), _ptr(ctx), _ptr(dY, bf),
                               _ptr(dx, bf), _ptr(dW_r, bf), _ptr(dW_gate, bf), _ptr(dW_up, bf),
                               _ptr(dW_down, bf), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream)), "moe_backward")


def moe_backward_accumulate(cfg: MoeConfig, x, W_r, W_gate, W_up, W_down, ctx, dY, dx, gW_r,
                            gW_gate, gW_up, gW_down, ws, stream=None) -> None:
    bf, f32 = torch.bfloat16, torch.float32
    _check(load().moe_backward_accumulate(
        ctypes.byref(cfg), _ptr(x, bf), _ptr(W_r, bf), _ptr(W_gate, bf), _ptr(W_up, bf),
        _ptr(W_down, bf), _ptr(ctx), _ptr(dY, bf), _ptr(dx, bf), _ptr(gW_r, f32),
        _ptr(gW_gate, f32), _ptr(gW_up, f32), _ptr(gW_down, f32), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_backward_accumulate")


def moe_prepared_weights_size(cfg: MoeConfig) -> int:
    n = _sz()
    _check(load().moe_prepared_weights_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_prepared_weights_size")
    return n.value


def moe_prepare_weights(cfg: MoeConfig, W_gate, W_up, W_down, wq, stream=None) -> None:
    bf = torch.bfloat16
    _check(load().moe_prepare_weights(ctypes.byref(cfg), _ptr(W_gate, bf), _ptr(W_up, bf),
                                      _ptr(W_down, bf), _ptr(wq), wq.numel() * wq.element_size(),
                                      _stream(stream)), "moe_prepare_weights")


def moe_gemm_bf16(A, a_kmajor: bool, B, b_kmajor: bool, D, ws, stream=None) -> None:
    """D[M,N] = sum_k A(m,k) B(n,k); A is [M,K] (a_kmajor) or [K,M], B is [N,K]
    (b_kmajor) or [K,N]; D fp32 [M,N]."""
    M, N = D.shape
    K = A.shape[1] if a_kmajor else A.shape[0]
    bf = torch.bfloat16
    _check(load().moe_gemm_bf16(M, N, K, _ptr(A, bf), int(bool(a_kmajor)), _ptr(B, bf),
                                int(bool(b_kmajor)), _ptr(D, torch.float32), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)),
           "moe_gemm_bf16")


def moe_gemm_mxfp8(A, B, D, stream=None) -> None:
    """D[M,N] = sum_k A_q(m,k) B_q(n,k) with A [M,K], B [N,K] bf16 quantised to
    MXFP8 along K by the library; D fp32 [M,N].  Sizes and owns its workspace."""
    M, K = A.shape
    N = B.shape[0]
    lib = load()
    need = _sz(0)
    _check(lib.moe_gemm_mxfp8(M, N, K, None, None, None, None, ctypes.byref(need), None),
           "moe_gemm_mxfp8")
    ws = torch.empty(max(need.value, 256), dtype=torch.uint8, device=A.device)
    have = _sz(ws.numel())
    bf = torch.bfloat16
    _check(lib.moe_gemm_mxfp8(M, N, K, _ptr(A, bf), _ptr(B, bf), _ptr(D, torch.float32),
                              _ptr(ws), ctypes.byref(have), _stream(stream)), "moe_gemm_mxfp8")


def moe_get_device_status(ws, stream=None) -> int:
    return int(load().moe_get_device_status(_ptr(ws), _stream(stream)))


def moe_status_string(code: int) -> str:
    return load().moe_status_string(int(code)).decode()


def moe_profile_enable(on: bool) -> None:
    load().moe_profile_enable(1 if on else 0)


def moe_profile_select(name: Optional[str]) -> None:
    """Times only the launches labelled `name` while profiling is enabled
    (None: every launch)."""
    load().moe_profile_select(None if name is None else name.encode())


def moe_profile_read(cap: int = 64) -> Dict[str, Tuple[int, float]]:
    names = (ctypes.c_char_p * cap)()
    launches = (_i64 * cap)()
    ms = (ctypes.c_double * cap)()
    n = load().moe_profile_read(names, launches, ms, cap)
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(min(n, cap))}


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def exported_symbols() -> List[str]:
    lib = load()
    return [name for name in EXPORTED if hasattr(lib, name)]

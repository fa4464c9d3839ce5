"""Python binding of libkmoe: the Kimi-K3 routed-expert MoE forward
(MXFP8 activations x MXFP4 weights, SiTU) for GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions carry the C entry points' names (include/kmoe.h); torch is used
for device memory and the current stream.  Importing this package loads the
in-tree libkmoe.so and raises if it is missing (build it with
`python -m mxfp8_mxfp4_moe_gb300.build` or __graft_entry__.build()).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkmoe.so")

KMOE_OK = 0
STATUS = {0: "KMOE_OK", 1: "KMOE_ERR_ARG", 2: "KMOE_ERR_SHAPE", 3: "KMOE_ERR_ALIGN", 4: "KMOE_ERR_ARCH",
          5: "KMOE_ERR_WORKSPACE", 6: "KMOE_ERR_CUDA", 7: "KMOE_ERR_TIMEOUT", 8: "KMOE_ERR_DEVICE"}
KMOE_MXFP8_E4M3 = 0
KMOE_MXFP4_E2M1 = 1

EXPORTS = ("kmoe_status_string", "kmoe_check_device", "kmoe_workspace_size", "kmoe_workspace_layout",
           "kmoe_route", "kmoe_quantize_mx", "kmoe_prepared_weight_bytes", "kmoe_prepare_weights",
           "kmoe_forward", "kmoe_forward_ex", "kmoe_device_error", "kmoe_tile_sf_offset",
           "kmoe_selftest_wait_timeout", "kmoe_forward_noalloc", "kmoe_mma_peak_run",
           "kmoe_router_workspace_size", "kmoe_router", "kmoe_forward_router", "kmoe_selftest_activation")
NOALLOC_SCRATCH_BYTES = 32 << 20


class kmoe_params(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("situ_beta", ctypes.c_float), ("situ_linear_beta", ctypes.c_float),
                ("routed_scaling_factor", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("swiglu_alpha", ctypes.c_float), ("swiglu_beta", ctypes.c_float), ("swiglu_limit", ctypes.c_float)]


class kmoe_ws_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("err", "topk_ids", "topk_w", "counts", "seg_start", "tile_start",
                                               "row_of_slot", "slot_of_row", "xq", "xsf", "iq", "isf", "y")] + \
               [("tile_rows", ctypes.c_int), ("max_tiles", ctypes.c_int), ("total", ctypes.c_size_t),
                ("logits", ctypes.c_size_t), ("tile_start_big", ctypes.c_size_t), ("xsf_big", ctypes.c_size_t),
                ("isf_big", ctypes.c_size_t), ("tile_rows_big", ctypes.c_int), ("max_tiles_big", ctypes.c_int),
                ("big_rows", ctypes.c_int)]


class kmoe_stage_events(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("start", "routed", "permuted", "quantized", "fc1", "fc2",
                                               "combined")]


STAGE_NAMES = ("route", "permute", "quantize", "fc1", "fc2", "combine")


class KmoeError(RuntimeError):
    def __init__(self, fn, status, lib=None):
        msg = STATUS.get(status, str(status))
        if lib is not None:
            msg += ": " + lib.kmoe_status_string(status).decode()
        super().__init__(f"{fn} failed with {msg}")
        self.status = status


def load_library(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libkmoe.so not built at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, S, I, V = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
    pp = ctypes.POINTER(kmoe_params)
    lib.kmoe_status_string.restype = ctypes.c_char_p
    lib.kmoe_status_string.argtypes = [I]
    lib.kmoe_check_device.argtypes = [I]
    lib.kmoe_workspace_size.restype = S
    lib.kmoe_workspace_size.argtypes = [pp]
    lib.kmoe_workspace_layout.argtypes = [pp, ctypes.POINTER(kmoe_ws_layout)]
    lib.kmoe_route.argtypes = [P, P, I, I, I, P, P, V]
    lib.kmoe_quantize_mx.argtypes = [P, I, I, I, P, P, V]
    lib.kmoe_prepared_weight_bytes.restype = S
    lib.kmoe_prepared_weight_bytes.argtypes = [pp, I]
    lib.kmoe_prepare_weights.argtypes = [pp, P, P, P, P, P, P, V]
    lib.kmoe_forward.argtypes = [pp, P, P, P, P, P, P, P, P, P, S, V]
    lib.kmoe_forward_ex.argtypes = [pp, P, P, P, P, P, P, P, P, P, S, V, ctypes.POINTER(kmoe_stage_events)]
    lib.kmoe_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), V]
    lib.kmoe_tile_sf_offset.restype = S
    lib.kmoe_tile_sf_offset.argtypes = [I, I, I, I, I, I]
    lib.kmoe_selftest_wait_timeout.argtypes = [P, I, V]
    lib.kmoe_mma_peak_run.argtypes = [I, I, P, V]
    lib.kmoe_mma_peak_run.restype = ctypes.c_int
    lib.kmoe_forward_noalloc.argtypes = [pp, P, P, P, P, P, P, P, P, P, V]
    lib.kmoe_forward_noalloc.restype = ctypes.c_int
    lib.kmoe_router_workspace_size.restype = S
    lib.kmoe_router_workspace_size.argtypes = [I, I, I]
    lib.kmoe_router.argtypes = [P, P, P, I, I, I, I, P, P, P, P, S, V]
    lib.kmoe_forward_router.argtypes = [pp, P, P, P, P, P, P, P, S, V, ctypes.POINTER(kmoe_stage_events)]
    lib.kmoe_selftest_activation.argtypes = [pp, P, P, I, P, V]
    for n in ("kmoe_check_device", "kmoe_workspace_layout", "kmoe_route", "kmoe_quantize_mx",
              "kmoe_prepare_weights", "kmoe_forward", "kmoe_forward_ex", "kmoe_device_error",
              "kmoe_selftest_wait_timeout", "kmoe_router", "kmoe_forward_router", "kmoe_selftest_activation"):
        getattr(lib, n).restype = ctypes.c_int
    return lib


_lib = load_library()


def lib():
    return _lib


def _check(fn, st):
    if st != KMOE_OK:
        raise KmoeError(fn, st, _lib)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _arg(t, name, dtype=None, shape=None, min_bytes=None):
    """Checks a caller tensor before its pointer reaches the library, which
    sees no sizes: dtype, exact shape or a minimum size in bytes, and
    contiguity.  None passes (optional arguments).  Each entry point checks
    every argument this way, then that all of them live on the GPU (_gpu)."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if min_bytes is not None and _nbytes(t) < min_bytes:
        raise ValueError(f"{name} holds {_nbytes(t)} bytes, needs at least {min_bytes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (strided input is rejected, not copied)")


def _gpu(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _nbytes(t):
    return t.numel() * t.element_size()


def _rows(t, name, ncols_name):
    """(rows, cols) of a 2-D argument."""
    if t is None or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor [rows, {ncols_name}]")
    return t.shape


KMOE_FLAG_SWIGLU = 1


def make_params(T, H, I, E, k, situ_beta=4.0, situ_linear_beta=25.0, routed_scaling_factor=1.0,
                activation="situ", swiglu_alpha=1.702, swiglu_beta=1.0, swiglu_limit=7.0):
    """`activation` is "situ" (the layer's) or "swiglu" (the clamped SwiGLU control)."""
    if activation not in ("situ", "swiglu"):
        raise ValueError(f"activation must be 'situ' or 'swiglu', got {activation!r}")
    flags = KMOE_FLAG_SWIGLU if activation == "swiglu" else 0
    return kmoe_params(T, H, I, E, k, situ_beta, situ_linear_beta, routed_scaling_factor, flags,
                       swiglu_alpha, swiglu_beta, swiglu_limit)


def kmoe_status_string(status: int) -> str:
    return _lib.kmoe_status_string(status).decode()


def kmoe_check_device(device: int = 0) -> int:
    return _lib.kmoe_check_device(device)


def kmoe_workspace_size(p: kmoe_params) -> int:
    return _lib.kmoe_workspace_size(ctypes.byref(p))


def kmoe_workspace_layout(p: kmoe_params) -> kmoe_ws_layout:
    out = kmoe_ws_layout()
    _check("kmoe_workspace_layout", _lib.kmoe_workspace_layout(ctypes.byref(p), ctypes.byref(out)))
    return out


def kmoe_route(logits, bias, k, topk_ids=None, topk_w=None, stream=None):
    T, E = _rows(logits, "logits", "E")
    _arg(logits, "logits", torch.float32)
    _arg(bias, "bias", torch.float32, (E,))
    _arg(topk_ids, "topk_ids", torch.int32, (T, k))
    _arg(topk_w, "topk_w", torch.float32, (T, k))
    _gpu(logits=logits, bias=bias, topk_ids=topk_ids, topk_w=topk_w)
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check("kmoe_route", _lib.kmoe_route(_ptr(logits), _ptr(bias), T, E, k, _ptr(topk_ids), _ptr(topk_w),
                                         _stream(stream)))
    return topk_ids, topk_w


def kmoe_quantize_mx(x, fmt=KMOE_MXFP8_E4M3, codes=None, scales=None, stream=None):
    rows, cols = _rows(x, "x", "cols")
    _arg(x, "x", torch.bfloat16)
    _arg(codes, "codes", torch.uint8, (rows, cols if fmt == KMOE_MXFP8_E4M3 else cols // 2))
    _arg(scales, "scales", torch.uint8, (rows, cols // 32))
    _gpu(x=x, codes=codes, scales=scales)
    if codes is None:
        codes = torch.empty((rows, cols if fmt == KMOE_MXFP8_E4M3 else cols // 2), dtype=torch.uint8,
                            device=x.device)
    if scales is None:
        scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    _check("kmoe_quantize_mx", _lib.kmoe_quantize_mx(_ptr(x), rows, cols, fmt, _ptr(codes), _ptr(scales),
                                                     _stream(stream)))
    return codes, scales


def kmoe_prepared_weight_bytes(p, which):
    return _lib.kmoe_prepared_weight_bytes(ctypes.byref(p), which)


def kmoe_prepare_weights(p, w13, w13_sf, w2, w2_sf, stream=None):
    """Raw checkpoint tensors -> (w13_k, w2_k) prepared weight blocks."""
    for n, t in (("w13", w13), ("w13_sf", w13_sf), ("w2", w2), ("w2_sf", w2_sf)):
        _arg(t, n, torch.uint8)
    _gpu(w13=w13, w13_sf=w13_sf, w2=w2, w2_sf=w2_sf)
    if (w13.numel() != p.E * 2 * p.I * p.H // 2 or w13_sf.numel() != p.E * 2 * p.I * p.H // 32 or
            w2.numel() != p.E * p.H * p.I // 2 or w2_sf.numel() != p.E * p.H * p.I // 32):
        raise ValueError("weight sizes do not match the parameters (w13 [E, 2I, H/2], w2 [E, H, I/2])")
    a = torch.empty(kmoe_prepared_weight_bytes(p, 0), dtype=torch.uint8, device=w13.device)
    b = torch.empty(kmoe_prepared_weight_bytes(p, 1), dtype=torch.uint8, device=w13.device)
    _check("kmoe_prepare_weights", _lib.kmoe_prepare_weights(ctypes.byref(p), _ptr(w13), _ptr(w13_sf), _ptr(w2),
                                                             _ptr(w2_sf), _ptr(a), _ptr(b), _stream(stream)))
    return a, b


def _layer_args(p, x, w13_k, w2_k, out, workspace=None):
    """Checks of the arguments every forward entry point shares."""
    _arg(x, "x", torch.bfloat16, (p.T, p.H))
    _arg(w13_k, "w13_k", torch.uint8, min_bytes=kmoe_prepared_weight_bytes(p, 0))
    _arg(w2_k, "w2_k", torch.uint8, min_bytes=kmoe_prepared_weight_bytes(p, 1))
    _arg(out, "out", torch.bfloat16, (p.T, p.H))
    _arg(workspace, "workspace", torch.uint8, min_bytes=kmoe_workspace_size(p))


def kmoe_forward(p, x, logits, bias, w13_k, w2_k, topk_ids=None, topk_w=None, out=None, workspace=None,
                 stream=None, stage_events=None):
    """stage_events: optional list of 7 torch.cuda.Event recorded between the stages (kmoe_forward_ex)."""
    _layer_args(p, x, w13_k, w2_k, out, workspace)
    if topk_ids is None:
        _arg(logits, "logits", torch.float32, (p.T, p.E))
        _arg(bias, "bias", torch.float32, (p.E,))
    else:
        _arg(topk_ids, "topk_ids", torch.int32, (p.T, p.k))
        _arg(topk_w, "topk_w", torch.float32, (p.T, p.k))
    _gpu(x=x, logits=logits, bias=bias, w13_k=w13_k, w2_k=w2_k, topk_ids=topk_ids, topk_w=topk_w, out=out,
         workspace=workspace)
    if out is None:
        out = torch.empty((p.T, p.H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(kmoe_workspace_size(p), dtype=torch.uint8, device=x.device)
    args = (ctypes.byref(p), _ptr(x), _ptr(logits), _ptr(bias), _ptr(w13_k), _ptr(w2_k), _ptr(topk_ids),
            _ptr(topk_w), _ptr(out), _ptr(workspace), _nbytes(workspace), _stream(stream))
    if stage_events is None:
        _check("kmoe_forward", _lib.kmoe_forward(*args))
    else:
        ev = kmoe_stage_events(*[e.cuda_event for e in stage_events])
        _check("kmoe_forward_ex", _lib.kmoe_forward_ex(*args, ctypes.byref(ev)))
    return out, workspace


def kmoe_router_workspace_size(T: int, H: int, E: int) -> int:
    return _lib.kmoe_router_workspace_size(T, H, E)


def kmoe_router(x, w_gate, bias, k, logits=None, topk_ids=None, topk_w=None, workspace=None, stream=None):
    """The fused router: logits = x @ w_gate^T (bf16 operands, fp32) and the
    top-k routing of kmoe_route, in one kernel.  Returns (topk_ids, topk_w,
    logits, workspace); the workspace's first word is the device error word."""
    T, H = _rows(x, "x", "H")
    E, _ = _rows(w_gate, "w_gate", "H")
    _arg(x, "x", torch.bfloat16)
    _arg(w_gate, "w_gate", torch.bfloat16, (E, H))
    _arg(bias, "bias", torch.float32, (E,))
    _arg(logits, "logits", torch.float32, (T, E))
    _arg(topk_ids, "topk_ids", torch.int32, (T, k))
    _arg(topk_w, "topk_w", torch.float32, (T, k))
    _arg(workspace, "workspace", torch.uint8, min_bytes=kmoe_router_workspace_size(T, H, E))
    _gpu(x=x, w_gate=w_gate, bias=bias, logits=logits, topk_ids=topk_ids, topk_w=topk_w, workspace=workspace)
    dev = x.device
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(kmoe_router_workspace_size(T, H, E), dtype=torch.uint8, device=dev)
    _check("kmoe_router", _lib.kmoe_router(_ptr(x), _ptr(w_gate), _ptr(bias), T, H, E, k, _ptr(logits),
                                           _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), _nbytes(workspace),
                                           _stream(stream)))
    return topk_ids, topk_w, logits, workspace


def kmoe_forward_router(p, x, w_gate, bias, w13_k, w2_k, out=None, workspace=None, stream=None,
                        stage_events=None):
    """kmoe_forward with the fused router (routing from x and the gate weight
    instead of given logits).  stage_events: optional list of 7 torch.cuda.Event."""
    _layer_args(p, x, w13_k, w2_k, out, workspace)
    _arg(w_gate, "w_gate", torch.bfloat16, (p.E, p.H))
    _arg(bias, "bias", torch.float32, (p.E,))
    _gpu(x=x, w_gate=w_gate, bias=bias, w13_k=w13_k, w2_k=w2_k, out=out, workspace=workspace)
    if out is None:
        out = torch.empty((p.T, p.H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(kmoe_workspace_size(p), dtype=torch.uint8, device=x.device)
    ev = None if stage_events is None else kmoe_stage_events(*[e.cuda_event for e in stage_events])
    _check("kmoe_forward_router", _lib.kmoe_forward_router(
        ctypes.byref(p), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w13_k), _ptr(w2_k), _ptr(out), _ptr(workspace),
        _nbytes(workspace), _stream(stream), None if ev is None else ctypes.byref(ev)))
    return out, workspace


def kmoe_forward_noalloc(p, x, logits, bias, w13_k, w2_k, topk_ids=None, topk_w=None, out=None,
                         device_error=None, stream=None):
    """kmoe_forward without a workspace argument, for hosts that cannot
    allocate device memory: the library's built-in scratch array
    (NOALLOC_SCRATCH_BYTES, shared by all calls) is used instead.  `out` and
    the optional `device_error` (one int32 on the device) are caller-owned."""
    _layer_args(p, x, w13_k, w2_k, out)
    if topk_ids is None:
        _arg(logits, "logits", torch.float32, (p.T, p.E))
        _arg(bias, "bias", torch.float32, (p.E,))
    else:
        _arg(topk_ids, "topk_ids", torch.int32, (p.T, p.k))
        _arg(topk_w, "topk_w", torch.float32, (p.T, p.k))
    _arg(device_error, "device_error", min_bytes=4)
    _gpu(x=x, logits=logits, bias=bias, w13_k=w13_k, w2_k=w2_k, topk_ids=topk_ids, topk_w=topk_w, out=out,
         device_error=device_error)
    if out is None:
        out = torch.empty((p.T, p.H), dtype=torch.bfloat16, device=x.device)
    _check("kmoe_forward_noalloc", _lib.kmoe_forward_noalloc(
        ctypes.byref(p), _ptr(x), _ptr(logits), _ptr(bias), _ptr(w13_k), _ptr(w2_k), _ptr(topk_ids), _ptr(topk_w),
        _ptr(out), _ptr(device_error), _stream(stream)))
    return out


def kmoe_selftest_activation(p, gate, up, out=None, stream=None):
    """The FC1 epilogue's activation of (gate, up), elementwise (fp32 device
    arrays of one shape), by the forward's own device functions."""
    _arg(gate, "gate", torch.float32, tuple(gate.shape))
    _arg(up, "up", torch.float32, tuple(gate.shape))
    if out is None:
        out = torch.empty_like(gate)
    _arg(out, "out", torch.float32, tuple(gate.shape))
    _gpu(gate=gate, up=up, out=out)
    _check("kmoe_selftest_activation", _lib.kmoe_selftest_activation(
        ctypes.byref(p), _ptr(gate), _ptr(up), gate.numel(), _ptr(out), _stream(stream)))
    return out


def kmoe_device_error(workspace, stream=None):
    _arg(workspace, "workspace", min_bytes=4)
    _gpu(workspace=workspace)
    word = ctypes.c_uint32(0)
    st = _lib.kmoe_device_error(_ptr(workspace), ctypes.byref(word), _stream(stream))
    return st, word.value


def kmoe_tile_sf_offset(tile, local_row, g, tile_rows, K, max_tiles):
    return _lib.kmoe_tile_sf_offset(tile, local_row, g, tile_rows, K, max_tiles)


def kmoe_mma_peak_run(iters, N, workspace, stream=None):
    """Launch the tensor-pipe roof kernel; returns the launch's FLOP count."""
    _arg(workspace, "workspace", min_bytes=4)
    _gpu(workspace=workspace)
    _check("kmoe_mma_peak_run", _lib.kmoe_mma_peak_run(iters, N, _ptr(workspace), _stream(stream)))
    sms = torch.cuda.get_device_properties(workspace.device).multi_processor_count
    return sms * iters * 4 * 2 * 128 * N * 32


def kmoe_selftest_wait_timeout(workspace, budget_us, stream=None):
    _arg(workspace, "workspace", min_bytes=4)
    _gpu(workspace=workspace)
    _check("kmoe_selftest_wait_timeout",
           _lib.kmoe_selftest_wait_timeout(_ptr(workspace), budget_us, _stream(stream)))


def stage_views(p, workspace):
    """Views of the stage tensors kmoe_forward leaves in the workspace."""
    L = kmoe_workspace_layout(p)
    R = p.T * p.k

    def v(off, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return workspace[off:off + nbytes].view(dtype)

    return {
        "layout": L,
        "topk_ids": v(L.topk_ids, R, torch.int32).view(p.T, p.k),
        "topk_w": v(L.topk_w, R, torch.float32).view(p.T, p.k),
        "counts": v(L.counts, p.E, torch.int32),
        "seg_start": v(L.seg_start, p.E + 1, torch.int32),
        "tile_start": v(L.tile_start, p.E + 1, torch.int32),
        "row_of_slot": v(L.row_of_slot, R, torch.int32),
        "slot_of_row": v(L.slot_of_row, R, torch.int32),
        "xq": v(L.xq, R * p.H, torch.uint8).view(R, p.H),
        "iq": v(L.iq, R * p.I, torch.uint8).view(R, p.I),
        "xsf": workspace[L.xsf:L.xsf + (p.H // 128) * L.max_tiles * ((L.tile_rows + 127) // 128) * 512],
        "isf": workspace[L.isf:L.isf + (p.I // 128) * L.max_tiles * ((L.tile_rows + 127) // 128) * 512],
        "tile_start_big": v(L.tile_start_big, p.E + 1, torch.int32),
        "xsf_big": workspace[L.xsf_big:L.xsf_big + (p.H // 128) * L.max_tiles_big * 2 * 512],
        "isf_big": workspace[L.isf_big:L.isf_big + (p.I // 128) * L.max_tiles_big * 2 * 512],
        "y": v(L.y, R * p.H, torch.float32).view(R, p.H),
        "logits": v(L.logits, p.T * p.E, torch.float32).view(p.T, p.E),
    }

"""Thin Python binding of libmoe_ffn_gb300 (include/moe_ffn.h), argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module checks tensor
dtypes/devices/contiguity, passes raw pointers and the current CUDA stream, and turns a non-zero
status into an exception. There is no fallback: if the library is missing it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_VALUE", -5: "MOE_ERR_CUDA", -6: "MOE_ERR_UNSUPPORTED",
          -7: "MOE_ERR_ALIGN"}
FMT_FP8 = 1
FMT_NVFP4 = 2
ERRBIT_BAD_ID = 1
ERRBIT_BARRIER = 2
ERRBIT_DRAIN = 4

EXPORTED = ("moe_workspace_bytes", "moe_route_permute", "moe_fp8_forward", "moe_nvfp4_forward",
            "moe_plan", "moe_fp8_gate_up", "moe_fp8_down_combine", "moe_nvfp4_gate_up",
            "moe_nvfp4_down_combine", "moe_build_arch", "moe_fp8_forward_noalloc",
            "moe_router_workspace_bytes", "moe_router", "moe_fp8_forward_layer",
            "moe_nvfp4_forward_layer", "moe_shared_expert_workspace_bytes", "moe_shared_expert_bf16",
            "moe_stage_timing", "moe_stage_times", "moe_test_barrier_timeout",
            "moe_nvfp4_forward_expert_scale2", "moe_nvfp4_forward_layer_expert_scale2",
            "moe_stream_read")

_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load the in-tree shared library. Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(p)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.moe_workspace_bytes.restype = sz
    lib.moe_workspace_bytes.argtypes = [i32] * 6
    lib.moe_route_permute.restype = i32
    lib.moe_route_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.moe_fp8_forward.restype = i32
    lib.moe_fp8_forward.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                    f32, vp, vp, sz, vp, vp]
    lib.moe_nvfp4_forward.restype = i32
    lib.moe_nvfp4_forward.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, f32, vp, vp,
                                      f32, vp, vp, f32, f32, vp, vp, sz, vp, vp]
    lib.moe_nvfp4_forward_expert_scale2.restype = i32
    lib.moe_nvfp4_forward_expert_scale2.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                    vp, vp, vp, vp, vp, i32, f32, vp, vp, sz, vp, vp]
    lib.moe_plan.restype = i32
    lib.moe_plan.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, sz, vp, vp]
    lib.moe_fp8_gate_up.restype = i32
    lib.moe_fp8_gate_up.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, f32, vp, sz,
                                    vp, vp]
    lib.moe_fp8_down_combine.restype = i32
    lib.moe_fp8_down_combine.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_nvfp4_gate_up.restype = i32
    lib.moe_nvfp4_gate_up.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, f32, vp, vp, f32,
                                      f32, vp, sz, vp, vp]
    lib.moe_nvfp4_down_combine.restype = i32
    lib.moe_nvfp4_down_combine.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, f32, vp, vp,
                                           sz, vp]
    lib.moe_build_arch.restype = ctypes.c_char_p
    lib.moe_build_arch.argtypes = []
    lib.moe_router_workspace_bytes.restype = sz
    lib.moe_router_workspace_bytes.argtypes = [i32, i32, i32]
    lib.moe_router.restype = i32
    lib.moe_router.argtypes = [vp, i32, i32, vp, vp, i32, i32, f32, i32, vp, vp, vp, vp, sz, vp]
    lib.moe_fp8_forward_layer.restype = i32
    lib.moe_fp8_forward_layer.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                          f32, vp, vp, vp, vp, sz, vp, vp]
    lib.moe_nvfp4_forward_layer.restype = i32
    lib.moe_nvfp4_forward_layer.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, f32, vp, vp,
                                            f32, vp, vp, f32, f32, vp, vp, vp, vp, sz, vp, vp]
    lib.moe_nvfp4_forward_layer_expert_scale2.restype = i32
    lib.moe_nvfp4_forward_layer_expert_scale2.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                                          vp, vp, vp, vp, vp, vp, i32, f32, vp, vp, vp, vp,
                                                          sz, vp, vp]
    lib.moe_shared_expert_workspace_bytes.restype = sz
    lib.moe_shared_expert_workspace_bytes.argtypes = [i32, i32, i32]
    lib.moe_shared_expert_bf16.restype = i32
    lib.moe_shared_expert_bf16.argtypes = [vp, i32, i32, i32, vp, vp, vp, f32, vp, vp, sz, vp]
    lib.moe_stage_timing.restype = i32
    lib.moe_stage_timing.argtypes = [i32]
    lib.moe_test_barrier_timeout.restype = i32
    lib.moe_test_barrier_timeout.argtypes = [i32]
    lib.moe_stream_read.restype = i32
    lib.moe_stream_read.argtypes = [vp, sz, vp, vp]
    lib.moe_stage_times.restype = i32
    lib.moe_stage_times.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), i32]
    if path is None:
        _lib = lib
    return lib


# ---- marshalling helpers -------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


# ---- public API ----------------------------------------------------------------------------------

def workspace_bytes(T: int, H: int, I: int, E: int, topk: int, fmt: int) -> int:
    return int(load().moe_workspace_bytes(T, H, I, E, topk, fmt))


def alloc_workspace(T, H, I, E, topk, fmt, device) -> torch.Tensor:
    n = workspace_bytes(T, H, I, E, topk, fmt)
    if n == 0:
        raise ValueError("invalid sizes for moe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)   # caching allocator: 256-B aligned


def route_permute(ids: torch.Tensor, num_experts: int, err: Optional[torch.Tensor] = None,
                  stream=None):
    """Stable counting sort of (token, slot) pairs by expert (moe_route_permute)."""
    dev = ids.device
    _need(ids, "ids", torch.int32, dev)
    T, topk = ids.shape
    P = T * topk
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    sorted_pair = torch.empty(P, dtype=torch.int32, device=dev)
    pair_to_sorted = torch.empty(P, dtype=torch.int32, device=dev)
    if err is not None:
        _need(err, "err", torch.int32, dev)
    rc = load().moe_route_permute(_ptr(ids), T, topk, num_experts, _ptr(counts), _ptr(offsets),
                                  _ptr(sorted_pair), _ptr(pair_to_sorted), _ptr(err),
                                  _stream(dev, stream))
    _check("moe_route_permute", rc)
    return dict(counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_to_sorted=pair_to_sorted)


def _common(x, ids, wts, out, workspace, err, fmt, E, I):
    dev = x.device
    _need(x, "x", torch.bfloat16, dev)
    _need(ids, "topk_ids", torch.int32, dev)
    _need(wts, "topk_weights", torch.float32, dev)
    T, H = x.shape
    topk = ids.shape[1]
    if ids.shape[0] != T or wts.shape != ids.shape:
        raise ValueError("topk_ids / topk_weights must be [T, topk]")
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    if workspace is None:
        workspace = alloc_workspace(T, H, I, E, topk, fmt, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if err is not None:
        _need(err, "err", torch.int32, dev)
    return dev, T, H, topk, out, workspace


def fp8_forward(x, ids, wts, bank, limit: float, out=None, workspace=None, err=None, stream=None):
    """Routed MoE FFN over an E4M3 bank with 128x128 block scales (moe_fp8_forward)."""
    E, I, _ = bank.w_gate.shape
    dev, T, H, topk, out, ws = _common(x, ids, wts, out, workspace, err, FMT_FP8, E, I)
    for n in ("w_gate", "w_up", "w_down"):
        _need(getattr(bank, n), n, torch.uint8, dev)
    for n in ("s_gate", "s_up", "s_down"):
        _need(getattr(bank, n), n, torch.float32, dev)
    rc = load().moe_fp8_forward(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                _ptr(bank.w_gate), _ptr(bank.s_gate), _ptr(bank.w_up),
                                _ptr(bank.s_up), _ptr(bank.w_down), _ptr(bank.s_down),
                                float(limit), _ptr(out), _ptr(ws), ws.numel(), _ptr(err),
                                _stream(dev, stream))
    _check("moe_fp8_forward", rc)
    return out


def nvfp4_forward(x, ids, wts, bank, limit: float, out=None, workspace=None, err=None, stream=None):
    """Routed MoE FFN over an NVFP4 (W4A16) bank (moe_nvfp4_forward; with one scale_2 per expert
    and projection, moe_nvfp4_forward_expert_scale2)."""
    E, I, _ = bank.w_gate.shape
    dev, T, H, topk, out, ws = _common(x, ids, wts, out, workspace, err, FMT_NVFP4, E, I)
    for n in ("w_gate", "w_up", "w_down", "sf_gate", "sf_up", "sf_down"):
        _need(getattr(bank, n), n, torch.uint8, dev)
    if _per_expert_scale2(bank):
        for n in ("scale2_gate", "scale2_up", "scale2_down"):
            t = getattr(bank, n)
            _need(t, n, torch.float32, dev)
            if tuple(t.shape) != (E,):
                raise ValueError(f"{n} must be [E] per expert")
        rc = load().moe_nvfp4_forward_expert_scale2(
            _ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
            _ptr(bank.w_gate), _ptr(bank.sf_gate), _ptr(bank.scale2_gate),
            _ptr(bank.w_up), _ptr(bank.sf_up), _ptr(bank.scale2_up),
            _ptr(bank.w_down), _ptr(bank.sf_down), _ptr(bank.scale2_down), 1,
            float(limit), _ptr(out), _ptr(ws), ws.numel(), _ptr(err), _stream(dev, stream))
        _check("moe_nvfp4_forward_expert_scale2", rc)
        return out
    rc = load().moe_nvfp4_forward(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                  _ptr(bank.w_gate), _ptr(bank.sf_gate), float(bank.scale2_gate),
                                  _ptr(bank.w_up), _ptr(bank.sf_up), float(bank.scale2_up),
                                  _ptr(bank.w_down), _ptr(bank.sf_down), float(bank.scale2_down),
                                  float(limit), _ptr(out), _ptr(ws), ws.numel(), _ptr(err),
                                  _stream(dev, stream))
    _check("moe_nvfp4_forward", rc)
    return out


def _per_expert_scale2(bank) -> bool:
    return isinstance(getattr(bank, "scale2_gate", None), torch.Tensor)


def _scalar_scale2_only(bank, fn: str):
    if _per_expert_scale2(bank):
        raise ValueError(f"{fn} takes one scale_2 per projection; a bank with one per expert goes "
                         "through nvfp4_forward (moe_nvfp4_forward_expert_scale2)")


def forward(x, ids, wts, bank, limit: float, **kw):
    """Dispatch on the bank's format."""
    if bank.fmt == "fp8":
        return fp8_forward(x, ids, wts, bank, limit, **kw)
    return nvfp4_forward(x, ids, wts, bank, limit, **kw)


def forward_layer(x, ids, wts, bank, limit: float, shared=None, residual=None, out=None,
                  workspace=None, err=None, stream=None):
    """moe_*_forward_layer: the forward with out = bf16((routed + shared) + residual) (an NVFP4 bank
    with one scale_2 per expert goes through moe_nvfp4_forward_layer_expert_scale2)."""
    E, I, _ = bank.w_gate.shape
    fmt = FMT_FP8 if bank.fmt == "fp8" else FMT_NVFP4
    dev, T, H, topk, out, ws = _common(x, ids, wts, out, workspace, err, fmt, E, I)
    for n, t in (("shared", shared), ("residual", residual)):
        if t is not None:
            _need(t, n, torch.bfloat16, dev)
            if tuple(t.shape) != (T, H):
                raise ValueError(f"{n} must be [T, H]")
    lib = load()
    if bank.fmt == "fp8":
        rc = lib.moe_fp8_forward_layer(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                       _ptr(bank.w_gate), _ptr(bank.s_gate), _ptr(bank.w_up),
                                       _ptr(bank.s_up), _ptr(bank.w_down), _ptr(bank.s_down),
                                       float(limit), _ptr(shared), _ptr(residual), _ptr(out), _ptr(ws),
                                       ws.numel(), _ptr(err), _stream(dev, stream))
    elif _per_expert_scale2(bank):
        for n in ("scale2_gate", "scale2_up", "scale2_down"):
            t = getattr(bank, n)
            _need(t, n, torch.float32, dev)
            if tuple(t.shape) != (E,):
                raise ValueError(f"{n} must be [E] per expert")
        rc = lib.moe_nvfp4_forward_layer_expert_scale2(
            _ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
            _ptr(bank.w_gate), _ptr(bank.sf_gate), _ptr(bank.scale2_gate),
            _ptr(bank.w_up), _ptr(bank.sf_up), _ptr(bank.scale2_up),
            _ptr(bank.w_down), _ptr(bank.sf_down), _ptr(bank.scale2_down), 1,
            float(limit), _ptr(shared), _ptr(residual), _ptr(out), _ptr(ws), ws.numel(), _ptr(err),
            _stream(dev, stream))
    else:
        rc = lib.moe_nvfp4_forward_layer(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                         _ptr(bank.w_gate), _ptr(bank.sf_gate), float(bank.scale2_gate),
                                         _ptr(bank.w_up), _ptr(bank.sf_up), float(bank.scale2_up),
                                         _ptr(bank.w_down), _ptr(bank.sf_down), float(bank.scale2_down),
                                         float(limit), _ptr(shared), _ptr(residual), _ptr(out), _ptr(ws),
                                         ws.numel(), _ptr(err), _stream(dev, stream))
    _check("moe_*_forward_layer", rc)
    return out


def shared_expert(x, w_gate, w_up, w_down, limit: float, out=None, workspace=None, stream=None):
    """moe_shared_expert_bf16: dense bf16 SwiGLU MLP, out [T, H] bf16."""
    dev = x.device
    _need(x, "x", torch.bfloat16, dev)
    for n, t in (("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down)):
        _need(t, n, torch.bfloat16, dev)
    T, H = x.shape
    S = w_gate.shape[0]
    lib = load()
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if workspace is None:
        n = int(lib.moe_shared_expert_workspace_bytes(T, H, S))
        if n == 0:
            raise ValueError("invalid sizes for moe_shared_expert_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    rc = lib.moe_shared_expert_bf16(_ptr(x), T, H, S, _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                    float(limit), _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream(dev, stream))
    _check("moe_shared_expert_bf16", rc)
    return out


# ---- stages (T <= 8), for profiling and interleaving ----------------------------------------------

def plan(ids, H, I, E, fmt, workspace, err=None, stream=None):
    T, topk = ids.shape
    rc = load().moe_plan(T, H, I, E, topk, fmt, _ptr(ids), _ptr(workspace), workspace.numel(),
                         _ptr(err), _stream(ids.device, stream))
    _check("moe_plan", rc)


def gate_up(x, ids, bank, limit, workspace, err=None, stream=None):
    _scalar_scale2_only(bank, "gate_up")
    T, H = x.shape
    topk = ids.shape[1]
    E, I, _ = bank.w_gate.shape
    lib = load()
    if bank.fmt == "fp8":
        rc = lib.moe_fp8_gate_up(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(bank.w_gate),
                                 _ptr(bank.s_gate), _ptr(bank.w_up), _ptr(bank.s_up), float(limit),
                                 _ptr(workspace), workspace.numel(), _ptr(err),
                                 _stream(x.device, stream))
    else:
        rc = lib.moe_nvfp4_gate_up(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(bank.w_gate),
                                   _ptr(bank.sf_gate), float(bank.scale2_gate), _ptr(bank.w_up),
                                   _ptr(bank.sf_up), float(bank.scale2_up), float(limit),
                                   _ptr(workspace), workspace.numel(), _ptr(err),
                                   _stream(x.device, stream))
    _check("moe_*_gate_up", rc)


def down_combine(ids, wts, bank, out, workspace, stream=None):
    _scalar_scale2_only(bank, "down_combine")
    T, H = out.shape
    topk = ids.shape[1]
    E, I, _ = bank.w_gate.shape
    lib = load()
    if bank.fmt == "fp8":
        rc = lib.moe_fp8_down_combine(T, H, I, E, topk, _ptr(ids), _ptr(wts), _ptr(bank.w_down),
                                      _ptr(bank.s_down), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(out.device, stream))
    else:
        rc = lib.moe_nvfp4_down_combine(T, H, I, E, topk, _ptr(ids), _ptr(wts), _ptr(bank.w_down),
                                        _ptr(bank.sf_down), float(bank.scale2_down), _ptr(out),
                                        _ptr(workspace), workspace.numel(),
                                        _stream(out.device, stream))
    _check("moe_*_down_combine", rc)


def test_barrier_timeout(enable: bool) -> None:
    """moe_test_barrier_timeout: make the cooperative forward's grid barrier time out (test hook)."""
    _check("moe_test_barrier_timeout", load().moe_test_barrier_timeout(1 if enable else 0))


def stream_read(buf: torch.Tensor, nbytes: int, sink: torch.Tensor, stream=None) -> None:
    """moe_stream_read: one plain streaming read of the first nbytes of buf (a device tensor),
    every 32-bit word XORed into sink (an int32 tensor of one element, not cleared). A
    measurement aid: the read throughput one kernel of nbytes reaches on the device."""
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    if nbytes > buf.numel() * buf.element_size():
        raise ValueError("nbytes exceeds the buffer")
    _need(sink, "sink", torch.int32, buf.device)
    _check("moe_stream_read", load().moe_stream_read(_ptr(buf), int(nbytes), _ptr(sink),
                                                      _stream(buf.device, stream)))


def build_arch() -> str:
    return load().moe_build_arch().decode()


def stage_timing(enable: bool) -> None:
    """moe_stage_timing: switch per-stage CUDA-event recording of the forward calls on or off."""
    _check("moe_stage_timing", load().moe_stage_timing(1 if enable else 0))


def stage_times(max_stages: int = 64):
    """moe_stage_times: [(stage name, device ms)] of the most recent timed forward (blocks on it)."""
    ms = (ctypes.c_float * max_stages)()
    names = (ctypes.c_char_p * max_stages)()
    n = load().moe_stage_times(ms, names, max_stages)
    if n < 0:
        _check("moe_stage_times", n)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def router(x: torch.Tensor, router_w: torch.Tensor, topk: int, routed_scale: float = 1.0,
           renormalize: bool = True, bias: Optional[torch.Tensor] = None, want_logits: bool = False,
           workspace: Optional[torch.Tensor] = None, stream=None):
    """moe_router: (topk_ids [T,topk] int32, topk_weights [T,topk] fp32, logits [T,E] fp32 or None)."""
    dev = x.device
    _need(x, "x", torch.bfloat16, dev)
    _need(router_w, "router_w", torch.bfloat16, dev)
    T, H = x.shape
    E = router_w.shape[0]
    if bias is not None:
        _need(bias, "bias", torch.float32, dev)
    lib = load()
    if workspace is None:
        n = int(lib.moe_router_workspace_bytes(T, H, E))
        if n == 0:
            raise ValueError("invalid sizes for moe_router_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    ids = torch.empty(T, topk, dtype=torch.int32, device=dev)
    wts = torch.empty(T, topk, dtype=torch.float32, device=dev)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None
    rc = lib.moe_router(_ptr(x), T, H, _ptr(router_w), _ptr(bias), E, topk, float(routed_scale),
                        int(bool(renormalize)), _ptr(logits), _ptr(ids), _ptr(wts), _ptr(workspace),
                        workspace.numel(), _stream(dev, stream))
    _check("moe_router", rc)
    return ids, wts, logits

"""Plain, slow, FP64 CPU reference for the routed MoE FFN ("the oracle").

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package. It shares no code with the CUDA library
in ``moe_expert_ffn_histogram_gb300`` and imports nothing from it.

The arithmetic lives in ``moe_oracle.cpp`` (host C++, no CUDA headers), compiled here with g++
into ``liboracle.so`` and called through ``ctypes``. This module only marshals numpy arrays.
See the header of ``moe_oracle.cpp`` for which page and section each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile moe_oracle.cpp with g++ (portable flags: no -march, builds on x86 and Arm)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_clamped_swiglu.restype = ctypes.c_double
        lib.oracle_clamped_swiglu.argtypes = [ctypes.c_double] * 3
        lib.oracle_hardware_threads.restype = ctypes.c_int
        for name in ("oracle_combine", "oracle_dequant_fp8", "oracle_dequant_nvfp4",
                     "oracle_route_permute", "oracle_moe_fp8", "oracle_moe_nvfp4",
                     "oracle_moe_nvfp4_expert_scale2",
                     "oracle_router_logits", "oracle_router_topk", "oracle_shared_expert",
                     "oracle_layer_epilogue"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar decoders / helpers -----------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code) & 0xFF)


def e2m1_value(nibble: int) -> float:
    return _load().oracle_e2m1_value(int(nibble) & 0xF)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(int(bits) & 0xFFFF)


def bf16_round(v: float) -> int:
    return int(_load().oracle_bf16_round(float(v)))


def clamped_swiglu(g: float, u: float, limit: float) -> float:
    return _load().oracle_clamped_swiglu(float(g), float(u), float(limit))


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def combine(down: np.ndarray, weights: np.ndarray, tokens: int, topk: int, width: int) -> np.ndarray:
    down = _c(down, np.float64)
    weights = _c(weights, np.float64)
    if down.size != tokens * topk * width or weights.size != tokens * topk:
        raise ValueError("combine: down/weights sizes do not match tokens x topk x width")
    out = np.zeros((tokens, width), np.float64)
    rc = _load().oracle_combine(_ptr(down), _ptr(weights), tokens, topk, width, _ptr(out))
    if rc:
        raise ValueError(f"oracle_combine failed: {rc}")
    return out


def dequant_fp8(codes: np.ndarray, scales: np.ndarray, expert: int) -> np.ndarray:
    """Dense float64 [N, K] of one expert of an E4M3 bank [E, N, K] with [E, N/128, K/128] scales."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    E, N, K = codes.shape
    out = np.empty((N, K), np.float64)
    rc = _load().oracle_dequant_fp8(_ptr(codes), _ptr(scales), E, N, K, int(expert), _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequant_fp8 failed: {rc}")
    return out


def dequant_nvfp4(packed: np.ndarray, sf: np.ndarray, scale_2: float, expert: int) -> np.ndarray:
    """Dense float64 [N, K] of one expert of an NVFP4 bank: packed [E, N, K/2], sf [E, N, K/16]."""
    packed = _c(packed, np.uint8)
    sf = _c(sf, np.uint8)
    E, N, K2 = packed.shape
    out = np.empty((N, 2 * K2), np.float64)
    rc = _load().oracle_dequant_nvfp4(_ptr(packed), _ptr(sf), ctypes.c_double(scale_2), E, N,
                                      2 * K2, int(expert), _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequant_nvfp4 failed: {rc}")
    return out


def route_permute(ids: np.ndarray, num_experts: int):
    """Counting sort of (token, slot) pairs by expert. Returns dict of int32 arrays and err."""
    ids = _c(ids, np.int32)
    T, topk = ids.shape
    P = T * topk
    counts = np.zeros(num_experts, np.int32)
    offsets = np.zeros(num_experts + 1, np.int32)
    sorted_pair = np.full(P, -1, np.int32)
    pair_to_sorted = np.full(P, -1, np.int32)
    err = np.zeros(1, np.int32)
    rc = _load().oracle_route_permute(_ptr(ids), T, topk, num_experts, _ptr(counts), _ptr(offsets),
                                      _ptr(sorted_pair), _ptr(pair_to_sorted), _ptr(err))
    if rc:
        raise ValueError(f"oracle_route_permute failed: {rc}")
    return dict(counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_to_sorted=pair_to_sorted, err=int(err[0]))


def _forward(kind, x_bf16_bits, ids, wts, bank, limit, tokens=None, intermediates=False,
             nthreads=0):
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(ids, np.int32)
    wts = _c(wts, np.float32)
    T, H = x.shape
    topk = ids.shape[1]
    tok = None if tokens is None else _c(tokens, np.int32)
    nt = T if tok is None else tok.size
    out = np.zeros((nt, H), np.float64)
    outb = np.zeros((nt, H), np.uint16)
    err = np.zeros(1, np.int32)
    if kind == "fp8":
        E, I, _ = bank["w_gate"].shape
    else:
        E, I, _ = bank["w_gate"].shape
    inter = {}
    if intermediates:
        for k in ("g", "u", "a"):
            inter[k] = np.zeros((nt * topk, I), np.float64)
        inter["y"] = np.zeros((nt * topk, H), np.float64)
    ip = lambda k: _ptr(inter[k]) if intermediates else None  # noqa: E731
    arrs = {k: _c(v, np.float32 if k.startswith("s_") else np.uint8)
            for k, v in bank.items() if isinstance(v, np.ndarray) and not k.startswith("scale2")}
    per_expert = kind == "nvfp4" and isinstance(bank["scale2_gate"], np.ndarray)
    if kind == "fp8":
        rc = lib.oracle_moe_fp8(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                _ptr(arrs["w_gate"]), _ptr(arrs["s_gate"]),
                                _ptr(arrs["w_up"]), _ptr(arrs["s_up"]),
                                _ptr(arrs["w_down"]), _ptr(arrs["s_down"]),
                                ctypes.c_double(limit), _ptr(tok), nt, _ptr(out), _ptr(outb),
                                ip("g"), ip("u"), ip("a"), ip("y"), int(nthreads), _ptr(err))
    elif per_expert:                   # one scale_2 per expert and projection, [E] float32 each
        s2 = {k: _c(bank[k], np.float32) for k in ("scale2_gate", "scale2_up", "scale2_down")}
        if any(v.shape != (E,) for v in s2.values()):
            raise ValueError("per-expert scale_2 arrays must have shape [E]")
        rc = lib.oracle_moe_nvfp4_expert_scale2(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                                _ptr(arrs["w_gate"]), _ptr(arrs["sf_gate"]), _ptr(s2["scale2_gate"]),
                                                _ptr(arrs["w_up"]), _ptr(arrs["sf_up"]), _ptr(s2["scale2_up"]),
                                                _ptr(arrs["w_down"]), _ptr(arrs["sf_down"]), _ptr(s2["scale2_down"]),
                                                1, ctypes.c_double(limit), _ptr(tok), nt, _ptr(out), _ptr(outb),
                                                ip("g"), ip("u"), ip("a"), ip("y"), int(nthreads), _ptr(err))
    else:
        rc = lib.oracle_moe_nvfp4(_ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(wts),
                                  _ptr(arrs["w_gate"]), _ptr(arrs["sf_gate"]),
                                  ctypes.c_float(bank["scale2_gate"]),
                                  _ptr(arrs["w_up"]), _ptr(arrs["sf_up"]),
                                  ctypes.c_float(bank["scale2_up"]),
                                  _ptr(arrs["w_down"]), _ptr(arrs["sf_down"]),
                                  ctypes.c_float(bank["scale2_down"]),
                                  ctypes.c_double(limit), _ptr(tok), nt, _ptr(out), _ptr(outb),
                                  ip("g"), ip("u"), ip("a"), ip("y"), int(nthreads), _ptr(err))
    if rc:
        raise ValueError(f"oracle forward ({kind}) failed: {rc}")
    res = dict(out=out, out_bf16=outb, err=int(err[0]))
    res.update(inter)
    return res


def moe_fp8(x_bf16_bits, ids, wts, bank, limit, tokens=None, intermediates=False, nthreads=0):
    """FP8 routed FFN. bank: dict w_gate/w_up [E,I,H] u8, w_down [E,H,I] u8, s_* fp32 block scales.

    x_bf16_bits: uint16 [T, H] (bf16 bit patterns). Returns dict(out float64 [n, H],
    out_bf16 uint16 [n, H], err, and g/u/a/y when intermediates=True).
    """
    return _forward("fp8", x_bf16_bits, ids, wts, bank, limit, tokens, intermediates, nthreads)


def moe_nvfp4(x_bf16_bits, ids, wts, bank, limit, tokens=None, intermediates=False, nthreads=0):
    """NVFP4 routed FFN. bank: w_* packed [E,N,K/2] u8, sf_* [E,N,K/16] u8, scale2_* floats, or
    float32 arrays [E] for one scale_2 per expert and projection."""
    return _forward("nvfp4", x_bf16_bits, ids, wts, bank, limit, tokens, intermediates, nthreads)


# ---- router (in front of the FFN) -----------------------------------------------------------------

def router_logits(x_bf16_bits: np.ndarray, w_bf16_bits: np.ndarray) -> np.ndarray:
    """FP64 logits [T][E] of bf16 x [T][H] against bf16 router rows [E][H]."""
    x = _c(x_bf16_bits, np.uint16)
    w = _c(w_bf16_bits, np.uint16)
    T, H = x.shape
    E = w.shape[0]
    out = np.zeros((T, E), dtype=np.float64)
    rc = _load().oracle_router_logits(_ptr(x), T, H, _ptr(w), E, _ptr(out))
    assert rc == 0, rc
    return out


def router_topk(logits: np.ndarray, bias, topk: int, routed_scale: float, renormalize: bool):
    """(ids [T][topk] int32, weights [T][topk] float64) from logits [T][E] (see moe_oracle.cpp)."""
    lg = _c(logits, np.float64)
    T, E = lg.shape
    b = None if bias is None else _c(bias, np.float64)
    ids = np.zeros((T, topk), dtype=np.int32)
    wts = np.zeros((T, topk), dtype=np.float64)
    rc = _load().oracle_router_topk(_ptr(lg), T, E, _ptr(b), topk, ctypes.c_double(routed_scale),
                                    int(bool(renormalize)), _ptr(ids), _ptr(wts))
    assert rc == 0, rc
    return ids, wts


# ---- shared expert and the layer epilogue -----------------------------------------------------

def shared_expert(x_bf16_bits, wg_bits, wu_bits, wd_bits, limit: float, nthreads: int = 0) -> np.ndarray:
    """FP64 dense SwiGLU MLP: x [T][H], wg/wu [S][H], wd [H][S] (bf16 bits) -> [T][H] float64."""
    x = _c(x_bf16_bits, np.uint16)
    wg, wu, wd = (_c(a, np.uint16) for a in (wg_bits, wu_bits, wd_bits))
    T, H = x.shape
    S = wg.shape[0]
    out = np.zeros((T, H), np.float64)
    rc = _load().oracle_shared_expert(_ptr(x), T, H, S, _ptr(wg), _ptr(wu), _ptr(wd),
                                      ctypes.c_double(limit), _ptr(out), int(nthreads))
    assert rc == 0, rc
    return out


def layer_epilogue(routed: np.ndarray, shared_bits=None, residual_bits=None):
    """(float64 sum, bf16 bits) of routed + shared + residual, rounded once."""
    r = _c(routed, np.float64)
    sh = None if shared_bits is None else _c(shared_bits, np.uint16)
    rs = None if residual_bits is None else _c(residual_bits, np.uint16)
    out = np.zeros(r.shape, np.float64)
    outb = np.zeros(r.shape, np.uint16)
    rc = _load().oracle_layer_epilogue(_ptr(r), _ptr(sh), _ptr(rs), ctypes.c_int64(r.size), _ptr(out),
                                       _ptr(outb))
    assert rc == 0, rc
    return out, outb

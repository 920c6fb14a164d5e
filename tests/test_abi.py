"""CPU-side checks of the C ABI: the library builds, loads and exports every declared symbol,
and the synchronous argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import math
import os
import re

import pytest

import __graft_entry__
from moe_expert_ffn_histogram_gb300 import _build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return capi.load()


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("moe_route_permute", "moe_fp8_forward", "moe_nvfp4_forward",
                     "moe_workspace_bytes"):
        assert required in names
    assert set(names) == set(capi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert capi.build_arch() == "sm_103a"


def test_build_entry_point_runs():
    __graft_entry__.build()


def test_workspace_bytes_is_pure_and_monotone(lib):
    a = capi.workspace_bytes(1, 7168, 2048, 256, 8, capi.FMT_FP8)
    assert a > 0 and a == capi.workspace_bytes(1, 7168, 2048, 256, 8, capi.FMT_FP8)
    b = capi.workspace_bytes(8, 7168, 2048, 256, 8, capi.FMT_FP8)
    assert b > a
    # NVFP4 with T > 8 and K not a multiple of 256 runs in sub-batches of <= 8 rows (the
    # workspace stops growing); otherwise T > 8 takes the grouped-GEMM tier, whose workspace holds
    # the expert-sorted rows
    n8 = capi.workspace_bytes(8, 5120, 1408, 160, 8, capi.FMT_NVFP4)
    assert capi.workspace_bytes(4096, 5120, 1408, 160, 8, capi.FMT_NVFP4) == n8
    assert capi.workspace_bytes(4096, 5120, 1536, 160, 8, capi.FMT_NVFP4) >= 4096 * 8 * 5120 * 2
    big = capi.workspace_bytes(4096, 7168, 2048, 256, 8, capi.FMT_FP8)
    assert big >= 4096 * 8 * 7168 * 4 + 4096 * 8 * 2048 * 2 + 4096 * 7168 * 2
    # a [P][I] f16 activation buffer is the bulk of it
    assert b >= 8 * 8 * 2048 * 2
    for bad in [(0, 256, 128, 16, 8), (1, 200, 128, 16, 8), (1, 256, 100, 16, 8),
                (1, 256, 128, 0, 8), (1, 256, 128, 16, 9), (1, 256, 128, 16, 0)]:
        assert capi.workspace_bytes(*bad, capi.FMT_FP8) == 0
    assert capi.workspace_bytes(1, 256, 128, 16, 8, 7) == 0


def test_nvfp4_workspace_holds_the_single_token_activation_scales(lib):
    """One NVFP4 token's gate/up writes one activation scale per 32 features (FP8: per 64), so its
    workspace's scale region holds topk * I/32 fp32 values instead of topk * I/64 (each region is
    rounded up to 256 bytes); everything else is the same."""
    def ru(n):
        return (n + 255) // 256 * 256
    for H, I in [(5120, 1536), (7168, 2048), (256, 128), (512, 8192)]:
        f8 = capi.workspace_bytes(1, H, I, 160, 8, capi.FMT_FP8)
        f4 = capi.workspace_bytes(1, H, I, 160, 8, capi.FMT_NVFP4)
        assert f4 - f8 == ru(8 * (I // 32) * 4) - ru(8 * (I // 64) * 4)


FAKE = ctypes.c_void_p(0x10000000)     # never dereferenced: every call below fails its checks


def _fp8_call(lib, **over):
    args = dict(x=FAKE, T=1, H=256, I=128, E=16, topk=8, ids=FAKE, wts=FAKE, wg=FAKE, sg=FAKE,
                wu=FAKE, su=FAKE, wd=FAKE, sd=FAKE, limit=7.0, out=FAKE, ws=FAKE, ws_bytes=1 << 30,
                err=None, stream=None)
    args.update(over)
    return lib.moe_fp8_forward(*args.values())


def test_fp8_forward_rejects_bad_arguments(lib):
    assert _fp8_call(lib, x=None) == -1
    assert _fp8_call(lib, wd=None) == -1
    assert _fp8_call(lib, out=None) == -1
    assert _fp8_call(lib, T=0) == -2
    assert _fp8_call(lib, H=200) == -2
    assert _fp8_call(lib, I=64) == -2
    assert _fp8_call(lib, topk=9) == -2
    assert _fp8_call(lib, E=0) == -2
    assert _fp8_call(lib, limit=0.0) == -4
    assert _fp8_call(lib, limit=-1.0) == -4
    assert _fp8_call(lib, limit=math.nan) == -4
    assert _fp8_call(lib, ws=None) == -3
    assert _fp8_call(lib, ws_bytes=16) == -3
    assert _fp8_call(lib, ws=ctypes.c_void_p(0x10000010)) == -3     # not 256-byte aligned
    assert _fp8_call(lib, wg=ctypes.c_void_p(0x10000008)) == -7     # weights not 16-B aligned
    assert _fp8_call(lib, x=ctypes.c_void_p(0x10000002)) == -7
    # x staging for 8 columns would not fit in shared memory
    assert _fp8_call(lib, T=8, H=128 * 128) == -6


def test_nvfp4_forward_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=FAKE, T=1, H=256, I=128, E=16, topk=8, ids=FAKE, wts=FAKE, wg=FAKE, sfg=FAKE,
                 s2g=1.0, wu=FAKE, sfu=FAKE, s2u=1.0, wd=FAKE, sfd=FAKE, s2d=1.0, limit=7.0,
                 out=FAKE, ws=FAKE, ws_bytes=1 << 30, err=None, stream=None)
        a.update(over)
        return lib.moe_nvfp4_forward(*a.values())
    assert call(sfd=None) == -1
    assert call(s2g=math.inf) == -4
    assert call(s2d=math.nan) == -4
    assert call(limit=math.nan) == -4
    assert call(T=-3) == -2
    assert call(ws_bytes=0) == -3


def test_nvfp4_expert_scale2_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=FAKE, T=1, H=256, I=128, E=16, topk=8, ids=FAKE, wts=FAKE, wg=FAKE, sfg=FAKE,
                 s2g=FAKE, wu=FAKE, sfu=FAKE, s2u=FAKE, wd=FAKE, sfd=FAKE, s2d=FAKE, stride=1,
                 limit=7.0, out=FAKE, ws=FAKE, ws_bytes=1 << 30, err=None, stream=None)
        a.update(over)
        return lib.moe_nvfp4_forward_expert_scale2(*a.values())
    assert call(s2u=None) == -1
    assert call(stride=0) == -4
    assert call(s2d=ctypes.c_void_p(FAKE.value + 2)) == -7   # a table that is not 4-byte aligned
    assert call(limit=math.nan) == -4
    assert call(T=-3) == -2
    assert call(ws_bytes=0) == -3


def test_nvfp4_layer_expert_scale2_rejects_bad_arguments(lib):
    def call(**over):
        a = dict(x=FAKE, T=1, H=256, I=128, E=16, topk=8, ids=FAKE, wts=FAKE, wg=FAKE, sfg=FAKE,
                 s2g=FAKE, wu=FAKE, sfu=FAKE, s2u=FAKE, wd=FAKE, sfd=FAKE, s2d=FAKE, stride=3,
                 limit=7.0, shared=None, residual=None, out=FAKE, ws=FAKE, ws_bytes=1 << 30, err=None,
                 stream=None)
        a.update(over)
        return lib.moe_nvfp4_forward_layer_expert_scale2(*a.values())
    assert call(s2g=None) == -1
    assert call(stride=-1) == -4
    assert call(shared=ctypes.c_void_p(FAKE.value + 8)) == -7
    assert call(ws_bytes=0) == -3


def test_route_permute_rejects_bad_arguments(lib):
    f = lib.moe_route_permute
    assert f(None, 1, 8, 16, FAKE, FAKE, FAKE, FAKE, None, None) == -1
    assert f(FAKE, 0, 8, 16, FAKE, FAKE, FAKE, FAKE, None, None) == -2
    assert f(FAKE, 1, 8, 0, FAKE, FAKE, FAKE, FAKE, None, None) == -2
    assert f(FAKE, 1, 8, 5000, FAKE, FAKE, FAKE, FAKE, None, None) == -6


def test_stage_entry_points_reject_wide_batches(lib):
    assert lib.moe_plan(9, 256, 128, 16, 8, capi.FMT_FP8, FAKE, FAKE, 1 << 30, None, None) == -6
    assert lib.moe_plan(2, 256, 128, 16, 8, 3, FAKE, FAKE, 1 << 30, None, None) == -4
    assert lib.moe_fp8_gate_up(FAKE, 9, 256, 128, 16, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 7.0, FAKE,
                               1 << 30, None, None) == -6


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        capi.load(str(tmp_path / "missing.so"))


def test_router_rejects_bad_arguments(lib):
    f = lib.moe_router

    def call(**over):
        a = dict(x=FAKE, T=2, H=256, w=FAKE, bias=None, E=64, topk=8, scale=1.0, renorm=1,
                 logits=None, ids=FAKE, wts=FAKE, ws=FAKE, ws_bytes=1 << 30, stream=None)
        a.update(over)
        return f(*a.values())
    assert call(x=None) == -1
    assert call(ids=None) == -1
    assert call(E=8) == -2                 # fewer than 16 experts
    assert call(E=100) == -2               # not a multiple of 16
    assert call(E=2048) == -2
    assert call(H=250) == -2
    assert call(topk=9) == -2
    assert call(topk=0) == -2
    assert call(scale=0.0) == -4
    assert call(scale=math.inf) == -4
    assert call(x=ctypes.c_void_p(0x10000008)) == -7
    assert call(ws=None) == -3
    assert lib.moe_router_workspace_bytes(2, 250, 64) == 0
    assert lib.moe_router_workspace_bytes(2, 256, 64) > 0


def test_stage_times_without_timing(lib):
    assert lib.moe_stage_times(None, None, 4) == -1
    assert capi.stage_times() == []            # timing off: nothing recorded


def test_stream_read_rejects_bad_arguments(lib):
    # argument checks come before any CUDA call, so they run without a GPU
    assert lib.moe_stream_read(None, 1024, FAKE, None) == -1
    assert lib.moe_stream_read(FAKE, 1024, None, None) == -1
    assert lib.moe_stream_read(FAKE, 0, FAKE, None) == -2
    assert lib.moe_stream_read(FAKE, 1000, FAKE, None) == -2
    assert lib.moe_stream_read(ctypes.c_void_p(FAKE.value + 8), 1024, FAKE, None) == -7
    assert lib.moe_stream_read(FAKE, 1024, ctypes.c_void_p(FAKE.value + 2), None) == -7

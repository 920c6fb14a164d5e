"""GPU test of moe_fp8_forward_noalloc, the forward for callers that cannot allocate device memory
(plugins that only get input/output pointers, loops that forbid cudaMalloc because it can
synchronise the device). It must give the same results as moe_fp8_forward with a caller-provided
workspace, on two calls in a row (its built-in scratch keeps the previous call's contents).

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_ffn_histogram_gb300 import _build, capi, inputs

from helpers import bf16_to_f64, check_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SCRATCH_BYTES = 1 << 20      # MOE_NOALLOC_SCRATCH_BYTES in include/moe_ffn.h


def _entry():
    _build.build()
    lib = capi.load()
    f = lib.moe_fp8_forward_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.restype = i32
    f.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                  vp, vp, vp]
    return f


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(f, wl, out, err=None):
    b = wl.bank
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return f(_p(wl.x), wl.T, wl.H, wl.I, wl.E, wl.topk, _p(wl.ids), _p(wl.wts), _p(b.w_gate),
             _p(b.s_gate), _p(b.w_up), _p(b.s_up), _p(b.w_down), _p(b.s_down), wl.limit, _p(out),
             _p(err), stream)


@pytest.fixture(scope="module")
def entry():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return _entry()


@pytest.mark.parametrize("T", [1, 5, 17])
def test_noalloc_matches_workspace_entry_point_two_calls(entry, T):
    """Two calls in a row with different inputs; each is bit-identical to moe_fp8_forward with a
    caller workspace (the same kernels on the same inputs). T = 5 runs the cooperative kernel
    (its barrier word in the scratch), T = 17 the grouped-GEMM tier, whose plan, sorted copies
    and intermediates fill most of the 1 MiB and are rewritten in stream order by each call."""
    assert capi.workspace_bytes(T, 1024, 512, 16, 8, capi.FMT_FP8) <= SCRATCH_BYTES
    bank = inputs.make_fp8_bank(16, 1024, 512, seed=404, device=DEV)
    for call in range(2):                      # two calls in a row, different inputs
        wl = inputs.make_custom("fp8", T, 1024, 512, 16, seed=500 + call, device=DEV)
        wl.bank = bank
        ref = capi.fp8_forward(wl.x, wl.ids, wl.wts, bank, wl.limit)
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _noalloc(entry, wl, out, err) == 0
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"noalloc T={T} call {call}"
        check_close(bf16_to_f64(out), bf16_to_f64(ref), f"noalloc T={T} call {call}")
        assert int(err.item()) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(entry):
    need = capi.workspace_bytes(8, 4096, 8192, 256, 8, capi.FMT_FP8)
    assert need > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000000)         # never dereferenced: rejected before any work
    rc = entry(fake, 8, 4096, 8192, 256, 8, fake, fake, fake, fake, fake, fake, fake, fake, 7.0,
               fake, None, None)
    assert rc == -3                            # MOE_ERR_WORKSPACE
    rc = entry(None, 1, 256, 128, 16, 8, fake, fake, fake, fake, fake, fake, fake, fake, 7.0,
               fake, None, None)
    assert rc == -1                            # same argument checks as moe_fp8_forward

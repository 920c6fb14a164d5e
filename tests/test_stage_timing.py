"""Stage timing (moe_stage_timing / moe_stage_times): the forward paths name their stages, the
times are positive device intervals that add up to the forward, and switching it off stops it."""
import pytest
import torch

from moe_expert_ffn_histogram_gb300 import capi, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _timed(wl):
    capi.stage_timing(True)
    try:
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
        e.record()
        st = capi.stage_times()
        torch.cuda.synchronize()
        return st, s.elapsed_time(e)
    finally:
        capi.stage_timing(False)


@pytest.mark.parametrize("T,names", [
    (1, ["plan", "gate_up", "down_combine"]),
    (5, ["fused"]),
    # a finite clamp limit bounds the activations: the gate/up GEMM writes them in f16 itself
    (64, ["route_plan", "tile_list", "x_prep", "gate_up_gemm", "down_gemm", "combine"]),
])
def test_stage_names_and_times(T, names):
    wl = inputs.make_custom("fp8", T, 512, 256, 16, seed=900 + T, device=DEV)
    capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)      # warm-up (module load, attributes)
    st, total = _timed(wl)
    assert [n for n, _ in st] == names
    assert all(ms >= 0.0 for _, ms in st)
    assert sum(ms for _, ms in st) <= total * 1.05 + 0.05


def test_stage_names_without_clamp():
    """No clamp (limit = +inf): the activations need their range scale, so act_prep runs."""
    wl = inputs.make_custom("fp8", 64, 512, 256, 16, seed=964, device=DEV, limit=float("inf"))
    capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
    st, _ = _timed(wl)
    assert [n for n, _ in st] == ["route_plan", "tile_list", "x_prep", "gate_up_gemm", "act_prep",
                                  "down_gemm", "combine"]


def test_timing_off_records_nothing():
    wl = inputs.make_custom("fp8", 1, 512, 256, 16, seed=990, device=DEV)
    _timed(wl)
    capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
    torch.cuda.synchronize()
    assert capi.stage_times() == []

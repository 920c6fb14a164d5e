"""GPU parity of the router (moe_router) against the FP64 oracle, and the router feeding the FFN.

The selection is an integer decision taken from floating-point scores: the oracle takes it from
the kernel's own fp32 logits (the kernel's precision), in FP64, and the indices must match exactly
except where the top-k boundary is a near-tie, where the kernel's pick only has to be valid.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_histogram_gb300 import capi, inputs
from helpers import bf16_to_f64, check_close, oracle_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _make(T, H, E, seed, bias=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    b = (torch.randn(E, generator=g) * 0.05).float() if bias else None
    return x.to(DEV), w.to(DEV), None if b is None else b.to(DEV)


def _check(x, w, b, topk, scale, renorm):
    ids, wts, logits = capi.router(x, w, topk, scale, renorm, bias=b, want_logits=True)
    torch.cuda.synchronize()
    lg = logits.double().cpu().numpy()
    ref = oracle.router_logits(_bits(x), _bits(w))
    err = np.abs(lg - ref)
    assert err.max() <= 1e-5 * max(1.0, np.abs(ref).max()), err.max()
    bias = None if b is None else b.double().cpu().numpy()
    o_ids, o_w = oracle.router_topk(lg, bias, topk, scale, renorm)      # decision on the kernel's logits
    g_ids = ids.cpu().numpy()
    g_w = wts.double().cpu().numpy()
    sig = 1.0 / (1.0 + np.exp(-lg))
    score = sig + (0.0 if bias is None else bias)
    E = lg.shape[1]
    near = 0
    for t in range(lg.shape[0]):
        srt = np.sort(score[t])[::-1]
        margin = srt[topk - 1] - srt[topk] if topk < E else 1.0
        gaps = np.diff(srt[:topk + 1])
        if margin > 1e-6 and (gaps.size == 0 or np.min(np.abs(gaps)) > 1e-6):
            assert g_ids[t].tolist() == o_ids[t].tolist(), (t, g_ids[t], o_ids[t])
            assert np.allclose(g_w[t], o_w[t], rtol=2e-6, atol=1e-7)
        else:                                   # near-tie: a valid pick, distinct, weights consistent
            near += 1
            assert len(set(g_ids[t].tolist())) == topk
            assert score[t, g_ids[t]].min() >= srt[topk - 1] - 1e-6
            picked = sig[t, g_ids[t]]
            ref_w = scale * (picked / picked.sum() if renorm else picked)
            assert np.allclose(g_w[t], ref_w, rtol=2e-6, atol=1e-7)
    return near


@pytest.mark.parametrize("T,H,E,topk,scale,renorm", [
    (1, 7168, 256, 8, 2.5, True),     # decode: K split over the grid
    (7, 1024, 64, 8, 1.0, True),
    (33, 512, 160, 6, 1.0, False),    # wide path with a ragged 32-token tile
    (300, 2048, 256, 8, 2.5, True),
])
def test_router_parity(T, H, E, topk, scale, renorm):
    x, w, b = _make(T, H, E, seed=100 + T)
    near = _check(x, w, b, topk, scale, renorm)
    assert near <= max(1, T // 50)


def test_router_exact_ties_go_to_the_lower_index():
    T, H, E = 9, 256, 32
    g = torch.Generator(device="cpu").manual_seed(7)
    u = torch.randn(H, generator=g)
    # a shared direction u with logits ~2-2.6 on it (sigmoid far from fp32 saturation), and small
    # random rows elsewhere
    x = (torch.randn(T, H, generator=g) + u).to(torch.bfloat16)
    w = (torch.randn(E, H, generator=g) * H ** -0.5 * 0.1)
    w[3] = w[20] = 0.01 * u                    # duplicate rows: bitwise-equal logits, the two best
    w[11] = w[30] = 0.008 * u                  # and the next two
    x, w = x.to(DEV), w.to(torch.bfloat16).to(DEV)
    ids, wts, logits = capi.router(x, w, 4, 1.0, True, want_logits=True)
    torch.cuda.synchronize()
    lg = logits.cpu()
    assert torch.equal(lg[:, 3], lg[:, 20]) and torch.equal(lg[:, 11], lg[:, 30])
    o_ids, _ = oracle.router_topk(lg.double().numpy(), None, 4, 1.0, True)
    assert ids.cpu().numpy().tolist() == o_ids.tolist()
    assert all(row == [3, 20, 11, 30] for row in ids.cpu().numpy().tolist())


def test_router_feeds_the_ffn():
    """Router picks and weights drive moe_fp8_forward; the result matches the oracle FFN."""
    T, H, I, E = 6, 256, 128, 16
    wl = inputs.make_custom("fp8", T, H, I, E, seed=55, device=DEV)
    x, w, b = _make(T, H, E, seed=56)
    wl.x = x
    ids, wts, _ = capi.router(wl.x, w, 8, 1.0, True, bias=b)
    wl.ids, wl.wts = ids, wts
    out = capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
    torch.cuda.synchronize()
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], "router -> ffn")


def test_router_workspace_and_errors():
    x, w, b = _make(4, 256, 64, seed=3)
    n = capi.load().moe_router_workspace_bytes(4, 256, 64)
    assert n > 0 and capi.load().moe_router_workspace_bytes(4, 250, 64) == 0
    with pytest.raises(capi.MoeError):
        capi.router(x, w, 9, 1.0, True)             # topk > 8
    with pytest.raises(capi.MoeError):
        capi.router(x, w, 8, 0.0, True)             # routed_scale must be > 0


def test_router_minus_inf_bias_leaves_fewer_finite_scores_than_topk():
    """A -inf bias masks all but topk-1 experts: the picks are those topk-1 and then the masked
    expert of lowest index (equal -inf scores go to the lower index), exactly the oracle's
    decision on the kernel's logits; ids stay distinct and in [0, E)."""
    T, H, E, topk = 5, 256, 64, 8
    x, w, _ = _make(T, H, E, seed=21, bias=False)
    b = torch.full((E,), float("-inf"), dtype=torch.float32, device=DEV)
    keep = torch.tensor([5, 17, 33, 40, 41, 50, 63], device=DEV)
    b[keep] = 0.0
    ids, wts, logits = capi.router(x, w, topk, 1.0, True, bias=b, want_logits=True)
    torch.cuda.synchronize()
    g_ids = ids.cpu().numpy()
    o_ids, o_w = oracle.router_topk(logits.double().cpu().numpy(), b.double().cpu().numpy(), topk, 1.0, True)
    assert g_ids.tolist() == o_ids.tolist()
    for t in range(T):
        assert sorted(g_ids[t, :topk - 1].tolist()) == keep.cpu().tolist()
        assert g_ids[t, topk - 1] == 0
    assert np.allclose(wts.double().cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)


def test_router_nan_logits_give_valid_distinct_ids():
    """NaN logits (a NaN router row, and a token whose x is NaN) never produce an index outside
    [0, E) or a repeated pick; experts with a number for a score come before NaN ones."""
    T, H, E, topk = 4, 256, 32, 8
    x, w, b = _make(T, H, E, seed=22)
    w = w.clone()
    w[[2, 9, 30]] = float("nan")                 # three experts score NaN for every token
    x = x.clone()
    x[3] = float("nan")                          # token 3 scores NaN for every expert
    ids, wts, _ = capi.router(x, w, topk, 1.0, True, bias=b)
    torch.cuda.synchronize()
    g = ids.cpu().numpy()
    assert ((g >= 0) & (g < E)).all()
    for t in range(T):
        assert len(set(g[t].tolist())) == topk
    for t in range(3):                           # finite scores exist for 29 experts: NaN ones lose
        assert not set(g[t].tolist()) & {2, 9, 30}
    assert g[3].tolist() == list(range(topk))    # all NaN: by index

"""GPU parity of the MoE layer epilogue (shared expert + residual fused into the combine) and of the
BF16 shared expert, against the FP64 oracle."""
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


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("fmt,T,H,I,E", [("fp8", 1, 256, 128, 16), ("fp8", 5, 384, 256, 12),
                                         ("fp8", 40, 256, 256, 10), ("nvfp4", 3, 256, 128, 9),
                                         ("nvfp4", 64, 512, 256, 12)])
def test_layer_epilogue_parity(fmt, T, H, I, E):
    wl = inputs.make_custom(fmt, T, H, I, E, seed=300 + T, device=DEV)
    shared = _rand_bf16((T, H), 301 + T, 0.05)
    resid = _rand_bf16((T, H), 302 + T, 1.0)
    out = capi.forward_layer(wl.x, wl.ids, wl.wts, wl.bank, wl.limit, shared=shared, residual=resid)
    plain = capi.forward_layer(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
    torch.cuda.synchronize()
    ref = oracle_for(wl)
    _, ref_b = oracle.layer_epilogue(ref["out"], _bits(shared), _bits(resid))
    want = np.array([oracle.bf16_value(int(v)) for v in ref_b.reshape(-1)]).reshape(ref_b.shape)
    check_close(bf16_to_f64(out), want, f"layer {fmt} T={T}")
    # without shared / residual the layer entry is the plain forward, bit for bit
    assert torch.equal(plain.view(torch.int16),
                       capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit).view(torch.int16))


@pytest.mark.parametrize("T", [1, 5, 40])
def test_layer_epilogue_with_expert_scale2(T):
    """moe_nvfp4_forward_layer_expert_scale2: one scale_2 per expert and projection, with the shared
    expert and the residual in the combine, on the single-token, fused and grouped tiers."""
    E, H, I = 10, 512, 256
    bank = inputs.make_nvfp4_bank_expert_scale2(E, H, I, seed=310 + T, device=DEV)
    x = inputs.normal_activations(T, H, 310 + T, DEV)
    ids = inputs.make_routes("uniform", T, E, 310 + T).to(DEV)
    wts = inputs.softmax_route_weights(T, 310 + T).to(DEV)
    wl = inputs.Workload(f"layer_s2_T{T}", "nvfp4", T, H, I, E, inputs.TOPK, x, ids, wts, bank, inputs.LIMIT)
    shared = _rand_bf16((T, H), 311 + T, 0.05)
    resid = _rand_bf16((T, H), 312 + T, 1.0)
    out = capi.forward_layer(wl.x, wl.ids, wl.wts, bank, wl.limit, shared=shared, residual=resid)
    plain = capi.forward_layer(wl.x, wl.ids, wl.wts, bank, wl.limit)
    torch.cuda.synchronize()
    ref = oracle_for(wl)
    _, ref_b = oracle.layer_epilogue(ref["out"], _bits(shared), _bits(resid))
    want = np.array([oracle.bf16_value(int(v)) for v in ref_b.reshape(-1)]).reshape(ref_b.shape)
    check_close(bf16_to_f64(out), want, f"layer per-expert scale_2 T={T}")
    assert torch.equal(plain.view(torch.int16),
                       capi.forward(wl.x, wl.ids, wl.wts, bank, wl.limit).view(torch.int16))


@pytest.mark.parametrize("T,H,S", [(1, 512, 256), (7, 256, 512), (100, 512, 256)])
def test_shared_expert_parity(T, H, S):
    x = _rand_bf16((T, H), 400 + T)
    wg = _rand_bf16((S, H), 401, H ** -0.5)
    wu = _rand_bf16((S, H), 402, H ** -0.5)
    wd = _rand_bf16((H, S), 403, S ** -0.5)
    out = capi.shared_expert(x, wg, wu, wd, 7.0)
    torch.cuda.synchronize()
    ref = oracle.shared_expert(_bits(x), _bits(wg), _bits(wu), _bits(wd), 7.0)
    check_close(bf16_to_f64(out), ref, f"shared expert T={T}")


def test_full_layer_router_shared_residual():
    """router -> routed FFN with the shared expert and residual in the combine."""
    T, H, I, E, S = 6, 256, 128, 16, 128
    wl = inputs.make_custom("fp8", T, H, I, E, seed=500, device=DEV)
    rw = _rand_bf16((E, H), 501, H ** -0.5)
    ids, wts, _ = capi.router(wl.x, rw, 8, 2.5, True)
    wl.ids, wl.wts = ids, wts
    sh = capi.shared_expert(wl.x, _rand_bf16((S, H), 502, H ** -0.5), _rand_bf16((S, H), 503, H ** -0.5),
                            _rand_bf16((H, S), 504, S ** -0.5), 7.0)
    resid = _rand_bf16((T, H), 505)
    out = capi.forward_layer(wl.x, wl.ids, wl.wts, wl.bank, wl.limit, shared=sh, residual=resid)
    torch.cuda.synchronize()
    _, ref_b = oracle.layer_epilogue(oracle_for(wl)["out"], _bits(sh), _bits(resid))
    want = np.array([oracle.bf16_value(int(v)) for v in ref_b.reshape(-1)]).reshape(ref_b.shape)
    check_close(bf16_to_f64(out), want, "router -> layer")

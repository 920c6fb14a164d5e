"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each test fixes a part of the oracle with an independent fact: a library decoder (torch's
float8_e4m3fn), the published E2M1 table, hand-built bytes with a closed-form answer, the pages'
worked combine example, brute-force dense float64 matmul, or a brute-force stable sort.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_histogram_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- number formats ------------------------------------------------------------------------

def test_e4m3_all_codes_match_torch_decoder():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if np.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
            assert math.copysign(1.0, v) == math.copysign(1.0, ref[c]), c


def test_e4m3_special_codes():
    assert oracle.e4m3_value(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x40) == 2.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e2m1_table():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for n in range(8):
        assert oracle.e2m1_value(n) == grid[n]
        assert oracle.e2m1_value(n | 8) == -grid[n]
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_bf16_widen_and_round():
    bits = np.random.default_rng(0).integers(0, 1 << 16, 4000, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits, ref):
        v = oracle.bf16_value(int(b))
        assert (math.isnan(v) and math.isnan(r)) or v == r
    # f32-representable values: torch's f32 -> bf16 cast is round-to-nearest-even
    vals = np.random.default_rng(1).standard_normal(4000).astype(np.float32) * 37.0
    ref_bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, rb in zip(vals, ref_bits):
        assert oracle.bf16_round(float(v)) == int(rb)
    # hand cases: ties to even, and one that a double->f32->bf16 path would round wrongly
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_round(-0.0) == 0x8000
    assert oracle.bf16_round(float("inf")) == 0x7F80


# ---- clamped SwiGLU (spark_model glm5next_mlp forward.rs, `swiglu_rows`) ------------------------

SILU_1 = 0.73105857863000487925   # 1/(1+e^-1), 20 digits (sympy)
SILU_7 = 6.9936226416391954825    # 7/(1+e^-7)
SILU_M9 = -0.0011105511838760855677  # -9/(1+e^9)


def test_swiglu_closed_form_values():
    L = 7.0
    assert oracle.clamped_swiglu(1.0, 1.0, L) == pytest.approx(SILU_1, rel=1e-15)
    assert oracle.clamped_swiglu(0.0, 5.0, L) == 0.0
    # gate is clamped from above only
    assert oracle.clamped_swiglu(8.0, 1.0, L) == oracle.clamped_swiglu(7.0, 1.0, L)
    assert oracle.clamped_swiglu(7.0, 1.0, L) == pytest.approx(SILU_7, rel=1e-15)
    assert oracle.clamped_swiglu(-9.0, 1.0, L) == pytest.approx(SILU_M9, rel=1e-12)
    assert oracle.clamped_swiglu(-100.0, 1.0, L) == pytest.approx(-100.0 / (1 + math.exp(100)), rel=1e-12)
    # up is clamped both ways
    assert oracle.clamped_swiglu(1.0, 9.0, L) == pytest.approx(SILU_1 * 7.0, rel=1e-15)
    assert oracle.clamped_swiglu(1.0, -9.0, L) == pytest.approx(-SILU_1 * 7.0, rel=1e-15)
    assert oracle.clamped_swiglu(1.0, 7.0, L) == oracle.clamped_swiglu(1.0, 9.0, L)
    assert oracle.clamped_swiglu(1.0, -7.0, L) == oracle.clamped_swiglu(1.0, -1e9, L)
    # no limit: plain silu(g) * u
    inf = float("inf")
    assert oracle.clamped_swiglu(20.0, 30.0, inf) == pytest.approx(20.0 / (1 + math.exp(-20)) * 30.0, rel=1e-15)


# ---- combine (ep_step_fp8_gate.rs, `combine_down_rows_host`) ------------------------------------

def test_combine_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "combine_worked_example.json")))
    down = np.array(g["down"], np.float64)
    w = np.array(g["weights"], np.float64)
    out = oracle.combine(down, w, 1, 8, 2)
    assert out.tolist() == [g["expected"]]
    with pytest.raises(ValueError):
        oracle.combine(down.reshape(-1)[:-1], w, 1, 8, 2)


# ---- route fixture and weights (input generator; worked values from the pages) ------------------

def test_route_fixture_worked_values():
    g = json.load(open(os.path.join(GOLDEN, "route_fixture.json")))
    r = inputs.fixture_routes(g["tokens"], g["experts"])
    assert r.tolist() == g["routes"]
    w = inputs.fixture_route_weights(g["tokens"], g["weight_shift"])
    expect = [float(np.float32(v) / np.float32(g["weights_denominator"])) for v in g["weights_sorted_per_token"]]
    for row in w:
        assert sorted(row.tolist()) == pytest.approx(expect, abs=0)
        assert abs(float(row.sum()) - 1.0) <= np.finfo(np.float32).eps
    assert w[0].tolist() != w[1].tolist()
    assert inputs.fixture_routes(1, 16).tolist() == [[0, 2, 4, 6, 8, 10, 12, 14]]


# ---- permutation: brute-force stable sort -------------------------------------------------------

@pytest.mark.parametrize("T,E,seed", [(1, 16, 0), (3, 5, 1), (37, 64, 2), (256, 256, 3)])
def test_route_permute_matches_bruteforce(T, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, 8)).astype(np.int32)
    ids[rng.random((T, 8)) < 0.1] = -1           # unfilled slots
    r = oracle.route_permute(ids, E)
    flat = ids.reshape(-1)
    valid = [p for p in range(flat.size) if 0 <= flat[p] < E]
    order = sorted(valid, key=lambda p: (flat[p], p))
    assert r["sorted_pair"][: len(order)].tolist() == order
    assert (r["sorted_pair"][len(order):] == -1).all()
    assert r["counts"].tolist() == [int((flat == e).sum()) for e in range(E)]
    assert r["offsets"][0] == 0 and r["offsets"][-1] == len(order)
    assert (np.diff(r["offsets"]) == r["counts"]).all()
    for s, p in enumerate(order):
        assert r["pair_to_sorted"][p] == s
    assert all(r["pair_to_sorted"][p] == -1 for p in range(flat.size) if p not in set(valid))
    assert r["err"] == 0


def test_route_permute_flags_out_of_range():
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 99]], np.int32)
    r = oracle.route_permute(ids, 8)
    assert r["err"] & 1
    assert r["offsets"][-1] == 7
    assert r["pair_to_sorted"][7] == -1


# ---- dequantisation with hand-built bytes -------------------------------------------------------

def test_fp8_dequant_hand_built():
    E, N, K = 2, 256, 128
    codes = np.zeros((E, N, K), np.uint8)
    scales = np.ones((E, N // 128, K // 128), np.float32)
    codes[1, 200, 5] = 0x38          # 1.0
    scales[1, 1, 0] = 0.5            # rows 128..255 of expert 1
    codes[1, 3, 7] = 0xC0            # -2.0, in block (0, 0) with scale 1
    d = oracle.dequant_fp8(codes, scales, 1)
    assert d[200, 5] == 0.5
    assert d[3, 7] == -2.0
    assert np.count_nonzero(d) == 2
    assert np.count_nonzero(oracle.dequant_fp8(codes, scales, 0)) == 0


def test_nvfp4_dequant_nibble_order_and_scales():
    E, N, K = 1, 2, 32
    packed = np.zeros((E, N, K // 2), np.uint8)
    sf = np.zeros((E, N, K // 16), np.uint8)
    packed[0, 0, 0] = 0x21            # element 0 = low nibble 0x1 (0.5), element 1 = 0x2 (1.0)
    sf[0, 0, 0] = 0x38                # 1.0
    packed[0, 1, 9] = 0x07            # element 18 = 6.0, element 19 = 0
    sf[0, 1, 1] = 0x38                # elements 16..31 of row 1
    d = oracle.dequant_nvfp4(packed, sf, 2.0, 0)
    assert d[0, 0] == 1.0 and d[0, 1] == 2.0          # x scale_2 = 2
    assert d[1, 18] == 12.0                           # 6 * 1.0 * 2.0
    assert np.count_nonzero(d) == 3


def test_hand_built_fp8_ffn_closed_form():
    """One expert, identity-like weights: every output is a closed-form number."""
    H = I = 128
    wg = np.zeros((1, I, H), np.uint8); wg[0, :, 0] = 0x38           # g_n = x0 * 1.0 * sg
    wu = np.zeros((1, I, H), np.uint8); wu[0, :, 1] = 0x40           # u_n = x1 * 2.0 * su
    wd = np.zeros((1, H, I), np.uint8); wd[0, np.arange(H), np.arange(I)] = 0x38   # y_j = a_j * sd
    bank = dict(w_gate=wg, s_gate=np.full((1, 1, 1), 0.5, np.float32),
                w_up=wu, s_up=np.full((1, 1, 1), 1.0, np.float32),
                w_down=wd, s_down=np.full((1, 1, 1), 0.25, np.float32))
    x = torch.zeros(1, H, dtype=torch.bfloat16); x[0, 0] = 1.0; x[0, 1] = 3.0
    xb = x.view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[0]], np.int32)
    w = np.array([[0.5]], np.float32)
    r = oracle.moe_fp8(xb, ids, w, bank, limit=7.0)
    g, u = 0.5, 6.0
    expect = 0.5 * (g / (1 + math.exp(-g))) * min(u, 7.0) * 0.25
    assert np.allclose(r["out"], expect, rtol=1e-15, atol=0)
    r2 = oracle.moe_fp8(xb, ids, w, bank, limit=4.0)          # up clamped to 4
    assert np.allclose(r2["out"], 0.5 * (g / (1 + math.exp(-g))) * 4.0 * 0.25, rtol=1e-15)


# ---- brute force: dense float64 matmul on tiny banks --------------------------------------------

def _dense_fp8(codes, scales):
    E, N, K = codes.shape
    w = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.repeat(np.repeat(scales.astype(np.float64), 128, axis=1), 128, axis=2)
    return w * s


def _dense_nvfp4(packed, sf, scale_2):
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6])
    lo = grid[packed & 0xF]
    hi = grid[packed >> 4]
    E, N, K2 = packed.shape
    w = np.empty((E, N, 2 * K2)); w[..., 0::2] = lo; w[..., 1::2] = hi
    s = torch.from_numpy(sf).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return w * np.repeat(s, 16, axis=2) * scale_2


def _bruteforce(x, ids, wts, Wg, Wu, Wd, limit):
    T, H = x.shape
    out = np.zeros((T, Wd.shape[1]))
    for t in range(T):
        for k in range(ids.shape[1]):
            e = ids[t, k]
            if e < 0:
                continue
            g = Wg[e] @ x[t]
            u = Wu[e] @ x[t]
            a = np.minimum(g, limit) / (1 + np.exp(-np.minimum(g, limit))) * np.clip(u, -limit, limit)
            out[t] += float(wts[t, k]) * (Wd[e] @ a)
    return out


@pytest.mark.parametrize("T,H,I,E", [(1, 256, 128, 16), (3, 384, 256, 5), (2, 128, 384, 9)])
def test_fp8_ffn_matches_dense_bruteforce(T, H, I, E):
    wl = inputs.make_custom("fp8", T, H, I, E, seed=11 + T, routes="uniform" if E >= 8 else "uniform",
                            topk=min(8, E), x_scale=3.0)
    b = wl.bank.numpy()
    # give every scale block its own value so a transposed scale index cannot pass
    rng = np.random.default_rng(5)
    for k in ("s_gate", "s_up", "s_down"):
        b[k] = (b[k] * rng.uniform(0.5, 2.0, b[k].shape)).astype(np.float32)
    ids = wl.ids.numpy().copy()
    if T > 1:
        ids[1, 0] = -1
    r = oracle.moe_fp8(wl.x_bits(), ids, wl.wts.numpy(), b, wl.limit)
    x = wl.x.to(torch.float64).numpy()
    ref = _bruteforce(x, ids, wl.wts.numpy(), _dense_fp8(b["w_gate"], b["s_gate"]),
                      _dense_fp8(b["w_up"], b["s_up"]), _dense_fp8(b["w_down"], b["s_down"]), wl.limit)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # bf16 output is the nearest-even rounding of the double result
    rb = torch.from_numpy(r["out_bf16"].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(rb - r["out"]) <= np.abs(r["out"]) * 2.0 ** -8 + 1e-30)


@pytest.mark.parametrize("T,H,I,E", [(1, 256, 128, 8), (4, 128, 256, 6)])
def test_nvfp4_ffn_matches_dense_bruteforce(T, H, I, E):
    wl = inputs.make_custom("nvfp4", T, H, I, E, seed=21 + T, topk=min(8, E), x_scale=2.0)
    b = wl.bank.numpy()
    ids = wl.ids.numpy()
    r = oracle.moe_nvfp4(wl.x_bits(), ids, wl.wts.numpy(), b, wl.limit)
    x = wl.x.to(torch.float64).numpy()
    ref = _bruteforce(x, ids, wl.wts.numpy(),
                      _dense_nvfp4(b["w_gate"], b["sf_gate"], b["scale2_gate"]),
                      _dense_nvfp4(b["w_up"], b["sf_up"], b["scale2_up"]),
                      _dense_nvfp4(b["w_down"], b["sf_down"], b["scale2_down"]), wl.limit)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def _nvfp4_expert_scale2_case(T=3, H=256, I=128, E=6, seed=31):
    bank = inputs.make_nvfp4_bank_expert_scale2(E, H, I, seed)
    x = inputs.normal_activations(T, H, seed, "cpu", scale=2.0)
    ids = inputs.make_routes("uniform", T, E, seed, min(8, E))
    wts = inputs.softmax_route_weights(T, seed, min(8, E))
    bits = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    return bank, x, ids.numpy(), wts.numpy(), bits


def test_nvfp4_expert_scale2_matches_dense_bruteforce():
    """One scale_2 per expert and projection (a per-expert checkpoint): the oracle against dense
    float64 matrices that multiply each expert's codes by its own scale_2."""
    bank, x, ids, wts, bits = _nvfp4_expert_scale2_case()
    b = bank.numpy()
    assert len(set(b["scale2_gate"].tolist())) > 1          # the experts' values differ
    r = oracle.moe_nvfp4(bits, ids, wts, b, inputs.LIMIT)
    per = lambda k: b[k].astype(np.float64)[:, None, None]  # noqa: E731
    ref = _bruteforce(x.to(torch.float64).numpy(), ids, wts,
                      _dense_nvfp4(b["w_gate"], b["sf_gate"], per("scale2_gate")),
                      _dense_nvfp4(b["w_up"], b["sf_up"], per("scale2_up")),
                      _dense_nvfp4(b["w_down"], b["sf_down"], per("scale2_down")), inputs.LIMIT)
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_nvfp4_expert_scale2_equal_values_are_the_scalar_path():
    bank, x, ids, wts, bits = _nvfp4_expert_scale2_case()
    b = bank.numpy()
    scalar = dict(b)
    for k in ("scale2_gate", "scale2_up", "scale2_down"):
        scalar[k] = float(b[k][2])
        b[k] = np.full_like(b[k], b[k][2])
    r1 = oracle.moe_nvfp4(bits, ids, wts, b, inputs.LIMIT)
    r2 = oracle.moe_nvfp4(bits, ids, wts, scalar, inputs.LIMIT)
    assert np.array_equal(r1["out"], r2["out"])


def test_nvfp4_expert_scale2_power_of_two_equals_scale_byte_shift():
    """scale_2 * 2^j for expert e is the same weight as adding j to the exponent field of each of
    e's E4M3 scale bytes (exact in float64): per-expert powers of two against the scalar path on
    the shifted bytes, bit for bit - an index or projection mix-up in the per-expert lookup
    cannot pass."""
    T, H, I, E = 3, 256, 128, 6
    rng = np.random.default_rng(7)
    base = inputs.make_custom("nvfp4", T, H, I, E, seed=41, topk=min(8, E), x_scale=2.0)
    b = base.bank.numpy()
    for k in ("sf_gate", "sf_up", "sf_down"):                 # exponents 3..11, any sign/mantissa
        exp_ = rng.integers(3, 12, b[k].shape)
        b[k] = ((rng.integers(0, 2, b[k].shape) << 7) | (exp_ << 3) | rng.integers(0, 8, b[k].shape)).astype(np.uint8)
    shifted = dict(b)
    per = dict(b)
    for k, sk in (("scale2_gate", "sf_gate"), ("scale2_up", "sf_up"), ("scale2_down", "sf_down")):
        j = rng.integers(-2, 3, E)
        per[k] = (np.float32(b[k]) * np.exp2(j)).astype(np.float32)
        e_field = ((b[sk] >> 3) & 0xF).astype(np.int64) + j[:, None, None]
        assert e_field.min() >= 1 and e_field.max() <= 13
        shifted[sk] = ((b[sk] & 0x87) | (e_field << 3)).astype(np.uint8)
    ids, wts = base.ids.numpy(), base.wts.numpy()
    r1 = oracle.moe_nvfp4(base.x_bits(), ids, wts, per, base.limit)
    r2 = oracle.moe_nvfp4(base.x_bits(), ids, wts, shifted, base.limit)
    assert np.array_equal(r1["out"], r2["out"])


def test_oracle_intermediates_and_token_subset():
    wl = inputs.make_custom("fp8", 4, 256, 128, 12, seed=3)
    b = wl.bank.numpy()
    full = oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, wl.limit, intermediates=True)
    sub = oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, wl.limit, tokens=[2, 0])
    assert np.array_equal(sub["out"][0], full["out"][2]) and np.array_equal(sub["out"][1], full["out"][0])
    # activation intermediates obey the clamp closed form
    g, u, a = full["g"], full["u"], full["a"]
    gl = np.minimum(g, 7.0)
    assert np.allclose(a, gl / (1 + np.exp(-gl)) * np.clip(u, -7, 7), rtol=1e-14, atol=0)


def test_oracle_thread_count_invariance():
    wl = inputs.make_custom("fp8", 3, 256, 256, 10, seed=4)
    b = wl.bank.numpy()
    r1 = oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, wl.limit, nthreads=1)
    r4 = oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, wl.limit, nthreads=5)
    assert np.array_equal(r1["out"], r4["out"])


def test_oracle_rejects_bad_shapes_and_limit():
    wl = inputs.make_custom("fp8", 1, 256, 128, 8, seed=1)
    b = wl.bank.numpy()
    with pytest.raises(ValueError):
        oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, limit=0.0)
    with pytest.raises(ValueError):
        oracle.moe_fp8(wl.x_bits(), wl.ids.numpy(), wl.wts.numpy(), b, limit=float("nan"))


# ---- router (in front of the FFN) -----------------------------------------------------------------

def test_router_logits_against_numpy_matmul():
    """FP64 logits of bf16 inputs equal a float64 matmul of the decoded bf16 values."""
    g = torch.Generator().manual_seed(11)
    x = torch.randn(3, 96, generator=g).to(torch.bfloat16)
    w = (torch.randn(16, 96, generator=g) * 0.1).to(torch.bfloat16)
    got = oracle.router_logits(x.view(torch.int16).numpy().view(np.uint16),
                               w.view(torch.int16).numpy().view(np.uint16))
    ref = x.to(torch.float64).numpy() @ w.to(torch.float64).numpy().T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # a transposed operand would change this row: one hot x picks one column of W
    x1 = torch.zeros(1, 96, dtype=torch.bfloat16)
    x1[0, 5] = 1.0
    got1 = oracle.router_logits(x1.view(torch.int16).numpy().view(np.uint16),
                                w.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got1[0], w[:, 5].to(torch.float64).numpy())


def test_router_topk_closed_forms_ties_and_bias():
    ln3 = np.log(3.0)
    # sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2, sigmoid(-ln 3) = 1/4
    lg = np.array([[0.0, -ln3, ln3, 0.0, -5.0]])
    ids, w = oracle.router_topk(lg, None, 3, 2.0, True)
    assert ids.tolist() == [[2, 0, 3]]                      # equal scores: lower index first
    assert np.allclose(w, [[2.0 * 0.75 / 1.75, 2.0 * 0.5 / 1.75, 2.0 * 0.5 / 1.75]], rtol=1e-14)
    ids, w = oracle.router_topk(lg, None, 2, 1.5, False)
    assert ids.tolist() == [[2, 0]] and np.allclose(w, [[1.125, 0.75]], rtol=1e-14)
    # the bias selects but does not weight: a large bias pulls expert 1 (sigmoid 1/4) to the front
    bias = np.array([0.0, 10.0, 0.0, 0.0, 0.0])
    ids, w = oracle.router_topk(lg, bias, 2, 1.0, False)
    assert ids.tolist() == [[1, 2]] and np.allclose(w, [[0.25, 0.75]], rtol=1e-14)


def test_router_topk_against_sort_and_expit():
    from scipy.special import expit
    rng = np.random.default_rng(5)
    T, E, k = 20, 64, 8
    lg = rng.normal(size=(T, E))
    lg[3, 10] = lg[3, 40] = lg[3].max() + 1.0               # an exact tie at the top
    bias = rng.normal(scale=0.1, size=E)
    bias[40] = bias[10]                                      # ... and equal scores
    ids, w = oracle.router_topk(lg, bias, k, 2.5, True)
    sig = expit(lg)
    score = sig + bias
    for t in range(T):
        order = np.lexsort((np.arange(E), -score[t]))[:k]    # descending score, then index
        assert ids[t].tolist() == order.tolist()
        sel = sig[t, order]
        assert np.allclose(w[t], 2.5 * sel / sel.sum(), rtol=1e-12)
    assert ids[3, 0] == 10 and ids[3, 1] == 40


# ---- shared expert and the layer epilogue -------------------------------------------------------

def test_shared_expert_against_numpy():
    from scipy.special import expit
    g = torch.Generator().manual_seed(21)
    T, H, S, L = 3, 64, 32, 7.0
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(S, H, generator=g) * 0.3).to(torch.bfloat16)
    wu = (torch.randn(S, H, generator=g) * 0.3).to(torch.bfloat16)
    wd = (torch.randn(H, S, generator=g) * 0.2).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    got = oracle.shared_expert(bits(x), bits(wg), bits(wu), bits(wd), L)
    f = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    gg, uu = f(x) @ f(wg).T, f(x) @ f(wu).T
    gc = np.minimum(gg, L)
    a = gc * expit(gc) * np.clip(uu, -L, L)
    assert np.allclose(got, a @ f(wd).T, rtol=1e-12, atol=1e-12)


def test_layer_epilogue_single_rounding():
    one = lambda v: torch.tensor([v], dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    s, b = oracle.layer_epilogue(np.array([1.0]), one(0.5), one(0.25))
    assert s[0] == 1.75 and oracle.bf16_value(int(b[0])) == 1.75
    # 1 + 2^-9 (+ 2^-9 + 2^-9): one rounding gives 1 + 2^-7; rounding the routed sum first would
    # give 1 (1 + 2^-8 is a tie that goes to even)
    s, b = oracle.layer_epilogue(np.array([1.0 + 2 ** -9]), one(2 ** -9), one(2 ** -9))
    assert oracle.bf16_value(int(b[0])) == 1.0 + 2 ** -7
    s, b = oracle.layer_epilogue(np.array([-3.0]))
    assert s[0] == -3.0

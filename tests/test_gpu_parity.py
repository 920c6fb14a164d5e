"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the same seeded inputs.

Integer outputs (route permutation) must match bit for bit; bf16 outputs must be within relative
L2 <= 5e-3 and max abs <= 2e-2 * RMS(out) of the oracle's double result.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_histogram_gb300 import capi, inputs

from helpers import bf16_to_f64, check_close, oracle_for, prefill_sample_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_ffn_histogram_gb300 import _build
    _build.build()
    capi.load()


def run(wl, **kw):
    out = capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit, **kw)
    torch.cuda.synchronize()
    return out


# ---- route permutation: exact ---------------------------------------------------------------------

def _check_permute(ids_np, E):
    ids = torch.from_numpy(ids_np).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = capi.route_permute(ids, E, err=err)
    torch.cuda.synchronize()
    ref = oracle.route_permute(ids_np, E)
    for k in ("counts", "offsets", "sorted_pair", "pair_to_sorted"):
        assert np.array_equal(r[k].cpu().numpy(), ref[k]), k
    assert int(err.item()) == ref["err"]


@pytest.mark.parametrize("T,E,kind", [(1, 16, "uniform"), (3, 5, "uniform"), (8, 256, "low64"),
                                      (37, 64, "uniform"), (1000, 256, "zipf"),
                                      (4096, 256, "zipf"), (129, 4096, "uniform")])
def test_route_permute_exact(T, E, kind):
    topk = min(8, E)
    ids = inputs.sampled_routes(T, E, kind, seed=T * 31 + E, topk=topk).numpy()
    rng = np.random.default_rng(T)
    ids[rng.random(ids.shape) < 0.05] = -1
    _check_permute(ids.astype(np.int32), E)


def test_route_permute_skew_and_degenerate():
    _check_permute(np.full((300, 8), 7, np.int32), 16)                  # every pair on one expert
    _check_permute(np.full((5, 8), -1, np.int32), 16)                   # nothing routed
    bad = np.zeros((4, 8), np.int32)
    bad[1, 3] = 99
    bad[2, 0] = -7
    _check_permute(bad, 16)                                             # out-of-range ids flagged


# ---- FFN parity on small shapes (several tiles, ragged T) -------------------------------------------

SMALL = [
    ("fp8", 1, 256, 128, 16), ("fp8", 1, 384, 256, 12), ("fp8", 2, 256, 384, 9),
    ("fp8", 3, 640, 256, 12), ("fp8", 5, 256, 128, 20), ("fp8", 8, 384, 256, 24),
    ("fp8", 11, 256, 256, 16), ("fp8", 20, 128, 128, 40),
    ("nvfp4", 1, 256, 128, 16), ("nvfp4", 1, 512, 384, 10), ("nvfp4", 3, 384, 256, 12),
    # one token: 1, 5 (a batch of 4 and a ragged 1) and 7 (4 + 3) super-segments of 128 along H
    ("nvfp4", 1, 128, 128, 8), ("nvfp4", 1, 640, 256, 12), ("nvfp4", 1, 896, 128, 9),
    ("nvfp4", 8, 256, 256, 24), ("nvfp4", 13, 256, 128, 16),
]


@pytest.mark.parametrize("fmt,T,H,I,E", SMALL)
def test_small_parity(fmt, T, H, I, E):
    wl = inputs.make_custom(fmt, T, H, I, E, seed=100 + T + H + E, device=DEV)
    out = run(wl)
    ref = oracle_for(wl)["out"]
    check_close(bf16_to_f64(out), ref, f"{fmt} T={T} H={H} I={I} E={E}")


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_topk_below_eight(fmt):
    wl = inputs.make_custom(fmt, 4, 256, 128, 6, seed=9, device=DEV, topk=3)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"{fmt} topk=3")


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("T,topk", [(1, 1), (1, 3), (1, 5), (40, 1), (40, 5)])
def test_topk_below_eight_single_token_and_grouped(fmt, T, topk):
    """Fewer than 8 slots through the single-token kernels (T = 1: a grid row per slot, the down
    kernel's warps past topk idle) and the grouped tier (T = 40: P = T * topk sorted rows)."""
    wl = inputs.make_custom(fmt, T, 512, 256, 12, seed=70 + 10 * T + topk, device=DEV, topk=topk)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"{fmt} T={T} topk={topk}")


def test_tiny_fp8_decode_config():
    wl = inputs.make_workload("tiny_fp8_decode", device=DEV)
    assert wl.ids.tolist() == [[0, 2, 4, 6, 8, 10, 12, 14]]
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], "tiny_fp8_decode")


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_clamp_stress(fmt):
    """Activations x40: many gates above the limit and ups outside +-limit."""
    wl = inputs.make_custom(fmt, 3, 512, 256, 12, seed=77, device=DEV, x_scale=40.0)
    res = oracle_for(wl)
    check_close(bf16_to_f64(run(wl)), res["out"], f"{fmt} clamp stress")


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_no_limit(fmt):
    wl = inputs.make_custom(fmt, 2, 256, 256, 10, seed=78, device=DEV, x_scale=20.0,
                            limit=float("inf"))
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"{fmt} limit=inf")


@pytest.mark.parametrize("T", [1, 4])
def test_unfilled_and_bad_ids(T):
    wl = inputs.make_custom("fp8", T, 256, 128, 16, seed=5, device=DEV)
    ids = wl.ids.clone()
    ids[0, 1] = -1
    ids[0, 5] = 16          # == E: out of range
    ids[T - 1, 7] = -9
    wl.ids = ids
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(wl, err=err)
    assert int(err.item()) & capi.ERRBIT_BAD_ID
    res = oracle_for(wl)
    assert res["err"] & 1
    check_close(bf16_to_f64(out), res["out"], "bad ids")


@pytest.mark.parametrize("T", [1, 3])
def test_nothing_routed_gives_zero(T):
    wl = inputs.make_custom("fp8", T, 256, 128, 16, seed=6, device=DEV)
    wl.ids = torch.full_like(wl.ids, -1)
    out = torch.full((T, 256), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run(wl, out=out, err=err)
    assert torch.equal(out.float(), torch.zeros_like(out.float()))
    assert int(err.item()) == 0


def test_duplicate_ids_in_a_token_are_summed():
    wl = inputs.make_custom("fp8", 3, 256, 128, 16, seed=7, device=DEV)
    ids = wl.ids.clone()
    ids[0, :] = 3           # all 8 slots of token 0 on expert 3
    ids[1, 2] = ids[1, 5]
    wl.ids = ids
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], "duplicates")
    wl1 = inputs.make_custom("nvfp4", 1, 256, 128, 16, seed=8, device=DEV)
    wl1.ids = torch.full_like(wl1.ids, 2)
    check_close(bf16_to_f64(run(wl1)), oracle_for(wl1)["out"], "duplicates T=1")


# ---- determinism, guards, stages -----------------------------------------------------------------

@pytest.mark.parametrize("fmt,T", [("fp8", 1), ("fp8", 6), ("nvfp4", 1), ("nvfp4", 5)])
def test_bitwise_repeatable(fmt, T):
    wl = inputs.make_custom(fmt, T, 384, 256, 16, seed=10 + T, device=DEV)
    a = run(wl).clone()
    for _ in range(3):
        assert torch.equal(run(wl).view(torch.int16), a.view(torch.int16))


@pytest.mark.parametrize("fmt,T", [("fp8", 1), ("fp8", 7), ("nvfp4", 2)])
def test_output_tail_sentinel_untouched(fmt, T):
    wl = inputs.make_custom(fmt, T, 256, 128, 16, seed=11, device=DEV)
    H = wl.H
    buf = torch.full((T * H + 17,), float("nan"), dtype=torch.bfloat16, device=DEV)
    sentinel = buf[T * H:].clone()
    out = buf[: T * H].view(T, H)
    run(wl, out=out)
    assert torch.equal(buf[T * H:].view(torch.int16), sentinel.view(torch.int16))
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("fmt,T", [("fp8", 1), ("fp8", 5), ("nvfp4", 1), ("nvfp4", 8)])
def test_stages_equal_forward(fmt, T):
    wl = inputs.make_custom(fmt, T, 256, 256, 16, seed=12, device=DEV)
    ref = run(wl).clone()
    f = capi.FMT_FP8 if fmt == "fp8" else capi.FMT_NVFP4
    ws = capi.alloc_workspace(T, wl.H, wl.I, wl.E, wl.topk, f, DEV)
    out = torch.empty_like(ref)
    capi.plan(wl.ids, wl.H, wl.I, wl.E, f, ws)
    capi.gate_up(wl.x, wl.ids, wl.bank, wl.limit, ws)
    capi.down_combine(wl.ids, wl.wts, wl.bank, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_workspace_too_small_is_rejected_on_device_path():
    wl = inputs.make_custom("fp8", 2, 256, 128, 16, seed=13, device=DEV)
    n = capi.workspace_bytes(2, 256, 128, 16, 8, capi.FMT_FP8)
    ws = torch.empty(n - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(capi.MoeError) as e:
        run(wl, workspace=ws)
    assert e.value.code == -3


def test_stream_ordering_on_a_side_stream():
    wl = inputs.make_custom("fp8", 4, 256, 128, 16, seed=14, device=DEV)
    ref = run(wl).clone()
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        out = capi.forward(wl.x, wl.ids, wl.wts, wl.bank, wl.limit)
    s.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


# ---- the named workloads at full size ---------------------------------------------------------------

@pytest.fixture(scope="module")
def fp8_bank():
    return inputs.make_bank("fp8_decode", DEV)


def test_fp8_decode_full_size(fp8_bank):
    for rs in range(2):
        wl = inputs.make_workload("fp8_decode", device=DEV, bank=fp8_bank, route_set=rs)
        check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"fp8_decode set {rs}")


def test_fp8_decode_clamp_stress_full_size(fp8_bank):
    wl = inputs.make_workload("fp8_decode", device=DEV, bank=fp8_bank, x_scale=8.0)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], "fp8_decode x8")


def test_fp8_batchm_full_size(fp8_bank):
    wl = inputs.make_workload("fp8_batchm", device=DEV, bank=fp8_bank)
    ids = wl.ids.cpu().numpy()
    assert ids.max() < 64 and len(set(ids.reshape(-1).tolist())) < 64
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], "fp8_batchm")


def test_fp8_prefill_full_size_sampled(fp8_bank):
    """The full prefill workload (4096 Zipf-routed tokens, 256 experts) in the launch
    configuration the bench times; compared with the oracle on sampled tokens whose pairs reach
    every routed expert and the edge rows of every multi-tile expert's m-tiles."""
    wl = inputs.make_workload("fp8_prefill", device=DEV, bank=fp8_bank)
    out = run(wl)
    toks = prefill_sample_tokens(wl.ids, wl.E)
    assert len(toks) < 200
    res = oracle_for(wl, tokens=toks)
    check_close(bf16_to_f64(out[toks]), res["out"], f"fp8_prefill on {len(toks)} sampled tokens")
    # route permutation at the full prefill size, exactly
    _check_permute(wl.ids.cpu().numpy(), wl.E)


def test_nvfp4_decode_full_size():
    bank = inputs.make_bank("nvfp4_decode", DEV)
    for rs in range(2):
        wl = inputs.make_workload("nvfp4_decode", device=DEV, bank=bank, route_set=rs)
        check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"nvfp4_decode set {rs}")


# ---- the grouped-GEMM (prefill) tier: FP8, T > 8 ----------------------------------------------------

@pytest.mark.parametrize("T,H,I,E,routes", [(28, 256, 128, 16, "uniform"), (64, 384, 256, 40, "zipf"),
                                            (300, 256, 256, 8, "uniform"), (130, 512, 384, 24, "zipf")])
def test_prefill_parity(T, H, I, E, routes):
    wl = inputs.make_custom("fp8", T, H, I, E, seed=700 + T, device=DEV, routes=routes)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"prefill T={T} E={E}")


def test_prefill_skewed_and_bad_ids():
    T, E = 200, 12
    wl = inputs.make_custom("fp8", T, 256, 256, E, seed=801, device=DEV)
    ids = wl.ids.clone()
    ids[:150, :4] = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=DEV)   # experts 0..3 get 150+ rows
    ids[5, 6] = -1
    ids[7, 2] = E + 3
    wl.ids = ids
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(wl, err=err)
    assert int(err.item()) & capi.ERRBIT_BAD_ID
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], "prefill skew")


def test_prefill_clamp_stress_and_no_limit():
    wl = inputs.make_custom("fp8", 40, 256, 256, 10, seed=802, device=DEV, x_scale=40.0)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], "prefill clamp stress")
    wl2 = inputs.make_custom("fp8", 30, 256, 128, 10, seed=803, device=DEV, x_scale=20.0,
                             limit=float("inf"))
    check_close(bf16_to_f64(run(wl2)), oracle_for(wl2)["out"], "prefill no limit")


# ---- the grouped-GEMM tier over NVFP4 banks (K multiples of 256) -------------------------------------

@pytest.mark.parametrize("T,H,I,E,routes", [(18, 256, 256, 16, "uniform"), (64, 512, 256, 40, "zipf"),
                                            (300, 256, 512, 8, "uniform"), (130, 768, 512, 24, "zipf")])
def test_nvfp4_prefill_parity(T, H, I, E, routes):
    wl = inputs.make_custom("nvfp4", T, H, I, E, seed=900 + T, device=DEV, routes=routes)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"nvfp4 prefill T={T} E={E}")


def test_nvfp4_prefill_skewed_bad_ids_and_clamp():
    T, E = 200, 12
    wl = inputs.make_custom("nvfp4", T, 512, 256, E, seed=901, device=DEV, x_scale=30.0)
    ids = wl.ids.clone()
    ids[:150, :4] = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=DEV)
    ids[5, 6] = -1
    ids[7, 2] = E + 3
    wl.ids = ids
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(wl, err=err)
    assert int(err.item()) & capi.ERRBIT_BAD_ID
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], "nvfp4 prefill skew")
    a = out.clone()
    assert torch.equal(run(wl, err=err).view(torch.int16), a.view(torch.int16))


def test_nvfp4_prefill_full_size_sampled():
    bank = inputs.make_bank("nvfp4_prefill", DEV)
    wl = inputs.make_workload("nvfp4_prefill", device=DEV, bank=bank)
    out = run(wl)
    toks = prefill_sample_tokens(wl.ids, wl.E)
    assert len(toks) < 200
    res = oracle_for(wl, tokens=toks)
    check_close(bf16_to_f64(out[toks]), res["out"], f"nvfp4_prefill on {len(toks)} sampled tokens")


@pytest.mark.parametrize("fmt,T,H,I", [("fp8", 8, 512, 256), ("fp8", 9, 512, 256), ("nvfp4", 8, 512, 256),
                                       ("nvfp4", 9, 512, 256), ("nvfp4", 9, 384, 256), ("nvfp4", 20, 512, 128)])
def test_tier_crossover_both_sides(fmt, T, H, I):
    """Both sides of the measured crossover: T = 8 (one cooperative sweep) and T = 9 (the grouped
    GEMM), and NVFP4 shapes the grouped tier does not cover (H or I not a multiple of 256), which
    run as sweeps of <= 8 tokens at any T."""
    wl = inputs.make_custom(fmt, T, H, I, 20, seed=950 + T, device=DEV)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"crossover {fmt} T={T} H={H} I={I}")


def test_prefill_bitwise_repeatable():
    wl = inputs.make_custom("fp8", 100, 256, 256, 16, seed=804, device=DEV, routes="zipf")
    a = run(wl).clone()
    for _ in range(2):
        assert torch.equal(run(wl).view(torch.int16), a.view(torch.int16))


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_prefill_multi_block_plan(fmt):
    """T*topk >= 4096 pairs: the permutation is planned over several blocks (a ragged last one),
    with skew, a dropped slot (-1) and an out-of-range id; bit-for-bit the single-block result's
    output, checked against the oracle."""
    T, E = 700, 33
    wl = inputs.make_custom(fmt, T, 256, 256, E, seed=960, device=DEV, routes="zipf")
    ids = wl.ids.clone()
    ids[:200, :3] = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    ids[9, 5] = -1
    ids[650, 1] = E + 7
    wl.ids = ids
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(wl, err=err)
    assert int(err.item()) & capi.ERRBIT_BAD_ID
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], f"{fmt} prefill wide plan")


@pytest.mark.parametrize("limit", [255.0, 300.0])
def test_prefill_activation_paths_at_the_limit_bound(limit):
    """limit <= 255: the gate/up GEMM stores the activations in f16 as they are (|a| <= limit^2
    fits f16); above it they keep the per-row range scale (act_prep). Both against the oracle
    with large activations."""
    wl = inputs.make_custom("fp8", 48, 256, 256, 10, seed=966, device=DEV, x_scale=60.0, limit=limit)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"prefill limit {limit}")


@pytest.mark.parametrize("fmt,x_scale,limit", [("fp8", 3e-3, 7.0), ("fp8", 2e3, float("inf")),
                                               ("fp8", 3e-3, float("inf")), ("nvfp4", 3e-3, 7.0),
                                               ("nvfp4", 2e3, float("inf"))])
def test_prefill_f16_scaling_across_magnitudes(fmt, x_scale, limit):
    """The grouped tier keeps its activations and the down GEMM's output y in f16 times powers of
    two (a fixed one for the clamped activations, one per sorted row and 128-row output block for
    y, from a bound on |y|): tiny inputs stay clear of f16's subnormal range and large ones (y far
    above 65504 without the clamp) below its largest value, both against the oracle."""
    H, I = (256, 256) if fmt == "fp8" else (512, 256)
    wl = inputs.make_custom(fmt, 40, H, I, 10, seed=970, device=DEV, x_scale=x_scale, limit=limit)
    ref = oracle_for(wl)["out"]
    if x_scale > 1.0:
        assert np.abs(ref).max() > 65504.0        # y itself leaves f16's range
    check_close(bf16_to_f64(run(wl)), ref, f"{fmt} prefill x*{x_scale} limit {limit}")


# ---- NVFP4 with one scale_2 per expert and projection ---------------------------------------------

def _expert_scale2_workload(T, E=12, H=512, I=256, seed=977):
    bank = inputs.make_nvfp4_bank_expert_scale2(E, H, I, seed, device=DEV)
    x = inputs.normal_activations(T, H, seed, DEV)
    ids = inputs.make_routes("uniform", T, E, seed).to(DEV)
    wts = inputs.softmax_route_weights(T, seed).to(DEV)
    return inputs.Workload(f"expert_scale2_T{T}", "nvfp4", T, H, I, E, inputs.TOPK, x, ids, wts, bank,
                           inputs.LIMIT)


@pytest.mark.parametrize("T", [1, 4, 12, 64])
def test_nvfp4_expert_scale2_parity(T):
    """moe_nvfp4_forward_expert_scale2 through every tier - one token, the fused batch-M kernel,
    sweeps of <= 8 tokens, the grouped GEMM - against the oracle with the same per-expert
    values (each expert quantised with its own scale_2)."""
    wl = _expert_scale2_workload(T)
    assert len(set(wl.bank.scale2_down.tolist())) > 1
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"nvfp4 per-expert scale_2 T={T}")


@pytest.mark.parametrize("T", [1, 6, 64])
def test_nvfp4_expert_scale2_zero_and_negative(T):
    """Per-expert values of 0 (an expert that contributes nothing) and of a negative sign (its
    outputs flip) on every tier; the grouped tier's f16 bound for y uses |scale_2|."""
    wl = _expert_scale2_workload(T, seed=978)
    b = wl.bank
    for t in (b.scale2_gate, b.scale2_up, b.scale2_down):
        t[3] = 0.0
        t[5] = -t[5]
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"nvfp4 scale_2 zero/negative T={T}")


@pytest.mark.parametrize("fmt,E", [("fp8", 4096), ("nvfp4", 1024)])
def test_grouped_tier_many_experts_few_tokens(fmt, E):
    """The grouped tier at its smallest width (T = 9) over a bank with thousands of experts: the
    route plan, the m-tile list (almost every expert empty) and the GEMMs' tile decode."""
    H, I = (256, 128) if fmt == "fp8" else (256, 256)
    wl = inputs.make_custom(fmt, 9, H, I, E, seed=981, device=DEV)
    check_close(bf16_to_f64(run(wl)), oracle_for(wl)["out"], f"{fmt} grouped T=9 E={E}")


def test_prefill_zero_token_rows():
    """Tokens whose x is all zero: their activation rows (and, when every token of an m-tile is zero,
    the m-tile maximum) are 0, so y's power of two falls back to 1 and their outputs are exactly 0."""
    wl = inputs.make_custom("fp8", 40, 256, 256, 10, seed=979, device=DEV)
    wl.x[3].zero_()
    wl.x[17].zero_()
    out = run(wl)
    assert torch.count_nonzero(out[3]) == 0 and torch.count_nonzero(out[17]) == 0
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], "prefill zero tokens")


@pytest.mark.parametrize("T", [1, 64])
def test_nvfp4_expert_scale2_table_with_stride(T):
    """The same values as one [E][3] table (gate, up, down columns; stride 3) give the same bits
    as three [E] arrays."""
    wl = _expert_scale2_workload(T)
    b = wl.bank
    table = torch.stack([b.scale2_gate, b.scale2_up, b.scale2_down], dim=1).contiguous()
    ref = run(wl)
    out = torch.empty_like(ref)
    E, I, _ = b.w_gate.shape
    ws = torch.empty(int(capi.load().moe_workspace_bytes(T, wl.H, I, E, wl.topk, capi.FMT_NVFP4)),
                     dtype=torch.uint8, device=DEV)
    col = lambda j: ctypes.c_void_p(table.data_ptr() + 4 * j)  # noqa: E731
    rc = capi.load().moe_nvfp4_forward_expert_scale2(
        ctypes.c_void_p(wl.x.data_ptr()), T, wl.H, I, E, wl.topk, ctypes.c_void_p(wl.ids.data_ptr()),
        ctypes.c_void_p(wl.wts.data_ptr()), ctypes.c_void_p(b.w_gate.data_ptr()),
        ctypes.c_void_p(b.sf_gate.data_ptr()), col(0), ctypes.c_void_p(b.w_up.data_ptr()),
        ctypes.c_void_p(b.sf_up.data_ptr()), col(1), ctypes.c_void_p(b.w_down.data_ptr()),
        ctypes.c_void_p(b.sf_down.data_ptr()), col(2), 3, wl.limit, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


# ---- bounded waits and buffer bounds -----------------------------------------------------------------

@pytest.mark.parametrize("fmt,T", [("fp8", 4), ("nvfp4", 7)])
def test_fused_barrier_timeout_reports_and_context_survives(fmt, T):
    """The test hook makes the cooperative kernel's grid barrier wait for one CTA more than the
    grid holds (a count nothing reaches) with a ~10 ms bound: every CTA gives up, sets
    MOE_ERRBIT_BARRIER and writes NaN to its output rows, and the context stays usable - the
    next call, with the hook off, is bit-identical to a clean run."""
    wl = inputs.make_custom(fmt, T, 256, 128, 16, seed=31 + T, device=DEV)
    ref = run(wl).clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(ref)
    capi.test_barrier_timeout(True)
    try:
        run(wl, out=out, err=err)
    finally:
        capi.test_barrier_timeout(False)
    torch.cuda.synchronize()
    assert int(err.item()) & capi.ERRBIT_BARRIER
    assert torch.isnan(out.float()).all()
    err.zero_()
    again = run(wl, err=err)
    assert int(err.item()) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("fmt,T", [("fp8", 1), ("fp8", 6), ("fp8", 19), ("nvfp4", 1), ("nvfp4", 8),
                                   ("fp8", 40), ("nvfp4", 40)])
def test_workspace_tail_sentinel_untouched(fmt, T):
    """Every tier stays inside moe_workspace_bytes(): NaN sentinel bytes right after the
    workspace (and after out) come back unchanged, and the result matches the oracle."""
    wl = inputs.make_custom(fmt, T, 512, 256, 16, seed=40 + T, device=DEV, routes="zipf")
    f = capi.FMT_FP8 if fmt == "fp8" else capi.FMT_NVFP4
    n = capi.workspace_bytes(T, wl.H, wl.I, wl.E, wl.topk, f)
    tail = 4096
    buf = torch.empty(n + tail, dtype=torch.uint8, device=DEV)
    buf[n:].view(torch.int32).fill_(0x7fc54321)
    sentinel = buf[n:].clone()
    obuf = torch.full((T * wl.H + 17,), float("nan"), dtype=torch.bfloat16, device=DEV)
    osent = obuf[T * wl.H:].clone()
    out = obuf[: T * wl.H].view(T, wl.H)
    run(wl, out=out, workspace=buf[:n])
    assert torch.equal(buf[n:], sentinel)
    assert torch.equal(obuf[T * wl.H:].view(torch.int16), osent.view(torch.int16))
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], f"{fmt} T={T} inside its workspace")


# expert row counts that put one m-tile of every height 1..128 (and the next tile of a
# multi-tile expert) through the grouped tier: the token boxes are loaded with the tile's valid
# rows rounded up to 16, one tensor map per height
_TILE_HEIGHT_COUNTS = [1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 63, 64, 65, 79, 80, 81, 95, 96, 97,
                       111, 112, 113, 127, 128, 129, 143, 144, 255, 256, 257]


def _routes_with_counts(counts, topk, pad_expert):
    """Route ids [T][topk] in which expert e appears counts[e] times; the slots past the total
    go to pad_expert. Duplicate ids within a token are legal (they are summed)."""
    flat = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    T = -(-flat.size // topk)
    ids = np.full(T * topk, pad_expert, dtype=np.int32)
    ids[:flat.size] = np.random.default_rng(77).permutation(flat)
    return torch.from_numpy(ids.reshape(T, topk))


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_prefill_every_token_box_height(fmt):
    E = len(_TILE_HEIGHT_COUNTS) + 1                 # the last expert takes the padding slots
    ids = _routes_with_counts(_TILE_HEIGHT_COUNTS, 8, E - 1)
    T = ids.shape[0]
    wl = inputs.make_custom(fmt, T, 256, 256, E, seed=1234, device=DEV)
    wl.ids = ids.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(wl, err=err)
    assert int(err.item()) == 0
    check_close(bf16_to_f64(out), oracle_for(wl)["out"], f"{fmt} prefill, every token-box height")

"""Seeded synthetic inputs for the routed MoE FFN (shared by the tests, the oracle checks and bench).

This module only draws random numbers and packs them into the byte layouts the library reads:
it holds none of the FFN's arithmetic (no decode, no projection, no activation, no combine).
Weight quantisation to E4M3 / NVFP4 is input preparation: the method under test starts from the
stored codes and scales, and both the CUDA path and the oracle read exactly the bytes made here.

Workloads (the real checkpoints and routing traces behind the pages are not available, so these
stand in for them, with the pages' shapes):

* ``tiny_fp8_decode`` - T=1, H=256, I=128, E=16, top-8; x from the gate binary's LCG activation
  fixture, routes from its route fixture ("memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs",
  ``activations_with_salt`` and ``grouped_selected_routes``).
* ``fp8_decode`` - T=1, H=7168, I=2048, E=256; routes uniform without replacement.
* ``fp8_batchm`` - T=8 over the same bank; each token picks 8 of experts 0..63, so expert sets
  overlap across tokens.
* ``nvfp4_decode`` - T=1, H=5120, I=1536, E=160, NVFP4 W4A16.
* ``fp8_prefill`` - T=4096 over the fp8_decode bank; routes from a Zipf(1.1) expert popularity.
* ``nvfp4_prefill`` - T=4096 over the nvfp4_decode bank; Zipf(1.1) routes (the second prefill
  workload: the grouped GEMM over W4A16 banks).

All weights are N(0, 0.02) in fp32 before quantisation; router weights are a softmax of N(0, 1)
logits over the 8 slots; activations are N(0, 1) bf16 (LCG for the tiny case); limit = 7.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np
import torch

TOPK = 8
E4M3_MAX = 448.0
E2M1_MAX = 6.0
# E2M1 magnitudes by code 0..7, and the midpoints between neighbours (for round-to-nearest-even).
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


CONFIGS = {
    "tiny_fp8_decode": dict(fmt="fp8", T=1, H=256, I=128, E=16, routes="fixture", x="lcg",
                            seed=1001, bank_seed=1001),
    "fp8_decode": dict(fmt="fp8", T=1, H=7168, I=2048, E=256, routes="uniform", x="normal",
                       seed=1002, bank_seed=1002),
    "fp8_batchm": dict(fmt="fp8", T=8, H=7168, I=2048, E=256, routes="low64", x="normal",
                       seed=1003, bank_seed=1002),
    "nvfp4_decode": dict(fmt="nvfp4", T=1, H=5120, I=1536, E=160, routes="uniform", x="normal",
                         seed=1004, bank_seed=1004),
    "fp8_prefill": dict(fmt="fp8", T=4096, H=7168, I=2048, E=256, routes="zipf", x="normal",
                        seed=1005, bank_seed=1002),
    "nvfp4_prefill": dict(fmt="nvfp4", T=4096, H=5120, I=1536, E=160, routes="zipf", x="normal",
                          seed=1006, bank_seed=1004),
}
LIMIT = 7.0


def _seed(*parts) -> int:
    """Stable 63-bit seed from a tuple of ints/strings (substreams per purpose)."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


# ---- activations -------------------------------------------------------------------------------

def lcg_activations(tokens: int, width: int, salt: int = 0) -> torch.Tensor:
    """The gate binary's LCG activation fixture, as bf16 [tokens, width] (CPU).

    value(i) = ((mix(i) mod 8191) - 4095) / 2048 with mix(i) = (i + salt*104729)*1664525 +
    1013904223 in wrapping 64-bit arithmetic; computed exactly in f32, then rounded to bf16.
    """
    i = np.arange(tokens * width, dtype=np.uint64)
    with np.errstate(over="ignore"):
        mixed = (i + np.uint64(salt) * np.uint64(104_729)) * np.uint64(1_664_525) + np.uint64(1_013_904_223)
    v = ((mixed % np.uint64(8191)).astype(np.float32) - np.float32(4095.0)) / np.float32(2048.0)
    return torch.from_numpy(v.reshape(tokens, width)).to(torch.bfloat16)


def normal_activations(tokens: int, width: int, seed: int, device="cpu", scale: float = 1.0) -> torch.Tensor:
    g = _gen(device, "x", seed)
    x = torch.randn(tokens, width, generator=g, device=device, dtype=torch.float32)
    return (x * scale).to(torch.bfloat16)


# ---- routes ------------------------------------------------------------------------------------

def fixture_routes(tokens: int, experts: int) -> torch.Tensor:
    """The gate binary's route fixture: ids[t, k] = (k * E/8 + t) mod E (needs E % 8 == 0)."""
    if tokens <= 0 or experts < TOPK or experts % TOPK:
        raise ValueError("route fixture needs tokens > 0 and an expert count divisible by 8")
    stride = experts // TOPK
    t = torch.arange(tokens).unsqueeze(1)
    k = torch.arange(TOPK).unsqueeze(0)
    return ((k * stride + t) % experts).to(torch.int32)


def fixture_route_weights(tokens: int, shift: int) -> torch.Tensor:
    """The gate binary's weight fixture: w[t, k] = ((k + t + shift) mod 8 + 1) / 36."""
    t = torch.arange(tokens).unsqueeze(1)
    k = torch.arange(TOPK).unsqueeze(0)
    return (((k + t + shift) % TOPK + 1).to(torch.float32) / 36.0)


def sampled_routes(tokens: int, experts: int, kind: str, seed: int, topk: int = TOPK,
                   zipf_s: float = 1.1) -> torch.Tensor:
    """Distinct top-k expert ids per token, drawn without replacement (CPU generator).

    kind: 'uniform' over all experts; 'low64' over experts 0..63; 'zipf' with popularity of
    expert e proportional to (e+1)^-s (sequential weighted sampling without replacement).
    """
    g = _gen("cpu", "routes", kind, seed)
    if kind == "uniform":
        p = torch.ones(experts, dtype=torch.float64)
    elif kind == "low64":
        p = torch.zeros(experts, dtype=torch.float64)
        p[: min(64, experts)] = 1.0
    elif kind == "zipf":
        p = (torch.arange(experts, dtype=torch.float64) + 1.0) ** (-zipf_s)
    else:
        raise ValueError(kind)
    ids = torch.multinomial(p.expand(tokens, experts), topk, replacement=False, generator=g)
    return ids.to(torch.int32)


def softmax_route_weights(tokens: int, seed: int, topk: int = TOPK) -> torch.Tensor:
    g = _gen("cpu", "router", seed)
    logits = torch.randn(tokens, topk, generator=g, dtype=torch.float32)
    return torch.softmax(logits, dim=1)


# ---- weight banks ------------------------------------------------------------------------------

@dataclasses.dataclass
class Fp8Bank:
    """E4M3 codes with one fp32 scale per 128x128 block. gate/up [E, I, H], down [E, H, I]."""
    w_gate: torch.Tensor
    s_gate: torch.Tensor
    w_up: torch.Tensor
    s_up: torch.Tensor
    w_down: torch.Tensor
    s_down: torch.Tensor
    fmt: str = "fp8"

    def numpy(self, experts: Optional[torch.Tensor] = None) -> dict:
        sel = (lambda t: t) if experts is None else (lambda t: t.index_select(0, experts.to(t.device)))
        return {k: sel(getattr(self, k)).cpu().numpy()
                for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")}


@dataclasses.dataclass
class Nvfp4Bank:
    """Packed E2M1 codes (element 2j in the low nibble of byte j), one E4M3 scale byte per 16
    elements along K, and one fp32 scale_2 per projection - or, in a bank from
    make_nvfp4_bank_expert_scale2, one per expert and projection (float32 tensors [E]).
    gate/up [E, I, H/2], down [E, H, I/2]."""
    w_gate: torch.Tensor
    sf_gate: torch.Tensor
    scale2_gate: float
    w_up: torch.Tensor
    sf_up: torch.Tensor
    scale2_up: float
    w_down: torch.Tensor
    sf_down: torch.Tensor
    scale2_down: float
    fmt: str = "nvfp4"

    def numpy(self, experts: Optional[torch.Tensor] = None) -> dict:
        sel = (lambda t: t) if experts is None else (lambda t: t.index_select(0, experts.to(t.device)))
        d = {k: sel(getattr(self, k)).cpu().numpy()
             for k in ("w_gate", "sf_gate", "w_up", "sf_up", "w_down", "sf_down")}
        for k in ("scale2_gate", "scale2_up", "scale2_down"):
            v = getattr(self, k)
            d[k] = sel(v).cpu().numpy().astype(np.float32) if isinstance(v, torch.Tensor) else v
        return d

    @property
    def per_expert_scale2(self) -> bool:
        return isinstance(self.scale2_gate, torch.Tensor)


def quantize_e4m3_blocks(w: torch.Tensor):
    """fp32 [N, K] -> (E4M3 codes u8 [N, K], fp32 scales [N/128, K/128]); scale = amax/448,
    code = RNE(clamp(w/scale, +-448)). An all-zero block gets scale 1 and zero codes."""
    N, K = w.shape
    blk = w.reshape(N // 128, 128, K // 128, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
    codes = q.reshape(N, K).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.to(torch.float32)


def e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """fp32 -> E2M1 nibbles (uint8 0..15), round to nearest, ties to the even code, saturating at 6."""
    mag = v.abs().clamp(max=E2M1_MAX)
    mids = torch.tensor(_E2M1_MID, dtype=mag.dtype, device=mag.device)
    idx = torch.bucketize(mag, mids, right=False)          # number of midpoints strictly below
    at_mid = (idx < len(_E2M1_MID)) & (mag == mids[idx.clamp(max=len(_E2M1_MID) - 1)])
    idx = torch.where(at_mid & (idx % 2 == 1), idx + 1, idx)
    sign = ((v < 0) & (idx > 0)).to(torch.uint8) << 3
    return idx.to(torch.uint8) | sign


def pack_e2m1(nibbles: torch.Tensor) -> torch.Tensor:
    """[..., K] nibbles -> [..., K/2] bytes, element 2j in the low nibble of byte j."""
    lo = nibbles[..., 0::2]
    hi = nibbles[..., 1::2]
    return lo | (hi << 4)


def quantize_nvfp4(w: torch.Tensor, scale_2: float):
    """fp32 [N, K] -> (packed [N, K/2] u8, sf [N, K/16] E4M3 u8) for a given per-projection scale_2.

    sf = E4M3_RNE(amax_16 / (6 * scale_2)); code = E2M1_RNE(clamp(w / (sf * scale_2), +-6)),
    code 0 where the scale byte decodes to 0.
    """
    N, K = w.shape
    g = w.reshape(N, K // 16, 16)
    amax = g.abs().amax(dim=2)
    sf_val = (amax / (E2M1_MAX * scale_2)).clamp(max=E4M3_MAX)
    sf = sf_val.to(torch.float8_e4m3fn)
    sf_dec = sf.to(torch.float32)
    denom = (sf_dec * scale_2)[:, :, None]
    q = torch.where(denom > 0, g / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(g))
    nib = e2m1_codes(q.clamp(-E2M1_MAX, E2M1_MAX)).reshape(N, K)
    return pack_e2m1(nib), sf.view(torch.uint8)


def _normal_matrix(seed: int, expert: int, proj: str, n: int, k: int, device) -> torch.Tensor:
    g = _gen(device, "w", seed, expert, proj)
    return torch.randn(n, k, generator=g, device=device, dtype=torch.float32) * 0.02


def make_fp8_bank(E: int, H: int, I: int, seed: int, device="cpu", experts=None) -> Fp8Bank:
    """Whole bank, or only the listed experts (in that order) of the same seeded bank."""
    experts = list(range(E)) if experts is None else [int(e) for e in experts]
    E = len(experts)
    wg = torch.empty(E, I, H, dtype=torch.uint8, device=device)
    wu = torch.empty(E, I, H, dtype=torch.uint8, device=device)
    wd = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    sg = torch.empty(E, I // 128, H // 128, dtype=torch.float32, device=device)
    su = torch.empty_like(sg)
    sd = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=device)
    for i, e in enumerate(experts):
        for proj, (wt, st, n, k) in {"gate": (wg, sg, I, H), "up": (wu, su, I, H),
                                     "down": (wd, sd, H, I)}.items():
            c, s = quantize_e4m3_blocks(_normal_matrix(seed, e, proj, n, k, device))
            wt[i].copy_(c)
            st[i].copy_(s)
    return Fp8Bank(wg, sg, wu, su, wd, sd)


def make_nvfp4_bank(E: int, H: int, I: int, seed: int, device="cpu", experts=None) -> Nvfp4Bank:
    """Whole bank, or only the listed experts of the same seeded bank (scale_2 is always taken
    over the whole bank, as the full bank defines it)."""
    shapes = {"gate": (I, H), "up": (I, H), "down": (H, I)}
    keep = list(range(E)) if experts is None else [int(e) for e in experts]
    scale2 = {}
    for proj, (n, k) in shapes.items():          # pass 1: bank-wide amax per projection
        amax = torch.zeros((), device=device)
        for e in range(E):
            amax = torch.maximum(amax, _normal_matrix(seed, e, proj, n, k, device).abs().amax())
        # scale_2 is an fp32 passed by value: keep exactly the fp32 the library will see
        scale2[proj] = float(np.float32(float(amax) / (E2M1_MAX * E4M3_MAX)))
    out = {}
    for proj, (n, k) in shapes.items():          # pass 2: regenerate and quantise
        packed = torch.empty(len(keep), n, k // 2, dtype=torch.uint8, device=device)
        sf = torch.empty(len(keep), n, k // 16, dtype=torch.uint8, device=device)
        for i, e in enumerate(keep):
            p, s = quantize_nvfp4(_normal_matrix(seed, e, proj, n, k, device), scale2[proj])
            packed[i].copy_(p)
            sf[i].copy_(s)
        out[proj] = (packed, sf)
    return Nvfp4Bank(out["gate"][0], out["gate"][1], scale2["gate"],
                     out["up"][0], out["up"][1], scale2["up"],
                     out["down"][0], out["down"][1], scale2["down"])


def make_nvfp4_bank_expert_scale2(E: int, H: int, I: int, seed: int, device="cpu") -> Nvfp4Bank:
    """The same matrices as make_nvfp4_bank, each expert quantised with its own scale_2 per
    projection (its amax / (6 * 448), as a per-expert checkpoint stores it), held as float32
    tensors [E] on the bank's device."""
    shapes = {"gate": (I, H), "up": (I, H), "down": (H, I)}
    out = {}
    for proj, (n, k) in shapes.items():
        packed = torch.empty(E, n, k // 2, dtype=torch.uint8, device=device)
        sf = torch.empty(E, n, k // 16, dtype=torch.uint8, device=device)
        s2 = torch.empty(E, dtype=torch.float32)
        for e in range(E):
            m = _normal_matrix(seed, e, proj, n, k, device)
            s2[e] = float(np.float32(float(m.abs().amax()) / (E2M1_MAX * E4M3_MAX)))
            p, s = quantize_nvfp4(m, float(s2[e]))
            packed[e].copy_(p)
            sf[e].copy_(s)
        out[proj] = (packed, sf, s2.to(device))
    return Nvfp4Bank(*out["gate"], *out["up"], *out["down"])


# ---- whole workloads ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    fmt: str
    T: int
    H: int
    I: int
    E: int
    topk: int
    x: torch.Tensor        # bf16 [T, H]
    ids: torch.Tensor      # int32 [T, topk]
    wts: torch.Tensor      # fp32 [T, topk]
    bank: object           # Fp8Bank | Nvfp4Bank
    limit: float

    def x_bits(self) -> np.ndarray:
        """bf16 bit patterns as uint16 [T, H] on the host (the oracle's input form)."""
        return self.x.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def to_device(wl: Workload, device) -> Workload:
    """The same workload with its tensors (bank included) copied to `device` (no arithmetic)."""
    def mv(obj):
        return dataclasses.replace(obj, **{f.name: getattr(obj, f.name).to(device)
                                          for f in dataclasses.fields(obj)
                                          if isinstance(getattr(obj, f.name), torch.Tensor)})
    out = mv(wl)
    out.bank = mv(wl.bank)
    return out


def make_routes(kind: str, T: int, E: int, seed: int, topk: int = TOPK) -> torch.Tensor:
    if kind == "fixture":
        return fixture_routes(T, E)
    return sampled_routes(T, E, kind, seed, topk)


def make_workload(name: str, device="cpu", bank=None, route_set: int = 0, T: Optional[int] = None,
                  x_scale: float = 1.0, E: Optional[int] = None) -> Workload:
    """Build one named workload. ``bank`` may be passed to reuse an already generated bank;
    ``route_set`` selects another seeded draw of routes/activations/weights for the same bank.
    ``E`` restricts the bank to its first E experts (same bytes) and routes over those only."""
    c = CONFIGS[name]
    T = c["T"] if T is None else T
    E = c["E"] if E is None else E
    seed = c["seed"] + 7919 * route_set
    if bank is None:
        bank = make_bank(name, device, experts=None if E == c["E"] else range(E))
    if c["x"] == "lcg":
        x = lcg_activations(T, c["H"], salt=route_set).to(device)
    else:
        x = normal_activations(T, c["H"], seed, device, scale=x_scale)
    ids = make_routes(c["routes"], T, E, seed).to(device)
    wts = softmax_route_weights(T, seed).to(device)
    return Workload(name, c["fmt"], T, c["H"], c["I"], E, TOPK, x, ids, wts, bank, LIMIT)


def make_bank(name: str, device="cpu", experts=None):
    c = CONFIGS[name]
    if c["fmt"] == "fp8":
        return make_fp8_bank(c["E"], c["H"], c["I"], c["bank_seed"], device, experts)
    return make_nvfp4_bank(c["E"], c["H"], c["I"], c["bank_seed"], device, experts)


def make_custom(fmt: str, T: int, H: int, I: int, E: int, seed: int, device="cpu",
                routes: str = "uniform", topk: int = TOPK, x_scale: float = 1.0,
                limit: float = LIMIT) -> Workload:
    """A small workload of arbitrary shape for parity tests (ragged T, several tiles)."""
    bank = (make_fp8_bank(E, H, I, seed, device) if fmt == "fp8"
            else make_nvfp4_bank(E, H, I, seed, device))
    x = normal_activations(T, H, seed, device, scale=x_scale)
    ids = make_routes(routes, T, E, seed, topk).to(device)
    wts = softmax_route_weights(T, seed, topk).to(device)
    return Workload(f"custom_{fmt}_{T}x{H}x{I}x{E}", fmt, T, H, I, E, topk, x, ids, wts, bank, limit)

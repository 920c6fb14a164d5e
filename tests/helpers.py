"""Shared test helpers: tolerance checks and oracle runs on (sub-banks of) seeded workloads."""
import numpy as np
import torch

import oracle

# Floating-point tolerance of the bf16 outputs against the FP64 oracle: relative L2 error
# <= 5e-3 and max abs error <= 2e-2 * RMS(out).
REL_L2_TOL = 5e-3
MAX_ABS_RMS_TOL = 2e-2


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    diff = got - ref
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(diff) / nref) if nref > 0 else float(np.linalg.norm(diff))
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert rel <= REL_L2_TOL, f"{what}: rel L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_RMS_TOL * rms + 1e-30, f"{what}: max abs {mx:.3e} > {MAX_ABS_RMS_TOL}*rms ({rms:.3e})"
    return rel, mx / rms if rms > 0 else 0.0


def oracle_for(wl, tokens=None, ids=None, x_bits=None, limit=None, nthreads=0):
    """Run the oracle on a workload, copying to the host only the experts the chosen tokens use
    (ids are remapped onto that sub-bank; -1 and out-of-range ids are kept as they are)."""
    ids = (wl.ids if ids is None else ids).detach().cpu().numpy().astype(np.int32)
    wts = wl.wts.detach().cpu().numpy()
    xb = wl.x_bits() if x_bits is None else x_bits
    limit = wl.limit if limit is None else limit
    rows = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    used = sorted({int(e) for e in ids[rows].reshape(-1) if 0 <= e < wl.E})
    remap = {e: i for i, e in enumerate(used)}
    sub_ids = np.full_like(ids, -1)          # rows outside `tokens` are never read
    for t in rows:
        for k, e in enumerate(ids[t]):
            if 0 <= e < wl.E:
                sub_ids[t, k] = remap[int(e)]
            elif e != -1:
                sub_ids[t, k] = len(used) + 10_000     # stays out of range for the sub-bank
    if not used:
        used = [0]
    if used == list(range(wl.E)):
        bank = wl.bank.numpy()                 # every expert: no gathered copy of the bank
    else:
        bank = wl.bank.numpy(torch.tensor(used, dtype=torch.long))
    fn = oracle.moe_fp8 if wl.fmt == "fp8" else oracle.moe_nvfp4
    return fn(xb, sub_ids, wts, bank, limit, tokens=tokens, nthreads=nthreads)


def prefill_sample_tokens(ids, E: int, tile_rows: int = 128):
    """Tokens whose routed pairs touch every expert that has a routed pair, and, for every expert
    with more than one m-tile of sorted rows, the first and last row of its last (partial) m-tile
    and the last row of its first m-tile (the grouped GEMM's tile edges). The pairs of an expert
    are taken in the stable sorted order (ascending pair index t*topk + k)."""
    ids = np.asarray(ids.detach().cpu().numpy() if isinstance(ids, torch.Tensor) else ids)
    T, topk = ids.shape
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    order = np.flatnonzero(valid)[np.argsort(flat[valid], kind="stable")]   # sorted pair indices
    keys = flat[order]
    starts = np.searchsorted(keys, np.arange(E), side="left")
    ends = np.searchsorted(keys, np.arange(E), side="right")
    chosen = set()
    for e in range(E):
        n = ends[e] - starts[e]
        if n > tile_rows:
            last0 = starts[e] + tile_rows * ((n - 1) // tile_rows)
            for pos in (starts[e] + tile_rows - 1, last0, ends[e] - 1):
                chosen.add(int(order[pos]) // topk)
    need = {e for e in range(E) if ends[e] > starts[e]}
    covered = {int(e) for t in chosen for e in ids[t] if 0 <= e < E}
    tok_sets = [{int(e) for e in row if 0 <= e < E} for row in ids]
    left = need - covered
    while left:                                   # greedy cover of the experts still missing
        best = max(range(T), key=lambda t: len(tok_sets[t] & left))
        chosen.add(best)
        left -= tok_sets[best]
    return sorted(chosen)

"""Shared pieces of the GPU parity tests: device setup, seeded inputs for both
sides, oracle construction, and the comparison rules.

Tolerances (floating point): router gates within 1e-5 absolute; layer output
relative L2 <= 5e-3 and max |diff| <= 2e-2 * RMS of the reference. Integer and
byte results (E4M3 codes, scales, histograms, permutation) are compared
bit for bit. Tokens whose routing hinges on a margin below 1e-6 (the oracle
reports them) are excluded from routing and layer comparisons.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

gpu = pytest.mark.gpu

GATE_ATOL = 1e-5
Y_REL_L2 = 5e-3
Y_MAX_RMS = 2e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def y_metrics(got: np.ndarray, want: np.ndarray):
    diff = got.astype(np.float64) - want.astype(np.float64)
    rel = np.linalg.norm(diff) / max(np.linalg.norm(want), 1e-300)
    rms = np.sqrt(np.mean(want.astype(np.float64) ** 2))
    return rel, np.abs(diff).max() / max(rms, 1e-300)


# The budget may explain at most this share of the output (Frobenius norm). One undecidable code
# at the maximum of a 128-token column of h moves that column's scale, and with it a whole column
# of a weight gradient, by up to 1/16: with 64-100 rows per expert (tiny width) that is up to
# about 2.5% of the gradient; outputs and input gradients stay near 1%.
BUDGET_CAP = 5e-2


def assert_y_close(got, want, budget=None, name="y", cap=True):
    """rel-L2 <= 5e-3 of the whole difference; max |diff| <= 2e-2 * RMS of what the budget does
    not explain. The budget (oracle/bounds.py: Layer.forward(budget=True), layer_backward) is
    how far another correct FP32 evaluation may lie from the oracle through its E4M3 rounding
    decisions alone, element by element; it is capped at BUDGET_CAP of the output as a whole
    (cap=False for sums over many tokens, whose budget adds every token's without the
    cancellation the sum itself has: the raw relative-L2 bar holds those)."""
    rel, mx = y_metrics(got, want)
    msg = f"[parity] {name}: rel-L2 {rel:.3e}  max-abs/RMS {mx:.3e}  over {got.shape[0]} rows"
    if budget is not None:
        diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
        rms = np.sqrt(np.mean(want.astype(np.float64) ** 2))
        resid = np.maximum(diff - budget, 0.0)
        mx = resid.max() / max(rms, 1e-300)
        share = np.linalg.norm(budget) / max(np.linalg.norm(want), 1e-300)
        material = float(np.mean(budget > 1e-3 * rms))
        msg += (f"; beyond the E4M3-decision budget max-abs/RMS {mx:.3e}; budget {share:.2e} of the output, "
                f"above 1e-3 RMS on {material:.2%} of elements")
        print(msg)
        if cap:
            assert share <= BUDGET_CAP, f"{name}: budget {share:.3e} of the output"
    else:
        print(msg)
    assert rel <= Y_REL_L2, f"{name}: rel-L2 {rel:.3e}"
    assert mx <= Y_MAX_RMS, f"{name}: max-abs/RMS {mx:.3e}"
    return rel, mx


# Oracle experts quantised so far in this test session, keyed by (expert seed,
# d, I, scale rule, expert): the full-width workloads share one set of expert
# weights, so their tests quantise each expert once.
_EXPERTS: dict = {}


def oracle_experts(cfg, experts, device="cuda", rule="fp32", batch: int = 48):
    """Quantised oracle experts for `experts`, built in parallel CPU workers.

    The fp32 weights come from the same seeded generator (on `device`) that
    fed the CUDA path; the workers run only the oracle's quantiser. Weights
    are drawn `batch` experts at a time to bound host memory.
    """
    from oracle.parallel import quantize_experts
    from sparse_moe_layer_13_b300.inputs import gen_expert
    key = (cfg.weight_seed, cfg.d, cfg.I, rule)
    want = sorted(set(int(e) for e in experts))
    missing = [e for e in want if key + (e,) not in _EXPERTS]
    for i in range(0, len(missing), batch):
        jobs = [(e, *(to_np(w) for w in gen_expert(cfg, e, device))) for e in missing[i:i + batch]]
        for e, q in quantize_experts(jobs, rule=rule).items():
            _EXPERTS[key + (e,)] = q
        del jobs
    return {e: _EXPERTS[key + (e,)] for e in want}


def oracle_route_chunked(x, Wr, bias, cfg, logit_offset=None, chunk: int = 8192):
    """The oracle router over a large batch, a slice of tokens at a time (routing is
    per token, so this is the same function; it only bounds the FP64 copies)."""
    from oracle.route import route as oracle_route
    parts = [oracle_route(np.asarray(x[i:i + chunk], np.float32), Wr, bias, cfg.G, cfg.M, cfg.K, cfg.gk,
                          logit_offset) for i in range(0, x.shape[0], chunk)]
    idx = np.concatenate([p[0] for p in parts])
    gate = np.concatenate([p[1] for p in parts])
    info = {k: np.concatenate([p[2][k] for p in parts]) for k in parts[0][2]}
    return idx, gate, info


def check_routing(cfg, idx_gpu, gate_gpu, ref_idx, ref_gate, info):
    """Bit-exact expert choice and order, gates within GATE_ATOL, on non-tie tokens."""
    from oracle.route import near_tie
    tie = near_tie(info)
    ok = ~tie
    gi = np.asarray(idx_gpu)
    gg = np.asarray(gate_gpu)
    assert np.array_equal(np.sort(gi[ok], 1), np.sort(ref_idx[ok], 1)), "chosen expert sets differ"
    strict = ok & (info["order_gap"] > 1e-6)
    assert np.array_equal(gi[strict], ref_idx[strict]), "order of chosen experts differs"
    o1 = np.argsort(gi[ok], 1)
    o2 = np.argsort(ref_idx[ok], 1)
    g1 = np.take_along_axis(gg[ok], o1, 1)
    g2 = np.take_along_axis(ref_gate[ok], o2, 1)
    err = np.abs(g1 - g2).max() if g1.size else 0.0
    assert err <= GATE_ATOL, f"gate error {err:.3e}"
    return tie, err


def check_load_and_bias(cfg, gpu_idx, gpu_counts, ref_idx, tie, b0, bias_after, T=None):
    """End-of-step checks (《DeepSeek-V3 Technical Report》深度解读报告 §2.3), every call:
    the device histogram is exactly that of the device's choice; with the near-tie tokens
    taken out of both, it equals the oracle's load; and the updated bias is, bit for bit,
    the update rule applied to the device's load."""
    from oracle.layer import bias_update
    T = cfg.T if T is None else T

    def histogram(idx, E):          # a library count (the oracle's own histogram is pinned to it)
        return np.bincount(np.asarray(idx).ravel(), minlength=E).astype(np.int32)

    assert np.array_equal(gpu_counts, histogram(gpu_idx, cfg.E))
    assert np.array_equal(histogram(gpu_idx[~tie], cfg.E), histogram(ref_idx[~tie], cfg.E))
    assert np.array_equal(bias_after, bias_update(b0, gpu_counts, T, cfg.K, cfg.gamma))
    # the oracle's own load gives the same bias except where near-tie tokens can move an
    # expert's load across the mean
    ob = bias_update(b0, histogram(ref_idx, cfg.E), T, cfg.K, cfg.gamma)
    moved = np.zeros(cfg.E, bool)
    moved[np.unique(np.concatenate([gpu_idx[tie].ravel(), ref_idx[tie].ravel()]))] = True
    assert np.all((ob == bias_after) | moved)

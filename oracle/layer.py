"""Whole DeepSeekMoE layer forward, combine and end-of-step bias update.

《DeepSeek-V3 Technical Report》深度解读报告 §2.2: output = u + sum over shared
experts of FFN(u) + sum over routed experts of g * FFN(u). Here there is one
shared expert (devpress blog §1: 256 routed + 1 shared). The residual u is
added only when asked for; the checks compare the expert sum itself.

§2.3: at the end of a step, an overloaded expert's bias drops by gamma and an
underloaded expert's bias rises by gamma. Reading: loads are compared with
the mean load T*K/E of the step's whole batch; an expert exactly at the mean
keeps its bias. Bias values are float32 and the update is one float32 add.
"""
from __future__ import annotations

import numpy as np

from . import route as _route
from .ffn import QuantExpert, expert_forward
from .permute import histogram
from .quant import quant_1x128


def combine(shared_out, routed_out, gate, residual=None) -> np.ndarray:
    """shared_out [T][d], routed_out [T][K][d], gate [T][K] -> float64 [T][d].

    The result is left unrounded: it is the exact layer value for these
    expert outputs, against which a bf16 result is judged (its own rounding
    to bf16 is part of the error it is charged with).
    """
    y = np.asarray(shared_out, np.float64).copy()
    for k in range(routed_out.shape[1]):
        y += np.asarray(gate, np.float64)[:, k][:, None] * routed_out[:, k, :]
    if residual is not None:
        y += np.asarray(residual, np.float64)
    return y


def bias_update(bias, counts, T: int, K: int, gamma: float) -> np.ndarray:
    """b_e <- b_e + gamma * sign(mean - c_e), mean = T*K/E, one float32 rounding."""
    bias = np.asarray(bias, np.float32)
    counts = np.asarray(counts, np.int64)
    E = bias.shape[0]
    sign = np.sign(T * K - counts * E)           # exact: compares c_e with T*K/E
    step = (np.float32(gamma) * sign.astype(np.float32)).astype(np.float32)
    return np.where(sign == 0, bias, (bias + step).astype(np.float32)).astype(np.float32)


class Layer:
    """Oracle for one layer instance.

    expert_weights(e) -> (W1 [I][d], W3 [I][d], W2 [d][I]) float32, with e == E
    the shared expert. Quantised experts are built on first use and cached;
    `experts` may pre-fill that cache with QuantExpert objects.
    """

    def __init__(self, cfg, Wr, bias, expert_weights, logit_offset=None, experts=None, rule: str = "fp32"):
        self.cfg = cfg
        self.rule = rule
        self.Wr = np.asarray(Wr, np.float32)
        self.bias = np.asarray(bias, np.float32)
        self.logit_offset = None if logit_offset is None else np.asarray(logit_offset, np.float32)
        self._weights = expert_weights
        self._experts: dict[int, QuantExpert] = dict(experts or {})

    def expert(self, e: int) -> QuantExpert:
        if e not in self._experts:
            self._experts[e] = QuantExpert(*[np.asarray(w, np.float32) for w in self._weights(e)], rule=self.rule)
        return self._experts[e]

    def route(self, x):
        c = self.cfg
        return _route.route(x, self.Wr, self.bias, c.G, c.M, c.K, c.gk, self.logit_offset)

    def forward(self, x, tokens=None, idx=None, gate=None, residual=False, budget=False):
        """x [T][d] float32 (bf16 values). Returns a dict with y for `tokens` (all by default).

        idx/gate may be given to evaluate the experts for a fixed routing. budget: also
        "budget", per element of y, how far another correct FP32 evaluation of the layer may
        lie from y through its E4M3 decisions on h (each expert's, expert_forward) and its
        gates' error bound (oracle/bounds.py, gate_err), combined with the gates.
        """
        c = self.cfg
        x = np.asarray(x, np.float32)
        info = None
        if idx is None:
            idx, gate, info = self.route(x)
        tokens = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
        xq, xs = quant_1x128(x[tokens], self.rule)
        n = len(tokens)
        routed = np.zeros((n, c.K, c.d), dtype=np.float64)
        b_routed = np.zeros((n, c.K, c.d), dtype=np.float64) if budget else None
        sub_idx = np.asarray(idx)[tokens]
        for e in np.unique(sub_idx):
            rows, slots = np.nonzero(sub_idx == e)
            if budget:
                routed[rows, slots], b_routed[rows, slots] = expert_forward(xq[rows], xs[rows], self.expert(int(e)),
                                                                            budget=True)
            else:
                routed[rows, slots] = expert_forward(xq[rows], xs[rows], self.expert(int(e)))
        if budget:
            shared, b_shared = expert_forward(xq, xs, self.expert(c.E), budget=True)
        else:
            shared = expert_forward(xq, xs, self.expert(c.E))
        res = x[tokens] if residual else None
        g = np.asarray(gate)[tokens]
        y = combine(shared, routed, g, res)
        out = {"y": y, "idx": idx, "gate": gate, "info": info, "tokens": tokens,
               "counts": histogram(idx, c.E), "routed": routed, "shared": shared}
        if budget:
            from .bounds import gate_err
            s = _route.affinity(x[tokens], self.Wr, self.logit_offset)
            ge = gate_err(np.take_along_axis(s, sub_idx, axis=1))
            out["budget"] = (b_shared + np.einsum("tk,tkd->td", np.abs(g), b_routed)
                             + np.einsum("tk,tkd->td", ge, np.abs(routed)))
        return out

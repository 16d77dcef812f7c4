"""Oracle evaluation of a synthetic layer whose weights live in device memory.

Test infrastructure only.  The weights come from the seeded generator
(:mod:`synth.device`); only the router and the experts the oracle itself
selects are copied to the host.  Nothing here touches the CUDA library.
"""
from __future__ import annotations

import numpy as np

from . import oracle

# Output tolerance for bf16 layers (max-abs, relative L2).
MAX_ABS = 2e-2
REL_L2 = 5e-3
# Tokens whose 6th and 7th oracle logits are closer than this may be routed
# either way by an fp32 router; for them both outcomes are accepted.
NEAR_TIE = 1e-5


def margins(logits: np.ndarray, k: int = 6) -> np.ndarray:
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


class LayerOracle:
    """Caches host copies of experts of one device layer (bf16 or NVFP4 Mats)."""

    def __init__(self, router_bits, bias, expert_mats, shared_mats, E: int = 256):
        self.router_bits = router_bits
        self.bias = bias
        self.expert_mats = expert_mats   # callable e -> (Mat gate_up, Mat down)
        self.shared = shared_mats
        self.E = E
        self._cache = {}

    @classmethod
    def from_bf16_layer(cls, lw):
        def mats(e):
            gu, dn = lw.expert_bits(e)
            return oracle.Mat(gu), oracle.Mat(dn)
        sgu, sdn = lw.expert_bits(lw.E)
        return cls(lw.router_bits(), lw.bias_host(), mats, (oracle.Mat(sgu), oracle.Mat(sdn)), lw.E)

    def _mats_for(self, experts):
        gus = [oracle.Mat.absent()] * self.E
        dns = [oracle.Mat.absent()] * self.E
        for e in experts:
            if e not in self._cache:
                self._cache[e] = self.expert_mats(int(e))
            gus[e], dns[e] = self._cache[e]
        return gus, dns

    def route(self, x_bits):
        logits = oracle.router_logits(x_bits, self.router_bits, self.bias)
        idx, w = oracle.select(logits)
        return logits, idx, w

    def forward(self, x_bits, idx_in=None):
        logits, idx, _ = self.route(x_bits)
        sel = idx if idx_in is None else idx_in
        gus, dns = self._mats_for(sorted(set(np.asarray(sel).ravel().tolist())))
        return oracle.moe_forward(x_bits, self.router_bits, self.bias, gus, dns, self.shared, idx_in=idx_in)

    def forward_with_alternatives(self, x_bits):
        """Oracle output, plus for near-tie tokens the output under the
        runner-up selection (6th choice replaced by the 7th-ranked expert)."""
        base = self.forward(x_bits)
        mg = margins(base["logits"])
        near = np.nonzero(mg < NEAR_TIE)[0]
        alt_y = {}
        if len(near):
            alt = base["idx"].copy()
            for t in near:
                order = np.argsort(-base["logits"][t], kind="stable")
                alt[t, 5] = order[6]
            r = self.forward(x_bits[near], idx_in=alt[near])
            for i, t in enumerate(near):
                alt_y[int(t)] = r["y"][i]
        return base, alt_y


def compare(y_gpu: np.ndarray, base, alt_y=None, max_abs=MAX_ABS, rel_l2=REL_L2):
    """Element-wise comparison of a device output (float array [T][H]) with
    the oracle.  Near-tie tokens may match the runner-up output instead.
    Returns a dict of error figures; 'ok' says whether both bounds hold."""
    y_ref = base["y"].copy()
    alt_y = alt_y or {}
    for t, ya in alt_y.items():
        if np.abs(y_gpu[t] - ya).max() < np.abs(y_gpu[t] - y_ref[t]).max():
            y_ref[t] = ya
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    mx = float(err.max())
    rel = float(np.linalg.norm(y_gpu.astype(np.float64) - y_ref) / max(np.linalg.norm(y_ref), 1e-300))
    return {"max_abs": mx, "rel_l2": rel, "ok": mx <= max_abs and rel <= rel_l2,
            "near_ties": len(alt_y)}

"""Write tau_decisions.json: the oracle's tau1/tau2 decisions on every full-size workload,
and how far the rel-MAE trace stands from each threshold that decides them.

Calls only the oracle (``oracle.cfg_oracle.run_sampler``) and the seeded input draws
(``workloads``); nothing here touches the CUDA library.  Run from the repository root:

    python tests/golden/make_tau_decisions.py

The rule (Hybridiff notes, key design 3) decides tau1' by comparing each slope
G_s = (M_s - M_{s-L}) / L with 0 and g_slope, and tau_cap by the argmin of the trace.  A
device whose trace differs from the oracle's by dM per step moves each G by at most
2 dM / L, so its decisions equal the oracle's whenever 2 max|dM| / L is below the margins
recorded here:

    g_margin_zero   min |G_s|            over L <= s <= s_end
    g_margin_slope  min |G_s - g_slope|  over L <= s <= s_end
    (s_end = tau1' if found, else the last step: a threshold crossing anywhere up to the
    decision could move it)
    m_argmin_gap    (second smallest M - smallest M), the distance that keeps the argmin
"""
from __future__ import annotations

import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402
from oracle import cfg_oracle as O  # noqa: E402

OUT = Path(__file__).resolve().parent / "tau_decisions.json"


def margins(M: np.ndarray, L: int, g_slope: float, tau1p: int) -> dict:
    N = M.shape[0]
    s_end = tau1p if tau1p != O.TAU_NONE else N - 1
    G = np.array([(M[s] - M[s - L]) / L for s in range(L, s_end + 1)])
    srt = np.sort(M[~np.isnan(M)])
    return {
        "g_margin_zero": float(np.min(np.abs(G))) if G.size else None,
        "g_margin_slope": float(np.min(np.abs(G - g_slope))) if G.size else None,
        "m_argmin_gap": float(srt[1] - srt[0]) if srt.size > 1 else None,
        "M_first": float(M[0]), "M_min": float(srt[0]), "M_last": float(M[-1]),
        "monotone_rising": bool(np.all(np.diff(M) > 0)),
        "monotone_falling": bool(np.all(np.diff(M) < 0)),
    }


def decisions(name: str) -> dict:
    wl = W.WORKLOADS[name]
    inputs = W.draw_inputs(wl)
    pert = (lambda s, b: W.draw_perturbation(wl, s, b)) if wl.perturb_std else None
    ref = O.run_sampler(wl, inputs, perturb=pert)
    row = dict(ref.sched.as_dict())
    row.update(margins(ref.M, wl.L, wl.g_slope, ref.sched.tau1p))
    row.update({"L": wl.L, "g_slope": wl.g_slope, "k": wl.k, "n_steps": wl.n_steps})
    return row


def main() -> None:
    table = {name: decisions(name) for name in W.WORKLOAD_ORDER}
    OUT.write_text(json.dumps(table, indent=1, sort_keys=True) + "\n")
    for name, row in table.items():
        print(name, {k: row[k] for k in ("tau1p", "tau_cap", "tau1", "tau2", "decided_at",
                                         "g_margin_zero", "g_margin_slope", "m_argmin_gap")})


if __name__ == "__main__":
    main()

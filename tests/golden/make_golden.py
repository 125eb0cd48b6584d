"""Writes the fixtures of this directory from the fp64 oracle (and nothing else).

The source pages print formulas but no numeric worked example, so these fixtures are
not page values: they are small problems with hand-picked inputs (multiples of 1/8, so
that fp32 and bf16 hold them exactly) and the oracle's results, stored so that
  * a change of the oracle's arithmetic shows up as a failing comparison (such a change
    must cite the passage that justifies it), and
  * the CUDA entry points can be checked against fixed numbers.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def eighths(rng, shape, lo=-16, hi=16):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) / 8.0


def scan_case():
    rng = np.random.default_rng(7)
    nb, L, D, N = 1, 6, 2, 3
    p = dict(x=eighths(rng, (nb, L, D)), delta=eighths(rng, (nb, L, D), -8, 4),
             A=-(np.arange(1, N + 1, dtype=np.float64)[None, :] * np.ones((D, 1))),
             B=eighths(rng, (nb, L, N)), C=eighths(rng, (nb, L, N)),
             D=np.array([0.5, -0.25]), z=eighths(rng, (nb, L, D)), bias=np.array([0.125, -0.5]))
    y, hf = oracle.scan(p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"], z=p["z"],
                        bias=p["bias"], softplus=True, threads=1)
    gy = eighths(rng, (nb, L, D))
    g = oracle.scan_bwd(gy, p["x"], p["delta"], p["A"], p["B"], p["C"], Dv=p["D"], z=p["z"],
                        bias=p["bias"], softplus=True)
    return {
        "what": "S6 scan with softplus step, Euler B, D skip and SiLU gate, and its "
                "gradients for the upstream gradient dy (final-state gradient zero)",
        "source": "tildalice review, sections \"Selection Mechanism\", \"Δ의 직관적 이해\", "
                  "\"Mamba 블록 아키텍처\"; yongggg review, section \"State Space Model\" "
                  "(D skip); backward: tildalice \"Hardware-Aware 병렬 알고리즘\"",
        "inputs": {k: v.tolist() for k, v in p.items()} | {"dy": gy.tolist()},
        "y": y.tolist(), "h_final": hf.tolist(),
        "grads": {k: v.tolist() for k, v in g.items()},
    }


def conv_case():
    rng = np.random.default_rng(8)
    nb, L, D, K = 2, 5, 8, 4
    x = eighths(rng, (nb, L, D))
    w = eighths(rng, (D, K), -4, 4)
    b = eighths(rng, (D,), -2, 2)
    out = oracle.conv1d(x, w, b, silu=True)
    return {
        "what": "causal depthwise Conv1D (K = 4, K - 1 steps of zero left padding) + SiLU",
        "source": "tildalice review, section \"Mamba 블록 아키텍처\" (Conv1D k=4, SiLU)",
        "inputs": {"x": x.tolist(), "w": w.tolist(), "bias": b.tolist()},
        "out": out.tolist(),
    }


def main():
    for name, fn in (("scan_small.json", scan_case), ("conv1d_small.json", conv_case)):
        with open(os.path.join(HERE, name), "w", encoding="utf-8") as f:
            json.dump(fn(), f, indent=1, ensure_ascii=False)
        print("wrote", name)


if __name__ == "__main__":
    main()

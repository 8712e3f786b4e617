"""Writes tiny_gqa_rope.txt: the oracle's outputs on one tiny GQA + RoPE case,
stored so that an unintended change to the oracle's arithmetic fails
tests/test_golden.py.

The pages print no attention values for a worked example (their gradient
check reports whole-model tensors only: "Rebuilding GPT-2 in one 100KB
C/CUDA file", section 2.1), so every stored value here comes from this
script, which calls only the oracle.  Inputs are a closed-form formula (no
random numbers), so they are reproducible anywhere.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

B, T, Hq, Hkv, d = 1, 6, 4, 2, 8
THETA = 10000.0
OUT = os.path.join(HERE, "tiny_gqa_rope.txt")


def inputs():
    """q, k, v, dO of shape [B, T, H, d] from smooth closed forms."""
    def f(H, a, b, c):
        t = np.arange(T)[None, :, None, None]
        h = np.arange(H)[None, None, :, None]
        e = np.arange(d)[None, None, None, :]
        x = np.sin(a * (t + 1) * (e + 1) + b * h + c) + 0.25 * np.cos(0.7 * e - 0.3 * t)
        return np.broadcast_to(x, (B, T, H, d)).copy()
    return f(Hq, 0.37, 0.11, 0.0), f(Hkv, 0.23, 0.41, 1.0), f(Hkv, 0.19, 0.29, 2.0), \
        f(Hq, 0.31, 0.17, 3.0)


def compute():
    q, k, v, do = inputs()
    o, lse = oracle.attn_fwd(q, k, v, THETA)
    r = oracle.attn_bwd(q, k, v, do, THETA)
    return {"o": o, "lse": lse, "dq": r["dq"], "dk": r["dk"], "dv": r["dv"]}


def main():
    out = compute()
    with open(OUT, "w") as f:
        f.write(f"# oracle outputs, B={B} T={T} Hq={Hq} Hkv={Hkv} d={d} rope_theta={THETA}; "
                "inputs: make_golden.inputs(); written by tests/golden/make_golden.py\n")
        for name, x in out.items():
            f.write(f"{name} {' '.join(str(s) for s in x.shape)}\n")
            f.write(" ".join(f"{v:.17e}" for v in x.reshape(-1)) + "\n")


if __name__ == "__main__":
    main()

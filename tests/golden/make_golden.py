"""Write tests/golden/oracle_d8_t40.npz from the oracle (calls only oracle/ and wkv7_inputs)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import wkv7_inputs  # noqa: E402


def main():
    x = wkv7_inputs.random_small(7, B=2, T=40, H=3, D=8, h0_std=0.1, dhT_std=1.0)
    y, ck, hT = oracle.forward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], chunk=16)
    g = oracle.backward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], ck, x["dy"], x["dhT"],
                        chunk=16, mode="full")
    names = ("dr", "dw", "dk", "dv", "da", "db", "dh0")
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_d8_t40.npz")
    np.savez(out, y=y, h_ckpt=ck, hT=hT, **dict(zip(names, g)))
    print("wrote", out)


if __name__ == "__main__":
    main()

"""Write the oracle regression fixture for the tiny workload (N=1, Hk=2, H=4, S=32, T=16).

Calls only the CPU oracle (double build) on the seeded inputs; the CUDA path is
never involved. The fixture pins the oracle against silent drift: a later change
to its arithmetic changes these numbers and fails tests/test_golden.py until the
fixture is regenerated on purpose.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402

OUT = os.path.join(HERE, "tiny_oracle_f64.txt")


def compute():
    cfg = I.get_config(0)
    rec = I.recurrence_batch(cfg)
    st = I.state_pool(cfg).astype(np.float64)
    y, _ = oracle.recurrence(st, rec["q"], rec["k"], rec["v"], rec["g"], rec["beta"], cfg.scale)
    res = {"scan_y_t15_h3": y[0, 15, 3, :8], "scan_state_sum": np.array([st.sum()]),
           "scan_y_abs_sum": np.array([np.abs(y).sum()])}
    stat = I.block_static(cfg)
    cs = I.conv_state_pool(cfg).astype(np.float64)
    st = I.state_pool(cfg).astype(np.float64)
    for step in range(cfg.steps):
        a = I.block_step(cfg, step)
        out, _ = oracle.block_decode(a["qkv"], stat["conv_w"], cs, a["alpha"], a["b"], stat["dt"],
                                     stat["a"], a["z"], stat["norm_w"], st, cfg.n_k_heads,
                                     cfg.scale, cfg.eps, cfg.eps)
    res["block_out_last_h1"] = out[0, 1, :8]
    res["block_state_sum"] = np.array([st.sum()])
    res["block_conv_state_sum"] = np.array([cs.sum()])
    return res


def main():
    res = compute()
    with open(OUT, "w") as f:
        f.write("# CPU oracle (double build) on the seeded tiny workload; written by make_golden.py\n")
        for key, val in res.items():
            f.write(key + " " + " ".join(repr(float(x)) for x in val) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()

"""Oracle results for single (sequence, v-head) units of a scan, computed in parallel
threads (the oracle is C called through ctypes, which releases the GIL), and the full
4 x 4096 prefill workload's results cached for the session: several GPU tests hold
their scan forms to every unit of it."""
import functools
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle
from gated_deltanet_linear_scan_gb300 import inputs as I


def oracle_units(cfg, x, st0, units):
    """{(n, vh): (y [T][S], final state [S][S])} from the oracle (double build)."""

    def one(unit):
        n, vh = unit
        kh = vh % cfg.n_k_heads
        sub = {"q": x["q"][n:n + 1, :, kh:kh + 1], "k": x["k"][n:n + 1, :, kh:kh + 1],
               "v": x["v"][n:n + 1, :, vh:vh + 1], "g": x["g"][n:n + 1, :, vh:vh + 1],
               "beta": x["beta"][n:n + 1, :, vh:vh + 1]}
        s_ref = np.ascontiguousarray(st0[n:n + 1, vh:vh + 1], dtype=np.float64)
        y_ref, _ = oracle.recurrence(s_ref, scale=cfg.scale, **sub)
        return unit, (y_ref[0, :, 0], s_ref[0, 0])

    oracle.sigmoid(np.zeros(1, np.float32))  # load the library before the threads start
    with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        return dict(ex.map(one, units))


@functools.lru_cache(maxsize=1)
def prefill_4x4096():
    """(cfg, inputs, initial state, {unit: (y, state)}) of the 4 x 4096 prefill workload
    for all 128 (sequence, v-head) units."""
    cfg = I.get_config(2)
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    units = [(n, vh) for n in range(cfg.n_seqs) for vh in range(cfg.n_v_heads)]
    return cfg, x, st0, oracle_units(cfg, x, st0, units)

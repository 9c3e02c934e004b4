"""Writes prev_comb_sinkhorn20.npy: the previous layer's residual mixes the seeded input generator
draws from.  The workload definition gives the previous comb_res_mix as the 20-iteration Sinkhorn
normalisation of exp(N(0, 0.5)) (0.5 the standard deviation, as for the other N(0, s) draws
there); the generator holds none of the op's arithmetic, so the normalisation happens here, once,
with the oracle's Sinkhorn (sinkhorn_eps = 3e-4, reading A5), over 1024 seeded matrices, stored as
float32 [1024, 4, 4].  Each token then takes one of them by a seeded index.

    python tests/golden/make_prev_comb_table.py      (from the repository root)
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

N, ITERS, EPS, SEED = 1024, 20, 3e-4, (2025, 11)
PATH = os.path.join(HERE, "prev_comb_sinkhorn20.npy")


def table():
    import oracle
    rng = np.random.default_rng(SEED)
    M = np.exp(0.5 * rng.standard_normal((N, 4, 4)))
    return np.stack([oracle.sinkhorn(m, ITERS, EPS) for m in M]).astype(np.float32)


if __name__ == "__main__":
    np.save(PATH, table())
    print("wrote", PATH)

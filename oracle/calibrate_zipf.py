"""Fix the strength of the prefill workload's Zipf logit skew.

Test infrastructure: it routes the seeded 35B prefill inputs with the oracle's
softmax-top-k for a few candidate strengths and prints the one whose realised
expert-load log-log slope is closest to -1.1.  The chosen value is stored as
``ZIPF_BETA`` in the synthetic-input module; tests/test_oracle_pins.py checks
the realised slope of that stored value.

    python -m oracle.calibrate_zipf
"""
import numpy as np

from int4_gathered_expert_gb300 import synth
from oracle import e0_oracle as O


def load_slope(counts: np.ndarray) -> float:
    """Least-squares slope of log(load) against log(rank), experts with load > 0."""
    c = np.sort(np.asarray(counts, np.float64))[::-1]
    c = c[c > 0]
    r = np.arange(1, len(c) + 1, dtype=np.float64)
    A = np.stack([np.log(r), np.ones_like(r)], 1)
    return float(np.linalg.lstsq(A, np.log(c), rcond=None)[0][0])


def realised(beta: float, T: int = 4096, seed: int = 4):
    s = synth.L35B
    Wr = synth.router(seed, 0, s)
    X = synth.normal_rows(seed, T, s.H).astype(np.float16)
    b = synth.zipf_logit_bias(seed, s.E, beta=beta)
    rt = O.route_softmax_topk(O.router_logits(Wr, X, b), s.K)
    counts = np.bincount(rt.inds.ravel(), minlength=s.E)
    return load_slope(counts), counts


def main():
    best = None
    for beta in np.arange(0.30, 0.4501, 0.005):
        slope, counts = realised(float(beta))
        print(f"beta={beta:.2f} slope={slope:+.3f} top={counts.max()} min={counts.min()}")
        if best is None or abs(slope + 1.1) < abs(best[1] + 1.1):
            best = (float(beta), slope)
    print("best beta %.2f slope %.3f" % best)


if __name__ == "__main__":
    main()

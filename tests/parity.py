"""Comparison helpers for GPU-vs-oracle parity (test infrastructure)."""
import numpy as np

TIE_REL = 1e-6      # routing: index mismatches allowed only below this relative score gap
REL_L2 = 2e-3       # MoE outputs: relative L2 bound
W_ATOL = 1e-5       # routing weights (fp32 arithmetic on the GPU)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (d if d > 0 else 1.0))


def _adjacent_tie(scores, order, K):
    """True when two neighbours among the top K+1 of ``order`` are closer than TIE_REL."""
    top = scores[order[:K + 1]] if K < len(order) else scores[order[:K]]
    for a, b in zip(top[:-1], top[1:]):
        if np.isfinite(b) and abs(a - b) <= TIE_REL * max(abs(a), 1e-300):
            return True
    return False


def routing_matches(gpu_inds, gpu_w, rt, allow_tie=True):
    """Compare a GPU routing [T,K] with an oracle Routing.  Returns
    (exempt_tokens, messages).  Non-exempt tokens must match exactly (ordered
    indices) with weights within W_ATOL; a token is exempt when the oracle's
    K-th and (K+1)-th scores (or its G-th and (G+1)-th group scores) differ by
    less than TIE_REL relative.  Within an exempt-free token, if two selected
    experts are themselves tied the sets are compared instead of the order.
    gpu_w None: indices only."""
    gpu_inds = np.asarray(gpu_inds)
    gpu_w = None if gpu_w is None else np.asarray(gpu_w, np.float64)
    T, K = rt.inds.shape
    exempt, msgs = [], []
    for t in range(T):
        if allow_tie and (rt.gap[t] < TIE_REL or rt.group_gap[t] < TIE_REL):
            exempt.append(t)
            continue
        order = np.argsort(-rt.scores[t], kind="stable")
        if list(gpu_inds[t]) != list(rt.inds[t]):
            if not (_adjacent_tie(rt.scores[t], order, K) and set(gpu_inds[t]) == set(rt.inds[t])):
                msgs.append(f"token {t}: gpu {list(gpu_inds[t])} oracle {list(rt.inds[t])} gap {rt.gap[t]:.3g}")
                continue
        if gpu_w is None:
            continue
        want = {int(e): float(w) for e, w in zip(rt.inds[t], rt.w[t])}
        for e, w in zip(gpu_inds[t], gpu_w[t]):
            if abs(want[int(e)] - w) > W_ATOL:
                msgs.append(f"token {t}: weight of expert {e} gpu {w} oracle {want[int(e)]}")
    return exempt, msgs


def tile_edge_tokens(inds, n_experts=3, tile=128, per_expert=8):
    """Tokens that sit at the edges of the token tiles of the ``n_experts``
    busiest experts: an expert's tokens, in token order (the order a stable
    sort by expert keeps), are cut into tiles of ``tile``; the first and last
    token of each tile and the expert's last token are taken, up to
    ``per_expert`` of them.  Tile-boundary mistakes in a grouped GEMM show up
    on exactly these tokens."""
    inds = np.asarray(inds)
    counts = np.bincount(inds.ravel(), minlength=int(inds.max()) + 1)
    out = set()
    for e in np.argsort(-counts, kind="stable")[:n_experts]:
        toks = np.nonzero((inds == e).any(axis=1))[0]
        n = len(toks)
        pos = []
        for t0 in range(0, n, tile):
            pos += [t0, min(t0 + tile, n) - 1]
        pos = sorted(set(pos))
        if len(pos) > per_expert:
            keep = np.linspace(0, len(pos) - 1, per_expert).round().astype(int)
            pos = [pos[i] for i in keep]
        out.update(int(toks[p]) for p in pos)
    return sorted(out)

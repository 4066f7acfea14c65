"""Seeded synthetic workloads with the shapes of the Edge0 release tiers.

This module is shared by the CUDA path and by the CPU oracle, so it holds no
arithmetic of the method itself: it only draws random numbers and lays them
out in the canonical tensor formats below.  Everything here is plain numpy on
the host; callers copy what they need to the device.

Canonical int4 "Q-tensor" for a projection with ``out`` rows and ``inn``
inputs (affine int4, group size 64 along the input dimension; the tier tables
of "Edge0: 35B MoE를 SSD에서 3GiB 메모리로 서빙하기" §"두 공개 티어" and the
release-tier list of the jaehun.me review of "The Other Half of the Memory
Wall" give "int4 affine g64"):

    codes  uint8   [out, inn/2]   element j of a row sits in byte j/2,
                                  low nibble if j is even, high nibble if odd
    scale  float16 [out, inn/64]
    bias   float16 [out, inn/64]

An expert is three Q-tensors: gate [I,H], up [I,H], down [H,I].  A layer's
bank stacks them over the expert axis, which gives the nine per-layer tensors
(gate/up/down x codes/scale/bias) that the pages describe for the whole-layer
path ("The Other Half of the Memory Wall", jaehun.me review, §3.1 staged /
whole-layer bullets).

Every array is drawn from ``numpy.random.default_rng(SeedSequence([seed,
*path]))`` so that each tensor of each layer has its own reproducible stream
and big banks can be drawn on several threads.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

GROUP = 64

# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class LayerShape:
    H: int
    I: int
    E: int
    K: int
    route: str = "softmax_topk"     # or "sigmoid_group"
    n_groups: int = 1
    topk_groups: int = 1
    route_scale: float = 1.0


@dataclass(frozen=True)
class StackShape:
    layer: LayerShape
    n_layers: int
    owners: tuple                    # layers that own a prerouter head
    head_hidden: int = 512
    shared_expert: bool = False
    lora_rank: int = 16
    lora_alpha: float = 32.0
    router_std: float = 0.02
    n_tokens: int = 256
    seed: int = 0

    @property
    def consumers(self) -> tuple:
        return tuple(o + 1 for o in self.owners)


TINY = LayerShape(H=256, I=128, E=16, K=4)
L35B = LayerShape(H=2048, I=512, E=256, K=4)
L8B = LayerShape(H=1536, I=384, E=128, K=8, route="sigmoid_group",
                 n_groups=8, topk_groups=4, route_scale=2.5)

# 35B tier: 40 layers, heads owned by layers 6..38, consumed by 7..39.
STACK35B = StackShape(layer=L35B, n_layers=40, owners=tuple(range(6, 39)),
                      shared_expert=True, router_std=0.02, seed=2)
# 8B tier: 24 layers, heads owned by 7..22, consumed by 8..23; no shared
# expert on this workload; router weights scaled so logits are ~N(0,1).
STACK8B = StackShape(layer=L8B, n_layers=24, owners=tuple(range(7, 23)),
                     shared_expert=False, router_std=1.0 / np.sqrt(1536.0),
                     seed=3)

# Zipf exponent of the prefill load skew and the logit-bias strength that
# realises it with softmax-top-4 over 256 experts.  The strength was fixed
# once by oracle/calibrate_zipf.py; tests check the realised slope.
ZIPF_EXPONENT = 1.1
ZIPF_BETA = 0.365


def _rng(seed: int, *path: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(p) for p in path]))


# --------------------------------------------------------------------------
# Q-tensors and experts
# --------------------------------------------------------------------------

_T_GATE, _T_UP, _T_DOWN = 0, 1, 2
_T_CODES, _T_SCALE, _T_BIAS = 0, 1, 2


def qtensor(g: np.random.Generator, out: int, inn: int, lead: tuple = ()) -> Dict[str, np.ndarray]:
    """One (or a stack of) canonical int4 Q-tensor(s).

    q ~ U{0..15} per element (so every code byte is uniform on 0..255),
    scale = |N(0, 0.02)| / 8, bias = -8*scale + N(0, 1e-3), both stored as fp16.
    """
    assert inn % GROUP == 0
    codes = g.integers(0, 256, size=lead + (out, inn // 2), dtype=np.uint8)
    ng = inn // GROUP
    s32 = np.abs(g.standard_normal(size=lead + (out, ng), dtype=np.float32)) * np.float32(0.02 / 8.0)
    scale = s32.astype(np.float16)
    noise = g.standard_normal(size=lead + (out, ng), dtype=np.float32) * np.float32(1e-3)
    bias = (np.float32(-8.0) * scale.astype(np.float32) + noise).astype(np.float16)
    return {"codes": codes, "scale": scale, "bias": bias}


def expert_bank(seed: int, layer: int, shape: LayerShape, n_experts: Optional[int] = None,
                threads: int = 0, tag: int = 1) -> Dict[str, Dict[str, np.ndarray]]:
    """Stacked per-layer bank: {'gate','up','down'} -> Q-tensor with a leading expert axis."""
    E = shape.E if n_experts is None else n_experts
    H, I = shape.H, shape.I
    jobs = {
        "gate": (_T_GATE, I, H),
        "up": (_T_UP, I, H),
        "down": (_T_DOWN, H, I),
    }

    def make(name):
        tid, out, inn = jobs[name]
        return name, qtensor(_rng(seed, tag, layer, tid), out, inn, lead=(E,))

    if threads and threads > 1:
        with _cf.ThreadPoolExecutor(min(threads, 3)) as ex:
            return dict(ex.map(make, list(jobs)))
    return dict(make(n) for n in jobs)


def expert_view(bank: Dict[str, Dict[str, np.ndarray]], e: int) -> Dict[str, Dict[str, np.ndarray]]:
    """The three Q-tensors of expert ``e`` of a stacked bank (views, no copy)."""
    return {p: {k: v[e] for k, v in bank[p].items()} for p in ("gate", "up", "down")}


def fp16_normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float16)


def router(seed: int, layer: int, shape: LayerShape, std: float = 0.02) -> np.ndarray:
    """Router weight W_r [E, H] fp16 ~ N(0, std)."""
    return fp16_normal(_rng(seed, 2, layer), (shape.E, shape.H), std)


def prerouter_head(seed: int, layer: int, shape: LayerShape, next_router: np.ndarray,
                   hidden: int = 512, std: float = 0.02) -> Dict[str, np.ndarray]:
    """A prerouter head owned by ``layer``: fc1 [hid, H+2E], b1 [hid], fc2 [E, hid],
    b2 [E] (fp16, biases zero) and the linear residual Lres [E, H+2E] laid out as
    [next layer's router | 0 | 0] (the warm start)."""
    H, E = shape.H, shape.E
    g = _rng(seed, 3, layer)
    fc1 = fp16_normal(g, (hidden, H + 2 * E), std)
    fc2 = fp16_normal(g, (E, hidden), std)
    lres = np.zeros((E, H + 2 * E), np.float16)
    lres[:, :H] = next_router
    return {"fc1": fc1, "b1": np.zeros(hidden, np.float16), "fc2": fc2,
            "b2": np.zeros(E, np.float16), "lres": lres}


def shared_expert(seed: int, layer: int, shape: LayerShape, rank: int = 16,
                  alpha: float = 32.0) -> Dict[str, object]:
    """Shared expert (int4 like the routed ones) with an unmerged LoRA on each
    projection: A ~ N(0, 0.01) [r, in], B ~ N(0, 0.0125) [out, r], fp16."""
    H, I = shape.H, shape.I
    q = expert_bank(seed, layer, shape, n_experts=1, tag=9)
    g = _rng(seed, 4, layer)
    lora = {}
    for p, (out, inn) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
        lora[p] = {"A": fp16_normal(g, (rank, inn), 0.01), "B": fp16_normal(g, (out, rank), 0.0125)}
    return {"q": expert_view(q, 0), "lora": lora, "rank": rank, "alpha": alpha}


def normal_rows(seed: int, T: int, H: int, tag: int = 5) -> np.ndarray:
    """x ~ N(0, 1), fp32 [T, H]."""
    return _rng(seed, tag).standard_normal(size=(T, H), dtype=np.float32)


def ar1_tokens(seed: int, T: int, H: int, rho: float = 0.8) -> np.ndarray:
    """x_0 = eps_0, x_t = rho*x_{t-1} + sqrt(1-rho^2)*eps_t, eps ~ N(0, I); fp32 [T, H].
    With rho = 0.8 the innovation weight is 0.6 and every x_t has unit variance."""
    g = _rng(seed, 6)
    eps = g.standard_normal(size=(T, H), dtype=np.float64)
    x = np.empty((T, H), np.float64)
    x[0] = eps[0]
    c = np.sqrt(1.0 - rho * rho)
    for t in range(1, T):
        x[t] = rho * x[t - 1] + c * eps[t]
    return x.astype(np.float32)


def random_topk_sets(seed: int, T: int, E: int, K: int, tag: int = 7) -> np.ndarray:
    """T rows of K distinct expert ids (a stand-in for a previous token's routing)."""
    g = _rng(seed, tag)
    return np.stack([g.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32)


def zipf_logit_bias(seed: int, E: int, exponent: float = ZIPF_EXPONENT,
                    beta: float = ZIPF_BETA) -> np.ndarray:
    """Per-expert additive logit skew b_e = beta * ln p_{pi(e)}, p_r ∝ r^-exponent,
    pi a seeded permutation of the ranks; fp32 [E]."""
    g = _rng(seed, 8)
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-exponent)
    p /= p.sum()
    perm = g.permutation(E)
    return (beta * np.log(p[perm])).astype(np.float32)


# --------------------------------------------------------------------------
# whole workloads
# --------------------------------------------------------------------------


def tiny_layer(seed: int = 0, T: int = 8) -> dict:
    """Tiny MoE layer: H=256, I=128, E=16, K=4, T=8; x ~ N(0,1) (the consumer
    RMS-normalises it); router W_r ~ N(0, 0.02)."""
    s = TINY
    return {"shape": s, "bank": expert_bank(seed, 0, s), "router": router(seed, 0, s),
            "x": normal_rows(seed, T, s.H)}


def layer35b(seed: int = 1, T: int = 1) -> dict:
    """35B-tier single decode layer with its prerouter head (predicting the next
    layer) and a previous-token routing for the head's second one-hot."""
    s = L35B
    bank = expert_bank(seed, 0, s, threads=3)
    w_r = router(seed, 0, s)
    w_next = router(seed, 1, s)
    head = prerouter_head(seed, 0, s, w_next)
    return {"shape": s, "bank": bank, "router": w_r, "router_next": w_next, "head": head,
            "x": normal_rows(seed, T, s.H), "inds_prev": random_topk_sets(seed, T, s.E, s.K)}


@dataclass
class StackModel:
    shape: StackShape
    banks: List[Dict[str, Dict[str, np.ndarray]]] = field(default_factory=list)
    routers: List[np.ndarray] = field(default_factory=list)
    heads: Dict[int, Dict[str, np.ndarray]] = field(default_factory=dict)
    shared: List[Optional[dict]] = field(default_factory=list)
    x: Optional[np.ndarray] = None


def stack_model(shape: StackShape, n_layers: Optional[int] = None, n_tokens: Optional[int] = None,
                threads: int = 0) -> StackModel:
    """Every weight of a decode stack plus its AR(1) token stream."""
    L = shape.n_layers if n_layers is None else n_layers
    T = shape.n_tokens if n_tokens is None else n_tokens
    s, seed = shape.layer, shape.seed
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(threads) as ex:
        banks = list(ex.map(lambda l: expert_bank(seed, l, s), range(L)))
    routers = [router(seed, l, s, shape.router_std) for l in range(L)]
    heads = {}
    for o in shape.owners:
        if o + 1 < L:
            heads[o] = prerouter_head(seed, o, s, routers[o + 1], hidden=shape.head_hidden)
    shared = [shared_expert(seed, l, s, shape.lora_rank, shape.lora_alpha) if shape.shared_expert else None
              for l in range(L)]
    return StackModel(shape=shape, banks=banks, routers=routers, heads=heads, shared=shared,
                      x=ar1_tokens(seed, T, s.H))


def prefill35b(seed: int = 4, T: int = 4096) -> dict:
    """35B-tier whole-layer prefill: X fp16 [T, H] ~ N(0,1), router N(0, 0.02)
    plus a Zipf(1.1) logit skew."""
    s = L35B
    return {"shape": s, "bank": expert_bank(seed, 0, s, threads=3), "router": router(seed, 0, s),
            "logit_bias": zipf_logit_bias(seed, s.E),
            "X": normal_rows(seed, T, s.H).astype(np.float16)}


def prefill8b(seed: int = 5, T: int = 4096) -> dict:
    """8B-tier whole-layer prefill: X fp16 [T, H] ~ N(0,1), router N(0, 1/sqrt(H))
    so the logits are ~N(0,1), sigmoid-group routing (n=8, G=4, s=2.5, K=8),
    no logit skew."""
    s = L8B
    return {"shape": s, "bank": expert_bank(seed, 0, s, threads=3),
            "router": router(seed, 0, s, std=1.0 / np.sqrt(s.H)),
            "X": normal_rows(seed, T, s.H).astype(np.float16)}


def expert_nbytes(shape: LayerShape) -> int:
    """Bytes of one expert in the canonical format (codes + fp16 scale + fp16 bias)."""
    H, I = shape.H, shape.I
    codes = 3 * H * I // 2
    groups = 2 * I * (H // GROUP) + H * (I // GROUP)
    return codes + groups * 2 * 2

"""CPU oracle for the int4 gathered-expert MoE block of Edge0.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
definition that the CUDA library is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product path never does and has no CPU fallback.  It shares no
code with ``int4_gathered_expert_gb300`` and imports nothing from it: callers
hand it numpy arrays in the canonical formats (see the ``synth`` module's
docstring for the layout of a Q-tensor).

Numerics: every floating-point step runs in float64.  Weights are dequantised
exactly (an fp16 scale times a 4-bit code plus an fp16 bias is exact in
float64), dot products accumulate in float64, softmax subtracts the row
maximum, GELU uses erf.  Top-k is a full stable sort on the scores: descending
score, ties to the lower expert index.

Sources (page title and section of each passage followed):
  [KOALA]   "Edge0: 35B MoE를 SSD에서 3GiB 메모리로 서빙하기 — 라우팅을 한
            토큰 먼저 예측한다" (koala.ai.kr): §1 "SSD 스트리밍 전문가 레이어",
            §2 "Prerouter", §3 "Recovery LoRA", table "두 공개 티어".
  [PTKR]    "edge0: 35B MoE 모델을 활성 메모리 3GiB로 실행하는 SSD 전문가
            스트리밍 추론 프레임워크" (discuss.pytorch.kr): "SSD 전문가 스트리밍",
            "라우팅을 한 스텝 먼저 예측하는 프리라우터".
  [JAEHUN]  "The Other Half of the Memory Wall: Serving 35B MoEs from SSD with
            Trained Routing Prediction" (jaehun.me review): "새로운 접근법: Edge0"
            (paper §3.1 math contract, Appx.A routing math), "작동 원리: 구체적인
            예시로 살펴보기" (paper §3.2 toy head), release tiers (paper Tab.1).
  [XYZNOT]  same title (xyznot.com summary): "Methode" — "Architektur des
            Prerouter-Heads" (head equation), "Ausführung des
            unzusammengeführten Adapters" (LoRA equation).

Readings where the pages are silent (each is listed in the design notes):
  * dequantisation is w = scale*q + bias with q the unsigned 4-bit code;
  * RMSNorm (the "post-attention norm" the heads read) is r/sqrt(mean(r^2)+1e-6)
    with no learned weight;
  * the head's one-hot vectors hold 1.0 at each of the K routed experts;
  * sigmoid-group: groups are contiguous blocks of E/n experts, the group score
    is the sum of the group's two largest sigmoids, group ties go to the lower
    group, experts of dropped groups cannot be chosen, no score-correction bias;
  * the decode stack is r_0 = x_t; per layer h = RMSNorm(r), r += MoE(h) +
    Shared(h); layers without a prediction (t = 0, or not a consumer) route
    with their own router.

Every function here is pinned by tests/test_oracle_pins.py against closed
forms, brute force or invariants; none is marked "parity unpinned".
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
from scipy.special import erf as _erf

F64 = np.float64
GROUP = 64

# ---------------------------------------------------------------------------
# affine int4, group 64
# ---------------------------------------------------------------------------


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[..., out, inn/2] uint8 -> [..., out, inn] int64 codes 0..15.

    Element j of a row is the low nibble of byte j/2 when j is even and the
    high nibble when j is odd."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = (codes & 0x0F).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    q = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.int64)
    q[..., 0::2] = lo
    q[..., 1::2] = hi
    return q


def dequant(q: Dict[str, np.ndarray]) -> np.ndarray:
    """w[o, j] = scale[o, j//64] * q[o, j] + bias[o, j//64] in float64.

    [KOALA] §1 and [PTKR] "SSD 전문가 스트리밍": "4-bit affine quantization,
    group size 64"; scale and bias are fp16 (the 1.77 MB per-expert figure of
    [KOALA] §1 only adds up with 2-byte scale and bias)."""
    codes = unpack_codes(q["codes"]).astype(F64)
    inn = codes.shape[-1]
    grp = np.arange(inn) // GROUP
    scale = np.asarray(q["scale"]).astype(F64)[..., grp]
    bias = np.asarray(q["bias"]).astype(F64)[..., grp]
    return scale * codes + bias


# ---------------------------------------------------------------------------
# elementwise pieces
# ---------------------------------------------------------------------------


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    x = np.asarray(x, F64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def sigmoid(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def gelu_erf(x: np.ndarray) -> np.ndarray:
    """Exact (erf) GELU: x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).

    [PTKR] "라우팅을 한 스텝 먼저 예측하는 프리라우터": fc1, then erf-based gelu."""
    x = np.asarray(x, F64)
    return 0.5 * x * (1.0 + _erf(x / np.sqrt(2.0)))


def rmsnorm(r: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """h = r / sqrt(mean(r^2) + eps) over the last axis, no learned weight
    (reading: the pages name the post-attention norm but print no formula)."""
    r = np.asarray(r, F64)
    return r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------------------
# experts
# ---------------------------------------------------------------------------


def linear_q(q: Dict[str, np.ndarray], x: np.ndarray) -> np.ndarray:
    """W_int4 x for x [..., inn] -> [..., out]."""
    W = dequant(q)
    return np.asarray(x, F64) @ W.T


def swiglu_expert(x: np.ndarray, expert: Dict[str, Dict[str, np.ndarray]]) -> np.ndarray:
    """y = down(silu(gate(x)) * up(x)).

    [JAEHUN] "새로운 접근법: Edge0", paper §3.1 math contract: every path
    computes down(silu(gate(x)) · up(x)) with the same kernel."""
    a = silu(linear_q(expert["gate"], x)) * linear_q(expert["up"], x)
    return linear_q(expert["down"], a)


def lora_linear(q: Dict[str, np.ndarray], A: np.ndarray, B: np.ndarray, alpha: float, rank: int,
                x: np.ndarray) -> np.ndarray:
    """Unmerged LoRA projection y = W_int4 x + (alpha/r) B (A x).

    [XYZNOT] "Ausführung des unzusammengeführten Adapters" and [JAEHUN]
    (paper §3.3): the delta runs beside the frozen int4 base, never merged."""
    x = np.asarray(x, F64)
    base = linear_q(q, x)
    ax = x @ np.asarray(A, F64).T
    return base + (alpha / rank) * (ax @ np.asarray(B, F64).T)


def shared_expert(x: np.ndarray, shared: dict) -> np.ndarray:
    """Shared expert with the unmerged LoRA on gate, up and down.

    [KOALA] §4 phase 2 / [JAEHUN] paper §4: the LoRA sits on the shared-expert
    projections, never on the routed experts."""
    q, lo, a, r = shared["q"], shared["lora"], shared["alpha"], shared["rank"]
    if lo is None:
        return swiglu_expert(x, q)
    g = lora_linear(q["gate"], lo["gate"]["A"], lo["gate"]["B"], a, r, x)
    u = lora_linear(q["up"], lo["up"]["A"], lo["up"]["B"], a, r, x)
    return lora_linear(q["down"], lo["down"]["A"], lo["down"]["B"], a, r, silu(g) * u)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------


def _stable_desc(scores: np.ndarray) -> np.ndarray:
    """Indices sorted by descending score; equal scores keep ascending index."""
    return np.argsort(-np.asarray(scores, F64), kind="stable")


def _rel_gap(a: float, b: float) -> float:
    if not np.isfinite(b):
        return np.inf
    return abs(a - b) / max(abs(a), 1e-300)


@dataclass
class Routing:
    inds: np.ndarray        # [T, K] int64, descending score
    w: np.ndarray           # [T, K] float64
    gap: np.ndarray         # [T] relative K-th vs (K+1)-th score gap
    group_gap: np.ndarray   # [T] relative G-th vs (G+1)-th group-score gap (inf if n/a)
    scores: np.ndarray      # [T, E] the scores top-k ran on


def route_softmax_topk(logits: np.ndarray, K: int) -> Routing:
    """g = softmax(l); inds = top-k(g, K); w = g[inds] / sum(g[inds]).

    [JAEHUN] "새로운 접근법: Edge0", paper Appx.A routing math."""
    L = np.atleast_2d(np.asarray(logits, F64))
    T, E = L.shape
    inds = np.empty((T, K), np.int64)
    w = np.empty((T, K), F64)
    gap = np.full(T, np.inf)
    g_all = np.empty_like(L)
    for t in range(T):
        z = L[t] - L[t].max()
        e = np.exp(z)
        g = e / e.sum()
        g_all[t] = g
        order = _stable_desc(g)
        sel = order[:K]
        inds[t] = sel
        w[t] = g[sel] / g[sel].sum()
        if K < E:
            gap[t] = _rel_gap(g[order[K - 1]], g[order[K]])
    return Routing(inds, w, gap, np.full(T, np.inf), g_all)


def route_sigmoid_group(logits: np.ndarray, n_groups: int, topk_groups: int, K: int,
                        s: float) -> Routing:
    """Sigmoid group-limited top-k.

    [JAEHUN] "새로운 접근법: Edge0", paper Appx.A: sigma = sigmoid(l); the top-2
    sum of each group keeps the best G groups; inds = top-k(sigma, K) over the
    kept groups; w = s * sigma[inds] / (sum sigma[inds] + 1e-20).  The 8B tier
    uses n = 8, G = 4, s = 2.5, K = 8 (release tiers, paper Tab.1)."""
    L = np.atleast_2d(np.asarray(logits, F64))
    T, E = L.shape
    assert E % n_groups == 0
    gs = E // n_groups
    inds = np.empty((T, K), np.int64)
    w = np.empty((T, K), F64)
    gap = np.full(T, np.inf)
    ggap = np.full(T, np.inf)
    sig_all = np.empty_like(L)
    for t in range(T):
        sig = sigmoid(L[t])
        sig_all[t] = sig
        gscore = np.empty(n_groups)
        for gi in range(n_groups):
            members = sig[gi * gs:(gi + 1) * gs]
            top = np.sort(members)[::-1][:2]
            gscore[gi] = top.sum()
        gorder = _stable_desc(gscore)
        kept = gorder[:topk_groups]
        if topk_groups < n_groups:
            ggap[t] = _rel_gap(gscore[gorder[topk_groups - 1]], gscore[gorder[topk_groups]])
        masked = np.full(E, -np.inf)
        for gi in kept:
            masked[gi * gs:(gi + 1) * gs] = sig[gi * gs:(gi + 1) * gs]
        order = _stable_desc(masked)
        sel = order[:K]
        inds[t] = sel
        w[t] = s * sig[sel] / (sig[sel].sum() + 1e-20)
        if K < E:
            gap[t] = _rel_gap(masked[order[K - 1]], masked[order[K]])
    return Routing(inds, w, gap, ggap, sig_all)


def route(logits: np.ndarray, shape) -> Routing:
    """Dispatch on a layer shape's routing rule (attributes K, route,
    n_groups, topk_groups, route_scale)."""
    if shape.route == "softmax_topk":
        return route_softmax_topk(logits, shape.K)
    return route_sigmoid_group(logits, shape.n_groups, shape.topk_groups, shape.K, shape.route_scale)


def router_logits(W_r: np.ndarray, h: np.ndarray, logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l = W_r h (+ a per-expert bias when a workload supplies one)."""
    out = np.asarray(h, F64) @ np.asarray(W_r, F64).T
    if logit_bias is not None:
        out = out + np.asarray(logit_bias, F64)
    return out


# ---------------------------------------------------------------------------
# MoE block
# ---------------------------------------------------------------------------


def moe_block(h: np.ndarray, experts, inds: np.ndarray, w: np.ndarray,
              shared: Optional[dict] = None) -> np.ndarray:
    """y[t] = sum_k w[t,k] * expert_{inds[t,k]}(h[t])  (+ shared(h[t])).

    ``experts`` maps an expert id to its three Q-tensors.  [KOALA] §2 (the
    routed set is the predicted set) and [JAEHUN] paper §3.1 / Appx.A."""
    h = np.atleast_2d(np.asarray(h, F64))
    T = h.shape[0]
    out = np.zeros((T, h.shape[1]), F64)
    for t in range(T):
        for k in range(inds.shape[1]):
            out[t] += float(w[t, k]) * swiglu_expert(h[t], experts[int(inds[t, k])])
    if shared is not None:
        out += shared_expert(h, shared)
    return out


class BankExperts:
    """Expert lookup over a stacked per-layer bank (views, nothing copied)."""

    def __init__(self, bank):
        self.bank = bank

    def __getitem__(self, e: int):
        return {p: {k: v[e] for k, v in self.bank[p].items()} for p in ("gate", "up", "down")}


# ---------------------------------------------------------------------------
# prerouter head
# ---------------------------------------------------------------------------


def onehot(inds: Optional[np.ndarray], E: int) -> np.ndarray:
    """1.0 at each of the K routed experts, 0 elsewhere; zeros when ``inds`` is None."""
    v = np.zeros(E, F64)
    if inds is not None:
        v[np.asarray(inds, np.int64)] = 1.0
    return v


def prerouter_features(h: np.ndarray, inds_cur: np.ndarray, inds_prev: Optional[np.ndarray],
                       E: int) -> np.ndarray:
    """f = [h ; onehot(top-K at this token) ; onehot(top-K at the previous token)].

    [KOALA] §2 and [XYZNOT] "Architektur des Prerouter-Heads": dim = d_model + 2E
    (2048 + 2*256 = 2560 for the 35B tier)."""
    return np.concatenate([np.asarray(h, F64), onehot(inds_cur, E), onehot(inds_prev, E)])


def prerouter(h: np.ndarray, inds_cur: np.ndarray, inds_prev: Optional[np.ndarray],
              head: Dict[str, np.ndarray]) -> np.ndarray:
    """head(f) = fc2(gelu_erf(fc1 f + b1)) + b2 + Lres f, for one token.

    [XYZNOT] "Architektur des Prerouter-Heads" head equation; [PTKR] "라우팅을 한
    스텝 먼저 예측하는 프리라우터" (fc1 -> erf gelu -> fc2 plus linear_init);
    [JAEHUN] "작동 원리" toy example (8 + 2*4 = 16 input features)."""
    E = head["fc2"].shape[0]
    f = prerouter_features(h, inds_cur, inds_prev, E)
    fc1 = np.asarray(head["fc1"], F64)
    fc2 = np.asarray(head["fc2"], F64)
    b1 = np.zeros(fc1.shape[0]) if head.get("b1") is None else np.asarray(head["b1"], F64)
    b2 = np.zeros(E) if head.get("b2") is None else np.asarray(head["b2"], F64)
    hid = gelu_erf(fc1 @ f + b1)
    return fc2 @ hid + b2 + np.asarray(head["lres"], F64) @ f


# ---------------------------------------------------------------------------
# slot pool (staged path, incr_stack)
# ---------------------------------------------------------------------------


def slot_update(table: np.ndarray, occupant: np.ndarray, inds_next: np.ndarray,
                inds_cur: np.ndarray) -> Tuple[np.ndarray, np.ndarray, List[Tuple[int, int]]]:
    """In-place replacement of changed slots.

    [KOALA] §1 staged path / [JAEHUN] paper §3.1 and Appx.B (incr_stack): fixed
    slots, a slot table maps expert id -> slot, and only slots whose expert
    changed are overwritten.  Reading: a slot is free when it holds no expert of
    the current or the next set; each missing next expert (in the order given,
    duplicates skipped) takes the lowest free slot.

    Returns (new table [E], new occupant [n_slots], list of (expert, slot) copies)."""
    table = np.array(table, np.int64, copy=True)
    occ = np.array(occupant, np.int64, copy=True)
    nxt = [int(e) for e in np.asarray(inds_next).ravel()]
    cur = [int(e) for e in np.asarray(inds_cur).ravel()] if inds_cur is not None else []
    protected = set()
    for e in nxt + cur:
        if table[e] >= 0:
            protected.add(int(table[e]))
    copies = []
    seen = set()
    for e in nxt:
        if e in seen:
            continue
        seen.add(e)
        if table[e] >= 0:
            continue
        free = [s for s in range(occ.shape[0]) if s not in protected]
        if not free:
            raise ValueError("slot pool too small for the current and next sets")
        s = free[0]
        if occ[s] >= 0:
            table[occ[s]] = -1
        occ[s] = e
        table[e] = s
        protected.add(s)
        copies.append((e, s))
    return table, occ, copies


# ---------------------------------------------------------------------------
# decode stack (prediction-as-routing, double shift)
# ---------------------------------------------------------------------------


@dataclass
class LayerTrace:
    r_in: np.ndarray
    h: np.ndarray
    inds: np.ndarray
    w: np.ndarray
    native: bool
    y: np.ndarray
    head_logits: Optional[np.ndarray]
    pred: Optional[Routing]
    routing: Routing


class StackState:
    """What a decode stream carries from one token to the next: each layer's
    routed set (the head's 'previous token' one-hot) and each consumer layer's
    pending prediction."""

    def __init__(self, n_layers: int):
        self.prev_inds: List[Optional[np.ndarray]] = [None] * n_layers
        self.pred: List[Optional[Tuple[np.ndarray, np.ndarray]]] = [None] * n_layers
        self.t = 0


def stack_layer(l: int, r: np.ndarray, model, shape, state: StackState,
                forced_inds: Optional[np.ndarray] = None,
                forced_w: Optional[np.ndarray] = None) -> LayerTrace:
    """One layer of the decode stack for one token.

    [KOALA] §2 / [PTKR] "프리라우터" / [XYZNOT] "Architektur des Prerouter-Heads":
    the head owned by layer N runs at token t on layer N's MoE input and
    predicts layer N+1's routing at token t+1; layer N+1 consumes that
    prediction one token later through the same routing math (prediction as
    routing).  [JAEHUN] "작동 원리": prefill and the first token do not predict,
    so they route natively.

    ``forced_inds`` / ``forced_w`` replace the routing this layer takes (used by
    teacher-forced checks after the routing itself has been compared)."""
    ls = shape.layer
    h = rmsnorm(r)
    bank = BankExperts(model.banks[l])
    native = state.pred[l] is None
    if native:
        rt = route(router_logits(model.routers[l], h), ls)
        inds, w = rt.inds[0], rt.w[0]
    else:
        rt = None
        inds, w = state.pred[l]
    routing = rt
    if forced_inds is not None:
        inds, w = np.asarray(forced_inds), np.asarray(forced_w, F64)
    sh = model.shared[l] if model.shared else None
    y = moe_block(h, bank, inds[None, :], np.asarray(w, F64)[None, :], sh)[0]
    head_logits = None
    pred = None
    if l in model.heads:
        head_logits = prerouter(h, inds, state.prev_inds[l], model.heads[l])
        pred = route(head_logits, ls)
    return LayerTrace(r_in=r, h=h, inds=np.asarray(inds), w=np.asarray(w, F64), native=native, y=y,
                      head_logits=head_logits, pred=pred, routing=routing)


def stack_commit(l: int, tr: LayerTrace, model, state: StackState) -> None:
    """Record what this layer leaves for the next token."""
    state.prev_inds[l] = tr.inds
    if tr.pred is not None and l + 1 < len(model.banks):
        state.pred[l + 1] = (tr.pred.inds[0], tr.pred.w[0])


def stack_token(x: np.ndarray, model, state: StackState) -> Tuple[np.ndarray, List[LayerTrace]]:
    """Decode one token through every layer: r_0 = x; r_{l+1} = r_l + MoE(h_l) + Shared(h_l).
    Predictions made at this token are only consumed at the next one."""
    shape = model.shape
    r = np.asarray(x, F64)
    traces = []
    pending = []
    for l in range(len(model.banks)):
        tr = stack_layer(l, r, model, shape, state)
        traces.append(tr)
        pending.append(tr)
        r = r + tr.y
    # the next token sees this token's routing and predictions
    for l, tr in enumerate(pending):
        stack_commit(l, tr, model, state)
    state.t += 1
    return r, traces


# ---------------------------------------------------------------------------
# whole-layer prefill (sorted gather)
# ---------------------------------------------------------------------------


def prefill_sort(inds: np.ndarray, E: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Group the T*K (token, k) assignments by expert.

    [PTKR] "SSD 전문가 스트리밍" (full-layer path computes with a sorted gather).
    Returns counts [E], offsets [E+1] (exclusive scan) and perm [T*K]: the
    assignment ids a = t*K + k ordered by expert, token order kept within one
    expert (a stable sort)."""
    flat = np.asarray(inds, np.int64).ravel()
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm = np.argsort(flat, kind="stable")
    return counts, offsets, perm


def prefill(X: np.ndarray, bank, W_r: np.ndarray, shape, logit_bias: Optional[np.ndarray] = None,
            tokens: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, Routing]:
    """Whole-layer prefill: route every token natively, then y_t = sum_k w_k expert(x_t).

    [JAEHUN] "작동 원리": prefill does not predict.  The sort of the sorted
    gather only orders the work, so this definition loops over tokens.
    ``tokens`` restricts the output rows computed (routing is per token)."""
    X = np.asarray(X, F64)
    rows = np.arange(X.shape[0]) if tokens is None else np.asarray(tokens)
    rt = route(router_logits(W_r, X[rows], logit_bias), shape)
    experts = BankExperts(bank)
    Y = moe_block(X[rows], experts, rt.inds, rt.w)
    return Y, rt

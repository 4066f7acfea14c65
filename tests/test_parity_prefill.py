"""GPU parity of the whole-layer prefill (router GEMM, routing, stable sort by
expert, tcgen05 grouped GEMMs, combine) against the CPU oracle."""
import numpy as np
import pytest

from int4_gathered_expert_gb300 import synth
from oracle import e0_oracle as O
from tests.parity import REL_L2, rel_l2, routing_matches, tile_edge_tokens

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_gathered_expert_gb300 import build, lib
    import os
    if not os.path.exists(lib.LIB_PATH):
        build.build()
    lib.load()
    return lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("T,K,E", [(1, 4, 16), (37, 4, 16), (4096, 4, 256), (300, 8, 128), (5, 1, 1024)])
def test_prefill_sort_is_exact(L, T, K, E):
    g = np.random.default_rng(T + K + E)
    inds = np.stack([g.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    if T > 10:
        inds[: T // 3, 0] = 3  # a crowded expert
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
    ws_bytes = L.e0_workspace_size(2, T, 64, 64, E, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    L.e0_prefill_sort(dev(inds), T, K, E, counts, offsets, perm, ws, ws_bytes)
    c, o, p = O.prefill_sort(inds, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(perm.cpu().numpy(), p)


def run_prefill(L, pool, X16, Wr, rp, T):
    s_H = pool.H
    ws_bytes = L.e0_workspace_size(2, T, pool.H, pool.I, pool.E, rp.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    Y = torch.empty((T, s_H), dtype=torch.float32, device="cuda")
    inds = torch.empty((T, rp.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, rp.K), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.e0_moe_prefill_forward(X16, T, pool.desc, Wr, rp, Y, inds, w, ws, ws_bytes, st)
    return Y.cpu().numpy(), inds.cpu().numpy(), w.cpu().numpy(), L.e0_read_status(st)


def test_prefill_many_experts(L):
    """E = 1024 (the largest E the library takes) at the tiny layer width,
    K = 2, T = 700: nearly every expert gets a partial tile, so the tile list
    ranks ~1000 partial tiles, and every token's routing and output is
    checked against the oracle."""
    import dataclasses
    from int4_gathered_expert_gb300.model import SlotPoolDev
    s = dataclasses.replace(synth.TINY, E=1024, K=2)
    T = 700
    bank = synth.expert_bank(11, 0, s)
    W_r = synth.router(11, 0, s)
    X = synth.normal_rows(11, T, s.H).astype(np.float16)
    pool = SlotPoolDev.resident(bank, s.H, s.I)
    Y, inds, w, st = run_prefill(L, pool, dev(X), dev(W_r), L.route_params(K=s.K), T)
    assert st == 0
    Yo, rt = O.prefill(X, bank, W_r, s)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs[:4]
    assert len(np.unique(inds)) > 600
    errs = [rel_l2(Y[t], Yo[t]) for t in range(T) if t not in ex]
    assert max(errs) <= REL_L2, max(errs)


@pytest.mark.parametrize("fixed_order", [False, True])
def test_prefill_repeated_calls_on_changing_buffers(L, fixed_order, monkeypatch):
    """Calls that alternate two input buffers (and a larger token count in
    between) through one workspace: each call matches the oracle (the encoded
    tensor maps are reused only for the buffers they were made for; no state
    leaks between calls).  A repeated call gives the same routing and, with
    E0MOE_PREFILL_FIXED_ORDER=1, the same bits; by default the K weighted
    rows of a token are added with atomics, so the sum may differ in its
    last bits from run to run."""
    monkeypatch.setenv("E0MOE_PREFILL_FIXED_ORDER", "1" if fixed_order else "0")
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d1 = synth.tiny_layer(3, T=200)
    d2 = synth.tiny_layer(4, T=200)
    d3 = synth.tiny_layer(5, T=390)
    s = d1["shape"]
    pool = SlotPoolDev.resident(d1["bank"], s.H, s.I)
    rp = L.route_params(K=s.K)
    ws_bytes = L.e0_workspace_size(2, 390, s.H, s.I, s.E, s.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wr = dev(d1["router"])

    def call(x):
        T = x.shape[0]
        Y = torch.empty((T, s.H), dtype=torch.float32, device="cuda")
        inds = torch.empty((T, s.K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, s.K), dtype=torch.float32, device="cuda")
        L.e0_moe_prefill_forward(dev(x), T, pool.desc, Wr, rp, Y, inds, w, ws, ws_bytes, st)
        return Y.cpu().numpy(), inds.cpu().numpy(), w.cpu().numpy()

    xs = [d["x"].astype(np.float16) for d in (d1, d2, d3)]
    runs = [call(xs[i]) for i in (0, 1, 2, 0, 1)]
    assert L.e0_read_status(st) == 0
    for i, (Y, inds, w) in zip((0, 1, 2, 0, 1), runs):
        Yo, rt = O.prefill(xs[i], d1["bank"], d1["router"], s)
        ex, msgs = routing_matches(inds, w, rt)
        assert not msgs, msgs[:4]
        errs = [rel_l2(Y[t], Yo[t]) for t in range(xs[i].shape[0]) if t not in ex]
        assert max(errs) <= REL_L2, max(errs)
    for a, b in ((runs[0], runs[3]), (runs[1], runs[4])):
        assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
        if fixed_order:
            assert np.array_equal(a[0], b[0])
        else:
            assert np.abs(a[0] - b[0]).max() <= 1e-6 * np.abs(a[0]).max()


@pytest.mark.parametrize("T", [1, 8, 130, 513])
def test_tiny_prefill(L, T):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.tiny_layer(0, T=T)
    s = d["shape"]
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I)
    X = d["x"].astype(np.float16)
    Y, inds, w, st = run_prefill(L, pool, dev(X), dev(d["router"]), L.route_params(K=s.K), T)
    assert st == 0
    Yo, rt = O.prefill(X, d["bank"], d["router"], s)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs[:4]
    errs = [rel_l2(Y[t], Yo[t]) for t in range(T) if t not in ex]
    assert max(errs) <= REL_L2, max(errs)


def test_prefill_one_crowded_expert_set(L):
    """Every token routed to the same 4 experts: each expert gets T rows, so
    the grouped GEMM runs several full N tiles plus a ragged tail."""
    from int4_gathered_expert_gb300.model import SlotPoolDev
    T = 300
    d = synth.tiny_layer(3, T=T)
    s = d["shape"]
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I)
    bias = np.zeros(s.E, np.float32)
    bias[[2, 5, 9, 14]] = 40.0
    X = d["x"].astype(np.float16)
    bias_d = dev(bias)  # the descriptor holds a raw pointer: keep the tensor alive
    rp = L.route_params(K=s.K, logit_bias=bias_d)
    Y, inds, w, st = run_prefill(L, pool, dev(X), dev(d["router"]), rp, T)
    assert st == 0
    assert set(np.unique(inds)) == {2, 5, 9, 14}
    Yo, rt = O.prefill(X, d["bank"], d["router"], s, logit_bias=bias)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs
    assert max(rel_l2(Y[t], Yo[t]) for t in range(T)) <= REL_L2


@pytest.mark.parametrize("mode", ["softmax_topk", "sigmoid_group"])
def test_prefill_planted_near_ties(L, mode):
    """Two router rows that differ in one fp16 ulp of one input: in every token
    their two logits differ by ulp * x_j, a few 1e-6 to 1e-5 at the 35B width,
    the size of the tensor-core logits' own error, so their order rests on the
    exact recomputation of the tokens flagged as near-ties.  Softmax top-k: a
    logit bias lifts both into every token's top K; sigmoid group-limited: the
    two share a group.  Every token whose gap is above the tie rule must route
    as the oracle does, and many such tokens must exist."""
    import dataclasses
    from int4_gathered_expert_gb300.model import SlotPoolDev
    if mode == "softmax_topk":
        s = dataclasses.replace(synth.TINY, H=2048, E=64, K=4)
    else:
        s = dataclasses.replace(synth.TINY, H=2048, E=64, K=8, route="sigmoid_group", n_groups=8, topk_groups=4,
                                route_scale=2.5)
    T = 600
    e0, e1 = 3, 5  # the same group of 8 experts in the sigmoid-group case
    W = synth.router(13, 0, s, std=1.0 / np.sqrt(s.H))
    j = int(np.argmin(np.abs(np.abs(W[e0].astype(np.float32)) - 0.02)))  # fp16 ulp 1.5e-5 there
    W[e1] = W[e0]
    W[e1, j] = np.nextafter(W[e0, j], np.float16(np.inf) if W[e0, j] > 0 else np.float16(-np.inf))
    X = synth.normal_rows(13, T, s.H).astype(np.float16)
    bank = synth.expert_bank(13, 0, s)
    pool = SlotPoolDev.resident(bank, s.H, s.I)
    bias = None
    if mode == "softmax_topk":
        bias = np.zeros(s.E, np.float32)
        bias[[e0, e1]] = 4.0
        bias_d = dev(bias)  # the descriptor holds a raw pointer: keep the tensor alive
        rp = L.route_params(K=s.K, logit_bias=bias_d)
    else:
        rp = L.route_params(mode=L.E0_ROUTE_SIGMOID_GROUP, K=s.K, n_groups=s.n_groups, topk_groups=s.topk_groups,
                            scale=s.route_scale)
    Y, inds, w, st = run_prefill(L, pool, dev(X), dev(W), rp, T)
    assert st == 0
    logits = O.router_logits(W, X, bias)
    rt = O.route(logits, s)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs[:4]
    # tokens where both planted experts were selected, their order decided by
    # a gap below 1e-4 and above the tie rule
    both = [t for t in range(T) if t not in ex and e0 in rt.inds[t] and e1 in rt.inds[t]
            and 0 < abs(logits[t, e0] - logits[t, e1]) < 1e-4]
    assert len(both) >= (300 if mode == "softmax_topk" else 20), len(both)
    sample = sorted(set(both[:12] + [0, T - 1]) - set(ex))
    Yo, _ = O.prefill(X, bank, W, s, logit_bias=bias, tokens=sample)
    assert max(rel_l2(Y[t], Yo[i]) for i, t in enumerate(sample)) <= REL_L2


@pytest.fixture(scope="module")
def prefill35(L):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.prefill35b(4, T=4096)
    s = d["shape"]
    d["pool"] = SlotPoolDev.resident(d["bank"], s.H, s.I)
    return d


def test_35b_prefill_full_size(L, prefill35):
    d = prefill35
    s = d["shape"]
    T = d["X"].shape[0]
    bias_d = dev(d["logit_bias"])
    rp = L.route_params(K=s.K, logit_bias=bias_d)
    Y, inds, w, st = run_prefill(L, d["pool"], dev(d["X"]), dev(d["router"]), rp, T)
    assert st == 0
    # routing of every token against the oracle (exact up to the tie rule)
    logits = O.router_logits(d["router"], d["X"], d["logit_bias"])
    rt = O.route_softmax_topk(logits, s.K)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs[:4]
    # expert load is Zipf-like (the workload's recipe)
    counts = np.bincount(inds.ravel(), minlength=s.E)
    assert counts.sum() == T * s.K and counts.max() > 20 * np.median(counts)
    # outputs on a sample of tokens: the first and the last, random ones, and
    # the tokens at the tile edges of the three busiest experts (several
    # 128-token tiles each)
    g = np.random.default_rng(0)
    edges = tile_edge_tokens(inds)
    sample = sorted(set([0, T - 1] + g.choice(T, 22, replace=False).tolist() + edges) - set(ex))
    Yo = O.moe_block(d["X"][sample].astype(np.float64), O.BankExperts(d["bank"]), rt.inds[sample], rt.w[sample])
    errs = [rel_l2(Y[t], Yo[i]) for i, t in enumerate(sample)]
    assert max(errs) <= REL_L2, max(errs)


@pytest.fixture(scope="module")
def prefill8(L):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.prefill8b(5, T=3100)
    s = d["shape"]
    d["pool"] = SlotPoolDev.resident(d["bank"], s.H, s.I)
    return d


def test_8b_prefill_sigmoid_group(L, prefill8):
    """The 8B-tier layer (H=1536, I=384, E=128) through the same sorted grouped
    GEMMs, with sigmoid-group routing (n=8, keep 4 groups, K=8, s=2.5) over a
    3.1k-token prompt: every token's routing against the oracle (exact up to
    the tie rule) and outputs on a sample of tokens."""
    d = prefill8
    s = d["shape"]
    T = d["X"].shape[0]
    rp = L.route_params(mode=L.E0_ROUTE_SIGMOID_GROUP, K=s.K, n_groups=s.n_groups, topk_groups=s.topk_groups,
                        scale=s.route_scale)
    Y, inds, w, st = run_prefill(L, d["pool"], dev(d["X"]), dev(d["router"]), rp, T)
    assert st == 0
    logits = O.router_logits(d["router"], d["X"])
    rt = O.route(logits, s)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs[:4]
    counts = np.bincount(inds.ravel(), minlength=s.E)
    assert counts.sum() == T * s.K
    g = np.random.default_rng(1)
    sample = sorted(set([0, T - 1] + g.choice(T, 22, replace=False).tolist() + tile_edge_tokens(inds)) - set(ex))
    Yo = O.moe_block(d["X"][sample].astype(np.float64), O.BankExperts(d["bank"]), rt.inds[sample], rt.w[sample])
    errs = [rel_l2(Y[t], Yo[i]) for i, t in enumerate(sample)]
    assert max(errs) <= REL_L2, max(errs)

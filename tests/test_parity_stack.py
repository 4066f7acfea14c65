"""Decode-stack parity (35B tier: 40 layers, heads owned by 6..38; 8B tier: 24
layers, sigmoid-group routing, heads owned by 7..22) against the CPU oracle,
teacher-forced layer by layer: the oracle recomputes every checked layer from
the GPU's residual stream and the GPU's routing, after checking that routing
itself (native router or the head prediction made one token earlier).

Routing must equal the oracle's exactly, except where the oracle's K-th and
(K+1)-th scores (or G-th and (G+1)-th group scores) are closer than 1e-6
relative; per-layer outputs must be within rel-L2 2e-3 of the oracle's."""
import dataclasses

import numpy as np
import pytest

from int4_gathered_expert_gb300 import synth
from oracle import e0_oracle as O
from tests.parity import REL_L2, rel_l2, routing_matches

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_TOK = 6
CHECK = (0, 1, 2, 5)
LL = 3  # the flag-carrying-word kernel (one launch per token)


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


def snapshot(sd):
    return {k: v.cpu().numpy().copy() for k, v in sd.tr.items()}


def run_stack(sd, m, n_tok, impl, traced=None):
    """Decode n_tok tokens; returns the trace of every token (or of the tokens
    in `traced`, None elsewhere)."""
    sd.prepare()
    traces = []
    full = sd.trace
    for t in range(n_tok):
        keep = traced is None or t in traced
        sd.trace = full if keep else None
        sd.step(torch.from_numpy(m.x[t]).cuda(), impl=impl)
        traces.append(snapshot(sd) if keep else None)
    sd.trace = full
    return traces


def check_stack(m, traces, check, L_check=None):
    shape = m.shape
    ls = shape.layer
    nL = len(m.banks)
    worst = 0.0
    n_exempt = 0
    for t in check:
        tr = traces[t]
        prev = traces[t - 1] if t > 0 else None
        for l in (range(nL) if L_check is None else L_check):
            r_in = tr["r"][l].astype(np.float64)
            h = O.rmsnorm(r_in)
            inds = tr["inds"][l]
            w = tr["w"][l]
            consumer = t > 0 and l in shape.consumers and (l - 1) in m.heads
            if consumer:
                # prediction as routing: exactly what the owner predicted one token earlier
                assert np.array_equal(inds, prev["pred_inds"][l]), (t, l)
            else:
                rt = O.route(O.router_logits(m.routers[l], h[None]), ls)
                ex, msgs = routing_matches(inds[None], w[None], rt)
                assert not msgs, (t, l, msgs)
                n_exempt += len(ex)
            y_gpu = tr["r"][l + 1].astype(np.float64) - r_in
            sh = m.shared[l] if m.shared else None
            y_or = O.moe_block(h[None], O.BankExperts(m.banks[l]), inds[None].astype(np.int64),
                               w[None].astype(np.float64), sh)[0]
            e = rel_l2(y_gpu, y_or)
            worst = max(worst, e)
            assert e <= REL_L2, (t, l, e)
            if l in m.heads:
                p_inds = prev["inds"][l] if prev is not None else None
                z = O.prerouter(h, inds, p_inds, m.heads[l])
                assert rel_l2(tr["head_logits"][l], z) < 1e-5, (t, l)
                if l + 1 < nL:
                    # the predicted routing: indices and weights as the oracle
                    # routes the head logits, exempt only at ties
                    rt = O.route(z[None], ls)
                    ex, msgs = routing_matches(tr["pred_inds"][l + 1][None],
                                               _pred_w(traces, t, l + 1, ls.K), rt)
                    assert not msgs, (t, l, msgs)
                    n_exempt += len(ex)
    return worst, n_exempt


def _pred_w(traces, t, l, K):
    """The weights of a prediction are what the consumer uses at the next token
    (the trace records the weights each layer used); without a next-token
    trace, the weight check is skipped (the indices are still compared)."""
    nxt = traces[t + 1] if t + 1 < len(traces) else None
    if nxt is not None and np.array_equal(nxt["inds"][l], traces[t]["pred_inds"][l]):
        return nxt["w"][l][None]
    return None


@pytest.fixture(scope="module")
def stack35(L):
    from int4_gathered_expert_gb300.model import StackDev
    m = synth.stack_model(synth.STACK35B, n_tokens=256)
    sd = StackDev(m, trace=True)
    yield m, sd
    del sd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("impl", [0, LL])
def test_35b_stack_teacher_forced(L, stack35, impl):
    m, sd = stack35
    traces = run_stack(sd, m, N_TOK, impl=impl)
    assert L.e0_read_status(sd.status) == 0
    worst, n_ex = check_stack(m, traces, CHECK)
    print("35B stack impl", impl, "worst per-layer rel-L2", worst, "tie-exempt", n_ex)


def test_35b_stack_late_token(L, stack35):
    """Token 255 of the 256-token AR(1) stream (experts recur): the state the
    kernel carries from token to token (routing history, predictions, flag
    epochs) still gives oracle results late in the stream."""
    m, sd = stack35
    traces = run_stack(sd, m, 256, impl=LL, traced={253, 254, 255})
    assert L.e0_read_status(sd.status) == 0
    worst, n_ex = check_stack(m, traces, (254, 255))
    print("35B stack token 255: worst per-layer rel-L2", worst, "tie-exempt", n_ex)


def test_35b_ll_kernel_agrees_with_persistent(L, stack35):
    """Both kernels are deterministic; their sums are taken in different orders,
    so the residual streams agree to rounding and the routing exactly (a routing
    difference would have to be a tie, which the oracle check above exempts)."""
    m, sd = stack35
    a = run_stack(sd, m, 4, impl=0)
    b = run_stack(sd, m, 4, impl=LL)
    for t in range(4):
        assert rel_l2(b[t]["r"], a[t]["r"]) < 1e-4, t
        assert np.array_equal(a[t]["inds"], b[t]["inds"]), t
        assert np.array_equal(a[t]["pred_inds"], b[t]["pred_inds"]), t


def test_35b_ll_kernel_is_deterministic(L, stack35):
    m, sd = stack35
    a = run_stack(sd, m, 3, impl=LL)
    b = run_stack(sd, m, 3, impl=LL)
    for t in range(3):
        for k in ("r", "inds", "w", "head_logits", "pred_inds"):
            assert np.array_equal(a[t][k], b[t][k]), (t, k)


def test_35b_stack_chain_equals_persistent(L, stack35):
    m, sd = stack35
    a = run_stack(sd, m, 3, impl=0)
    b = run_stack(sd, m, 3, impl=1)
    for t in range(3):
        for k in ("r", "inds", "pred_inds"):
            assert np.array_equal(a[t][k], b[t][k]), (t, k)
    check_stack(m, b, (1, 2), L_check=range(0, 40, 7))


@pytest.fixture(scope="module")
def stack8(L):
    from int4_gathered_expert_gb300.model import StackDev
    m = synth.stack_model(synth.STACK8B, n_tokens=N_TOK)
    sd = StackDev(m, trace=True)
    yield m, sd
    del sd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("impl", [0, LL])
def test_8b_stack_teacher_forced(L, stack8, impl):
    m, sd = stack8
    traces = run_stack(sd, m, N_TOK, impl=impl)
    assert L.e0_read_status(sd.status) == 0
    worst, n_ex = check_stack(m, traces, CHECK)
    print("8B stack impl", impl, "worst per-layer rel-L2", worst, "tie-exempt", n_ex)


def test_tiny_stack_ll_kernel(L):
    """A 5-layer tiny stack (H=256, E=16: eight rows a warp) through the kernel."""
    from int4_gathered_expert_gb300.model import StackDev
    shape = synth.StackShape(layer=synth.TINY, n_layers=5, owners=(1, 2, 3), shared_expert=True, seed=13)
    m = synth.stack_model(shape, n_tokens=4, threads=2)
    sd = StackDev(m, trace=True)
    traces = run_stack(sd, m, 4, impl=LL)
    assert L.e0_read_status(sd.status) == 0
    check_stack(m, traces, (0, 1, 2, 3))


@pytest.mark.parametrize("K,prerouter", [(2, True), (8, True), (4, False)])
def test_35b_shape_route_k_and_prerouter_variants(L, K, prerouter):
    """The K / prerouter arms of the harness (softmax-top-K on the 35B layer
    shape, 8 layers): K = 2 and K = 8 with heads owned by 2..6, and K = 4 with
    no heads (every layer routes with its own router)."""
    from int4_gathered_expert_gb300.model import StackDev
    shape = dataclasses.replace(synth.STACK35B, layer=dataclasses.replace(synth.L35B, K=K), n_layers=8,
                                owners=tuple(range(2, 7)) if prerouter else (), seed=40 + K)
    m = synth.stack_model(shape, n_tokens=4)
    sd = StackDev(m, trace=True)
    traces = run_stack(sd, m, 4, impl=LL)
    assert L.e0_read_status(sd.status) == 0
    worst, n_ex = check_stack(m, traces, (0, 1, 2, 3))
    print("K", K, "prerouter", prerouter, "worst", worst, "tie-exempt", n_ex)
    del sd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("K,prerouter", [(2, True), (4, False)])
def test_stack_variant_equals_fresh_stack(L, K, prerouter):
    """StackDev.variant (the same device weights with another K, or without
    heads) gives the bits of a stack built from scratch with that shape."""
    from int4_gathered_expert_gb300.model import StackDev
    base = dataclasses.replace(synth.STACK35B, n_layers=6, owners=tuple(range(1, 5)), seed=50)
    m = synth.stack_model(base, n_tokens=4)
    sd = StackDev(m)
    v = sd.variant(K=K, prerouter=prerouter)
    shape = dataclasses.replace(base, layer=dataclasses.replace(synth.L35B, K=K),
                                owners=base.owners if prerouter else ())
    m2 = synth.stack_model(shape, n_tokens=4)
    fresh = StackDev(m2)
    X = torch.from_numpy(m.x).cuda()
    for t in range(4):
        a = v.step(X[t], impl=LL).cpu().numpy()
        b = fresh.step(X[t], impl=LL).cpu().numpy()
        assert np.array_equal(a, b), t
    assert L.e0_read_status(v.status) == 0 and L.e0_read_status(fresh.status) == 0
    del sd, v, fresh
    torch.cuda.empty_cache()


def test_stack_range_launches_equal_one_launch(L, stack35):
    """A token split into two launches at any layer gives the same bits as one."""
    m, sd = stack35
    from int4_gathered_expert_gb300 import lib
    a = run_stack(sd, m, 3, impl=LL)
    sd.prepare()
    for t in range(3):
        x = torch.from_numpy(m.x[t]).cuda()
        split = (7, 22, 39)[t]
        lib.e0_stack_step_range(x, None, sd.ws, 0, split, sd.trace, sd.status)
        lib.e0_stack_step_range(None, sd.r_out, sd.ws, split, sd.L, sd.trace, sd.status)
        b = snapshot(sd)
        for k in ("r", "inds", "w", "head_logits", "pred_inds"):
            assert np.array_equal(a[t][k], b[k]), (t, k)
    assert L.e0_read_status(sd.status) == 0


def _run_streamed(ss, sd, X, n_tok, overlap=True):
    got = []
    ss.start(X[0])
    torch.cuda.synchronize()
    got.append(snapshot(sd))
    for t in range(1, n_tok):
        ss.step(X[t], overlap=overlap)
        torch.cuda.synchronize()
        got.append(snapshot(sd))
    return got


def _tiny_stream_model():
    shape = synth.StackShape(layer=synth.TINY, n_layers=8, owners=(1, 2, 3, 4, 5, 6), shared_expert=True, seed=21)
    return synth.stack_model(shape, n_tokens=6, threads=2)


@pytest.mark.parametrize("overlap", [True, False])
def test_streamed_stack_matches_oracle(L, overlap):
    """Host-tier staged streaming: the consumer layers hold 2K slots filled from
    pinned host memory with the experts the prerouter predicted one token
    earlier, copied on a second stream while the other half of the token runs.
    Every token is teacher-forced against the oracle, with no slot miss."""
    from int4_gathered_expert_gb300.model import StackDev, StreamedStack
    m = _tiny_stream_model()
    sd = StackDev(m, trace=True)
    ss = StreamedStack(sd, split=5)
    assert ss.batch1 == [2, 3] and ss.batch2 == [5, 6, 7]
    got = _run_streamed(ss, sd, torch.from_numpy(m.x).cuda(), 6, overlap)
    assert L.e0_read_status(sd.status) == 0
    check_stack(m, got, range(6))
    # the staged layers really run from their slot pools: each holds at most 2K experts
    for l in ss.staged:
        tab = ss.pools[l].table.cpu().numpy()
        assert 0 < (tab >= 0).sum() <= 2 * m.shape.layer.K


@pytest.mark.parametrize("capacity", [0, 3])
def test_streamed_stack_per_layer_prefetch_equals_batched(L, capacity):
    """The per-layer prefetch calls (plain, and through a small cache that
    evicts) fill the slots exactly as the batched calls do: the decode of
    every token gives the same bits."""
    from int4_gathered_expert_gb300.model import ExpertCacheDev, StackDev, StreamedStack
    m = _tiny_stream_model()
    X = torch.from_numpy(m.x).cuda()
    runs = []
    for batched in (True, False):
        sd = StackDev(m, trace=True)
        cache = ExpertCacheDev(capacity, sd.L, sd.H, sd.I, sd.E) if capacity else None
        ss = StreamedStack(sd, split=5, cache=cache, batched=batched)
        ss.start(X[0])
        got = [snapshot(sd)]
        for t in range(1, 6):
            ss.step(X[t])
            torch.cuda.synchronize()
            got.append(snapshot(sd))
        assert L.e0_read_status(sd.status) == 0
        runs.append(got)
        del ss, sd, cache
    for t in range(6):
        for k in ("r", "inds", "w", "pred_inds"):
            assert np.array_equal(runs[0][t][k], runs[1][t][k]), (t, k)


@pytest.mark.parametrize("capacity", [3, 64])
def test_streamed_stack_with_expert_cache(L, capacity):
    """Staged streaming with a cross-layer LRU cache of expert bundles in front
    of the host bank: oracle results token by token, and the counters add up
    (every copy is a hit or a miss; a cache smaller than the working set evicts)."""
    from int4_gathered_expert_gb300.model import ExpertCacheDev, StackDev, StreamedStack
    m = _tiny_stream_model()
    sd = StackDev(m, trace=True)
    cache = ExpertCacheDev(capacity, sd.L, sd.H, sd.I, sd.E)
    ss = StreamedStack(sd, split=5, cache=cache)
    X = torch.from_numpy(m.x).cuda()
    copies = 0
    ss.start(X[0])
    got = [snapshot(sd)]
    occ = {l: ss.pools[l].occupant.cpu().numpy().copy() for l in ss.staged}
    copies += sum(int((o >= 0).sum()) for o in occ.values())
    for t in range(1, 6):
        ss.step(X[t])
        torch.cuda.synchronize()
        got.append(snapshot(sd))
        for l in ss.staged:
            now = ss.pools[l].occupant.cpu().numpy()
            copies += int((now != occ[l]).sum())
            occ[l] = now.copy()
    assert L.e0_read_status(sd.status) == 0
    check_stack(m, got, range(6))
    st = cache.stats()
    assert st["hits"] + st["misses"] == copies
    if capacity < 5 * 4:
        assert st["evictions"] > 0


@pytest.mark.parametrize("cache_capacity", [0, 64])
def test_streamed_stack_35b_shape_matches_oracle(L, cache_capacity):
    """Staged streaming (and with a 64-bundle LRU in front of the host bank) on
    the 35B layer shape: 12 layers, heads owned by 2..10, two launches a token
    split at layer 6, 2K = 8 slots per staged layer; teacher-forced against the
    oracle on every token."""
    from int4_gathered_expert_gb300.model import ExpertCacheDev, StackDev, StreamedStack
    shape = dataclasses.replace(synth.STACK35B, n_layers=12, owners=tuple(range(2, 11)), seed=31)
    m = synth.stack_model(shape, n_tokens=5)
    sd = StackDev(m, trace=True)
    cache = ExpertCacheDev(cache_capacity, sd.L, sd.H, sd.I, sd.E) if cache_capacity else None
    ss = StreamedStack(sd, split=6, cache=cache)
    assert ss.batch1 == [3, 4] and ss.batch2 == [6, 7, 8, 9, 10, 11]
    got = _run_streamed(ss, sd, torch.from_numpy(m.x).cuda(), 5)
    assert L.e0_read_status(sd.status) == 0
    worst, n_ex = check_stack(m, got, range(5))
    print("35B-shape streaming, cache", cache_capacity, "worst", worst, "tie-exempt", n_ex)
    del ss, sd
    torch.cuda.empty_cache()

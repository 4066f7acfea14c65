"""GPU parity of the decode entry points against the CPU oracle: routing,
RMSNorm, the MoE block (tiny and 35B-tier layer, resident and staged slot
pools, native and predicted routing), the prerouter head, slot_update and the
device status word."""
import numpy as np
import pytest

from int4_gathered_expert_gb300 import synth
from oracle import e0_oracle as O
from tests.parity import REL_L2, rel_l2, routing_matches

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


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------ routing


@pytest.mark.parametrize("T,E,K", [(1, 16, 4), (37, 256, 4), (64, 128, 8), (5, 8, 8), (3, 1024, 32), (9, 33, 3)])
def test_softmax_topk(L, T, E, K):
    g = np.random.default_rng(E * 100 + K)
    logits = g.standard_normal((T, E)).astype(np.float32)
    logits[0, :4] = logits[0, 5]  # exact ties: lower index first
    inds = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    st = status_word()
    L.e0_route_softmax_topk(dev(logits), T, E, K, inds, w, st)
    rt = O.route_softmax_topk(logits.astype(np.float64), K)
    ex, msgs = routing_matches(inds.cpu().numpy(), w.cpu().numpy(), rt, allow_tie=False)
    assert not msgs, msgs[:5]
    assert L.e0_read_status(st) == 0


def test_softmax_topk_signed_zero_and_extremes(L):
    """Ranking compares scores as floats: -0 and +0 tie (lower id first), the
    smallest subnormal ranks above zero, and the largest finite magnitudes
    keep their order."""
    E, K = 64, 6
    logits = np.full((3, E), -1.0, np.float32)
    logits[0, [9, 3, 5]] = [0.0, 0.0, -0.0]                      # three-way tie at zero
    logits[1, [7, 2]] = [30.0, -3.0e38]                          # far apart
    logits[1, 11] = np.float32(1.0e-45)                          # smallest subnormal beats -0
    logits[1, 12] = -0.0
    logits[2, :] = -3.0e38
    logits[2, [40, 20]] = [-2.9e38, -2.9e38]
    inds = torch.empty((3, K), dtype=torch.int32, device="cuda")
    w = torch.empty((3, K), dtype=torch.float32, device="cuda")
    st = status_word()
    L.e0_route_softmax_topk(dev(logits), 3, E, K, inds, w, st)
    got = inds.cpu().numpy()
    assert list(got[0, :3]) == [3, 5, 9]
    assert list(got[1, :3]) == [7, 11, 12]
    assert list(got[2, :2]) == [20, 40]
    rt = O.route_softmax_topk(logits.astype(np.float64), K)
    ex, msgs = routing_matches(got, w.cpu().numpy(), rt, allow_tie=False)
    assert not msgs, msgs[:5]
    assert L.e0_read_status(st) == 0


@pytest.mark.parametrize("T,E,n,G,K,s", [(40, 128, 8, 4, 8, 2.5), (16, 8, 4, 2, 2, 2.5), (8, 64, 1, 1, 6, 1.0),
                                          (8, 64, 8, 8, 4, 1.5), (7, 256, 32, 3, 5, 2.0)])
def test_sigmoid_group(L, T, E, n, G, K, s):
    g = np.random.default_rng(E + n + G)
    logits = (g.standard_normal((T, E)) * 2).astype(np.float32)
    inds = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    L.e0_route_sigmoid_group(dev(logits), T, E, n, G, K, s, inds, w)
    rt = O.route_sigmoid_group(logits.astype(np.float64), n, G, K, s)
    ex, msgs = routing_matches(inds.cpu().numpy(), w.cpu().numpy(), rt)
    assert not msgs, msgs[:5]
    assert len(ex) < T


def test_nonfinite_logits_set_status(L):
    logits = np.zeros((2, 16), np.float32)
    logits[1, 3] = np.nan
    inds = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    w = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    st = status_word()
    L.e0_route_softmax_topk(dev(logits), 2, 16, 4, inds, w, st)
    assert L.e0_read_status(st) & L.E0_ST_NONFINITE
    assert 3 not in inds[1].cpu().numpy().tolist()


def test_rmsnorm(L):
    x = np.random.default_rng(0).standard_normal((5, 2048)).astype(np.float32) * 3
    h = torch.empty((5, 2048), dtype=torch.float32, device="cuda")
    L.e0_rmsnorm(dev(x), 5, 2048, 1e-6, h)
    assert rel_l2(h.cpu().numpy(), O.rmsnorm(x.astype(np.float64))) < 1e-6


# ------------------------------------------------------------------ MoE block


def run_block(L, pool, x, W_r, rp, inds_in=None, w_in=None, shared=None):
    T = x.shape[0]
    ws_bytes = L.e0_workspace_size(0, T, pool.H, pool.I, pool.E, rp.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.empty((T, pool.H), dtype=torch.float32, device="cuda")
    io = torch.empty((T, rp.K), dtype=torch.int32, device="cuda")
    wo = torch.empty((T, rp.K), dtype=torch.float32, device="cuda")
    st = status_word()
    L.e0_moe_block_forward(x, T, pool.desc, W_r, rp, inds_in, w_in, shared, y, io, wo, ws, ws_bytes, st)
    return y.cpu().numpy(), io.cpu().numpy(), wo.cpu().numpy(), L.e0_read_status(st)


def test_tiny_layer_native_routing(L):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.tiny_layer(0)
    s = d["shape"]
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I)
    x = dev(d["x"])
    h = torch.empty_like(x)
    L.e0_rmsnorm(x, x.shape[0], s.H, 1e-6, h)
    Wr = dev(d["router"])
    y, inds, w, st = run_block(L, pool, h, Wr, L.route_params(K=s.K))
    assert st == 0
    hh = O.rmsnorm(d["x"].astype(np.float64))
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w)
    for t in range(len(yo)):
        if t not in ex:
            assert rel_l2(y[t], yo[t]) <= REL_L2, (t, rel_l2(y[t], yo[t]))


def test_tiny_layer_gate_up_swap_is_detected(L):
    """The same check fails loudly on a swapped gate/up bank (the oracle keeps the right one)."""
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.tiny_layer(0)
    s = d["shape"]
    bad = dict(d["bank"], gate=d["bank"]["up"], up=d["bank"]["gate"])
    pool = SlotPoolDev.resident(bad, s.H, s.I)
    hh = O.rmsnorm(d["x"].astype(np.float64))
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K)
    y, _, _, _ = run_block(L, pool, dev(hh.astype(np.float32)), None, L.route_params(K=s.K),
                           dev(rt.inds.astype(np.int32)), dev(rt.w.astype(np.float32)))
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w)
    assert rel_l2(y, yo) > 0.1


@pytest.fixture(scope="module")
def layer35(L):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.layer35b(1, T=8)
    s = d["shape"]
    d["pool"] = SlotPoolDev.resident(d["bank"], s.H, s.I)
    return d


@pytest.mark.parametrize("T", [1, 8])
def test_35b_layer_resident_native(L, layer35, T):
    d = layer35
    s = d["shape"]
    hh = O.rmsnorm(d["x"][:T].astype(np.float64))
    y, inds, w, st = run_block(L, d["pool"], dev(hh.astype(np.float32)), dev(d["router"]), L.route_params(K=s.K))
    assert st == 0
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K)
    ex, msgs = routing_matches(inds, w, rt)
    assert not msgs, msgs
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w)
    errs = [rel_l2(y[t], yo[t]) for t in range(T) if t not in ex]
    assert max(errs) <= REL_L2, errs


@pytest.mark.parametrize("T", [1, 8])
def test_35b_layer_staged_slots_predicted_routing(L, layer35, T):
    """2KT fixed slots filled by e0_slot_update from the resident bank, routing
    handed in (prediction-as-routing), experts read through the slot table."""
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = layer35
    s = d["shape"]
    hh = O.rmsnorm(d["x"][:T].astype(np.float64))
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K)
    n_slots = 2 * s.K * T
    staged = SlotPoolDev(s.H, s.I, s.E, n_slots)
    st = status_word()
    prev = d["inds_prev"][:T].ravel().astype(np.int32)
    nxt = rt.inds.ravel().astype(np.int32)
    # previous set first (as if it were the current one), then the predicted set
    L.e0_slot_update(staged.desc, dev(prev), prev.size, None, 0, d["pool"].data, st)
    L.e0_slot_update(staged.desc, dev(nxt), nxt.size, dev(prev), prev.size, d["pool"].data, st)
    assert L.e0_read_status(st) == 0
    # integer work is bit-exact against the oracle's slot_update
    tab = np.full(s.E, -1)
    occ = np.full(n_slots, -1)
    tab, occ, _ = O.slot_update(tab, occ, prev, None)
    tab, occ, copies = O.slot_update(tab, occ, nxt, prev)
    assert np.array_equal(staged.table.cpu().numpy(), tab)
    assert np.array_equal(staged.occupant.cpu().numpy(), occ)
    sb = staged.slot_bytes
    data = staged.data.view(n_slots, sb)
    bank = d["pool"].data.view(s.E, sb)
    for e, slot in enumerate(tab):
        if slot >= 0:
            assert torch.equal(data[slot], bank[e])
    y, inds, w, st2 = run_block(L, staged, dev(hh.astype(np.float32)), None, L.route_params(K=s.K),
                                dev(rt.inds.astype(np.int32)), dev(rt.w.astype(np.float32)))
    assert st2 == 0
    assert np.array_equal(inds, rt.inds)
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w)
    assert max(rel_l2(y[t], yo[t]) for t in range(T)) <= REL_L2


def test_slot_miss_contributes_zero_and_sets_status(L, layer35):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = layer35
    s = d["shape"]
    staged = SlotPoolDev(s.H, s.I, s.E, 8)
    hh = O.rmsnorm(d["x"][:1].astype(np.float64))
    inds = np.array([[3, 7, 11, 200]], np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1]], np.float32)
    st = status_word()
    present = np.array([3, 7, 11], np.int32)
    L.e0_slot_update(staged.desc, dev(present), 3, None, 0, d["pool"].data, st)
    y, _, _, code = run_block(L, staged, dev(hh.astype(np.float32)), None, L.route_params(K=4), dev(inds), dev(w))
    assert code & L.E0_ST_SLOT_MISS
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), inds[:, :3], w[:, :3].astype(np.float64))
    assert rel_l2(y[0], yo[0]) <= REL_L2


def test_slot_update_pool_full(L, layer35):
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = layer35
    s = d["shape"]
    staged = SlotPoolDev(s.H, s.I, s.E, 4)
    st = status_word()
    a = np.array([1, 2, 3, 4], np.int32)
    b = np.array([5, 6, 7, 8], np.int32)
    L.e0_slot_update(staged.desc, dev(a), 4, None, 0, d["pool"].data, st)
    L.e0_slot_update(staged.desc, dev(b), 4, dev(a), 4, d["pool"].data, st)
    assert L.e0_read_status(st) & L.E0_ST_POOL_FULL
    assert staged.table.cpu().numpy()[[1, 2, 3, 4]].tolist() == [0, 1, 2, 3]


def test_resident_slot_update_moves_nothing(L, layer35):
    d = layer35
    before = d["pool"].table.clone()
    st = status_word()
    nxt = np.array([1, 2, 3, 4], np.int32)
    L.e0_slot_update(d["pool"].desc, dev(nxt), 4, dev(nxt), 4, d["pool"].data, st)
    assert torch.equal(before, d["pool"].table)
    assert L.e0_read_status(st) == 0


# ------------------------------------------------------------------ shared expert + LoRA


def test_shared_expert_with_lora(L, layer35):
    from int4_gathered_expert_gb300.model import SharedDev
    d = layer35
    s = d["shape"]
    sh = synth.shared_expert(5, 0, s)
    shd = SharedDev(sh, s.H, s.I)
    T = 3
    hh = O.rmsnorm(d["x"][:T].astype(np.float64))
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K)
    y, _, _, st = run_block(L, d["pool"], dev(hh.astype(np.float32)), None, L.route_params(K=s.K),
                            dev(rt.inds.astype(np.int32)), dev(rt.w.astype(np.float32)), shd.desc)
    yo = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w, sh)
    assert max(rel_l2(y[t], yo[t]) for t in range(T)) <= REL_L2
    # the LoRA delta is really applied: without it the result is measurably different
    y_nolora = O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w, dict(sh, lora=None))
    assert rel_l2(y, y_nolora) > 5 * max(rel_l2(y[t], yo[t]) for t in range(T))


# ------------------------------------------------------------------ prerouter head


@pytest.mark.parametrize("T,first", [(1, False), (8, False), (2, True)])
def test_prerouter_head(L, layer35, T, first):
    from int4_gathered_expert_gb300.model import HeadDev
    d = layer35
    s = d["shape"]
    head = HeadDev(d["head"], s.H, s.E)
    hh = O.rmsnorm(d["x"][:T].astype(np.float64))
    cur = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K).inds.astype(np.int32)
    prev = None if first else d["inds_prev"][:T]
    ws_bytes = L.e0_workspace_size(1, T, s.H, head.hidden, s.E, s.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    z = torch.empty((T, s.E), dtype=torch.float32, device="cuda")
    inds = torch.empty((T, s.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, s.K), dtype=torch.float32, device="cuda")
    L.e0_prerouter_forward(dev(hh.astype(np.float32)), T, dev(cur), None if prev is None else dev(prev), head.desc,
                           L.route_params(K=s.K), z, inds, w, ws, ws_bytes)
    zo = np.stack([O.prerouter(hh[t], cur[t], None if prev is None else prev[t], d["head"]) for t in range(T)])
    assert rel_l2(z.cpu().numpy(), zo) < 1e-5
    rt = O.route_softmax_topk(zo, s.K)
    ex, msgs = routing_matches(inds.cpu().numpy(), w.cpu().numpy(), rt)
    assert not msgs, msgs


def test_prerouter_warm_start_reproduces_next_router_on_gpu(L, layer35):
    from int4_gathered_expert_gb300.model import HeadDev
    d = layer35
    s = d["shape"]
    hd = dict(d["head"], fc2=np.zeros_like(d["head"]["fc2"]))
    head = HeadDev(hd, s.H, s.E)
    T = 8
    hh = O.rmsnorm(d["x"][:T].astype(np.float64))
    cur = O.route_softmax_topk(O.router_logits(d["router"], hh), s.K).inds.astype(np.int32)
    ws_bytes = L.e0_workspace_size(1, T, s.H, head.hidden, s.E, s.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    z = torch.empty((T, s.E), dtype=torch.float32, device="cuda")
    inds = torch.empty((T, s.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, s.K), dtype=torch.float32, device="cuda")
    L.e0_prerouter_forward(dev(hh.astype(np.float32)), T, dev(cur), dev(d["inds_prev"][:T]), head.desc,
                           L.route_params(K=s.K), z, inds, w, ws, ws_bytes)
    rt_next = O.route_softmax_topk(O.router_logits(d["router_next"], hh), s.K)
    ex, msgs = routing_matches(inds.cpu().numpy(), w.cpu().numpy(), rt_next)
    assert not msgs, msgs

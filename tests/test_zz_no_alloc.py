"""The workspace-free MoE block entry point (for callers that cannot give the
library scratch memory: plugins whose host framework owns every device
allocation, or serving loops that must not allocate once they run) gives the
same results as e0_moe_block_forward, on two calls in a row through the C ABI.
Collected last on purpose; it builds its own inputs, so it also runs alone."""
import os

import numpy as np
import pytest

from int4_gathered_expert_gb300 import synth
from oracle import e0_oracle as O
from tests.parity import REL_L2, rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_gathered_expert_gb300 import build, lib
    if not os.path.exists(lib.LIB_PATH):
        build.build()
    lib.load()
    return lib


def test_noalloc_block_matches_workspace_block_twice(L):
    from int4_gathered_expert_gb300.model import SharedDev, SlotPoolDev
    d = synth.layer35b(1, T=8)
    s = d["shape"]
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I)
    sh = SharedDev(synth.shared_expert(5, 0, s), s.H, s.I)
    Wr = torch.from_numpy(d["router"]).cuda()
    rp = L.route_params(K=s.K)
    hh = O.rmsnorm(d["x"].astype(np.float64)).astype(np.float32)

    def both(T, shared, inds_in=None, w_in=None):
        x = torch.from_numpy(hh[:T]).cuda()
        outs = []
        for noalloc in (False, True):
            y = torch.full((T, s.H), np.nan, dtype=torch.float32, device="cuda")
            io = torch.full((T, s.K), -7, dtype=torch.int32, device="cuda")
            wo = torch.zeros((T, s.K), dtype=torch.float32, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            if noalloc:
                L.e0_moe_block_forward_noalloc(x, T, pool.desc, Wr, rp, inds_in, w_in, shared, y, io, wo, st)
            else:
                ws_bytes = L.e0_workspace_size(0, T, s.H, s.I, s.E, s.K)
                ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
                L.e0_moe_block_forward(x, T, pool.desc, Wr, rp, inds_in, w_in, shared, y, io, wo, ws, ws_bytes, st)
            assert L.e0_read_status(st) == 0
            outs.append((y.cpu().numpy(), io.cpu().numpy(), wo.cpu().numpy()))
        (y0, i0, w0), (y1, i1, w1) = outs
        assert np.array_equal(i0, i1)
        assert np.allclose(w0, w1, atol=1e-6)
        assert np.isfinite(y1).all()
        assert rel_l2(y1, y0) <= REL_L2
        return y1, i1

    # first call: 8 tokens, native routing, shared expert with LoRA
    y_a, inds_a = both(8, sh.desc)
    # second call in a row: fewer tokens, routing handed in, no shared expert;
    # the scratch still holds the first call's contents
    rt = O.route_softmax_topk(O.router_logits(d["router"], hh[:3].astype(np.float64)), s.K)
    inds_in = torch.from_numpy(rt.inds.astype(np.int32)).cuda()
    w_in = torch.from_numpy(rt.w.astype(np.float32)).cuda()
    y_b, inds_b = both(3, None, inds_in, w_in)
    assert np.array_equal(inds_b, rt.inds)


def test_noalloc_rejects_oversized_calls(L):
    """A call whose scratch need exceeds the fixed array is refused up front."""
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.tiny_layer(0)
    s = d["shape"]
    pool = SlotPoolDev(2048, 2048, 1024, 1)
    need = L.e0_workspace_size(0, 64, 2048, 2048, 1024, 32)
    assert need > (1 << 20)
    rp = L.route_params(K=32)
    x = torch.zeros((64, 2048), dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    rc = L.e0_moe_block_forward_noalloc(x, 64, pool.desc, x, rp, None, None, None, y, None, None,
                                        raise_on_error=False)
    assert rc == L.E0_ERR_UNSUPPORTED
    del s

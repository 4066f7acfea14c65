"""Failure detection without a GPU fault.

Host side: malformed calls are refused with a return code before anything is
launched.  Device side: every spin of the library is bounded; a wait that
nothing ends turns into E0_ST_TIMEOUT in the caller's status word and the
context stays usable (checked with a flag that no one sets).  Injected
faults (poisoned slot tables, NaN logits, full pools) are covered by the
decode parity tests."""
import ctypes as C
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    from int4_gathered_expert_gb300 import build, lib
    if not os.path.exists(lib.LIB_PATH):
        try:
            build.nvcc()
        except RuntimeError:
            pytest.skip("nvcc unavailable and the library is not built")
        build.build()
    lib.load()
    return lib


def test_selftest_rejects_bad_arguments_on_the_host(L):
    lib = L.load()
    assert lib.e0_selftest_bounded_wait(None, 10, C.c_void_p(256), None) == L.E0_ERR_NULL
    assert lib.e0_selftest_bounded_wait(C.c_void_p(256), 10, None, None) == L.E0_ERR_NULL
    assert lib.e0_selftest_bounded_wait(C.c_void_p(256), 0, C.c_void_p(256), None) == L.E0_ERR_ARG
    assert lib.e0_selftest_bounded_wait(C.c_void_p(256), L.E0_SELFTEST_MAX_WAIT_US + 1, C.c_void_p(256),
                                        None) == L.E0_ERR_ARG


def test_stack_step_refuses_an_unprepared_workspace(L):
    lib = L.load()
    # a workspace e0_stack_prepare never saw: refused before any launch
    assert lib.e0_stack_step(C.c_void_p(4096), C.c_void_p(4096), C.c_void_p(4096), None, 2, None,
                             None) == L.E0_ERR_ARG
    assert lib.e0_stack_step(C.c_void_p(4096), C.c_void_p(4096), C.c_void_p(4096), None, 7, None,
                             None) == L.E0_ERR_ARG


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.gpu
def test_bounded_wait_times_out_into_a_status_bit(L):
    _gpu()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")  # nothing ever sets it
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.e0_selftest_bounded_wait(flag, 2000, st)  # 2 ms of device time
    code = L.e0_read_status(st)
    assert code & L.E0_ST_TIMEOUT
    # the context is still usable: a compute call right after gives right answers
    r = torch.randn(3, 256, device="cuda")
    h = torch.empty_like(r)
    L.e0_rmsnorm(r, 3, 256, 1e-6, h)
    torch.cuda.synchronize()
    ref = r.double() / torch.sqrt((r.double() ** 2).mean(dim=1, keepdim=True) + 1e-6)
    assert torch.allclose(h.double(), ref, rtol=1e-5, atol=1e-6)


@pytest.mark.gpu
def test_bounded_wait_ends_early_when_the_flag_is_set(L):
    _gpu()
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.e0_selftest_bounded_wait(flag, L.E0_SELFTEST_MAX_WAIT_US, st)
    assert L.e0_read_status(st) == 0


@pytest.mark.gpu
def test_stack_status_clean_on_a_normal_token(L):
    """A prepared tiny stack runs a token with a clean status word, after a
    timed-out self-test on the same stream (the status words are separate)."""
    _gpu()
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import StackDev
    shape = synth.StackShape(layer=synth.TINY, n_layers=3, owners=(0, 1), shared_expert=True, seed=9)
    m = synth.stack_model(shape, n_tokens=2, threads=2)
    sd = StackDev(m, trace=False)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.e0_selftest_bounded_wait(flag, 1000, st)
    X = torch.from_numpy(m.x).cuda()
    for t in range(2):
        sd.step(X[t], impl=3)
    torch.cuda.synchronize()
    assert int(sd.status.item()) == 0
    assert L.e0_read_status(st) & L.E0_ST_TIMEOUT


@pytest.mark.gpu
def test_stack_ll_wait_limit_ends_in_timeout_and_recovers(L):
    """impl 3 with a 1 us wait limit (E0MOE_WAIT_US, read at prepare): at
    token 0 every layer routes natively, so each block waits for the gate/up
    copies it issued right after the routing, longer than 1 us; the launch
    returns with E0_ST_TIMEOUT in the status word (every block leaves after
    draining its own bulk copies), and after a prepare with the normal limit
    the same stack decodes the same bits as a stack that never timed out."""
    _gpu()
    import dataclasses
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import StackDev
    shape = dataclasses.replace(synth.STACK35B, n_layers=6, owners=(1, 2, 3, 4), seed=50)
    m = synth.stack_model(shape, n_tokens=2)
    X = torch.from_numpy(m.x).cuda()
    ref = StackDev(m, trace=False)
    want = [ref.step(X[t], impl=3).cpu().numpy().copy() for t in range(2)]
    assert int(ref.status.item()) == 0
    sd = StackDev(m, trace=False)
    old = os.environ.get("E0MOE_WAIT_US")
    os.environ["E0MOE_WAIT_US"] = "1"
    try:
        sd.prepare()
    finally:
        if old is None:
            del os.environ["E0MOE_WAIT_US"]
        else:
            os.environ["E0MOE_WAIT_US"] = old
    sd.step(X[0], impl=3)
    torch.cuda.synchronize()
    assert L.e0_read_status(sd.status) & L.E0_ST_TIMEOUT
    sd.status.zero_()
    sd.prepare()
    got = [sd.step(X[t], impl=3).cpu().numpy().copy() for t in range(2)]
    assert int(sd.status.item()) == 0
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    del ref, sd
    torch.cuda.empty_cache()

"""The C-ABI library builds, loads and exports every entry point that
include/e0moe.h declares; host-side argument checks answer without a GPU.
No compute call is made here (CPU only)."""
import ctypes as C
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "e0moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(e0_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from int4_gathered_expert_gb300 import build, lib as L
    if not os.path.exists(L.LIB_PATH):
        try:
            build.nvcc()
        except RuntimeError:
            pytest.skip("nvcc unavailable and the library is not built")
        build.build()
    return L.load()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for must in ["e0_moe_block_forward", "e0_route_softmax_topk", "e0_route_sigmoid_group", "e0_prerouter_forward",
                 "e0_slot_update", "e0_moe_prefill_forward", "e0_stack_step", "e0_pack_experts"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from int4_gathered_expert_gb300 import lib as L
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
    # the binding covers the same names
    assert set(L.exported_symbols()) == set(names)


def test_sizes_without_gpu(lib):
    from int4_gathered_expert_gb300 import lib as L
    assert L.e0_slot_bytes(2048, 512) == 1_769_472
    assert L.e0_slot_bytes(1536, 384) == 995_328
    assert L.e0_slot_bytes(100, 64) == 0
    assert L.e0_workspace_size(0, 8, 2048, 512, 256, 4) > 0
    assert L.e0_stack_workspace_size(40, 2048, 512, 256, 4, 512) > 0
    assert L.e0_stack_workspace_size(0, 2048, 512, 256, 4, 512) == 0


def test_host_validation_codes(lib):
    from int4_gathered_expert_gb300 import lib as L
    # K > E, unsupported E, bad groups: rejected before any launch
    assert lib.e0_route_softmax_topk(None, 4, 8, 9, None, None, None, None) == L.E0_ERR_ARG
    assert lib.e0_route_softmax_topk(None, 4, 4096, 4, None, None, None, None) == L.E0_ERR_UNSUPPORTED
    assert lib.e0_route_softmax_topk(None, 0, 16, 4, None, None, None, None) == L.E0_OK
    assert lib.e0_route_softmax_topk(None, 4, 16, 4, None, None, None, None) == L.E0_ERR_NULL
    assert lib.e0_route_sigmoid_group(None, 4, 128, 7, 4, 8, 2.5, None, None, None, None) == L.E0_ERR_ARG
    assert lib.e0_route_sigmoid_group(None, 4, 128, 8, 9, 8, 2.5, None, None, None, None) == L.E0_ERR_ARG
    assert lib.e0_route_sigmoid_group(None, 4, 128, 8, 1, 32, 2.5, None, None, None, None) == L.E0_ERR_ARG
    pool = L.SlotPool(None, None, None, 8, 2048, 512, 256)
    rp = L.route_params(K=4)
    assert L.e0_moe_block_forward(None, 1, pool, None, rp, None, None, None, None, None, None, None, 0,
                                  raise_on_error=False, stream=0) == L.E0_ERR_NULL
    pool = L.SlotPool(16, 16, 16, 8, 2000, 512, 256)
    assert L.e0_moe_block_forward(None, 1, pool, None, rp, None, None, None, None, None, None, None, 0,
                                  raise_on_error=False, stream=0) == L.E0_ERR_UNSUPPORTED
    assert lib.e0_stack_step(None, None, None, None, 0, None, None) == L.E0_ERR_NULL
    assert lib.e0_stack_step(C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), None, 0, None, None) == L.E0_ERR_ARG
    assert lib.e0_status_string(L.E0_ERR_CUDA).decode().startswith("CUDA")


def test_host_validation_of_ranges_prefetch_and_selftest(lib):
    """Layer ranges, the host-tier prefetch (plain and through the expert
    cache), layer updates and the bounded-wait self-test reject null
    pointers, workspaces that no stack was prepared in, and out-of-range
    waits on the host, before any launch."""
    from int4_gathered_expert_gb300 import lib as L
    unknown = C.c_void_p(256)   # never passed to e0_stack_prepare
    some = C.c_void_p(512)
    assert lib.e0_stack_step_range(None, None, None, 0, 1, None, None, None) == L.E0_ERR_NULL
    assert lib.e0_stack_step_range(some, some, unknown, 0, 1, None, None, None) == L.E0_ERR_ARG
    layer = L.StackLayer()
    assert lib.e0_stack_update_layers(None, C.byref(layer), 1, None) == L.E0_ERR_NULL
    assert lib.e0_stack_update_layers(unknown, None, 1, None) == L.E0_ERR_NULL
    assert lib.e0_stack_update_layers(unknown, C.byref(layer), 1, None) == L.E0_ERR_ARG
    pool = L.SlotPool(16, 16, 16, 8, 2048, 512, 256)
    assert lib.e0_stack_prefetch_experts(None, 7, 1, C.byref(pool), some, None, None) == L.E0_ERR_NULL
    assert lib.e0_stack_prefetch_experts(unknown, 7, 1, None, some, None, None) == L.E0_ERR_NULL
    assert lib.e0_stack_prefetch_experts(unknown, 7, 1, C.byref(pool), None, None, None) == L.E0_ERR_NULL
    assert lib.e0_stack_prefetch_experts(unknown, 7, 1, C.byref(pool), some, None, None) == L.E0_ERR_ARG
    cache = L.ExpertCache(16, 16, 16, 16, 16, 16, 64, 40 * 256)
    assert lib.e0_stack_prefetch_experts_cached(unknown, 7, 1, C.byref(pool), some, None, None,
                                                None) == L.E0_ERR_NULL
    assert lib.e0_stack_prefetch_experts_cached(unknown, 7, 1, C.byref(pool), some, C.byref(cache), None,
                                                None) == L.E0_ERR_ARG
    assert lib.e0_selftest_bounded_wait(None, 1000, some, None) == L.E0_ERR_NULL
    assert lib.e0_selftest_bounded_wait(some, 1000, None, None) == L.E0_ERR_NULL
    assert lib.e0_selftest_bounded_wait(some, 0, some, None) == L.E0_ERR_ARG
    assert lib.e0_selftest_bounded_wait(some, L.E0_SELFTEST_MAX_WAIT_US + 1, some, None) == L.E0_ERR_ARG


def test_tile_edge_sampler_covers_every_tile_of_the_busiest_expert():
    """The parity sampler of the full-size prefill tests: for a hand-made
    routing where expert 5 takes tokens 0..299 (three 128-token tiles), the
    tokens picked for it are the first and last of each tile."""
    import numpy as np
    from tests.parity import tile_edge_tokens
    inds = np.zeros((400, 2), np.int32)
    inds[:300, 0] = 5
    inds[300:, 0] = 7
    inds[:, 1] = np.arange(400) % 3
    inds[:300, 1] = 1 + np.arange(300) % 2  # no token holds expert 5 twice
    got = tile_edge_tokens(inds, n_experts=1, tile=128, per_expert=8)
    assert got == [0, 127, 128, 255, 256, 299]


def test_route_params_keeps_its_logit_bias_alive():
    """The routing struct carries the bias tensor's device address; the tensor
    must live as long as the struct, also when the caller passed a temporary."""
    import gc
    import weakref
    torch = pytest.importorskip("torch")
    from int4_gathered_expert_gb300 import lib as L
    bias = torch.arange(16, dtype=torch.float32)
    ref = weakref.ref(bias)
    rp = L.route_params(K=2, logit_bias=bias)
    addr = bias.data_ptr()
    del bias
    gc.collect()
    assert ref() is not None and rp.logit_bias == addr
    del rp
    gc.collect()
    assert ref() is None


def test_host_validation_of_batched_prefetch(lib):
    """The batched host-tier prefetch rejects null arrays, null banks and
    workspaces no stack was prepared in before any launch."""
    from int4_gathered_expert_gb300 import lib as L
    unknown = C.c_void_p(256)   # never passed to e0_stack_prepare
    pools = (L.SlotPool * 2)(L.SlotPool(16, 16, 16, 8, 2048, 512, 256), L.SlotPool(32, 32, 32, 8, 2048, 512, 256))
    layers = (C.c_int32 * 2)(7, 8)
    banks = (C.c_void_p * 2)(512, 1024)
    nobank = (C.c_void_p * 2)(512, None)
    f = lib.e0_stack_prefetch_experts_batch
    assert f(None, layers, 2, 1, pools, banks, None, None) == L.E0_ERR_NULL
    assert f(unknown, None, 2, 1, pools, banks, None, None) == L.E0_ERR_NULL
    assert f(unknown, layers, 2, 1, None, banks, None, None) == L.E0_ERR_NULL
    assert f(unknown, layers, 2, 1, pools, None, None, None) == L.E0_ERR_NULL
    assert f(unknown, layers, 2, 1, pools, banks, None, None) == L.E0_ERR_ARG
    assert f(unknown, None, 0, 1, None, None, None, None) == L.E0_ERR_ARG   # no stack there, even for n = 0
    # the binding marshals Python lists into the same call
    # a null bank is caught per entry, after the workspace is known
    assert f(unknown, layers, 2, 1, pools, nobank, None, None) == L.E0_ERR_ARG
    assert L.e0_stack_prefetch_experts_batch(256, [7, 8], 1, list(pools), [512, 1024], stream=0,
                                             raise_on_error=False) == L.E0_ERR_ARG
    g = lib.e0_stack_prefetch_experts_cached_batch
    cache = L.ExpertCache()
    assert g(unknown, layers, 2, 1, pools, banks, None, None, None) == L.E0_ERR_NULL
    assert g(None, layers, 2, 1, pools, banks, C.byref(cache), None, None) == L.E0_ERR_NULL
    assert g(unknown, layers, 2, 1, pools, banks, C.byref(cache), None, None) == L.E0_ERR_ARG

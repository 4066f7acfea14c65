#!/usr/bin/env python
"""Decode throughput of the 35B-tier 40-layer int4 MoE stack at batch 1.

One step = 256 consecutive decode tokens of an AR(1) token stream through the
40 layers (H=2048, I=512, E=256, softmax-top-4, shared expert with an
unmerged rank-16 LoRA, 33 prerouter heads owned by layers 6..38 whose
predictions route layers 7..39 one token later).  Each token is one launch of
the flag-carrying-word whole-token kernel (--kernel-impl 3; 0 = persistent
cooperative kernel, 1 = per-phase chain).  Weights are synthetic (seeded),
resident in HBM (18.1 GB expert bank); every token streams ~484 MB of
weights, far more than the 129 MB L2, so no flush is needed between
iterations.

The same JSON line also carries: the end-to-end rate through the C ABI with
host buffers (e2e), the CPU oracle on all host cores (cpu_baseline) and on one
thread for the single-layer workloads and the 8B and 35B stacks
(cpu_oracle_one_thread, run in a child process beside the GPU work), the K x
prerouter on/off sweep on the same weights (route_sweep), the 35B-tier single
layer alone at T=1 and T=8 (block_35b), the 8B-tier 24-layer stack
(stack_8b), the host-tier staged streaming run (streaming: consumer layers'
experts in pinned host memory, copied one token ahead of use), and the
T=4096 whole-layer prefill of the 35B and the 8B tier (prefill, prefill_8b).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun every rank runs an independent replica ("replicas only": the
path has no cross-GPU exchange); value = all ranks' tokens / max rank time.
The reference arm (--impl reference) times the CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s + expert-weight HBM GB/s (35B-tier MoE stack, batch 1)"
WORKLOAD = ("35B-tier 40-layer MoE stack decode, batch 1: H=2048, I=512, E=256, softmax-top-k K=4, "
            "shared expert + unmerged LoRA r=16 alpha=32, 33 prerouter heads (owners 6..38, hidden 512), "
            "AR(1) rho=0.8 token stream")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--tokens-per-step", type=int, default=256)
    p.add_argument("--no-cpu", action="store_true", help="skip the timed CPU-oracle baseline")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--kernel-impl", type=int, default=3,
                   help="3 flag-carrying-word kernel (default), 0 persistent cooperative kernel, 1 per-phase chain")
    p.add_argument("--layers", type=int, default=40, help="fewer layers: a small case for profiling only")
    p.add_argument("--no-prefill", action="store_true", help="skip the whole-layer prefill measurement")
    p.add_argument("--prefill-only", action="store_true")
    p.add_argument("--route-k", type=int, default=4, help="routed experts per token (the 35B tier uses 4)")
    p.add_argument("--no-prerouter", action="store_true",
                   help="every layer routes with its own router; no prerouter heads")
    p.add_argument("--no-streaming", action="store_true", help="skip the host-tier staged-streaming measurement")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the K / prerouter sweep, the single-layer block and the 8B-tier stack measurements")
    p.add_argument("--stream-split", type=int, default=22,
                   help="first layer of the second launch of a token in the staged-streaming run")
    return p.parse_args()


# ---------------------------------------------------------------- prefill (T=4096 whole-layer)


def run_prefill_bench(dev, reps: int = 5, tier: str = "35b"):
    """Whole-layer prefill, T=4096: the 35B-tier layer with a Zipf(1.1) expert
    load (softmax-top-4), or the 8B-tier layer (sigmoid-group, K=8); the L2 is
    flushed (a 256 MB write) before every timed call."""
    import torch
    from int4_gathered_expert_gb300 import lib as L
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import SlotPoolDev
    d = synth.prefill35b(4, T=4096) if tier == "35b" else synth.prefill8b(5, T=4096)
    s = d["shape"]
    T = d["X"].shape[0]
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I)
    X = torch.from_numpy(d["X"]).to(dev)
    Wr = torch.from_numpy(d["router"]).to(dev)
    if tier == "35b":
        bias = torch.from_numpy(d["logit_bias"]).to(dev)
        rp = L.route_params(K=s.K, logit_bias=bias)
    else:
        rp = L.route_params(mode=L.E0_ROUTE_SIGMOID_GROUP, K=s.K, n_groups=s.n_groups, topk_groups=s.topk_groups,
                            scale=s.route_scale)
    ws_bytes = L.e0_workspace_size(2, T, s.H, s.I, s.E, s.K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    Y = torch.empty((T, s.H), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    for _ in range(3):
        L.e0_moe_prefill_forward(X, T, pool.desc, Wr, rp, Y, None, None, ws, ws_bytes, st, stream=stream)
    torch.cuda.synchronize()
    # device time of a call: the GPU is held in a sleep while the host enqueues
    # every (flush, call) pair, so no call waits for its launches
    evs = []
    with torch.cuda.stream(stream):
        torch.cuda._sleep(20_000_000)
        for _ in range(reps):
            flush.fill_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            L.e0_moe_prefill_forward(X, T, pool.desc, Wr, rp, Y, None, None, ws, ws_bytes, st, stream=stream)
            b.record(stream)
            evs.append((a, b))
    torch.cuda.synchronize()
    t = float(np.median([a.elapsed_time(b) / 1e3 for a, b in evs]))
    # latency of a call that starts on an idle GPU: includes the host's encoding
    # and launching of the call's kernels
    sync = []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            L.e0_moe_prefill_forward(X, T, pool.desc, Wr, rp, Y, None, None, ws, ws_bytes, st, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        sync.append(a.elapsed_time(b) / 1e3)
    t_sync = float(np.median(sync))
    flops = 2.0 * T * s.K * 3 * s.H * s.I
    pk = peaks()
    peak = pk["bf16_tflops"] if pk else 1900.0
    name = ("35B-tier whole-layer prefill, T=4096, K=4, Zipf(1.1) expert load" if tier == "35b" else
            "8B-tier whole-layer prefill, T=4096, H=1536, I=384, E=128, sigmoid-group n=8 G=4 K=8")
    return {"workload": name,
            "value": T / t, "unit": "tok/s", "ms": t * 1e3, "useful_tflops": flops / t / 1e12,
            "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peak, "unit": "TFLOP/s",
                         "frac": flops / t / 1e12 / peak,
                         # DRAM bytes of one launch of the dominant kernel (the
                         # gate/up grouped GEMM), 35B tier only
                         "traffic": recorded_traffic("k_umma2<1>") if tier == "35b" else None,
                         "traffic_kernel": "k_umma2<1>" if tier == "35b" else None,
                         "peak_source": "MEASURED_PEAKS.json bf16_tflops (measured, fp16 = bf16 rate)"
                         if pk else "fallback",
                         # the same rate against the GEMM rate held for seconds under the power cap
                         "peak_sustained": pk.get("bf16_tflops_sustained") if pk else 1700.0,
                         "frac_sustained": flops / t / 1e12 / (pk.get("bf16_tflops_sustained") if pk else 1700.0)},
            "l2": "flushed (256 MB write) before each timed call",
            "timing": "device time, calls enqueued ahead of the GPU; ms_idle_start: the same call started on an "
                      "idle GPU (host encoding and launches inside the timed region)",
            "ms_idle_start": t_sync * 1e3, "device_status": int(st.item())}


# ---------------------------------------------------------------- one layer alone


def _timed(fn, stream, flush, reps: int):
    """Median device time (s) of fn() on ``stream``, the L2 flushed (a 256 MB
    write) before each call."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    return float(np.median(times))


def run_block_bench(dev, reps: int = 20):
    """The 35B-tier single decode layer (H=2048, I=512, E=256, K=4) at T=1 and
    T=8: the MoE block with native routing on the resident bank, the same
    block on a 2KT-slot staged pool with the routing handed in, the slot
    update that fills that pool, and the prerouter head.  Bytes are the
    weights the call must read: the union of the selected experts (plus the
    router for native routing, the head's weights for the head)."""
    import torch
    from int4_gathered_expert_gb300 import lib as L
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import HeadDev, SlotPoolDev
    d = synth.layer35b(1, T=8)
    s = d["shape"]
    eb = synth.expert_nbytes(s)
    pool = SlotPoolDev.resident(d["bank"], s.H, s.I, dev)
    Wr = torch.from_numpy(d["router"]).to(dev)
    head = HeadDev(d["head"], s.H, s.E, dev)
    head_bytes = sum(int(np.asarray(v).nbytes) for v in d["head"].values())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    pk = peaks()
    peak = pk["hbm_gbs"] if pk else 6800.0
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {"workload": "35B-tier single layer decode: H=2048, I=512, E=256, softmax-top-k K=4, prerouter head "
                       "hidden 512; seed 1", "l2": "flushed (256 MB write) before each timed call",
           "peak_gbs": peak}
    x = torch.from_numpy(d["x"]).to(dev)
    for T in (1, 8):
        h = torch.empty((T, s.H), dtype=torch.float32, device=dev)
        L.e0_rmsnorm(x[:T].contiguous(), T, s.H, 1e-6, h)
        ws_bytes = L.e0_workspace_size(0, T, s.H, s.I, s.E, s.K)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        y = torch.empty((T, s.H), dtype=torch.float32, device=dev)
        io = torch.empty((T, s.K), dtype=torch.int32, device=dev)
        wo = torch.empty((T, s.K), dtype=torch.float32, device=dev)
        rp = L.route_params(K=s.K)

        def native():
            L.e0_moe_block_forward(h, T, pool.desc, Wr, rp, None, None, None, y, io, wo, ws, ws_bytes, st,
                                   stream=stream)
        t_nat = _timed(native, stream, flush, reps)
        inds = io.cpu().numpy()
        n_union = len(set(int(e) for e in inds.ravel()))
        b_nat = n_union * eb + s.E * s.H * 2
        # staged: 2KT slots filled from the resident bank (previous set, then this one)
        n_slots = 2 * s.K * T
        staged = SlotPoolDev(s.H, s.I, s.E, n_slots, dev)
        prev = torch.from_numpy(d["inds_prev"][:T].ravel().astype(np.int32)).to(dev)
        cur = io.reshape(-1).clone()
        L.e0_slot_update(staged.desc, prev, prev.numel(), None, 0, pool.data, st, stream=stream)
        torch.cuda.synchronize()
        tab0, occ0 = staged.table.clone(), staged.occupant.clone()
        n_new = len(set(cur.cpu().tolist()) - set(prev.cpu().tolist()))

        def update():
            staged.table.copy_(tab0)
            staged.occupant.copy_(occ0)
            L.e0_slot_update(staged.desc, cur, cur.numel(), prev, prev.numel(), pool.data, st, stream=stream)
        t_upd = _timed(update, stream, flush, reps)
        wi = wo.clone()

        def staged_block():
            L.e0_moe_block_forward(h, T, staged.desc, None, rp, cur, wi, None, y, io, wo, ws, ws_bytes, st,
                                   stream=stream)
        t_stg = _timed(staged_block, stream, flush, reps)
        b_stg = n_union * eb
        # prerouter head of the same layer
        hws_bytes = L.e0_workspace_size(1, T, s.H, head.hidden, s.E, s.K)
        hws = torch.empty(hws_bytes, dtype=torch.uint8, device=dev)
        z = torch.empty((T, s.E), dtype=torch.float32, device=dev)
        ni = torch.empty((T, s.K), dtype=torch.int32, device=dev)
        nw = torch.empty((T, s.K), dtype=torch.float32, device=dev)
        pv = prev.reshape(T, s.K)

        def head_call():
            L.e0_prerouter_forward(h, T, io, pv, head.desc, rp, z, ni, nw, hws, hws_bytes, st, stream=stream)
        t_head = _timed(head_call, stream, flush, reps)
        out["T%d" % T] = {
            "block_native": {"us": t_nat * 1e6, "bytes": b_nat, "gbs": b_nat / t_nat / 1e9,
                             "frac": b_nat / t_nat / 1e9 / peak, "experts_read": n_union},
            "block_staged": {"us": t_stg * 1e6, "bytes": b_stg, "gbs": b_stg / t_stg / 1e9,
                             "frac": b_stg / t_stg / 1e9 / peak, "n_slots": n_slots},
            "slot_update": {"us": t_upd * 1e6, "experts_copied": n_new,
                            "copy_gbs": n_new * eb * 2 / t_upd / 1e9 if n_new else None},
            "prerouter": {"us": t_head * 1e6, "bytes": head_bytes, "gbs": head_bytes / t_head / 1e9}}
    out["device_status"] = int(st.item())
    return out


# ---------------------------------------------------------------- other stacks and variants


def _time_tokens(sd, X, t0: int, t1: int, stream, impl: int = 3) -> float:
    """Seconds per token of sd over tokens t0..t1 (device time, one launch a token)."""
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for t in range(t0, t1):
            sd.step(X[t], impl=impl, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / (t1 - t0)


def run_stack8b_bench(dev, n_warm: int = 8, n_timed: int = 128):
    """8B-tier 24-layer stack decode (H=1536, I=384, E=128, sigmoid-group n=8
    G=4 s=2.5 K=8, heads owned by 7..22), one flag-carrying-word launch a
    token; token 0 (every layer routes natively) is in the warm-up."""
    import torch
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import StackDev
    shape = synth.STACK8B
    model = synth.stack_model(shape, n_tokens=n_warm + n_timed)
    sd = StackDev(model, device=dev)
    X = torch.from_numpy(model.x).to(dev)
    stream = torch.cuda.Stream()
    _time_tokens(sd, X, 0, n_warm, stream)
    s_tok = _time_tokens(sd, X, n_warm, n_warm + n_timed, stream)
    nb = bytes_per_token(shape, native_layers=sum(1 for l in range(shape.n_layers) if l not in shape.consumers))
    pk = peaks()
    peak = pk["hbm_gbs"] if pk else 6800.0
    st = int(sd.status.item())
    del sd
    torch.cuda.empty_cache()
    return {"workload": "8B-tier 24-layer stack decode, batch 1: H=1536, I=384, E=128, sigmoid group-limited "
                        "n=8 G=4 s=2.5 K=8, 16 prerouter heads (owners 7..22, hidden 512), AR(1) rho=0.8 stream",
            "value": 1.0 / s_tok, "unit": "tok/s", "us_per_token": s_tok * 1e6, "tokens": n_timed,
            "bytes_per_token": nb, "weight_gbs": nb["total"] / s_tok / 1e9,
            "roofline": {"bound": "hbm", "achieved": nb["total"] / s_tok / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": nb["total"] / s_tok / 1e9 / peak, "kernel": "k_stack_ll",
                         "peak_nominal": HBM_NOMINAL_GBS,
                         "frac_nominal": nb["total"] / s_tok / 1e9 / HBM_NOMINAL_GBS},
            "device_status": st}


def run_route_sweep(sd, X, n_warm: int = 8, n_timed: int = 96):
    """The 35B-tier stack with K = 2, 4, 8 routed experts, each with the
    prerouter on (layers 7..39 take the prediction made one token earlier) and
    off (every layer routes with its own router, no heads): same weights."""
    import torch
    stream = torch.cuda.Stream()
    rows = []
    for K in (2, 4, 8):
        r = {"K": K}
        for on in (True, False):
            v = sd.variant(K=K, prerouter=on)
            _time_tokens(v, X, 0, n_warm, stream)
            s_tok = _time_tokens(v, X, n_warm, n_warm + n_timed, stream)
            key = "on" if on else "off"
            r[key] = {"tok_s": 1.0 / s_tok, "us_per_token": s_tok * 1e6, "device_status": int(v.status.item())}
            del v
        r["on_over_off"] = r["on"]["tok_s"] / r["off"]["tok_s"]
        rows.append(r)
    torch.cuda.empty_cache()
    return {"workload": "35B-tier 40-layer stack, K in {2, 4, 8} x prerouter on/off, same weights and stream",
            "tokens": n_timed, "rows": rows}


def oracle_config_timings(stacks):
    """The oracle as it stands on the workloads other than the headline
    line: one call of the routing + MoE block of the tiny layer (T=8, best
    of three) and of the 35B-tier single layer (T=1, T=8), and, for each
    named stack ("stack_8b", "stack_35b"), token 0 (every layer routes
    natively) and one steady-state token; eight tokens are extrapolated as
    token 0 + 7 steady tokens."""
    import gc
    from oracle import e0_oracle as O
    from int4_gathered_expert_gb300 import synth
    res = {}

    def blk(d, T):
        hh = O.rmsnorm(d["x"][:T].astype(np.float64))
        t0 = time.perf_counter()
        rt = O.route_softmax_topk(O.router_logits(d["router"], hh), d["shape"].K)
        O.moe_block(hh, O.BankExperts(d["bank"]), rt.inds, rt.w)
        return time.perf_counter() - t0

    d = synth.tiny_layer(0, T=8)
    blk(d, 8)
    res["tiny_T8_ms"] = 1e3 * min(blk(d, 8) for _ in range(3))
    d = synth.layer35b(1, T=8)
    for T in (1, 8):
        res["l35b_T%d_ms" % T] = 1e3 * blk(d, T)
    del d
    shapes = {"stack_8b": synth.STACK8B, "stack_35b": synth.STACK35B}
    for name in stacks:
        shape = shapes[name]
        m = synth.stack_model(shape, n_tokens=2)
        st = O.StackState(shape.n_layers)
        t = []
        for i in range(2):
            t0 = time.perf_counter()
            O.stack_token(m.x[i], m, st)
            t.append(time.perf_counter() - t0)
        res[name] = {"token0_s": t[0], "steady_token_s": t[1], "tok_s": 1.0 / t[1],
                     "tokens_8_s_extrapolated": t[0] + 7 * t[1]}
        del m, st
        gc.collect()
    return res


ORACLE_ONE_THREAD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
print(json.dumps(bench.oracle_config_timings(("stack_8b", "stack_35b"))))
"""


def start_oracle_one_thread():
    """Starts, in a child process with BLAS limited to one thread, the
    oracle's MoE block (routing + experts) on the tiny layer (T=8) and the
    35B-tier single layer (T=1, T=8), then the 8B and 35B stacks for two
    tokens each: token 0 (every layer routes natively) and one steady-state
    token.  Eight tokens are extrapolated as token 0 + 7 steady tokens.  The
    child runs on one host core while the GPU measurements go on."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    return subprocess.Popen([sys.executable, "-c", ORACLE_ONE_THREAD, ROOT], env=env, stdout=subprocess.PIPE,
                            stderr=subprocess.PIPE, text=True)


def finish_oracle_one_thread(proc, timeout: float = 600.0):
    try:
        out, _ = proc.communicate(timeout=timeout)
        r = json.loads(out.strip().splitlines()[-1])
    except subprocess.TimeoutExpired as ex:
        proc.kill()
        proc.communicate()
        return {"error": repr(ex)[:200]}
    except (ValueError, IndexError) as ex:
        return {"error": repr(ex)[:200]}
    r.update({"cores": 1, "kind": "oracle",
              "sample": "float64 numpy oracle, BLAS limited to one thread: one call of the routing + MoE block "
                        "(tiny layer, 35B-tier layer); the 8B and 35B stacks for token 0 and one steady token, "
                        "tokens_8_s_extrapolated = token 0 + 7 x the steady token (extrapolated, not measured)"})
    return r


# ---------------------------------------------------------------- host-tier staged streaming


def run_streaming_bench(model, X, args, tps: int):
    """Decode with the consumer layers' experts in pinned host memory and 2K
    device slots per layer, filled with the prerouter's prediction one token
    ahead (model.StreamedStack).  Reports tok/s with the copies overlapped on a
    second stream, with the copies serialised on the compute stream, and with
    the same two-launch token from the resident bank; plus the expert bytes
    copied per token (measured from the slot pools' occupant tables)."""
    import torch
    from int4_gathered_expert_gb300.model import StackDev, StreamedStack
    sd = StackDev(model, trace=False)
    ss = StreamedStack(sd, split=args.stream_split)
    n_tok = min(tps, X.shape[0] - 1)

    def timed(fn, n):
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(ss.cs)
        for i in range(n):
            fn(i)
        b.record(ss.cs)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    ss.start(X[0])
    # expert copies per token, from the occupant tables (untimed pass)
    occ = {l: ss.pools[l].occupant.clone() for l in ss.staged}
    n_count = min(16, n_tok)
    copied = 0
    for i in range(n_count):
        ss.step(X[1 + i])
        torch.cuda.synchronize()
        for l in ss.staged:
            now = ss.pools[l].occupant
            copied += int((now != occ[l]).sum().item())
            occ[l] = now.clone()
    per_token_bytes = copied / n_count * ss.copy_bytes_per_expert()
    base = 1 + n_count
    n = max(1, min(n_tok, X.shape[0] - base) // 2)
    t_overlap = timed(lambda i: ss.step(X[base + i], overlap=True), n)
    t_serial = timed(lambda i: ss.step(X[base + n + i], overlap=False), n)
    status = int(ss.status.item())
    n_staged = len(ss.staged)
    host = ss.host
    del ss
    torch.cuda.empty_cache()
    # the same two launches per token from the resident bank
    rd = sd
    rd.prepare()
    cs = torch.cuda.Stream()
    L_ = rd.L
    from int4_gathered_expert_gb300 import lib as L

    def resident_token(i):
        L.e0_stack_step_range(X[i], None, rd.ws, 0, args.stream_split, None, rd.status, stream=cs)
        L.e0_stack_step_range(None, rd.r_out, rd.ws, args.stream_split, L_, None, rd.status, stream=cs)

    for i in range(3):
        resident_token(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(cs)
    for i in range(n):
        resident_token(3 + i)
    b.record(cs)
    torch.cuda.synchronize()
    t_res = a.elapsed_time(b) / 1e3
    exposed = max(0.0, t_serial - t_res)
    # the same streaming with a cross-layer LRU cache of bundles in device memory in front of the host bank
    caches = {}
    for cap in (64, 1024):
        from int4_gathered_expert_gb300.model import ExpertCacheDev
        sd.prepare()
        cache = ExpertCacheDev(cap, sd.L, sd.H, sd.I, sd.E)
        ssc = StreamedStack(sd, split=args.stream_split, cache=cache, host=host)
        ssc.start(X[0])
        for i in range(8):  # warm the cache
            ssc.step(X[1 + i])
        torch.cuda.synchronize()
        c0 = cache.stats()
        torch.cuda.synchronize()
        a2 = torch.cuda.Event(enable_timing=True)
        b2 = torch.cuda.Event(enable_timing=True)
        a2.record(ssc.cs)
        for i in range(n):
            ssc.step(X[9 + i], overlap=True)
        b2.record(ssc.cs)
        torch.cuda.synchronize()
        tc = a2.elapsed_time(b2) / 1e3
        c1 = cache.stats()
        hits, misses = c1["hits"] - c0["hits"], c1["misses"] - c0["misses"]
        caches[str(cap)] = {"tok_s_streamed_overlapped": n / tc, "hit_rate": hits / max(1, hits + misses),
                            "host_bytes_per_token": misses / n * ssc.copy_bytes_per_expert(),
                            "device_status": int(ssc.status.item())}
        del ssc, cache
        torch.cuda.empty_cache()
    del sd, host
    torch.cuda.empty_cache()
    return {"workload": "35B-tier stack decode with host-tier staged streaming: consumer layers hold 2K device "
                        "slots filled from pinned host memory with the prediction one token ahead",
            "expert_cache": caches,
            "tokens": n, "split": args.stream_split, "staged_layers": n_staged,
            "tok_s_streamed_overlapped": n / t_overlap, "tok_s_streamed_serial": n / t_serial,
            "tok_s_resident_two_launch": n / t_res,
            "expert_bytes_copied_per_token": per_token_bytes,
            "exposed_copy_us_per_token_serial": 1e6 * exposed / n,
            "exposed_copy_us_per_token_overlapped": 1e6 * max(0.0, t_overlap - t_res) / n,
            "device_status": status}


# ---------------------------------------------------------------- algorithmic bytes


def bytes_per_token(shape, native_layers: int):
    """Weight bytes one steady-state token must read (each selected expert
    counted once), split by kind."""
    from int4_gathered_expert_gb300 import synth
    s = shape.layer
    expert = synth.expert_nbytes(s)
    Lyr = shape.n_layers
    routed = Lyr * s.K * expert
    shared = Lyr * expert if shape.shared_expert else 0
    r = shape.lora_rank
    lora = Lyr * 2 * r * (2 * (s.H + s.I) + (s.I + s.H)) if shape.shared_expert else 0
    hid = shape.head_hidden
    head = (hid * s.H * 2 + s.E * s.H * 2 + s.E * hid * 2 + 2 * s.K * (hid + s.E) * 2 + (hid + s.E) * 2)
    heads = len(shape.owners) * head
    routers = native_layers * s.E * s.H * 2
    return {"routed": routed, "shared": shared, "lora": lora, "heads": heads, "routers": routers,
            "total": routed + shared + lora + heads + routers}


# ---------------------------------------------------------------- clocks


class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[2]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- helpers


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


# the sources each profiled kernel is compiled from (a change to any of them
# voids its recorded DRAM traffic)
KERNEL_SOURCES = {
    "k_stack_ll": ("e0_common.cuh", "e0_decode.cuh", "e0_decode.cu", "e0_internal.h", "e0_stack_ll.cuh"),
    "k_umma2<1>": ("e0_common.cuh", "e0_decode.cuh", "e0_internal.h", "e0_prefill.cu", "e0_umma.cuh"),
}


def kernel_source_digest(kernel: str = "k_stack_ll"):
    """Digest of a kernel's source files with comments and whitespace left
    out: an edit that cannot change the compiled code keeps the digest."""
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "int4_gathered_expert_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(d, f), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    except (OSError, ValueError):
        return None
    k = rec.get(kernel)
    if not k or kernel not in KERNEL_SOURCES or k.get("source_digest") != kernel_source_digest(kernel):
        return None
    return k.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (x itself without a process
    group).  Works on any backend: the tensor lives on ``device`` (a CUDA
    device for NCCL, the CPU for gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Units processed by all ranks together over the slowest rank's time
    (replicas: every rank does the same amount of work)."""
    return world * units_per_rank / seconds_max


# GB300 HBM3e bandwidth as specified (the measured copy rate is the roofline's peak)
HBM_NOMINAL_GBS = 8000.0

# launches of this library's kernels per decode token, by stack implementation
LAUNCHES_PER_TOKEN = {0: 1, 3: 1}
KERNEL_NAME = {0: "k_stack_token", 1: "k_stack_gateup/k_stack_down chain", 3: "k_stack_ll"}


# ---------------------------------------------------------------- CPU oracle timing


def time_oracle(model, n_tokens: int):
    """The oracle as it stands, decoding the first ``n_tokens`` of the stream."""
    from oracle import e0_oracle as O
    st = O.StackState(len(model.banks))
    t0 = time.perf_counter()
    for t in range(n_tokens):
        O.stack_token(model.x[t], model, st)
    return time.perf_counter() - t0


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- arms


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from int4_gathered_expert_gb300 import synth
    shape = synth.STACK35B
    n = args.warmup + args.steps
    model = synth.stack_model(shape, n_tokens=max(n, 2))
    # each step: one decode token of the same workload through all 40 layers
    from oracle import e0_oracle as O
    st = O.StackState(shape.n_layers)
    for t in range(args.warmup):
        O.stack_token(model.x[t], model, st)
    t0 = time.perf_counter()
    for t in range(args.warmup, n):
        O.stack_token(model.x[t], model, st)
    el = time.perf_counter() - t0
    v = args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": 1, "sample": "one decode token per step"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cores(), "kind": "oracle",
                             "sample": f"{args.steps} decode tokens (after {args.warmup} warm-up tokens) of the "
                                       "40-layer stack, float64 numpy oracle"},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    import __graft_entry__
    __graft_entry__.build()
    from int4_gathered_expert_gb300 import synth
    from int4_gathered_expert_gb300.model import StackDev

    if args.prefill_only:
        print(json.dumps({"prefill": run_prefill_bench(dev), "prefill_8b": run_prefill_bench(dev, tier="8b")}),
              flush=True)
        return 0
    shape = synth.STACK35B
    import dataclasses
    if args.layers != shape.n_layers:
        shape = dataclasses.replace(shape, n_layers=args.layers,
                                    owners=tuple(o for o in shape.owners if o + 1 < args.layers))
    if args.route_k != shape.layer.K:
        shape = dataclasses.replace(shape, layer=dataclasses.replace(shape.layer, K=args.route_k))
    if args.no_prerouter:
        shape = dataclasses.replace(shape, owners=())
    tps = args.tokens_per_step
    n_tok = (args.warmup + args.steps) * tps
    model = synth.stack_model(shape, n_tokens=n_tok)
    sd = StackDev(model, trace=False)
    X = torch.from_numpy(model.x).to(dev)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def decode(t0, t1, ev=None):
        with torch.cuda.stream(stream):
            for t in range(t0, t1):
                if ev is not None:
                    ev[t - t0][0].record(stream)
                sd.step(X[t], impl=args.kernel_impl, stream=stream)
                if ev is not None:
                    ev[t - t0][1].record(stream)

    # warm-up (includes token 0, which routes every layer natively)
    decode(0, args.warmup * tps)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()

    clk = ClockSampler(dev)
    clk.start()
    n_timed = args.steps * tps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_timed)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    decode(args.warmup * tps, n_tok, ev)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    el_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    st = int(sd.status.cpu().item())
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    el_ms = max_over_ranks(el_ms, device=dev)

    value = whole_job_rate(n_timed, ws, el_ms / 1e3)
    nb = bytes_per_token(shape, native_layers=sum(1 for l in range(shape.n_layers) if l not in shape.consumers))
    mean_launch_s = float(np.mean(launch_ms)) / 1e3
    pk = peaks()
    peak = pk["hbm_gbs"] if pk else 6800.0
    achieved = nb["total"] / mean_launch_s / 1e9
    kname = KERNEL_NAME.get(args.kernel_impl, "?")
    traffic = recorded_traffic(kname)

    # end to end: the same decode through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        Xh = torch.from_numpy(model.x).pin_memory()
        out_h = torch.empty((tps, shape.layer.H), dtype=torch.float32).pin_memory()
        xin = torch.empty(shape.layer.H, dtype=torch.float32, device=dev)
        rout = torch.empty(shape.layer.H, dtype=torch.float32, device=dev)
        sd.prepare()
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        w0 = time.perf_counter()
        for sstep in range(args.warmup + args.steps):
            if sstep == args.warmup:
                torch.cuda.synchronize()
                w0 = time.perf_counter()
            with torch.cuda.stream(stream):
                for i in range(tps):
                    t = sstep * tps + i
                    xin.copy_(Xh[t], non_blocking=True)
                    sd.step(xin, impl=args.kernel_impl, stream=stream, out=rout)
                    out_h[i].copy_(rout, non_blocking=True)
            stream.synchronize()
        e2e_s = time.perf_counter() - w0
        if ws > 1:
            torch.distributed.barrier()
        e2e_s = max_over_ranks(e2e_s, device=dev)
        e2e = {"value": whole_job_rate(n_timed, ws, e2e_s), "unit": "tok/s", "h2d_bytes_per_step": tps * shape.layer.H * 4,
               "d2h_bytes_per_step": tps * shape.layer.H * 4}

    cpu = cpu_all = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        n_cpu = 3
        el = time_oracle(model, n_cpu)
        cpu = {"value": n_cpu / el, "unit": "tok/s", "cores": cores(), "kind": "oracle",
               "sample": f"first {n_cpu} tokens of the same stream (token 0 routes all 40 layers natively) "
                         "through the 40-layer stack, float64 numpy oracle"}
        try:
            cpu_all = oracle_config_timings(("stack_8b",))
            cpu_all.update({"cores": cores(), "kind": "oracle",
                            "sample": "float64 numpy oracle on all host cores (numpy's BLAS threads): one call of "
                                      "the routing + MoE block (tiny layer, 35B-tier layer); the 8B stack for "
                                      "token 0 and one steady token, tokens_8_s_extrapolated = token 0 + 7 x "
                                      "the steady token (extrapolated, not measured); the 35B stack is "
                                      "cpu_baseline"})
        except Exception as ex:  # a measurement that cannot run here is reported, not fatal
            cpu_all = {"error": repr(ex)[:300]}

    sweep = None
    if rank == 0 and not args.no_extras and args.kernel_impl == 3 and args.layers == 40 and args.route_k == 4 \
            and not args.no_prerouter:
        sweep = run_route_sweep(sd, X)

    streaming = None
    if rank == 0 and not args.no_streaming and args.kernel_impl == 3:
        del sd
        torch.cuda.empty_cache()
        try:
            streaming = run_streaming_bench(model, X, args, tps)
        except Exception as ex:  # a measurement that cannot run here is reported, not fatal
            streaming = {"error": repr(ex)[:300]}
        sd = None

    block = stack8b = oracle1 = None
    oracle1_proc = None
    if rank == 0 and ws == 1 and not args.no_extras and not args.no_cpu:
        oracle1_proc = start_oracle_one_thread()
    if rank == 0 and not args.no_extras:
        del sd
        sd = None
        torch.cuda.empty_cache()
        block = run_block_bench(dev)
        torch.cuda.empty_cache()
        stack8b = run_stack8b_bench(dev)
        torch.cuda.empty_cache()

    prefill = prefill8 = None
    if rank == 0 and not args.no_prefill:
        del sd
        sd = None
        torch.cuda.empty_cache()
        prefill = run_prefill_bench(dev)
        torch.cuda.empty_cache()
        prefill8 = run_prefill_bench(dev, tier="8b")
    if oracle1_proc is not None:
        oracle1 = finish_oracle_one_thread(oracle1_proc)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": el_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int4 x int16 dp4a -> int32, f32 epilogue",
                "data": "synthetic",
                "config": {"workload": WORKLOAD if (args.route_k == 4 and not args.no_prerouter and args.layers == 40)
                           else WORKLOAD + " [variant: K=%d, prerouter %s, %d layers]" % (
                               args.route_k, "off" if args.no_prerouter else "on", args.layers),
                           "tokens_per_step": tps, "batch": 1,
                           "l2": "no flush: each token streams %.0f MB of weights, more than the 129 MB L2"
                                 % (nb["total"] / 1e6),
                           "kernel": {0: "persistent cooperative kernel, one launch per token",
                                      1: "per-phase kernel chain",
                                      3: "flag-carrying-word kernel (one CTA per SM, no grid barrier), one "
                                         "launch per token"}.get(args.kernel_impl)},
                "expert_weight_gbs": value * nb["routed"] / 1e9 / ws if ws else None,
                "weight_gbs": value * nb["total"] / 1e9 / ws if ws else None,
                "bytes_per_token": nb,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": traffic,
                             "kernel": kname, "launch_us": mean_launch_s * 1e6,
                             "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if pk else "fallback",
                             "peak_nominal": HBM_NOMINAL_GBS, "frac_nominal": achieved / HBM_NOMINAL_GBS},
                "cpu_baseline": cpu, "cpu_oracle_all_cores": cpu_all, "cpu_oracle_one_thread": oracle1, "e2e": e2e, "prefill": prefill,
                "prefill_8b": prefill8, "stack_8b": stack8b, "block_35b": block, "route_sweep": sweep,
                "streaming": streaming,
                "gpu_launches": n_timed * LAUNCHES_PER_TOKEN.get(args.kernel_impl, 6 * shape.n_layers + 1),
                "clocks": clocks, "device_status": st}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())

"""Device-resident weights for the C ABI: uploads the canonical tensors drawn
by ``synth``, packs experts into slot pools with e0_pack_experts and keeps the
ctypes descriptors (and the torch tensors they point into) alive.  PyTorch is
used for device memory and streams only; all arithmetic runs in libe0moe.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional

import numpy as np
import torch

from . import lib as L


def _dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device, non_blocking=False)


class DeviceQBank:
    """A layer's canonical stacked bank on the device (gate/up/down x codes/scale/bias)."""

    def __init__(self, bank_np: Dict[str, Dict[str, np.ndarray]], device="cuda"):
        self.t = {p: {k: _dev(v, device) for k, v in bank_np[p].items()} for p in ("gate", "up", "down")}
        self.E = self.t["gate"]["codes"].shape[0]

    def expert_q(self, e: int) -> L.ExpertQ:
        def q(p):
            d = self.t[p]
            return L.QTensor(d["codes"][e].data_ptr(), d["scale"][e].data_ptr(), d["bias"][e].data_ptr())
        return L.ExpertQ(q("gate"), q("up"), q("down"))


class SlotPoolDev:
    """n_slots experts in the kernel layout, a slot table [E] and an occupant
    table [n_slots] (all -1 until something is packed)."""

    def __init__(self, H: int, I: int, E: int, n_slots: int, device="cuda"):
        self.H, self.I, self.E, self.n_slots = H, I, E, n_slots
        self.slot_bytes = L.e0_slot_bytes(H, I)
        self.data = torch.empty(n_slots * self.slot_bytes, dtype=torch.uint8, device=device)
        self.table = torch.full((E,), -1, dtype=torch.int32, device=device)
        self.occupant = torch.full((n_slots,), -1, dtype=torch.int32, device=device)
        self.desc = L.SlotPool(self.data.data_ptr(), self.table.data_ptr(), self.occupant.data_ptr(),
                               n_slots, H, I, E)

    def pack(self, qbank: DeviceQBank, experts: List[int], slots: List[int], set_table=True, stream=None):
        src = [qbank.expert_q(e) for e in experts]
        L.e0_pack_experts(src, self.desc, slots, experts if set_table else None, stream=stream)

    @classmethod
    def resident(cls, bank_np, H, I, device="cuda", stream=None) -> "SlotPoolDev":
        """Every expert of a layer in slot e (identity table)."""
        qb = DeviceQBank(bank_np, device)
        pool = cls(H, I, qb.E, qb.E, device)
        ids = list(range(qb.E))
        pool.pack(qb, ids, ids, stream=stream)
        del qb
        return pool


class SharedDev:
    """Shared expert (one packed slot) plus its LoRA tensors."""

    def __init__(self, shared_np: dict, H: int, I: int, device="cuda", with_lora=True):
        qb = DeviceQBank({p: {k: v[None] for k, v in shared_np["q"][p].items()} for p in ("gate", "up", "down")},
                         device)
        self.pool = SlotPoolDev(H, I, 1, 1, device)
        self.pool.pack(qb, [0], [0])
        self.lora = None
        null = None
        if with_lora and shared_np.get("lora") is not None:
            self.lora = {p: {k: _dev(v, device) for k, v in shared_np["lora"][p].items()}
                         for p in ("gate", "up", "down")}
            lo = self.lora
            self.desc = L.SharedExpert(self.pool.data.data_ptr(),
                                       lo["gate"]["A"].data_ptr(), lo["gate"]["B"].data_ptr(),
                                       lo["up"]["A"].data_ptr(), lo["up"]["B"].data_ptr(),
                                       lo["down"]["A"].data_ptr(), lo["down"]["B"].data_ptr(),
                                       int(shared_np["rank"]), float(shared_np["alpha"]))
        else:
            self.desc = L.SharedExpert(self.pool.data.data_ptr(), null, null, null, null, null, null, 0, 0.0)


class HeadDev:
    def __init__(self, head_np: dict, H: int, E: int, device="cuda"):
        self.t = {k: _dev(v, device) for k, v in head_np.items() if v is not None}
        hidden = self.t["fc1"].shape[0]
        g = lambda k: self.t[k].data_ptr() if k in self.t else None  # noqa: E731
        self.desc = L.Prerouter(g("fc1"), g("b1"), g("fc2"), g("b2"), g("lres"), H, E, hidden)
        self.hidden = hidden


class StackDev:
    """A whole decode stack on the device plus its workspace and optional trace."""

    def __init__(self, model, device="cuda", trace=False, with_lora=True):
        sh = model.shape
        s = sh.layer
        self.shape = sh
        self.H, self.I, self.E, self.K = s.H, s.I, s.E, s.K
        self.L = len(model.banks)
        self.pools = [SlotPoolDev.resident(b, s.H, s.I, device) for b in model.banks]
        self.routers = [_dev(w, device) for w in model.routers]
        self.heads = {l: HeadDev(h, s.H, s.E, device) for l, h in model.heads.items()}
        self.shared = [SharedDev(x, s.H, s.I, device, with_lora) if x is not None else None for x in model.shared]
        hidden = max([h.hidden for h in self.heads.values()], default=0)
        self._sh_descs = [C.pointer(x.desc) if x is not None else None for x in self.shared]
        self._hd_descs = {l: C.pointer(h.desc) for l, h in self.heads.items()}
        consumers = set(sh.consumers)
        layers = []
        for l in range(self.L):
            layers.append(L.StackLayer(self.pools[l].desc, self.routers[l].data_ptr(),
                                       self._sh_descs[l] if self._sh_descs[l] is not None else None,
                                       self._hd_descs.get(l), 1 if (l in consumers and (l - 1) in self.heads) else 0))
        self.layers = layers
        self.rp = L.route_params(0 if s.route == "softmax_topk" else 1, s.K, s.n_groups, s.topk_groups,
                                 s.route_scale)
        self.ws_bytes = L.e0_stack_workspace_size(self.L, s.H, s.I, s.E, s.K, hidden)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.r_out = torch.empty(s.H, dtype=torch.float32, device=device)
        self.trace = None
        if trace:
            self.tr = {"r": torch.zeros((self.L + 1, s.H), dtype=torch.float32, device=device),
                       "inds": torch.full((self.L, s.K), -1, dtype=torch.int32, device=device),
                       "w": torch.zeros((self.L, s.K), dtype=torch.float32, device=device),
                       "head_logits": torch.zeros((self.L, s.E), dtype=torch.float32, device=device),
                       "pred_inds": torch.full((self.L, s.K), -1, dtype=torch.int32, device=device)}
            self.trace = L.StackTrace(*[self.tr[k].data_ptr() for k in ("r", "inds", "w", "head_logits",
                                                                           "pred_inds")])
        self.prepare()

    def variant(self, K: Optional[int] = None, prerouter: bool = True, device="cuda") -> "StackDev":
        """The same device weights with another routed-expert count K and/or
        without the prerouter heads (every layer then routes with its own
        router); its own workspace and status word, no trace."""
        import copy
        v = copy.copy(self)
        s = self.shape.layer
        v.K = self.K if K is None else int(K)
        consumers = set(self.shape.consumers) if prerouter else set()
        heads = self._hd_descs if prerouter else {}
        v.layers = [L.StackLayer(self.pools[l].desc, self.routers[l].data_ptr(),
                                 self._sh_descs[l] if self._sh_descs[l] is not None else None,
                                 heads.get(l), 1 if (l in consumers and (l - 1) in heads) else 0)
                    for l in range(self.L)]
        v.rp = L.route_params(0 if s.route == "softmax_topk" else 1, v.K, s.n_groups, s.topk_groups, s.route_scale)
        hidden = max([h.hidden for h in self.heads.values()], default=0) if prerouter else 0
        v.ws_bytes = L.e0_stack_workspace_size(self.L, s.H, s.I, s.E, v.K, hidden)
        v.ws = torch.empty(v.ws_bytes, dtype=torch.uint8, device=device)
        v.status = torch.zeros(1, dtype=torch.int32, device=device)
        v.r_out = torch.empty(s.H, dtype=torch.float32, device=device)
        v.trace = None
        v.prepare()
        return v

    def prepare(self, stream=None):
        L.e0_stack_prepare(self.layers, self.H, self.I, self.E, self.rp, self.ws, self.ws_bytes, stream=stream)

    def step(self, x: torch.Tensor, impl: int = 0, stream=None, out: Optional[torch.Tensor] = None):
        out = self.r_out if out is None else out
        L.e0_stack_step(x, out, self.ws, self.trace, impl, self.status, stream=stream)
        return out


class ExpertCacheDev:
    """A cross-layer cache of `capacity` expert bundles in device memory (keys
    layer * E + expert), least recently used first out."""

    def __init__(self, capacity: int, n_layers: int, H: int, I: int, E: int, device="cuda"):
        self.capacity = capacity
        sb = L.e0_slot_bytes(H, I)
        self.data = torch.empty(max(capacity, 1) * sb, dtype=torch.uint8, device=device)
        self.key = torch.full((max(capacity, 1),), -1, dtype=torch.int32, device=device)
        self.stamp = torch.zeros(max(capacity, 1), dtype=torch.int32, device=device)
        self.map = torch.full((n_layers * E,), -1, dtype=torch.int32, device=device)
        self.counters = torch.zeros(4, dtype=torch.int32, device=device)
        self.scratch = torch.zeros(4 + 4 * 32, dtype=torch.int32, device=device)
        self.desc = L.ExpertCache(self.data.data_ptr(), self.key.data_ptr(), self.stamp.data_ptr(),
                                  self.map.data_ptr(), self.counters.data_ptr(), self.scratch.data_ptr(),
                                  capacity, n_layers * E)

    def stats(self) -> dict:
        c = self.counters.cpu().tolist()
        return {"hits": c[1], "misses": c[2], "evictions": c[3]}


class StreamedStack:
    """Host-tier staged streaming on top of a StackDev (flag-carrying-word kernel).

    Each staged layer keeps its experts (kernel layout) in pinned host memory
    and only 2K slots in device memory.  A token runs as two launches, layers
    [0, split) and [split, L); the experts the prerouter predicted for the next
    token are copied host -> device by e0_stack_prefetch_experts on a second
    stream: layers below split - 1 while the second half of the token runs,
    layers from split on while the first half of the next token runs.  Layer
    split - 1, whose prediction is final only once the token has ended but
    which the next token's first half uses, stays in the resident bank, as do
    the layers that route natively.  With an ExpertCacheDev the copies first
    look in a cross-layer cache of recently used bundles in device memory.

    The decode launches leave ``free_sms`` SMs to the copy kernels, which run
    on that many blocks: a cooperative launch over every SM would wait for a
    running copy kernel instead of overlapping it.  The layers of one half
    are prefetched with one batched call (``batched=False``: one call per
    layer, the same slot contents)."""

    def __init__(self, sd: "StackDev", split: int, device="cuda", cache: Optional["ExpertCacheDev"] = None,
                 host: Optional[dict] = None, free_sms: int = 24, batched: bool = True):
        self.batched = batched
        import os
        old = os.environ.get("E0MOE_LL_FREE_SMS")
        os.environ["E0MOE_LL_FREE_SMS"] = str(int(free_sms))
        try:
            sd.prepare()
        finally:
            if old is None:
                del os.environ["E0MOE_LL_FREE_SMS"]
            else:
                os.environ["E0MOE_LL_FREE_SMS"] = old
        self.sd = sd
        self.split = split
        self.cache = cache
        consumers = [l for l in range(sd.L) if sd.layers[l].consumer]
        self.batch1 = [l for l in consumers if l <= split - 2]
        self.batch2 = [l for l in consumers if l >= split]
        self.staged = self.batch1 + self.batch2
        self.host = {}
        self.pools = {}
        n_slots = 2 * sd.K
        for l in self.staged:
            if host is not None and l in host:  # the pinned copies of an earlier run of the same stack
                self.host[l] = host[l]
            else:
                src = sd.pools[l].data
                h = torch.empty(src.shape, dtype=torch.uint8, pin_memory=True)
                h.copy_(src)
                self.host[l] = h
            self.pools[l] = SlotPoolDev(sd.H, sd.I, sd.E, n_slots, device)
        torch.cuda.synchronize()
        self.cs = torch.cuda.Stream()
        self.ps = torch.cuda.Stream()
        self.ev1 = torch.cuda.Event()
        self.ev2 = torch.cuda.Event()
        self.status = sd.status
        self.t = 0

    def copy_bytes_per_expert(self) -> int:
        return L.e0_slot_bytes(self.sd.H, self.sd.I)

    def _prefetch(self, layers, t_next, stream):
        if not self.batched:
            for l in layers:
                if self.cache is None:
                    L.e0_stack_prefetch_experts(self.sd.ws, l, t_next, self.pools[l].desc, self.host[l], self.status,
                                                stream=stream)
                else:
                    L.e0_stack_prefetch_experts_cached(self.sd.ws, l, t_next, self.pools[l].desc, self.host[l],
                                                       self.cache.desc, self.status, stream=stream)
            return
        # every layer of the batch in one copy launch and one commit launch
        pools = [self.pools[l].desc for l in layers]
        banks = [self.host[l] for l in layers]
        if self.cache is None:
            L.e0_stack_prefetch_experts_batch(self.sd.ws, layers, t_next, pools, banks, self.status, stream=stream)
        else:
            L.e0_stack_prefetch_experts_cached_batch(self.sd.ws, layers, t_next, pools, banks, self.cache.desc,
                                                     self.status, stream=stream)

    def start(self, x0: torch.Tensor, out: Optional[torch.Tensor] = None):
        """Token 0 (every layer routes natively) from the resident bank, then the
        staged layers switch to their slot pools holding the predicted experts
        of token 1."""
        sd = self.sd
        out = sd.r_out if out is None else out
        with torch.cuda.stream(self.cs):
            L.e0_stack_step_range(x0, out, sd.ws, 0, sd.L, sd.trace, self.status, stream=self.cs)
            self._prefetch(self.staged, 1, self.cs)
        self.cs.synchronize()
        layers = list(sd.layers)
        for l in self.staged:
            layers[l] = L.StackLayer(self.pools[l].desc, layers[l].W_router, layers[l].shared, layers[l].head,
                                     layers[l].consumer)
        L.e0_stack_update_layers(sd.ws, layers, stream=self.cs)
        self.layers = layers
        self.ev1.record(self.cs)
        self.ev2.record(self.cs)
        self.t = 1
        return out

    def step(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, overlap: bool = True):
        """Token self.t; the copies for token self.t + 1 are issued behind it."""
        sd = self.sd
        out = sd.r_out if out is None else out
        t = self.t
        cs, ps = self.cs, (self.ps if overlap else self.cs)
        cs.wait_event(self.ev1)
        L.e0_stack_step_range(x, None, sd.ws, 0, self.split, sd.trace, self.status, stream=cs)
        ev_a = torch.cuda.Event()
        ev_a.record(cs)
        ps.wait_event(ev_a)
        self._prefetch(self.batch1, t + 1, ps)
        self.ev1.record(ps)
        cs.wait_event(self.ev2)
        L.e0_stack_step_range(None, out, sd.ws, self.split, sd.L, sd.trace, self.status, stream=cs)
        ev_b = torch.cuda.Event()
        ev_b.record(cs)
        ps.wait_event(ev_b)
        self._prefetch(self.batch2, t + 1, ps)
        self.ev2.record(ps)
        self.t = t + 1
        return out

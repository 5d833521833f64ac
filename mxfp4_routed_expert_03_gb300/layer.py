"""Buffer bookkeeping around the C ABI for one routed layer.

Holds torch-owned device buffers (weights, plan, workspace) and calls the C
entry points; it computes nothing itself.
"""
from __future__ import annotations

import torch

from . import (MOE_OP_DECODE, MOE_OP_FORWARD, MOE_OP_PLAN, MOE_ROUTER_XWR, check, moe_create,
               moe_create_streaming, moe_create_streaming_store, moe_decode, moe_desc,
               moe_destroy, moe_forward, moe_plan, moe_plan_buf, moe_prepare, moe_prepared_bytes,
               moe_router_logits, moe_status, moe_store, moe_store_blob_bound, moe_store_encode,
               moe_store_tiles_per_expert, moe_stream_state_bytes, moe_stream_stats, moe_weights,
               moe_workspace_bytes)

WEIGHT_NAMES = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def alloc_weights(E: int, D: int, F: int, device="cuda") -> dict:
    """Uninitialised uint8 weight tensors in the library's layout."""
    return {
        "gate_q": torch.empty((E, F, D // 2), dtype=torch.uint8, device=device),
        "gate_s": torch.empty((E, F, D // 32), dtype=torch.uint8, device=device),
        "up_q": torch.empty((E, F, D // 2), dtype=torch.uint8, device=device),
        "up_s": torch.empty((E, F, D // 32), dtype=torch.uint8, device=device),
        "down_q": torch.empty((E, D, F // 2), dtype=torch.uint8, device=device),
        "down_s": torch.empty((E, D, F // 32), dtype=torch.uint8, device=device),
    }


def alloc_fp8_weights(E: int, D: int, F: int, device="cuda") -> dict:
    """Uninitialised FP8 expert tensors: E4M3FN codes (uint8) and fp32 scales
    per 128 x 128 block, in the library's layout."""
    nb = lambda n: (n + 127) // 128
    return {
        "gate_q": torch.empty((E, F, D), dtype=torch.uint8, device=device),
        "gate_s": torch.empty((E, nb(F), nb(D)), dtype=torch.float32, device=device),
        "up_q": torch.empty((E, F, D), dtype=torch.uint8, device=device),
        "up_s": torch.empty((E, nb(F), nb(D)), dtype=torch.float32, device=device),
        "down_q": torch.empty((E, D, F), dtype=torch.uint8, device=device),
        "down_s": torch.empty((E, nb(D), nb(F)), dtype=torch.float32, device=device),
    }


class Plan:
    def __init__(self, T: int, E: int, k: int, device="cuda"):
        dev = device
        self.T, self.E, self.k = T, E, k
        n = max(T * k, 1)
        self.topk_idx = torch.empty((max(T, 1), k), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((max(T, 1), k), dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.perm = torch.empty(n, dtype=torch.int32, device=dev)
        self.inv = torch.empty(n, dtype=torch.int32, device=dev)
        self.active = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.buf = moe_plan_buf(*[t.data_ptr() for t in (self.topk_idx, self.topk_w, self.counts,
                                                         self.offsets, self.perm, self.inv,
                                                         self.active)])


class Layer:
    """One routed layer: weights (device tensors) + the library handle."""

    def __init__(self, D: int, F: int, E: int, k: int, weights: dict, router_mode: int = 0,
                 w_router=None, shared=None, act_mode: int = 0, weight_format: int = 0):
        self.D, self.F, self.E, self.k = D, F, E, k
        self.router_mode = router_mode
        self.weights = weights
        self.w_router = w_router
        self.shared = shared
        ptr = lambda t: None if t is None else t.data_ptr()
        sh = shared or {}
        self.desc = moe_desc(D, F, E, k, router_mode, 1 if shared else 0, act_mode, weight_format)
        self.wdesc = moe_weights(*[weights[n].data_ptr() for n in WEIGHT_NAMES], ptr(w_router),
                                 ptr(sh.get("sh_gate")), ptr(sh.get("sh_up")),
                                 ptr(sh.get("sh_down")))
        self.h = moe_create(self.desc, self.wdesc)
        self._ws = None
        self.atoms = None

    def prepare(self, stream=None) -> None:
        """One-time weight-scale re-layout (and W_r split) for the tensor-core paths."""
        if self.atoms is None:
            n = moe_prepared_bytes(self.h)
            self.atoms = torch.empty(n, dtype=torch.uint8, device="cuda")
            check(moe_prepare(self.h, self.atoms, n, stream), "moe_prepare")

    def close(self):
        if self.h:
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, T: int, op: int) -> tuple:
        n = moe_workspace_bytes(self.h, T, op)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
        return self._ws, n

    def router_logits(self, T, x, logits, stream=None) -> int:
        self.prepare(stream)
        return moe_router_logits(self.h, T, x, logits, stream)

    def plan(self, T, logits, x, plan: Plan, stream=None) -> int:
        if self.router_mode == MOE_ROUTER_XWR:
            self.prepare(stream)
        ws, n = self.workspace(T, MOE_OP_PLAN)
        return moe_plan(self.h, T, logits, x, plan.buf, ws, ws.numel(), stream)

    def decode(self, T, x, plan: Plan, out, stream=None) -> int:
        ws, n = self.workspace(T, MOE_OP_DECODE)
        return moe_decode(self.h, T, x, plan.buf, out, ws, ws.numel(), stream)

    def forward(self, T, x, plan: Plan, out, stream=None) -> int:
        self.prepare(stream)
        ws, n = self.workspace(T, MOE_OP_FORWARD)
        return moe_forward(self.h, T, x, plan.buf, out, ws, ws.numel(), stream)

    def status(self, stream=None) -> int:
        return moe_status(self.h, stream)


class ExpertStore:
    """The compressed expert store of a layer: blob in pinned host memory,
    tile records and frequency tables on the device, built by the library's
    host encoder from host weight arrays (CPU tensors or numpy arrays in the
    library's layouts)."""

    def __init__(self, E: int, D: int, F: int, host_weights: dict, n_threads: int = 0,
                 device="cuda"):
        import numpy as np
        self.E, self.D, self.F = E, D, F
        self.tpe = moe_store_tiles_per_expert(D, F)
        cap = moe_store_blob_bound(E, D, F)
        if self.tpe <= 0 or cap <= 0:
            raise ValueError("bad layer shape for a store")
        arrays = {n: host_weights[n] for n in WEIGHT_NAMES}
        ptrs = []
        for n in WEIGHT_NAMES:
            a = arrays[n]
            ptrs.append(a.data_ptr() if isinstance(a, torch.Tensor) else a.ctypes.data)
        hw = moe_weights(*ptrs, None, None, None, None)
        blob = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
        tiles = np.zeros((E, self.tpe, 8), np.uint32)
        tables = np.zeros((E, 6, 256), np.uint16)
        self.blob_bytes = moe_store_encode(E, D, F, hw, blob.data_ptr(), cap, tiles.ctypes.data,
                                           tables.ctypes.data, n_threads)
        self.blob = blob
        self.raw_bytes = sum(int(arrays[n].numel() if isinstance(arrays[n], torch.Tensor)
                                 else arrays[n].size) for n in WEIGHT_NAMES)
        self.tiles = torch.from_numpy(tiles).to(device)
        self.tables = torch.from_numpy(tables.view(np.int16)).to(device)
        self.records = tiles

    def desc(self) -> moe_store:
        return moe_store(self.blob.data_ptr(), self.blob_bytes, self.tiles.data_ptr(),
                         self.tables.data_ptr())


class StreamingLayer(Layer):
    """A routed layer whose experts stay in pinned host memory; the library
    keeps an HBM cache of n_slots of them (expert streaming). host_weights:
    CPU tensors in the library's layouts, pinned (tensor.pin_memory())."""

    def __init__(self, D: int, F: int, E: int, k: int, host_weights: dict | None, n_slots: int,
                 router_mode: int = 0, w_router=None, shared=None, store: ExpertStore | None = None,
                 act_mode: int = 0):
        """host_weights: pinned CPU tensors of all experts, or None with `store`
        (an ExpertStore): the misses are then decoded from the store."""
        self.D, self.F, self.E, self.k = D, F, E, k
        self.router_mode = router_mode
        self.host_weights = host_weights
        self.store = store
        self.n_slots = n_slots
        self.weights = alloc_weights(n_slots, D, F)  # the slot cache
        self.w_router = w_router
        self.shared = shared
        ptr = lambda t: None if t is None else t.data_ptr()
        sh = shared or {}
        self.desc = moe_desc(D, F, E, k, router_mode, 1 if shared else 0, act_mode)
        self.wdesc = moe_weights(*[self.weights[n].data_ptr() for n in WEIGHT_NAMES],
                                 ptr(w_router), ptr(sh.get("sh_gate")), ptr(sh.get("sh_up")),
                                 ptr(sh.get("sh_down")))
        self.state = torch.empty(moe_stream_state_bytes(E, n_slots), dtype=torch.uint8,
                                 device="cuda")
        if store is not None:
            self.sdesc = store.desc()
            self.h = moe_create_streaming_store(self.desc, self.sdesc, self.wdesc, n_slots,
                                                self.state)
        else:
            self.hdesc = moe_weights(*[host_weights[n].data_ptr() for n in WEIGHT_NAMES], None,
                                     None, None, None)
            self.h = moe_create_streaming(self.desc, self.hdesc, self.wdesc, n_slots, self.state)
        self._ws = None
        self.atoms = None

    def stats(self, stream=None) -> tuple:
        """(hits, misses, misses of the last call)."""
        return moe_stream_stats(self.h, stream)

    def cache_state(self) -> dict:
        """slot_of [E] and expert_of / stamp [S] read back from the device."""
        import numpy as np
        raw = self.state.cpu().numpy()
        words = raw[32:].view(np.int32)
        E, S = self.E, self.n_slots
        return {"clock": int(raw[:4].view(np.int32)[0]), "slot_of": words[:E].copy(),
                "expert_of": words[E:E + S].copy(), "stamp": words[E + S:E + 2 * S].copy()}

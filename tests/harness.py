"""Shared helpers of the GPU parity tests (inputs from synth, expected values
from the CPU oracle, outputs through the C ABI)."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Normwise reading of "max relative error 2e-2, mean absolute error 1e-3",
# measured against the oracle's largest output magnitude.
MAX_REL = 2e-2
MAE_REL = 1e-3


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return a.view(np.float32).astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    scale = float(np.abs(ref).max())
    err = np.abs(got - ref)
    return {"max_rel": float(err.max() / scale), "mae_rel": float(err.mean() / scale),
            "max_abs": float(err.max()), "mae_abs": float(err.mean()), "scale": scale}


def assert_close(got: np.ndarray, ref: np.ndarray, max_rel=MAX_REL, mae_rel=MAE_REL) -> dict:
    e = errors(got, ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    assert e["max_rel"] <= max_rel and e["mae_rel"] <= mae_rel, e
    return e


def to_dev_bf16(x_np: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).to(device)


def host_layer_weights(w: synth.Workload, device="cuda") -> dict:
    """Whole layer generated on the host (small layers only)."""
    from mxfp4_routed_expert_03_gb300.layer import alloc_weights
    weights = alloc_weights(w.E, w.D, w.F, device)
    for e in range(w.E):
        for name, arr in synth.expert_weights(w.seed, e, w.D, w.F, dist=w.codes).items():
            weights[name][e].copy_(torch.from_numpy(arr))
    return weights


def device_layer_weights(w: synth.Workload, device="cuda") -> dict:
    """Whole layer generated on the GPU by the device half of the generator."""
    from mxfp4_routed_expert_03_gb300.layer import alloc_weights
    weights = alloc_weights(w.E, w.D, w.F, device)
    synth.dev_fill_layer(w.seed, w.E, w.D, w.F, {k: v.data_ptr() for k, v in weights.items()},
                         torch.cuda.current_stream().cuda_stream, dist=w.codes)
    torch.cuda.synchronize()
    return weights


def router_and_shared(w: synth.Workload, shared: bool = True, device="cuda"):
    """Device copies of the workload's fp32 W_r [E][D] and bf16 shared expert (host-generated)."""
    wr = torch.from_numpy(synth.make_w_router(w)).to(device)
    if not shared:
        return wr, None
    sh = {k: to_dev_bf16(v, device) for k, v in synth.make_shared(w).items()}
    return wr, sh

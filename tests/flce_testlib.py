"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, and compare with the CPU oracle at the
tolerances of the numerics gate (loss rel 1e-3, per-token lse abs 2e-3, dH and
dW relative Frobenius 5e-3)."""
from __future__ import annotations

import numpy as np

import flce_inputs

TOL_LOSS_REL = 1e-3
TOL_LSE_ABS = 2e-3
TOL_GRAD_FRO = 5e-3


def to_device(Hb, Wb, y, dev="cuda:0"):
    import torch
    H = torch.from_numpy(np.ascontiguousarray(Hb).view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(np.ascontiguousarray(Wb).view(np.int16)).to(dev).view(torch.bfloat16)
    lab = torch.from_numpy(np.ascontiguousarray(y, dtype=np.int32)).to(dev)
    return H, W, lab


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return flce_inputs.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def tensor_to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_tensor_to_f64(t)
    return t.double().cpu().numpy()


def rel_fro(a, b) -> float:
    nb = float(np.linalg.norm(b))
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def compare(res, ref, dh_rows=None, dw_rows=None) -> dict:
    loss = float(res.loss.item())
    lse = res.lse.double().cpu().numpy()
    out = {"loss_gpu": loss, "loss_ref": ref["loss"]}
    out["loss_rel"] = abs(loss - ref["loss"]) / max(abs(ref["loss"]), 1e-30) if ref["loss"] else abs(loss)
    out["lse_abs"] = float(np.max(np.abs(lse - ref["lse"])))
    if res.dH is not None and ref["dH"] is not None:
        dH = tensor_to_f64(res.dH if dh_rows is None else res.dH[dh_rows])
        out["dH_fro"] = rel_fro(dH, ref["dH"])
    if res.dW is not None and ref["dW"] is not None:
        dW = tensor_to_f64(res.dW if dw_rows is None else res.dW[dw_rows])
        out["dW_fro"] = rel_fro(dW, ref["dW"])
    return out


def assert_within(errs: dict):
    assert errs["loss_rel"] <= TOL_LOSS_REL, errs
    assert errs["lse_abs"] <= TOL_LSE_ABS, errs
    if "dH_fro" in errs:
        assert errs["dH_fro"] <= TOL_GRAD_FRO, errs
    if "dW_fro" in errs:
        assert errs["dW_fro"] <= TOL_GRAD_FRO, errs

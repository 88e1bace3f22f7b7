"""Helpers shared by the GPU tests: move a workload to the device, run the
CUDA path through the C ABI, compare with the oracle at the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import mla_sparse_top_gb300 as mla
import workloads

# tolerance: rtol 0.005 / atol 0.0001 on the bf16 output (the operator spec's
# precision standard), 1e-3 relative on the fp32 lse
RTOL, ATOL = 5e-3, 1e-4
LSE_RTOL, LSE_ATOL = 1e-3, 1e-5


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_device(inp: dict, device="cuda") -> dict:
    return workloads.to_device(inp, device)


def dims_of(inp: dict) -> "mla.MlaDims":
    return mla.dims_from_workload(inp["dims"])


def launch(inp: dict, dev: dict, mode=None):
    mla.mla_sparse_attn_fwd(dev["q_nope"], dev["q_rope"], dev["kv_nope"], dev["kv_rope"], dev["kv_scales"],
                            dev["topk_idx"], dev["block_table"], dev["act_seqs"], dev["out"], dev["lse"],
                            softmax_scale=inp["softmax_scale"], mode=inp.get("mode", "decode") if mode is None else mode,
                            dims=dims_of(inp))


def run_gpu(inp: dict, mode=None, dev=None):
    """Returns (out fp64 (T, H, 512), lse fp64 (T, H), status bits)."""
    if dev is None:
        dev = to_device(inp)
    dev["out"].fill_(float("nan"))
    dev["lse"].fill_(float("nan"))
    launch(inp, dev, mode)
    status = mla.device_status(clear=True)
    torch.cuda.synchronize()
    out = bf16_to_f64(dev["out"].view(torch.int16).cpu().numpy().view(np.uint16))
    lse = dev["lse"].cpu().numpy().astype(np.float64)
    return out, lse, status


def assert_out_close(g, o, label=""):
    err = np.abs(g - o)
    bound = ATOL + RTOL * np.abs(o)
    bad = ~(err <= bound)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.nanargmax(np.where(np.isfinite(err), err / bound, np.inf))
        raise AssertionError(f"{label}: {int(bad.sum())}/{bad.size} out elements outside rtol {RTOL}/atol {ATOL}; "
                             f"first {idx.tolist()}; worst gpu={g.flat[worst]!r} oracle={o.flat[worst]!r}")


def assert_lse_close(g, o, label=""):
    both_inf = np.isneginf(g) & np.isneginf(o)
    # the difference is taken only where it is defined (-inf - -inf is not)
    err = np.abs(np.where(both_inf, 0.0, g) - np.where(both_inf, 0.0, o))
    bound = LSE_ATOL + LSE_RTOL * np.abs(np.where(both_inf, 0.0, o))
    bad = ~(both_inf | (err <= bound))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{label}: {int(bad.sum())}/{bad.size} lse values outside 1e-3 relative; first {idx.tolist()} "
                             f"gpu={g[tuple(idx[0])]!r} oracle={o[tuple(idx[0])]!r}")

"""Helpers shared by the GPU tests: move a workload to the device, run the
CUDA path through the C ABI, compare with the oracle at the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import mla_sparse_top_gb300 as mla

# tolerance: rtol 0.005 / atol 0.0001 on the bf16 output (the operator spec's
# precision standard), 1e-3 relative on the fp32 lse
RTOL, ATOL = 5e-3, 1e-4
LSE_RTOL, LSE_ATOL = 1e-3, 1e-5


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_device(inp: dict, device="cuda") -> dict:
    d = inp["dims"]
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    dev = dict(
        q_nope=bf(inp["q_nope"]),
        q_rope=bf(inp["q_rope"]),
        kv_nope=(torch.from_numpy(np.ascontiguousarray(inp["kv_nope"])).to(device) if d["kv_int8"] else bf(inp["kv_nope"])),
        kv_rope=bf(inp["kv_rope"]),
        kv_scales=(torch.from_numpy(np.ascontiguousarray(inp["kv_scales"])).to(device) if d["kv_int8"] else None),
        topk_idx=torch.from_numpy(np.ascontiguousarray(inp["topk_idx"])).to(device),
        block_table=torch.from_numpy(np.ascontiguousarray(inp["block_table"])).to(device),
        act_seqs=torch.from_numpy(np.ascontiguousarray(inp["act_seqs"])).to(device),
    )
    T, H = d["B"] * d["S1"], d["n_q"]
    dev["out"] = torch.empty((T, H, d["d_nope"]), dtype=torch.bfloat16, device=device)
    dev["lse"] = torch.empty((T, H), dtype=torch.float32, device=device)
    return dev


def dims_of(inp: dict) -> "mla.MlaDims":
    d = inp["dims"]
    return mla.MlaDims(B=d["B"], S1=d["S1"], n_q=d["n_q"], n_kv=d["n_kv"], d_nope=d["d_nope"], d_rope=d["d_rope"],
                       block_size=d["block_size"], num_blocks=d["num_blocks"],
                       max_blocks_per_seq=d["max_blocks_per_seq"], topk=d["topk"],
                       kv_dtype=mla.MLA_KV_INT8 if d["kv_int8"] else mla.MLA_KV_BF16)


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
    err = np.abs(g - o)
    bound = LSE_ATOL + LSE_RTOL * np.abs(o)
    bad = ~(both_inf | (err <= bound))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{label}: {int(bad.sum())}/{bad.size} lse values outside 1e-3 relative; first {idx.tolist()} "
                             f"gpu={g[tuple(idx[0])]!r} oracle={o[tuple(idx[0])]!r}")

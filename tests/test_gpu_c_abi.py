"""The C ABI on its own: a plain C program (tests/c_abi/attn_from_file.c,
compiled here with gcc against include/mla_sparse.h and the CUDA runtime, no
Python or torch in it) runs mla_sparse_attn_fwd on seeded inputs written to a
file, and its out / lse match the oracle at the operator's tolerance."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import assert_lse_close, assert_out_close, bf16_to_f64

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def compile_caller(tmp_path):
    from mla_sparse_top_gb300 import build
    lib = build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "attn_from_file")
    cmd = ["gcc", "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", "attn_from_file.c"), "-o", exe,
           "-L", os.path.dirname(lib), "-lmla_sparse", "-Wl,-rpath," + os.path.dirname(lib),
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


def write_problem(inp, path, mode=0):
    d = inp["dims"]
    with open(path, "wb") as f:
        np.array([d["B"], d["S1"], d["n_q"], d["num_blocks"], d["max_blocks_per_seq"], d["topk"], d["kv_int8"], mode,
                  0, 0, 0], dtype=np.int32).tofile(f)
        np.array([inp["softmax_scale"]], dtype=np.float32).tofile(f)
        for key in ("q_nope", "q_rope", "kv_nope", "kv_rope"):
            np.ascontiguousarray(inp[key]).tofile(f)
        if d["kv_int8"]:
            np.ascontiguousarray(inp["kv_scales"], dtype=np.float32).tofile(f)
        for key in ("topk_idx", "block_table", "act_seqs"):
            np.ascontiguousarray(inp[key], dtype=np.int32).tofile(f)


@pytest.mark.parametrize("kv_int8", [False, True])
def test_plain_c_caller_matches_the_oracle(tmp_path, kv_int8):
    exe = compile_caller(tmp_path)
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[700, 1500], topk=300, seed=50, kv_int8=kv_int8)
    src, dst = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    write_problem(inp, src)
    subprocess.run([exe, src, dst], check=True)
    d = inp["dims"]
    T, H = d["B"] * d["S1"], d["n_q"]
    raw = np.fromfile(dst, dtype=np.uint8)
    out = bf16_to_f64(raw[: T * H * 512 * 2].view(np.uint16)).reshape(T, H, 512)
    lse = raw[T * H * 512 * 2:].view(np.float32).astype(np.float64).reshape(T, H)
    ref_out, ref_lse, _ = oracle.forward(inp)
    assert_out_close(out, ref_out, "C caller")
    assert_lse_close(lse, ref_lse, "C caller")

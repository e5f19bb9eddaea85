"""The library driven from a plain C program through include/moe_ffn.h alone
(no Python binding, no PyTorch on the call path): the program is compiled and
linked against libmoe_ffn.so on the CPU (not gpu-marked), and on a GPU its
output is compared with the oracle at the bf16 parity tolerances, through
device buffers and through the host-buffer entry point."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import grouped_gemm_gb300 as moe
from grouped_gemm_gb300 import build as libbuild
from grouped_gemm_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "forward_from_c.c")


def compile_program(tmp_path):
    lib = moe.library_path() if os.path.exists(moe.library_path()) else libbuild.build()
    exe = str(tmp_path / "forward_from_c")
    cuda = os.path.dirname(os.path.dirname(libbuild.nvcc()))
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", SRC, "-o", exe, "-I", libbuild.INCLUDE,
           "-I", os.path.join(cuda, "include"), "-L", os.path.dirname(lib), "-lmoe_ffn",
           f"-Wl,-rpath,{os.path.dirname(lib)}", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    assert os.path.exists(compile_program(tmp_path))


@pytest.mark.gpu
@pytest.mark.parametrize("host_chunk", [None, 64])   # device buffers; host buffers in chunks of 64 tokens
@pytest.mark.parametrize("pipeline", [0, 1])
def test_c_program_matches_oracle(tmp_path, pipeline, host_chunk):
    import oracle
    from helpers import assert_close
    import torch

    exe = compile_program(tmp_path)
    T, D, H, E, k = 200, 512, 256, 16, 4
    inp = wl.make_custom(T, D, H, E, k, seed=77, routing="uniform")
    for name, arr in (("x", inp["x"]), ("w1", inp["w1"]), ("w2", inp["w2"]),
                      ("ids", np.ascontiguousarray(inp["topk_ids"], np.int32)),
                      ("w", np.ascontiguousarray(inp["topk_w"], np.float32))):
        arr.tofile(str(tmp_path / f"{name}.bin"))
    argv = [exe, str(tmp_path), str(T), str(E), str(D), str(H), str(k), str(pipeline)]
    if host_chunk is not None:
        argv.append(str(host_chunk))
    r = subprocess.run(argv, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out_bits = np.fromfile(str(tmp_path / "out.bin"), dtype=np.uint16).reshape(T, D)
    out = torch.from_numpy(out_bits.view(np.int16)).view(torch.bfloat16)
    ref = oracle.moe_ffn(inp["x"], inp["w1"], inp["w2"], inp["topk_ids"], inp["topk_w"], act=oracle.ACT_BF16)
    assert_close(out, ref, label=f"C program pipeline={pipeline} host_chunk={host_chunk}")

"""The C ABI used from a plain C program (tests/c/forward_from_c.c): it is
valid C, links against the library and the CUDA runtime, and on a GPU its
forward equals the Python binding's bit for bit and the oracle's within the
layer tolerance."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import moe_synth
from gpu_util import assert_y_close, bf16_bits_to_float

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "forward_from_c.c")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _compile(out_dir):
    from moe_expert_ffn_gb300 import build
    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    libdir = os.path.dirname(lib)
    exe = os.path.join(out_dir, "forward_from_c")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-lmoe_gb300", "-Wl,-rpath," + libdir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(str(tmp_path)))


@pytest.mark.gpu
def test_c_program_forward_matches_binding_and_oracle(tmp_path, orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(str(tmp_path))
    wl = moe_synth.custom(T=96, H=512, I=256, E=8, k=2, seed=91, name="c_program")
    inp = moe_synth.make_inputs(wl)
    bundle = os.path.join(str(tmp_path), "bundle.bin")
    with open(bundle, "wb") as fh:
        fh.write(np.array([wl.T, wl.H, wl.I, wl.E, wl.k], dtype=np.int32).tobytes())
        for n in ("x", "x_sf", "topk_idx", "topk_weights", "w1", "w1_sf", "w2", "w2_sf"):
            fh.write(inp[n].contiguous().numpy().tobytes())
    y_path = os.path.join(str(tmp_path), "y.bin")
    r = subprocess.run([exe, bundle, y_path], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    y_bits = np.fromfile(y_path, dtype=np.uint16).reshape(wl.T, wl.H)

    import moe_expert_ffn_gb300 as m
    dev = torch.device("cuda:0")
    layer = m.MoELayer(wl.T, wl.H, wl.I, wl.E, wl.k, device=dev)
    g = {n: t.to(dev) for n, t in inp.items()}
    layer.transform_weights(g["w1"], g["w1_sf"], g["w2"], g["w2_sf"])
    y = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"])
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), y_bits)

    ref = bf16_bits_to_float(orc.forward(inp))
    assert_y_close(bf16_bits_to_float(y_bits), ref, "forward_from_c")

"""The C boundary from C: tests/c_consumer.c is compiled with gcc against include/sp_fused.h and
linked with libspfused.so. On the CPU it checks the host-side helpers; on the GPU it runs the
fused stage from C and its outputs are compared with the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import sequence_reduce_add_gb300 as sp
from sequence_reduce_add_gb300 import build as sp_build
from sequence_reduce_add_gb300 import synth

from parity_util import compare

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    lib = sp_build.build()
    exe = str(tmp_path_factory.mktemp("c") / "c_consumer")
    subprocess.run(["gcc", "-std=c11", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_consumer.c"),
                    "-o", exe, lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.dirname(lib)}:{os.path.join(CUDA, 'lib64')}"],
                   check=True)
    return exe


def test_c_consumer_host_helpers(consumer):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")  # host-only path, also on a GPU machine
    out = subprocess.run([consumer], capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "host-only checks passed" in out.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("wi,rows", [(1, None), (4, 48), (5, 40)])
def test_c_consumer_device_call_matches_oracle(consumer, tmp_path, wi, rows):
    w = synth.workload(wi)
    kw = {} if rows is None else dict(T_pad=rows, T_valid=rows - 3)
    inp = synth.make_inputs(w, device="cpu", **kw)
    b = synth.bf16_bits
    tp, T_pad, Tv, H = inp["tp"], inp["T_pad"], inp["T_valid"], inp["H"]
    mode = sp.QUANT_MODES[inp["mode"]]
    path_in, path_out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(path_in, "wb") as f:
        f.write(np.array([tp, T_pad, Tv, H, mode], np.int32).tobytes())
        f.write(np.array([inp["eps"], inp["scale"] or 0.0], np.float32).tobytes())
        for k in ("partials", "residual", "weight", "bias"):
            f.write(b(inp[k]).tobytes())
    run = subprocess.run([consumer, str(path_in), str(path_out)], capture_output=True, text=True,
                         timeout=300)
    assert run.returncode == 0, run.stderr
    raw = np.fromfile(path_out, np.uint8)
    oshape, odt, sshape, sdt = oracle.out_layout(T_pad, H, inp["mode"])
    ob, sb = sp.sp_out_bytes(T_pad, H, mode), sp.sp_out_scales_bytes(T_pad, H, mode)
    got = {"out": raw[:ob].view(odt).reshape(oshape),
           "out_scales": raw[ob:ob + sb].view(sdt).reshape(sshape) if sb else None,
           "residual_out": raw[ob + sb:].view(np.uint16).reshape(T_pad, H)}
    ref = oracle.fused_reduce_norm(b(inp["partials"]), b(inp["residual"]), b(inp["weight"]),
                                   b(inp["bias"]), inp["eps"], inp["mode"], inp["scale"], Tv,
                                   want_y=True)
    compare(got, ref, inp)

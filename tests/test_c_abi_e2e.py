"""A plain C program drives the library through include/aq.h with host
buffers (tests/c_abi_e2e.c): the weight quantised once, then per call the
activations copied host -> device, aq_gemv_nvfp4, and the outputs copied
back, timed with CUDA events.  It compiles against the header alone and
links libaq.so and the CUDA runtime.  On a GPU its outputs meet the GEMV
tolerance against the oracle and equal the Python binding's bit for bit."""
import glob
import json
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "nvfp4_block_scaled_aq_gb300")


def cuda_home():
    from nvfp4_block_scaled_aq_gb300 import build
    return os.path.dirname(os.path.dirname(os.path.realpath(build.nvcc())))


def cudart_dir(home):
    for cand in [os.path.join(home, "lib64")] + sorted(glob.glob(os.path.join(home, "targets", "*", "lib"))):
        if glob.glob(os.path.join(cand, "libcudart.so*")):
            return cand
    raise RuntimeError("libcudart.so not found under %s" % home)


def build_c_program(out_dir):
    from nvfp4_block_scaled_aq_gb300 import build
    build.build()
    home = cuda_home()
    exe = os.path.join(out_dir, "c_abi_e2e")
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
                    os.path.join(ROOT, "tests", "c_abi_e2e.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(home, "include"),
                    "-L", LIB_DIR, "-laq", "-L", cudart_dir(home), "-lcudart",
                    "-Wl,-rpath," + LIB_DIR, "-o", exe], check=True)
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    """No GPU needed: the program builds with -Werror against aq.h, links,
    loads libaq.so and rejects a call without arguments before any CUDA
    call."""
    exe = build_c_program(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 2 and "usage" in r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("n,k,m", [(1536, 1152, 1), (5376, 4096, 3)])
def test_c_program_host_buffers_matches_oracle_and_binding(tmp_path, n, k, m):
    """The 1B fused QKV at m = 1 and the ~31B o_proj at m = 3, seeded."""
    import torch

    import oracle
    from gpu_helpers import DEV, assert_gemv_close, bits, require_gpu
    from nvfp4_block_scaled_aq_gb300 import aq, inputs
    require_gpu()
    W = inputs.weight(n, k, seed=n + k)
    x = inputs.tokens(m, k, seed=n + k + 1)
    Wb, xb = bits(W), bits(x)
    paths = [str(tmp_path / name) for name in ("W.bin", "x.bin", "y.bin")]
    Wb.astype("<u2").tofile(paths[0])
    xb.astype("<u2").tofile(paths[1])
    exe = build_c_program(str(tmp_path))
    r = subprocess.run([exe, str(n), str(k), str(m), "20"] + paths, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["h2d_bytes_per_call"] == m * k * 2 and line["d2h_bytes_per_call"] == m * n * 2
    assert line["us_per_call"] > 0
    y_c = np.fromfile(paths[2], dtype="<u2").reshape(m, n)

    packed, scales, _, gd = oracle.quantize(Wb)
    y_ref = oracle.gemv(packed, scales, gd, xb)
    assert_gemv_close(torch.from_numpy(y_c.view(np.int16)).view(torch.bfloat16), y_ref,
                      "C caller [%d, %d] m = %d" % (n, k, m))

    w = aq.Nvfp4Weight.empty(n, k, device=DEV)
    qws = torch.zeros(aq.quantize_workspace_bytes(), dtype=torch.uint8, device=DEV)
    aq.quantize(W.to(DEV), w, qws)
    y_py = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    gws = torch.zeros(aq.gemv_workspace_bytes(n, k, m), dtype=torch.uint8, device=DEV)
    aq.gemv(w, x.to(DEV), y_py, gws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y_py), y_c), "the C caller and the binding differ"
    assert aq.poll_device_status() == aq.OK

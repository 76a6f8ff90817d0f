"""The C ABI used from plain C (tests/c_abi_forward.c compiled with gcc against
include/moe_gb300.h and the built library): the forward it runs must equal the Python
binding's, bit for bit, on the same inputs (the same kernels behind both)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from tests.conftest import ROOT, ensure_built
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _cuda_home():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else "/usr/local/cuda"


def test_forward_from_c_equals_python(tmp_path):
    ensure_built()
    import routing_shared_expert_gb300 as moe
    pkg = os.path.join(ROOT, "routing_shared_expert_gb300")
    cuda = _cuda_home()
    exe = str(tmp_path / "c_abi_forward")
    subprocess.run(["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi_forward.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", pkg, "-lmoe_gb300", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{pkg}", "-o", exe], check=True)
    # an olmo-shaped layer at reduced size: softmax, L1, alpha = K, constant shared gain
    spec = CONFIGS["olmo"].replace(T=700, d_model=512, N=16, K=4, d_expert=384, d_shared=256)
    inp = make_inputs(spec, "cuda")
    layer = moe.MoELayer(moe.config_from_spec(spec), inp, "cuda")
    y_py = layer.forward(inp["x"]).cpu()
    idx_py = layer.out["topk_idx"].cpu()
    assert layer.status() == 0
    (tmp_path / "layer.txt").write_text(
        f"{spec.T} {spec.d_model} {spec.N} {spec.K} {spec.d_expert} {spec.d_shared}\n")
    for name in ("x", "W_router", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        t = inp[name].contiguous().cpu()
        assert t.dtype == torch.bfloat16
        t.view(torch.int16).numpy().tofile(str(tmp_path / f"{name}.bin"))
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    y_c = torch.from_numpy(np.fromfile(str(tmp_path / "y.bin"), dtype=np.float32)).view(spec.T, -1)
    idx_c = torch.from_numpy(np.fromfile(str(tmp_path / "topk_idx.bin"), dtype=np.int32))
    assert torch.equal(idx_c.view(spec.T, spec.K), idx_py)
    assert torch.equal(y_c, y_py)

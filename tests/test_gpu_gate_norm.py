"""kda_gate_norm on the GPU against the oracle's output gate (same bf16/fp32 inputs)."""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import host, rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dv", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gate_norm(kda_lib, cuda_dev, dv, dtype):
    import serving_kda_chunked_gated_gb300.kda as kda
    r = np.random.default_rng(dv)
    rows = 1000 + 3
    o = r.standard_normal((rows, dv)).astype(np.float32)
    g = r.standard_normal((rows, dv)).astype(np.float32)
    w = (r.random(dv) + 0.5).astype(np.float32)
    if dtype == "bf16":
        ob, gb = I.bf16_bits(o), I.bf16_bits(g)
        y = kda.gate_norm(to_dev(ob, cuda_dev, True), to_dev(gb, cuda_dev, True), to_dev(w, cuda_dev))
        ref = oracle.gate_norm(I.bf16_to_f32(ob), I.bf16_to_f32(gb), norm_w=w)
        tol = 2e-3
    else:
        y = kda.gate_norm(to_dev(o, cuda_dev), to_dev(g, cuda_dev), to_dev(w, cuda_dev))
        ref = oracle.gate_norm(o, g, norm_w=w)
        tol = 1e-5
    torch.cuda.synchronize()
    assert rel(host(y), ref) < tol


def test_gate_norm_empty(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    o = torch.empty((0, 128), dtype=torch.bfloat16, device=cuda_dev)
    y = kda.gate_norm(o, o.clone())
    assert y.shape == (0, 128)

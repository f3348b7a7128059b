"""The prefill kernels' give-up path, exercised without faulting the GPU.

Every wait of a prefill kernel is bounded.  With the test hook
kda_debug_set_wait_limit(0) every wait on a local copy or tensor-core
operation gives up at once: the kernels record it in the call's error word,
stop issuing asynchronous work, drain what they had issued and finish.  The
host reads the error with kda_get_last_device_error (KDA_ERR_TIMEOUT), the
CUDA context stays usable, and the same call with the default bound afterwards
is correct and reports KDA_OK.  Nothing here traps, faults or hangs: a wait
that gives up is an ordinary branch in the kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, parity, qkv_to_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def wait_limit_zero(kda_lib):
    import serving_kda_chunked_gated_gb300.kda as kda
    prev = kda.set_wait_limit(0)
    yield
    kda.set_wait_limit(kda.WAIT_LIMIT_DEFAULT)
    assert prev == kda.WAIT_LIMIT_DEFAULT


def _inputs(dev, gate):
    d = I.make_prefill(I.workload("prefill_128k", T=0, H=2, varlen=(3, 40, 300), S0_std=0.02))
    q, k, v = qkv_to_dev(d, dev)
    t = dict(q=q, k=k, v=v, z=to_dev(d["z"], dev), beta=to_dev(d["beta"], dev), A=to_dev(d["A"], dev),
             cu=to_dev(d["cu_seqlens"], dev), S0=to_dev(d["S0"], dev),
             g_in=to_dev(d["g_in"], dev, True) if gate else None)
    return d, t


def _prefill(kda, t, ws):
    return kda.prefill(t["q"], t["k"], t["v"], t["z"], t["beta"], t["A"], cu_seqlens=t["cu"], S0=t["S0"],
                       g_in=t["g_in"], workspace=ws)


@pytest.mark.parametrize("schedule", ["chunk-parallel", "single-pass"])
@pytest.mark.parametrize("gate", [False, True])
def test_wait_that_gives_up_is_reported_and_context_survives(kda_lib, cuda_dev, wait_limit_zero, schedule, gate):
    import serving_kda_chunked_gated_gb300.kda as kda
    d, t = _inputs(cuda_dev, gate)
    cu_host = t["cu"].cpu()          # kept alive: the args hold its address
    probe = kda.make_prefill_args(t["q"], t["k"], t["v"], t["z"], t["beta"], t["A"], t["cu"], cu_host,
                                  torch.empty_like(t["v"]))
    size = kda.prefill_workspace_size(probe) if schedule == "chunk-parallel" else kda.PREFILL_MIN_WORKSPACE
    ws = torch.empty(size, dtype=torch.uint8, device=cuda_dev)
    _prefill(kda, t, ws)
    assert kda.device_error(ws) == kda.KDA_ERR_TIMEOUT
    assert kda.device_error(ws) == kda.KDA_OK          # the read cleared the word
    kda.set_wait_limit(kda.WAIT_LIMIT_DEFAULT)
    o, S_T, y = _prefill(kda, t, ws)
    torch.cuda.synchronize()
    assert kda.device_error(ws) == kda.KDA_OK
    ro, rS, ry = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                cu_seqlens=d["cu_seqlens"], S0=d["S0"], g_in=f64(d, "g_in") if gate else None)
    parity("o", host(o), ro, TOL_O, bf16_out=True)
    parity("S_T", host(S_T), rS, TOL_S)
    if gate:
        parity("y", host(y), ry, TOL_O, bf16_out=True, floor_ref=ro)


def test_noalloc_wait_that_gives_up_is_reported(kda_lib, cuda_dev, wait_limit_zero):
    """kda_prefill_noalloc keeps its error word in the library's fixed array;
    kda_get_last_device_error(NULL) reads it."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d, t = _inputs(cuda_dev, True)
    cu_host = t["cu"].cpu()
    o, y = torch.empty_like(t["v"]), torch.empty_like(t["v"])
    S_T = torch.empty_like(t["S0"])
    args = kda.make_prefill_args(t["q"], t["k"], t["v"], t["z"], t["beta"], t["A"], t["cu"], cu_host, o,
                                 S0=t["S0"], S_T=S_T, g_in=t["g_in"], y=y)
    kda.prefill_noalloc_raw(args)
    assert kda.device_error(None) == kda.KDA_ERR_TIMEOUT
    kda.set_wait_limit(kda.WAIT_LIMIT_DEFAULT)
    kda.prefill_noalloc_raw(args)
    assert kda.device_error(None) == kda.KDA_OK
    ro, rS, ry = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                cu_seqlens=d["cu_seqlens"], S0=d["S0"], g_in=f64(d, "g_in"))
    parity("o", host(o), ro, TOL_O, bf16_out=True)
    parity("S_T", host(S_T), rS, TOL_S)

"""kda_prefill_noalloc, the allocation-free prefill entry point.

Some callers cannot allocate device memory while they run -- for example a
serving engine that hands all device memory to its own pool up front and forbids
allocation during requests -- so they cannot supply the workspace kda_prefill
asks for.  kda_prefill_noalloc takes the same arguments, ignores the workspace
and uses a fixed scratch array inside the library instead.  This test calls it
through the C ABI twice in a row and checks each result against kda_prefill's
on the same inputs, within the tolerances of the other prefill tests, that no
device memory was allocated, and that no bounded wait gave up (the error word,
kept in the library's array, is read with kda_get_last_device_error(NULL)).

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import pytest
import torch

from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, host, qkv_to_dev, rel, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_prefill_twice(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=0, H=4, varlen=(3, 40, 300), S0_std=0.02))
    q, k, v = qkv_to_dev(d, cuda_dev)
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    cu = to_dev(d["cu_seqlens"], cuda_dev)
    S0 = to_dev(d["S0"], cuda_dev)
    g_in = to_dev(d["g_in"], cuda_dev, True)
    ref_o, ref_S, ref_y = kda.prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=S0, g_in=g_in)
    torch.cuda.synchronize()
    cu_host = cu.cpu()
    free_after = []
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        y = torch.full_like(ref_y, float("nan"))
        S_T = torch.full_like(ref_S, float("nan"))
        args = kda.make_prefill_args(q, k, v, z, beta, A, cu, cu_host, o, S0=S0, S_T=S_T,
                                     g_in=g_in, y=y)
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated(cuda_dev)
        kda.prefill_noalloc_raw(args)
        torch.cuda.synchronize()
        # no device memory was taken: neither through torch nor from the driver
        # (the driver's count is compared across the second call, after the
        # first has loaded whatever the runtime loads lazily)
        assert torch.cuda.memory_allocated(cuda_dev) == allocated
        free_after.append(torch.cuda.mem_get_info(cuda_dev)[0])
        # no bounded wait gave up (the word lives in the library's fixed array)
        assert kda.device_error(None) == kda.KDA_OK
        assert rel(host(o), host(ref_o)) < TOL_O
        assert rel(host(y), host(ref_y)) < TOL_O
        assert rel(host(S_T), host(ref_S)) < TOL_S
        del o, y, S_T
    assert free_after[1] == free_after[0]

"""The routing entry point that allocates nothing (moe_route_noalloc) against moe_route.

Some callers cannot call cudaMalloc: code running while another framework captures the stream into a
CUDA graph, code confined to a memory pool it was handed, or latency-critical threads that cannot take
the synchronisation an allocation may cause.  For them the library offers one routing call whose
scratch is a fixed device array inside the library.  This file runs last in the suite; each test
builds what it needs, so it also passes when run on its own in a fresh process.
"""
import numpy as np
import pytest

from routed_expert_ffn_07_b300 import inputs
from routed_expert_ffn_07_b300.workloads import WORKLOADS, Workload, alloc_and_fill, create_handle
from tests.parity import W_ATOL, to_torch_act

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["small", "full"])
def test_noalloc_route_matches_moe_route(case):
    import torch
    from routed_expert_ffn_07_b300 import capi
    if case == "small":
        wl = Workload(500, "noalloc_small", 5, 1024, 64, 4, 128, True, "int4", "bf16", 1, False)
        Ts = (1, 3, 5)
    else:
        wl = WORKLOADS[2]
        Ts = (1, 4, 16)
    wts = alloc_and_fill(wl, n_layers=1)
    h = create_handle(wl, wts, max_tokens=max(Ts), n_layers=1)
    try:
        x_np = inputs.gen_activations(wl.seed, max(Ts), wl.d, "bf16", layer=3)
        x = to_torch_act(x_np)
        E, K = wl.E, wl.K
        for T in Ts:
            ref = [torch.empty(T * K, dtype=torch.int32, device="cuda"),
                   torch.empty(T * K, dtype=torch.float32, device="cuda"),
                   torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                   torch.empty(T * K, dtype=torch.int32, device="cuda")]
            capi.moe_route(h, 0, x, T, *ref)
            for _ in range(2):  # two calls in a row share (and reuse) the library's scratch
                out = [torch.full_like(r, -7) for r in ref]
                capi.moe_route_noalloc(wts["router"][0], None, x, capi.MOE_ACT_BF16, T, wl.d, E, K, *out)
                torch.cuda.synchronize()
                assert torch.equal(out[0], ref[0])
                np.testing.assert_allclose(out[1].cpu().numpy(), ref[1].cpu().numpy(), rtol=0, atol=W_ATOL)
                assert torch.equal(out[2], ref[2])
                assert torch.equal(out[3], ref[3])
    finally:
        capi.moe_destroy(h)


def test_noalloc_route_rejects_sizes_beyond_its_scratch():
    import torch
    from routed_expert_ffn_07_b300 import capi
    w = torch.zeros((8, 256), dtype=torch.float32, device="cuda")
    x = torch.zeros((32, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_route_noalloc(w, None, x, capi.MOE_ACT_BF16, 17, 256, 8, 2)   # T > 16
    assert ei.value.status == 2
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_route_noalloc(w, None, x, capi.MOE_ACT_BF16, 4, 256, 8, 9)    # K > E
    assert ei.value.status == 1


def test_noalloc_route_inside_stream_capture_and_with_null_outputs():
    """After one warm-up call (which looks up the scratch address), the call can be recorded into a
    CUDA graph by the caller and replayed; outputs left NULL go to the library's scratch."""
    import torch
    from routed_expert_ffn_07_b300 import capi
    wl = Workload(501, "noalloc_capture", 4, 1024, 64, 4, 128, True, "int4", "bf16", 1, False)
    wts = alloc_and_fill(wl, n_layers=1)
    h = create_handle(wl, wts, max_tokens=4, n_layers=1)
    try:
        T, E, K = 4, wl.E, wl.K
        x = to_torch_act(inputs.gen_activations(wl.seed, T, wl.d, "bf16", layer=1))
        ref = [torch.empty(T * K, dtype=torch.int32, device="cuda"),
               torch.empty(T * K, dtype=torch.float32, device="cuda"),
               torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               torch.empty(T * K, dtype=torch.int32, device="cuda")]
        capi.moe_route(h, 0, x, T, *ref)
        # only the permutation requested
        perm = torch.full_like(ref[3], -7)
        capi.moe_route_noalloc(wts["router"][0], None, x, capi.MOE_ACT_BF16, T, wl.d, E, K, None, None, None, perm)
        torch.cuda.synchronize()
        assert torch.equal(perm, ref[3])
        # recorded into a graph on a side stream, replayed twice
        out = [torch.full_like(r, -7) for r in ref]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            capi.moe_route_noalloc(wts["router"][0], None, x, capi.MOE_ACT_BF16, T, wl.d, E, K, *out,
                                   stream=s.cuda_stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            capi.moe_route_noalloc(wts["router"][0], None, x, capi.MOE_ACT_BF16, T, wl.d, E, K, *out,
                                   stream=torch.cuda.current_stream().cuda_stream)
        for _ in range(2):
            for o in out:
                o.fill_(-7)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out[0], ref[0]) and torch.equal(out[2], ref[2]) and torch.equal(out[3], ref[3])
            np.testing.assert_allclose(out[1].cpu().numpy(), ref[1].cpu().numpy(), rtol=0, atol=W_ATOL)
        del g
    finally:
        capi.moe_destroy(h)

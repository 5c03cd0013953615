"""GPU tensor-core (tcgen05) prefill path vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from routed_expert_ffn_07_b300 import inputs
from routed_expert_ffn_07_b300.workloads import WORKLOADS, Workload, alloc_and_fill, create_handle, host_experts
from tests.parity import Y_TOL, W_ATOL, check_dispatch, check_routing, from_torch_act, to_torch_act, y_error

pytestmark = pytest.mark.gpu


def run_prefill(h, wl, wts, x_np, T, layer=0, sample=None, repeat=False):
    import torch
    from routed_expert_ffn_07_b300 import capi
    K, E = wl.K, wl.E
    x = to_torch_act(x_np)
    idx = torch.empty(T * K, dtype=torch.int32, device="cuda")
    w = torch.empty(T * K, dtype=torch.float32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
    capi.moe_route(h, layer, x, T, idx, w, offs, perm)
    y = torch.empty_like(x)
    capi.moe_layer_forward(h, layer, x, T, y)
    torch.cuda.synchronize()
    assert capi.moe_get_device_status(h) == 0
    if repeat:
        y2 = torch.empty_like(x)
        capi.moe_layer_forward(h, layer, x, T, y2)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "prefill output not bit-identical run to run"
    Wr = wts["router"][layer].cpu().numpy()
    bias = None if wts["bias"] is None else wts["bias"][layer].cpu().numpy()
    logits, idx_ref, _, gap = oracle.route(x_np, Wr, bias, K)
    idx_g = idx.cpu().numpy().reshape(T, K)
    flagged = check_routing(logits, idx_ref, gap, idx_g)
    check_dispatch(idx_g, E, offs.cpu().numpy(), perm.cpu().numpy())
    np.testing.assert_allclose(w.cpu().numpy().reshape(T, K), oracle.weights_for(logits, idx_g), rtol=0, atol=W_ATOL)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    used = sorted(set(idx_g[rows].ravel().tolist()))
    ex = host_experts(wl, layer, used + ([E] if wl.shared else []))
    sh = ex.pop(E) if wl.shared else None
    y_ref, _, _ = oracle.layer(x_np[rows], Wr, bias, ex, E, K, shared=sh, idx=idx_g[rows])
    y_g = oracle.widen(from_torch_act(y))[rows]
    err = y_error(y_g, y_ref)
    assert err <= Y_TOL, f"max err {err:.3e}"
    return err, flagged, idx_g


SMALL = [
    # d, f, E, K, shared, T values
    (256, 256, 16, 4, True, (17, 33, 100, 300)),
    (512, 256, 8, 2, False, (600,)),          # ~150 tokens per expert: two tiles per expert
    (256, 512, 32, 8, True, (129, 257)),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_prefill_small_shapes(case):
    from routed_expert_ffn_07_b300 import capi
    d, f, E, K, sh, Ts = SMALL[case]
    wl = Workload(400 + case, f"prefill_small{case}", max(Ts), d, E, K, f, sh, "int4", "bf16", 1, False)
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, max(Ts), d, "bf16")
        for T in Ts:
            run_prefill(h, wl, wts, x[:T], T, repeat=(T == Ts[0]))
    finally:
        capi.moe_destroy(h)


def test_prefill_full_width_T200():
    from routed_expert_ffn_07_b300 import capi
    wl = Workload(410, "prefill_fullwidth", 200, 2048, 64, 4, 768, True, "int4", "bf16", 1, False)
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, 200, wl.d, "bf16")
        run_prefill(h, wl, wts, x, 200, sample=np.arange(0, 200, 5))
        # the GEMV path (T <= 16) and the tensor-core path agree with the oracle on the same tokens
        run_prefill(h, wl, wts, x[:16], 16)
    finally:
        capi.moe_destroy(h)


def test_prefill_chunk_T4096_full_size():
    import torch
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[4]
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, wl.T, wl.d, "bf16")
        rng = np.random.default_rng(4)
        sample = np.unique(np.concatenate([[0, 1, wl.T - 1], rng.choice(wl.T, 45, replace=False)]))
        err, flagged, idx_g = run_prefill(h, wl, wts, x, wl.T, sample=sample, repeat=True)
        counts = np.bincount(idx_g.ravel(), minlength=wl.E)
        assert counts.sum() == wl.T * wl.K
        assert (counts > 0).sum() >= 500  # a prefill chunk reaches almost every expert
    finally:
        capi.moe_destroy(h)
        del wts
        torch.cuda.empty_cache()

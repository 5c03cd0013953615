"""GPU tensor-core (tcgen05) prefill path vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from routed_expert_ffn_07_b300 import inputs
from routed_expert_ffn_07_b300.workloads import WORKLOADS, Workload, alloc_and_fill, create_handle, host_experts
from tests.parity import (TIE_EPS, Y_TOL, W_ATOL, check_dispatch, check_routing, from_torch_act, to_torch_act,
                          y_error)

pytestmark = pytest.mark.gpu


def tile_edge_tokens(idx_g: np.ndarray, E: int, tile: int = 128) -> np.ndarray:
    """Tokens whose assignment is the first or the last row of a `tile`-row tile of its expert's
    token group (the dispatch order: ascending token within an expert)."""
    T, K = idx_g.shape
    _, offs, perm, _ = oracle.dispatch(idx_g, E)
    rows = []
    for e in range(E):
        for a in range(offs[e], offs[e + 1], tile):
            rows += [perm[a], perm[min(a + tile, offs[e + 1]) - 1]]
    return np.unique(np.asarray(rows, dtype=np.int64) // K)


def run_prefill(h, wl, wts, x_np, T, layer=0, sample=None, repeat=False, edges=0, n_random=0, seed=0,
                max_edge_tokens=None):
    """Forward one layer; check the routing the forward used (bit-exact), its dispatch, the
    stand-alone routing call, and the output on `sample` tokens (all tokens if None), plus, when
    `edges`, every token at the first or last row of a 128-row tile of an expert and `n_random`
    random tokens."""
    import torch
    from routed_expert_ffn_07_b300 import capi
    K, E = wl.K, wl.E
    x = to_torch_act(x_np)
    idx = torch.full((T * K,), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T * K,), -1.0, dtype=torch.float32, device="cuda")
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * K,), -1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(x)
    capi.moe_layer_forward(h, layer, x, T, y)
    capi.moe_get_last_routing(h, T, idx, w, offs, perm)
    torch.cuda.synchronize()
    assert capi.moe_get_device_status(h) == 0
    if repeat:
        y2 = torch.empty_like(x)
        capi.moe_layer_forward(h, layer, x, T, y2)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "prefill output not bit-identical run to run"
    r = [torch.empty_like(t) for t in (idx, w, offs, perm)]
    capi.moe_route(h, layer, x, T, *r)
    torch.cuda.synchronize()
    Wr = wts["router"][layer].cpu().numpy()
    bias = None if wts["bias"] is None else wts["bias"][layer].cpu().numpy()
    logits, idx_ref, _, gap = oracle.route(x_np, Wr, bias, K)
    idx_g = idx.cpu().numpy().reshape(T, K)
    flagged = check_routing(logits, idx_ref, gap, idx_g)
    check_dispatch(idx_g, E, offs.cpu().numpy(), perm.cpu().numpy())
    np.testing.assert_allclose(w.cpu().numpy().reshape(T, K), oracle.weights_for(logits, idx_g), rtol=0, atol=W_ATOL)
    # the stand-alone routing call agrees (bit for bit away from near-ties: for T <= 16 the forward's
    # one-launch layer sums its logits in another order)
    r_idx_g = r[0].cpu().numpy().reshape(T, K)
    check_routing(logits, idx_ref, gap, r_idx_g)
    clear = gap >= TIE_EPS
    np.testing.assert_array_equal(r_idx_g[clear], idx_g[clear])
    if clear.all():
        assert torch.equal(r[2], offs) and torch.equal(r[3], perm)
        np.testing.assert_allclose(r[1].cpu().numpy(), w.cpu().numpy(), rtol=0, atol=W_ATOL)
    if sample is None and not edges and not n_random:
        rows = np.arange(T)
    else:
        parts = [np.asarray([] if sample is None else sample, dtype=np.int64)]
        if edges:
            ed = tile_edge_tokens(idx_g, E)
            if max_edge_tokens is not None and len(ed) > max_edge_tokens:
                ed = np.random.default_rng(seed + 1).choice(ed, max_edge_tokens, replace=False)
            parts.append(ed)
        if n_random:
            parts.append(np.random.default_rng(seed).choice(T, n_random, replace=False))
        rows = np.unique(np.concatenate(parts))
    used = sorted(set(idx_g[rows].ravel().tolist()))
    ex = host_experts(wl, layer, used + ([E] if wl.shared else []))
    sh = ex.pop(E) if wl.shared else None
    y_ref, _, _ = oracle.layer(x_np[rows], Wr, bias, ex, E, K, shared=sh, idx=idx_g[rows])
    y_g = oracle.widen(from_torch_act(y))[rows]
    err = y_error(y_g, y_ref)
    assert err <= Y_TOL, f"max err {err:.3e}"
    return err, flagged, idx_g, rows


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
        run_prefill(h, wl, wts, x, 200, sample=np.arange(0, 200, 5), edges=True)
        # the one-launch decode layer (T <= 16) and the tensor-core path agree with the oracle on the same tokens
        run_prefill(h, wl, wts, x[:16], 16)
    finally:
        capi.moe_destroy(h)


def test_prefill_chunk_T4096_full_size():
    """The full 4096-token chunk: routing and dispatch of every token; outputs of every token at the
    first or last row of any 128-row tile of an expert, plus 256 random tokens."""
    import torch
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[4]
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, wl.T, wl.d, "bf16")
        err, flagged, idx_g, rows = run_prefill(h, wl, wts, x, wl.T, sample=[0, 1, wl.T - 1], repeat=True,
                                                edges=True, n_random=256, seed=4)
        counts = np.bincount(idx_g.ravel(), minlength=wl.E)
        assert counts.sum() == wl.T * wl.K
        assert (counts > 0).sum() >= 500  # a prefill chunk reaches almost every expert
        assert len(rows) >= 500
    finally:
        capi.moe_destroy(h)
        del wts
        torch.cuda.empty_cache()


def test_prefill_chunk_T4096_skewed_multi_tile():
    """Full-size shapes (d = 2048, f = 768, 512 experts) with the Zipf(1.1) popularity prior as the
    router bias: the popular experts receive thousands of tokens, i.e. many 128-row tiles each."""
    import dataclasses
    import torch
    from routed_expert_ffn_07_b300 import capi
    wl = dataclasses.replace(WORKLOADS[5], idx=6, name="prefill_skewed", T=4096, layers=1, prenorm=False,
                             stack=False)
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, wl.T, wl.d, "bf16")
        err, flagged, idx_g, rows = run_prefill(h, wl, wts, x, wl.T, edges=True, n_random=64, seed=6,
                                                max_edge_tokens=384)
        counts = np.bincount(idx_g.ravel(), minlength=wl.E)
        assert counts.max() > 4 * 128  # several tiles for the popular experts
    finally:
        capi.moe_destroy(h)
        del wts
        torch.cuda.empty_cache()


def test_prefill_fp32_activations_T40():
    """int4 experts with fp32 activations above the small-T limit: the fp32 SIMT router GEMM (the
    tensor-core router serves bf16 activations) and the grouped GEMM's fp32 -> fp16 staging."""
    from routed_expert_ffn_07_b300 import capi
    wl = Workload(420, "prefill_fp32_act", 40, 256, 16, 4, 256, True, "int4", "f32", 1, False)
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, 40, wl.d, "f32")
        run_prefill(h, wl, wts, x, 40, repeat=True)
        run_prefill(h, wl, wts, x[:17], 17)
    finally:
        capi.moe_destroy(h)

"""GPU (CUDA library, through the C ABI) vs the fp64 oracle: router, dispatch, GEMV experts, stack."""
import numpy as np
import pytest

import oracle
from routed_expert_ffn_07_b300 import inputs
from routed_expert_ffn_07_b300.workloads import WORKLOADS, Workload, alloc_and_fill, create_handle, host_experts
from tests.parity import (TIE_EPS, Y_TOL, W_ATOL, check_dispatch, check_routing, from_torch_act, to_torch_act,
                          y_error)

pytestmark = pytest.mark.gpu

PATHS = {  # decode path -> (MOE_OPT_FUSED_MAX_TOKENS, MOE_OPT_GEMV_MAX_TOKENS)
    "one_launch": (16, 16),
    "gemv": (0, 16),
    "tensor_core": (0, 0),
}


def _torch():
    import torch
    return torch


def run_layer(h, wl, weights, x_np, T, layer=0, gen_layer=0):
    """Forward one layer on the GPU and check the routing that forward pass used (read back with
    moe_get_last_routing), its dispatch and its output against the oracle; then check that the
    stand-alone routing call agrees with the forward's routing."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    K, E = wl.K, wl.E
    n_layers = weights["router"].shape[0]
    x = to_torch_act(x_np)

    def outs():
        return (torch.full((T * K,), -1, dtype=torch.int32, device="cuda"),
                torch.full((T * K,), -1.0, dtype=torch.float32, device="cuda"),
                torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
                torch.full((T * K,), -1, dtype=torch.int32, device="cuda"))

    idx, w, offs, perm = outs()
    y = torch.empty_like(x)
    capi.moe_layer_forward(h, layer, x, T, y)
    capi.moe_get_last_routing(h, T, idx, w, offs, perm)
    torch.cuda.synchronize()
    assert capi.moe_get_device_status(h) == 0
    n_active_fwd = int(capi.moe_get_active_counts(h, n_layers)[layer])
    Wr = weights["router"][layer].cpu().numpy()
    bias = None if weights["bias"] is None else weights["bias"][layer].cpu().numpy()
    logits, idx_ref, w_ref, gap = oracle.route(x_np, Wr, bias, K)
    idx_g = idx.cpu().numpy().reshape(T, K)
    flagged = check_routing(logits, idx_ref, gap, idx_g)
    active = check_dispatch(idx_g, E, offs.cpu().numpy(), perm.cpu().numpy())
    assert n_active_fwd == len(active)
    w_exp = oracle.weights_for(logits, idx_g)
    np.testing.assert_allclose(w.cpu().numpy().reshape(T, K), w_exp, rtol=0, atol=W_ATOL)
    # the stand-alone routing call picks the same experts in the same slots (its logits are summed
    # in another order, so a near-tie token may legitimately go either way there)
    r_idx, r_w, r_offs, r_perm = outs()
    capi.moe_route(h, layer, x, T, r_idx, r_w, r_offs, r_perm)
    torch.cuda.synchronize()
    r_idx_g = r_idx.cpu().numpy().reshape(T, K)
    check_routing(logits, idx_ref, gap, r_idx_g)
    clear = gap >= TIE_EPS
    np.testing.assert_array_equal(r_idx_g[clear], idx_g[clear])
    if clear.all():
        assert torch.equal(r_offs, offs) and torch.equal(r_perm, perm)
        np.testing.assert_allclose(r_w.cpu().numpy(), w.cpu().numpy(), rtol=0, atol=W_ATOL)
    used = sorted(set(idx_g.ravel().tolist()))
    ex = host_experts(wl, gen_layer, used + ([E] if wl.shared else []))
    sh = ex.pop(E) if wl.shared else None
    y_ref, _, _ = oracle.layer(x_np, Wr, bias, ex, E, K, shared=sh, idx=idx_g)
    err = y_error(oracle.widen(from_torch_act(y)), y_ref)
    assert err <= Y_TOL, f"max err {err:.3e} > {Y_TOL}"
    return y, err, flagged


def test_device_generator_matches_host():
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[2]
    d, f = 1024, 256
    for layer, e0, n in ((0, 0, 3), (7, 511, 2)):
        gu = torch.empty((n, 2 * f, d // 2), dtype=torch.uint8, device="cuda")
        gs = torch.empty((n, 2 * f, d // 32), dtype=torch.float16, device="cuda")
        dn = torch.empty((n, d, f // 2), dtype=torch.uint8, device="cuda")
        ds = torch.empty((n, d, f // 32), dtype=torch.float16, device="cuda")
        capi.moe_gen_int4_planes(gu, wl.seed, layer, inputs.T_GU_Q, e0, n, gu[0].numel())
        capi.moe_gen_scale_planes(gs, wl.seed, layer, inputs.T_GU_S, e0, n, gs[0].numel())
        capi.moe_gen_int4_planes(dn, wl.seed, layer, inputs.T_DN_Q, e0, n, dn[0].numel())
        capi.moe_gen_scale_planes(ds, wl.seed, layer, inputs.T_DN_S, e0, n, ds[0].numel())
        torch.cuda.synchronize()
        for i in range(n):
            ref = inputs.gen_expert_int4(wl.seed, layer, e0 + i, d, f)
            np.testing.assert_array_equal(gu[i].cpu().numpy(), ref["gu_q"])
            np.testing.assert_array_equal(gs[i].cpu().numpy().view(np.uint16), ref["gu_s"])
            np.testing.assert_array_equal(dn[i].cpu().numpy(), ref["dn_q"])
            np.testing.assert_array_equal(ds[i].cpu().numpy().view(np.uint16), ref["dn_s"])


def test_tiny_fp32_layer():
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[1]
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        x = inputs.gen_activations(wl.seed, wl.T, wl.d, "f32")
        _, err, _ = run_layer(h, wl, wts, x, wl.T)
        assert err < 1e-4  # fp32 everywhere
        for T in (1, 3, 7):
            run_layer(h, wl, wts, x[:T], T)
    finally:
        capi.moe_destroy(h)


SMALL = [
    # d, f, E, K, shared, T values
    (1024, 256, 32, 4, True, (1, 2, 5, 16)),
    (2048, 128, 16, 3, False, (1, 4, 9)),
    (3072, 384, 24, 6, True, (1, 7, 16)),
    (1024, 512, 8, 8, True, (1, 3)),     # K = E: every expert for every token
    (2048, 256, 64, 1, True, (1, 16)),   # K = 1
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_int4_shapes(case):
    from routed_expert_ffn_07_b300 import capi
    d, f, E, K, sh, Ts = SMALL[case]
    wl = Workload(200 + case, f"small{case}", max(Ts), d, E, K, f, sh, "int4", "bf16", 2, False)
    wts = alloc_and_fill(wl)
    h = create_handle(wl, wts)
    try:
        for layer in (0, 1):
            x = inputs.gen_activations(wl.seed, max(Ts), d, "bf16", layer=layer)
            for T in Ts:
                run_layer(h, wl, wts, x[:T], T, layer=layer, gen_layer=layer)
    finally:
        capi.moe_destroy(h)


@pytest.mark.parametrize("path", ["one_launch", "gemv", "tensor_core"])
def test_exact_ties_lower_index_on_gpu(path):
    """Duplicated router rows give bit-identical logits on both sides: the lower index must win, on
    every decode path and at T = 1, 2 (the one-launch layer's block-wide selection) and 4, 16."""
    from routed_expert_ffn_07_b300 import capi
    wl = Workload(250, "ties", 16, 1024, 32, 4, 128, True, "int4", "bf16", 1, False)
    wts = alloc_and_fill(wl)
    r = wts["router"][0]
    for a, b in ((3, 17), (5, 6), (9, 30), (12, 2), (20, 21), (0, 31)):
        r[b] = r[a]
    h = create_handle(wl, wts)
    fz, gv = PATHS[path]
    capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, fz)
    capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, gv)
    try:
        x = inputs.gen_activations(wl.seed, 16, wl.d, "bf16")
        for T in (1, 2, 4, 16):
            run_layer(h, wl, wts, x[:T], T)
    finally:
        capi.moe_destroy(h)


@pytest.mark.parametrize("path", ["one_launch", "gemv", "tensor_core"])
def test_all_logits_equal_picks_the_first_k_experts(path):
    """A zero router makes every logit of every token exactly 0: all E experts tie, so each token
    must get experts 0 .. K-1 in that order with weights 1/K (ties go to the lower index)."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[2]
    wts = alloc_and_fill(wl, n_layers=1)
    wts["router"].zero_()
    h = create_handle(wl, wts, max_tokens=16, n_layers=1)
    fz, gv = PATHS[path]
    capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, fz)
    capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, gv)
    try:
        x_all = inputs.gen_activations(wl.seed, 16, wl.d, "bf16", layer=4)
        for T in (1, 2, 4, 16):
            y, err, flagged = run_layer(h, wl, wts, x_all[:T], T)
            assert flagged == T
            idx = torch.empty(T * wl.K, dtype=torch.int32, device="cuda")
            w = torch.empty(T * wl.K, dtype=torch.float32, device="cuda")
            capi.moe_layer_forward(h, 0, to_torch_act(x_all[:T]), T, y)
            capi.moe_get_last_routing(h, T, idx, w)
            torch.cuda.synchronize()
            expect = np.tile(np.arange(wl.K, dtype=np.int32), T)
            np.testing.assert_array_equal(idx.cpu().numpy(), expect)
            np.testing.assert_allclose(w.cpu().numpy(), 1.0 / wl.K, rtol=0, atol=W_ATOL)
    finally:
        capi.moe_destroy(h)


@pytest.fixture(scope="module")
def decode_layer():
    from routed_expert_ffn_07_b300 import capi
    wl = WORKLOADS[2]
    wts = alloc_and_fill(wl, n_layers=3)
    h = create_handle(wl, wts, max_tokens=16)
    yield wl, wts, h
    capi.moe_destroy(h)


def test_decode_layer_full_size(decode_layer):
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    for layer in range(3):
        x = inputs.gen_activations(wl.seed, 1, wl.d, "bf16", layer=layer)
        y, err, _ = run_layer(h, wl, wts, x, 1, layer=layer, gen_layer=layer)
        # run-to-run bit identity
        y2 = torch.empty_like(y)
        capi.moe_layer_forward(h, layer, to_torch_act(x), 1, y2)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
        # the host-buffer entry point gives the same bits
        yh = np.zeros_like(x)
        capi.moe_layer_forward_host(h, layer, np.ascontiguousarray(x), 1, yh)
        np.testing.assert_array_equal(yh, from_torch_act(y))


def test_host_entry_point_pinned_and_pageable_buffers(decode_layer):
    """moe_layer_forward_host moves page-locked, device-mapped buffers with a small kernel over the
    host link and pageable ones with copies: both must give moe_layer_forward's bits, T = 1, 5, 16,
    including a pinned buffer at an odd byte offset (the byte-wise form of the kernel)."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    x_all = inputs.gen_activations(wl.seed, 16, wl.d, "bf16", layer=11)
    for T in (1, 5, 16):
        x = np.ascontiguousarray(x_all[:T])
        y = torch.empty((T, wl.d), dtype=torch.bfloat16, device="cuda")
        capi.moe_layer_forward(h, 0, to_torch_act(x), T, y)
        torch.cuda.synchronize()
        ref = from_torch_act(y)
        # pageable numpy buffers: the copy path
        yn = np.zeros_like(x)
        capi.moe_layer_forward_host(h, 0, x, T, yn)
        np.testing.assert_array_equal(yn, ref)
        # page-locked torch buffers: the kernel path
        xp = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
        yp = torch.zeros_like(xp).pin_memory()
        capi.moe_layer_forward_host(h, 0, xp, T, yp)
        np.testing.assert_array_equal(yp.numpy().view(np.uint16), ref)
        # pinned, but one byte into the allocation: byte-wise loads and stores
        nb = x.nbytes
        xb = torch.zeros(nb + 1, dtype=torch.uint8).pin_memory()
        yb = torch.zeros(nb + 1, dtype=torch.uint8).pin_memory()
        xb[1:] = torch.from_numpy(x.view(np.uint8).reshape(-1).copy())
        capi.moe_layer_forward_host(h, 0, xb.data_ptr() + 1, T, yb.data_ptr() + 1)
        assert capi.moe_get_device_status(h) == 0
        np.testing.assert_array_equal(yb[1:].numpy().view(np.uint16).reshape(T, wl.d), ref)
        assert int(yb[0]) == 0  # nothing written before y


def test_decode_layer_batch_sizes(decode_layer):
    wl, wts, h = decode_layer
    x = inputs.gen_activations(wl.seed, 16, wl.d, "bf16", layer=5)
    for T in (2, 4, 16):
        run_layer(h, wl, wts, x[:T], T, layer=1, gen_layer=1)


def _stack_parity(wl, sample_layers, gemv_max=None, fused_max=None):
    """The stack, checked teacher-forced per layer: each sampled layer's input, normalised input and
    the routing that layer used come from a traced run; the oracle recomputes that layer from the
    traced input."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wts = alloc_and_fill(wl)
    L, T, d, K, E = wl.layers, wl.T, wl.d, wl.K, wl.E
    h = create_handle(wl, wts)
    if gemv_max is not None:
        capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, gemv_max)
    if fused_max is not None:
        capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, fused_max)
    try:
        x0 = inputs.gen_activations(wl.seed, T, d, "bf16")
        xa = to_torch_act(x0)
        trace = torch.empty((L, 2, T, d), dtype=torch.bfloat16, device="cuda")
        r_idx = torch.full((L, T * K), -1, dtype=torch.int32, device="cuda")
        r_w = torch.full((L, T * K), -1.0, dtype=torch.float32, device="cuda")
        r_offs = torch.full((L, E + 1), -1, dtype=torch.int32, device="cuda")
        r_perm = torch.full((L, T * K), -1, dtype=torch.int32, device="cuda")
        capi.moe_stack_forward_traced(h, xa, T, trace, r_idx, r_w, r_offs, r_perm)
        xg = to_torch_act(x0)
        capi.moe_stack_forward(h, xg, T)   # graph replay
        capi.moe_stack_forward(h, xg2 := to_torch_act(x0), T)
        torch.cuda.synchronize()
        assert capi.moe_get_device_status(h) == 0
        assert torch.equal(xa.view(torch.int16), xg.view(torch.int16)), "graph replay != eager launches"
        assert torch.equal(xg.view(torch.int16), xg2.view(torch.int16)), "graph replays differ"
        tr = trace.view(torch.int16).cpu().numpy().view(np.uint16)
        final = from_torch_act(xa)
        counts = capi.moe_get_active_counts(h, L)
        ri, rw, ro, rp = (t.cpu().numpy() for t in (r_idx, r_w, r_offs, r_perm))
        flagged_total = 0
        worst = 0.0
        for l in sample_layers:
            x_l, xn_l = tr[l, 0], tr[l, 1]
            x_next = tr[l + 1, 0] if l + 1 < L else final
            # RMSNorm (fp32 on the GPU, rounded to bf16) vs fp64: within one bf16 ulp
            ref_n = oracle.rmsnorm(x_l, 1e-6)
            got_n = oracle.widen(xn_l)
            assert np.all(np.abs(got_n - ref_n) <= 2.0 ** -8 * np.abs(ref_n) + 1e-30)
            # the routing this layer of the stack used, against the oracle on the traced input
            Wr = wts["router"][l].cpu().numpy()
            bias = None if wts["bias"] is None else wts["bias"][l].cpu().numpy()
            logits, idx_ref, _, gap = oracle.route(xn_l, Wr, bias, K)
            idx_g = ri[l].reshape(T, K)
            flagged_total += check_routing(logits, idx_ref, gap, idx_g)
            active = check_dispatch(idx_g, E, ro[l], rp[l])
            np.testing.assert_allclose(rw[l].reshape(T, K), oracle.weights_for(logits, idx_g), rtol=0, atol=W_ATOL)
            assert counts[l] == len(active)
            ex = host_experts(wl, l, sorted(set(idx_g.ravel().tolist())) + [E])
            sh = ex.pop(E)
            y_ref, _, _ = oracle.layer(xn_l, Wr, bias, ex, E, K, shared=sh, idx=idx_g)
            x_ref = oracle.widen(x_l) + y_ref
            got = oracle.widen(x_next)
            tol = Y_TOL * np.abs(y_ref).max() + 2.0 ** -8 * np.abs(x_ref)
            bad = np.abs(got - x_ref) > tol
            assert not bad.any(), f"layer {l}: {bad.sum()} elements out of tolerance"
            worst = max(worst, float((np.abs(got - x_ref) / (np.abs(y_ref).max())).max()))
        return counts, flagged_total, worst
    finally:
        capi.moe_destroy(h)
        del wts
        torch.cuda.empty_cache()


def test_verify_stack_T4_48_layers():
    wl = WORKLOADS[3]
    counts, flagged, worst = _stack_parity(wl, sample_layers=[0, 1, 2, 7, 15, 23, 24, 31, 40, 45, 46, 47])
    assert all(10 <= c <= 40 for c in counts)


def test_skewed_stack_T16_zipf():
    wl = WORKLOADS[5]
    counts, flagged, worst = _stack_parity(wl, sample_layers=[0, 5, 17, 29, 41, 47])
    assert all(10 <= c <= 160 for c in counts)
    assert np.mean(counts) < 120  # the popularity prior concentrates the routing


def test_invalid_arguments_rejected():
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl = Workload(260, "args", 4, 1024, 16, 2, 128, True, "int4", "bf16", 2, False)
    wts = alloc_and_fill(wl, n_layers=1)
    h = capi.moe_create(wl.d, wl.f, wl.E, wl.K, 2, 4, has_shared=True)
    try:
        x = torch.zeros((8, wl.d), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros_like(x)
        with pytest.raises(capi.MoeError) as ei:
            capi.moe_layer_forward(h, 0, x, 2, y)
        assert ei.value.status == 6  # weights not set
        capi.moe_set_layer(h, 0, wts["router"][0], wts["gu_q"][0], wts["gu_s"][0], wts["dn_q"][0], wts["dn_s"][0],
                           sh_gu_q=wts["sh_gu_q"][0], sh_gu_s=wts["sh_gu_s"][0], sh_dn_q=wts["sh_dn_q"][0],
                           sh_dn_s=wts["sh_dn_s"][0])
        for bad in (lambda: capi.moe_layer_forward(h, 0, x, 5, y),          # T > max_tokens
                    lambda: capi.moe_layer_forward(h, 0, x, 0, y),          # T = 0
                    lambda: capi.moe_layer_forward(h, 2, x, 2, y),          # layer out of range
                    lambda: capi.moe_layer_forward(h, 0, x, 2, x),          # y overlaps x
                    lambda: capi.moe_layer_forward(h, 0, 0, 2, y),          # null x
                    lambda: capi.moe_layer_forward(h, 0, x.data_ptr() + 2, 2, y)):  # misaligned
            with pytest.raises(capi.MoeError) as ei:
                bad()
            assert ei.value.status == 1
        with pytest.raises(capi.MoeError):
            capi.moe_set_layer(h, 1, 0, wts["gu_q"][0], wts["gu_s"][0], wts["dn_q"][0], wts["dn_s"][0])
        capi.moe_layer_forward(h, 0, x, 2, y)
        torch.cuda.synchronize()
        assert capi.moe_get_device_status(h) == 0
    finally:
        capi.moe_destroy(h)




@pytest.mark.parametrize("path", list(PATHS))
def test_decode_sizes_on_every_expert_path(decode_layer, path):
    """T <= 16 through the one-launch layer (T <= 8), the split-K GEMV experts and the grouped GEMM."""
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    fz, gv = PATHS[path]
    got = capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, fz)
    assert (got >= 4) if fz else (got == 0)  # the one-launch layer serves at least decode and 1 + 3 verify
    capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, gv)
    try:
        x = inputs.gen_activations(wl.seed, 16, wl.d, "bf16", layer=9)
        for T in (1, 2, 3, 4, 5, 8, 16):
            run_layer(h, wl, wts, x[:T], T, layer=2, gen_layer=2)
    finally:
        capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, 16)
        capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, 4)


def test_one_launch_layer_matches_gemv_path_closely(decode_layer):
    """Same routing, same per-product arithmetic: the two decode paths agree to fp32 rounding."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    x = to_torch_act(inputs.gen_activations(wl.seed, 4, wl.d, "bf16", layer=11))
    out = {}
    try:
        for path in ("one_launch", "gemv"):
            fz, gv = PATHS[path]
            capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, fz)
            capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, gv)
            y = torch.empty_like(x)
            capi.moe_layer_forward(h, 1, x, 4, y)
            torch.cuda.synchronize()
            assert capi.moe_get_device_status(h) == 0
            out[path] = y.float()
    finally:
        capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, 16)
        capi.moe_set_option(h, capi.MOE_OPT_GEMV_MAX_TOKENS, 4)
    a, b = out["one_launch"], out["gemv"]
    # The GEMV path multiplies in fp32; the one-launch layer feeds its tensor cores fp16 operands
    # (exact int4 codes and bf16 activations, but w * h rounded to an 11-bit significand) and
    # accumulates in fp32.  Both round once to bf16 (2 ulps, 2^-7 relative).  The fp16 rounding of
    # h adds up to 2^-11 relative per term of the down sum, so the difference scales with the size
    # of the summed terms (the layer's output scale), not with an output that cancels to near zero:
    # 2^-9 of max|y| bounds it with room to spare.
    tol = 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 2.0 ** -9 * b.abs().max()
    assert torch.all((a - b).abs() <= tol)


def test_verify_stack_on_gemv_path():
    wl = WORKLOADS[3]
    import dataclasses
    wl_small = dataclasses.replace(wl, layers=8)
    counts, flagged, worst = _stack_parity(wl_small, sample_layers=[0, 3, 7], fused_max=0, gemv_max=16)
    assert all(10 <= c <= 40 for c in counts)


def test_skewed_stack_on_gemv_path():
    wl = WORKLOADS[5]
    import dataclasses
    wl_small = dataclasses.replace(wl, layers=8)
    counts, flagged, worst = _stack_parity(wl_small, sample_layers=[0, 3, 7], gemv_max=16)
    assert all(10 <= c <= 160 for c in counts)


def test_bounded_waits_give_up_and_the_context_survives(decode_layer):
    """A wait that nothing can satisfy (an mbarrier nobody arrives at, a barrier counter nobody
    bumps) gives up within its budget and reports a timeout; the library keeps working after it."""
    from routed_expert_ffn_07_b300 import capi
    assert capi.moe_selftest_bounded_waits(2_000_000) == 5  # MOE_ERR_TIMEOUT
    wl, wts, h = decode_layer
    x = inputs.gen_activations(wl.seed, 1, wl.d, "bf16", layer=3)
    run_layer(h, wl, wts, x, 1, layer=0, gen_layer=0)


def test_usage_histogram_counts_every_forward_exactly(decode_layer):
    """The per-expert usage counters equal the sum of the oracle's dispatch counts of the routings
    the forward passes used, over several calls, layers and token counts; moe_route adds nothing."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    L, E, K = wts["router"].shape[0], wl.E, wl.K
    capi.moe_usage_read(h, L, E, reset=True)
    capi.moe_usage_enable(h, True)
    expect = np.zeros((L, E), dtype=np.uint64)
    try:
        x_all = inputs.gen_activations(wl.seed, 16, wl.d, "bf16", layer=13)
        for i, (layer, T) in enumerate([(0, 1), (1, 4), (2, 16), (0, 2), (0, 1), (1, 16)]):
            x = to_torch_act(x_all[:T])
            y = torch.empty_like(x)
            idx = torch.empty(T * K, dtype=torch.int32, device="cuda")
            capi.moe_layer_forward(h, layer, x, T, y)
            capi.moe_get_last_routing(h, T, idx)
            capi.moe_route(h, layer, x, T)          # not counted
            torch.cuda.synchronize()
            counts, _, _, _ = oracle.dispatch(idx.cpu().numpy().reshape(T, K), E)
            expect[layer] += counts.astype(np.uint64)
        got = capi.moe_usage_read(h, L, E, reset=True)
        np.testing.assert_array_equal(got, expect)
        assert not capi.moe_usage_read(h, L, E).any()
    finally:
        capi.moe_usage_enable(h, False)


def test_one_launch_layer_gives_up_on_a_reported_timeout_and_recovers(decode_layer):
    """Host-side fault injection: with the status word's timeout bit set (as a launch whose wait gave
    up leaves it), the one-launch layer returns NaN instead of a silently wrong y, the status call
    reports MOE_ERR_TIMEOUT and resets, and the next launch is correct again.  No GPU fault."""
    torch = _torch()
    from routed_expert_ffn_07_b300 import capi
    wl, wts, h = decode_layer
    assert capi.moe_set_option(h, capi.MOE_OPT_FUSED_MAX_TOKENS, -1) >= 1
    x_np = inputs.gen_activations(wl.seed, 1, wl.d, "bf16", layer=21)
    x = to_torch_act(x_np)
    y = torch.zeros_like(x)
    capi.moe_inject_device_status(h, 2)
    capi.moe_layer_forward(h, 0, x, 1, y)
    capi.moe_layer_forward(h, 1, x, 1, y)   # still refused: the status has not been read yet
    torch.cuda.synchronize()
    assert torch.isnan(y.float()).all()
    assert capi.moe_get_device_status(h) == 5  # MOE_ERR_TIMEOUT, then cleared
    assert capi.moe_get_device_status(h) == 0
    run_layer(h, wl, wts, x_np, 1, layer=0, gen_layer=0)

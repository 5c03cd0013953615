"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, a hand-written fixture, a brute force on tiny
inputs, or a library routine (numpy / torch) computing a special case the method reduces to.
Together they are chosen so that a dropped term, a wrong sign, a swapped nibble, a transposed
operand or a wrong tie-break fails at least one of them (test_oracle_mutants.py checks that).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_07_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ number formats
def test_int4_nibbles_match_hand_table():
    rows = _read_table("int4_nibbles.txt")
    nbytes = len(rows)
    pad = (-nbytes) % 16
    q = np.array([int(r[0], 16) for r in rows] + [0] * pad, dtype=np.uint8).reshape(1, -1)
    cols = q.shape[1] * 2
    s = np.full((1, cols // 32), 0x3C00, dtype=np.uint16)  # fp16 1.0
    w = oracle.dequant(q, s, 1, cols)[0]
    for b, r in enumerate(rows):
        assert w[2 * b] == int(r[1]), r
        assert w[2 * b + 1] == int(r[2]), r


def test_int4_group_scales_apply_per_32_columns():
    # two groups, codes -8..7 repeated; scales 0.5 (0x3800) and -2 (0xC000)
    vals = np.tile(np.arange(-8, 8), 4).reshape(1, 64)
    q = inputs.pack_int4(vals)
    s = np.array([[0x3800, 0xC000]], dtype=np.uint16)
    w = oracle.dequant(q, s, 1, 64)[0]
    np.testing.assert_array_equal(w[:32], vals[0, :32] * 0.5)
    np.testing.assert_array_equal(w[32:], vals[0, 32:] * -2.0)


def test_f16_decode_matches_numpy_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = oracle.f16_to_double(h)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.all(np.isinf(got[np.isinf(ref)]))
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_bf16_widen_matches_torch():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4096)
    bits = inputs.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.widen(bits.reshape(64, 64)).ravel(), ref)


# ------------------------------------------------------------------ routing
def _tiny_router(seed, T, d, E):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32)
    Wr = rng.standard_normal((E, d)).astype(np.float32)
    return x, Wr


@pytest.mark.parametrize("E,K", [(8, 1), (16, 4), (64, 10), (64, 64)])
def test_topk_equals_bruteforce_full_sort(E, K):
    x, Wr = _tiny_router(E * 100 + K, 12, 32, E)
    bias = np.random.default_rng(7).standard_normal(E).astype(np.float32)
    logits, idx, w, gap = oracle.route(x, Wr, bias, K)
    ref_logits = x.astype(np.float64) @ Wr.astype(np.float64).T + bias.astype(np.float64)
    np.testing.assert_allclose(logits, ref_logits, rtol=1e-12, atol=1e-12)
    for t in range(x.shape[0]):
        order = np.lexsort((np.arange(E), -ref_logits[t]))  # logit desc, then index asc
        np.testing.assert_array_equal(idx[t], order[:K])
        if K < E:
            assert gap[t] == pytest.approx(ref_logits[t, order[K - 1]] - ref_logits[t, order[K]], abs=1e-12)


def test_exact_ties_go_to_lower_index():
    d, E, K = 16, 12, 3
    rng = np.random.default_rng(3)
    Wr = rng.standard_normal((E, d)).astype(np.float32) * 0.01
    x = np.ones((1, d), np.float32)
    # experts 2, 5 and 9 get identical rows with the largest logit, expert 7 the same row too
    top = np.full(d, 0.5, np.float32)
    for e in (9, 5, 2, 7):
        Wr[e] = top
    logits, idx, w, _ = oracle.route(x, Wr, None, K)
    assert list(idx[0]) == [2, 5, 7]
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=0, atol=1e-15)


def test_two_expert_weights_closed_form():
    # E=3, K=2: renormalised weights of the kept pair are a logistic function of their logit gap,
    # independent of the third logit.
    d = 4
    Wr = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0]], np.float32)
    x = np.array([[0.75, -0.5, 0.25, 9.0]], np.float32)
    logits, idx, w, gap = oracle.route(x, Wr, None, 2)
    assert list(idx[0]) == [0, 2]
    a = 1.0 / (1.0 + math.exp(-(0.75 - 0.25)))
    assert w[0, 0] == pytest.approx(a, abs=1e-15)
    assert w[0, 1] == pytest.approx(1 - a, abs=1e-15)
    assert gap[0] == pytest.approx(0.25 - (-0.5), abs=1e-15)


def test_weights_sum_to_one_and_k_distinct_full_size_router():
    seed = inputs.workload_seed(2)
    T, d, E, K = 6, 2048, 512, 10
    x = inputs.gen_activations(seed, T, d)
    Wr = inputs.gen_router(seed, 0, E, d)
    _, idx, w, _ = oracle.route(x, Wr, None, K)
    for t in range(T):
        assert len(set(idx[t].tolist())) == K
        assert idx[t].min() >= 0 and idx[t].max() < E
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(w[t]) <= 1e-15)  # slot order = selection order (largest first)


def test_full_softmax_when_k_equals_e():
    # K = E keeps every expert: the weights are the plain softmax of the logits (torch.softmax).
    x, Wr = _tiny_router(11, 5, 24, 16)
    logits, idx, w, _ = oracle.route(x, Wr, None, 16)
    ref = torch.softmax(torch.from_numpy(logits), dim=-1).numpy()
    for t in range(5):
        np.testing.assert_allclose(w[t], ref[t, idx[t]], rtol=1e-13, atol=1e-16)


# ------------------------------------------------------------------ dispatch
@pytest.mark.parametrize("T,K,E", [(1, 10, 512), (7, 4, 16), (64, 10, 512), (300, 3, 5)])
def test_dispatch_matches_stable_argsort(T, K, E):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offs, perm, active = oracle.dispatch(idx, E)
    flat = idx.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(active, np.nonzero(np.bincount(flat, minlength=E))[0])
    assert sorted(perm.tolist()) == list(range(T * K))
    for e in range(E):
        seg = perm[offs[e]:offs[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // K) > 0)  # ascending token within an expert


# ------------------------------------------------------------------ experts and the layer
def _torch_ffn(Wgu, Wdn, x):
    f = Wgu.shape[0] // 2
    xt = torch.from_numpy(x)
    g = xt @ torch.from_numpy(Wgu[:f]).T
    u = xt @ torch.from_numpy(Wgu[f:]).T
    return (torch.nn.functional.silu(g) * u) @ torch.from_numpy(Wdn).T


def _deq(planes, d, f):
    if planes["gu_s"] is None:
        return planes["gu_q"].astype(np.float64), planes["dn_q"].astype(np.float64)
    return (oracle.dequant(planes["gu_q"], planes["gu_s"], 2 * f, d),
            oracle.dequant(planes["dn_q"], planes["dn_s"], d, f))


@pytest.mark.parametrize("wfmt,d,f", [("f32", 64, 32), ("int4", 128, 64), ("int4", 64, 192)])
def test_single_expert_is_dense_swiglu(wfmt, d, f):
    # E = 1, K = 1: the weight renormalises to exactly 1 and the layer is one dense SwiGLU FFN.
    seed = 99
    ex = inputs.gen_layer_experts(seed, 0, 1, d, f, wfmt)
    x = inputs.gen_activations(seed, 5, d, "bf16")
    Wr = inputs.gen_router(seed, 0, 1, d)
    y, idx, w = oracle.layer(x, Wr, None, ex, E=1, K=1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    Wgu, Wdn = _deq(ex[0], d, f)
    ref = _torch_ffn(Wgu, Wdn, oracle.widen(x)).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("shared", [False, True])
def test_k_equals_e_is_full_softmax_mixture(shared):
    d, f, E = 64, 32, 6
    seed = 123
    ex = inputs.gen_layer_experts(seed, 0, E + 1, d, f, "int4")
    sh_planes = ex.pop(E)
    sh = sh_planes if shared else None
    x = inputs.gen_activations(seed, 4, d, "bf16")
    Wr = inputs.gen_router(seed, 0, E, d) * 20.0
    y, idx, w = oracle.layer(x, Wr, None, ex, E=E, K=E, shared=sh)
    xd = oracle.widen(x)
    probs = torch.softmax(torch.from_numpy(xd @ Wr.astype(np.float64).T), dim=-1)
    ref = torch.zeros(4, d, dtype=torch.float64)
    for e in range(E):
        Wgu, Wdn = _deq(ex[e], d, f)
        ref += probs[:, e:e + 1] * _torch_ffn(Wgu, Wdn, xd)
    if shared:
        Wgu, Wdn = _deq(sh, d, f)
        ref += _torch_ffn(Wgu, Wdn, xd)
    ref = ref.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())


def test_topk_layer_matches_torch_gather_mixture():
    # K < E with a bias: torch.topk on the fp64 logits (no exact ties here) picks the experts,
    # the kept softmax mass is renormalised, the shared expert is added with weight 1.
    d, f, E, K, T = 64, 64, 16, 4, 6
    seed = 5
    ex = inputs.gen_layer_experts(seed, 0, E + 1, d, f, "int4")
    sh = ex.pop(E)
    x = inputs.gen_activations(seed, T, d, "bf16")
    Wr = inputs.gen_router(seed, 0, E, d) * 10.0
    bias = inputs.gen_zipf_prior(seed, 0, E)
    y, idx, w = oracle.layer(x, Wr, bias, ex, E=E, K=K, shared=sh)
    xd = torch.from_numpy(oracle.widen(x))
    lg = xd @ torch.from_numpy(Wr.astype(np.float64)).T + torch.from_numpy(bias.astype(np.float64))
    p = torch.softmax(lg, -1)
    top = torch.topk(lg, K, dim=-1)
    pk = torch.gather(p, 1, top.indices)
    wk = pk / pk.sum(-1, keepdim=True)
    outs = []
    for e in range(E):
        Wgu, Wdn = _deq(ex[e], d, f)
        outs.append(_torch_ffn(Wgu, Wdn, xd.numpy()))
    outs = torch.stack(outs, 1)  # [T, E, d]
    ref = (wk.unsqueeze(-1) * torch.gather(outs, 1, top.indices.unsqueeze(-1).expand(-1, -1, d))).sum(1)
    Wgu, Wdn = _deq(sh, d, f)
    ref = (ref + _torch_ffn(Wgu, Wdn, xd.numpy())).numpy()
    np.testing.assert_array_equal(idx, top.indices.numpy())
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())


def test_idx_override_uses_given_routing():
    d, f, E, K = 32, 32, 8, 2
    ex = inputs.gen_layer_experts(1, 0, E, d, f, "f32")
    x = inputs.gen_activations(1, 1, d, "f32")
    Wr = inputs.gen_router(1, 0, E, d)
    forced = np.array([[6, 1]], np.int32)
    y, idx, w = oracle.layer(x, Wr, None, ex, E=E, K=K, idx=forced)
    logits, _, _, _ = oracle.route(x, Wr, None, K)
    p = np.exp(logits[0] - logits[0].max())
    ww = p[[6, 1]] / p[[6, 1]].sum()
    np.testing.assert_allclose(w[0], ww, rtol=1e-14)
    ref = ww[0] * oracle.expert(ex[6], oracle.widen(x)[0]) + ww[1] * oracle.expert(ex[1], oracle.widen(x)[0])
    np.testing.assert_allclose(y[0], ref, rtol=1e-14, atol=1e-18)


# ------------------------------------------------------------------ RMSNorm (stack pre-norm)
def test_rmsnorm_closed_forms():
    d = 8
    x = np.array([[3, 4, 3, 4, 3, 4, 3, 4], [2] * 8], np.float32)
    out = oracle.rmsnorm(x, 0.0)
    np.testing.assert_allclose(out[0], x[0].astype(np.float64) / math.sqrt(12.5), rtol=1e-15)
    np.testing.assert_allclose(out[1], np.ones(d), rtol=1e-15)
    out_eps = oracle.rmsnorm(x[1:], 1.0)
    np.testing.assert_allclose(out_eps[0], 2 / math.sqrt(5.0) * np.ones(d), rtol=1e-15)
    # scale invariance with eps = 0
    np.testing.assert_allclose(oracle.rmsnorm(x * 8, 0.0), out, rtol=1e-15)


# ------------------------------------------------------------------ the pages' structural constants
def test_model_constants():
    c = {r[0]: int(r[1]) for r in _read_table("model_constants.txt")}
    assert c["layers"] * c["experts_per_layer"] == c["experts_total"]
    assert c["layers"] * c["top_k"] == c["experts_per_token_all_layers"]
    assert c["verify_window"] == c["max_drafts"] + 1
    assert abs(c["experts_per_token_all_layers"] / c["experts_total"] - 0.02) < 0.001
    # the oracle picks exactly top_k of experts_per_layer
    seed = inputs.workload_seed(2)
    x = inputs.gen_activations(seed, 2, 256)
    Wr = inputs.gen_router(seed, 0, c["experts_per_layer"], 256)
    _, idx, _, _ = oracle.route(x, Wr, None, c["top_k"])
    assert idx.shape == (2, c["top_k"]) and all(len(set(r)) == c["top_k"] for r in idx.tolist())

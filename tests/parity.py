"""Shared helpers of the GPU-vs-oracle parity tests (routing acceptance, tolerances, transfers)."""
from __future__ import annotations

import numpy as np

import oracle

# Layer output tolerance: max |y_gpu - y_ref| <= 2e-2 * max |y_ref| (bf16 activations, fp32 accumulation).
Y_TOL = 2e-2
# Near-tie threshold on the fp64 logits: tokens whose K-th / (K+1)-th logit gap is below it may
# legitimately pick either expert (fp32 logits on the GPU, fp64 in the oracle).
TIE_EPS = 1e-5
# Renormalised weights: fp32 softmax on the GPU vs fp64.
W_ATOL = 2e-6


def to_torch_act(x: np.ndarray, device="cuda"):
    import torch
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(x.copy()).to(device)


def from_torch_act(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def check_routing(logits: np.ndarray, idx_ref: np.ndarray, gap: np.ndarray, idx_gpu: np.ndarray):
    """Bit-exact routing except at near-ties.  Returns the number of flagged tokens.

    A token whose oracle gap between the K-th and (K+1)-th logit is below TIE_EPS is flagged; its GPU
    set is accepted if it differs from the oracle set only by experts whose logits are within TIE_EPS
    of the oracle's K-th logit.  Inside the kept set the slot order must follow the oracle logits,
    except between experts whose logits are within TIE_EPS of each other.
    """
    T, K = idx_ref.shape
    E = logits.shape[1]
    flagged = 0
    for t in range(T):
        g, r = idx_gpu[t], idx_ref[t]
        assert len(set(g.tolist())) == K, f"token {t}: repeated expert {g}"
        assert g.min() >= 0 and g.max() < E, f"token {t}: expert out of range {g}"
        lg = logits[t]
        if gap[t] < TIE_EPS:
            flagged += 1
            kth = lg[r[K - 1]]
            diff = set(g.tolist()) ^ set(r.tolist())
            assert all(abs(lg[e] - kth) < TIE_EPS for e in diff), f"token {t}: {g} vs {r}"
        else:
            assert set(g.tolist()) == set(r.tolist()), f"token {t}: gpu {sorted(g)} oracle {sorted(r)}"
        for k in range(K - 1):
            a, b = g[k], g[k + 1]
            ok = lg[a] > lg[b] or (lg[a] == lg[b] and a < b) or abs(lg[a] - lg[b]) < TIE_EPS
            assert ok, f"token {t}: slot order {g}"
        if gap[t] >= TIE_EPS and not np.array_equal(g, r):
            # only near-equal neighbours may swap
            for k in range(K):
                if g[k] != r[k]:
                    assert abs(lg[g[k]] - lg[r[k]]) < TIE_EPS, f"token {t}: order {g} vs {r}"
    return flagged


def check_dispatch(idx_gpu: np.ndarray, E: int, offs_gpu: np.ndarray, perm_gpu: np.ndarray):
    counts, offs, perm, active = oracle.dispatch(idx_gpu, E)
    np.testing.assert_array_equal(offs_gpu, offs)
    np.testing.assert_array_equal(perm_gpu, perm)
    return active


def y_error(y_gpu: np.ndarray, y_ref: np.ndarray) -> float:
    return float(np.abs(y_gpu - y_ref).max() / max(np.abs(y_ref).max(), 1e-30))

"""The five synthetic workloads and device-resident weight sets for them.

Shapes follow the model on the pages: 48 layers of 512 experts, 10 picked per token, a shared
expert ('Strata はなぜ少ない VRAM でも速いのか' (modeldock.net), section '問題：1,250 億パラメータと
12 GB'); verify passes of 1 + 3 tokens (section '予測してから検証する'); prefill chunks of thousands
of tokens (section '長いプロンプトを読む：大きなまとまりで流す').  Hidden size 2048 and expert width
768 are our choice (the pages fix neither; 24,576 experts of 3*2048*768 weights is about 116 B
parameters, close to the ~125 B the pages give for the model).

Weights are generated on the device (routed_expert_ffn_07_b300.capi.moe_gen_*) with the same
counter-based definition as routed_expert_ffn_07_b300.inputs, so any expert can be reproduced on
the host bit for bit.  Nothing here does MoE arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import inputs


@dataclass(frozen=True)
class Workload:
    idx: int
    name: str
    T: int
    d: int
    E: int
    K: int
    f: int
    shared: bool
    wfmt: str          # "int4" or "f32"
    act: str           # "bf16" or "f32"
    layers: int
    prenorm: bool
    zipf: float = 0.0  # > 0: router bias = Zipf(s) popularity prior
    stack: bool = False

    @property
    def seed(self) -> int:
        return inputs.workload_seed(self.idx)


WORKLOADS = {
    1: Workload(1, "tiny_layer_T8_d256_E64_k4_f128_fp32", 8, 256, 64, 4, 128, False, "f32", "f32", 1, False),
    2: Workload(2, "decode_layer_T1_d2048_E512_k10_f768_int4", 1, 2048, 512, 10, 768, True, "int4", "bf16", 1, False),
    3: Workload(3, "verify_stack_T4_L48_d2048_E512_k10_f768_int4", 4, 2048, 512, 10, 768, True, "int4", "bf16", 48,
                True, stack=True),
    4: Workload(4, "prefill_layer_T4096_d2048_E512_k10_f768_int4", 4096, 2048, 512, 10, 768, True, "int4", "bf16", 1,
                False),
    5: Workload(5, "skewed_decode_stack_T16_L48_zipf1.1_d2048_E512_k10_f768_int4", 16, 2048, 512, 10, 768, True,
                "int4", "bf16", 48, True, zipf=1.1, stack=True),
}


def expert_bytes(d: int, f: int) -> int:
    """Bytes of one int4 group-32 expert: 3*d*f/2 weight bytes + 3*d*f/32 fp16 scales."""
    return 3 * d * f // 2 + 3 * d * f // 32 * 2


@dataclass
class DeviceWeights:
    """All layers' planes on one device plus the registered library handle."""
    wl: Workload
    n_layers: int
    tensors: dict = field(default_factory=dict)


def alloc_and_fill(wl: Workload, n_layers: int | None = None, device: str = "cuda", layer0: int = 0):
    """Allocate and fill the weight planes of `n_layers` layers (default: the workload's count).

    Returns a dict of torch tensors: router [L,E,d] fp32, bias [L,E] fp32 or None, gu_q, gu_s, dn_q,
    dn_s (routed, stacked by layer then expert) and sh_gu_q, sh_gu_s, sh_dn_q, sh_dn_s (shared).
    Layer l of the returned set is generator layer layer0 + l.
    """
    import torch
    from . import capi

    L = wl.layers if n_layers is None else n_layers
    d, f, E = wl.d, wl.f, wl.E
    out = {}
    routers = np.stack([inputs.gen_router(wl.seed, layer0 + l, E, d) for l in range(L)])
    out["router"] = torch.from_numpy(routers).to(device)
    if wl.zipf > 0:
        b = np.stack([inputs.gen_zipf_prior(wl.seed, layer0 + l, E, wl.zipf) for l in range(L)])
        out["bias"] = torch.from_numpy(b).to(device)
    else:
        out["bias"] = None
    if wl.wfmt == "f32":
        ex = [inputs.gen_layer_experts(wl.seed, layer0 + l, E + 1, d, f, "f32") for l in range(L)]
        out["gu_q"] = torch.from_numpy(np.stack([np.stack([ex[l][e]["gu_q"] for e in range(E)]) for l in range(L)])).to(device)
        out["dn_q"] = torch.from_numpy(np.stack([np.stack([ex[l][e]["dn_q"] for e in range(E)]) for l in range(L)])).to(device)
        out["gu_s"] = out["dn_s"] = None
        out["sh_gu_q"] = torch.from_numpy(np.stack([ex[l][E]["gu_q"] for l in range(L)])).to(device)
        out["sh_dn_q"] = torch.from_numpy(np.stack([ex[l][E]["dn_q"] for l in range(L)])).to(device)
        out["sh_gu_s"] = out["sh_dn_s"] = None
        return out
    gu_b, dn_b = 2 * f * d // 2, d * f // 2
    gu_n, dn_n = 2 * f * d // 32, d * f // 32
    u8, f16 = torch.uint8, torch.float16
    out["gu_q"] = torch.empty((L, E, 2 * f, d // 2), dtype=u8, device=device)
    out["gu_s"] = torch.empty((L, E, 2 * f, d // 32), dtype=f16, device=device)
    out["dn_q"] = torch.empty((L, E, d, f // 2), dtype=u8, device=device)
    out["dn_s"] = torch.empty((L, E, d, f // 32), dtype=f16, device=device)
    out["sh_gu_q"] = torch.empty((L, 2 * f, d // 2), dtype=u8, device=device)
    out["sh_gu_s"] = torch.empty((L, 2 * f, d // 32), dtype=f16, device=device)
    out["sh_dn_q"] = torch.empty((L, d, f // 2), dtype=u8, device=device)
    out["sh_dn_s"] = torch.empty((L, d, f // 32), dtype=f16, device=device)
    st = torch.cuda.current_stream().cuda_stream
    for l in range(L):
        g = layer0 + l
        capi.moe_gen_int4_planes(out["gu_q"][l], wl.seed, g, inputs.T_GU_Q, 0, E, gu_b, st)
        capi.moe_gen_scale_planes(out["gu_s"][l], wl.seed, g, inputs.T_GU_S, 0, E, gu_n, st)
        capi.moe_gen_int4_planes(out["dn_q"][l], wl.seed, g, inputs.T_DN_Q, 0, E, dn_b, st)
        capi.moe_gen_scale_planes(out["dn_s"][l], wl.seed, g, inputs.T_DN_S, 0, E, dn_n, st)
        capi.moe_gen_int4_planes(out["sh_gu_q"][l], wl.seed, g, inputs.T_GU_Q, E, 1, gu_b, st)
        capi.moe_gen_scale_planes(out["sh_gu_s"][l], wl.seed, g, inputs.T_GU_S, E, 1, gu_n, st)
        capi.moe_gen_int4_planes(out["sh_dn_q"][l], wl.seed, g, inputs.T_DN_Q, E, 1, dn_b, st)
        capi.moe_gen_scale_planes(out["sh_dn_s"][l], wl.seed, g, inputs.T_DN_S, E, 1, dn_n, st)
    return out


def create_handle(wl: Workload, weights: dict, max_tokens: int | None = None, n_layers: int | None = None,
                  prenorm: bool | None = None):
    """moe_create + moe_set_layer for every layer of `weights`."""
    from . import capi

    L = weights["router"].shape[0] if n_layers is None else n_layers
    h = capi.moe_create(wl.d, wl.f, wl.E, wl.K, L, max_tokens or wl.T, has_shared=wl.shared,
                        prenorm=wl.prenorm if prenorm is None else prenorm, norm_eps=1e-6,
                        wfmt=capi.MOE_W_INT4_G32 if wl.wfmt == "int4" else capi.MOE_W_F32,
                        act=capi.MOE_ACT_BF16 if wl.act == "bf16" else capi.MOE_ACT_F32)
    for l in range(L):
        sh = wl.shared
        capi.moe_set_layer(
            h, l, weights["router"][l], weights["gu_q"][l],
            None if weights["gu_s"] is None else weights["gu_s"][l], weights["dn_q"][l],
            None if weights["dn_s"] is None else weights["dn_s"][l],
            router_b=None if weights["bias"] is None else weights["bias"][l],
            sh_gu_q=weights["sh_gu_q"][l] if sh else None,
            sh_gu_s=(weights["sh_gu_s"][l] if weights["sh_gu_s"] is not None else None) if sh else None,
            sh_dn_q=weights["sh_dn_q"][l] if sh else None,
            sh_dn_s=(weights["sh_dn_s"][l] if weights["sh_dn_s"] is not None else None) if sh else None)
    return h


def host_experts(wl: Workload, layer: int, experts) -> dict:
    """Host (numpy) copies of the listed experts of generator layer `layer` (index E = shared)."""
    return inputs.gen_layer_experts(wl.seed, layer, wl.E + 1, wl.d, wl.f, wl.wfmt, experts=experts)


def activations(wl: Workload, T: int | None = None, layer: int = 0) -> np.ndarray:
    return inputs.gen_activations(wl.seed, wl.T if T is None else T, wl.d, wl.act, layer=layer)

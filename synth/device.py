"""Synthetic model weights and KV pools on the GPU, filled by the generator of
synth.h (the same values the CPU oracle regenerates on demand).

Layouts are the ones the decode step's C ABI takes: [out][in] row-major
weights stacked over layers (and experts); KV pools [L][pages][n_kv][P][d].
"""
from __future__ import annotations

import torch

from . import (EMB, WQKV, WO, WR, WG, WU, WD, WLM, KPOOL, VPOOL, SG, SU, SD, BG, BU, BD, fill_device,
               fill_fp4_device, fill_bscales_device, fill_scales4_device, fill_fp8_device,
               fill_scales_device, fill_gains_device)
from .workloads import ModelShape


def _fill(t: torch.Tensor, n_streams: int, per: int, seed: int, kind: int, layer0=0, expert0=0,
          vary_layer=False, sigma=0.02, stream=0):
    assert t.dtype == torch.uint16 or t.dtype == torch.bfloat16
    assert t.numel() == n_streams * per
    fill_device(t.data_ptr(), n_streams, per, seed, kind, layer0, expert0, vary_layer, sigma, stream)


def device_weights(shape: ModelShape, seed: int, device="cuda", router_bias=None, gains=False) -> dict:
    """All weights of the model as torch tensors (BF16 stored as uint16; with
    expert_fp8 the expert matrices as uint8 E4M3 codes plus fp32 row scales; with
    expert_fp4 packed E2M1 codes, E4M3 block scales and fp32 row scales).  The
    RMSNorm gains are ones, or with `gains` the generator's seeded gains in
    [0.5, 2) (synth.h, "RMSNorm gains")."""
    st = torch.cuda.current_stream(device).cuda_stream
    L, H, E, I, V = shape.n_layers, shape.hidden, shape.n_experts, shape.inter, shape.vocab
    QKV, NQD = shape.qkv_rows(), shape.n_q * shape.head_dim
    sg = shape.weight_sigma
    u16 = dict(dtype=torch.uint16, device=device)
    w = {
        "embedding": torch.empty(V, H, **u16),
        "w_qkv": torch.empty(L, QKV, H, **u16),
        "w_o": torch.empty(L, H, NQD, **u16),
        "w_router": torch.empty(L, E, H, **u16),
        "w_lm": torch.empty(V, H, **u16),
        "norm_gamma": torch.ones(L, H, dtype=torch.float32, device=device),
        "final_gamma": torch.ones(H, dtype=torch.float32, device=device),
        "router_bias": (torch.as_tensor(router_bias, dtype=torch.float32).to(device)
                        if router_bias is not None else None),
    }
    if gains:
        fill_gains_device(w["norm_gamma"].data_ptr(), L, H, seed, stream=st)
        fill_gains_device(w["final_gamma"].data_ptr(), 1, H, seed, layer0=L, stream=st)
    _fill(w["embedding"], 1, V * H, seed, EMB, sigma=sg, stream=st)
    _fill(w["w_qkv"], L, QKV * H, seed, WQKV, vary_layer=True, sigma=sg, stream=st)
    _fill(w["w_o"], L, H * NQD, seed, WO, vary_layer=True, sigma=sg, stream=st)
    _fill(w["w_router"], L, E * H, seed, WR, vary_layer=True, sigma=sg, stream=st)
    if getattr(shape, "expert_fp8", False):
        # E4M3 codes and one fp32 scale per output row (synth.h, "FP8 expert weights")
        u8 = dict(dtype=torch.uint8, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        w["w_gate"] = torch.empty(L, E, I, H, **u8)
        w["w_up"] = torch.empty(L, E, I, H, **u8)
        w["w_down"] = torch.empty(L, E, H, I, **u8)
        w["w_gate_scale"] = torch.empty(L, E, I, **f32)
        w["w_up_scale"] = torch.empty(L, E, I, **f32)
        w["w_down_scale"] = torch.empty(L, E, H, **f32)
        for l in range(L):
            for t, kind in ((w["w_gate"], WG), (w["w_up"], WU), (w["w_down"], WD)):
                fill_fp8_device(t[l].data_ptr(), E, t[l].numel() // E, seed, kind, layer0=l, stream=st)
            for t, kind in ((w["w_gate_scale"], SG), (w["w_up_scale"], SU), (w["w_down_scale"], SD)):
                fill_scales_device(t[l].data_ptr(), E, t[l].numel() // E, seed, kind, layer0=l, sigma=sg,
                                   stream=st)
        return _rest(w, shape, seed, sg, st)
    if getattr(shape, "expert_fp4", False):
        # two E2M1 codes per byte, an E4M3 scale per 16 inputs, a scale per output row
        # (synth.h, "FP4 expert weights")
        u8 = dict(dtype=torch.uint8, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        w["w_gate"] = torch.empty(L, E, I, H // 2, **u8)
        w["w_up"] = torch.empty(L, E, I, H // 2, **u8)
        w["w_down"] = torch.empty(L, E, H, I // 2, **u8)
        w["w_gate_bscale"] = torch.empty(L, E, I, H // 16, **u8)
        w["w_up_bscale"] = torch.empty(L, E, I, H // 16, **u8)
        w["w_down_bscale"] = torch.empty(L, E, H, I // 16, **u8)
        w["w_gate_scale"] = torch.empty(L, E, I, **f32)
        w["w_up_scale"] = torch.empty(L, E, I, **f32)
        w["w_down_scale"] = torch.empty(L, E, H, **f32)
        for l in range(L):
            for t, kind in ((w["w_gate"], WG), (w["w_up"], WU), (w["w_down"], WD)):
                fill_fp4_device(t[l].data_ptr(), E, t[l].numel() // E, seed, kind, layer0=l, stream=st)
            for t, kind in ((w["w_gate_bscale"], BG), (w["w_up_bscale"], BU), (w["w_down_bscale"], BD)):
                fill_bscales_device(t[l].data_ptr(), E, t[l].numel() // E, seed, kind, layer0=l, stream=st)
            for t, kind in ((w["w_gate_scale"], SG), (w["w_up_scale"], SU), (w["w_down_scale"], SD)):
                fill_scales4_device(t[l].data_ptr(), E, t[l].numel() // E, seed, kind, layer0=l, sigma=sg,
                                    stream=st)
        return _rest(w, shape, seed, sg, st)
    w["w_gate"] = torch.empty(L, E, I, H, **u16)
    w["w_up"] = torch.empty(L, E, I, H, **u16)
    w["w_down"] = torch.empty(L, E, H, I, **u16)
    for l in range(L):
        _fill(w["w_gate"][l], E, I * H, seed, WG, layer0=l, sigma=sg, stream=st)
        _fill(w["w_up"][l], E, I * H, seed, WU, layer0=l, sigma=sg, stream=st)
        _fill(w["w_down"][l], E, H * I, seed, WD, layer0=l, sigma=sg, stream=st)
    return _rest(w, shape, seed, sg, st)


def _rest(w, shape, seed, sg, st):
    V, H = shape.vocab, shape.hidden
    _fill(w["w_lm"], 1, V * H, seed, WLM, sigma=sg, stream=st)
    return w


def device_pools(shape: ModelShape, seed: int, num_pages: int, device="cuda"):
    """K and V pools [L][num_pages][n_kv][P][d], every slot filled with the
    generator's values (slots past a sequence's length are never read)."""
    st = torch.cuda.current_stream(device).cuda_stream
    L, nkv, P, d = shape.n_layers, shape.n_kv, shape.page_size, shape.head_dim
    per = num_pages * nkv * P * d
    k = torch.empty(L, num_pages, nkv, P, d, dtype=torch.uint16, device=device)
    v = torch.empty_like(k)
    _fill(k, L, per, seed, KPOOL, vary_layer=True, sigma=shape.kv_sigma, stream=st)
    _fill(v, L, per, seed, VPOOL, vary_layer=True, sigma=shape.kv_sigma, stream=st)
    return k, v

"""Seeded synthetic inputs for the decode step.

`synth.h` defines one counter-based generator (splitmix64 + an Irwin-Hall sum,
rounded to BF16).  `libsynth.so` evaluates it on the host (for the oracle and
the tests) or fills device buffers with it (for the GPU path).  The module holds
no arithmetic of the decode step.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .workloads import (MODELS, WORKLOADS, ModelShape, Workload, StepInputs, make_inputs,  # noqa: F401
                        step_kv_bytes, seq_lens_for, block_tables_for, tokens_for,
                        zipf_router_bias)

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsynth.so")

EMB, WQKV, WO, WR, WG, WU, WD, WLM, KPOOL, VPOOL, SG, SU, SD, BG, BU, BD, GAMMA = range(1, 18)

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            from .build import build
            build()
        L = ctypes.CDLL(LIB_PATH)
        u64, u32 = ctypes.c_uint64, ctypes.c_uint32
        L.synth_fill_device.restype = ctypes.c_int
        L.synth_fill_device.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_void_p]
        L.synth_fill_host.restype = None
        L.synth_fill_host.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int,
                                      ctypes.c_double]
        L.synth_raw.restype = u64
        L.synth_raw.argtypes = [u64, u64]
        L.synth_fill_fp8_device.restype = ctypes.c_int
        L.synth_fill_fp8_device.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int,
                                            ctypes.c_void_p]
        L.synth_fill_scales_device.restype = ctypes.c_int
        L.synth_fill_scales_device.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int,
                                               ctypes.c_double, ctypes.c_void_p]
        L.synth_fill_fp8_host.restype = None
        L.synth_fill_fp8_host.argtypes = [ctypes.c_void_p, u64, u64, u32, u32, u32]
        L.synth_fill_scales_host.restype = None
        L.synth_fill_scales_host.argtypes = [ctypes.c_void_p, u64, u64, u32, u32, u32, ctypes.c_double]
        L.synth_e4m3.restype = ctypes.c_uint8
        L.synth_e4m3.argtypes = [ctypes.c_float]
        for name in ("synth_fill_fp4_device", "synth_fill_bscales_device"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_scales_base_device.restype = ctypes.c_int
        L.synth_fill_scales_base_device.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, u32, u32, ctypes.c_int,
                                                    ctypes.c_float, ctypes.c_void_p]
        for name in ("synth_fill_fp4_host", "synth_fill_bscales_host"):
            f = getattr(L, name)
            f.restype = None
            f.argtypes = [ctypes.c_void_p, u64, u64, u32, u32, u32]
        L.synth_fill_scales_base_host.restype = None
        L.synth_fill_scales_base_host.argtypes = [ctypes.c_void_p, u64, u64, u32, u32, u32, ctypes.c_float]
        L.synth_fp4_base_of.restype = ctypes.c_float
        L.synth_fp4_base_of.argtypes = [ctypes.c_double]
        L.synth_e2m1.restype = ctypes.c_uint8
        L.synth_e2m1.argtypes = [ctypes.c_float]
        L.synth_fill_gains_device.restype = ctypes.c_int
        L.synth_fill_gains_device.argtypes = [ctypes.c_void_p, u64, u64, u64, u32, ctypes.c_void_p]
        L.synth_fill_gains_host.restype = None
        L.synth_fill_gains_host.argtypes = [ctypes.c_void_p, u64, u64, u64, u32]
        _lib = L
    return _lib


def fill_host(n_streams: int, per_stream: int, seed: int, kind: int, layer0: int = 0,
              expert0: int = 0, vary_layer: bool = False, sigma: float = 0.02) -> np.ndarray:
    """uint16 BF16 bit patterns, shape [n_streams, per_stream]."""
    out = np.empty((n_streams, per_stream), dtype=np.uint16)
    lib().synth_fill_host(out.ctypes.data, n_streams, per_stream, seed, kind, layer0, expert0,
                          int(vary_layer), sigma)
    return out


def fill_device(ptr: int, n_streams: int, per_stream: int, seed: int, kind: int, layer0: int = 0,
                expert0: int = 0, vary_layer: bool = False, sigma: float = 0.02,
                stream: int = 0) -> None:
    rc = lib().synth_fill_device(ptr, n_streams, per_stream, seed, kind, layer0, expert0,
                                 int(vary_layer), sigma, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed with CUDA error {rc}")


def fill_fp8_host(n: int, seed: int, kind: int, layer: int = 0, expert: int = 0) -> np.ndarray:
    """uint8 E4M3 codes of one FP8 expert matrix (n elements, row-major)."""
    out = np.empty(n, dtype=np.uint8)
    lib().synth_fill_fp8_host(out.ctypes.data, n, seed, kind, layer, expert)
    return out


def fill_scales_host(rows: int, seed: int, kind: int, layer: int = 0, expert: int = 0,
                     sigma: float = 0.02) -> np.ndarray:
    """float32 row scales of one FP8 expert matrix (kind SG, SU or SD)."""
    out = np.empty(rows, dtype=np.float32)
    lib().synth_fill_scales_host(out.ctypes.data, rows, seed, kind, layer, expert, sigma)
    return out


def e4m3(f: float) -> int:
    """The generator's E4M3 encoding of one binary32 (|f| <= 448)."""
    return int(lib().synth_e4m3(f))


def fill_fp8_device(ptr: int, n_streams: int, per_stream: int, seed: int, kind: int, layer0: int = 0,
                    expert0: int = 0, vary_layer: bool = False, stream: int = 0) -> None:
    rc = lib().synth_fill_fp8_device(ptr, n_streams, per_stream, seed, kind, layer0, expert0,
                                     int(vary_layer), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_fp8_device failed with CUDA error {rc}")


def fill_scales_device(ptr: int, n_streams: int, rows: int, seed: int, kind: int, layer0: int = 0,
                       expert0: int = 0, vary_layer: bool = False, sigma: float = 0.02,
                       stream: int = 0) -> None:
    rc = lib().synth_fill_scales_device(ptr, n_streams, rows, seed, kind, layer0, expert0,
                                        int(vary_layer), sigma, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_scales_device failed with CUDA error {rc}")


def fill_fp4_host(n_bytes: int, seed: int, kind: int, layer: int = 0, expert: int = 0) -> np.ndarray:
    """uint8 packed E2M1 codes of one FP4 expert matrix (element 2j in the low
    nibble of byte j), n_bytes = elements / 2."""
    out = np.empty(n_bytes, dtype=np.uint8)
    lib().synth_fill_fp4_host(out.ctypes.data, n_bytes, seed, kind, layer, expert)
    return out


def fill_bscales_host(n: int, seed: int, kind: int, layer: int = 0, expert: int = 0) -> np.ndarray:
    """uint8 E4M3 block scales of one FP4 expert matrix (kind BG, BU or BD)."""
    out = np.empty(n, dtype=np.uint8)
    lib().synth_fill_bscales_host(out.ctypes.data, n, seed, kind, layer, expert)
    return out


def fp4_base(sigma: float = 0.02) -> float:
    return float(lib().synth_fp4_base_of(sigma))


def fill_scales4_host(rows: int, seed: int, kind: int, layer: int = 0, expert: int = 0,
                      sigma: float = 0.02) -> np.ndarray:
    """float32 row scales of one FP4 expert matrix (kind SG, SU or SD)."""
    out = np.empty(rows, dtype=np.float32)
    lib().synth_fill_scales_base_host(out.ctypes.data, rows, seed, kind, layer, expert, fp4_base(sigma))
    return out


def e2m1(f: float) -> int:
    """The generator's E2M1 encoding of one binary32 (|f| <= 6)."""
    return int(lib().synth_e2m1(f))


def fill_fp4_device(ptr: int, n_streams: int, per_stream: int, seed: int, kind: int, layer0: int = 0,
                    expert0: int = 0, vary_layer: bool = False, stream: int = 0) -> None:
    rc = lib().synth_fill_fp4_device(ptr, n_streams, per_stream, seed, kind, layer0, expert0,
                                     int(vary_layer), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_fp4_device failed with CUDA error {rc}")


def fill_bscales_device(ptr: int, n_streams: int, per_stream: int, seed: int, kind: int, layer0: int = 0,
                        expert0: int = 0, vary_layer: bool = False, stream: int = 0) -> None:
    rc = lib().synth_fill_bscales_device(ptr, n_streams, per_stream, seed, kind, layer0, expert0,
                                         int(vary_layer), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_bscales_device failed with CUDA error {rc}")


def fill_scales4_device(ptr: int, n_streams: int, rows: int, seed: int, kind: int, layer0: int = 0,
                        expert0: int = 0, vary_layer: bool = False, sigma: float = 0.02,
                        stream: int = 0) -> None:
    rc = lib().synth_fill_scales_base_device(ptr, n_streams, rows, seed, kind, layer0, expert0,
                                             int(vary_layer), fp4_base(sigma), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_scales_base_device failed with CUDA error {rc}")


def fill_gains_host(n_layers: int, per_layer: int, seed: int, layer0: int = 0) -> np.ndarray:
    """float32 RMSNorm gains [n_layers][per_layer] of layers layer0 .. (stream (GAMMA, l, 0))."""
    out = np.empty((n_layers, per_layer), dtype=np.float32)
    lib().synth_fill_gains_host(out.ctypes.data, n_layers, per_layer, seed, layer0)
    return out


def gains_host(shape, seed: int):
    """The seeded gains of a model: (layer norms [L][H], final norm [H]), float32;
    the final norm's stream is layer n_layers."""
    return (fill_gains_host(shape.n_layers, shape.hidden, seed),
            fill_gains_host(1, shape.hidden, seed, layer0=shape.n_layers)[0])


def fill_gains_device(ptr: int, n_layers: int, per_layer: int, seed: int, layer0: int = 0,
                      stream: int = 0) -> None:
    rc = lib().synth_fill_gains_device(ptr, n_layers, per_layer, seed, layer0, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_gains_device failed with CUDA error {rc}")


def raw(key: int, idx: int) -> int:
    return int(lib().synth_raw(key, idx))


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)

"""ctypes front end of the counter-based generator in ``gen.c``.

Everything here produces input DATA (activations, router weights, quantised
expert weights).  None of the layer's arithmetic lives here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

from .configs import (Family, TID_ROUTER_BIAS, TID_ROUTER_W, TID_W13, TID_W2, TID_X)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_gen.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so (gcc, portable C: no -march flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC,
                        "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i64, dbl, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        L.gen_stream_key.argtypes = [u64, u64]
        L.gen_stream_key.restype = u64
        L.gen_normal_at.argtypes = [u64, u64, u64]
        L.gen_normal_at.restype = dbl
        L.gen_e4m3_encode.argtypes = [ctypes.c_float]
        L.gen_e4m3_encode.restype = ctypes.c_uint8
        L.gen_e4m3_encode_array.argtypes = [vp, i64, vp]
        L.gen_e4m3_encode_array.restype = None
        L.gen_normal_f32.argtypes = [u64, u64, i64, dbl, vp, i32]
        L.gen_normal_bf16.argtypes = [u64, u64, i64, dbl, vp, i32]
        L.gen_blockwise_e4m3.argtypes = [u64, u64, i64, i64, i64, dbl, vp, vp, i32]
        L.gen_nvfp4.argtypes = [u64, u64, i64, i64, i64, dbl, vp, vp, vp, i32]
        L.gen_e2m1_encode.argtypes = [ctypes.c_float]
        L.gen_e2m1_encode.restype = ctypes.c_uint8
        for f in (L.gen_normal_f32, L.gen_normal_bf16, L.gen_blockwise_e4m3, L.gen_nvfp4):
            f.restype = i32
        _lib = L
    return _lib


def _threads(n: int | None) -> int:
    return n if n else (os.cpu_count() or 1)


def normal_f32(seed: int, tid: int, shape, std: float, nthreads=None) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().gen_normal_f32(seed, tid, out.size, std, out.ctypes.data, _threads(nthreads))
    return out


def normal_bf16(seed: int, tid: int, shape, std: float = 1.0, nthreads=None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, std) values."""
    out = np.empty(shape, dtype=np.uint16)
    lib().gen_normal_bf16(seed, tid, out.size, std, out.ctypes.data, _threads(nthreads))
    return out


def blockwise_e4m3(seed: int, tid: int, E: int, R: int, C: int, std: float, nthreads=None):
    codes = np.empty((E, R, C), dtype=np.uint8)
    scales = np.empty((E, R // 128, C // 128), dtype=np.float32)
    rc = lib().gen_blockwise_e4m3(seed, tid, E, R, C, std, codes.ctypes.data,
                                  scales.ctypes.data, _threads(nthreads))
    if rc != 0:
        raise ValueError("R and C must be multiples of 128")
    return codes, scales


def nvfp4(seed: int, tid: int, E: int, R: int, C: int, std: float, nthreads=None):
    """E matrices R x C of N(0, std) values in the FP4 expert format: packed
    e2m1 codes [E, R, C/2], e4m3 block scales [E, R, C/16], f32 global
    scales [E] (the same normal streams as ``blockwise_e4m3``)."""
    codes = np.empty((E, R, C // 2), dtype=np.uint8)
    bsc = np.empty((E, R, C // 16), dtype=np.uint8)
    gsc = np.empty((E,), dtype=np.float32)
    rc = lib().gen_nvfp4(seed, tid, E, R, C, std, codes.ctypes.data, bsc.ctypes.data,
                         gsc.ctypes.data, _threads(nthreads))
    if rc != 0:
        raise ValueError("C must be a multiple of 16")
    return codes, bsc, gsc


def e4m3_encode(values: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().gen_e4m3_encode_array(v.ctypes.data, v.size, out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to f32 (a bf16 is the top half of an f32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerWeights:
    router_w: np.ndarray            # f32 [E, H]
    router_bias: np.ndarray | None  # f32 [E] or None
    w13: np.ndarray                 # u8 e4m3 [E, 2I, H]; rows [0,I) gate, [I,2I) up
    s13: np.ndarray                 # f32 [E, 2I/128, H/128]
    w2: np.ndarray                  # u8 e4m3 [E, H, I]
    s2: np.ndarray                  # f32 [E, H/128, I/128]


def make_weights(fam: Family, nthreads=None) -> LayerWeights:
    E, H, I, s = fam.n_experts, fam.hidden, fam.inter, fam.seed
    router_w = normal_f32(s, TID_ROUTER_W, (E, H), fam.router_std, nthreads)
    bias = None
    if fam.bias_std is not None:
        bias = normal_f32(s, TID_ROUTER_BIAS, (E,), fam.bias_std, nthreads)
    w13, s13 = blockwise_e4m3(s, TID_W13, E, 2 * I, H, fam.w_std, nthreads)
    w2, s2 = blockwise_e4m3(s, TID_W2, E, H, I, fam.w_std, nthreads)
    return LayerWeights(router_w, bias, w13, s13, w2, s2)


@dataclass
class LayerWeightsFP4:
    router_w: np.ndarray            # f32 [E, H]
    router_bias: np.ndarray | None  # f32 [E] or None
    w13: np.ndarray                 # u8 [E, 2I, H/2] packed e2m1; rows [0,I) gate, [I,2I) up
    sf13: np.ndarray                # u8 e4m3 [E, 2I, H/16]
    g13: np.ndarray                 # f32 [E]
    w2: np.ndarray                  # u8 [E, H, I/2]
    sf2: np.ndarray                 # u8 e4m3 [E, H, I/16]
    g2: np.ndarray                  # f32 [E]


def make_weights_fp4(fam: Family, nthreads=None) -> LayerWeightsFP4:
    """The family's layer with FP4 experts: the same router and the same
    normal streams as ``make_weights``, quantised to the FP4 format."""
    E, H, I, s = fam.n_experts, fam.hidden, fam.inter, fam.seed
    router_w = normal_f32(s, TID_ROUTER_W, (E, H), fam.router_std, nthreads)
    bias = None
    if fam.bias_std is not None:
        bias = normal_f32(s, TID_ROUTER_BIAS, (E,), fam.bias_std, nthreads)
    w13, sf13, g13 = nvfp4(s, TID_W13, E, 2 * I, H, fam.w_std, nthreads)
    w2, sf2, g2 = nvfp4(s, TID_W2, E, H, I, fam.w_std, nthreads)
    return LayerWeightsFP4(router_w, bias, w13, sf13, g13, w2, sf2, g2)


def make_x(fam: Family, T: int, nthreads=None) -> np.ndarray:
    """bf16 bits [T, H] of x ~ N(0, 1)."""
    return normal_bf16(fam.x_seed(T), TID_X, (T, fam.hidden), 1.0, nthreads)

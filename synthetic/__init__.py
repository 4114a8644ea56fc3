"""Seeded, position-addressable synthetic inputs for the CSA KV compressor.

Test and benchmark infrastructure shared by the oracle side and the GPU side.
It holds none of the compressor's arithmetic: it only draws numbers (SplitMix64
streams, Box-Muller normals) and lays them out in the shapes of the workloads
below.  The generator itself is the small C file ``synth.c`` beside this module,
built on first use with the host C compiler.

Tensor ids (the ``tid`` of a stream):
  1 token hidden states x, one stream per sequence b, index t*dim + k
  2 wkv, 3 wgate, 4 RMSNorm gain, 5 decode start positions, 6 outlier-token mask
A workload's seed is fixed per workload (tiny 0, Flash CSA 1, HCA 2, decode 3,
long sweep 4).  Each compressor instance inside a workload gets its own weight
stream number, so several layers can be drawn from one seed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcsa_synth.so")
_lock = threading.Lock()
_lib = None

TID_X, TID_WKV, TID_WGATE, TID_GAIN, TID_START, TID_OUTLIER = 1, 2, 3, 4, 5, 6


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library (idempotent)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl, ptr, cint = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p,
                                         ctypes.c_int)
            lib.synth_normal.argtypes = [u64, u64, u64, u64, i64, dbl, dbl, ptr, cint]
            lib.synth_normal.restype = None
            lib.synth_uniform.argtypes = [u64, u64, u64, u64, i64, ptr, cint]
            lib.synth_uniform.restype = None
            lib.synth_uniform1.argtypes = [u64, u64, u64, u64]
            lib.synth_uniform1.restype = dbl
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal(seed: int, tid: int, stream: int, first: int, count: int, mean: float = 0.0,
           scale: float = 1.0) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    if count:
        _load().synth_normal(seed, tid, stream, first, count, mean, scale, out.ctypes.data, _threads())
    return out


def uniform(seed: int, tid: int, stream: int, first: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    if count:
        _load().synth_uniform(seed, tid, stream, first, count, out.ctypes.data, _threads())
    return out


def uniform1(seed: int, tid: int, stream: int, index: int) -> float:
    return _load().synth_uniform1(seed, tid, stream, index)


# --------------------------------------------------------------------------------------------
# workload recipes


@dataclass(frozen=True)
class Layer:
    """One compressor instance: its shape and the distributions of its weights."""
    dim: int
    head_dim: int
    ratio: int
    overlap: int
    w_std: float
    gate_scale: float = 1.0  # wgate std = w_std * gate_scale
    rope_dim: int = 64
    fp4: int = 1
    weight_stream: int = 0

    @property
    def width(self) -> int:  # rows of wkv (and of wgate)
        return (1 + self.overlap) * self.head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: tuple
    batch: int
    tokens: tuple  # sequence lengths exercised (prefill) or steps (decode)
    outlier_frac: float = 0.0
    outlier_scale: float = 20.0
    decode_steps: int = 0
    start_pos_hi: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)


FLASH_DIM, FLASH_H = 4096, 512

TINY = Workload("tiny parity: B=1 N=64 dim=256 head_dim=64 ratio=2", 0,
                (Layer(256, 64, 2, 0, 1.0 / 16, rope_dim=0, fp4=0),), 1, (64,), decode_steps=64)
FLASH_CSA = Workload("Flash CSA prefill: B=1 N=4096 dim=4096 ratio=4 overlapped", 1,
                     (Layer(FLASH_DIM, FLASH_H, 4, 1, 1.0 / 64),), 1, (4096,))
HCA = Workload("HCA prefill: B=4 N=16461 dim=4096 ratio=128", 2,
               (Layer(FLASH_DIM, FLASH_H, 128, 0, 1.0 / 64, gate_scale=4.0),), 4, (16384 + 77,))
DECODE = Workload("batched decode: B=128, ratio 4 overlapped + ratio 128, 512 steps", 3,
                  (Layer(FLASH_DIM, FLASH_H, 4, 1, 1.0 / 64, weight_stream=0),
                   Layer(FLASH_DIM, FLASH_H, 128, 0, 1.0 / 64, weight_stream=1)), 128, (1,),
                  decode_steps=512, start_pos_hi=8192)
LONG = Workload("long-context prefill sweep", 4,
                (Layer(FLASH_DIM, FLASH_H, 4, 1, 1.0 / 64, weight_stream=0),
                 Layer(FLASH_DIM, FLASH_H, 128, 0, 1.0 / 64, weight_stream=1)), 1,
                (16384, 65536, 131072), outlier_frac=0.01, outlier_scale=20.0,
                extra={"batched": (8, 8192)})

# the indexer's 128-wide compressor of a CSA layer (its keys take the power-of-two fp4 round
# trip), and the ratio-2 "pool token pairs" layers, at the Flash width
INDEXER = Workload("Flash CSA indexer compressor: B=1 N=4096 dim=4096 head_dim=128 ratio=4 overlapped", 5,
                   (Layer(FLASH_DIM, 128, 4, 1, 1.0 / 64, fp4=2),), 1, (4096,))
PAIRS = Workload("pool token pairs: B=2 N=4096 dim=4096 head_dim=512 ratio=2", 6,
                 (Layer(FLASH_DIM, FLASH_H, 2, 0, 1.0 / 64),), 2, (4096,))

WORKLOADS = {"tiny": TINY, "flash_csa": FLASH_CSA, "hca": HCA, "decode": DECODE, "long": LONG,
             "indexer": INDEXER, "pairs": PAIRS}


def weights(seed: int, layer: Layer):
    """(wkv [C, dim], wgate [C, dim], gain [head_dim]) as float32 arrays, C = layer.width."""
    c, d = layer.width, layer.dim
    s = layer.weight_stream
    wkv = normal(seed, TID_WKV, s, 0, c * d, 0.0, layer.w_std).reshape(c, d)
    wgate = normal(seed, TID_WGATE, s, 0, c * d, 0.0, layer.w_std * layer.gate_scale).reshape(c, d)
    gain = normal(seed, TID_GAIN, s, 0, layer.head_dim, 1.0, 0.02)
    return wkv, wgate, gain


def outlier_mask(seed: int, b: int, t0: int, t1: int, frac: float) -> np.ndarray:
    if frac <= 0.0:
        return np.zeros(t1 - t0, dtype=bool)
    u = uniform(seed, TID_OUTLIER, b, t0, t1 - t0)
    return u < frac


def tokens(seed: int, b: int, t0: int, t1: int, dim: int, outlier_frac: float = 0.0,
           outlier_scale: float = 20.0) -> np.ndarray:
    """float32 hidden states of tokens [t0, t1) of sequence b, shape [t1-t0, dim].

    Standard normal; a token flagged by the outlier mask is scaled by outlier_scale.
    Round to bf16 (the recipe's input type) with torch on the caller's side.
    """
    x = normal(seed, TID_X, b, t0 * dim, (t1 - t0) * dim).reshape(t1 - t0, dim)
    if outlier_frac > 0.0:
        m = outlier_mask(seed, b, t0, t1, outlier_frac)
        x[m] *= np.float32(outlier_scale)
    return x


def start_positions(seed: int, batch: int, hi: int) -> np.ndarray:
    """Per-sequence decode start positions, uniform on {0, ..., hi-1}."""
    u = uniform(seed, TID_START, 0, 0, batch).astype(np.float64)
    return np.minimum((u * hi).astype(np.int64), hi - 1).astype(np.int32)

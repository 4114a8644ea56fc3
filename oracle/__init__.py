"""ctypes wrapper of the CPU oracle (``csa_oracle.cpp``).

TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow C++ restatement of the
compressed-sparse-attention KV Compressor written from the pages it cites
(header of ``csa_oracle.h``).  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module; the library in
``deepseek_v4_compressed_wkv_gb300`` never does, and shares no code with it.

Arrays cross the boundary as numpy arrays; bf16 values travel as their uint16
bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (idempotent)."""
    srcs = [os.path.join(_HERE, f) for f in ("csa_oracle.cpp", "csa_oracle.h")]
    newest = max(os.path.getmtime(s) for s in srcs)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-o", tmp, srcs[0]], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Options(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("rope_dim", ctypes.c_int), ("rope_base", ctypes.c_double),
                ("rope_factor", ctypes.c_double), ("rope_orig_len", ctypes.c_int), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("fp4", ctypes.c_int), ("eps", ctypes.c_double)]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, I64, D, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
        U16, U8 = ctypes.c_uint16, ctypes.c_uint8
        sig = {
            "oracle_bf16_from_f32": ([F], U16), "oracle_bf16_from_f64": ([D], U16),
            "oracle_bf16_to_f32": ([U16], F), "oracle_e4m3_from_f32": ([F], U8),
            "oracle_e4m3_to_f64": ([U8], D), "oracle_e2m1_from_f32": ([F], U8), "oracle_e2m1_to_f64": ([U8], D),
            "oracle_fp4_e4m3": ([P, I64, P, P, P], None),
            "oracle_fp4_e8m0": ([P, I64, P, P, P], None),
            "oracle_yarn_freqs": ([I, D, D, I, D, D, P], None),
            "oracle_yarn_bounds": ([I, D, I, D, D, P, P], None),
            "oracle_pool": ([P, P, I, I, P, P], None),
            "oracle_epilogue": ([P, P, I64, P], None),
            "oracle_linear": ([P, I64, I, P, I, P, I], None),
            "oracle_create": ([I, I, I, I, P], P), "oracle_destroy": ([P], None),
            "oracle_set_weights": ([P, P, P, P], None),
            "oracle_prefill": ([P, P, I, I, I, P, P, P, P, I], I),
            "oracle_prefill_groups": ([P, P, I, P, I, P, P, P, P, I], I),
            "oracle_prefill_chunk": ([P, P, I, I, I, I, P, P, P, P, I], I),
            "oracle_decode": ([P, P, I, P, P, P, P, P, P, I], I),
            "oracle_state_reset": ([P], None), "oracle_state_elems": ([P], I64),
            "oracle_set_gate_bias": ([P, P], None),
            "oracle_state_export": ([P, P, P], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def lib():
    return _load()


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---- number formats -----------------------------------------------------------------------

def bf16_from_f32(v: float) -> int:
    return int(_load().oracle_bf16_from_f32(v))


def bf16_from_f64(v: float) -> int:
    return int(_load().oracle_bf16_from_f64(v))


def bf16_to_f32(h: int) -> float:
    return float(_load().oracle_bf16_to_f32(h))


def e4m3_from_f32(v: float) -> int:
    return int(_load().oracle_e4m3_from_f32(v))


def e4m3_to_f64(b: int) -> float:
    return float(_load().oracle_e4m3_to_f64(b))


def e2m1_from_f32(v: float) -> int:
    return int(_load().oracle_e2m1_from_f32(v))


def e2m1_to_f64(c: int) -> float:
    return float(_load().oracle_e2m1_to_f64(c))


def fp4_e4m3(bf16_bits: np.ndarray):
    """fp4 round trip of a uint16 (bf16 bits) array whose size is a multiple of 16.

    Returns (codes uint8 [n/2], scales uint8 [n/16], out uint16 [n])."""
    x = np.ascontiguousarray(bf16_bits, dtype=np.uint16).reshape(-1)
    nb = x.size // 16
    codes = np.zeros(nb * 8, np.uint8)
    scales = np.zeros(nb, np.uint8)
    out = np.zeros(nb * 16, np.uint16)
    _load().oracle_fp4_e4m3(_ptr(x), nb, _ptr(codes), _ptr(scales), _ptr(out))
    return codes, scales, out


def fp4_e8m0(bf16_bits: np.ndarray):
    """The indexer's fp4 round trip (power-of-two scales, block 32) of a uint16 (bf16 bits)
    array whose size is a multiple of 32.  Returns (codes uint8 [n/2], scales uint8 [n/32]
    e8m0 bytes, out uint16 [n])."""
    x = np.ascontiguousarray(bf16_bits, dtype=np.uint16).reshape(-1)
    nb = x.size // 32
    codes = np.zeros(nb * 16, np.uint8)
    scales = np.zeros(nb, np.uint8)
    out = np.zeros(nb * 32, np.uint16)
    _load().oracle_fp4_e8m0(_ptr(x), nb, _ptr(codes), _ptr(scales), _ptr(out))
    return codes, scales, out


def yarn_freqs(rope_dim=64, base=160000.0, factor=16.0, orig_len=4096, beta_fast=32.0, beta_slow=1.0):
    f = np.zeros(rope_dim // 2, np.float64)
    _load().oracle_yarn_freqs(rope_dim, base, factor, orig_len, beta_fast, beta_slow, _ptr(f))
    return f


def yarn_bounds(rope_dim=64, base=160000.0, orig_len=4096, beta_fast=32.0, beta_slow=1.0):
    lo, hi = ctypes.c_double(), ctypes.c_double()
    _load().oracle_yarn_bounds(rope_dim, base, orig_len, beta_fast, beta_slow, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def pool(kv: np.ndarray, score: np.ndarray):
    """kv, score float32 [n, H] -> (pooled float32 [H], weights float64 [n, H])."""
    kv = np.ascontiguousarray(kv, np.float32)
    score = np.ascontiguousarray(score, np.float32)
    n, H = kv.shape
    out = np.zeros(H, np.float32)
    w = np.zeros((n, H), np.float64)
    _load().oracle_pool(_ptr(kv), _ptr(score), n, H, _ptr(out), _ptr(w))
    return out, w


def linear(x_bf16: np.ndarray, w: np.ndarray, nthreads: int = 1) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, np.uint16)
    w = np.ascontiguousarray(w, np.float32)
    M, D = x.shape
    C = w.shape[0]
    out = np.zeros((M, C), np.float32)
    _load().oracle_linear(_ptr(x), M, D, _ptr(w), C, _ptr(out), nthreads)
    return out


# ---- the compressor ----------------------------------------------------------------------

FLASH_ROPE = dict(rope_dim=64, rope_base=160000.0, rope_factor=16.0, rope_orig_len=4096, beta_fast=32.0,
                  beta_slow=1.0)


class Compressor:
    """The oracle compressor: prefill / decode / state, mirroring the library's calls."""

    def __init__(self, dim, head_dim, ratio, overlap, max_batch=1, rope_dim=64, rope_base=160000.0,
                 rope_factor=16.0, rope_orig_len=4096, beta_fast=32.0, beta_slow=1.0, fp4=1, eps=1e-6):
        self.dim, self.H, self.ratio, self.overlap = dim, head_dim, ratio, overlap
        self.fp4 = fp4
        self.opt = Options(max_batch, rope_dim, rope_base, rope_factor, rope_orig_len, beta_fast, beta_slow, fp4,
                           eps)
        self._lib = _load()
        self.h = self._lib.oracle_create(dim, head_dim, ratio, overlap, ctypes.byref(self.opt))
        if not self.h:
            raise ValueError("oracle_create rejected the arguments")

    def __del__(self):
        if getattr(self, "h", None):
            self._lib.oracle_destroy(self.h)
            self.h = None

    def set_weights(self, wkv, wgate, gain):
        self._w = (np.ascontiguousarray(wkv, np.float32),
                   None if wgate is None else np.ascontiguousarray(wgate, np.float32),
                   np.ascontiguousarray(gain, np.float32))
        self._lib.oracle_set_weights(self.h, _ptr(self._w[0]), _ptr(self._w[1]), _ptr(self._w[2]))

    @property
    def scale_block(self):
        """Values per fp4 scale: 16 (e4m3 scales, the latent) or 32 (power-of-two scales)."""
        return 32 if self.fp4 == 2 else 16

    def set_gate_bias(self, ape):
        """ape float32 [ratio, (1 + overlap) * H] added to the gate logits by position within the
        group, or None to remove it."""
        self._ape = None if ape is None else np.ascontiguousarray(ape, np.float32)
        self._lib.oracle_set_gate_bias(self.h, None if self._ape is None else _ptr(self._ape))

    def _outs(self, n):
        H = self.H
        return (np.zeros((n, H), np.uint16), np.zeros((n, H // 2), np.uint8),
                np.zeros((n, H // self.scale_block), np.uint8), np.zeros((n, H), np.uint16))

    def prefill(self, x_bf16, slot_offset=0, nthreads=None, start_pos=0):
        """x uint16 [B, N, dim] (tokens start_pos .. start_pos+N-1 of each sequence) ->
        dict(latent [B,G,H], codes, scales, prequant, G), G the groups completing in the chunk."""
        x = np.ascontiguousarray(x_bf16, np.uint16)
        B, N, _ = x.shape
        G = (start_pos + N) // self.ratio - start_pos // self.ratio
        lat, cd, sc, pq = self._outs(max(B * G, 1))
        g = self._lib.oracle_prefill_chunk(self.h, _ptr(x), B, N, start_pos, slot_offset, _ptr(lat), _ptr(cd),
                                           _ptr(sc), _ptr(pq), nthreads or default_threads())
        if g < 0:
            raise ValueError("oracle_prefill rejected the arguments")
        H = self.H
        return dict(G=g, latent=lat[:B * G].reshape(B, G, H), codes=cd[:B * G].reshape(B, G, H // 2),
                    scales=sc[:B * G].reshape(B, G, H // self.scale_block), prequant=pq[:B * G].reshape(B, G, H))

    def prefill_groups(self, x_seq_bf16, groups, nthreads=None):
        """x uint16 [N, dim] (one sequence); groups: list of group indices -> outputs [ng, ...]."""
        x = np.ascontiguousarray(x_seq_bf16, np.uint16)
        N = x.shape[0]
        g = np.ascontiguousarray(groups, np.int32)
        lat, cd, sc, pq = self._outs(max(g.size, 1))
        rc = self._lib.oracle_prefill_groups(self.h, _ptr(x), N, _ptr(g), g.size, _ptr(lat), _ptr(cd), _ptr(sc),
                                             _ptr(pq), nthreads or default_threads())
        if rc < 0:
            raise ValueError("oracle_prefill_groups rejected the arguments")
        n = g.size
        return dict(latent=lat[:n], codes=cd[:n], scales=sc[:n], prequant=pq[:n])

    def decode(self, x_tok_bf16, start_pos, nthreads=None):
        x = np.ascontiguousarray(x_tok_bf16, np.uint16)
        B = x.shape[0]
        sp = np.ascontiguousarray(start_pos, np.int32)
        lat, cd, sc, pq = self._outs(B)
        em = np.zeros(B, np.uint8)
        n = self._lib.oracle_decode(self.h, _ptr(x), B, _ptr(sp), _ptr(lat), _ptr(cd), _ptr(sc), _ptr(pq), _ptr(em),
                                    nthreads or default_threads())
        if n < 0:
            raise ValueError("oracle_decode rejected the arguments")
        return dict(n=n, emitted=em, latent=lat, codes=cd, scales=sc, prequant=pq)

    def state_reset(self):
        self._lib.oracle_state_reset(self.h)

    def state(self):
        n = self._lib.oracle_state_elems(self.h)
        kv = np.zeros(n, np.float32)
        sc = np.zeros(n, np.float32)
        self._lib.oracle_state_export(self.h, _ptr(kv), _ptr(sc))
        mb = self.opt.max_batch
        if self.overlap:
            shape = (mb, 2, 4, 2 * self.H)
        else:
            shape = (mb, self.ratio, self.H)
        return kv.reshape(shape), sc.reshape(shape)


def _epilogue(self, pooled, pos):
    """bf16 round + RMSNorm + RoPE at position pos of one pooled float32 row [H] -> bf16 bits [H]."""
    p = np.ascontiguousarray(pooled, np.float32)
    out = np.zeros(self.H, np.uint16)
    self._lib.oracle_epilogue(self.h, _ptr(p), int(pos), _ptr(out))
    return out


Compressor.epilogue = _epilogue

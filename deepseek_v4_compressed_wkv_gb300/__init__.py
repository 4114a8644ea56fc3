"""GB300 (sm_103a) compressed-sparse-attention KV Compressor.

Thin Python binding over the C ABI in ``include/csa.h`` (``libcsa.so``): it only marshals
arguments.  PyTorch provides device memory and streams; every step of the compressor runs
in the library's CUDA kernels.  There is no CPU path: if the library is missing or no GPU
is present, calls fail with an error.

    from deepseek_v4_compressed_wkv_gb300 import Compressor
    c = Compressor(dim=4096, head_dim=512, ratio=4, overlap=1)
    c.set_weights(wkv, wgate, gain)          # f32 CUDA tensors [C, dim], [C, dim], [H]
    out = c.prefill(x)                       # x bf16 CUDA [B, N, dim] -> dict of tensors or None
    step = c.decode(x_tok, start_pos)        # x_tok bf16 [B, dim]; start_pos int32 [B] on the host
                                             # (returns the emitting count) or on the device
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build_mod

__all__ = ["Compressor", "CSAError", "load_library", "fp4_e4m3_roundtrip", "fp4_e8m0_roundtrip", "rope_table",
           "default_options",
           "library_path", "ABI_FUNCTIONS"]

_lock = threading.Lock()
_lib = None

# every entry point declared in include/csa.h
ABI_FUNCTIONS = ("csa_options_default", "csa_compressor_create", "csa_compressor_create_ex",
                 "csa_compressor_set_weights", "csa_compress_prefill", "csa_compress_decode",
                 "csa_compress_decode_dev", "csa_state_reset", "csa_state_elems",
                 "csa_state_export", "csa_state_import", "csa_device_status", "csa_compressor_destroy", "csa_last_error",
                 "csa_fp4_e4m3_roundtrip", "csa_rope_table", "csa_set_profile_events", "csa_kernel_launches",
                 "csa_uses_tensor_cores", "csa_compress_prefill_noalloc", "csa_compress_prefill_into",
                 "csa_prefill_geometry",
                 "csa_fp4_e8m0_roundtrip", "csa_compressor_set_gate_bias")


class CSAError(RuntimeError):
    pass


class Options(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("rope_dim", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("rope_factor", ctypes.c_float), ("rope_orig_len", ctypes.c_int), ("beta_fast", ctypes.c_float),
                ("beta_slow", ctypes.c_float), ("max_pos", ctypes.c_int), ("fp4", ctypes.c_int),
                ("eps", ctypes.c_float), ("prefill_split", ctypes.c_int), ("prefill_pair", ctypes.c_int)]


class Out(ctypes.Structure):
    _fields_ = [("latent", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("prequant", ctypes.c_void_p)]


def _variant() -> str:
    # CSA_LIBRARY_VARIANT=bounds selects the bounds-checked build (for tests)
    return os.environ.get("CSA_LIBRARY_VARIANT", "")


def library_path() -> str:
    return _build_mod.lib_path(_variant())


def load_library(build_if_missing: bool = True):
    """Loads libcsa.so (building it first if it is missing and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build_mod.lib_path(_variant())
        if not os.path.exists(path):
            if not build_if_missing:
                raise CSAError(f"{path} is missing: build it with deepseek_v4_compressed_wkv_gb300.build")
            _build_mod.build(variant=_variant())
        lib = ctypes.CDLL(path)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        sig = {
            "csa_options_default": ([P], None),
            "csa_compressor_create": ([I, I, I, I, P], I),
            "csa_compressor_create_ex": ([I, I, I, I, P, P], I),
            "csa_compressor_set_weights": ([P, P, P, P, P], I),
            "csa_compress_prefill": ([P, P, I, I, I, I, P, P], I),
            "csa_compress_decode": ([P, P, I, P, P, P, P], I),
            "csa_compress_decode_dev": ([P, P, I, P, P, P, P], I),
            "csa_state_reset": ([P, I, I, P], I),
            "csa_state_elems": ([P], I64),
            "csa_state_export": ([P, P, P, P], I),
            "csa_state_import": ([P, P, P, P], I),
            "csa_device_status": ([P, P], I),
            "csa_compressor_destroy": ([P], None),
            "csa_last_error": ([], ctypes.c_char_p),
            "csa_fp4_e4m3_roundtrip": ([P, I64, P, P, P, P], I),
            "csa_fp4_e8m0_roundtrip": ([P, I64, P, P, P, P], I),
            "csa_compressor_set_gate_bias": ([P, P, P], I),
            "csa_rope_table": ([P, I, I, P, P], I),
            "csa_set_profile_events": ([P, P, P], I),
            "csa_kernel_launches": ([P], I64),
            "csa_uses_tensor_cores": ([P], I),
            "csa_prefill_geometry": ([P, I, I, I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_int)], I),
            "csa_compress_prefill_noalloc": ([P, P, I, I, I, I, P, P], I),
            "csa_compress_prefill_into": ([P, P, I, I, I, I, P, I, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, what: str) -> int:
    if rc < 0:
        msg = load_library().csa_last_error().decode(errors="replace")
        raise CSAError(f"{what} failed ({rc}): {msg}")
    return rc


def default_options(**overrides) -> Options:
    o = Options()
    load_library().csa_options_default(ctypes.byref(o))
    for k, v in overrides.items():
        if not hasattr(o, k):
            raise TypeError(f"unknown option {k}")
        setattr(o, k, v)
    return o


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda or not t.is_contiguous():
        raise CSAError("tensors passed to the library must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _u16(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _on_current_device(*tensors):
    """The library launches on the current CUDA device: every tensor it reads or writes must
    live there (a pointer into another GPU's memory would fault)."""
    dev = torch.cuda.current_device()
    for t in tensors:
        if t is not None and (not t.is_cuda or t.device.index != dev):
            raise CSAError(f"tensor on {t.device}, but the current CUDA device is cuda:{dev}")




class Compressor:
    """One compressor instance (one attention layer's wkv / wgate / norm / state)."""

    def __init__(self, dim: int, head_dim: int, ratio: int, overlap: int = 0, **options):
        self._lib = load_library()
        self.dim, self.head_dim, self.ratio, self.overlap = dim, head_dim, ratio, overlap
        self.options = default_options(**options)
        h = ctypes.c_void_p()
        _check(self._lib.csa_compressor_create_ex(dim, head_dim, ratio, overlap, ctypes.byref(self.options),
                                                  ctypes.byref(h)), "csa_compressor_create_ex")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.csa_compressor_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def set_weights(self, wkv, wgate, gain, stream=None):
        _check(self._lib.csa_compressor_set_weights(self._h, _dptr(wkv), _dptr(wgate), _dptr(gain),
                                                    _stream(stream)), "csa_compressor_set_weights")

    def set_gate_bias(self, ape, stream=None):
        """ape f32 CUDA [ratio, (1 + overlap) * head_dim] added to the gate logits by position within
        the group, or None to remove it."""
        _check(self._lib.csa_compressor_set_gate_bias(self._h, _dptr(ape), _stream(stream)),
               "csa_compressor_set_gate_bias")

    @property
    def scale_block(self) -> int:
        """Features per fp4 scale: 16 (e4m3 scales, fp4 = 1) or 32 (power-of-two scales, fp4 = 2)."""
        return 32 if self.options.fp4 == 2 else 16

    def _alloc_out(self, rows, device, prequant=True):
        H = self.head_dim
        fp4 = bool(self.options.fp4)
        d = dict(latent=torch.empty(rows, H, dtype=torch.bfloat16, device=device),
                 codes=torch.empty(rows, H // 2, dtype=torch.uint8, device=device) if fp4 else None,
                 scales=torch.empty(rows, H // self.scale_block, dtype=torch.uint8, device=device) if fp4 else None,
                 prequant=torch.empty(rows, H, dtype=torch.bfloat16, device=device) if prequant else None)
        return d

    def _check_out(self, d, rows):
        """Caller-provided outputs: the library writes `rows` rows of each array given, so each
        must be a contiguous CUDA tensor of the right type holding at least that many."""
        H = self.head_dim
        widths = {"latent": H, "codes": H // 2, "scales": H // self.scale_block, "prequant": H}
        types = {"latent": torch.bfloat16, "codes": torch.uint8, "scales": torch.uint8, "prequant": torch.bfloat16}
        if d.get("latent") is None:
            raise CSAError("out['latent'] is required")
        for k, t in d.items():
            if t is None or k not in widths:
                continue
            if t.dtype != types[k]:
                raise CSAError(f"out['{k}'] must be {types[k]}")
            if t.numel() < rows * widths[k]:
                raise CSAError(f"out['{k}'] holds {t.numel()} elements, the call writes {rows} x {widths[k]}")
        _on_current_device(*[t for t in d.values() if t is not None])

    @staticmethod
    def _out_struct(d):
        return Out(_dptr(d["latent"]).value, _dptr(d.get("codes")).value, _dptr(d.get("scales")).value,
                   _dptr(d.get("prequant")).value)

    def prefill(self, x, slot_offset: int = 0, out=None, prequant: bool = True, stream=None, start_pos: int = 0):
        """x bf16 [B, N, dim] CUDA: tokens start_pos .. start_pos+N-1 of each sequence (start_pos > 0:
        a chunk continuing the sequences in the state).  Returns None when no group completes,
        else a dict of latent [B, G, H] bf16, codes [B, G, H/2] u8, scales [B, G, H/16] u8 and
        prequant [B, G, H] bf16 (codes/scales None when fp4 is off)."""
        B, N, D = x.shape
        if D != self.dim or x.dtype != torch.bfloat16:
            raise CSAError("x must be bf16 [B, N, dim]")
        G = (start_pos + N) // self.ratio - start_pos // self.ratio
        _on_current_device(x)
        if out is None:
            out = self._alloc_out(max(B * G, 1), x.device, prequant)
        else:
            self._check_out(out, B * G)
        o = self._out_struct(out)
        g = _check(self._lib.csa_compress_prefill(self._h, _dptr(_u16(x)), B, N, start_pos, slot_offset,
                                                  ctypes.byref(o), _stream(stream)), "csa_compress_prefill")
        if g == 0:
            return None
        H = self.head_dim
        shp = {"latent": (B, g, H), "codes": (B, g, H // 2), "scales": (B, g, H // self.scale_block),
               "prequant": (B, g, H)}
        return {k: (None if v is None else v[:B * g].view(*shp[k])) for k, v in out.items()}

    def prefill_noalloc(self, x, out, slot_offset: int = 0, start_pos: int = 0, stream=None):
        """The same prefill through the entry point that allocates no device memory (its scratch
        is a fixed array in the library; tensor-core shapes up to that array's size).  `out` is
        required (the caller owns every buffer); returns the entries per sequence."""
        B, N, D = x.shape
        if D != self.dim or x.dtype != torch.bfloat16:
            raise CSAError("x must be bf16 [B, N, dim]")
        _on_current_device(x)
        G = (start_pos + N) // self.ratio - start_pos // self.ratio
        self._check_out(out, B * G)
        o = self._out_struct(out)
        return _check(self._lib.csa_compress_prefill_noalloc(self._h, _dptr(_u16(x)), B, N, start_pos, slot_offset,
                                                             ctypes.byref(o), _stream(stream)),
                      "csa_compress_prefill_noalloc")

    def prefill_into(self, x, cache, start_pos: int = 0, slot_offset: int = 0, stream=None) -> int:
        """Prefill (or a chunk at start_pos) writing entry g of sequence b into row g of
        cache["latent"][b] ([B, rows, H] bf16; optional "codes" [B, rows, H/2], "scales"
        [B, rows, H/16], "prequant" [B, rows, H]).  Returns the entries written per sequence."""
        B, N, D = x.shape
        if D != self.dim or x.dtype != torch.bfloat16:
            raise CSAError("x must be bf16 [B, N, dim]")
        lat = cache["latent"]
        if lat.dim() != 3 or lat.shape[0] != B or lat.shape[2] != self.head_dim:
            raise CSAError("cache['latent'] must be [B, rows, head_dim]")
        _on_current_device(x)
        self._check_out({k: cache.get(k) for k in ("latent", "codes", "scales", "prequant")}, B * lat.shape[1])
        o = self._out_struct({k: cache.get(k) for k in ("latent", "codes", "scales", "prequant")})
        return _check(self._lib.csa_compress_prefill_into(self._h, _dptr(_u16(x)), B, N, start_pos, slot_offset,
                                                          ctypes.byref(o), lat.shape[1], _stream(stream)),
                      "csa_compress_prefill_into")

    def decode(self, x_tok, start_pos, out=None, emitted=None, prequant: bool = True, stream=None):
        """One decode step: x_tok bf16 CUDA [B, dim]; start_pos int32 [B], either on the host (a
        numpy array, a list or a CPU tensor: csa_compress_decode, which returns the number of
        emitting sequences) or a CUDA tensor (csa_compress_decode_dev, for positions that live on
        the device and for graph capture).  Returns a dict with latent/codes/scales/prequant
        [B, ...] (rows valid where emitted), emitted u8 [B] (a CPU tensor for host positions
        unless a device `emitted` is given, else on the device) and, for host positions, count."""
        B, D = x_tok.shape
        if D != self.dim or x_tok.dtype != torch.bfloat16:
            raise CSAError("x_tok must be bf16 [B, dim]")
        on_device = isinstance(start_pos, torch.Tensor) and start_pos.is_cuda
        if on_device:
            if start_pos.numel() != B:
                raise CSAError(f"start_pos has {start_pos.numel()} elements for {B} sequences")
            if start_pos.dtype != torch.int32:
                raise CSAError("start_pos must be int32")
            _on_current_device(x_tok, start_pos)
        else:
            import numpy as np
            sp = np.ascontiguousarray(start_pos.numpy() if isinstance(start_pos, torch.Tensor) else start_pos,
                                      dtype=np.int32).reshape(-1)
            if sp.size != B:
                raise CSAError(f"start_pos has {sp.size} elements for {B} sequences")
            _on_current_device(x_tok)
        if out is None:
            out = self._alloc_out(B, x_tok.device, prequant)
        else:
            self._check_out(out, B)
        o = self._out_struct(out)
        if on_device:
            if emitted is None:
                emitted = torch.empty(B, dtype=torch.uint8, device=x_tok.device)
            elif emitted.dtype != torch.uint8 or emitted.numel() < B or not emitted.is_cuda:
                raise CSAError("emitted must be a uint8 CUDA tensor with at least B elements")
            _on_current_device(emitted)
            _check(self._lib.csa_compress_decode_dev(self._h, _dptr(_u16(x_tok)), B, _dptr(start_pos),
                                                     ctypes.byref(o), _dptr(emitted), _stream(stream)),
                   "csa_compress_decode_dev")
            d = dict(out)
            d["emitted"] = emitted
            return d
        if emitted is None:
            emitted = torch.empty(B, dtype=torch.uint8)
        elif emitted.dtype != torch.uint8 or emitted.numel() < B or not emitted.is_contiguous():
            raise CSAError("emitted must be a contiguous uint8 tensor with at least B elements")
        if emitted.is_cuda:
            _on_current_device(emitted)
        n = _check(self._lib.csa_compress_decode(self._h, _dptr(_u16(x_tok)), B, ctypes.c_void_p(sp.ctypes.data),
                                                 ctypes.byref(o), ctypes.c_void_p(emitted.data_ptr()),
                                                 _stream(stream)), "csa_compress_decode")
        d = dict(out)
        d["emitted"] = emitted
        d["count"] = n
        return d

    def state_reset(self, slot_begin: int = 0, slot_count: int | None = None, stream=None):
        if slot_count is None:
            slot_count = self.options.max_batch - slot_begin
        _check(self._lib.csa_state_reset(self._h, slot_begin, slot_count, _stream(stream)), "csa_state_reset")

    def state_export(self, device="cuda", stream=None):
        n = _check(self._lib.csa_state_elems(self._h), "csa_state_elems")
        kv = torch.empty(n, dtype=torch.float32, device=device)
        sc = torch.empty(n, dtype=torch.float32, device=device)
        _check(self._lib.csa_state_export(self._h, _dptr(kv), _dptr(sc), _stream(stream)), "csa_state_export")
        mb, H = self.options.max_batch, self.head_dim
        shape = (mb, 2, 4, 2 * H) if self.overlap else (mb, self.ratio, H)
        return kv.view(shape), sc.view(shape)

    def state_import(self, kv, score, stream=None):
        """Replaces the whole state with kv and score (f32 CUDA tensors in the layout state_export
        returns, e.g. another handle's)."""
        n = _check(self._lib.csa_state_elems(self._h), "csa_state_elems")
        kv, score = kv.contiguous(), score.contiguous()
        for t in (kv, score):
            if t.dtype != torch.float32 or not t.is_cuda or t.numel() != n:
                raise CSAError(f"state arrays must be f32 CUDA tensors of {n} elements")
            _on_current_device(t)
        _check(self._lib.csa_state_import(self._h, _dptr(kv), _dptr(score), _stream(stream)), "csa_state_import")

    def set_profile_events(self, start=None, stop=None):
        """torch.cuda.Event pair (enable_timing=True) recorded around the dominant kernel."""
        _check(self._lib.csa_set_profile_events(self._h, ctypes.c_void_p(start.cuda_event if start else 0),
                                                ctypes.c_void_p(stop.cuda_event if stop else 0)),
               "csa_set_profile_events")

    def uses_tensor_cores(self) -> bool:
        return bool(_check(self._lib.csa_uses_tensor_cores(self._h), "csa_uses_tensor_cores"))

    def prefill_geometry(self, B: int, N: int, start_pos: int = 0) -> dict:
        """The tensor-core prefill's launch geometry for B sequences of N tokens at start_pos:
        {"token_tile": 256 | 224 | 128, "k_split": 1 | 2, "cta_pair": 1 | 2}."""
        tok, split, pair = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(self._lib.csa_prefill_geometry(self._h, B, N, start_pos, ctypes.byref(tok), ctypes.byref(split),
                                              ctypes.byref(pair)), "csa_prefill_geometry")
        return {"token_tile": tok.value, "k_split": split.value, "cta_pair": pair.value}

    def kernel_launches(self) -> int:
        return _check(self._lib.csa_kernel_launches(self._h), "csa_kernel_launches")

    def device_status(self, stream=None):
        return _check(self._lib.csa_device_status(self._h, _stream(stream)), "csa_device_status")


def fp4_e4m3_roundtrip(x, stream=None):
    """bf16 CUDA tensor (size a multiple of 16) -> (codes u8 [n/2], scales u8 [n/16], out bf16 [n])."""
    lib = load_library()
    x = x.contiguous().view(-1)
    if x.dtype != torch.bfloat16 or x.numel() % 16:
        raise CSAError("x must be bf16 with a multiple of 16 elements")
    _on_current_device(x)
    nb = x.numel() // 16
    codes = torch.empty(nb * 8, dtype=torch.uint8, device=x.device)
    scales = torch.empty(nb, dtype=torch.uint8, device=x.device)
    out = torch.empty(nb * 16, dtype=torch.bfloat16, device=x.device)
    _check(lib.csa_fp4_e4m3_roundtrip(_dptr(_u16(x)), nb, _dptr(codes), _dptr(scales), _dptr(_u16(out)),
                                      _stream(stream)), "csa_fp4_e4m3_roundtrip")
    return codes, scales, out


def fp4_e8m0_roundtrip(x, stream=None):
    """The indexer's fp4 round trip: bf16 CUDA tensor (size a multiple of 32) -> (codes u8 [n/2],
    scales u8 [n/32] e8m0 bytes, out bf16 [n])."""
    lib = load_library()
    x = x.contiguous().view(-1)
    if x.dtype != torch.bfloat16 or x.numel() % 32:
        raise CSAError("x must be bf16 with a multiple of 32 elements")
    _on_current_device(x)
    nb = x.numel() // 32
    codes = torch.empty(nb * 16, dtype=torch.uint8, device=x.device)
    scales = torch.empty(nb, dtype=torch.uint8, device=x.device)
    out = torch.empty(nb * 32, dtype=torch.bfloat16, device=x.device)
    _check(lib.csa_fp4_e8m0_roundtrip(_dptr(_u16(x)), nb, _dptr(codes), _dptr(scales), _dptr(_u16(out)),
                                      _stream(stream)), "csa_fp4_e8m0_roundtrip")
    return codes, scales, out


def rope_table(pos0: int, npos: int, **options):
    """Host-side RoPE table of the library: (cos, sin) float32 numpy [npos, rope_dim/2]."""
    import numpy as np
    o = default_options(**options)
    hr = o.rope_dim // 2
    cs = np.zeros((npos, hr), np.float32)
    sn = np.zeros((npos, hr), np.float32)
    _check(load_library().csa_rope_table(ctypes.byref(o), pos0, npos, cs.ctypes.data, sn.ctypes.data),
           "csa_rope_table")
    return cs, sn


def state_window_start(pos: int, ratio: int, overlap: int) -> int:
    """First token whose projection the state at position `pos` still holds.

    Prefilling tokens [state_window_start(pos), pos) of a sequence (as a sequence of its
    own, in a fresh state slot) leaves exactly the state that prefilling all `pos` tokens
    leaves: the unfinished group's tokens and, at ratio 4 overlapped, the last complete
    group's tokens in the parity slot of their absolute group index (so the start is a
    multiple of 8 tokens there).  Entries that this shorter prefill emits are not the
    sequence's entries and should be discarded."""
    g = pos // ratio
    if not overlap or g == 0:
        return ratio * g
    k0 = (g - 1) - ((g - 1) % 2)
    return 4 * k0

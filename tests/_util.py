"""Small helpers shared by the tests: bf16 bit conversions (via torch) and layer set-up."""
import numpy as np
import torch

import synthetic


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), rounded to nearest even by torch."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def layer_inputs(seed, layer, B, N, outlier_frac=0.0, t0=0):
    """(x bf16 bits [B, N, dim], wkv, wgate, gain) for one compressor layer of a workload."""
    x = np.stack([synthetic.tokens(seed, b, t0, t0 + N, layer.dim, outlier_frac) for b in range(B)])
    wkv, wgate, gain = synthetic.weights(seed, layer)
    return to_bf16_bits(x), wkv, wgate, gain


def ulp_distance_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two bf16 bit arrays (monotone integer mapping)."""
    def key(h):
        h = np.asarray(h, np.uint16).astype(np.int32)
        return np.where(h & 0x8000, -(h & 0x7FFF), h)
    return np.abs(key(a) - key(b))

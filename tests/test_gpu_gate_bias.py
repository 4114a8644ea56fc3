"""The gate positional bias (score = wgate(x) + ape[position in group]) on the GPU: prefill, a
chunk and decode steps against the oracle with the same bias, on the tensor-core and CUDA-core
paths; then the bias removed again."""
import math

import numpy as np
import pytest
import torch

import synthetic
from _util import layer_inputs
from test_gpu_parity import DEV, check_entries, dev_bits, make_pair, to_np

pytestmark = pytest.mark.gpu

SHAPES = [
    # dim, H, ratio, overlap, B, prefill N, chunk N
    (256, 128, 4, 1, 2, 4 * 60 + 1, 4 * 20 + 3),
    (256, 512, 128, 0, 2, 128 * 2 + 30, 128 + 9),
    (192, 256, 8, 0, 1, 8 * 40 + 3, 13),
    (1024, 128, 4, 1, 1, 4 * 120 + 1, 4 * 30 + 2),
    (128, 32, 3, 0, 2, 3 * 40 + 2, 7),           # CUDA-core path
    (128, 64, 300, 0, 1, 300 * 2 + 7, 301),      # CUDA-core path
]


@pytest.mark.parametrize("split,pair", [(1, 0), (2, 0), (1, 2)])
@pytest.mark.parametrize("dim,H,ratio,overlap,B,N,Nc", SHAPES)
def test_gate_bias_prefill_chunk_decode(dim, H, ratio, overlap, B, N, Nc, split, pair):
    """The bias where the prefill adds it (overlapped and one CTA per tile: where the pool and the
    state writes read the scores; otherwise in a pass over the staged rows), in decode and in the
    CUDA-core path, against the oracle's biased logits."""
    layer = synthetic.Layer(dim, H, ratio, overlap, 1.0 / math.sqrt(dim), gate_scale=2.0, rope_dim=min(64, H), fp4=1)
    g, o = make_pair(13, layer, max_batch=B, split=split, pair=pair)
    ape = np.random.default_rng(ratio).standard_normal((ratio, (1 + overlap) * H)).astype(np.float32) * 2
    g.set_gate_bias(torch.from_numpy(ape).to(DEV))
    o.set_gate_bias(ape)
    x, *_ = layer_inputs(13, layer, B, N + Nc + 6)
    p = 0
    for n in (N, Nc):
        xc = np.ascontiguousarray(x[:, p:p + n])
        got = g.prefill(dev_bits(xc), start_pos=p)
        torch.cuda.synchronize()
        ref = o.prefill(xc, start_pos=p)
        if ref["G"]:
            check_entries(to_np(got), ref["prequant"], 1, f"biased prefill at {p}")
        p += n
    for k in range(6):
        sp = np.full(B, p + k, np.int32)
        xt = np.ascontiguousarray(x[:, p + k])
        r = o.decode(xt, sp)
        d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"])
        rows = np.flatnonzero(em)
        if rows.size:
            check_entries(to_np(d, rows=rows), r["prequant"][rows], 1, f"biased decode {k}")
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    ko, so = o.state()
    fin = np.isfinite(so)
    assert np.array_equal(np.isinf(sg), np.isinf(so))
    assert np.allclose(sg[fin], so[fin], rtol=2e-5, atol=2e-5 * np.abs(so[fin]).max(initial=1.0))
    # removing the bias: a fresh prefill matches the unbiased oracle
    g.set_gate_bias(None)
    o.set_gate_bias(None)
    xc = np.ascontiguousarray(x[:, :N])
    got = g.prefill(dev_bits(xc))
    torch.cuda.synchronize()
    check_entries(to_np(got), o.prefill(xc)["prequant"], 1, "bias removed")
    assert g.device_status() == 0

"""Two more compressor instances of the model at the Flash width, on the same kernels:

- the indexer's 128-wide compressor of a CSA layer ("Compressed Sparse Attention": a separate
  128-D indexer compressor; "Module compress": the indexer's q and k take the e2m1 round trip
  with power-of-two scales, block 32), prefill, a chunk and decode steps;
- the ratio-2 layers that pool token pairs ("Pool token pairs"), a batch of two sequences.

Every entry is compared with the oracle (same tolerance as the other parity tests; the fp4
outputs bit for bit against the oracle's round trip of the GPU's own prequant).
"""
import numpy as np
import pytest
import torch

import deepseek_v4_compressed_wkv_gb300 as csa
import synthetic
from _util import layer_inputs
from test_gpu_parity import DEV, check_entries, dev_bits, make_pair, to_np

pytestmark = pytest.mark.gpu


def test_indexer_compressor_prefill_chunk_and_decode():
    wl = synthetic.INDEXER
    layer = wl.layers[0]
    g, o = make_pair(wl.seed, layer)
    assert g.uses_tensor_cores()
    N = wl.tokens[0]
    x, *_ = layer_inputs(wl.seed, layer, 1, N + 1003 + 9)
    got = g.prefill(dev_bits(np.ascontiguousarray(x[:, :N])))
    torch.cuda.synchronize()
    ref = o.prefill(np.ascontiguousarray(x[:, :N]))
    assert got["scales"].shape == (1, N // 4, 128 // 32)
    check_entries(to_np(got), ref["prequant"], 2, "indexer prefill")
    xc = np.ascontiguousarray(x[:, N:N + 1003])
    got = g.prefill(dev_bits(xc), start_pos=N)
    torch.cuda.synchronize()
    ref = o.prefill(xc, start_pos=N)
    check_entries(to_np(got), ref["prequant"], 2, "indexer chunk")
    p = N + 1003
    for k in range(9):
        sp = np.array([p + k], np.int32)
        xt = np.ascontiguousarray(x[:, p + k])
        r = o.decode(xt, sp)
        d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"])
        if em[0]:
            check_entries(to_np(d, rows=[0]), r["prequant"][[0]], 2, f"indexer decode {k}")
    assert g.device_status() == 0


def test_pool_token_pairs_ratio2_prefill():
    wl = synthetic.PAIRS
    layer = wl.layers[0]
    B, N = wl.batch, wl.tokens[0]
    g, o = make_pair(wl.seed, layer, max_batch=B)
    assert g.uses_tensor_cores()
    x, *_ = layer_inputs(wl.seed, layer, B, N)
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    ref = o.prefill(x)
    assert ref["G"] == N // 2
    check_entries(to_np(got), ref["prequant"], 1, "pairs prefill")
    assert g.device_status() == 0


def test_launch_geometry_of_the_measured_instances():
    """The launch geometry the prefill chooses (csa_prefill_geometry): the indexer's 4 packed tiles
    split over K at the 224-token tile (76 clusters of two CTAs fill the 152 SMs), the Flash CSA
    layer's 16 tiles one CTA each at 224 tokens (two full waves), HCA and one long ratio-128
    sequence at the 256-token tile; a forced split is reported as forced, and a shape the
    CUDA-core projection runs is refused."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    def geo(wl, **opt):
        L = wl.layers[0]
        c = csa.Compressor(L.dim, L.head_dim, L.ratio, L.overlap, max_batch=max(wl.batch, 1), **opt)
        try:
            return c.prefill_geometry(wl.batch, wl.tokens[0])
        finally:
            c.close()
    if sms == 152:  # the choices below are the model's for the 152-SM part
        assert geo(synthetic.INDEXER) == {"token_tile": 224, "k_split": 2, "cta_pair": 1}
        assert geo(synthetic.FLASH_CSA) == {"token_tile": 224, "k_split": 1, "cta_pair": 1}
        assert geo(synthetic.HCA) == {"token_tile": 256, "k_split": 1, "cta_pair": 1}
    assert geo(synthetic.INDEXER, prefill_split=1)["k_split"] == 1
    assert geo(synthetic.FLASH_CSA, prefill_split=2)["k_split"] == 2
    # CTA pairs where asked for and the tiles are not split
    assert geo(synthetic.FLASH_CSA, prefill_pair=2)["cta_pair"] == 2
    assert geo(synthetic.INDEXER, prefill_pair=2, prefill_split=2)["cta_pair"] == 1
    narrow = csa.Compressor(128, 32, 3, 0, rope_dim=16)  # packed tile narrower than 128 rows: the CUDA-core projection
    try:
        with pytest.raises(csa.CSAError):
            narrow.prefill_geometry(1, 30)
    finally:
        narrow.close()

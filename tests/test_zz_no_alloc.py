"""The prefill entry point that allocates nothing (csa_compress_prefill_noalloc).

Callers such as serving runtimes that reserve all device memory for their own pool, or code
that enqueues work while a CUDA graph is being captured, cannot let the library call
cudaMalloc.  This entry point runs the same tensor-core kernel with its scratch in a fixed
device array compiled into the library.  The test calls it through the C ABI twice in a row
(the shared array keeps the previous call's contents) and checks each result against the
ordinary entry point on the same input, within the parity tolerance of the other tests
(they come out identical), including the state it leaves behind.  This file is collected
last so that a failure here does not hide the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import deepseek_v4_compressed_wkv_gb300 as csa
import synthetic
from _util import ulp_distance_bf16

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _call_noalloc(lib, comp, x, out, slot_offset=0, start_pos=0):
    B, N, _ = x.shape
    o = csa.Out(out["latent"].data_ptr(), out["codes"].data_ptr(), out["scales"].data_ptr(),
                out["prequant"].data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.csa_compress_prefill_noalloc(comp.handle, ctypes.c_void_p(x.data_ptr()), B, N, start_pos,
                                            slot_offset, ctypes.byref(o), stream)


def test_noalloc_prefill_matches_the_allocating_entry_point_twice():
    lib = csa.load_library()
    layer = synthetic.Layer(1024, 512, 4, 1, 1.0 / 32, gate_scale=2.0)
    wkv, wgate, gain = synthetic.weights(7, layer)
    comps = []
    for _ in range(2):
        c = csa.Compressor(layer.dim, layer.head_dim, 4, 1, max_batch=3, max_pos=8192)
        c.set_weights(torch.from_numpy(wkv).to(DEV), torch.from_numpy(wgate).to(DEV), torch.from_numpy(gain).to(DEV))
        comps.append(c)
    ref_c, na_c = comps
    for call, (B, N) in enumerate([(2, 4 * 300 + 3), (3, 4 * 151 + 1)]):
        x = torch.from_numpy(np.stack([synthetic.tokens(7 + call, b, 0, N, layer.dim) for b in range(B)])) \
            .to(torch.bfloat16).to(DEV)
        G = N // 4
        ref = ref_c.prefill(x)
        out = ref_c._alloc_out(B * G, x.device, prequant=True)
        g = _call_noalloc(lib, na_c, x, out)
        assert g == G, lib.csa_last_error().decode()
        torch.cuda.synchronize()
        for k in ("latent", "prequant"):
            a, b = _bits(out[k]).reshape(B, G, -1), _bits(ref[k])
            u = ulp_distance_bf16(a, b)
            assert np.mean(u <= 2) >= 0.999 and np.array_equal(a, b), (call, k, int(u.max()))
        for k in ("codes", "scales"):
            assert torch.equal(out[k].view(B, G, -1), ref[k]), (call, k)
        ka, sa = na_c.state_export()
        kb, sb = ref_c.state_export()
        assert torch.equal(ka, kb) and torch.equal(sa, sb), call
    # a chunk continuing the last call's sequences (its carried values also live in the array)
    B, p0, N = 3, 4 * 151 + 1, 4 * 60 + 2
    x = torch.from_numpy(np.stack([synthetic.tokens(9, b, p0, p0 + N, layer.dim) for b in range(B)])) \
        .to(torch.bfloat16).to(DEV)
    G = (p0 + N) // 4 - p0 // 4
    ref = ref_c.prefill(x, start_pos=p0)
    out = ref_c._alloc_out(B * G, x.device, prequant=True)
    assert na_c.prefill_noalloc(x, out, start_pos=p0) == G  # through the binding this time
    torch.cuda.synchronize()
    for k in ("latent", "prequant", "codes", "scales"):
        assert torch.equal(out[k].view(B, G, -1), ref[k]), ("chunk", k)
    assert na_c.device_status() == 0


def test_noalloc_prefill_rejects_sizes_beyond_its_scratch():
    lib = csa.load_library()
    layer = synthetic.Layer(1024, 512, 4, 1, 1.0 / 32)
    wkv, wgate, gain = synthetic.weights(7, layer)
    c = csa.Compressor(layer.dim, layer.head_dim, 4, 1, max_batch=1)
    c.set_weights(torch.from_numpy(wkv).to(DEV), torch.from_numpy(wgate).to(DEV), torch.from_numpy(gain).to(DEV))
    N = 131072  # 521 token tiles x 63 groups x 512 features x 2 bytes > 16 MiB
    x = torch.zeros(1, N, layer.dim, dtype=torch.bfloat16, device=DEV)
    out = c._alloc_out(N // 4, x.device, prequant=True)
    rc = _call_noalloc(lib, c, x, out)
    assert rc == -1 and b"too large" in lib.csa_last_error()

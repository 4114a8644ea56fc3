"""The time-out path of the tensor-core prefill, exercised without any fault: in the bounds-checked
build of the library (CSA_LIBRARY_VARIANT=bounds) the environment variable
CSA_TEST_STALL_LAST_STAGE makes the kernel's producer leave out its last pipeline stage and
shortens every device-side wait to 0.2 s.  The MMA issuer's wait for that stage then runs out: the
kernel raises its abort flag, lets the copies already in flight land and the issued tensor-core
operations complete, frees its TMEM and returns; csa_device_status reports CSA_ERR_TIMEOUT, and the
next ordinary call on the same handle is correct against the oracle.  Both launch geometries: one CTA
per tile, a tile split over K between the two CTAs of a cluster (both stall, both give up, and
they still meet at the cluster barriers and exchange their staged sums before leaving), and two
CTAs sharing one MMA (the leader's MMA wait runs out, the other CTA's wait for the accumulator
does too; the leader waits for its issued MMAs before both free their TMEM together).  The product
build has no such hook, so this file only runs inside the bounds-checked run
(tests/test_gpu_bounds.py)."""
import ctypes
import math
import os

import pytest
import torch

import deepseek_v4_compressed_wkv_gb300 as csa
import synthetic
from _util import layer_inputs
from test_gpu_parity import check_entries, dev_bits, make_pair, to_np

pytestmark = pytest.mark.gpu

CSA_ERR_TIMEOUT = -4


@pytest.mark.parametrize("split,pair", [(1, 0), (2, 0), (1, 2)])
def test_a_wait_that_runs_out_is_reported_and_the_handle_recovers(monkeypatch, split, pair):
    if os.environ.get("CSA_LIBRARY_VARIANT") != "bounds":
        pytest.skip("the stall hook exists only in the bounds-checked build")
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / math.sqrt(256), gate_scale=2.0, rope_dim=64, fp4=1)
    g, o = make_pair(23, layer, max_batch=2, split=split, pair=pair)
    assert g.uses_tensor_cores()
    x, *_ = layer_inputs(23, layer, 2, 4 * 40 + 1)
    lib = csa.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("CSA_TEST_STALL_LAST_STAGE", "1")
    g.prefill(dev_bits(x))  # enqueued; its projection gives up on the missing stage
    rc = lib.csa_device_status(g.handle, stream)
    assert rc == CSA_ERR_TIMEOUT, (rc, lib.csa_last_error())
    assert b"wait budget exhausted" in lib.csa_last_error()
    monkeypatch.delenv("CSA_TEST_STALL_LAST_STAGE")
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    check_entries(to_np(got), o.prefill(x)["prequant"], 1, "prefill after a timed-out call")
    assert g.device_status() == 0

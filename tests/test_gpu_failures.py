"""Failure paths on the GPU, injected on the host (no device fault): a forced scratch allocation
failure is reported as an error code with a message, leaves the handle usable, and the next call
succeeds; an ABI call whose kernel flags an input reports it through csa_device_status."""
import math

import numpy as np
import pytest
import torch

import deepseek_v4_compressed_wkv_gb300 as csa
import synthetic
from _util import layer_inputs
from test_gpu_parity import DEV, check_entries, dev_bits, make_pair, to_np

pytestmark = pytest.mark.gpu


def test_forced_allocation_failure_is_reported_and_the_handle_recovers(monkeypatch):
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / math.sqrt(256), gate_scale=2.0, rope_dim=64, fp4=1)
    g, o = make_pair(17, layer, max_batch=2)
    x, *_ = layer_inputs(17, layer, 2, 4 * 40 + 1)
    monkeypatch.setenv("CSA_TEST_FAIL_ALLOC", "1")
    with pytest.raises(csa.CSAError, match="forced failure"):
        g.prefill(dev_bits(x))  # the first prefill of a handle grows its scratch
    monkeypatch.delenv("CSA_TEST_FAIL_ALLOC")
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    check_entries(to_np(got), o.prefill(x)["prequant"], 1, "prefill after a failed allocation")
    assert g.device_status() == 0


def test_flagged_decode_input_is_reported_once():
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / 16, rope_dim=64, fp4=1)
    g, _ = make_pair(18, layer, max_batch=2)
    x = torch.zeros(2, 256, dtype=torch.bfloat16, device=DEV)
    d = g.decode(x, torch.tensor([5, -2], dtype=torch.int32, device=DEV))
    assert d["emitted"].cpu().tolist() == [0, 0]
    with pytest.raises(csa.CSAError, match="negative start_pos"):
        g.device_status()
    assert g.device_status() == 0  # read and cleared

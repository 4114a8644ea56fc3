"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a, loads,
exports every entry point that include/csa.h declares, rejects bad shapes before touching
the device, and builds the same YaRN RoPE table as the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import deepseek_v4_compressed_wkv_gb300 as csa
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "csa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(csa.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol():
    lib = csa.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the artefact is an sm_103a CUDA build
    assert os.path.exists(csa.library_path())


def test_default_options():
    o = csa.default_options()
    assert (o.max_batch, o.rope_dim, o.rope_base, o.rope_factor, o.rope_orig_len) == (128, 64, 160000.0, 16.0, 4096)
    assert (o.beta_fast, o.beta_slow, o.max_pos, o.fp4) == (32.0, 1.0, 262144, 1)
    assert abs(o.eps - 1e-6) < 1e-12
    assert o.prefill_split == 0 and o.prefill_pair == 0


@pytest.mark.parametrize("args,frag", [((100, 512, 4, 1), "dim"), ((4096, 500, 4, 0), "head_dim"),
                                       ((4096, 1024, 4, 0), "head_dim"), ((4096, 512, 0, 0), "ratio"),
                                       ((4096, 512, 2, 1), "overlapped"), ((4096, 512, 4, 2), "overlap")])
def test_create_rejects_bad_shapes_without_a_device(args, frag):
    lib = csa.load_library()
    h = ctypes.c_void_p()
    o = csa.default_options()
    rc = lib.csa_compressor_create_ex(*args, ctypes.byref(o), ctypes.byref(h))
    assert rc == -1 and not h.value
    assert frag in lib.csa_last_error().decode()
    # the form without options checks the same shapes
    h2 = ctypes.c_void_p()
    assert lib.csa_compressor_create(*args, ctypes.byref(h2)) == -1 and not h2.value
    assert frag in lib.csa_last_error().decode()


def test_create_rejects_bad_options():
    lib = csa.load_library()
    h = ctypes.c_void_p()
    for kw in (dict(rope_dim=63), dict(rope_dim=1024), dict(max_batch=0), dict(fp4=3), dict(fp4=-1),
               dict(prefill_split=3), dict(prefill_split=-1), dict(prefill_pair=1), dict(prefill_pair=3)):
        o = csa.default_options(**kw)
        assert lib.csa_compressor_create_ex(4096, 512, 4, 1, ctypes.byref(o), ctypes.byref(h)) == -1
    # the power-of-two quantiser takes blocks of 32 features
    o = csa.default_options(fp4=2, rope_dim=16)
    assert lib.csa_compressor_create_ex(4096, 48, 4, 0, ctypes.byref(o), ctypes.byref(h)) == -1
    assert "multiple of 32" in lib.csa_last_error().decode()


def test_null_handle_calls_fail_cleanly():
    lib = csa.load_library()
    assert lib.csa_compress_prefill(None, None, 1, 4, 0, 0, None, None) == -1
    assert lib.csa_compress_decode(None, None, 1, None, None, None, None) == -1
    assert lib.csa_compress_decode_dev(None, None, 1, None, None, None, None) == -1
    assert lib.csa_compressor_create(256, 64, 4, 1, None) == -1  # no place for the handle
    assert lib.csa_state_reset(None, 0, 1, None) == -1
    assert lib.csa_state_elems(None) == -1
    assert lib.csa_state_export(None, None, None, None) == -1
    assert lib.csa_state_import(None, None, None, None) == -1
    assert lib.csa_compress_prefill_into(None, None, 1, 4, 0, 0, None, 8, None) == -1
    assert lib.csa_compress_prefill_noalloc(None, None, 1, 4, 0, 0, None, None) == -1
    assert lib.csa_compressor_set_gate_bias(None, None, None) == -1
    assert lib.csa_fp4_e8m0_roundtrip(None, -1, None, None, None, None) == -1
    assert lib.csa_fp4_e8m0_roundtrip(None, 4, None, None, None, None) == -1  # buffers required
    assert lib.csa_fp4_e4m3_roundtrip(None, 4, None, None, None, None) == -1
    assert lib.csa_fp4_e8m0_roundtrip(None, 0, None, None, None, None) == 0  # nothing to do
    lib.csa_compressor_destroy(None)


@pytest.mark.parametrize("pos0,npos", [(0, 64), (131000, 72), (262080, 64)])
def test_rope_table_matches_oracle_frequencies(pos0, npos):
    cs, sn = csa.rope_table(pos0, npos)
    f = oracle.yarn_freqs(64, 160000.0, 16.0, 4096, 32.0, 1.0)
    th = (np.arange(pos0, pos0 + npos, dtype=np.float64)[:, None]) * f[None, :]
    # one rounding from the double-precision angle: at most one float32 ulp from the oracle's angle
    for got, ref in ((cs, np.cos(th)), (sn, np.sin(th))):
        r32 = ref.astype(np.float32)
        ulps = np.abs(got.view(np.int32).astype(np.int64) - r32.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1
    assert np.allclose(cs.astype(np.float64) ** 2 + sn.astype(np.float64) ** 2, 1.0, atol=2e-7)


def test_rope_table_rejects_bad_arguments():
    with pytest.raises(csa.CSAError):
        csa.rope_table(-1, 4)
    with pytest.raises(csa.CSAError):
        csa.rope_table(0, 4, rope_dim=0)


def test_state_window_reproduces_the_full_prefill_state():
    """Prefilling only the tokens the state keeps gives the full prefill's state (oracle)."""
    import synthetic
    from _util import to_bf16_bits
    dim, H = 32, 16
    for ratio, overlap in ((4, 1), (8, 0)):
        for pos in (0, 3, 4, 9, 12, 21, 30, 33):
            layer = synthetic.Layer(dim, H, ratio, overlap, 0.2)
            wkv, wg, gain = synthetic.weights(0, layer)
            full = oracle.Compressor(dim, H, ratio, overlap, rope_dim=0, fp4=0)
            part = oracle.Compressor(dim, H, ratio, overlap, rope_dim=0, fp4=0)
            for c in (full, part):
                c.set_weights(wkv, wg, gain)
            x = to_bf16_bits(synthetic.tokens(0, 0, 0, max(pos, 1), dim))[None]
            t0 = csa.state_window_start(pos, ratio, overlap)
            if pos > 0:
                full.prefill(x[:, :pos])
                if pos > t0:
                    part.prefill(x[:, t0:pos])
            kf, sf = full.state()
            kp, sp = part.state()
            g, rem = pos // ratio, pos % ratio
            if overlap:
                q = g % 2
                assert np.array_equal(kf[:, q, :rem], kp[:, q, :rem]) and np.array_equal(sf[:, q, :rem], sp[:, q, :rem])
                assert np.array_equal(kf[:, 1 - q, :, H:], kp[:, 1 - q, :, H:])
                assert np.array_equal(sf[:, 1 - q, :, H:], sp[:, 1 - q, :, H:])
            else:
                assert np.array_equal(kf[:, :rem], kp[:, :rem]) and np.array_equal(sf[:, :rem], sp[:, :rem])

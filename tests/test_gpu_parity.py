"""Parity of the CUDA library (through its C ABI) with the CPU oracle, on seeded inputs.

Acceptance (per entry, on the pre-fp4 bf16 latent "prequant"):
  - at least 99.9% of elements within 2 bf16 ulps of the oracle;
  - max relative error at most 1e-2: over entries, the largest relative error of an entry
    vector, ||gpu - ref||_2 <= 1e-2 * ||ref||_2 (an elementwise ratio is not meaningful where
    RoPE outputs cancel to near zero, and a max-norm ratio of 1e-2 would forbid the 2-ulp
    differences the first criterion allows: 2 ulps of an element just above a power of two
    are 2^-6 of it);
  - and, per entry, max_i |gpu_i - ref_i| <= 2^-6 * max_i |ref_i|: exactly the 2-ulp allowance
    of the entry's largest element, so that no element (not even among the 0.1% allowed
    outside 2 ulps) is off by more than what two ulps of the entry's top binade allow;
  - the fp4 outputs (codes, scales, dequantised latent) equal the oracle's fp4 round trip
    (e4m3 scales per 16, or power-of-two scales per 32 for the indexer's keys) of the GPU's
    own prequant bit for bit (the quantisers are pinned separately on the oracle's bf16
    input, bit-exact);
  - decode emission flags exact.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import deepseek_v4_compressed_wkv_gb300 as csa
import oracle
import synthetic
from _util import bf16_bits_to_f32, layer_inputs, to_bf16_bits, ulp_distance_bf16

pytestmark = pytest.mark.gpu

DEV = "cuda"


def dev_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def opts_of(layer, max_batch=1, max_pos=262144):
    return dict(max_batch=max_batch, rope_dim=layer.rope_dim, fp4=layer.fp4, max_pos=max_pos)


def make_pair(seed, layer, max_batch=1, max_pos=262144, split=0, pair=0):
    """The library's compressor and the oracle's, with the same synthetic weights.  split forces
    the tensor-core prefill's launch geometry (1: one CTA per tile, 2: two CTAs of a cluster each
    taking half of K; 0: chosen per call); pair = 2 asks for two CTAs sharing one MMA of 256 rows
    where the tiles are not split."""
    wkv, wgate, gain = synthetic.weights(seed, layer)
    g = csa.Compressor(layer.dim, layer.head_dim, layer.ratio, layer.overlap, prefill_split=split,
                       prefill_pair=pair, **opts_of(layer, max_batch, max_pos))
    g.set_weights(torch.from_numpy(wkv).to(DEV), torch.from_numpy(wgate).to(DEV), torch.from_numpy(gain).to(DEV))
    o = oracle.Compressor(layer.dim, layer.head_dim, layer.ratio, layer.overlap, max_batch=max_batch,
                          rope_dim=layer.rope_dim, fp4=layer.fp4)
    o.set_weights(wkv, wgate, gain)
    return g, o


def check_entries(gpu: dict, ref_prequant: np.ndarray, fp4: int, what=""):
    """gpu: dict of numpy arrays (latent, codes, scales, prequant) [..., H]; ref: oracle prequant.
    Returns (fraction within 2 ulps, largest ulp distance) and prints them."""
    gp = gpu["prequant"].reshape(-1, ref_prequant.shape[-1])
    rp = ref_prequant.reshape(gp.shape)
    ulps = ulp_distance_bf16(gp, rp)
    frac2 = float(np.mean(ulps <= 2))
    assert frac2 >= 0.999, f"{what}: only {frac2:.5f} of elements within 2 ulps (max {ulps.max()})"
    g = bf16_bits_to_f32(gp).astype(np.float64)
    r = bf16_bits_to_f32(rp).astype(np.float64)
    rel = np.linalg.norm(g - r, axis=-1) / np.maximum(np.linalg.norm(r, axis=-1), 1e-30)
    w = int(np.argmax(rel))
    assert rel.max() <= 1e-2, f"{what}: entry {w} relative error {rel.max():.3g} (max ulps there {ulps[w].max()})"
    dmax = np.max(np.abs(g - r), axis=-1)
    amax = np.max(np.abs(r), axis=-1)
    over = dmax > 2.0 ** -6 * amax
    if over.any():
        e = int(np.flatnonzero(over)[0])
        raise AssertionError(f"{what}: entry {e} max |diff| {dmax[e]:.4g} > 2^-6 x max |ref| {amax[e]:.4g}"
                             f" ({int(over.sum())} entries; max ulps there {ulps[e].max()})")
    if fp4:
        codes, scales, lat = (oracle.fp4_e8m0 if fp4 == 2 else oracle.fp4_e4m3)(gp)
        assert np.array_equal(gpu["scales"].reshape(-1), scales), f"{what}: scales differ from fp4(prequant)"
        assert np.array_equal(gpu["codes"].reshape(-1), codes), f"{what}: codes differ from fp4(prequant)"
        assert np.array_equal(gpu["latent"].reshape(-1), lat), f"{what}: latent differs from fp4(prequant)"
    else:
        assert np.array_equal(gpu["latent"].reshape(gp.shape), gp)
    print(f"[parity] {what}: {frac2:.6f} within 2 ulps, max {int(ulps.max())} ulps, "
          f"max relative (2-norm) {rel.max():.3g}, entries {gp.shape[0]}")
    return frac2, int(ulps.max())


def to_np(d: dict, rows=None):
    out = {}
    for k, v in d.items():
        if v is None or k in ("emitted", "count") or not isinstance(v, torch.Tensor):
            continue
        a = v.contiguous()
        a = host_bits(a) if a.dtype == torch.bfloat16 else a.cpu().numpy()
        out[k] = a if rows is None else a[rows]
    return out


# ---- the quantiser alone, fed the oracle's bf16 values ---------------------------------------

def test_fp4_quantiser_bit_exact_on_oracle_input():
    rng = np.random.default_rng(0)
    nb = 20000
    mags = 10.0 ** rng.uniform(-4, 4, size=(nb, 1))
    vals = (rng.standard_normal((nb, 16)) * mags).astype(np.float32)
    vals[:50] = 0.0                      # all-zero blocks: floored amax
    vals[50:60, 3] = 6.375               # tie in the scale rounding
    vals[60:70] *= 1e-30                 # tiny blocks
    vals[70:80, 0] = 3.0e38              # saturating scale
    # the latent prequant of a real run, too
    bits = to_bf16_bits(vals)
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite((pats.astype(np.uint32) << 16).view(np.float32))
    sweep = np.zeros((int(finite.sum()), 16), np.uint16)
    sweep[:, 0] = pats[finite]
    sweep[:, 1:] = to_bf16_bits(np.linspace(-1.5, 1.7, 15, dtype=np.float32))
    allb = np.concatenate([bits, sweep])
    codes, scales, out = csa.fp4_e4m3_roundtrip(dev_bits(allb))
    torch.cuda.synchronize()
    rc, rs, ro = oracle.fp4_e4m3(allb)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(host_bits(out), ro)


def test_fp4_e8m0_quantiser_bit_exact_on_oracle_input():
    """The indexer's round trip (power-of-two scales, block 32) against the oracle: random
    blocks over 60 decades, all-zero blocks, exact powers, and every finite bf16 pattern."""
    rng = np.random.default_rng(1)
    nb = 20000
    mags = 10.0 ** rng.uniform(-30, 30, size=(nb, 1))
    vals = (rng.standard_normal((nb, 32)) * mags).astype(np.float32)
    vals[:50] = 0.0
    vals[50:90, 9] = (6.0 * 2.0 ** rng.integers(-60, 60, size=40)).astype(np.float32)
    bits = to_bf16_bits(vals)
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite((pats.astype(np.uint32) << 16).view(np.float32))
    sweep = np.zeros((int(finite.sum()), 32), np.uint16)
    sweep[:, 0] = pats[finite]
    sweep[:, 1:] = to_bf16_bits(np.linspace(-1.5, 1.7, 31, dtype=np.float32))
    allb = np.concatenate([bits, sweep])
    codes, scales, out = csa.fp4_e8m0_roundtrip(dev_bits(allb))
    torch.cuda.synchronize()
    rc, rs, ro = oracle.fp4_e8m0(allb)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(host_bits(out), ro)


# ---- tiny parity workload: prefill, then 64 decode steps from start_pos 0 ---------------------

def test_tiny_prefill_then_decode():
    wl = synthetic.TINY
    layer = wl.layers[0]
    g, o = make_pair(wl.seed, layer)
    x, *_ = layer_inputs(wl.seed, layer, 1, 64)
    ref = o.prefill(x)
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    check_entries(to_np(got), ref["prequant"], layer.fp4, "tiny prefill")
    g.state_reset()
    o.state_reset()
    for p in range(64):
        sp = np.array([p], np.int32)
        r = o.decode(x[:, p], sp)
        d = g.decode(dev_bits(x[:, p]), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"]), p
        if em[0]:
            check_entries(to_np(d, rows=[0]), r["prequant"][[0]], layer.fp4, f"tiny decode p={p}")
    assert g.device_status() == 0


# ---- small shapes over several tiles, ragged tails, odd batches -------------------------------

SMALL = [
    # dim, H, ratio, overlap, B, N
    (256, 128, 4, 1, 3, 4 * 67 + 3),
    (256, 128, 4, 1, 1, 3),          # no complete group: padded previous branch only
    (256, 128, 4, 1, 2, 4),
    (128, 64, 2, 0, 3, 2 * 70 + 1),
    (256, 512, 4, 1, 2, 128 + 5),
    (256, 512, 128, 0, 2, 128 * 3 + 77),
    (256, 256, 64, 0, 2, 64 * 9 + 13),  # long groups at ratio 64 (the two-thread pool, four groups a tile)
    (192, 256, 8, 0, 1, 8 * 40),
    (128, 64, 1, 0, 2, 37),
    (128, 32, 3, 0, 1, 2),
    (128, 32, 3, 0, 2, 3 * 90 + 2),  # packed tile narrower than 128 rows: CUDA-core projection
    (128, 64, 300, 0, 1, 300 * 2 + 7),  # ratio above one token tile: CUDA-core projection
]


SMALL_FP4 = [(d, H, r, ov, B, N, 1) for d, H, r, ov, B, N in SMALL] + [
    # the indexer's 128-wide instance with its power-of-two quantiser (fp4 = 2, block 32)
    (256, 128, 4, 1, 2, 4 * 60 + 1, 2),
    (128, 32, 3, 0, 2, 3 * 40 + 2, 2),   # CUDA-core path with the block-32 quantiser (lane pairs)
    (256, 64, 8, 0, 1, 8 * 30 + 5, 2),
    # few packed tiles at a wider dim (the 128-token tile)
    (1024, 128, 4, 1, 2, 4 * 150 + 3, 2),
    (1024, 128, 8, 0, 1, 8 * 70 + 5, 1),
]


@pytest.mark.parametrize("split,pair", [(1, 0), (2, 0), (1, 2)])
@pytest.mark.parametrize("dim,H,ratio,overlap,B,N,fp4", SMALL_FP4)
def test_small_prefill_state_and_decode(dim, H, ratio, overlap, B, N, fp4, split, pair):
    layer = synthetic.Layer(dim, H, ratio, overlap, 1.0 / math.sqrt(dim), gate_scale=2.0,
                            rope_dim=min(64, H), fp4=fp4)
    g, o = make_pair(5, layer, max_batch=B + 1, split=split, pair=pair)
    x, *_ = layer_inputs(5, layer, B, N + 6)
    xp = np.ascontiguousarray(x[:, :N])
    ref = o.prefill(xp, slot_offset=1)
    G = N // ratio
    canary = 1  # rows past the last entry must stay untouched
    out = {"latent": torch.full((B * G + canary, H), 7.0, dtype=torch.bfloat16, device=DEV),
           "codes": torch.full((B * G + canary, H // 2), 0xA5, dtype=torch.uint8, device=DEV),
           "scales": torch.full((B * G + canary, H // (32 if fp4 == 2 else 16)), 0x5A, dtype=torch.uint8,
                                device=DEV),
           "prequant": torch.full((B * G + canary, H), 7.0, dtype=torch.bfloat16, device=DEV)}
    got = g.prefill(dev_bits(xp), slot_offset=1, out=out)
    torch.cuda.synchronize()
    assert (got is None) == (G == 0)
    if G:
        check_entries(to_np(got), ref["prequant"], fp4, f"prefill {ratio}/{overlap}")
    assert torch.all(out["latent"][B * G:] == 7.0) and torch.all(out["codes"][B * G:] == 0xA5)
    assert torch.all(out["scales"][B * G:] == 0x5A) and torch.all(out["prequant"][B * G:] == 7.0)
    # state after prefill: the meaningful slots equal the oracle's (f32, from f32 projections)
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    ko, so = o.state()
    assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0))
    assert np.array_equal(np.isinf(sg), np.isinf(so))
    fin = np.isfinite(so)
    assert np.allclose(sg[fin], so[fin], rtol=2e-5, atol=2e-5 * np.abs(so[fin]).max(initial=1.0))
    # six decode steps continuing every sequence (slots 0..B: slot 0 is fresh, starts at p=0)
    xall, *_ = layer_inputs(5, layer, B + 1, N + 6)
    xall[1:] = x
    for k in range(6):
        sp = np.array([k] + [N + k] * B, np.int32)
        xt = np.ascontiguousarray(xall[np.arange(B + 1), sp])
        r = o.decode(xt, sp)
        if k % 2:  # positions on the device (csa_compress_decode_dev)
            d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        else:  # positions on the host (csa_compress_decode): the call returns the emitting count
            d = g.decode(dev_bits(xt), sp)
            assert d["count"] == int(np.sum((sp + 1) % ratio == 0)) == int(r["emitted"].sum())
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"]), (k, em, r["emitted"])
        rows = np.flatnonzero(em)
        if rows.size:
            check_entries(to_np(d, rows=rows), r["prequant"][rows], fp4, f"decode step {k}")
    assert g.device_status() == 0


# ---- full-size workloads ------------------------------------------------------------------

def test_flash_csa_prefill_full():
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    g, o = make_pair(wl.seed, layer)
    x, *_ = layer_inputs(wl.seed, layer, 1, 4096)
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    ref = o.prefill(x)
    frac, mx = check_entries(to_np(got), ref["prequant"], 1, "Flash CSA prefill")
    assert ref["G"] == 1024


def test_cta_pairs_give_the_single_cta_results():
    """Two CTAs sharing one MMA of 256 rows (prefill_pair = 2) form the same products and add them
    in the same order as one CTA per packed tile: the Flash CSA prefill's entries (before and after
    fp4) and its state are bit-identical, and a chunk continuing it is too."""
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    x, *_ = layer_inputs(wl.seed, layer, 1, 4096 + 300)
    res = []
    for pair in (0, 2):
        g, _ = make_pair(wl.seed, layer, pair=pair)
        assert g.prefill_geometry(1, 4096)["cta_pair"] == (2 if pair else 1)
        a = g.prefill(dev_bits(np.ascontiguousarray(x[:, :4096])))
        b = g.prefill(dev_bits(np.ascontiguousarray(x[:, 4096:])), start_pos=4096)
        torch.cuda.synchronize()
        res.append((a, b, [t.cpu() for t in g.state_export()]))
        assert g.device_status() == 0
        g.close()
    (a0, b0, s0), (a1, b1, s1) = res
    for k in ("latent", "codes", "scales", "prequant"):
        assert torch.equal(a0[k].cpu(), a1[k].cpu()), k
        assert torch.equal(b0[k].cpu(), b1[k].cpu()), k
    assert all(torch.equal(u, v) for u, v in zip(s0, s1))


def sampled_groups(G, k, seed):
    rng = np.random.default_rng(seed)
    picks = {0, 1, G - 1, G // 2} | set(rng.choice(G, size=min(k, G), replace=False).tolist())
    return sorted(p for p in picks if 0 <= p < G)


def test_hca_prefill_sampled_groups_and_tail_state():
    wl = synthetic.HCA
    layer = wl.layers[0]
    B, N = wl.batch, wl.tokens[0]
    g, o = make_pair(wl.seed, layer, max_batch=B)
    x, wkv, wgate, _ = layer_inputs(wl.seed, layer, B, N)
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    G = N // layer.ratio
    assert G == 128 and N % layer.ratio == 77
    gn = to_np(got)
    for b in range(B):
        grp = sampled_groups(G, 4, b)
        ref = o.prefill_groups(x[b], grp)
        sel = {k: v[b][grp] for k, v in gn.items()}
        check_entries(sel, ref["prequant"], 1, f"HCA b={b}")
    # the 77-token tail sits in state slots 0..76 of each sequence
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    for b in range(B):
        tail = x[b, 128 * G:]
        kv = oracle.linear(tail, wkv, nthreads=8)
        sc = oracle.linear(tail, wgate, nthreads=8)
        assert np.allclose(kg[b, :77], kv, rtol=1e-5, atol=1e-5 * np.abs(kv).max())
        assert np.allclose(sg[b, :77], sc, rtol=1e-5, atol=1e-5 * np.abs(sc).max())


@pytest.mark.parametrize("N,layer_idx", [(131072, 0), (131072, 1), (16384, 0)])
def test_long_prefill_sampled(N, layer_idx):
    wl = synthetic.LONG
    layer = wl.layers[layer_idx]
    g, o = make_pair(wl.seed, layer)
    x, *_ = layer_inputs(wl.seed, layer, 1, N, outlier_frac=wl.outlier_frac)
    got = g.prefill(dev_bits(x), prequant=True)
    torch.cuda.synchronize()
    G = N // layer.ratio
    grp = sampled_groups(G, 24, N)
    # include groups that hold outlier tokens
    mask = synthetic.outlier_mask(wl.seed, 0, 0, N, wl.outlier_frac)
    out_groups = np.unique(np.flatnonzero(mask) // layer.ratio)
    grp = sorted(set(grp) | set(out_groups[:8].tolist()))
    ref = o.prefill_groups(x[0], grp)
    gn = {k: v[0][grp] for k, v in to_np(got).items()}
    check_entries(gn, ref["prequant"], 1, f"long N={N} ratio={layer.ratio}")


def test_long_batched_prefill_sampled():
    wl = synthetic.LONG
    layer = wl.layers[0]
    B, N = wl.extra["batched"]
    g, o = make_pair(wl.seed, layer, max_batch=B)
    x, *_ = layer_inputs(wl.seed, layer, B, N, outlier_frac=wl.outlier_frac)
    got = g.prefill(dev_bits(x))
    torch.cuda.synchronize()
    gn = to_np(got)
    G = N // 4
    for b in (0, 3, 7):
        grp = sampled_groups(G, 6, b)
        ref = o.prefill_groups(x[b], grp)
        check_entries({k: v[b][grp] for k, v in gn.items()}, ref["prequant"], 1, f"B8 b={b}")


def test_batched_decode_both_compressors():
    wl = synthetic.DECODE
    B = wl.batch
    sp0 = synthetic.start_positions(wl.seed, B, wl.start_pos_hi)
    steps = 12
    for layer in wl.layers:
        g, o = make_pair(wl.seed, layer, max_batch=B)
        # bring every sequence's state to its start position
        for b in range(B):
            s = int(sp0[b])
            t0 = csa.state_window_start(s, layer.ratio, layer.overlap)
            if s > t0:
                xb = to_bf16_bits(synthetic.tokens(wl.seed, b, t0, s, layer.dim))[None]
                o.prefill(xb, slot_offset=b)
                g.prefill(dev_bits(xb), slot_offset=b, prequant=False)
        for k in range(steps):
            sp = (sp0 + k).astype(np.int32)
            xt = to_bf16_bits(np.stack([synthetic.tokens(wl.seed, b, int(sp[b]), int(sp[b]) + 1, layer.dim)[0]
                                        for b in range(B)]))
            r = o.decode(xt, sp)
            d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
            em = d["emitted"].cpu().numpy()
            assert np.array_equal(em, r["emitted"])
            assert np.array_equal(em, ((sp + 1) % layer.ratio == 0).astype(np.uint8))
            rows = np.flatnonzero(em)
            if rows.size:
                check_entries(to_np(d, rows=rows), r["prequant"][rows], 1, f"decode r={layer.ratio} k={k}")
        assert g.device_status() == 0


# ---- error paths on the device --------------------------------------------------------------

def test_errors_are_reported_not_raised_on_the_device():
    layer = synthetic.Layer(128, 64, 4, 1, 0.1, rope_dim=64)
    g = csa.Compressor(128, 64, 4, 1, max_batch=2, max_pos=64)
    x = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(csa.CSAError, match="weights not set"):
        g.prefill(x)
    wkv, wgate, gain = synthetic.weights(0, layer)
    g.set_weights(torch.from_numpy(wkv).to(DEV), torch.from_numpy(wgate).to(DEV), torch.from_numpy(gain).to(DEV))
    with pytest.raises(csa.CSAError, match="max_batch"):
        g.prefill(torch.zeros(3, 8, 128, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(csa.CSAError, match="RoPE table"):
        g.prefill(torch.zeros(1, 4 * 20, 128, dtype=torch.bfloat16, device=DEV))
    lib = csa.load_library()
    assert lib.csa_compress_prefill(g.handle, x.data_ptr(), 1, 8, -1, 0, None, None) == -1  # negative start_pos
    assert lib.csa_compress_prefill(g.handle, x.data_ptr(), 1, 8, 5, 0, None, None) == -1  # entries but no out
    # the binding refuses outputs too small for what the call writes, and mismatched lengths
    small = g._alloc_out(1, DEV)
    with pytest.raises(csa.CSAError, match="holds"):
        g.prefill(torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=DEV), out=small)  # 4 entries
    with pytest.raises(csa.CSAError, match="start_pos has"):
        g.decode(torch.zeros(2, 128, dtype=torch.bfloat16, device=DEV), torch.zeros(3, dtype=torch.int32, device=DEV))
    with pytest.raises(csa.CSAError, match="multiple of 16"):
        csa.fp4_e4m3_roundtrip(torch.zeros(24, dtype=torch.bfloat16, device=DEV))
    # empty calls are argument errors that enqueue nothing (the oracle rejects them alike)
    n0 = g.kernel_launches()
    assert lib.csa_compress_prefill(g.handle, x.data_ptr(), 1, 0, 0, 0, None, None) == -1
    assert lib.csa_compress_prefill(g.handle, x.data_ptr(), 0, 8, 0, 0, None, None) == -1
    sp1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    em1 = torch.zeros(1, dtype=torch.uint8, device=DEV)
    o1 = csa.Out(torch.zeros(1, 64, dtype=torch.bfloat16, device=DEV).data_ptr(), None, None, None)
    assert lib.csa_compress_decode_dev(g.handle, x.data_ptr(), 0, sp1.data_ptr(), ctypes.byref(o1), em1.data_ptr(),
                                       None) == -1
    hp = np.zeros(2, np.int32)
    assert lib.csa_compress_decode(g.handle, x.data_ptr(), 0, hp.ctypes.data, ctypes.byref(o1), None, None) == -1
    # host positions are checked on the host: a negative one, or an entry beyond the RoPE table
    # (max_pos 64), is an argument error that enqueues nothing
    for bad in ([-3, 5], [4, 67]):
        hp = np.array(bad, np.int32)
        assert lib.csa_compress_decode(g.handle, x.data_ptr(), 2, hp.ctypes.data, ctypes.byref(o1), None, None) == -1
    assert "negative" in lib.csa_last_error().decode() or "RoPE" in lib.csa_last_error().decode()
    with pytest.raises(csa.CSAError, match="negative"):
        g.decode(torch.zeros(2, 128, dtype=torch.bfloat16, device=DEV), np.array([-1, 3], np.int32))
    assert g.kernel_launches() == n0
    # decode positions the kernel cannot serve: flagged, rows not emitted, context still usable
    sp = torch.tensor([-3, 67], dtype=torch.int32, device=DEV)
    d = g.decode(torch.zeros(2, 128, dtype=torch.bfloat16, device=DEV), sp)
    assert d["emitted"].cpu().tolist() == [0, 0]
    with pytest.raises(csa.CSAError, match="device flag"):
        g.device_status()
    assert g.device_status() == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("ratio,overlap", [(4, 1), (16, 0)])
def test_host_position_decode_through_the_c_abi(ratio, overlap):
    """csa_compress_decode with host positions: its return value is the number of sequences whose
    token completes a group ((start_pos + 1) % ratio == 0, the pages' "None" for the others), a
    host emitted array is filled before it returns, a device one by the kernels; the entries match
    the oracle and the device-position form (csa_compress_decode_dev) on a twin handle, bit for
    bit."""
    B = 37
    layer = synthetic.Layer(256, 128, ratio, overlap, 1.0 / 16, gate_scale=2.0, rope_dim=64, fp4=1)
    g, o = make_pair(21, layer, max_batch=B)
    twin, _ = make_pair(21, layer, max_batch=B)
    lib = csa.load_library()
    sp0 = (np.arange(B) * 5 % 23).astype(np.int32)
    for b in range(B):
        s0 = int(sp0[b])
        t0 = csa.state_window_start(s0, ratio, overlap)
        if s0 > t0:
            xb = to_bf16_bits(synthetic.tokens(21, b, t0, s0, layer.dim))[None]
            o.prefill(xb, slot_offset=b)
            for h in (g, twin):
                h.prefill(dev_bits(xb), slot_offset=b, prequant=False)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    total = 0
    for k in range(ratio + 2):
        sp = (sp0 + k).astype(np.int32)
        xt = to_bf16_bits(np.stack([synthetic.tokens(21, b, int(sp[b]), int(sp[b]) + 1, layer.dim)[0]
                                    for b in range(B)]))
        xd = dev_bits(xt)
        r = o.decode(xt, sp)
        outs = [g._alloc_out(B, DEV) for _ in range(2)]
        os_ = [g._out_struct(d) for d in outs]
        em_host = np.full(B, 9, np.uint8)
        em_dev = torch.full((B,), 9, dtype=torch.uint8, device=DEV)
        # host emitted on even steps, device emitted on odd ones
        em_ptr = em_host.ctypes.data if k % 2 == 0 else em_dev.data_ptr()
        n = lib.csa_compress_decode(g.handle, xd.data_ptr(), B, sp.ctypes.data, ctypes.byref(os_[0]), em_ptr, stream)
        assert n == int(np.sum((sp + 1) % ratio == 0)), (k, n, lib.csa_last_error())
        em = em_host if k % 2 == 0 else em_dev.cpu().numpy()
        assert np.array_equal(em, r["emitted"]) and int(em.sum()) == n
        spd = torch.from_numpy(sp).to(DEV)
        em2 = torch.zeros(B, dtype=torch.uint8, device=DEV)
        assert lib.csa_compress_decode_dev(twin.handle, xd.data_ptr(), B, spd.data_ptr(), ctypes.byref(os_[1]),
                                           em2.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert np.array_equal(em2.cpu().numpy(), r["emitted"])
        rows = np.flatnonzero(r["emitted"])
        total += rows.size
        if rows.size:
            check_entries(to_np(outs[0], rows=rows), r["prequant"][rows], 1, f"host-position decode k={k}")
            for key in ("latent", "prequant", "codes", "scales"):
                assert torch.equal(outs[0][key][rows], outs[1][key][rows]), key
    assert total > 0
    assert g.device_status() == 0 and twin.device_status() == 0


@pytest.mark.parametrize("B,ratio,overlap", [(200, 4, 1), (130, 16, 0)])
def test_decode_batch_beyond_one_token_tile(B, ratio, overlap):
    """More sequences than one MMA token tile (128): the decode runs in token chunks."""
    layer = synthetic.Layer(256, 128, ratio, overlap, 1.0 / 16, rope_dim=64, fp4=1)
    g, o = make_pair(9, layer, max_batch=B)
    sp0 = (np.arange(B) * 7 % 61).astype(np.int32)
    for b in range(B):
        s = int(sp0[b])
        t0 = csa.state_window_start(s, ratio, overlap)
        if s > t0:
            xb = to_bf16_bits(synthetic.tokens(9, b, t0, s, layer.dim))[None]
            o.prefill(xb, slot_offset=b)
            g.prefill(dev_bits(xb), slot_offset=b, prequant=False)
    for k in range(ratio + 1):
        sp = (sp0 + k).astype(np.int32)
        xt = to_bf16_bits(np.stack([synthetic.tokens(9, b, int(sp[b]), int(sp[b]) + 1, layer.dim)[0]
                                    for b in range(B)]))
        r = o.decode(xt, sp)
        d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"])
        rows = np.flatnonzero(em)
        if rows.size:
            check_entries(to_np(d, rows=rows), r["prequant"][rows], 1, f"decode B={B} k={k}")
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    ko, so = o.state()
    assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0))
    assert g.device_status() == 0


@pytest.mark.parametrize("B", [4096, 4097])
def test_decode_at_the_batch_limit_of_the_tensor_core_path(B):
    """4096 sequences, the most the tensor-core decode takes in one call, and one more, which
    runs the CUDA-core decode: states from four batched prefills of different lengths (so that
    the sequences emit at different steps), then five steps against the oracle."""
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / 16, gate_scale=2.0, rope_dim=64, fp4=1)
    g, o = make_pair(13, layer, max_batch=B)
    lens = [5, 6, 7, 8]
    x, *_ = layer_inputs(13, layer, B, max(lens) + 5)
    q = -(-B // len(lens))
    sp0 = np.zeros(B, np.int32)
    for i, n in enumerate(lens):
        b0, b1 = i * q, min(B, (i + 1) * q)
        xp = np.ascontiguousarray(x[b0:b1, :n])
        o.prefill(xp, slot_offset=b0)
        g.prefill(dev_bits(xp), slot_offset=b0, prequant=False)
        sp0[b0:b1] = n
    emitted_any = 0
    for k in range(5):
        sp = (sp0 + k).astype(np.int32)
        xt = np.ascontiguousarray(x[np.arange(B), sp])
        r = o.decode(xt, sp)
        d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"]), k
        rows = np.flatnonzero(em)
        emitted_any += rows.size
        if rows.size:
            check_entries(to_np(d, rows=rows), r["prequant"][rows], 1, f"decode B={B} step {k}")
    assert emitted_any == B + q  # positions n .. n+4 complete one group each, two from n = 7
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    ko, so = o.state()
    assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0))
    assert g.device_status() == 0


# ---- decode calls queued back to back (launches that start before the previous one ends) -----

def _decode_setup(seed, layers, B, pos_hi):
    """Two compressors, every sequence's state brought to its start position on both sides."""
    sp0 = (np.arange(B) * 37 % pos_hi).astype(np.int32)
    pairs = []
    for layer in layers:
        g, o = make_pair(seed, layer, max_batch=B)
        for b in range(B):
            s = int(sp0[b])
            t0 = csa.state_window_start(s, layer.ratio, layer.overlap)
            if s > t0:
                xb = to_bf16_bits(synthetic.tokens(seed, b, t0, s, layer.dim))[None]
                o.prefill(xb, slot_offset=b)
                g.prefill(dev_bits(xb), slot_offset=b, prequant=False)
        pairs.append((g, o))
    return sp0, pairs


def _step_inputs(seed, layer, sp):
    return to_bf16_bits(np.stack([synthetic.tokens(seed, b, int(sp[b]), int(sp[b]) + 1, layer.dim)[0]
                                  for b in range(len(sp))]))


DECODE_PAIR = [synthetic.Layer(512, 512, 4, 1, 1.0 / 22, gate_scale=2.0, rope_dim=64, fp4=1),
               synthetic.Layer(512, 512, 16, 0, 1.0 / 22, gate_scale=2.0, rope_dim=64, fp4=1, weight_stream=3)]


def _check_steps(pairs, seed, sp0, steps, outs, layers=DECODE_PAIR):
    # the entries of all steps of a layer are checked together: the 2-ulp share is a property
    # of a sample, and one step may emit a single entry
    got = [[] for _ in pairs]
    ref = [[] for _ in pairs]
    for k in range(steps):
        sp = (sp0 + k).astype(np.int32)
        for li, (g, o) in enumerate(pairs):
            xt = _step_inputs(seed, layers[li], sp)
            r = o.decode(xt, sp)
            d = outs[k][li]
            em = d["emitted"].cpu().numpy()
            assert np.array_equal(em, r["emitted"]), (k, li)
            rows = np.flatnonzero(em)
            if rows.size:
                got[li].append(to_np(d, rows=rows))
                ref[li].append(r["prequant"][rows])
    for li in range(len(pairs)):
        assert got[li], li
        merged = {kk: np.concatenate([gd[kk] for gd in got[li]]) for kk in got[li][0]}
        check_entries(merged, np.concatenate(ref[li]), 1, f"queued decode layer {li}")
    for g, o in pairs:
        kg, sg = (t.cpu().numpy() for t in g.state_export())
        ko, so = o.state()
        assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0))
        assert g.device_status() == 0


def test_decode_steps_queued_without_host_sync():
    """Steps of two compressors enqueued back to back with no synchronisation between them
    (each call's projection may start while the previous call's kernels run): every step's
    entries and the final state equal the oracle's step-by-step results."""
    seed, B, steps = 21, 40, 20
    sp0, pairs = _decode_setup(seed, DECODE_PAIR, B, 97)
    xs = {}
    for k in range(steps):
        sp = (sp0 + k).astype(np.int32)
        for li in range(2):
            xs[k, li] = (dev_bits(_step_inputs(seed, DECODE_PAIR[li], sp)), torch.from_numpy(sp).to(DEV))
    torch.cuda.synchronize()
    outs = [[pairs[li][0].decode(*xs[k, li]) for li in range(2)] for k in range(steps)]
    torch.cuda.synchronize()
    _check_steps(pairs, seed, sp0, steps, outs)


@pytest.mark.parametrize("case", ["small", "decode_workload"])
def test_decode_steps_in_a_cuda_graph(case):
    """The same steps captured once in a CUDA graph and replayed (the way bench.py times decode):
    identical to the oracle.  "decode_workload" is the benchmark's pair of Flash-width
    compressors (ratio 4 overlapped and ratio 128, dim 4096, head_dim 512) with 128 sequences
    at positions up to 8191."""
    if case == "small":
        layers, seed, B, pos_hi, steps = DECODE_PAIR, 23, 40, 97, 12
    else:
        layers, seed, B, pos_hi, steps = synthetic.DECODE.layers, 25, synthetic.DECODE.batch, 8191, 12
    sp0, pairs = _decode_setup(seed, layers, B, pos_hi)
    xs = {}
    for k in range(steps):
        sp = (sp0 + k).astype(np.int32)
        for li in range(2):
            xs[k, li] = (dev_bits(_step_inputs(seed, layers[li], sp)), torch.from_numpy(sp).to(DEV))
    outs = [[{"emitted": torch.empty(B, dtype=torch.uint8, device=DEV),
              **pairs[li][0]._alloc_out(B, DEV, prequant=True)} for li in range(2)] for k in range(steps)]

    def run():
        for k in range(steps):
            for li in range(2):
                o = outs[k][li]
                pairs[li][0].decode(*xs[k, li], out={kk: v for kk, v in o.items() if kk != "emitted"},
                                    emitted=o["emitted"])

    # one eager step first (the library sizes its scratch on first use), then back to the start
    pairs[0][0].decode(*xs[0, 0])
    pairs[1][0].decode(*xs[0, 1])
    torch.cuda.synchronize()
    for li, (g, _) in enumerate(pairs):
        layer = layers[li]
        g.state_reset()
        for b in range(B):
            s = int(sp0[b])
            t0 = csa.state_window_start(s, layer.ratio, layer.overlap)
            if s > t0:
                g.prefill(dev_bits(to_bf16_bits(synthetic.tokens(seed, b, t0, s, layer.dim))[None]), slot_offset=b,
                          prequant=False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    graph.replay()
    torch.cuda.synchronize()
    _check_steps(pairs, seed, sp0, steps, outs, layers)


def test_decode_rollback_and_reset_between_steps():
    """Positions decoded a second time with other tokens (a rollback), and the state reset and
    partly prefilled again mid-stream: each decode emits what the oracle emits from the same
    state.
    (The non-overlapped decode keeps running softmax values of the open group between calls;
    they must not outlive a change of the state slots they summarise.)"""
    seed, B = 31, 24
    layers = [DECODE_PAIR[1], synthetic.Layer(512, 256, 8, 0, 1.0 / 22, gate_scale=2.0, rope_dim=64, fp4=1,
                                              weight_stream=5)]
    got, ref = [[], []], [[], []]
    for li, layer in enumerate(layers):
        sp0, (pair,) = _decode_setup(seed, [layer], B, 97)
        g, o = pair

        def step(k, salt=0):
            sp = (sp0 + k).astype(np.int32)
            xt = to_bf16_bits(np.stack([synthetic.tokens(seed + salt, b, int(sp[b]), int(sp[b]) + 1, layer.dim)[0]
                                        for b in range(B)]))
            r = o.decode(xt, sp)
            d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
            em = d["emitted"].cpu().numpy()
            assert np.array_equal(em, r["emitted"]), (li, k, salt)
            rows = np.flatnonzero(em)
            if rows.size:
                got[li].append(to_np(d, rows=rows))
                ref[li].append(r["prequant"][rows])

        for k in range(10):
            step(k)
        for k in range(4, 14):  # roll back six positions, other tokens
            step(k, salt=1)
        # reset every slot, bring half of the sequences back to their start positions; the
        # other half continues from the reset state
        half = B // 2
        g.state_reset()
        o.state_reset()
        for b in range(half):
            s = int(sp0[b])
            t0 = csa.state_window_start(s, layer.ratio, layer.overlap)
            if s > t0:
                xb = to_bf16_bits(synthetic.tokens(seed, b, t0, s, layer.dim))[None]
                o.prefill(xb, slot_offset=b)
                g.prefill(dev_bits(xb), slot_offset=b, prequant=False)
        for k in range(0, 2 * layer.ratio):
            step(k, salt=2)
        kg, sg = (t.cpu().numpy() for t in g.state_export())
        ko, so = o.state()
        assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0))
        assert g.device_status() == 0
    for li in range(2):
        assert got[li], li
        merged = {kk: np.concatenate([gd[kk] for gd in got[li]]) for kk in got[li][0]}
        check_entries(merged, np.concatenate(ref[li]), 1, f"rollback/reset layer {li}")


@pytest.mark.parametrize("li", [0, 1])
def test_state_moves_to_another_handle(li):
    """csa_state_import: the state exported from one handle and imported into another of the same
    shape continues the same sessions.  Both handles then decode the same tokens: the overlapped
    compressor's entries are bit-identical to the first handle's; the non-overlapped one rebuilds
    its running softmax values from the imported slots (the same softmax in another order), so its
    entries are checked against the oracle, which continues the sessions as well."""
    seed, B = 41, 16
    layer = DECODE_PAIR[li]
    sp0, ((g, o),) = _decode_setup(seed, [layer], B, 61)
    for k in range(3):  # a few steps first, so that the running values are in use
        sp = (sp0 + k).astype(np.int32)
        xt = _step_inputs(seed, layer, sp)
        o.decode(xt, sp)
        g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
    h, _ = make_pair(seed, layer, max_batch=B)
    kv, sc = g.state_export()
    h.state_import(kv, sc)
    k2, s2 = h.state_export()
    assert torch.equal(kv, k2) and torch.equal(sc, s2)
    got, ref = [], []
    for k in range(3, 3 + 2 * layer.ratio):
        sp = (sp0 + k).astype(np.int32)
        xt = _step_inputs(seed, layer, sp)
        r = o.decode(xt, sp)
        a = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        b_ = h.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = b_["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"]) and np.array_equal(em, a["emitted"].cpu().numpy())
        rows = np.flatnonzero(em)
        if rows.size:
            if layer.overlap:
                assert torch.equal(a["latent"][rows], b_["latent"][rows])
            got.append(to_np(b_, rows=rows))
            ref.append(r["prequant"][rows])
    assert got
    merged = {kk: np.concatenate([gd[kk] for gd in got]) for kk in got[0]}
    check_entries(merged, np.concatenate(ref), 1, "decode after the state moved")
    assert g.device_status() == 0 and h.device_status() == 0
    with pytest.raises(csa.CSAError):
        h.state_import(kv[:-1], sc)

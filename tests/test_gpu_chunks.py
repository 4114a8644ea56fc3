"""Prefill chunks at start_pos > 0 and prefill straight into a caller's compressed-KV cache.

A chunk continues sequences whose earlier tokens are in the state: its entries and the state
it leaves must be those of the oracle's chunk (itself pinned to token-by-token decode and to
one whole prefill).  Each call of a chain is compared with the oracle (entries within the
parity tolerance of the other tests, state within f32 rounding), then decode steps continue
the chain.  Shapes cover both projection paths (tensor-core and CUDA-core), chunks that start
mid-group, complete no group, span several token tiles, and the ratios 1, 3, 4 (overlapped),
8, 128 and 300.
"""
import math

import numpy as np
import pytest
import torch

import synthetic
from _util import layer_inputs
from test_gpu_parity import DEV, check_entries, dev_bits, make_pair, to_np

pytestmark = pytest.mark.gpu


def check_state(g, o, what):
    kg, sg = (t.cpu().numpy() for t in g.state_export())
    ko, so = o.state()
    assert np.allclose(kg, ko, rtol=2e-5, atol=2e-5 * np.abs(ko).max(initial=1.0)), what
    assert np.array_equal(np.isinf(sg), np.isinf(so)), what
    fin = np.isfinite(so)
    assert np.allclose(sg[fin], so[fin], rtol=2e-5, atol=2e-5 * np.abs(so[fin]).max(initial=1.0)), what


CHAINS = [
    # dim, H, ratio, overlap, B, chunk lengths (the first call starts at position 0)
    (256, 128, 4, 1, 2, (6, 1, 2, 4 * 70 + 3, 9, 500)),
    (256, 512, 4, 1, 1, (1, 2, 260, 4)),
    (256, 512, 128, 0, 2, (100, 30, 128 * 3 + 77, 5)),
    (192, 256, 8, 0, 2, (13, 8 * 40 + 3, 4, 8)),
    (128, 64, 1, 0, 2, (5, 7)),
    (1024, 128, 4, 1, 1, (9, 4 * 100 + 2, 301)),
    (128, 32, 3, 0, 2, (4, 3 * 90 + 2, 1)),      # packed tile narrower than 128 rows: CUDA-core path
    (128, 64, 300, 0, 1, (310, 300 * 2 + 7, 5)),  # ratio above one token tile: CUDA-core path
]


@pytest.mark.parametrize("split,pair", [(1, 0), (2, 0), (1, 2)])
@pytest.mark.parametrize("dim,H,ratio,overlap,B,chunks", CHAINS)
def test_prefill_chunks_then_decode(dim, H, ratio, overlap, B, chunks, split, pair):
    layer = synthetic.Layer(dim, H, ratio, overlap, 1.0 / math.sqrt(dim), gate_scale=2.0, rope_dim=min(64, H), fp4=1)
    g, o = make_pair(11, layer, max_batch=B + 1, split=split, pair=pair)
    P = sum(chunks)
    x, *_ = layer_inputs(11, layer, B, P + 5)
    p0 = 0
    for n in chunks:
        xc = np.ascontiguousarray(x[:, p0:p0 + n])
        ref = o.prefill(xc, slot_offset=1, start_pos=p0)
        got = g.prefill(dev_bits(xc), slot_offset=1, start_pos=p0)
        torch.cuda.synchronize()
        G = (p0 + n) // ratio - p0 // ratio
        assert ref["G"] == G and (got is None) == (G == 0)
        if G:
            check_entries(to_np(got), ref["prequant"], 1, f"chunk at {p0} (+{n})")
        check_state(g, o, f"state after the chunk at {p0}")
        p0 += n
    # decode continues the chained sequences
    for k in range(5):
        sp = np.full(B, P + k, np.int32)
        xt = np.ascontiguousarray(x[:, P + k])
        xt_all = np.concatenate([np.zeros((1, dim), np.uint16), xt])  # slot 0 restarts at position 0
        sp_all = np.concatenate([[0], sp]).astype(np.int32)
        r = o.decode(xt_all, sp_all)
        d = g.decode(dev_bits(xt_all), torch.from_numpy(sp_all).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"])
        rows = np.flatnonzero(em)
        if rows.size:
            check_entries(to_np(d, rows=rows), r["prequant"][rows], 1, f"decode after chunks, step {k}")
    assert g.device_status() == 0


def _random_chains(n, seed=2027):
    """Seeded random chunk chains: shape, ratio and chunk lengths drawn so that chunks start
    anywhere in a group, span zero to several token tiles, and mix both projection paths."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        ratio, overlap = [(1, 0), (2, 0), (3, 0), (4, 1), (4, 0), (8, 0), (16, 0), (128, 0)][rng.integers(8)]
        dim = int(rng.choice([128, 256]))
        H = int(rng.choice([32, 64, 128, 128, 256]))
        B = int(rng.integers(1, 4))
        lens = tuple(int(v) for v in rng.integers(1, 700, size=int(rng.integers(2, 5))))
        out.append((dim, H, ratio, overlap, B, lens))
    return out


@pytest.mark.parametrize("dim,H,ratio,overlap,B,chunks", _random_chains(12))
def test_random_chunk_chains(dim, H, ratio, overlap, B, chunks):
    layer = synthetic.Layer(dim, H, ratio, overlap, 1.0 / math.sqrt(dim), gate_scale=2.0, rope_dim=min(64, H), fp4=1)
    g, o = make_pair(17, layer, max_batch=B)
    x, *_ = layer_inputs(17, layer, B, sum(chunks))
    p0 = 0
    for n in chunks:
        xc = np.ascontiguousarray(x[:, p0:p0 + n])
        ref = o.prefill(xc, start_pos=p0)
        got = g.prefill(dev_bits(xc), start_pos=p0)
        torch.cuda.synchronize()
        assert (got is None) == (ref["G"] == 0)
        if ref["G"]:
            check_entries(to_np(got), ref["prequant"], 1, f"chunk at {p0} (+{n})")
        p0 += n
    check_state(g, o, "state after the chain")
    assert g.device_status() == 0


@pytest.mark.parametrize("split,pair", [(1, 0), (1, 2)])
def test_chunk_of_many_sequences_across_waves(split, pair):
    """A chunk whose first token tile reads candidates from the state that its later tiles rewrite,
    for 64 sequences at once: the grid (packed tiles x token tiles x sequences) runs in several
    waves, so a later tile's CTA may start before or long after the first tile of its sequence;
    it writes the state only once that tile has read it.  Entries and state against the oracle,
    and no time-out."""
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / 16, gate_scale=2.0, rope_dim=64, fp4=1)
    B, p0, n = 64, 4 * 20 + 2, 4 * 75 + 1  # the chunk starts two tokens into a group
    g, o = make_pair(31, layer, max_batch=B, split=split, pair=pair)
    x, *_ = layer_inputs(31, layer, B, p0 + n)
    for q0, q1 in ((0, p0), (p0, p0 + n)):
        xc = np.ascontiguousarray(x[:, q0:q1])
        ref = o.prefill(xc, start_pos=q0)
        got = g.prefill(dev_bits(xc), start_pos=q0)
        torch.cuda.synchronize()
        check_entries(to_np(got), ref["prequant"], 1, f"chunk at {q0} (+{q1 - q0})")
    T = g.prefill_geometry(B, n, p0)["token_tile"] - 4  # tokens a tile owns (overlapped: less the halo)
    assert -(-(p0 % 4 + n) // T) >= 2  # several token tiles per sequence
    check_state(g, o, "state after the chunk")
    assert g.device_status() == 0


def test_prefill_into_cache_rows():
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / 16, gate_scale=2.0, rope_dim=64, fp4=1)
    B, rows = 2, 100
    g, _ = make_pair(12, layer, max_batch=B)
    h, _ = make_pair(12, layer, max_batch=B)
    x, *_ = layer_inputs(12, layer, B, 300)
    H = layer.head_dim
    cache = {"latent": torch.full((B, rows, H), 7.0, dtype=torch.bfloat16, device=DEV),
             "codes": torch.full((B, rows, H // 2), 0xA5, dtype=torch.uint8, device=DEV),
             "scales": torch.full((B, rows, H // 16), 0x5A, dtype=torch.uint8, device=DEV),
             "prequant": torch.full((B, rows, H), 7.0, dtype=torch.bfloat16, device=DEV)}
    p0 = 0
    for n in (10, 50, 3, 201):
        xc = dev_bits(np.ascontiguousarray(x[:, p0:p0 + n]))
        wrote = g.prefill_into(xc, cache, start_pos=p0)
        ref = h.prefill(xc, start_pos=p0)
        g0, g1 = p0 // 4, (p0 + n) // 4
        assert wrote == g1 - g0
        if ref is not None:
            for k in cache:  # the same kernels: identical bits
                assert torch.equal(cache[k][:, g0:g1], ref[k]), (p0, k)
        p0 += n
    end = p0 // 4
    assert torch.all(cache["latent"][:, end:] == 7.0) and torch.all(cache["codes"][:, end:] == 0xA5)
    assert torch.all(cache["scales"][:, end:] == 0x5A) and torch.all(cache["prequant"][:, end:] == 7.0)
    ka, sa = g.state_export()
    kb, sb = h.state_export()
    assert torch.equal(ka, kb) and torch.equal(sa, sb)
    small = {k: v[:, :10].contiguous() for k, v in cache.items()}
    with pytest.raises(Exception, match="does not fit"):
        g.prefill_into(dev_bits(np.ascontiguousarray(x[:, :44])), small, start_pos=0)
    assert g.device_status() == 0


def test_flash_csa_chunked_prefill_full():
    """Flash CSA shapes: a prefill of 1001 tokens, then a chunk of 2000 starting mid-group
    (several token tiles), every entry against the oracle."""
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    g, o = make_pair(wl.seed, layer)
    x, *_ = layer_inputs(wl.seed, layer, 1, 3001)
    p0 = 0
    for n in (1001, 2000):
        xc = np.ascontiguousarray(x[:, p0:p0 + n])
        got = g.prefill(dev_bits(xc), start_pos=p0)
        torch.cuda.synchronize()
        ref = o.prefill(xc, start_pos=p0)
        check_entries(to_np(got), ref["prequant"], 1, f"Flash CSA chunk at {p0}")
        p0 += n
    check_state(g, o, "Flash CSA state after the chunks")


def test_hca_chunked_prefill():
    """HCA shapes (ratio 128): a chunk that completes no group, then one starting 74 tokens into a
    group and spanning three token tiles."""
    wl = synthetic.HCA
    layer = wl.layers[0]
    g, o = make_pair(wl.seed, layer, max_batch=2)
    x, *_ = layer_inputs(wl.seed, layer, 2, 1000)
    p0 = 0
    for n in (300, 30, 670):
        xc = np.ascontiguousarray(x[:, p0:p0 + n])
        got = g.prefill(dev_bits(xc), start_pos=p0)
        torch.cuda.synchronize()
        ref = o.prefill(xc, start_pos=p0)
        if ref["G"]:
            check_entries(to_np(got), ref["prequant"], 1, f"HCA chunk at {p0}")
        p0 += n
    check_state(g, o, "HCA state after the chunks")


@pytest.mark.parametrize("layer_idx,split", [(0, 65537), (1, 70000)])
def test_long_context_in_two_chunks_sampled(layer_idx, split):
    """The long-context workload (131072 tokens, 1 % outlier tokens) as a prefill and a chunk
    split mid-group: sampled entries of both calls against the oracle's groups of the whole
    sequence (a chunk gives the entries a whole prefill gives)."""
    from test_gpu_parity import sampled_groups
    wl = synthetic.LONG
    layer = wl.layers[layer_idx]
    N = 131072
    g, o = make_pair(wl.seed, layer)
    x, *_ = layer_inputs(wl.seed, layer, 1, N, outlier_frac=wl.outlier_frac)
    r = layer.ratio
    got = []
    for p0, p1 in ((0, split), (split, N)):
        out = g.prefill(dev_bits(np.ascontiguousarray(x[:, p0:p1])), start_pos=p0, prequant=True)
        torch.cuda.synchronize()
        got.append((p0 // r, to_np(out)))
    for gfirst, gn in got:
        G = gn["prequant"].shape[1]
        loc = sampled_groups(G, 12, gfirst)
        ref = o.prefill_groups(x[0], [gfirst + j for j in loc])
        check_entries({k: v[0][loc] for k, v in gn.items()}, ref["prequant"], 1, f"long chunk from group {gfirst}")
    assert g.device_status() == 0


@pytest.mark.parametrize("ratio,overlap", [(16, 0), (4, 1)])
def test_chunk_rewriting_decoded_positions_then_decode(ratio, overlap):
    """Decode steps, then a chunk that rewrites the last three decoded positions with other tokens,
    then decode again across the end of the group: the decode must pool the rewritten tokens (the
    running values it kept before the chunk summarise the old ones and may not be reused)."""
    layer = synthetic.Layer(256, 128, ratio, overlap, 1.0 / 16, gate_scale=2.0, rope_dim=64, fp4=1)
    B, p_start = 4, 2 * ratio + 5
    g, o = make_pair(19, layer, max_batch=B)
    x, *_ = layer_inputs(19, layer, B, 3 * ratio + 16)
    y, *_ = layer_inputs(29, layer, B, 3 * ratio + 16)  # the rewriting tokens
    xp = np.ascontiguousarray(x[:, :p_start])
    o.prefill(xp)
    g.prefill(dev_bits(xp), prequant=False)

    def decode(p, src):
        sp = np.full(B, p, np.int32)
        xt = np.ascontiguousarray(src[:, p])
        r = o.decode(xt, sp)
        d = g.decode(dev_bits(xt), torch.from_numpy(sp).to(DEV))
        em = d["emitted"].cpu().numpy()
        assert np.array_equal(em, r["emitted"]), p
        if em.any():
            check_entries(to_np(d, rows=np.flatnonzero(em)), r["prequant"][np.flatnonzero(em)], 1, f"decode at {p}")
        return int(em.sum())

    for p in range(p_start, p_start + 6):
        decode(p, x)
    p1 = p_start + 6
    yc = np.ascontiguousarray(y[:, p1 - 3:p1])
    ref = o.prefill(yc, start_pos=p1 - 3)
    got = g.prefill(dev_bits(yc), start_pos=p1 - 3)
    if ref["G"]:
        check_entries(to_np(got), ref["prequant"], 1, "rewriting chunk")
    emitted = sum(decode(p, x) for p in range(p1, p1 + ratio))
    assert emitted >= B  # the group completes within the steps
    check_state(g, o, "state after the chunk and the decode steps")
    assert g.device_status() == 0


@pytest.mark.parametrize("split", [1, 2])
def test_prefill_and_chunk_in_a_cuda_graph(split):
    """A prefill and a chunk continuing it, captured once in a CUDA graph after one eager pass (the
    library sets its kernel attributes, queries the device and sizes its scratch on first use) and
    replayed twice: the entries equal the eager pass's bit for bit and the oracle's within the
    parity tolerance, in both launch geometries."""
    layer = synthetic.Layer(256, 128, 4, 1, 1.0 / math.sqrt(256), gate_scale=2.0, rope_dim=64, fp4=1)
    B, N1, N2 = 2, 4 * 45 + 2, 4 * 20 + 3
    g, o = make_pair(29, layer, max_batch=B, split=split)
    x, *_ = layer_inputs(29, layer, B, N1 + N2)
    x1, x2 = (dev_bits(np.ascontiguousarray(x[:, a:b])) for a, b in ((0, N1), (N1, N1 + N2)))
    outs = [g._alloc_out(B * ((p + n) // 4 - p // 4), DEV, prequant=True) for p, n in ((0, N1), (N1, N2))]

    def run():
        g.prefill(x1, start_pos=0, out=outs[0])
        g.prefill(x2, start_pos=N1, out=outs[1])

    run()
    torch.cuda.synchronize()
    eager = [to_np(ob) for ob in outs]
    for ob in outs:
        for t in ob.values():
            t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for k, ob in enumerate(outs):
        got = to_np(ob)
        for key in eager[k]:
            assert np.array_equal(got[key], eager[k][key]), (k, key)
    r1 = o.prefill(np.ascontiguousarray(x[:, :N1]))
    r2 = o.prefill(np.ascontiguousarray(x[:, N1:]), start_pos=N1)
    check_entries(to_np(outs[0]), r1["prequant"], 1, "graph prefill")
    check_entries(to_np(outs[1]), r2["prequant"], 1, "graph chunk")
    assert g.device_status() == 0

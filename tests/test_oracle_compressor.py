"""Pins of the oracle's compressor against what the pages and the mathematics fix.

- pooling: closed forms (equal scores give the mean, one dominant score selects), the
  weights sum to one, padded candidates count for nothing, order within a group does not
  matter, and torch's own float64 softmax in the pages' reshape form ("Pool token pairs");
- projection: numpy's float64 matmul ("linear_f32": x . w^T, w [out, in]);
- ratio 1 reduces to projection + RMSNorm ("Pool token pairs" Compressor excerpt);
- the ratio-4 worked example (16 tokens -> 4 entries -> 32 candidate uses);
- prefill equals token-by-token decode ("Prefill and decode use the same rule");
- RMSNorm closed forms; YaRN RoPE: factor 1 is textbook RoPE, the ramp follows the
  rotation counts, position 0 is the identity, the rotation keeps pair norms and turns
  each pair by pos * f_i.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from _util import bf16_bits_to_f32, layer_inputs, to_bf16_bits, ulp_distance_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make(dim, H, ratio, overlap, rope_dim=0, fp4=0, max_batch=1, seed=0, gate_scale=1.0, eps=1e-6):
    c = oracle.Compressor(dim, H, ratio, overlap, max_batch=max_batch, rope_dim=rope_dim, fp4=fp4, eps=eps)
    layer = synthetic.Layer(dim, H, ratio, overlap, 1.0 / math.sqrt(dim), gate_scale=gate_scale)
    wkv, wgate, gain = synthetic.weights(seed, layer)
    c.set_weights(wkv, wgate, gain)
    return c, (wkv, wgate, gain)


def rand_x(seed, B, N, dim):
    return to_bf16_bits(np.stack([synthetic.tokens(seed, b, 0, N, dim) for b in range(B)]))


# ---- pooling ------------------------------------------------------------------------------

def test_pool_weights_sum_to_one_and_match_torch_softmax():
    rng = np.random.default_rng(0)
    for n in (1, 2, 4, 8, 128):
        kv = rng.standard_normal((n, 24)).astype(np.float32)
        sc = (rng.standard_normal((n, 24)) * 3).astype(np.float32)
        out, w = oracle.pool(kv, sc)
        assert np.allclose(w.sum(0), 1.0, rtol=0, atol=1e-14)
        ref_w = torch.softmax(torch.from_numpy(sc).double(), dim=0)
        ref = (torch.from_numpy(kv).double() * ref_w).sum(0).float().numpy()
        assert np.allclose(w, ref_w.numpy(), rtol=1e-13, atol=1e-15)
        assert np.array_equal(out, ref) or np.max(np.abs(out - ref) / np.abs(ref)) < 2e-7


def test_pool_equal_scores_give_the_mean():
    rng = np.random.default_rng(1)
    kv = rng.standard_normal((8, 40)).astype(np.float32)
    sc = np.full((8, 40), 0.7, np.float32)
    out, w = oracle.pool(kv, sc)
    assert np.all(w == 1.0 / 8)
    assert np.array_equal(out, kv.astype(np.float64).mean(0).astype(np.float32))


def test_pool_dominant_score_selects_and_padded_slots_count_for_nothing():
    rng = np.random.default_rng(2)
    kv = rng.standard_normal((8, 16)).astype(np.float32)
    sc = rng.standard_normal((8, 16)).astype(np.float32)
    sc[5, :] += 1.0e4
    out, _ = oracle.pool(kv, sc)
    assert np.array_equal(out, kv[5])
    sc2 = rng.standard_normal((8, 16)).astype(np.float32)
    sc2[:4] = -np.inf
    kv2 = kv.copy()
    kv2[:4] = 0.0
    a, w = oracle.pool(kv2, sc2)
    b, _ = oracle.pool(kv[4:], sc2[4:])
    assert np.array_equal(a, b) and np.all(w[:4] == 0.0)


def test_pool_is_symmetric_in_candidate_order():
    rng = np.random.default_rng(3)
    kv = rng.standard_normal((8, 16)).astype(np.float32)
    sc = rng.standard_normal((8, 16)).astype(np.float32)
    a, _ = oracle.pool(kv, sc)
    perm = rng.permutation(8)
    b, _ = oracle.pool(kv[perm], sc[perm])
    assert np.max(np.abs(a - b)) <= 1e-6 * np.max(np.abs(a))


# ---- projection ---------------------------------------------------------------------------

def test_linear_matches_float64_matmul():
    x = rand_x(5, 1, 37, 96)[0]
    w = synthetic.normal(5, 2, 0, 0, 80 * 96, 0.0, 0.1).reshape(80, 96)
    got = oracle.linear(x, w, nthreads=2)
    ref = (bf16_bits_to_f32(x).astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1 and np.mean(ulps == 0) > 0.999


# ---- torch float64 restatement of the pages' reshape form, for brute force on tiny shapes ---

def torch_reference_prequant(x_bits, wkv, wgate, gain, ratio, overlap, eps=1e-6):
    """[B, N, dim] -> pre-RoPE latent as float64 (before the final bf16 rounding).

    Follows "Pool token pairs": kv, score = wkv(x.float()), wgate(x.float()); unflatten(1, (-1, r));
    (kv * score.softmax(dim=2)).sum(dim=2); then norm(kv.to(bf16)).  At ratio 4 overlapped the
    candidates are [previous group's branch B, current group's branch A] ("Compressed Sparse
    Attention - ratio m = 4", overlap transform), the first entry's previous branch padded."""
    x = torch.from_numpy(bf16_bits_to_f32(x_bits)).double()
    kv = (x @ torch.from_numpy(wkv).double().T).float().double()
    sc = (x @ torch.from_numpy(wgate).double().T).float().double()
    B, N, _ = x.shape
    G = N // ratio
    kv, sc = kv[:, :G * ratio], sc[:, :G * ratio]
    if overlap:
        H = wkv.shape[0] // 2
        kv = kv.unflatten(1, (G, 4))
        sc = sc.unflatten(1, (G, 4))
        kvA, kvB = kv[..., :H], kv[..., H:]
        scA, scB = sc[..., :H], sc[..., H:]
        padk = torch.zeros_like(kvB[:, :1])
        pads = torch.full_like(scB[:, :1], -math.inf)
        kv = torch.cat([torch.cat([padk, kvB[:, :-1]], 1), kvA], 2)
        sc = torch.cat([torch.cat([pads, scB[:, :-1]], 1), scA], 2)
    else:
        kv = kv.unflatten(1, (G, ratio))
        sc = sc.unflatten(1, (G, ratio))
    pooled = (kv * sc.softmax(dim=2)).sum(dim=2).float()
    u = pooled.to(torch.bfloat16).double()
    g = torch.from_numpy(gain).double()
    return u * torch.rsqrt(u.pow(2).mean(-1, keepdim=True) + eps) * g


def assert_correctly_rounded(bits, exact):
    """Each bf16 value is the rounding of the float64 value: within half an ulp (+ float64 noise)."""
    got = bf16_bits_to_f32(bits).astype(np.float64)
    exact = np.asarray(exact, np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(got - exact) <= 0.5 * ulp * (1 + 1e-9) + 1e-300), np.max(np.abs(got - exact) / ulp)


@pytest.mark.parametrize("ratio,overlap,N", [(2, 0, 20), (3, 0, 17), (4, 0, 22), (4, 1, 16), (4, 1, 27),
                                             (8, 0, 40), (1, 0, 9)])
def test_bruteforce_against_reshape_form(ratio, overlap, N):
    dim, H = 48, 32
    c, (wkv, wgate, gain) = make(dim, H, ratio, overlap, max_batch=2, seed=ratio + overlap)
    x = rand_x(11, 2, N, dim)
    out = c.prefill(x, nthreads=2)
    assert out["G"] == N // ratio
    ref = torch_reference_prequant(x, wkv, wgate, gain, ratio, overlap).numpy()
    assert_correctly_rounded(out["prequant"], ref)
    assert np.array_equal(out["latent"], out["prequant"])  # fp4 off


def test_ratio_one_is_projection_plus_norm():
    dim, H = 64, 32
    c, (wkv, _, gain) = make(dim, H, 1, 0)
    x = rand_x(12, 1, 13, dim)
    out = c.prefill(x)
    kv = (bf16_bits_to_f32(x[0]).astype(np.float64) @ wkv.astype(np.float64).T).astype(np.float32)
    u = bf16_bits_to_f32(to_bf16_bits(kv)).astype(np.float64)
    y = u / np.sqrt((u * u).mean(-1, keepdims=True) + 1e-6) * gain
    assert out["G"] == 13
    assert_correctly_rounded(out["prequant"][0], y)


def test_worked_example_ratio4_overlap():
    with open(os.path.join(GOLDEN, "csa4_worked_example.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    N, r, entries, uses = map(int, rows[0])
    dim, H = 32, 16
    c = oracle.Compressor(dim, H, r, 1, rope_dim=0, fp4=0)
    wkv = synthetic.normal(7, 2, 0, 0, 2 * H * dim, 0.0, 0.2).reshape(2 * H, dim)
    c.set_weights(wkv, np.zeros_like(wkv), np.ones(H, np.float32))  # zero gate: equal scores
    x = rand_x(13, 1, N, dim)
    out = c.prefill(x)
    assert out["G"] == entries and 8 * out["G"] == uses
    kv = (bf16_bits_to_f32(x[0]).astype(np.float64) @ wkv.astype(np.float64).T).astype(np.float32)
    A, Bh = kv[:, :H].astype(np.float64), kv[:, H:].astype(np.float64)
    for j in range(entries):
        # equal scores: the mean of the live candidates; the padded slots of entry 0 count for nothing
        cands = A[4 * j:4 * j + 4] if j == 0 else np.concatenate([Bh[4 * j - 4:4 * j], A[4 * j:4 * j + 4]])
        m = cands.mean(0).astype(np.float32)
        u = bf16_bits_to_f32(to_bf16_bits(m)).astype(np.float64)
        y = u / np.sqrt((u * u).mean() + 1e-6)
        assert_correctly_rounded(out["prequant"][0, j], y)


# ---- prefill == decode ----------------------------------------------------------------------

@pytest.mark.parametrize("ratio,overlap,N,rope,fp4", [(2, 0, 64, 0, 0), (4, 1, 37, 16, 1), (4, 1, 3, 16, 1),
                                                      (3, 0, 29, 16, 1), (1, 0, 6, 16, 1), (16, 0, 50, 16, 1),
                                                      (4, 1, 21, 16, 2)])
def test_prefill_equals_token_by_token_decode(ratio, overlap, N, rope, fp4):
    dim, H = 64, 32
    B = 2
    pre, _ = make(dim, H, ratio, overlap, rope_dim=rope, fp4=fp4, max_batch=B, seed=3)
    dec, _ = make(dim, H, ratio, overlap, rope_dim=rope, fp4=fp4, max_batch=B, seed=3)
    x = rand_x(14, B, N, dim)
    full = pre.prefill(x, nthreads=2)
    got = {b: [] for b in range(B)}
    for p in range(N):
        o = dec.decode(x[:, p], np.full(B, p, np.int32), nthreads=2)
        for b in range(B):
            assert o["emitted"][b] == ((p + 1) % ratio == 0)
            if o["emitted"][b]:
                got[b].append((o["latent"][b].copy(), o["codes"][b].copy(), o["scales"][b].copy(),
                               o["prequant"][b].copy()))
    for b in range(B):
        assert len(got[b]) == full["G"]
        for j, (lat, cd, sc, pq) in enumerate(got[b]):
            assert np.array_equal(lat, full["latent"][b, j])
            assert np.array_equal(pq, full["prequant"][b, j])
            if fp4:
                assert np.array_equal(cd, full["codes"][b, j]) and np.array_equal(sc, full["scales"][b, j])
    # the state holds the same unfinished group (and, overlapped, the previous group's tokens)
    kp, sp = pre.state()
    kd, sd = dec.state()
    G, rem = N // ratio, N % ratio
    if overlap:
        q = G % 2
        assert np.array_equal(kp[:, q, :rem], kd[:, q, :rem]) and np.array_equal(sp[:, q, :rem], sd[:, q, :rem])
        if G >= 1:
            assert np.array_equal(kp[:, 1 - q], kd[:, 1 - q]) and np.array_equal(sp[:, 1 - q], sd[:, 1 - q])
        else:
            assert np.all(sp[:, 1, :, 32:] == -np.inf) and np.all(sd[:, 1, :, 32:] == -np.inf)
    else:
        assert np.array_equal(kp[:, :rem], kd[:, :rem]) and np.array_equal(sp[:, :rem], sd[:, :rem])


def live_state_equal(ka, sa, kb, sb, ratio, overlap, P, H):
    """The state slots a later call can still read after P tokens: non-overlapped the
    unfinished group's slots; overlapped also the last complete group's parity."""
    if overlap:
        q, rem = (P // 4) % 2, P % 4
        ok = np.array_equal(ka[:, q, :rem], kb[:, q, :rem]) and np.array_equal(sa[:, q, :rem], sb[:, q, :rem])
        if P >= 4:
            return ok and np.array_equal(ka[:, 1 - q], kb[:, 1 - q]) and np.array_equal(sa[:, 1 - q], sb[:, 1 - q])
        return ok and np.all(sa[:, 1, :, H:] == -np.inf) and np.all(sb[:, 1, :, H:] == -np.inf)
    rem = P % ratio
    return np.array_equal(ka[:, :rem], kb[:, :rem]) and np.array_equal(sa[:, :rem], sb[:, :rem])


# chunk lengths: the first call is a prefill at position 0, the others continue at the position
# the previous one reached (mid-group, group-aligned, chunks that complete no group, p < ratio)
CHUNKS = [(4, 1, (5, 2, 9, 1, 7)), (4, 1, (2, 1, 13, 4)), (3, 0, (4, 5, 1, 11)), (16, 0, (7, 20, 3, 40)),
          (1, 0, (3, 4)), (2, 0, (1, 1, 1, 5))]


@pytest.mark.parametrize("ratio,overlap,chunks", CHUNKS)
def test_prefill_chunks_equal_token_by_token_decode(ratio, overlap, chunks):
    dim, H, B = 64, 32, 2
    chk, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=B, seed=5)
    dec, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=B, seed=5)
    P = sum(chunks)
    x = rand_x(18, B, P, dim)
    want = {b: [] for b in range(B)}
    for p in range(P):
        o = dec.decode(x[:, p], np.full(B, p, np.int32), nthreads=2)
        for b in range(B):
            if o["emitted"][b]:
                want[b].append({k: o[k][b].copy() for k in ("latent", "codes", "scales", "prequant")})
    got = {b: [] for b in range(B)}
    p0 = 0
    for n in chunks:
        out = chk.prefill(x[:, p0:p0 + n], start_pos=p0, nthreads=2)
        assert out["G"] == (p0 + n) // ratio - p0 // ratio
        for b in range(B):
            for j in range(out["G"]):
                got[b].append({k: out[k][b, j] for k in ("latent", "codes", "scales", "prequant")})
        p0 += n
    for b in range(B):
        assert len(got[b]) == len(want[b]) == P // ratio
        for g, w in zip(got[b], want[b]):
            for k in w:
                assert np.array_equal(g[k], w[k]), k
    kc, sc = chk.state()
    kd, sd = dec.state()
    assert live_state_equal(kc, sc, kd, sd, ratio, overlap, P, H)


@pytest.mark.parametrize("ratio,overlap", [(4, 1), (8, 0)])
def test_prefill_then_chunks_equal_one_prefill(ratio, overlap):
    dim, H = 64, 32
    one, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=3, seed=6)
    parts, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=3, seed=6)
    x = rand_x(19, 2, 11 * ratio + 3, dim)
    full = one.prefill(x, slot_offset=1)
    got = []
    p0 = 0
    for n in (2 * ratio + 1, 5 * ratio - 2, 4 * ratio + 4):
        got.append(parts.prefill(x[:, p0:p0 + n], slot_offset=1, start_pos=p0)["latent"])
        p0 += n
    assert np.array_equal(np.concatenate(got, axis=1), full["latent"])
    ka, sa = one.state()
    kb, sb = parts.state()
    assert live_state_equal(ka[1:], sa[1:], kb[1:], sb[1:], ratio, overlap, p0, H)
    assert np.all(ka[0] == 0) and np.all(kb[0] == 0) and np.all(sb[0] == -np.inf)  # slot 0 untouched


def test_prefill_chunk_reads_its_own_slots():
    dim, H, r = 32, 16, 4
    c, _ = make(dim, H, r, 1, rope_dim=16, fp4=1, max_batch=3, seed=7)
    x = rand_x(20, 3, 14, dim)
    c.prefill(x[:, :6])  # three different histories
    first = c.prefill(x[:, 6:], start_pos=6)
    d, _ = make(dim, H, r, 1, rope_dim=16, fp4=1, max_batch=3, seed=7)
    d.prefill(x[1:2, :6], slot_offset=2)
    second = d.prefill(x[1:2, 6:], slot_offset=2, start_pos=6)
    assert np.array_equal(first["latent"][1], second["latent"][0])
    assert not np.array_equal(first["latent"][0], first["latent"][1])


def test_indexer_quantiser_applies_to_the_prequant_latent():
    """fp4 = 2 (the indexer's keys): the latent is the e8m0 / block-32 round trip of prequant,
    one scale per 32 features."""
    c, _ = make(64, 64, 4, 1, rope_dim=16, fp4=2)
    out = c.prefill(rand_x(21, 1, 4 * 9 + 1, 64))
    codes, scales, lat = oracle.fp4_e8m0(out["prequant"])
    assert out["scales"].shape == (1, 9, 2)
    assert np.array_equal(out["scales"].reshape(-1), scales) and np.array_equal(out["codes"].reshape(-1), codes)
    assert np.array_equal(out["latent"].reshape(-1), lat)


# ---- gate positional bias ([CSA4] "wgate(x) + positional bias") ------------------------------

@pytest.mark.parametrize("ratio,overlap,s0", [(4, 0, 2), (4, 1, 1), (8, 0, 7)])
def test_gate_bias_on_one_slot_selects_that_token(ratio, overlap, s0):
    """A bias of 1000 on one position of the group (branch A when overlapped) gives that token
    softmax weight 1 (the others exp(-1000) = 0), so each entry is the epilogue of that token's
    kv row, computed here from numpy's float64 projection rounded to float32."""
    dim, H = 64, 32
    c, (wkv, _, _) = make(dim, H, ratio, overlap, rope_dim=16)
    ape = np.zeros((ratio, (1 + overlap) * H), np.float32)
    ape[s0, :H] = 1000.0
    c.set_gate_bias(ape)
    x = rand_x(22, 1, 5 * ratio + 1, dim)
    out = c.prefill(x)
    xf = bf16_bits_to_f32(x[0]).astype(np.float64)
    for j in range(5):
        kv = (xf[ratio * j + s0] @ wkv.astype(np.float64).T).astype(np.float32)[:H]
        assert np.array_equal(out["prequant"][0, j], c.epilogue(kv, ratio * j)), j


@pytest.mark.parametrize("ratio,overlap", [(4, 1), (3, 0)])
def test_gate_bias_constant_per_feature_changes_nothing(ratio, overlap):
    """The softmax is unchanged by adding one constant to every candidate's logit: a bias that
    depends only on the feature (same for every position and both branches) leaves the entries
    as they are, up to the float32 rounding of the shifted logits."""
    dim, H = 64, 32
    a, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=2)
    b, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=2)
    cf = np.random.default_rng(5).standard_normal(H).astype(np.float32) * 3
    b.set_gate_bias(np.tile(np.concatenate([cf] * (1 + overlap)), (ratio, 1)))
    x = rand_x(23, 2, 40 * ratio + 2, dim)
    pa, pb = a.prefill(x)["prequant"], b.prefill(x)["prequant"]
    u = ulp_distance_bf16(pa, pb)
    assert u.max() <= 1 and np.mean(u == 0) >= 0.99


@pytest.mark.parametrize("ratio,overlap,chunks", [(4, 1, (6, 5, 13)), (3, 0, (4, 8, 1, 9))])
def test_gate_bias_prefill_chunks_equal_decode(ratio, overlap, chunks):
    """With a random bias, prefill chunks still equal token-by-token decode, bit for bit: both
    add the bias of the token's position within its group."""
    dim, H, B = 64, 32, 2
    ape = np.random.default_rng(6).standard_normal((ratio, (1 + overlap) * H)).astype(np.float32)
    chk, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=B, seed=8)
    dec, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=B, seed=8)
    chk.set_gate_bias(ape)
    dec.set_gate_bias(ape)
    P = sum(chunks)
    x = rand_x(24, B, P, dim)
    want = []
    for p in range(P):
        o = dec.decode(x[:, p], np.full(B, p, np.int32))
        if o["emitted"][0]:
            want.append(o["latent"].copy())
    got = []
    p0 = 0
    for n in chunks:
        out = chk.prefill(x[:, p0:p0 + n], start_pos=p0)
        got += [out["latent"][:, j] for j in range(out["G"])]
        p0 += n
    assert len(got) == len(want) == P // ratio
    for g, w in zip(got, want):
        assert np.array_equal(g, w)
    # the bias matters: without it the entries differ
    plain, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1, max_batch=B, seed=8)
    assert not np.array_equal(plain.prefill(x)["latent"][:, 0], got[0])


def test_prefill_state_holds_the_tail_projections():
    dim, H, r = 48, 16, 8
    c, (wkv, wgate, _) = make(dim, H, r, 0, max_batch=3)
    x = rand_x(15, 2, 2 * r + 5, dim)
    c.prefill(x, slot_offset=1)
    kv, sc = c.state()
    for b in range(2):
        tail = bf16_bits_to_f32(x[b, 2 * r:]).astype(np.float64)
        assert np.allclose(kv[1 + b, :5], tail @ wkv.astype(np.float64).T, rtol=1e-6, atol=1e-6)
        assert np.allclose(sc[1 + b, :5], tail @ wgate.astype(np.float64).T, rtol=1e-6, atol=1e-6)
    assert np.all(kv[0] == 0) and np.all(sc[0] == -np.inf)  # slot 0 untouched


def test_empty_calls_are_rejected_and_change_nothing():
    """Empty batches and zero-token prefills are argument errors (the library's ABI returns
    CSA_ERR_ARG for the same calls); the state keeps what an earlier prefill left."""
    dim, H, r = 32, 16, 4
    c, _ = make(dim, H, r, 1, max_batch=2)
    c.prefill(rand_x(17, 2, 2 * r + 3, dim))
    kv0, sc0 = (a.copy() for a in c.state())
    with pytest.raises(ValueError):
        c.prefill(np.zeros((2, 0, dim), np.uint16))
    with pytest.raises(ValueError):
        c.prefill(np.zeros((0, 5, dim), np.uint16))
    with pytest.raises(ValueError):
        c.decode(np.zeros((0, dim), np.uint16), np.zeros(0, np.int32))
    kv1, sc1 = c.state()
    assert np.array_equal(kv0, kv1) and np.array_equal(sc0, sc1)


def test_decode_emission_timing_per_sequence():
    dim, H, r = 32, 16, 4
    c, _ = make(dim, H, r, 1, max_batch=6)
    sp = np.array([1, 2, 3, 7, 8, 11], np.int32)
    x = rand_x(16, 6, 1, dim)[:, 0]
    o = c.decode(x, sp)
    assert list(o["emitted"]) == [int((p + 1) % r == 0) for p in sp] and o["n"] == 3


def test_prefill_groups_match_full_prefill():
    dim, H = 64, 32
    for ratio, overlap in ((4, 1), (8, 0)):
        c, _ = make(dim, H, ratio, overlap, rope_dim=16, fp4=1)
        x = rand_x(17, 1, 8 * ratio + 3, dim)
        full = c.prefill(x)
        groups = [0, 3, 7, 1]
        part = c.prefill_groups(x[0], groups)
        for k in ("latent", "prequant", "codes", "scales"):
            assert np.array_equal(part[k], full[k][0, groups])


# ---- RMSNorm --------------------------------------------------------------------------------

def test_rmsnorm_closed_forms():
    H = 64
    c = oracle.Compressor(64, H, 2, 0, rope_dim=0, fp4=0)
    gain = synthetic.normal(0, 4, 0, 0, H, 1.0, 0.02)
    c.set_weights(np.zeros((H, 64), np.float32), np.zeros((H, 64), np.float32), gain)
    # constant input c: y = c g / sqrt(c^2 + eps)
    for cval in (3.0, -0.5, 1e-3, 1e-4):
        y = bf16_bits_to_f32(c.epilogue(np.full(H, cval, np.float32), 0)).astype(np.float64)
        u = float(bf16_bits_to_f32(to_bf16_bits(np.array([cval], np.float32)))[0])
        expect = u * gain.astype(np.float64) / math.sqrt(u * u + 1e-6)
        assert np.all(np.abs(y - expect) <= np.abs(expect) * 2.0 ** -8)
    # unit gain: the output's RMS is one
    c.set_weights(np.zeros((H, 64), np.float32), np.zeros((H, 64), np.float32), np.ones(H, np.float32))
    v = synthetic.normal(9, 1, 0, 0, H, 0.0, 5.0)
    y = bf16_bits_to_f32(c.epilogue(v, 0)).astype(np.float64)
    assert abs(math.sqrt((y * y).mean()) - 1.0) < 4e-3


# ---- YaRN RoPE ----------------------------------------------------------------------------

def test_yarn_factor_one_is_textbook_rope():
    f = oracle.yarn_freqs(64, 10000.0, 1.0, 4096)
    ref = 10000.0 ** (-np.arange(0, 64, 2) / 64.0)
    assert np.allclose(f, ref, rtol=1e-14, atol=0)


def test_yarn_ramp_follows_rotation_counts():
    d, base, factor, L = 64, 160000.0, 16.0, 4096
    f = oracle.yarn_freqs(d, base, factor, L, 32.0, 1.0)
    f0 = base ** (-np.arange(0, d, 2) / d)
    ratio = f / f0
    rotations = L * f0 / (2 * math.pi)  # turns each pair makes over the original context
    assert np.all(np.diff(ratio) <= 1e-15)  # monotone: faster dims keep more of their frequency
    assert np.allclose(ratio[rotations > 32.0], 1.0, rtol=1e-14)  # more than beta_fast turns: kept
    assert np.allclose(ratio[rotations < 1.0], 1.0 / factor, rtol=1e-14)  # fewer than beta_slow: interpolated
    mid = (rotations < 32.0) & (rotations > 1.0)
    assert np.all((ratio[mid] < 1.0) & (ratio[mid] > 1.0 / factor))
    # for the Flash compressor (theta 160000, factor 16, original length 4096) the ramp runs
    # from dim 8 (32.6 turns) to dim 18 (0.77 turns)
    assert oracle.yarn_bounds(d, base, L, 32.0, 1.0) == (8.0, 18.0)


def _rope_pair_views(pos, rope_dim=16, H=32):
    c0 = oracle.Compressor(64, H, 2, 0, rope_dim=0, fp4=0)
    c1 = oracle.Compressor(64, H, 2, 0, rope_dim=rope_dim, fp4=0)
    gain = np.ones(H, np.float32)
    for c in (c0, c1):
        c.set_weights(np.zeros((H, 64), np.float32), np.zeros((H, 64), np.float32), gain)
    v = synthetic.normal(21, 1, 0, 0, H, 0.0, 1.0)
    y0 = bf16_bits_to_f32(c0.epilogue(v, pos)).astype(np.float64)
    y1 = bf16_bits_to_f32(c1.epilogue(v, pos)).astype(np.float64)
    return y0, y1


def test_rope_position_zero_is_identity():
    y0, y1 = _rope_pair_views(0)
    assert np.array_equal(y0, y1)


@pytest.mark.parametrize("pos", [1, 4, 4096, 131068])
def test_rope_rotates_pairs_by_pos_times_freq(pos):
    rd, H = 16, 32
    y0, y1 = _rope_pair_views(pos, rd, H)
    assert np.array_equal(y0[:H - rd], y1[:H - rd])  # features before the rotary slice untouched
    f = oracle.yarn_freqs(rd, 160000.0, 16.0, 4096)
    a, b = y0[H - rd::2], y0[H - rd + 1::2]
    a1, b1 = y1[H - rd::2], y1[H - rd + 1::2]
    r0, r1 = np.hypot(a, b), np.hypot(a1, b1)
    assert np.all(np.abs(r1 - r0) <= r0 * 2.0 ** -7)
    turn = np.angle((a1 + 1j * b1) / (a + 1j * b))  # counter-clockwise by +theta
    want = np.angle(np.exp(1j * pos * f))
    err = np.abs(np.angle(np.exp(1j * (turn - want))))
    assert np.all(err <= 2.0 ** -6), (turn, want)

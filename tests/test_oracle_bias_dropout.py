"""Pins for the oracle's attention bias, dbias and dropout (CPU, fp64).

The bias follows TransformerEngine PR #446 (review of ck_fused_attn_bwd.cpp:
bias of shape (bias_b, bias_h, s_q, s_kv) in the BiasShape kinds 11SS, 1HSS,
BHSS, B1SS; dbias in the BHSS shape); dropout is driven by a philox seed and
offset (the philox_seed_ptr / philox_offset_ptr pair of the same page).  The
checks:

* Philox: the oracle's generator at W = 64 reproduces numpy's Philox4x64-10
  bit generator word for word (the same code at W = 32 makes the dropout
  mask); keep rates and independence of the mask by statistics;
* bias: torch's scaled_dot_product_attention with the bias as a float
  attn_mask (forward, and autograd for dQ, dK, dV and the bias gradient, the
  broadcast shapes summed), central finite differences of dbias, and the
  softmax's invariance to a per-row shift of the bias;
* dropout: central finite differences with the mask held fixed, p = 0 equal to
  no dropout, and E[O] over seeds equal to the undropped O (the 1 / (1 - p)
  scaling).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attn_ref as R

F64 = torch.float64


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64)


def fd_grad(x, f, h=1e-6):
    g = torch.zeros_like(x)
    flat, gflat = x.view(-1), g.view(-1)
    for i in range(flat.numel()):
        x0 = flat[i].item()
        flat[i] = x0 + h
        fp = f()
        flat[i] = x0 - h
        fm = f()
        flat[i] = x0
        gflat[i] = (fp - fm) / (2 * h)
    return g


def rel_err(a, b):
    return float((a - b).abs().max() / max(float(b.abs().max()), 1e-300))


# ------------------------------------------------------------------ Philox

@pytest.mark.parametrize("seed", [1, 2, 3])
def test_philox64_matches_numpy_bit_generator(seed):
    rng = np.random.default_rng(seed)
    for _ in range(8):
        ctr = [int(x) for x in rng.integers(0, 2**63, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2**63, size=2, dtype=np.uint64)]
        bg = np.random.Philox(key=0)
        st = bg.state
        st["state"]["counter"] = np.array(ctr, dtype=np.uint64)
        st["state"]["key"] = np.array(key, dtype=np.uint64)
        st["buffer_pos"] = 4          # the next draw increments the counter, then runs the rounds
        bg.state = st
        want = [int(x) for x in bg.random_raw(4)]
        ctr1 = ctr[:]
        ctr1[0] = (ctr1[0] + 1) & (2**64 - 1)
        assert list(R.philox(ctr1, key, 64)) == want


def test_philox32_vectorised_equals_scalar():
    ctr = [np.array([0, 5, 2**32 - 1], dtype=np.uint64), np.array([7, 0, 3], dtype=np.uint64),
           np.array([1, 2**31, 9], dtype=np.uint64), np.array([0, 1, 2**32 - 2], dtype=np.uint64)]
    key = (np.uint64(0x12345678), np.uint64(0x9ABCDEF0))
    vec = R.philox(ctr, key, 32)
    for n in range(3):
        sc = R.philox([int(c[n]) for c in ctr], [int(key[0]), int(key[1])], 32)
        assert [int(w[n]) for w in vec] == list(sc)


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_dropout_keep_rate(p):
    keep = R.dropout_keep(256, 256, 3, p, seed=1234, offset=77)
    n = keep.numel()
    frac = float(keep.double().mean())
    sigma = math.sqrt(p * (1 - p) / n)
    assert abs(frac - (1 - p)) < 5 * sigma


def test_dropout_masks_independent_across_heads_offsets_and_seeds():
    base = R.dropout_keep(64, 64, 5, 0.5, seed=9, offset=0)
    for other in (R.dropout_keep(64, 64, 6, 0.5, seed=9, offset=0),
                  R.dropout_keep(64, 64, 5, 0.5, seed=10, offset=0),
                  R.dropout_keep(64, 64, 5, 0.5, seed=9, offset=1000)):
        agree = float((base == other).double().mean())
        assert abs(agree - 0.5) < 5 * math.sqrt(0.25 / base.numel())
    # the same (head, seed, offset) gives the same mask; rows i and i + 4 use
    # counters one apart, so an offset of 1 shifts the rows by 4
    assert torch.equal(base, R.dropout_keep(64, 64, 5, 0.5, seed=9, offset=0))
    shifted = R.dropout_keep(64, 64, 5, 0.5, seed=9, offset=1)
    assert torch.equal(shifted[:60], base[4:])


# -------------------------------------------------------------------- bias

BIAS_SHAPES = {"11SS": (1, 1), "1HSS": (1, None), "BHSS": (None, None), "B1SS": (None, 1)}


def _bias(kind, B, H, sq, sk, seed):
    bb, bh = BIAS_SHAPES[kind]
    return rnd((bb or B, bh or H, sq, sk), seed)


@pytest.mark.parametrize("kind", sorted(BIAS_SHAPES))
@pytest.mark.parametrize("mask", [0, 1, 3])
def test_bias_matches_sdpa_float_mask_and_autograd(kind, mask):
    F = torch.nn.functional
    B, sq, sk, hq, hkv, d, dv_ = 2, 7, 9, 4, 2, 8, 5
    left, right = (3, 1) if mask == 3 else (-1, -1)
    q, k, v, do = rnd((B, sq, hq, d), 61), rnd((B, sk, hkv, d), 62), rnd((B, sk, hkv, dv_), 63), rnd((B, sq, hq, dv_), 64)
    bias = _bias(kind, B, hq, sq, sk, 65)
    vis = R.visible(sq, sk, mask, left, right)
    qt, kt, vt = (x.permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    bt = bias.clone().requires_grad_(True)
    additive = bt.masked_fill(~vis, -math.inf)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=additive, scale=0.45, enable_gqa=True)
    ref.backward(do.permute(0, 2, 1, 3))
    kw = dict(mask=mask, left=left, right=right, bias=bias)
    o, lse = R.attn_forward(q, k, v, 0.45, **kw)
    assert torch.allclose(o, ref.detach().permute(0, 2, 1, 3), atol=1e-12)
    dq, dk, dv, dbias = R.attn_backward(q, k, v, o, do, lse, 0.45, return_dbias=True, **kw)
    assert torch.allclose(dq, qt.grad.permute(0, 2, 1, 3), atol=1e-12)
    assert torch.allclose(dk, kt.grad.permute(0, 2, 1, 3), atol=1e-12)
    assert torch.allclose(dv, vt.grad.permute(0, 2, 1, 3), atol=1e-12)
    # dbias comes in the full [B, Hq, Sq, Sk] shape; the gradient of a
    # broadcast bias is its sum over the broadcast dimensions
    assert dbias.shape == (B, hq, sq, sk)
    red = dbias.sum(dim=0, keepdim=True) if bias.shape[0] == 1 else dbias
    red = red.sum(dim=1, keepdim=True) if bias.shape[1] == 1 else red
    assert torch.allclose(red, bt.grad, atol=1e-12)


def test_dbias_finite_differences():
    B, sq, sk, hq, hkv, d = 1, 5, 6, 2, 1, 4
    q, k, v, do = rnd((B, sq, hq, d), 71), rnd((B, sk, hkv, d), 72), rnd((B, sk, hkv, d), 73), rnd((B, sq, hq, d), 74)
    bias = rnd((B, hq, sq, sk), 75)
    kw = dict(mask=2, bias=bias)

    def L():
        o, _ = R.attn_forward(q, k, v, 0.7, **kw)
        return float((o * do).sum())

    o, lse = R.attn_forward(q, k, v, 0.7, **kw)
    *_, dbias = R.attn_backward(q, k, v, o, do, lse, 0.7, return_dbias=True, **kw)
    assert rel_err(dbias, fd_grad(bias, L)) < 1e-6


def test_bias_row_shift_invariance():
    """Adding a constant per query row to the bias leaves O, dQ, dK, dV and
    dbias unchanged (the softmax is shift-invariant per row)."""
    B, sq, sk, hq, d = 1, 8, 8, 2, 8
    q, k, v, do = rnd((B, sq, hq, d), 81), rnd((B, sk, hq, d), 82), rnd((B, sk, hq, d), 83), rnd((B, sq, hq, d), 84)
    bias = rnd((1, hq, sq, sk), 85)
    shift = rnd((1, hq, sq, 1), 86) * 5
    outs = []
    for b in (bias, bias + shift):
        o, lse = R.attn_forward(q, k, v, 0.3, mask=1, bias=b)
        outs.append((o,) + R.attn_backward(q, k, v, o, do, lse, 0.3, mask=1, bias=b, return_dbias=True))
    for a, b in zip(*outs):
        assert torch.allclose(a, b, atol=1e-11)


def test_bias_rejected_in_group_mode():
    cu = torch.tensor([0, 3, 5], dtype=torch.int32)
    q = rnd((5, 2, 4), 1)
    with pytest.raises(ValueError):
        R.attn_forward(q, q, q, 0.5, cu_seqlens_q=cu, cu_seqlens_k=cu, bias=rnd((1, 1, 3, 3), 2))


# ----------------------------------------------------------------- dropout

@pytest.mark.parametrize("mask", [0, 1])
def test_dropout_finite_differences_with_fixed_mask(mask):
    B, sq, sk, hq, hkv, d = 1, 6, 7, 2, 1, 4
    q, k, v, do = rnd((B, sq, hq, d), 91), rnd((B, sk, hkv, d), 92), rnd((B, sk, hkv, d), 93), rnd((B, sq, hq, d), 94)
    kw = dict(mask=mask, dropout_p=0.3, philox_seed=5, philox_offset=11)

    def L():
        o, _ = R.attn_forward(q, k, v, 0.6, **kw)
        return float((o * do).sum())

    o, lse = R.attn_forward(q, k, v, 0.6, **kw)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.6, **kw)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert rel_err(g, fd_grad(x, L)) < 1e-6


def test_dropout_zero_probability_is_no_dropout():
    B, sq, sk, h, d = 1, 9, 9, 2, 8
    q, k, v, do = rnd((B, sq, h, d), 101), rnd((B, sk, h, d), 102), rnd((B, sk, h, d), 103), rnd((B, sq, h, d), 104)
    o0, l0 = R.attn_forward(q, k, v, 0.4, mask=1)
    o1, l1 = R.attn_forward(q, k, v, 0.4, mask=1, dropout_p=0.0, philox_seed=3)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_dropout_unbiased_over_seeds():
    """E[O] over independent masks is the undropped O (the kept weights are
    scaled by 1 / (1 - p)); 600 seeds, checked to 5 standard errors."""
    B, sq, sk, h, d = 1, 4, 6, 1, 3
    q, k, v = rnd((B, sq, h, d), 111), rnd((B, sk, h, d), 112), rnd((B, sk, h, d), 113)
    o_ref, _ = R.attn_forward(q, k, v, 0.5)
    samples = torch.stack([R.attn_forward(q, k, v, 0.5, dropout_p=0.4, philox_seed=s)[0] for s in range(600)])
    mean, se = samples.mean(0), samples.std(0) / math.sqrt(samples.shape[0])
    assert bool(((mean - o_ref).abs() <= 5 * se + 1e-12).all())

"""Pins of the oracle's layer math against closed forms and independent library routines."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import spd_inputs as si
from oracle import KVCache, Model, layer_block, rmsnorm, rope, silu, argmax_fp32
from oracle.model import Layer

def test_rmsnorm_hand_example():
    # x = [3, 4, 0, 12]: mean square = 169/4, rms = 13/2, so x/rms = [6/13, 8/13, 0, 24/13]
    out = rmsnorm(np.array([3.0, 4.0, 0.0, 12.0]), np.array([1.0, 2.0, 0.5, 1.0]), 0.0)
    np.testing.assert_allclose(out, [6 / 13, 16 / 13, 0.0, 24 / 13], rtol=1e-14)


def test_rmsnorm_matches_torch_library():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 37))
    w = rng.normal(size=37)
    ref = F.rms_norm(torch.from_numpy(x), (37,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(rmsnorm(x, w, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_rope_hand_example_and_complex_form():
    # hd = 4, theta = 100, pos = 2: pair (0, 2) turns by 2 * 100^0 = 2 rad,
    # pair (1, 3) by 2 * 100^(-1/2) = 0.2 rad
    out = rope(np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4), np.array([2]), 100.0).reshape(-1)
    c2, s2, c02, s02 = math.cos(2.0), math.sin(2.0), math.cos(0.2), math.sin(0.2)
    np.testing.assert_allclose(out, [1 * c2 - 3 * s2, 2 * c02 - 4 * s02, 3 * c2 + 1 * s2, 4 * c02 + 2 * s02],
                               rtol=1e-12)
    # complex form: pair (i, i + hd/2) is one complex number rotated by pos * theta^(-2i/hd)
    rng = np.random.default_rng(1)
    hd, theta = 16, 1.0e4
    v = rng.normal(size=(3, 2, hd))
    pos = np.array([0, 5, 1234])
    z = v[..., : hd // 2] + 1j * v[..., hd // 2:]
    w = theta ** (-np.arange(0, hd, 2) / hd)
    zr = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    expect = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(rope(v, pos, theta), expect, rtol=1e-10, atol=1e-12)


def test_rope_relative_position_property():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 1, 32))
    k = rng.normal(size=(1, 1, 32))
    d1 = np.sum(rope(q, [17], 1e4) * rope(k, [5], 1e4))
    d2 = np.sum(rope(q, [117], 1e4) * rope(k, [105], 1e4))
    assert abs(d1 - d2) < 1e-10
    np.testing.assert_allclose(rope(q, [0], 1e4), q)


def _torch_layer(dm, w, H, pos0, Kpast, Vpast):
    """Same layer through torch library primitives (fp64): F.rms_norm,
    scaled_dot_product_attention over [past K/V ; new K/V] with GQA expansion, F.silu.
    RoPE via torch complex multiplication."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    H = t(H)
    M = H.shape[0]
    x = F.rms_norm(H, (dm.d,), t(w.g1), eps=dm.rms_eps)
    q = (x @ t(w.wq).T).view(M, dm.Hq, dm.hd)
    k = (x @ t(w.wk).T).view(M, dm.Hkv, dm.hd)
    v = (x @ t(w.wv).T).view(M, dm.Hkv, dm.hd)
    pos = torch.arange(pos0, pos0 + M, dtype=torch.float64)
    freqs = dm.rope_theta ** (-torch.arange(0, dm.hd, 2, dtype=torch.float64) / dm.hd)
    rot = torch.polar(torch.ones(M, dm.hd // 2, dtype=torch.float64), pos[:, None] * freqs[None, :])

    def ap(a):
        c = torch.complex(a[..., : dm.hd // 2], a[..., dm.hd // 2:]) * rot[:, None, :]
        return torch.cat([c.real, c.imag], dim=-1)

    q, k = ap(q), ap(k)
    Kall = torch.cat([t(Kpast), k], 0)
    Vall = torch.cat([t(Vpast), v], 0)
    S = Kall.shape[0]
    rep = dm.Hq // dm.Hkv
    Kh = Kall.repeat_interleave(rep, dim=1).permute(1, 0, 2)
    Vh = Vall.repeat_interleave(rep, dim=1).permute(1, 0, 2)
    mask = (torch.arange(S)[None, :] <= (torch.arange(M)[:, None] + pos0))
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), Kh, Vh, attn_mask=mask)
    H = H + o.permute(1, 0, 2).reshape(M, -1) @ t(w.wo).T
    y = F.rms_norm(H, (dm.d,), t(w.g2), eps=dm.rms_eps)
    return (H + (F.silu(y @ t(w.wg).T) * (y @ t(w.wu).T)) @ t(w.wd).T).numpy()


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 1)])
def test_layer_matches_torch_library(Hq, Hkv):
    dm = si.ModelDims(L=1, d=48, Hq=Hq, Hkv=Hkv, hd=12, F=40, V=11, dtype="fp32")
    w = Layer(si.make_layer(dm, 3, "L", norms="perturbed"))
    rng = np.random.default_rng(3)
    cache = KVCache(1, 32, Hkv, 12)
    past = 7
    Hp = rng.normal(size=(past, 48))
    layer_block(dm, w, Hp, 0, cache, 0)
    H = rng.normal(size=(3, 48))
    Kpast, Vpast = cache.K[0][:past].copy(), cache.V[0][:past].copy()
    out = layer_block(dm, w, H, past, cache, 0)
    ref = _torch_layer(dm, w, H, past, Kpast, Vpast)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    assert cache.length[0] == past + 3


def test_single_position_attention_returns_value():
    """With one cached position softmax is 1: the attention output is W_o applied to v."""
    dm = si.ModelDims(L=1, d=16, Hq=2, Hkv=1, hd=8, F=8, V=5, dtype="fp32")
    lw = si.make_layer(dm, 4, "L")
    lw["w_gate"] = torch.zeros_like(lw["w_gate"])        # MLP contributes silu(0)*u = 0
    w = Layer(lw)
    cache = KVCache(1, 4, 1, 8)
    h = np.random.default_rng(5).normal(size=(1, 16))
    out = layer_block(dm, w, h, 0, cache, 0)
    x = rmsnorm(h, w.g1, dm.rms_eps)
    v = x @ w.wv.T                                         # [1][8]; both query heads read it
    expect = h + np.concatenate([v, v], axis=1) @ w.wo.T
    np.testing.assert_allclose(out, expect, rtol=1e-12)


def test_silu_values():
    np.testing.assert_allclose(silu(np.array([0.0, 1.0, -2.0])),
                               [0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2))], rtol=1e-14)


def test_block_equals_token_by_token():
    """Prefill as one causal block equals feeding the tokens one at a time."""
    w = si.TINY
    dm = si.shrink(w.dims, L=2, V=64)
    tg = si.make_target(dm, 0, norms="perturbed")
    m = Model(dm, tg)
    ids = [3, 9, 27, 1, 60, 2]
    c1, c2 = m.new_cache(16), m.new_cache(16)
    Hb = m.target_layers(m.embed[ids], 0, c1, 0, dm.L)
    rows = [m.target_layers(m.embed[[t]], p, c2, 0, dm.L)[0] for p, t in enumerate(ids)]
    np.testing.assert_allclose(Hb, np.stack(rows), rtol=1e-11, atol=1e-12)
    for li in range(dm.L):
        np.testing.assert_allclose(c1.K[li][:6], c2.K[li][:6], rtol=1e-11, atol=1e-13)


def test_argmax_lowest_index_on_ties():
    assert argmax_fp32(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    # values equal after rounding to fp32 count as a tie
    assert argmax_fp32(np.array([1.0, 1.0 + 1e-12, 0.5])) == 0


def test_feature_masks_deeper_anchors():
    dm = si.ModelDims(L=4, d=3, Hq=1, Hkv=1, hd=2, F=4, V=5, dtype="fp32")
    m = Model.__new__(Model)
    m.dm, m.anchors = dm, (0, 2, 4)
    vals = {0: np.array([1.0, 2, 3]), 2: np.array([4.0, 5, 6]), 4: np.array([7.0, 8, 9])}
    np.testing.assert_array_equal(m.feature(vals, 0), [1, 2, 3, 0, 0, 0, 0, 0, 0])
    np.testing.assert_array_equal(m.feature(vals, 3), [1, 2, 3, 4, 5, 6, 0, 0, 0])
    np.testing.assert_array_equal(m.feature(vals, 4), [1, 2, 3, 4, 5, 6, 7, 8, 9])


@pytest.mark.parametrize("Hq,Hkv,S", [(4, 4, 1), (8, 2, 9), (8, 1, 33)])
def test_attend_matches_torch_sdpa(Hq, Hkv, S):
    """Single decode query (position S-1) against torch's scaled_dot_product_attention."""
    from oracle import attend
    rng = np.random.default_rng(S)
    hd = 16
    q = rng.normal(size=(1, Hq, hd))
    K = rng.normal(size=(S, Hkv, hd))
    V = rng.normal(size=(S, Hkv, hd))
    out = attend(q, K, V, np.array([S - 1]))
    t = torch.from_numpy
    rep = Hq // Hkv
    ref = F.scaled_dot_product_attention(t(q).permute(1, 0, 2), t(K).repeat_interleave(rep, 1).permute(1, 0, 2),
                                         t(V).repeat_interleave(rep, 1).permute(1, 0, 2))
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)

"""Pins of the CPU oracle against what the Prism pages and plain mathematics fix.

Each test checks the oracle against something other than itself: printed
values (Table 11's shape names), closed forms, invariants, special cases that
reduce to a textbook routine, and brute force on tiny inputs.
"""
import itertools
import math
import os
import statistics

import numpy as np
import pytest
import torch

from content_adaptive_block_02_b300 import synth
from oracle import prism_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(**kw):
    """A small padded workload: 5x7x9 grid, 2x4x4 zones, 16-token blocks."""
    base = synth.WORKLOADS["tiny"].with_(T=5, Hg=7, W=9, H=2, d=8, Ca=8, Na=4)
    return base.with_(**kw)


# ---------------------------------------------------------------- menu ------

def test_table11_shape_names_have_class_token_count():
    """Prism Table 11: every printed shape bT bH bW multiplies to its class."""
    n = 0
    with open(os.path.join(GOLDEN, "table11_shape_names.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            cls, *names = line.split()
            for s in names:
                assert int(s[0]) * int(s[1]) * int(s[2]) == int(cls)
                n += 1
    assert n == 16


@pytest.mark.parametrize("menu,S", [(synth.MENU_TINY, 16), (synth.MENU_128, 128)])
def test_menus_have_equal_token_count(menu, S):
    assert all(a * b * c == S for a, b, c in menu)


def test_admissible_shapes():
    assert orc.admissible_shapes(synth.MENU_128, (3, 16, 16)) == [0, 1]
    assert orc.admissible_shapes(synth.MENU_128, (4, 16, 16)) == list(range(7))
    assert orc.admissible_shapes(synth.MENU_TINY, (2, 4, 4)) == [0, 1, 2]


def test_geometry_matches_2k_token_count():
    """Table 5 caption: 10 s of 2K video at 24 fps is about 870K tokens;
    the 2K-like frame is 90 x 160 latent tokens (61 latent frames)."""
    w = synth.WORKLOADS["2k"]
    assert abs(61 * w.Hg * w.W - 870_000) / 870_000 < 0.01
    assert w.Np == 322_560 and w.n_zones == 420 and w.n_blocks == 2520


# ----------------------------------------------------------- statistics -----

def _grid(w, fn, C):
    x = np.zeros((w.T, w.Hg, w.W, C))
    for t, y, z in itertools.product(range(w.T), range(w.Hg), range(w.W)):
        x[t, y, z] = fn(t, y, z)
    return x.reshape(w.N, C)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_line_variance_linear_ramp_closed_form(axis):
    """A ramp of slope s along one axis over n tokens has population variance
    s^2 (n^2 - 1) / 12 on every full line of that axis, and none across."""
    w = synth.WORKLOADS["tiny"].with_(H=1, d=3)        # 4x8x8 grid, zones 2x4x4, no padding
    slopes = np.array([0.5, -1.25, 3.0])
    x = _grid(w, lambda t, y, z: slopes * (t, y, z)[axis], 3)
    g, m = orc._grid_views(x, w, 3)
    n = w.zone[axis]
    for a in range(3):
        got = orc.line_variance(g, m, a)
        want = (slopes ** 2).mean() * (n * n - 1) / 12.0 if a == axis else 0.0
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_line_variance_constant_field_is_zero():
    w = _small()
    x = np.full((w.N, 4), 2.75)
    g, m = orc._grid_views(x, w, 4)
    for a in range(3):
        assert np.all(orc.line_variance(g, m, a) == 0.0)


def test_line_variance_brute_force_with_padding():
    """Explicit per-line loop with statistics.pvariance on a padded grid."""
    w = _small()
    rng = np.random.default_rng(5)
    C = 3
    x = rng.normal(size=(w.N, C))
    g, m = orc._grid_views(x, w, C)
    Tp, Hp, Wp = orc.padded_grid(w.T, w.Hg, w.W, w.zone)
    zT, zH, zW = w.zone
    xs = x.reshape(w.T, w.Hg, w.W, C)
    for axis in range(3):
        got = orc.line_variance(g, m, axis)
        for zt, zh, zw in itertools.product(range(Tp // zT), range(Hp // zH), range(Wp // zW)):
            vals = []
            ext = (zT, zH, zW)
            others = [a for a in range(3) if a != axis]
            for u in range(ext[others[0]]):
                for v in range(ext[others[1]]):
                    coords = []
                    for s in range(ext[axis]):
                        c = [0, 0, 0]
                        c[axis], c[others[0]], c[others[1]] = s, u, v
                        tt, yy, xx = zt * zT + c[0], zh * zH + c[1], zw * zW + c[2]
                        if tt < w.T and yy < w.Hg and xx < w.W:
                            coords.append((tt, yy, xx))
                    if len(coords) >= 2:
                        for ch in range(C):
                            vals.append(statistics.pvariance([xs[p][ch] for p in coords]))
            want = sum(vals) / len(vals) if vals else 0.0
            assert abs(got[zt, zh, zw] - want) < 1e-12


def test_zone_stats_audio_fields():
    """Constant-norm A2V output: nbar is that norm, no directional variance;
    n_valid counts the zone's real tokens."""
    w = _small()
    rng = np.random.default_rng(1)
    a2v = rng.normal(size=(1, w.N, w.Ca))
    a2v /= np.linalg.norm(a2v, axis=-1, keepdims=True) / 3.0
    V = rng.normal(size=(1, w.N, w.H, w.d))
    st = orc.zone_stats(w, V, a2v)
    assert st.shape == (1, w.H, w.n_zones, 8)
    np.testing.assert_allclose(st[..., 6], 3.0, rtol=1e-12)
    np.testing.assert_allclose(st[..., 3:6], 0.0, atol=1e-12)
    assert st[0, 0, :, 7].sum() == w.N
    # zone 0 is a full 2x4x4 zone
    assert st[0, 0, 0, 7] == 32


# ----------------------------------------------------------- shape rule -----

def test_shape_rule_exact_inverse_guidance_has_zero_cost():
    """g_d proportional to 1/b_d for a menu shape b makes b the continuous
    optimum of Eq. 7 with alpha = 1, so it is chosen with cost 0."""
    w = synth.WORKLOADS["2k"].with_(zone=(4, 16, 16))
    for k, b in enumerate(w.menu):
        g = 0.37 / np.array(b, dtype=float)
        costs, idx = orc.shape_costs(w, g)
        j = int(np.argmin(costs))
        assert idx[j] == k and costs[j] < 1e-24


@pytest.mark.parametrize("alpha", [1.0 / 3.0, 2.0])
def test_shape_rule_exponent_alpha(alpha):
    """The shape-mapping ablation's exponents (Table 10: alpha = 1/3, 2): with
    b*_d proportional to g_d^-alpha, guidance g_d proportional to
    b_d^(-1/alpha) makes the menu shape b the exact optimum (cost 0)."""
    w = synth.WORKLOADS["2k"].with_(zone=(4, 16, 16), alpha=alpha)
    for k, b in enumerate(w.menu):
        g = 0.37 * np.array(b, dtype=float) ** (-1.0 / alpha)
        costs, idx = orc.shape_costs(w, g)
        j = int(np.argmin(costs))
        assert idx[j] == k and costs[j] < 1e-24
    # and alpha scales the deviation of log2 b* from the cube root linearly
    g = np.array([1.0, 2.0, 8.0])
    c1, _ = orc.shape_costs(w.with_(alpha=1.0), g)
    assert not np.allclose(orc.shape_costs(w, g)[0], c1)


def test_shape_rule_equal_guidance_takes_lowest_index():
    w = synth.WORKLOADS["2k"]
    costs, idx = orc.shape_costs(w, np.ones(3))
    assert costs[0] == costs[1] and idx[int(np.argmin(costs))] == 0
    w4 = w.with_(zone=(4, 16, 16))
    costs, idx = orc.shape_costs(w4, np.ones(3))
    # (4,4,8) and (4,8,4) sit nearest to the cube root of 128 and tie
    assert idx[int(np.argmin(costs))] == 3 and abs(costs[3] - costs[4]) < 1e-15


def test_shape_rule_dominant_axis_gets_finest_extent():
    w = synth.WORKLOADS["2k"].with_(zone=(4, 16, 16))
    for axis in range(3):
        g = np.full(3, 1e-3)
        g[axis] = 10.0
        costs, idx = orc.shape_costs(w, g)
        best = w.menu[idx[int(np.argmin(costs))]]
        assert best[axis] == min(s[axis] for s in w.menu)


def test_guidance_zero_statistics_is_isotropic():
    w = synth.WORKLOADS["2k"]
    g = orc.guidance(w, np.zeros(8), 0.0)
    np.testing.assert_allclose(g, 1.0 / 3.0 + w.eps)
    g = orc.guidance(w.with_(use_video=False), np.array([1, 2, 3, 0, 0, 4, 2.0, 5]), 4.0)
    np.testing.assert_allclose(g, 0.5 * np.array([0, 0, 1.0]) + w.eps)


def test_audio_guidance_of_a_constant_norm_map_is_isotropic():
    """A zone whose A2V norms are all equal has no audio direction: round-off
    variances (any size up to 1e-10 nbar^2: a norm spread below 1e-5, which
    fp32 norms do not resolve) give v_hat = 1/3 each, while a small real
    variance keeps its direction."""
    w = synth.WORKLOADS["2k"]
    for noise in ([3e-30, 1e-31, 0.0], [0.0, 9e-13 / 1e9, 0.0], [5e-9, 3e-9, 4e-9]):
        st = np.array([1.0, 2.0, 3.0] + noise + [11.0, 768.0])
        g = orc.guidance(w, st, 11.0)
        np.testing.assert_allclose(g, np.array([1, 2, 3]) / 6.0 + 1.0 / 3.0 + w.eps)
    st = np.array([1.0, 2.0, 3.0, 1e-8, 0.0, 3e-8, 11.0, 768.0])
    g = orc.guidance(w, st, 11.0)
    np.testing.assert_allclose(g, np.array([1, 2, 3]) / 6.0 + np.array([0.25, 0, 0.75]) + w.eps)


def test_assign_shapes_follow_directional_variance():
    """A zone whose values vary only along W must get the finer W extent."""
    w = synth.WORKLOADS["2k"].with_(T=3, Hg=16, W=32, H=1, d=4, use_audio=False)
    x = _grid(w, lambda t, y, z: np.array([z, -z, 2 * z, z]) if z < 16 else
              np.array([y, y, -y, 3 * y]), 4)
    a2v = np.ones((1, w.N, 4))
    st = orc.zone_stats(w, x[None, :, None, :], a2v)
    sid, tie = orc.assign_shapes(w, st)
    assert w.menu[sid[0, 0, 0]] == (1, 16, 8)          # fine along W
    assert w.menu[sid[0, 0, 1]] == (1, 8, 16)          # fine along H
    assert not tie.any()


# ----------------------------------------------------- block-size classes ---

def _tiny_mc(**kw):
    """tiny with a second class: 32-token blocks (2,4,4) next to the 16-token
    menu; about half the zones fall below the threshold."""
    return synth.WORKLOADS["tiny"].with_(menu=synth.MENU_TINY + ((2, 4, 4),),
                                         class_tau=(1.4,), **kw)


def test_single_class_block_table_is_trivial():
    w = _small()
    sid = _random_shapes(w, 4)
    perm, inv, nval = orc.build_permutation(w, sid)
    p2, i2, nv2, tiles, nblk = orc.build_permutation(w, sid, table=True)
    assert np.array_equal(perm, p2) and np.array_equal(nval, nv2)
    assert np.all(tiles == 1) and np.array_equal(nblk, nval)
    X = np.random.default_rng(0).standard_normal((w.B, w.N, w.H, w.d))
    Xp = orc.permute(X, perm)
    assert np.array_equal(orc.pool_blocks(Xp, tiles, nblk, w.block), orc.pool(Xp, nval, w.block))
    L = [np.array([0, 3]), np.array([1]), np.zeros(0, dtype=np.int64)] + \
        [np.zeros(0, dtype=np.int64)] * (len(tiles[0, 0]) - 3)
    out = orc.expand_lists(L, tiles[0, 0])
    assert all(np.array_equal(a, b) for a, b in zip(out, L))


def test_classes_follow_the_thresholds():
    """Complexity above the threshold keeps the smaller class, below it the
    larger; exactly at it the larger is not taken (c >= tau stays fine), and
    a complexity within CLASS_TIE of it is flagged."""
    assert orc.menu_classes(_tiny_mc().menu) == [16, 32]
    taus = (1.5, 0.8)
    assert [orc.zone_class(c, taus) for c in (2.0, 1.5, 1.0, 0.8, 0.1)] == [0, 0, 1, 1, 2]
    w = _tiny_mc(T=4, Hg=4, W=8, H=1, d=4)      # two zones
    st = np.zeros((1, 1, 2, 8))
    st[0, 0, 0, :3] = [2.0, 0.7, 0.3]           # V = 3 (relative 1.5 + gate 1.0)
    st[0, 0, 1, :3] = [0.5, 0.25, 0.25]         # V = 1 (relative 0.5 + gate 1.0)
    st[0, 0, :, 6] = 1.0
    st[0, 0, :, 7] = 32
    sid, tie = orc.assign_shapes(w.with_(class_tau=(1.9,)), st)
    assert [int(np.prod(w.menu[k])) for k in sid[0, 0]] == [16, 32]
    assert not tie.any()
    _, tie = orc.assign_shapes(w.with_(class_tau=(1.5 + 1e-7,)), st)
    assert tie[0, 0, 1] and not tie[0, 0, 0]


def test_multi_tile_blocks_tile_their_zones():
    w = _tiny_mc(T=5, Hg=7, W=9, H=2, d=8, Ca=8, Na=4)
    sid = _random_shapes(w, 6)
    perm, inv, nval, tiles, nblk = orc.build_permutation(w, sid, table=True)
    T_ = w.block
    for b in range(w.B):
        for h in range(w.H):
            assert sorted(perm[b, h][perm[b, h] >= 0]) == list(range(w.N))
            assert np.array_equal(perm[b, h, inv[b, h]], np.arange(w.N))
            i = 0
            while i < len(tiles[b, h]):
                n = int(tiles[b, h, i])
                assert n in (1, 2)
                assert nblk[b, h, i] == nval[b, h, i:i + n].sum()
                # the block's real tokens come first: full tiles, then the rest
                for q in range(n):
                    assert nval[b, h, i + q] == min(T_, max(0, nblk[b, h, i] - q * T_))
                    assert np.all(perm[b, h, (i + q) * T_:(i + q) * T_ + nval[b, h, i + q]] >= 0)
                assert np.all(tiles[b, h, i + 1:i + n] == 0)
                i += n
    assert (tiles == 2).any() and (tiles == 1).any()


def test_mixed_class_path_equals_brute_force_masked_attention():
    """Blocks of two sizes in one head: the tile-level attention over the
    expanded lists equals masked attention whose token mask is built from the
    BLOCK lists (a query token sees every real token of every block its
    block selected), forward and backward, in the original token order."""
    w = _tiny_mc()
    x = _tiny_inputs(w)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
    assert (r["tiles"] == 2).any() and (r["tiles"] == 1).any()
    T_ = w.block
    for h in range(w.H):
        perm, tiles, L = r["perm"][0, h], r["tiles"][0, h], r["block_lists"][(0, h)]
        blk_of = np.zeros(w.N, dtype=np.int64)           # token -> first tile of its block
        i = 0
        while i < len(tiles):
            n = int(tiles[i])
            toks = perm[i * T_:(i + n) * T_]
            blk_of[toks[toks >= 0]] = i
            i += n
        mask = np.zeros((w.N, w.N), bool)
        for q in range(w.N):
            sel = L[blk_of[q]]
            mask[q] = np.isin(blk_of, sel)
        O, dQ, dK, dV = orc.masked_attention(x["Q"][0, :, h], x["K"][0, :, h], x["V"][0, :, h],
                                             mask, r["scale"], dO=x["dO"][0, :, h])
        assert np.abs(O - r["O"][0, :, h]).max() <= 1e-12
        assert np.abs(dQ - r["dQ"][0, :, h]).max() <= 1e-11
        assert np.abs(dK - r["dK"][0, :, h]).max() <= 1e-11
        assert np.abs(dV - r["dV"][0, :, h]).max() <= 1e-11


def _tiny_mc3(**kw):
    """tiny with three classes: 8-token blocks (half a 16-slot tile), the
    16-token menu and (2,4,4); the 4 x 8 x 8 grid has no padding."""
    half = ((1, 2, 4), (2, 2, 2), (1, 4, 2), (2, 1, 4), (2, 4, 1))
    return synth.WORKLOADS["tiny"].with_(menu=half + synth.MENU_TINY + ((2, 4, 4),),
                                         class_tau=(1.6, 1.3), **kw)


def test_block_level_attention_equals_tile_level_attention():
    """attn_blocks (blocks of any size, at block level) equals the tile-level
    forward and backward over the expanded lists, for one class and for
    blocks of one and two tiles."""
    for w in (synth.WORKLOADS["tiny"], _tiny_mc()):
        x = _tiny_inputs(w)
        r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
        U = orc.slot_tokens(w)
        assert U == w.block
        Op, lse, dQ, dK, dV = orc.attn_blocks(r["Qp"], r["Kp"], r["Vp"], r["tiles"], r["n_block"],
                                              r["block_lists"], U, r["scale"], dOp=r["dOp"])
        for a, b_ in ((Op, r["Op"]), (dQ, r["dQp"]), (dK, r["dKp"]), (dV, r["dVp"])):
            np.testing.assert_allclose(a, b_, atol=1e-12)
        np.testing.assert_allclose(lse, r["lse"], atol=1e-12)


def test_half_tile_blocks_equal_brute_force_masked_attention():
    """Three classes, one of them half a tile: the block-level path equals
    masked attention whose token mask comes from the block lists (forward and
    backward, original order), and the masked tile lists describe the same
    token pairs."""
    w = _tiny_mc3()
    x = _tiny_inputs(w)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
    U, T_ = orc.slot_tokens(w), w.block
    assert U == T_ // 2
    sizes = set((r["tiles"] * U)[r["tiles"] > 0].tolist())
    assert sizes == {8, 16, 32}, sizes
    for h in range(w.H):
        perm, units, L = r["perm"][0, h], r["tiles"][0, h], r["block_lists"][(0, h)]
        blk_of = np.zeros(w.N, dtype=np.int64)           # token -> first unit of its block
        i = 0
        while i < len(units):
            n = int(units[i])
            toks = perm[i * U:(i + n) * U]
            blk_of[toks[toks >= 0]] = i
            i += n
        mask = np.zeros((w.N, w.N), bool)
        for q in range(w.N):
            mask[q] = np.isin(blk_of, L[blk_of[q]])
        O, dQ, dK, dV = orc.masked_attention(x["Q"][0, :, h], x["K"][0, :, h], x["V"][0, :, h],
                                             mask, r["scale"], dO=x["dO"][0, :, h])
        assert np.abs(O - r["O"][0, :, h]).max() <= 1e-12
        assert np.abs(dQ - r["dQ"][0, :, h]).max() <= 1e-11
        assert np.abs(dK - r["dK"][0, :, h]).max() <= 1e-11
        assert np.abs(dV - r["dV"][0, :, h]).max() <= 1e-11
        # tile lists with masks: (tile t half qh, tile v half kh) is selected
        # exactly when a token there may attend a token there
        tl, tm = r["lists"][(0, h)]
        tok_slot = np.zeros(w.N, dtype=np.int64)
        tok_slot[perm[perm >= 0]] = np.nonzero(perm >= 0)[0]
        for t in range(len(tl)):
            for v, mbits in zip(tl[t], tm[t]):
                for qh in range(2):
                    for kh in range(2):
                        qs = perm[t * T_ + qh * U:t * T_ + (qh + 1) * U]
                        ks = perm[v * T_ + kh * U:v * T_ + (kh + 1) * U]
                        qs, ks = qs[qs >= 0], ks[ks >= 0]
                        want = bool(mask[np.ix_(qs, ks)].any()) if len(qs) and len(ks) else False
                        assert want == (not (mbits >> (qh * 2 + kh)) & 1), (t, v, qh, kh)
        nsel = sum(len(a) for a in tl)
        assert nsel > 0 and any((m > 0).any() for m in tm if len(m))


def test_padded_zones_skip_the_half_tile_class():
    """A zone with padding never takes a class smaller than the tile."""
    w = _tiny_mc3(T=5, Hg=7, W=9)
    x = _tiny_inputs(w)
    st = orc.zone_stats(w, x["V"], x["a2v"])
    sid, _ = orc.assign_shapes(w, st)
    vol = w.zone[0] * w.zone[1] * w.zone[2]
    small = np.array([np.prod(w.menu[k]) < w.block for k in sid.ravel()]).reshape(sid.shape)
    assert small.any()
    assert not (small & (st[..., 7] < vol)).any()


# ------------------------------------------------ A2V cross-attention -------

def test_a2v_norms_special_cases():
    """One audio token: every output is that token's value; equal logits (zero
    keys): the output is the mean of the values; a dominant key: its value."""
    rng = np.random.default_rng(7)
    B, N, Na, Ca = 2, 9, 5, 8
    Qa = rng.standard_normal((B, N, Ca))
    Va = rng.standard_normal((B, Na, Ca))
    n1 = orc.a2v_norms(Qa, rng.standard_normal((B, 1, Ca)), Va[:, :1])
    np.testing.assert_allclose(n1, np.linalg.norm(Va[:, 0], axis=-1)[:, None].repeat(N, 1),
                               rtol=1e-14)
    n0 = orc.a2v_norms(Qa, np.zeros((B, Na, Ca)), Va)
    np.testing.assert_allclose(n0, np.linalg.norm(Va.mean(axis=1), axis=-1)[:, None].repeat(N, 1),
                               rtol=1e-14)
    Ka = np.zeros((B, Na, Ca))
    Ka[:, 3] = 1e3 * Qa[:, 0] / np.linalg.norm(Qa[:, 0], axis=-1, keepdims=True)
    nd = orc.a2v_norms(Qa[:, :1], Ka, Va)
    np.testing.assert_allclose(nd[:, 0], np.linalg.norm(Va[:, 3], axis=-1), rtol=1e-12)


def test_a2v_norms_match_the_generators_cross_attention():
    """The generator's stand-in for the model's A2V layer (torch, fp32, from
    the same bf16 queries and audio tokens) against the oracle's norms."""
    w = synth.WORKLOADS["tiny"]
    x = synth.generate(w, "cpu", a2v_f32=True)
    n_ref = np.linalg.norm(x["a2v_f32"].double().numpy(), axis=-1)
    qa = x["qa"].float().numpy()
    au = x["audio"].float().numpy()
    n = orc.a2v_norms(qa, au, au)
    np.testing.assert_allclose(n, n_ref, rtol=2e-5)
    # and zone statistics from the norms equal those from the output itself
    a2v = x["a2v_f32"].double().numpy()
    V = x["V"].float().numpy()
    np.testing.assert_allclose(orc.zone_stats_from_norms(w, V, np.linalg.norm(a2v, axis=-1)),
                               orc.zone_stats(w, V, a2v), rtol=1e-12, atol=1e-300)


def test_line_variance_bound_holds_and_is_reached():
    """Brute force: relative perturbations of a scalar map within tau move
    every zone's line variance by at most the bound; perturbing each line's
    values away from its mean (sign of n - mean) comes within O(tau^2) of it."""
    w = _small()
    rng = np.random.default_rng(9)
    n = 3.0 + rng.random(w.N)
    tau = 1e-3
    g, m = orc._grid_views(n[:, None], w, 1)
    for axis in range(3):
        v0 = orc.line_variance(g, m, axis)
        bnd = orc.line_variance_bound(g, m, axis, tau)
        for _ in range(30):
            gp, _ = orc._grid_views((n * (1 + rng.uniform(-tau, tau, n.shape)))[:, None], w, 1)
            assert np.all(np.abs(orc.line_variance(gp, m, axis) - v0) <= bnd * (1 + 1e-9))
    # the extreme perturbation of the W lines: e_i = tau sign(n_i - line mean)
    inner = 5
    mean = (g * m[..., None]).sum(axis=inner, keepdims=True) / m[..., None].sum(axis=inner, keepdims=True).clip(1)
    gp = g * (1 + tau * np.sign(g - mean))
    lin = orc.line_variance_bound(g, m, 2, tau) - orc.line_variance_bound(g, m, 2, 0.0)
    move = orc.line_variance(gp, m, 2) - orc.line_variance(g, m, 2)
    np.testing.assert_allclose(move, lin, rtol=1e-2, atol=1e-12)


def test_norm_sensitive_zones_cover_every_flip_under_bounded_norm_errors():
    """Brute force over norm maps perturbed within tau (relative): every zone
    whose shape changes is flagged (as a near tie or as norm-sensitive); tau
    = 0 flags nothing beyond the near ties; one zone with a constant norm map
    (audio floor) is flagged once tau can lift it over the floor."""
    w = _small(H=2, d=4)
    rng = np.random.default_rng(21)
    t, y, x = np.meshgrid(np.arange(w.T), np.arange(w.Hg), np.arange(w.W), indexing="ij")
    n = (4.0 + np.sin(0.9 * x + 0.3 * t) + 0.6 * np.cos(0.7 * y) + 0.3 * rng.random(x.shape))
    n[:2, :4, :4] = 2.5                                  # zone 0: a constant map
    n = n.reshape(1, -1)
    V = rng.standard_normal((1, w.N, w.H, w.d))
    st = orc.zone_stats_from_norms(w, V, n)
    sid, tie = orc.assign_shapes(w, st)
    assert np.array_equal(orc.norm_sensitive_zones(w, n, st, 0.0) | tie, tie)
    seen_flip = False
    for tau in (1e-4, 3e-3, 1e-2):
        flags = orc.norm_sensitive_zones(w, n, st, tau) | tie
        assert not flags.all()
        for trial in range(60):
            if trial % 3 == 0:
                e = tau * rng.choice([-1.0, 1.0], size=n.shape)
            else:
                e = rng.uniform(-tau, tau, n.shape)
            s2, _ = orc.assign_shapes(w, orc.zone_stats_from_norms(w, V, n * (1 + e)))
            flips = s2 != sid
            seen_flip |= bool(flips.any())
            assert not (flips & ~flags).any(), (tau, np.nonzero(flips & ~flags))
        if tau >= 3e-3:
            assert flags[0, :, 0].all()                    # the constant zone
    assert seen_flip


# ------------------------------------------------------------ permutation ---

def _random_shapes(w, seed):
    rng = np.random.default_rng(seed)
    adm = orc.admissible_shapes(w.menu, w.zone)
    return rng.choice(adm, size=(w.B, w.H, w.n_zones))


def test_permutation_is_a_blockwise_bijection():
    w = _small()
    sid = _random_shapes(w, 3)
    perm, inv, nval = orc.build_permutation(w, sid)
    S = w.block
    for h in range(w.H):
        p = perm[0, h]
        real = p[p >= 0]
        assert sorted(real.tolist()) == list(range(w.N))
        assert np.all(p[inv[0, h]] == np.arange(w.N))
        for blk in range(w.n_blocks):
            seg = p[blk * S:(blk + 1) * S]
            nv = int(nval[0, h, blk])
            assert np.all(seg[:nv] >= 0) and np.all(seg[nv:] == -1)
            if nv == 0:
                continue
            t, r = np.divmod(seg[:nv], w.Hg * w.W)
            y, x = np.divmod(r, w.W)
            # one zone, and inside the box of the zone's chosen shape
            z = set(zip(t // w.zone[0], y // w.zone[1], x // w.zone[2]))
            assert len(z) == 1
            zt, zh, zw = z.pop()
            Z = ((zt * (orc.padded_grid(w.T, w.Hg, w.W, w.zone)[1] // w.zone[1]) + zh)
                 * (orc.padded_grid(w.T, w.Hg, w.W, w.zone)[2] // w.zone[2]) + zw)
            bT, bH, bW = w.menu[sid[0, h, Z]]
            assert t.max() - t.min() < bT and y.max() - y.min() < bH and x.max() - x.min() < bW
            # valid tokens in raster order
            assert np.all(np.diff(seg[:nv]) > 0)


def test_permutation_orders_zones_then_blocks_in_raster_order():
    """Reading 7: zones in raster (zt, zh, zw) order, and inside a zone its
    blocks in raster order of the zone's block grid: block k lies in zone
    k // blocks_per_zone, at grid position k % blocks_per_zone."""
    w = _small()
    sid = _random_shapes(w, 8)
    perm, inv, nval = orc.build_permutation(w, sid)
    S = w.block
    zT, zH, zW = w.zone
    Tp, Hp, Wp = orc.padded_grid(w.T, w.Hg, w.W, w.zone)
    nzH, nzW = Hp // zH, Wp // zW
    bpz = (zT * zH * zW) // S
    for h in range(w.H):
        for blk in range(w.n_blocks):
            nv = int(nval[0, h, blk])
            if nv == 0:
                continue
            Z, local = divmod(blk, bpz)
            zt, rest = divmod(Z, nzH * nzW)
            zh, zw = divmod(rest, nzW)
            bT, bH, bW = w.menu[sid[0, h, Z]]
            it, rest = divmod(local, (zH // bH) * (zW // bW))
            ih, iw = divmod(rest, zW // bW)
            t0, y0, x0 = zt * zT + it * bT, zh * zH + ih * bH, zw * zW + iw * bW
            seg = perm[0, h, blk * S: blk * S + nv]
            t, r = np.divmod(seg, w.Hg * w.W)
            y, x = np.divmod(r, w.W)
            assert t.min() >= t0 and t.max() < t0 + bT, (h, blk)
            assert y.min() >= y0 and y.max() < y0 + bH, (h, blk)
            assert x.min() >= x0 and x.max() < x0 + bW, (h, blk)
            # every real token of that box is in the block
            box = [(tt * w.Hg + yy) * w.W + xx for tt in range(t0, min(t0 + bT, w.T))
                   for yy in range(y0, min(y0 + bH, w.Hg)) for xx in range(x0, min(x0 + bW, w.W))]
            assert sorted(box) == seg.tolist()


def test_permute_unpermute_identity():
    w = _small()
    sid = _random_shapes(w, 4)
    perm, inv, _ = orc.build_permutation(w, sid)
    X = np.random.default_rng(0).normal(size=(1, w.N, w.H, w.d))
    Xp = orc.permute(X, perm)
    assert np.all(Xp[perm < 0] == 0.0)
    np.testing.assert_array_equal(orc.unpermute(Xp, inv), X)


def test_pool_is_mean_of_the_blocks_tokens():
    w = _small()
    sid = _random_shapes(w, 5)
    perm, inv, nval = orc.build_permutation(w, sid)
    X = np.random.default_rng(2).normal(size=(1, w.N, w.H, w.d))
    Xb = orc.pool(orc.permute(X, perm), nval, w.block)
    for h in range(w.H):
        for blk in range(w.n_blocks):
            toks = [n for n in perm[0, h, blk * w.block:(blk + 1) * w.block] if n >= 0]
            if toks:
                want = np.mean([X[0, n, h] for n in toks], axis=0)
                np.testing.assert_allclose(Xb[0, h, blk], want, rtol=1e-13, atol=1e-15)
            else:
                assert np.all(Xb[0, h, blk] == 0)


# -------------------------------------------------------------- selection ---

def test_topp_strictly_exceeds():
    """Table 7 caption: the set's cumulative weight must exceed p."""
    pr = np.array([0.5, 0.25, 0.125, 0.125])
    assert orc.topp_count(pr, 0.75) == 3      # 0.75 does not exceed 0.75
    assert orc.topp_count(pr, 0.74) == 2
    assert orc.topp_count(pr, 0.0) == 1
    assert orc.topp_count(pr, 0.875) == 4
    assert orc.topp_count(pr, 1.0) == 4


def test_topp_is_the_smallest_exceeding_set_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(200):
        n = int(rng.integers(1, 8))
        pr = rng.dirichlet(np.ones(n) * 0.7)
        p = float(rng.uniform(0, 0.999))
        best = min(len(c) for r in range(1, n + 1) for c in itertools.combinations(range(n), r)
                   if sum(pr[list(c)]) > p)
        assert orc.topp_count(np.sort(pr)[::-1], p) == best


def test_select_p0_is_topk_by_score():
    rng = np.random.default_rng(9)
    for trial in range(50):
        nb = int(rng.integers(3, 40))
        s = rng.normal(size=nb) * 3
        s[rng.integers(0, nb)] = s[0]                   # a duplicated score
        valid = rng.random(nb) > 0.2
        valid[0] = True
        kf = int(rng.integers(1, 6))
        sel, _ = orc.hybrid_select_row(s, valid, kf, 0.0)
        cand = [j for j in range(nb) if valid[j]]
        want = sorted(sorted(cand, key=lambda j: (-s[j], j))[:min(kf, len(cand))])
        assert sel.tolist() == want


def test_select_p1_keeps_every_valid_block():
    rng = np.random.default_rng(10)
    s = rng.normal(size=30) * 40                        # very peaked softmax
    valid = np.ones(30, bool)
    valid[[3, 17]] = False
    sel, _ = orc.hybrid_select_row(s, valid, 2, 1.0)
    assert sel.tolist() == [j for j in range(30) if valid[j]]


def test_select_hybrid_is_max_of_floor_and_topp():
    s = np.log(np.array([0.5, 0.25, 0.125, 0.0625, 0.0625]))
    valid = np.ones(5, bool)
    sel, _ = orc.hybrid_select_row(s, valid, 1, 0.7)   # Top-p needs 2
    assert sel.tolist() == [0, 1]
    sel, _ = orc.hybrid_select_row(s, valid, 4, 0.7)   # floor 4 wins
    assert sel.tolist() == [0, 1, 2, 3]
    sel, _ = orc.hybrid_select_row(s, valid, 9, 0.7)   # floor capped at the candidates
    assert sel.tolist() == [0, 1, 2, 3, 4]


def test_select_flags_near_ties():
    s = np.array([1.0, 0.5, 0.5 + 1e-9, -3.0])
    sel, flag = orc.hybrid_select_row(s, np.ones(4, bool), 2, 0.0)
    assert flag and sel.tolist() == [0, 2]
    sel, flag = orc.hybrid_select_row(np.array([2.0, 0.0, -2.0]), np.ones(3, bool), 1, 0.1)
    assert not flag


# -------------------------------------------------------------- attention ---

def _tiny_inputs(w, seed=0):
    torch.manual_seed(seed)
    d = synth.generate(w, "cpu")
    return {k: (v.float().numpy().astype(np.float64) if torch.is_tensor(v) else v)
            for k, v in d.items()}


def test_dense_special_case_equals_plain_attention():
    """Top-p = 1 keeps every block, so the path is plain softmax attention."""
    w = synth.WORKLOADS["tiny"].with_(topp=1.0)
    x = _tiny_inputs(w)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"])
    for h in range(w.H):
        ref = orc.dense_attention(x["Q"][0, :, h], x["K"][0, :, h], x["V"][0, :, h], r["scale"])
        assert np.abs(r["O"][0, :, h] - ref).max() <= 1e-12
    w2 = synth.WORKLOADS["tiny"].with_(topk_floor=10 ** 6)
    r2 = orc.run(w2, x["Q"], x["K"], x["V"], x["a2v"])
    assert np.abs(r2["O"] - r["O"]).max() <= 1e-12


def _token_mask(w, r, b, h):
    S = w.block
    perm, L = r["perm"][b, h], r["lists"][(b, h)]
    mask = np.zeros((w.N, w.N), bool)
    for i, sel in enumerate(L):
        qs = [n for n in perm[i * S:(i + 1) * S] if n >= 0]
        ks = [n for j in sel for n in perm[j * S:(j + 1) * S] if n >= 0]
        for q in qs:
            mask[q, ks] = True
    return mask


def test_block_sparse_equals_brute_force_masked_attention():
    """Permuted block-sparse forward and backward equal masked attention with
    the explicit N x N token mask, in the original order."""
    w = synth.WORKLOADS["tiny"]
    x = _tiny_inputs(w)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
    sparsity = []
    for h in range(w.H):
        mask = _token_mask(w, r, 0, h)
        sparsity.append(1 - mask.mean())
        O, dQ, dK, dV = orc.masked_attention(x["Q"][0, :, h], x["K"][0, :, h], x["V"][0, :, h],
                                             mask, r["scale"], dO=x["dO"][0, :, h])
        assert np.abs(O - r["O"][0, :, h]).max() <= 1e-12
        assert np.abs(dQ - r["dQ"][0, :, h]).max() <= 1e-11
        assert np.abs(dK - r["dK"][0, :, h]).max() <= 1e-11
        assert np.abs(dV - r["dV"][0, :, h]).max() <= 1e-11
    assert max(sparsity) > 0.2                          # the case is genuinely sparse


def test_gradients_match_central_finite_differences():
    """d<O, dO>/dX by central differences with the selection held fixed."""
    w = _small(H=1, d=6, Ca=6, topp=0.6, topk_floor=1)
    x = _tiny_inputs(w, seed=3)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
    rng = np.random.default_rng(0)
    perm, inv, nval = r["perm"], r["inv"], r["n_valid"]

    def objective(Q, K, V):
        Qp, Kp, Vp = orc.permute(Q, perm), orc.permute(K, perm), orc.permute(V, perm)
        Op, _ = orc.attn_fwd(w, Qp, Kp, Vp, nval, r["lists"], r["scale"])
        return float((orc.unpermute(Op, inv) * x["dO"]).sum())

    eps = 1e-6
    for name, grad in (("Q", r["dQ"]), ("K", r["dK"]), ("V", r["dV"])):
        for _ in range(6):
            n, c = int(rng.integers(0, w.N)), int(rng.integers(0, w.d))
            args = {k: x[k].copy() for k in ("Q", "K", "V")}
            args[name][0, n, 0, c] += eps
            fp = objective(args["Q"], args["K"], args["V"])
            args[name][0, n, 0, c] -= 2 * eps
            fm = objective(args["Q"], args["K"], args["V"])
            fd = (fp - fm) / (2 * eps)
            assert abs(fd - grad[0, n, 0, c]) <= 1e-6 * max(1.0, abs(fd))


def test_lse_is_log_sum_exp_of_selected_scores():
    w = synth.WORKLOADS["tiny"]
    x = _tiny_inputs(w)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"])
    S = w.block
    h = 1
    mask = _token_mask(w, r, 0, h)
    q, k = x["Q"][0, :, h], x["K"][0, :, h]
    for n in range(0, w.N, 37):
        s = [math.fsum([q[n, c] * k[m, c] for c in range(w.d)]) * r["scale"]
             for m in range(w.N) if mask[n, m]]
        want = max(s) + math.log(math.fsum(math.exp(v - max(s)) for v in s))
        slot = r["inv"][0, h, n]
        assert abs(r["lse"][0, h, slot] - want) < 1e-12


# ------------------------------------------------------- bf16 rounding ------

def test_round_bf16_matches_the_library_conversion_and_ties_to_even():
    rng = np.random.default_rng(3)
    # values exactly representable in fp32, so the library's conversion has a
    # single rounding too
    x = rng.standard_normal(20000).astype(np.float32).astype(np.float64) * 10.0 ** rng.integers(-8, 8, 20000)
    x = x.astype(np.float32).astype(np.float64)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(orc.round_bf16(x), ref)
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (even: 1);
    # 1 + 3 * 2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (even: 1 + 2^-6)
    t = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 0.0, -0.0])
    assert orc.round_bf16(t).tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 0.0, -0.0]


def test_backward_from_stored_bf16_output_differs_by_the_rounding_of_o_only():
    """o_bf16 changes only D = rowsum(dO * O): dV is unchanged and dQ moves by
    at most scale * max|K| * 2^-8 * sum_c |dO_c| |O_c| per row (each P row sums
    to one; bf16 rounding is within 2^-8 relative)."""
    rng = np.random.default_rng(5)
    S, d, nb = 8, 16, 4
    Qp = rng.standard_normal((nb * S, d)); Kp = rng.standard_normal((nb * S, d))
    Vp = rng.standard_normal((nb * S, d)); dOp = rng.standard_normal((nb * S, d))
    nv = np.full(nb, S)
    sel = np.array([0, 2, 3])
    scale = 1 / math.sqrt(d)
    dq0, dk0, dv0 = orc.attn_bwd_row(Qp, Kp, Vp, dOp, nv, 1, sel, S, scale)
    dq1, dk1, dv1 = orc.attn_bwd_row(Qp, Kp, Vp, dOp, nv, 1, sel, S, scale, o_bf16=True)
    assert np.array_equal(dv0, dv1)
    o, _ = orc.attn_fwd_row(Qp, Kp, Vp, nv, 1, sel, S, scale)
    bound = scale * np.abs(Kp).max() * 2.0 ** -8 * (np.abs(dOp[S:2 * S]) * np.abs(o)).sum(1)
    assert np.all(np.abs(dq1 - dq0).max(1) <= bound + 1e-15)
    assert np.abs(dq1 - dq0).max() > 0


def _bwd_case(seed=11, positive=()):
    rng = np.random.default_rng(seed)
    S, d, nb = 8, 4, 4
    X = {k: rng.standard_normal((nb * S, d)) for k in ("Q", "K", "V", "dO")}
    for k in positive:
        X[k] = np.abs(X[k])
    nv = np.array([S, 5, S, S])                       # query block 1 partly real
    return X, nv, S, d, np.array([0, 1, 3]), 1 / math.sqrt(d)


def _dq_dk_at(X, nv, S, sel, scale, o_given, i=1):
    dq, dk, _ = orc.attn_bwd_row(X["Q"], X["K"], X["V"], X["dO"], nv, i, sel, S, scale,
                                 o_given=o_given)
    return dq, dk


def test_bound_terms_are_the_worst_case_over_bf16_output_errors_brute_force():
    """abs_terms: the per-element sizes by which dq and dk move when the O
    that D is formed from carries bf16 forward errors (|dO_ic| <= u (|O_ic| +
    (P|V|)_ic)).  Brute force over perturbations of O: every one of the 2^d
    extreme sign patterns of a query row, and random interior ones, stays
    within u * terms; the worst pattern reaches it for dq exactly, and, with
    Q >= 0 (no cancellation over rows), for dk too."""
    u = 2.0 ** -9
    i = 1
    for positive in ((), ("Q",)):
        X, nv, S, d, sel, scale = _bwd_case(positive=positive)
        o, _ = orc.attn_fwd_row(X["Q"], X["K"], X["V"], nv, i, sel, S, scale)
        _, _, _, aq, ak = orc.attn_bwd_row(X["Q"], X["K"], X["V"], X["dO"], nv, i, sel, S,
                                           scale, abs_terms=True)
        dq0, dk0 = _dq_dk_at(X, nv, S, sel, scale, o)
        # the allowed size of the error of each element of O
        k = np.concatenate([X["K"][j * S:j * S + nv[j]] for j in sel])
        v = np.concatenate([X["V"][j * S:j * S + nv[j]] for j in sel])
        s = X["Q"][i * S:(i + 1) * S] @ k.T * scale
        P = np.exp(s - s.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        room = u * (np.abs(o) + P @ np.abs(v))
        worst_q = np.zeros_like(dq0)
        for signs in itertools.product((-1.0, 1.0), repeat=d):
            dq, dk = _dq_dk_at(X, nv, S, sel, scale, o + room * np.array(signs))
            worst_q = np.maximum(worst_q, np.abs(dq - dq0))
            assert np.all(np.abs(dq - dq0) <= u * aq * (1 + 1e-9) + 1e-300)
            assert np.all(np.abs(dk - dk0) <= u * ak * (1 + 1e-9) + 1e-300)
        rng = np.random.default_rng(2)
        for _ in range(50):
            dq, dk = _dq_dk_at(X, nv, S, sel, scale, o + room * rng.uniform(-1, 1, o.shape))
            assert np.all(np.abs(dq - dq0) <= u * aq * (1 + 1e-9) + 1e-300)
            assert np.all(np.abs(dk - dk0) <= u * ak * (1 + 1e-9) + 1e-300)
        np.testing.assert_allclose(worst_q, u * aq, rtol=1e-9, atol=1e-300)
        assert np.all(aq[nv[i]:] == 0) and aq[:nv[i]].min() > 0
        if positive:
            # every D_i moved up by u b_i at once (signs of dO): dk's terms align
            dq, dk = _dq_dk_at(X, nv, S, sel, scale, o + room * np.sign(X["dO"][i * S:(i + 1) * S]))
            np.testing.assert_allclose(np.abs(dk - dk0), u * ak, rtol=1e-9, atol=1e-300)


def test_bound_terms_vanish_without_upstream_gradient():
    """A query row with zero upstream gradient has nothing to move: its dq
    sizes are zero, and a query block whose dO is zero throughout adds nothing
    to the dk sizes."""
    X, nv, S, d, sel, scale = _bwd_case(seed=4)
    X["dO"][1 * S:1 * S + 2] = 0.0
    _, _, _, aq, ak = orc.attn_bwd_row(X["Q"], X["K"], X["V"], X["dO"], nv, 1, sel, S, scale,
                                       abs_terms=True)
    assert np.all(aq[:2] == 0)
    # dk collects over the rows of the query block: a block whose dO is all
    # zero contributes nothing
    X["dO"][1 * S:2 * S] = 0.0
    _, _, _, aq0, ak0 = orc.attn_bwd_row(X["Q"], X["K"], X["V"], X["dO"], nv, 1, sel, S, scale,
                                         abs_terms=True)
    assert np.all(aq0 == 0) and np.all(ak0 == 0)


def test_key_block_gradients_equal_the_full_backward():
    """attn_bwd_key_blocks is attn_bwd restricted to some key blocks."""
    w = _small(H=1, d=6, Ca=6, topp=0.6, topk_floor=2)
    x = _tiny_inputs(w, seed=5)
    r = orc.run(w, x["Q"], x["K"], x["V"], x["a2v"], dO=x["dO"])
    S, L = w.block, r["lists"][(0, 0)]
    for o_bf16 in (False, True):
        _, dK, dV = orc.attn_bwd(w, r["Qp"], r["Kp"], r["Vp"], r["dOp"], r["n_valid"], r["lists"],
                                 r["scale"], o_bf16=o_bf16)
        kb = [j for j in range(len(L)) if r["n_valid"][0, 0, j] > 0][::3]
        got = orc.attn_bwd_key_blocks(r["Qp"][0, 0], r["Kp"][0, 0], r["Vp"][0, 0], r["dOp"][0, 0],
                                      r["n_valid"][0, 0], L, kb, S, r["scale"], o_bf16=o_bf16)
        for j in kb:
            np.testing.assert_allclose(got[j][0], dK[0, 0, j * S:(j + 1) * S], atol=1e-13)
            np.testing.assert_allclose(got[j][1], dV[0, 0, j * S:(j + 1) * S], atol=1e-13)
        assert max(np.abs(got[j][0]).max() for j in kb) > 0
    # the dK sizes (per unit roundoff of the O behind D) are the full
    # backward's, whose per-row terms the brute-force pin above holds
    _, _, _, _, aK = orc.attn_bwd(w, r["Qp"], r["Kp"], r["Vp"], r["dOp"], r["n_valid"],
                                  r["lists"], r["scale"], o_bf16=True, abs_terms=True)
    got = orc.attn_bwd_key_blocks(r["Qp"][0, 0], r["Kp"][0, 0], r["Vp"][0, 0], r["dOp"][0, 0],
                                  r["n_valid"][0, 0], L, kb, S, r["scale"], o_bf16=True,
                                  abs_terms=True)
    for j in kb:
        np.testing.assert_allclose(got[j][2], aK[0, 0, j * S:(j + 1) * S], rtol=1e-12, atol=1e-300)
    assert max(got[j][2].max() for j in kb) > 0


# ------------------------------------------------- library and structure ----

def test_masked_attention_vjp_equals_torch_autograd():
    """The reference masked attention's VJP (used by the brute-force pin)
    against torch's autograd of the same masked softmax attention in fp64."""
    rng = np.random.default_rng(11)
    N, d = 40, 12
    Q, K, V, dO = (rng.standard_normal((N, d)) for _ in range(4))
    mask = rng.random((N, N)) < 0.3
    mask[np.arange(N), rng.integers(0, N, N)] = True          # every row keeps a key
    scale = 1 / math.sqrt(d)
    O, dQ, dK, dV = orc.masked_attention(Q, K, V, mask, scale, dO=dO)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    s = (tq @ tk.T * scale).masked_fill(~torch.tensor(mask), float("-inf"))
    to = torch.softmax(s, dim=-1) @ tv
    to.backward(torch.tensor(dO, dtype=torch.float64))
    assert np.abs(O - to.detach().numpy()).max() <= 1e-12
    for got, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        assert np.abs(got - ref.numpy()).max() <= 1e-12


def test_csc_is_the_transpose_of_the_lists():
    rng = np.random.default_rng(2)
    nb = 23
    L = [None if i % 7 == 3 else np.sort(rng.choice(nb, rng.integers(0, 9), replace=False))
         for i in range(nb)]
    cols = orc.csc_from_lists(L, nb)
    pairs_rows = {(i, int(j)) for i, s in enumerate(L) if s is not None for j in s}
    pairs_cols = {(int(i), j) for j, c in enumerate(cols) for i in c}
    assert pairs_rows == pairs_cols
    assert all(np.all(np.diff(c) > 0) for c in cols)


def test_block_scores_are_bilinear_and_scaled():
    rng = np.random.default_rng(4)
    d = 16
    Qb, Kb = rng.standard_normal((5, d)), rng.standard_normal((7, d))
    S = orc.block_scores(Qb, Kb, d)
    assert np.allclose(orc.block_scores(3.0 * Qb, Kb, d), 3.0 * S, rtol=0, atol=1e-12)
    e = np.eye(d) * d ** 0.25                                   # e_i . e_i / sqrt(d) = 1
    assert np.allclose(orc.block_scores(e[:4], e[:4], d), np.eye(4), rtol=0, atol=1e-14)
    assert np.allclose(orc.block_scores(e[:2], e[2:4], d), 0.0, rtol=0, atol=0)


def test_select_blocks_applies_the_row_rule_and_skips_empty_blocks():
    w = synth.WORKLOADS["tiny"].with_(B=1, H=2, topk_floor=2, topp=0.7)
    rng = np.random.default_rng(9)
    nb, d = 16, w.d
    Qb, Kb = rng.standard_normal((1, 2, nb, d)), rng.standard_normal((1, 2, nb, d))
    nv = np.full((1, 2, nb), 16)
    nv[0, 0, [3, 11]] = 0                                       # blocks without real tokens
    L, F = orc.select_blocks(w, Qb, Kb, nv)
    for h in range(2):
        S = orc.block_scores(Qb[0, h], Kb[0, h], d)
        valid = nv[0, h] > 0
        for i in range(nb):
            if not valid[i]:
                assert len(L[(0, h)][i]) == 0
                continue
            ref, flag = orc.hybrid_select_row(S[i], valid, w.topk_floor, w.topp)
            assert np.array_equal(L[(0, h)][i], ref) and F[(0, h)][i] == flag
            assert not np.isin(L[(0, h)][i], np.flatnonzero(~valid)).any()

"""Plain fp64 CPU oracle of the Prism hot path.  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference leg of ``bench.py`` may import this module.  The CUDA path shares no
code with it and never calls it.

"Prism" below is the paper *Prism: Dynamic Sparse Attention for Native 2K
Joint Video-Audio Generation Model Training* (arXiv 2610.05416) as printed on
its abstract, figure and table pages.  The pages give the method only in prose
(Abstract; Fig. 2 caption) and table captions (Tables 7, 9, 10, 11, 12); the
equations they refer to (Eq. 1, Eq. 7) are not printed.  Where a step is left
open, the plainest reading is taken and marked READING.

Steps, in the order the pages give them:
  1. zone statistics            -- ``zone_stats``
  2. block shape per zone       -- ``assign_shapes``
     and the token permutation  -- ``build_permutation`` / ``permute``
  3. block-mean Q/K, scores     -- ``pool``, ``block_scores``
  4. hybrid Top-k / Top-p       -- ``hybrid_select_row`` / ``select_blocks``
  5. block-sparse attention     -- ``attn_fwd_row`` / ``attn_bwd``
     and the inverse permutation-- ``unpermute``
plus two independent references used as pins: ``dense_attention`` (plain
softmax attention in the original token order) and ``masked_attention``
(explicit N x N token mask, original order, forward and VJP).

Everything is computed in float64 from the bf16-rounded inputs.
Parity pinned by the tests in tests/test_oracle_*.py, except the reading of the
unprinted Eq. 1 / Eq. 7 / gate / combination, which is parity unpinned: the
pages do not print them, so only their special cases can be checked.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

f64 = np.float64


# --------------------------------------------------------------------------
# geometry
# --------------------------------------------------------------------------

def padded_grid(T: int, Hg: int, W: int, zone: Sequence[int]) -> Tuple[int, int, int]:
    """READING (Prism, Abstract: macro-zones tile the token grid): each axis is
    padded up to a multiple of the zone extent; padded tokens are not real."""
    zT, zH, zW = zone
    return (-(-T // zT) * zT, -(-Hg // zH) * zH, -(-W // zW) * zW)


def admissible_shapes(menu: Sequence[Sequence[int]], zone: Sequence[int]) -> List[int]:
    """READING: a menu shape (bT, bH, bW) may be given to a zone only when it
    tiles the zone exactly, i.e. each block extent divides the zone extent."""
    return [k for k, b in enumerate(menu)
            if zone[0] % b[0] == 0 and zone[1] % b[1] == 0 and zone[2] % b[2] == 0]


def _grid_views(x: np.ndarray, w, C: int) -> Tuple[np.ndarray, np.ndarray]:
    """Scatter a real-token array x [N, C] onto the padded grid and view it as
    [Zt, zT, Zh, zH, Zw, zW, C]; also return the matching validity mask."""
    Tp, Hp, Wp = padded_grid(w.T, w.Hg, w.W, w.zone)
    zT, zH, zW = w.zone
    g = np.zeros((Tp, Hp, Wp, C), dtype=f64)
    g[: w.T, : w.Hg, : w.W] = x.reshape(w.T, w.Hg, w.W, C)
    m = np.zeros((Tp, Hp, Wp), dtype=bool)
    m[: w.T, : w.Hg, : w.W] = True
    g = g.reshape(Tp // zT, zT, Hp // zH, zH, Wp // zW, zW, C)
    m = m.reshape(Tp // zT, zT, Hp // zH, zH, Wp // zW, zW)
    return g, m


# --------------------------------------------------------------------------
# step 1: zone statistics
# --------------------------------------------------------------------------

def line_variance(g: np.ndarray, m: np.ndarray, axis: int) -> np.ndarray:
    """Directional variance of every zone along one grid axis.

    g: [Zt, zT, Zh, zH, Zw, zW, C] values, m: the validity mask without C.
    axis: 0 = T, 1 = H, 2 = W.
    READING of Prism's per-channel variance (Table 9 caption, "Eq. 1", not
    printed): a line along an axis is the set of valid tokens of a zone that
    share the other two coordinates.  For each line with at least two valid
    tokens and each channel, take the population variance of the values on the
    line; the zone's statistic is the plain mean of those over all such lines
    and all channels.  Returns [Zt, Zh, Zw]; 0 where no line qualifies.
    """
    inner = (1, 3, 5)[axis]
    mf = m.astype(f64)[..., None]
    n = mf.sum(axis=inner, keepdims=True)                      # valid tokens per line
    mean = (g * mf).sum(axis=inner, keepdims=True) / np.maximum(n, 1.0)
    var = (mf * (g - mean) ** 2).sum(axis=inner, keepdims=True) / np.maximum(n, 1.0)
    ok = (n >= 2.0)                                            # qualifying lines
    var = np.where(ok, var, 0.0)
    # mean over the lines (the other two in-zone axes) and the channels
    other = tuple(a for a in (1, 3, 5) if a != inner)
    num = var.sum(axis=(inner,) + other + (6,))
    cnt = ok.astype(f64).sum(axis=(inner,) + other) * g.shape[6]
    cnt = cnt[..., 0] if cnt.ndim == num.ndim + 1 else cnt
    return np.where(cnt > 0, num / np.maximum(cnt, 1.0), 0.0)


def a2v_norms(Qa: np.ndarray, Ka: np.ndarray, Va: np.ndarray) -> np.ndarray:
    """Per-token norm of the audio-to-video (A2V) cross-attention output
    (Prism, Abstract: the zone signals use feature norms from the
    audio-to-video cross-attention).

    READING (the pages give no formula): one attention head in which every
    video token's cross-attention query Qa_i attends to the audio tokens'
    keys Ka and values Va with scale 1/sqrt(Ca) and a softmax over the audio
    tokens; n_i = ||softmax(Qa_i Ka^T / sqrt(Ca)) Va||_2.
    Qa [B, N, Ca], Ka / Va [B, Na, Ca] (any float dtype) -> n [B, N] float64."""
    B, N, Ca = Qa.shape
    out = np.zeros((B, N), dtype=f64)
    for b in range(B):
        s = (Qa[b].astype(f64) @ Ka[b].astype(f64).T) / math.sqrt(Ca)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)
        out[b] = np.sqrt(((P @ Va[b].astype(f64)) ** 2).sum(axis=1))
    return out


def zone_stats(w, V: np.ndarray, a2v: np.ndarray) -> np.ndarray:
    """Per (b, h, zone) statistics, [B, H, Z, 8] float64:
    (var_v_T, var_v_H, var_v_W, var_n_T, var_n_H, var_n_W, nbar, n_valid),
    from the value features V [B, N, H, d] and the A2V cross-attention output
    a2v [B, N, Ca] (its per-token norms n_i = ||a2v_i||_2; see
    ``zone_stats_from_norms``)."""
    return zone_stats_from_norms(w, V, np.sqrt((a2v.astype(f64) ** 2).sum(axis=-1)))


def zone_stats_from_norms(w, V: np.ndarray, n: np.ndarray) -> np.ndarray:
    """Per (b, h, zone) statistics, [B, H, Z, 8] float64:
    (var_v_T, var_v_H, var_v_W, var_n_T, var_n_H, var_n_W, nbar, n_valid).

    * var_v_d: directional variance of the VALUE features of head h
      (Prism, Table 9 caption: the default uses value features; the query/key
      variants are ablations) -- ``line_variance`` along d.
    * n [B, N]: per-token norm of the audio-to-video cross-attention output
      (Prism, Abstract: feature norms from the A2V cross-attention).
      var_n_d: the same directional variance of the scalar map n (READING of
      the audio directional variance v_hat_{a,d} of Table 9's caption).
      nbar: mean of n over the zone's valid tokens (READING of the audio
      coupling gate's input, Table 9 caption).
    V: [B, N, H, d] (any float dtype; used as float64).
    """
    B, N, H, d = V.shape
    out = []
    for b in range(B):
        gn, m = _grid_views(np.asarray(n[b], dtype=f64)[:, None], w, 1)
        sn = np.stack([line_variance(gn, m, a) for a in range(3)], -1)    # [Zt,Zh,Zw,3]
        mf = m.astype(f64)
        cnt = mf.sum(axis=(1, 3, 5))
        nbar = np.where(cnt > 0, (gn[..., 0] * mf).sum(axis=(1, 3, 5)) / np.maximum(cnt, 1), 0.0)
        per_h = []
        for h in range(H):
            gv, _ = _grid_views(V[b, :, h, :].astype(f64), w, d)
            sv = np.stack([line_variance(gv, m, a) for a in range(3)], -1)
            st = np.concatenate([sv, sn, nbar[..., None], cnt[..., None]], -1)
            per_h.append(st.reshape(-1, 8))
        out.append(np.stack(per_h))
    return np.stack(out)


# --------------------------------------------------------------------------
# step 2: block shape per zone (Eq. 7) and token permutation
# --------------------------------------------------------------------------

# A2V norm maps that are constant over a zone (e.g. a zone where one audio
# token dominates the cross-attention) have no directional variance; what any
# arithmetic returns for them is round-off, and its ratios are meaningless.
# A directional variance whose sum is at most AUDIO_VAR_FLOOR * nbar^2 counts
# as zero: a spread of the norms below 1e-5 of their size, which a norm map
# computed in fp32 (relative error ~1e-7, variance ~1e-14 nbar^2 from
# rounding alone) cannot resolve.  Round-off of a constant map is ~1e-30
# nbar^2 in fp64; the zones of the synthetic grids that do vary have at least
# ~1e-3 nbar^2.
AUDIO_VAR_FLOOR = 1e-10


def guidance(w, st: np.ndarray, nbar_max: float) -> np.ndarray:
    """g_d for one zone from its statistics row st[8].

    READING (Prism, Table 9 caption names r_{v,d}, a_bar and v_hat_{a,d};
    Table 12 ablates each guidance):
      r_{v,d}     = var_v_d / sum_d var_v_d      (1/3 each when the sum is 0)
      v_hat_{a,d} = var_n_d / sum_d var_n_d      (1/3 each when there is no
                    variance: sum <= AUDIO_VAR_FLOOR * nbar^2)
      a_bar       = nbar / max over zones of nbar (0 when that max is 0)
      g_d = u_v r_{v,d} + u_a a_bar v_hat_{a,d} + eps
    with u_v, u_a the video/audio guidance switches.
    """
    sv, sn = st[0:3], st[3:6]
    r = sv / sv.sum() if sv.sum() > 0 else np.full(3, 1.0 / 3.0)
    no_var = not (sn.sum() > AUDIO_VAR_FLOOR * st[6] * st[6])
    vh = np.full(3, 1.0 / 3.0) if no_var else sn / sn.sum()
    abar = st[6] / nbar_max if nbar_max > 0 else 0.0
    uv = 1.0 if w.use_video else 0.0
    ua = 1.0 if w.use_audio else 0.0
    return uv * r + ua * abar * vh + w.eps


def menu_classes(menu: Sequence[Sequence[int]]) -> List[int]:
    """The block-size classes of a menu: its distinct token counts bT bH bW,
    ascending (Prism, Table 11: classes C_64, C_128, C_256 by token count)."""
    return sorted(set(int(b[0] * b[1] * b[2]) for b in menu))


def class_admissible(w, S: int) -> List[int]:
    """Admissible menu shapes of the class of S tokens."""
    return [k for k in admissible_shapes(w.menu, w.zone)
            if w.menu[k][0] * w.menu[k][1] * w.menu[k][2] == S]


def shape_costs(w, g: np.ndarray, S: int = None) -> Tuple[np.ndarray, np.ndarray]:
    """Eq. 7 (Prism, Table 10 caption: b*_d is proportional to g_d^-alpha).

    READING: with the token count fixed at S = bT bH bW (the zone's class;
    the workload's block size for a single-class menu), the continuous
    optimum is log2 b*_d = log2(S)/3 + alpha (mean_d log2 g_d - log2 g_d).
    Each admissible menu shape of that class is scored by
    sum_d (log2 b_d - log2 b*_d)^2.
    Returns (costs over those shapes, their menu indices)."""
    S = w.block if S is None else S
    lg = np.log2(g)
    lstar = math.log2(S) / 3.0 + w.alpha * (lg.mean() - lg)
    idx = class_admissible(w, S)
    costs = np.array([sum((math.log2(w.menu[k][dd]) - lstar[dd]) ** 2 for dd in range(3))
                      for k in idx], dtype=f64)
    return costs, np.array(idx)


SHAPE_TIE = 1e-4
CLASS_TIE = 1e-5


def zone_complexity(w, st_h: np.ndarray) -> np.ndarray:
    """Per-zone complexity c_z that picks the block-size class, for one
    (b, h): st_h [Z, 8] statistics rows.

    READING (Table 10 caption: thresholds tau_128 / tau_256 assign a block
    size class; Abstract: fine blocks where the content varies fast and
    couples strongly to the audio; the pages print no formula):
      c_z = u_v V_z / mean_z' V_z' + u_a a_bar_z,
    with V_z = sum_d var_v_d(z) (0 / 0 -> 0) and a_bar_z the audio gate."""
    V = st_h[:, 0:3].sum(axis=1)
    Vm = V.mean()
    nmax = st_h[:, 6].max()
    uv = 1.0 if w.use_video else 0.0
    ua = 1.0 if w.use_audio else 0.0
    rel = V / Vm if Vm > 0 else np.zeros_like(V)
    abar = st_h[:, 6] / nmax if nmax > 0 else np.zeros_like(V)
    return uv * rel + ua * abar


def zone_class(c: float, taus: Sequence[float]) -> int:
    """Class index (into menu_classes, ascending block size) of a zone of
    complexity c: the number of thresholds c is below, taus descending
    (tau_128 > tau_256: c >= tau_128 -> C_64, tau_256 <= c < tau_128 ->
    C_128, c < tau_256 -> C_256)."""
    return sum(1 for t in taus if c < t)


def zone_class_tokens(w, classes, cz: float, taus, n_real: float) -> int:
    """Token count of a zone's class.  READING: a class smaller than the
    tile (w.block, the tensor cores' row tile; two such blocks share one) is
    taken only by zones without padding, so that both halves of every shared
    tile are real; a zone with padding takes the smallest class of at least
    a tile instead."""
    S = classes[zone_class(cz, taus)]
    vol = w.zone[0] * w.zone[1] * w.zone[2]
    if S < w.block and n_real < vol:
        S = min(c for c in classes if c >= w.block)
    return S


def assign_shapes(w, stats: np.ndarray):
    """Shape id per (b, h, zone) -> (shape_id [B,H,Z] int, near_tie [B,H,Z] bool).

    A menu with several block-size classes first gives each zone its class
    (``zone_complexity`` against the thresholds ``w.class_tau``); then, in
    the class, the admissible shape of least Eq. 7 cost wins; an exact tie
    goes to the lowest menu index.  A zone whose best and second-best costs
    differ by less than SHAPE_TIE, or whose complexity lies within CLASS_TIE
    (relative) of a threshold, is flagged as a near tie (either decision is
    then accepted).  With per_head False, the video statistics are averaged
    over heads first and every head gets the same shape (Prism, Table 10
    caption ablates per-head shapes)."""
    B, H, Z, _ = stats.shape
    classes = menu_classes(w.menu)
    taus = tuple(getattr(w, "class_tau", ()) or ())
    if len(taus) != len(classes) - 1:
        raise ValueError("one threshold per class boundary expected")
    for S in classes:
        if not class_admissible(w, S):
            raise ValueError("no admissible shape for this zone")
    sid = np.zeros((B, H, Z), dtype=np.int64)
    tie = np.zeros((B, H, Z), dtype=bool)
    for b in range(B):
        for h in range(H):
            st_h = stats[b, h] if w.per_head else stats[b].mean(axis=0)
            nmax = st_h[:, 6].max()
            cz = zone_complexity(w, st_h) if taus else np.zeros(Z)
            for z in range(Z):
                S = zone_class_tokens(w, classes, cz[z], taus, st_h[z][7])
                costs, idx = shape_costs(w, guidance(w, st_h[z], nmax), S)
                k = int(np.argmin(costs))            # first minimum = lowest menu index
                sid[b, h, z] = idx[k]
                if len(costs) > 1:
                    srt = np.sort(costs)
                    tie[b, h, z] = (srt[1] - srt[0]) < SHAPE_TIE
                for t in taus:
                    tie[b, h, z] |= abs(cz[z] - t) <= CLASS_TIE * max(1.0, abs(t))
    return sid, tie


def line_variance_bound(g: np.ndarray, m: np.ndarray, axis: int, tau: float) -> np.ndarray:
    """How far ``line_variance`` of a scalar map (C = 1) can move when every
    value n_i is replaced by n_i (1 + e_i) with |e_i| <= tau.

    On a line of L values with mean mu the variance moves by
    (2/L) sum_i (n_i - mu) n_i e_i + (1/L) sum_i (n_i e_i)^2 - (mean of n_i e_i)^2,
    so by at most (2 tau / L) sum_i |n_i - mu| n_i + (tau^2 / L) sum_i n_i^2;
    the zone's statistic is the mean over its qualifying lines, and so is the
    bound.  Returns [Zt, Zh, Zw]."""
    inner = (1, 3, 5)[axis]
    mf = m.astype(f64)[..., None]
    n = mf.sum(axis=inner, keepdims=True)
    mean = (g * mf).sum(axis=inner, keepdims=True) / np.maximum(n, 1.0)
    lin = (mf * np.abs(g - mean) * np.abs(g)).sum(axis=inner, keepdims=True)
    sq = (mf * g * g).sum(axis=inner, keepdims=True)
    bnd = (2.0 * tau * lin + tau * tau * sq) / np.maximum(n, 1.0)
    ok = (n >= 2.0)
    bnd = np.where(ok, bnd, 0.0)
    other = tuple(a for a in (1, 3, 5) if a != inner)
    num = bnd.sum(axis=(inner,) + other + (6,))
    cnt = ok.astype(f64).sum(axis=(inner,) + other) * g.shape[6]
    cnt = cnt[..., 0] if cnt.ndim == num.ndim + 1 else cnt
    return np.where(cnt > 0, num / np.maximum(cnt, 1.0), 0.0)


def _shape_decision_reachable(w, st: np.ndarray, nmax: float, dvar: np.ndarray,
                              tau: float, S: int = None, cz: float = 0.0) -> bool:
    """True when the shape chosen from the statistics row ``st`` could change
    if the audio statistics came from norms off by at most tau relative:
    var_n_d by at most dvar[d], nbar and the zones' max nbar by at most tau
    relative.  Every bound below is a worst case over that box (first order
    where the quantity is linear in the perturbation, exact otherwise)."""
    if not w.use_audio:
        return False
    sv, sn, nbar = st[0:3], st[3:6], st[6]
    ssv, ssn, dss = sv.sum(), sn.sum(), dvar.sum()
    # the audio-direction floor: the decision "no direction" must be the same
    # everywhere in the box
    fl_lo = AUDIO_VAR_FLOOR * (nbar * (1.0 - tau)) ** 2
    fl_hi = AUDIO_VAR_FLOOR * (nbar * (1.0 + tau)) ** 2
    if ssn - dss > fl_hi:
        vh = sn / ssn
        dvh = (dvar + vh * dss) / (ssn - dss)
    elif ssn + dss <= fl_lo:
        vh, dvh = np.full(3, 1.0 / 3.0), np.zeros(3)
    else:
        return True
    abar = nbar / nmax if nmax > 0 else 0.0
    dab = abar * 2.0 * tau / (1.0 - tau)
    # the class: the complexity moves with the gate only
    for t in tuple(getattr(w, "class_tau", ()) or ()):
        if abs(cz - t) <= dab + CLASS_TIE * max(1.0, abs(t)):
            return True
    r = sv / ssv if ssv > 0 else np.full(3, 1.0 / 3.0)
    uv = 1.0 if w.use_video else 0.0
    g = uv * r + abar * vh + w.eps
    dg = dab * (vh + dvh) + abar * dvh
    if np.any(dg >= g):
        return True
    dL = np.log2(g / (g - dg))                         # largest move of log2 g_d
    dl = abs(w.alpha) * (dL.sum() / 3.0 + dL / 3.0)    # of log2 b*_d: |mean - own|
    costs, idx = shape_costs(w, g, S)
    kb = int(np.argmin(costs))
    lb = np.array([[math.log2(e) for e in w.menu[k]] for k in idx])
    for q in range(len(idx)):
        if q == kb:
            continue
        reach = 2.0 * (np.abs(lb[q] - lb[kb]) * dl).sum()
        if costs[q] - costs[kb] < SHAPE_TIE + reach:
            return True
    return False


def norm_sensitive_zones(w, n: np.ndarray, stats: np.ndarray, tau: float) -> np.ndarray:
    """Zones whose block shape could change if every A2V norm n_i [B, N] were
    off by up to tau * n_i (a norm map computed in another precision): the
    near ties of a path whose norms carry that error.  stats [B, H, Z, 8] are
    the statistics from n itself.  Returns bool [B, H, Z]."""
    B, H, Z, _ = stats.shape
    flags = np.zeros((B, H, Z), dtype=bool)
    for b in range(B):
        gn, m = _grid_views(np.asarray(n[b], dtype=f64)[:, None], w, 1)
        dv = np.stack([line_variance_bound(gn, m, a, tau) for a in range(3)], -1).reshape(-1, 3)
        classes = menu_classes(w.menu)
        taus = tuple(getattr(w, "class_tau", ()) or ())
        for h in range(H):
            st_h = stats[b, h] if w.per_head else stats[b].mean(axis=0)
            nmax = st_h[:, 6].max()
            cz = zone_complexity(w, st_h) if taus else np.zeros(Z)
            for z in range(Z):
                S = zone_class_tokens(w, classes, cz[z], taus, st_h[z][7])
                flags[b, h, z] = _shape_decision_reachable(w, st_h[z], nmax, dv[z], tau, S,
                                                           cz[z])
    return flags


def slot_tokens(w) -> int:
    """Granularity of the block table: the tile (w.block), or half of it when
    the menu has a class of half a tile."""
    return min([w.block] + menu_classes(w.menu))


def build_permutation(w, shape_id: np.ndarray, table: bool = False):
    """Token order for every (b, h): zones in raster (zt, zh, zw) order, the
    zone's blocks in raster order of its chosen shape, and inside a block its
    valid tokens first in (t, h, w) raster order, then its padding slots.

    READING (Prism, Abstract: tokens inside a block stay together; the pages do
    not give an order).  A block of S tokens fills S / w.block consecutive
    tiles of w.block slots (one tile when the menu has a single class of
    w.block tokens; two blocks of half a tile share one).  Returns perm
    [B,H,Np] (slot -> real token, -1 for a padding slot), inv [B,H,N]
    (token -> slot), n_valid [B,H,nb] (real tokens in each tile: a block's
    real tokens sit at its start, so they fill its first tiles); with
    ``table`` also, per unit of ``slot_tokens(w)`` tokens, units [B,H,nu]
    (a block's unit count at its first unit, 0 on the units that continue
    it) and n_block [B,H,nu] (a block's real tokens at its first unit, 0
    elsewhere)."""
    B, H, Z = shape_id.shape
    Tp, Hp, Wp = padded_grid(w.T, w.Hg, w.W, w.zone)
    zT, zH, zW = w.zone
    nzT, nzH, nzW = Tp // zT, Hp // zH, Wp // zW
    T_ = w.block
    U = slot_tokens(w)
    Np = Tp * Hp * Wp
    nb = Np // T_
    perm = np.full((B, H, Np), -1, dtype=np.int64)
    inv = np.full((B, H, w.N), -1, dtype=np.int64)
    nvalid = np.zeros((B, H, nb), dtype=np.int64)
    units = np.zeros((B, H, Np // U), dtype=np.int64)
    nblock = np.zeros((B, H, Np // U), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            slot = 0
            for z in range(Z):
                zt, zh, zw = z // (nzH * nzW), (z // nzW) % nzH, z % nzW
                bT, bH, bW = w.menu[int(shape_id[b, h, z])]
                S = bT * bH * bW
                for it in range(zT // bT):
                    for ih in range(zH // bH):
                        for iw in range(zW // bW):
                            toks = []
                            for t in range(bT):
                                for y in range(bH):
                                    for x in range(bW):
                                        tt = zt * zT + it * bT + t
                                        yy = zh * zH + ih * bH + y
                                        xx = zw * zW + iw * bW + x
                                        if tt < w.T and yy < w.Hg and xx < w.W:
                                            toks.append((tt * w.Hg + yy) * w.W + xx)
                            for k, n in enumerate(toks):
                                perm[b, h, slot + k] = n
                                inv[b, h, n] = slot + k
                            units[b, h, slot // U] = S // U
                            nblock[b, h, slot // U] = len(toks)
                            slot += S
            for t in range(nb):
                nvalid[b, h, t] = int((perm[b, h, t * T_:(t + 1) * T_] >= 0).sum())
    if table:
        return perm, inv, nvalid, units, nblock
    return perm, inv, nvalid


def pool_blocks(Xp: np.ndarray, tiles: np.ndarray, n_block: np.ndarray, T_: int) -> np.ndarray:
    """Block-level feature of blocks that span one or more units of T_
    slots: the mean of the block's real tokens (its first n_block slots),
    stored at its first unit; 0 on continuation units and for blocks without
    real tokens."""
    B, H, Np, d = Xp.shape
    nb = Np // T_
    out = np.zeros((B, H, nb, d), dtype=f64)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                nv = int(n_block[b, h, i])
                if tiles[b, h, i] > 0 and nv > 0:
                    out[b, h, i] = Xp[b, h, i * T_:i * T_ + nv].sum(axis=0) / nv
    return out


def expand_lists_masked(L, units: np.ndarray, U: int, T_: int):
    """Block lists over first units (of U slots) -> lists over tiles of T_ =
    2U slots with, per entry, a 4-bit mask of the sub-tile pairs that are NOT
    selected: bit 2 qh + kh for the query tile's half qh and the key tile's
    half kh (0: the whole tile pair is selected).  A tile pair is listed when
    any of its four halves is selected."""
    per = T_ // U
    nu = len(units)
    nt = nu // per
    start = np.zeros(nu, dtype=np.int64)                 # first unit of every unit's block
    i = 0
    while i < nu:
        n = max(1, int(units[i]))
        start[i:i + n] = i
        i += n
    sel = [set() if L[int(start[u])] is None else set(int(j) for j in L[int(start[u])])
           for u in range(nu)]
    lists, masks = [], []
    for t in range(nt):
        cols, ms = [], []
        for v in range(nt):
            bits = 0
            for qh in range(per):
                for kh in range(per):
                    if int(start[v * per + kh]) in sel[t * per + qh]:
                        bits |= 1 << (qh * per + kh)
            if bits:
                cols.append(v)
                ms.append((~bits) & ((1 << (per * per)) - 1))
        lists.append(np.array(cols, dtype=np.int64))
        masks.append(np.array(ms, dtype=np.int64))
    return lists, masks


def _rows_of(Xp_bh, blocks, U, n_block_bh):
    """Real rows of the given blocks (first units), concatenated in order."""
    return np.concatenate([Xp_bh[int(j) * U: int(j) * U + int(n_block_bh[int(j)])] for j in blocks],
                          axis=0)


def attn_blocks(Qp, Kp, Vp, units, n_block, L, U, scale, dOp=None, o_bf16=False):
    """Block-sparse attention at block level for blocks of any size (units of
    U slots): every real query token of block i attends to every real token of
    the blocks in L[(b, h)][i] (Prism, Fig. 2 caption; readings as
    ``attn_fwd_row``), and with dOp its VJP (as ``attn_bwd_row``; ``o_bf16``
    forms D from O rounded to bf16).  Returns (Op, lse) or
    (Op, lse, dQp, dKp, dVp), all in the permuted layout."""
    B, H, Np, d = Qp.shape
    Op = np.zeros((B, H, Np, d), dtype=f64)
    lse = np.zeros((B, H, Np), dtype=f64)
    if dOp is not None:
        dQ, dK, dV = (np.zeros((B, H, Np, d), dtype=f64) for _ in range(3))
    for (b, h), Lbh in L.items():
        nb_ = n_block[b, h]
        for i, sel in enumerate(Lbh):
            if sel is None or len(sel) == 0 or units[b, h, i] == 0 or nb_[i] == 0:
                continue
            r0, nq = i * U, int(nb_[i])
            q = Qp[b, h, r0:r0 + nq].astype(f64)
            k = _rows_of(Kp[b, h], sel, U, nb_).astype(f64)
            v = _rows_of(Vp[b, h], sel, U, nb_).astype(f64)
            s = (q @ k.T) * scale
            mx = s.max(axis=1, keepdims=True)
            e = np.exp(s - mx)
            l = e.sum(axis=1, keepdims=True)
            P = e / l
            o = P @ v
            Op[b, h, r0:r0 + nq] = o
            lse[b, h, r0:r0 + nq] = (mx + np.log(l))[:, 0]
            if dOp is None:
                continue
            do = dOp[b, h, r0:r0 + nq].astype(f64)
            dv = P.T @ do
            dP = do @ v.T
            Dr = (do * (round_bf16(o) if o_bf16 else o)).sum(axis=1, keepdims=True)
            dS = P * (dP - Dr)
            dQ[b, h, r0:r0 + nq] = (dS @ k) * scale
            dk = (dS.T @ q) * scale
            off = 0
            for j in sel:
                nv = int(nb_[int(j)])
                dK[b, h, int(j) * U:int(j) * U + nv] += dk[off:off + nv]
                dV[b, h, int(j) * U:int(j) * U + nv] += dv[off:off + nv]
                off += nv
    if dOp is None:
        return Op, lse
    return Op, lse, dQ, dK, dV


def expand_lists(L, tiles: np.ndarray):
    """Block lists over first tiles -> lists over tiles: every tile of a
    query block gets the tiles of every key block its block selected,
    ascending.  L [nb] (lists at first tiles; other entries ignored),
    tiles [nb] (one (b, h))."""
    nb = len(tiles)
    out = [np.zeros(0, dtype=np.int64) for _ in range(nb)]
    for i in range(nb):
        n = int(tiles[i])
        if n == 0 or L[i] is None:
            continue
        sel = np.concatenate([np.arange(int(j), int(j) + int(tiles[int(j)])) for j in L[i]]
                             ) if len(L[i]) else np.zeros(0, dtype=np.int64)
        for q in range(n):
            out[i + q] = sel.astype(np.int64)
    return out


def permute(X: np.ndarray, perm: np.ndarray) -> np.ndarray:
    """X [B, N, H, d] -> Xp [B, H, Np, d] in block order; padding slots are 0."""
    B, N, H, d = X.shape
    Np = perm.shape[2]
    Xp = np.zeros((B, H, Np, d), dtype=f64)
    for b in range(B):
        for h in range(H):
            ok = perm[b, h] >= 0
            Xp[b, h, ok] = X[b, perm[b, h, ok], h].astype(f64)
    return Xp


def unpermute(Xp: np.ndarray, inv: np.ndarray) -> np.ndarray:
    """Inverse of ``permute``: Xp [B, H, Np, d] -> X [B, N, H, d]."""
    B, H, Np, d = Xp.shape
    N = inv.shape[2]
    X = np.zeros((B, N, H, d), dtype=f64)
    for b in range(B):
        for h in range(H):
            X[b, :, h] = Xp[b, h, inv[b, h]]
    return X


# --------------------------------------------------------------------------
# step 3: block-level features and scores
# --------------------------------------------------------------------------

def pool(Xp: np.ndarray, n_valid: np.ndarray, S: int) -> np.ndarray:
    """Block-level feature = mean of the block's valid tokens (READING of the
    pages' block-level features, Prism Abstract; valid slots come first in a
    block).  Xp [B,H,Np,d], n_valid [B,H,nb] -> [B,H,nb,d]; 0 for empty blocks."""
    B, H, Np, d = Xp.shape
    nb = Np // S
    out = np.zeros((B, H, nb, d), dtype=f64)
    blocks = Xp.reshape(B, H, nb, S, d)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                nv = int(n_valid[b, h, i])
                if nv > 0:
                    out[b, h, i] = blocks[b, h, i, :nv].sum(axis=0) / nv
    return out


def block_scores(Qbar: np.ndarray, Kbar: np.ndarray, d: int) -> np.ndarray:
    """Query-block x key-block score Qbar Kbar^T / sqrt(d) for one (b, h)
    (Prism, Fig. 2 caption: block-sparse attention over block scores; READING:
    the usual 1/sqrt(d) scale, no bias)."""
    return (Qbar @ Kbar.T) / math.sqrt(d)


# --------------------------------------------------------------------------
# step 4: hybrid Top-k / Top-p selection
# --------------------------------------------------------------------------

TIE_SCORE = 1e-6
TIE_MASS = 1e-6


def topp_count(probs_sorted: np.ndarray, p: float) -> int:
    """Top-p (Prism, Table 7 caption): the smallest number of key blocks, taken
    in decreasing weight, whose cumulative weight is strictly greater than p;
    all of them when no prefix gets there.  READING: for p >= 1 no prefix can
    exceed p (the weights sum to 1), so every candidate is kept; this is
    stated explicitly so that rounding of the running sum cannot end early."""
    if p >= 1.0:
        return len(probs_sorted)
    acc = 0.0
    for m, q in enumerate(probs_sorted, start=1):
        acc += q
        if acc > p:
            return m
    return len(probs_sorted)


def hybrid_select_probs(probs: np.ndarray, order: np.ndarray, kf: int, p: float) -> int:
    """Number of blocks kept for one query block given its candidates'
    probabilities and their ranking: at least the Top-k floor (capped at the
    candidate count) and at least the Top-p count (READING of Prism's hybrid
    rule, Abstract and Fig. 2 caption: the count varies per query block)."""
    nv = len(order)
    mp = topp_count(probs[order], p)
    return max(min(kf, nv), mp)


def hybrid_select_row(scores: np.ndarray, valid: np.ndarray, kf: int, p: float):
    """Selection for one query block.

    scores: [nb] block scores, valid: [nb] bool (key block has valid tokens).
    Candidates are ranked by (score descending, block index ascending); their
    weights are the softmax of the scores over the candidates.
    Returns (ascending list of selected block ids, near_tie flag)."""
    cand = np.nonzero(valid)[0]
    if cand.size == 0:
        return np.zeros(0, dtype=np.int64), False
    s = scores[cand]
    order = np.lexsort((cand, -s))                    # primary -s, secondary index
    e = np.exp(s - s.max())
    probs = e / e.sum()
    m = hybrid_select_probs(probs, order, kf, p)
    sel = np.sort(cand[order[:m]])
    # near tie: the boundary scores are within TIE_SCORE, or a cumulative mass
    # at the Top-p boundary is within TIE_MASS of p
    flag = False
    if m < cand.size:
        a, b = s[order[m - 1]], s[order[m]]
        flag |= abs(a - b) <= TIE_SCORE * max(1.0, abs(a))
    cum = np.cumsum(probs[order])
    mp = topp_count(probs[order], p)
    flag |= abs(cum[mp - 1] - p) <= TIE_MASS
    if mp >= 2:
        flag |= abs(cum[mp - 2] - p) <= TIE_MASS
    return sel, bool(flag)


def select_blocks(w, Qbar: np.ndarray, Kbar: np.ndarray, n_valid: np.ndarray, heads=None,
                  rows=None):
    """Hybrid selection for every (b, h, query block).

    Returns (lists, flags): lists[(b, h)][i] = ascending selected key blocks
    (empty for an empty query block), flags[(b, h)][i] = near-tie flag.
    ``heads`` / ``rows`` restrict the work to a sample."""
    B, H, nb, d = Qbar.shape
    lists, flags = {}, {}
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            S = block_scores(Qbar[b, h], Kbar[b, h], d)
            valid = n_valid[b, h] > 0
            L, F = [None] * nb, [False] * nb
            for i in (range(nb) if rows is None else rows):
                if not valid[i]:
                    L[i] = np.zeros(0, dtype=np.int64)
                    continue
                L[i], F[i] = hybrid_select_row(S[i], valid, w.topk_floor, w.topp)
            lists[(b, h)], flags[(b, h)] = L, F
    return lists, flags


# --------------------------------------------------------------------------
# step 5: block-sparse attention, forward and backward
# --------------------------------------------------------------------------

def _gather_keys(Xp_bh: np.ndarray, n_valid_bh: np.ndarray, sel, S: int) -> np.ndarray:
    """Valid rows of the selected key blocks, concatenated in list order."""
    return np.concatenate([Xp_bh[j * S: j * S + int(n_valid_bh[j])] for j in sel], axis=0)


def attn_fwd_row(Qp_bh, Kp_bh, Vp_bh, n_valid_bh, i: int, sel, S: int, scale: float):
    """Exact softmax attention of query block i over the valid tokens of its
    selected key blocks (Prism, Fig. 2 caption; READING: bidirectional, no
    dropout, no correction for the dropped blocks).
    Returns (O rows [S, d] with padding rows 0, natural-log LSE [S])."""
    d = Qp_bh.shape[1]
    q = Qp_bh[i * S:(i + 1) * S].astype(f64)
    k = _gather_keys(Kp_bh, n_valid_bh, sel, S).astype(f64)
    v = _gather_keys(Vp_bh, n_valid_bh, sel, S).astype(f64)
    s = (q @ k.T) * scale
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    l = e.sum(axis=1, keepdims=True)
    o = (e / l) @ v
    lse = (mx + np.log(l))[:, 0]
    nv = int(n_valid_bh[i])
    o[nv:] = 0.0
    lse[nv:] = 0.0
    return o, lse


def attn_fwd(w, Qp, Kp, Vp, n_valid, lists, scale):
    """Forward over every (b, h, query block) present in ``lists``."""
    B, H, Np, d = Qp.shape
    S = w.block
    Op = np.zeros((B, H, Np, d), dtype=f64)
    lse = np.zeros((B, H, Np), dtype=f64)
    for (b, h), L in lists.items():
        for i, sel in enumerate(L):
            if sel is None or len(sel) == 0:
                continue
            o, l = attn_fwd_row(Qp[b, h], Kp[b, h], Vp[b, h], n_valid[b, h], i, sel, S, scale)
            Op[b, h, i * S:(i + 1) * S] = o
            lse[b, h, i * S:(i + 1) * S] = l
    return Op, lse


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even: 8 significant bits),
    returned as float64.  Done on the float64 bit pattern: keep the sign, the
    exponent and the top 7 fraction bits, rounding on the 45 bits below."""
    u = np.ascontiguousarray(a, dtype=f64).view(np.uint64)
    low = u & np.uint64((1 << 45) - 1)
    keep = u >> np.uint64(45)
    half = np.uint64(1 << 44)
    up = (low > half) | ((low == half) & ((keep & np.uint64(1)) == np.uint64(1)))
    r = (keep + up.astype(np.uint64)) << np.uint64(45)
    return r.view(f64).reshape(np.shape(a))


def attn_bwd_row(Qp_bh, Kp_bh, Vp_bh, dOp_bh, n_valid_bh, i, sel, S, scale, o_bf16=False,
                 abs_terms=False, o_given=None):
    """VJP of ``attn_fwd_row`` (Prism trains through this attention: Table 2
    caption -- it replaces video self-attention during training).  Gradients
    flow only through the attention; the discrete steps are constants.
    Returns (dq [S, d], dk [rows, d], dv [rows, d]) with dk/dv in the order of
    ``_gather_keys``.

    The VJP's row term D = rowsum(dO * O) (equal to sum_j P_ij dP_ij) is formed
    from O itself.  READING of the boundary: the backward entry point takes
    the forward's output O as the forward stores it, in bf16; with
    ``o_bf16`` D is formed from O rounded to bf16, which is what a backward
    given that stored O computes; ``o_given`` ([S, d]) forms D from that O
    instead (a backward handed some other forward output).  The default
    (exact O) is the plain VJP.

    ``abs_terms`` also returns how far dq and dk move, per element, when the O
    that D is formed from carries the errors of a forward that rounds to bf16
    (unit roundoff u): P rounded before the P V product moves O_ic by at most
    u (P |V|)_ic, and storing O moves it by at most u |O_ic|, so D_i moves by
    at most u b_i with b_i = sum_c |dO_ic| (|O_ic| + (P |V|)_ic).  D enters
    dq_i as -scale D_i (P K)_i and dk_j as -scale sum_i D_i P_ij Q_i, so the
    returned sizes (per unit u) are scale b_i |(P K)_ic| for dq and
    scale sum_i b_i P_ij |Q_ic| for dk.  Rows whose softmax is nearly one-hot
    make dq and dk cancel to about these sizes times u."""
    q = Qp_bh[i * S:(i + 1) * S].astype(f64)
    k = _gather_keys(Kp_bh, n_valid_bh, sel, S).astype(f64)
    v = _gather_keys(Vp_bh, n_valid_bh, sel, S).astype(f64)
    do = dOp_bh[i * S:(i + 1) * S].astype(f64).copy()
    nv = int(n_valid_bh[i])
    do[nv:] = 0.0                                     # padding query rows carry no gradient
    s = (q @ k.T) * scale
    e = np.exp(s - s.max(axis=1, keepdims=True))
    P = e / e.sum(axis=1, keepdims=True)
    o = P @ v
    dv = P.T @ do
    dP = do @ v.T
    if o_given is not None:
        o_used = np.asarray(o_given, dtype=f64)
    else:
        o_used = round_bf16(o) if o_bf16 else o
    Dr = (do * o_used).sum(axis=1, keepdims=True)
    dS = P * (dP - Dr)
    dq = (dS @ k) * scale
    dk = (dS.T @ q) * scale
    dq[nv:] = 0.0
    if abs_terms:
        b = (np.abs(do) * (np.abs(o) + P @ np.abs(v))).sum(axis=1, keepdims=True)
        dq_abs = scale * b * np.abs(P @ k)
        dq_abs[nv:] = 0.0
        return dq, dk, dv, dq_abs, scale * ((P * b).T @ np.abs(q))
    return dq, dk, dv


def attn_bwd(w, Qp, Kp, Vp, dOp, n_valid, lists, scale, rows_only=None, o_bf16=False,
             abs_terms=False):
    """Backward over every (b, h, query block) in ``lists``; returns permuted
    dQp, dKp, dVp [B, H, Np, d] (float64).  ``rows_only`` restricts the query
    blocks that are processed (dK/dV then hold partial sums); ``o_bf16`` and
    ``abs_terms`` as in ``attn_bwd_row`` (with ``abs_terms`` two more arrays,
    the summed sizes of the dQ and dK terms, are returned)."""
    B, H, Np, d = Qp.shape
    S = w.block
    dQ = np.zeros((B, H, Np, d), dtype=f64)
    dK = np.zeros((B, H, Np, d), dtype=f64)
    dV = np.zeros((B, H, Np, d), dtype=f64)
    if abs_terms:
        aQ = np.zeros((B, H, Np, d), dtype=f64)
        aK = np.zeros((B, H, Np, d), dtype=f64)
    for (b, h), L in lists.items():
        for i, sel in enumerate(L):
            if sel is None or len(sel) == 0:
                continue
            if rows_only is not None and i not in rows_only:
                continue
            r = attn_bwd_row(Qp[b, h], Kp[b, h], Vp[b, h], dOp[b, h], n_valid[b, h],
                             i, sel, S, scale, o_bf16, abs_terms)
            dq, dk, dv = r[:3]
            dQ[b, h, i * S:(i + 1) * S] += dq
            if abs_terms:
                aQ[b, h, i * S:(i + 1) * S] += r[3]
            off = 0
            for j in sel:
                nv = int(n_valid[b, h, j])
                dK[b, h, j * S: j * S + nv] += dk[off: off + nv]
                dV[b, h, j * S: j * S + nv] += dv[off: off + nv]
                if abs_terms:
                    aK[b, h, j * S: j * S + nv] += r[4][off: off + nv]
                off += nv
    if abs_terms:
        return dQ, dK, dV, aQ, aK
    return dQ, dK, dV


def attn_bwd_key_blocks(Qp_bh, Kp_bh, Vp_bh, dOp_bh, n_valid_bh, L, key_blocks, S, scale,
                        o_bf16=False, abs_terms=False):
    """dK and dV of the key blocks ``key_blocks`` of one (b, h): the same VJP
    as ``attn_bwd_row`` summed over every query block whose list L[i] holds
    one of them, with only those key blocks' columns formed in full (each
    query row still needs its whole softmax for P and its whole O for D).
    Returns {j: (dK_j [S, d], dV_j [S, d])}, rows past n_valid[j] zero; with
    ``abs_terms`` {j: (dK_j, dV_j, dK_abs_j)}, dK_abs_j the sizes of
    ``attn_bwd_row`` (scale sum_i b_i P_ij |Q_i|, per unit roundoff of the O
    that D is formed from) over the same query blocks."""
    d = Qp_bh.shape[1]
    want = set(int(j) for j in key_blocks)
    out = {j: (np.zeros((S, d)), np.zeros((S, d))) + ((np.zeros((S, d)),) if abs_terms else ())
           for j in want}
    for i, sel in enumerate(L):
        if sel is None or len(sel) == 0 or not want.intersection(int(j) for j in sel):
            continue
        q = Qp_bh[i * S:(i + 1) * S].astype(f64)
        k = _gather_keys(Kp_bh, n_valid_bh, sel, S).astype(f64)
        v = _gather_keys(Vp_bh, n_valid_bh, sel, S).astype(f64)
        do = dOp_bh[i * S:(i + 1) * S].astype(f64).copy()
        do[int(n_valid_bh[i]):] = 0.0
        s = (q @ k.T) * scale
        e = np.exp(s - s.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)
        o = P @ v
        Dr = (do * (round_bf16(o) if o_bf16 else o)).sum(axis=1, keepdims=True)
        if abs_terms:
            b = (np.abs(do) * (np.abs(o) + P @ np.abs(v))).sum(axis=1, keepdims=True)
        off = 0
        for j in sel:
            nv = int(n_valid_bh[j])
            j = int(j)
            if j in want:
                Pj = P[:, off:off + nv]
                dSj = Pj * (do @ v[off:off + nv].T - Dr)
                out[j][0][:nv] += (dSj.T @ q) * scale
                out[j][1][:nv] += Pj.T @ do
                if abs_terms:
                    out[j][2][:nv] += ((Pj * b).T @ np.abs(q)) * scale
            off += nv
    return out


def csc_from_lists(L, nb: int):
    """Key block -> ascending list of the query blocks that selected it."""
    cols = [[] for _ in range(nb)]
    for i, sel in enumerate(L):
        if sel is None:
            continue
        for j in sel:
            cols[int(j)].append(i)
    return [np.array(c, dtype=np.int64) for c in cols]


# --------------------------------------------------------------------------
# independent references (pins)
# --------------------------------------------------------------------------

def dense_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Plain softmax attention in the original token order, one query at a
    time: Q, K, V [N, d] -> O [N, d]."""
    N = Q.shape[0]
    O = np.zeros_like(Q, dtype=f64)
    for n in range(N):
        s = K.astype(f64) @ Q[n].astype(f64) * scale
        e = np.exp(s - s.max())
        O[n] = (e[:, None] * V.astype(f64)).sum(axis=0) / e.sum()
    return O


def masked_attention(Q, K, V, mask, scale, dO=None):
    """Softmax attention of every query over the keys its row of ``mask``
    allows (original token order), and its VJP when dO is given.
    Q, K, V, dO [N, d]; mask [N, N] bool.  Returns O or (O, dQ, dK, dV)."""
    Q, K, V = Q.astype(f64), K.astype(f64), V.astype(f64)
    s = np.where(mask, (Q @ K.T) * scale, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    e = np.where(mask, np.exp(s - mx), 0.0)
    P = e / e.sum(axis=1, keepdims=True)
    O = P @ V
    if dO is None:
        return O
    dO = dO.astype(f64)
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - (dO * O).sum(axis=1, keepdims=True))
    return O, (dS @ K) * scale, (dS.T @ Q) * scale, dV


# --------------------------------------------------------------------------
# whole path
# --------------------------------------------------------------------------

def run(w, Q, K, V, a2v, dO=None, heads=None):
    """The whole hot path on one batch, every step in the pages' order.
    Inputs in [B, N, H, d] / [B, N, Ca] (any float dtype); returns a dict of
    every intermediate and output in float64 / int64.  Blocks of a class
    larger than w.block span several tiles: selection runs over blocks
    (their first tiles), and the attention over the tiles of the selected
    blocks (``expand_lists``).  With a class of half a tile the block table
    is kept per half tile, the attention runs at block level
    (``attn_blocks``) and ``lists`` holds the tile lists with their sub-tile
    masks (``expand_lists_masked``)."""
    stats = zone_stats(w, V, a2v)
    sid, stie = assign_shapes(w, stats)
    perm, inv, nval, tiles, nblk = build_permutation(w, sid, table=True)
    U = slot_tokens(w)
    Qp, Kp, Vp = permute(Q, perm), permute(K, perm), permute(V, perm)
    Qb, Kb = pool_blocks(Qp, tiles, nblk, U), pool_blocks(Kp, tiles, nblk, U)
    blists, flags = select_blocks(w, Qb, Kb, nblk, heads=heads)
    scale = 1.0 / math.sqrt(w.d)
    if U < w.block:
        # blocks of half a tile: attention at block level; the tile lists with
        # their sub-tile masks are what the tensor-core kernels walk
        lists = {(b, h): expand_lists_masked(L, tiles[b, h], U, w.block)
                 for (b, h), L in blists.items()}
        dOp = permute(dO, perm) if dO is not None else None
        r = attn_blocks(Qp, Kp, Vp, tiles, nblk, blists, U, scale, dOp=dOp)
        Op, lse = r[0], r[1]
    else:
        lists = {(b, h): expand_lists(L, tiles[b, h]) for (b, h), L in blists.items()}
        Op, lse = attn_fwd(w, Qp, Kp, Vp, nval, lists, scale)
    res = dict(stats=stats, shape_id=sid, shape_tie=stie, perm=perm, inv=inv, n_valid=nval,
               tiles=tiles, n_block=nblk, Qp=Qp, Kp=Kp, Vp=Vp, Qbar=Qb, Kbar=Kb,
               block_lists=blists, lists=lists, flags=flags, Op=Op, lse=lse,
               O=unpermute(Op, inv), scale=scale)
    if dO is not None:
        if U < w.block:
            dQp, dKp, dVp = r[2], r[3], r[4]
        else:
            dOp = permute(dO, perm)
            dQp, dKp, dVp = attn_bwd(w, Qp, Kp, Vp, dOp, nval, lists, scale)
        res.update(dOp=dOp, dQp=dQp, dKp=dKp, dVp=dVp, dQ=unpermute(dQp, inv),
                   dK=unpermute(dKp, inv), dV=unpermute(dVp, inv))
    return res

"""Step-by-step comparison of the CUDA path (through the C ABI) with the CPU
oracle on the same seeded inputs.

Contract (checked per step):
  * zone statistics: relative 2e-5 of the column's scale (fp32 vs fp64);
  * shape ids: identical, except zones the oracle flags as near ties (either
    shape is then accepted and the CUDA choice is carried into the oracle);
  * perm / inv / n_valid and the permuted Q, K, V: bit-exact;
  * block means: |(hi + lo) - oracle| <= 1e-11 max(1, |mean|);
  * block lists: identical per query block, except rows the oracle flags as
    near ties (then the CUDA list is carried into the oracle);
  * CSC lists: exactly the transpose of the CSR lists;
  * attention: max|gpu - ref| / max|ref| per head <= 2e-2 for O and <= 5e-2
    for dQ, dK, dV (bf16 tensor-core arithmetic against fp64).  The oracle's
    backward forms its row term D = rowsum(dO * O) from its own O rounded to
    bf16 (o_bf16): the backward entry point receives O as the forward stores
    it, in bf16.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from content_adaptive_block_02_b300 import prism, synth
from oracle import prism_oracle as orc

O_TOL = 2e-2
G_TOL = 5e-2
# bf16 unit roundoff 2^-9, twice: the forward rounds P before the P V product
# and O when it stores it (u |O| + u P|V|, the oracle's bound terms), and a
# forward that walks the keys in ranges also rounds each range's partial O
# (another u P|V|)
TERMS_U = 2.0 ** -8
# relative tolerance of dQ and dK on inputs whose softmax rows are nearly
# one-hot (grad_scale "terms"): there dQ and dK cancel to about 1e-6 of their
# ingredients, and the forward's bf16 roundings of P and O, carried through
# D = rowsum(dO * O), leave them with errors of several percent (8 % measured
# for dK, 4 % for dQ on the white-field stress input)
ILL_COND_TOL = 0.15
# relative error allowed on the A2V norms the device computes (fp32 logits
# and softmax, P V with P in two fp16 terms)
TAU_N = 4e-6


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(w, inputs, attn_kernel=0, shape_id=None, key_chunk_blocks=0, fused_a2v=False):
    dev = torch.device("cuda")
    x = {k: inputs[k].to(dev) for k in ("Q", "K", "V", "a2v", "dO", "qa", "audio")}
    att = prism.PrismAttention(w, dev, attn_kernel=attn_kernel, key_chunk_blocks=key_chunk_blocks)
    sid = None if shape_id is None else torch.as_tensor(shape_id, dtype=torch.uint8).to(dev)
    if fused_a2v:
        O = att.forward(x["Q"], x["K"], x["V"], qa=x["qa"], audio=x["audio"], shape_id=sid)
    else:
        O = att.forward(x["Q"], x["K"], x["V"], x["a2v"], shape_id=sid)
    dQ, dK, dV = att.backward(x["dO"])
    torch.cuda.synchronize()
    assert att.status() == 0, "device status word set"
    g = {k: v.cpu() for k, v in att.perm_out.items()}
    g.update({k: v.cpu() for k, v in att.lists.items()})
    if fused_a2v:
        g["nrm"] = att.nrm.cpu()
    sz = att.plan.sz
    if sz.half_tile:
        # the sub-tile masks prism_block_select left in the workspace
        nnz = int(att.lists["row_ptr"][-1].item())
        g["csr_mask"] = att.ws[sz.ws_csr_mask:sz.ws_csr_mask + nnz].cpu()
        g["csc_mask"] = att.ws[sz.ws_csc_mask:sz.ws_csc_mask + nnz].cpu()
    g.update(stats=att.stats.cpu(), Op=att.Op.cpu(), lse=att.lse.cpu(), O=O.cpu(),
             dQ=dQ.cpu(), dK=dK.cpu(), dV=dV.cpu(), dQp=att.dQp.cpu(), dKp=att.dKp.cpu(),
             dVp=att.dVp.cpu(), dOp=att.dOp.cpu())
    return att, g


def gpu_lists(w, g, nb):
    """CSR lists of every (b, h) as python lists of ascending arrays."""
    rp = g["row_ptr"].numpy()
    ci = g["col_idx"].numpy()
    out = {}
    for b in range(w.B):
        for h in range(w.H):
            L = []
            for i in range(nb):
                r = (b * w.H + h) * nb + i
                L.append(ci[rp[r]:rp[r + 1]].astype(np.int64))
            out[(b, h)] = L
    return out


def rel_err(a, b):
    den = np.abs(b).max()
    return np.abs(a - b).max() / (den if den > 0 else 1.0)


def compare(w, heads=None, rows=None, key_blocks=None, check_bwd=True, report=None,
            attn_kernel=0, shape_id=None, key_chunk_blocks=0, grad_scale="result",
            fused_a2v=False):
    """Run both sides on the seeded inputs of `w`; assert the contract.
    heads / rows / key_blocks restrict the oracle's attention work (a sample
    of the (b, h), query blocks and key blocks).  shape_id ([B, H, Z] ints):
    block shapes given to both sides instead of the statistics and Eq. 7.
    grad_scale "terms" (inputs whose softmax rows are nearly one-hot, where
    dQ and dK cancel to the size of the forward's bf16 roundings): dQ and dK
    within ILL_COND_TOL relative, and element by element within G_TOL *
    max|ref| plus what those roundings can move the element by through
    D = rowsum(dO * O) (the oracle's bound terms times TERMS_U; the largest
    ratio of error to allowance is reported as <name>_bound_use).
    fused_a2v: the device computes the A2V norms from the cross-attention
    queries and the audio tokens (prism_a2v_norms) instead of taking the A2V
    output; the norms are held to TAU_N relative, the audio statistics to
    what TAU_N can move them by, and a shape may differ from the oracle's on
    zones whose decision that error can reach (orc.norm_sensitive_zones)."""
    inputs = synth.generate(w, "cpu")
    att, g = run_gpu(w, inputs, attn_kernel, shape_id, key_chunk_blocks, fused_a2v)
    rep_ = {} if report is None else report
    rep_["key_chunks"] = att.plan.sz.key_chunks
    nb = att.plan.nb
    X = {k: f64(inputs[k]) for k in ("Q", "K", "V", "a2v", "dO")}
    rep = {} if report is None else report
    hs = list(range(w.H)) if heads is None else list(heads)

    w_h = w.with_(H=len(hs))
    if shape_id is not None:
        sid_use = np.asarray(shape_id, dtype=np.int64)[:, hs]
        assert np.array_equal(g["shape_id"].numpy().astype(np.int64)[:, hs], sid_use)
        return _compare_from_shapes(w, w_h, hs, g, X, nb, sid_use, rows, key_blocks, check_bwd,
                                    rep, heads, grad_scale)

    # ---- step 1: zone statistics ----
    Vs = X["V"][:, :, hs, :]
    if fused_a2v:
        n_o = orc.a2v_norms(f64(inputs["qa"]), f64(inputs["audio"]), f64(inputs["audio"]))
        n_g = f64(g["nrm"])
        rep["a2v_norm_max_rel"] = float((np.abs(n_g - n_o) / n_o).max())
        assert rep["a2v_norm_max_rel"] <= TAU_N, rep["a2v_norm_max_rel"]
        st_o = orc.zone_stats_from_norms(w_h, Vs, n_o)
        slack = audio_stats_slack(w, n_o, TAU_N)
    else:
        st_o = orc.zone_stats(w_h, Vs, X["a2v"])
        slack = None
    st_g = f64(g["stats"])[:, hs]
    for k in range(8):
        scale = max(1e-30, np.abs(st_o[..., k]).max())
        err = np.abs(st_g[..., k] - st_o[..., k])
        if slack is not None and 3 <= k <= 6:
            err = np.maximum(err - slack[:, None, :, k - 3], 0.0)
        assert err.max() / scale <= 2e-5, (k, err.max() / scale)
    if not w.per_head:
        st_o = (orc.zone_stats_from_norms(w, X["V"], n_o) if fused_a2v else
                orc.zone_stats(w, X["V"], X["a2v"]))

    # ---- step 2: shapes, permutation, pooling ----
    if w.per_head:
        sid_o, tie_o = orc.assign_shapes(w_h, st_o)
    else:
        sid_o, tie_o = orc.assign_shapes(w, st_o)
        sid_o, tie_o = sid_o[:, hs], tie_o[:, hs]
    sid_g = g["shape_id"].numpy().astype(np.int64)[:, hs]
    if fused_a2v:
        sens = orc.norm_sensitive_zones(w, n_o, st_o, TAU_N)
        if not w.per_head:                   # st_o holds every head here
            sens = sens[:, hs]
        tie_o = tie_o | sens
        rep["zones_norm_sensitive"] = int(sens.sum())
    mism = sid_g != sid_o
    assert not (mism & ~tie_o).any(), "shape id differs on a zone that is not a near tie"
    rep["shape_ties_taken"] = int(mism.sum())
    sid_use = np.where(mism, sid_g, sid_o)
    return _compare_from_shapes(w, w_h, hs, g, X, nb, sid_use, rows, key_blocks, check_bwd, rep,
                                heads, grad_scale)


def _compare_half_tile(w, w_h, hs, g, X, nb, perm_o, inv_o, units_o, nblk_o, Qp_o, Kp_o, Vp_o,
                       Qb_o, Kb_o, check_bwd, rep):
    """Steps 3+ of ``compare`` for plans with blocks of half a tile: the
    device's tile lists and sub-tile masks are read back as block lists (a
    query block of half tile qh selects the key blocks of the halves kh its
    mask leaves on), compared with the oracle's selection, checked to expand
    back exactly (``orc.expand_lists_masked``), and the attention is compared
    with the oracle's block-level attention."""
    U, T_ = orc.slot_tokens(w), w.block
    per = T_ // U
    nu = units_o.shape[2]
    Lg_all = gpu_lists(w, g, nb)
    rp = g["row_ptr"].numpy()
    cm = g["csr_mask"].numpy().astype(np.int64)
    cp, ri = g["col_ptr"].numpy(), g["row_idx"].numpy()
    ccm = g["csc_mask"].numpy().astype(np.int64)
    Lo, Fo = orc.select_blocks(w_h, Qb_o, Kb_o, nblk_o)
    L_use = {}
    diff_rows = flagged = 0
    for b in range(w.B):
        for hi, h in enumerate(hs):
            ul = units_o[b, hi]
            start = np.zeros(nu, dtype=np.int64)
            i = 0
            while i < nu:
                n = max(1, int(ul[i]))
                start[i:i + n] = i
                i += n
            Lg = Lg_all[(b, h)]
            masks = [cm[rp[(b * w.H + h) * nb + t]:rp[(b * w.H + h) * nb + t + 1]] for t in range(nb)]
            Lb = [None] * nu
            for t in range(nb):
                for qh in range(per):
                    i = t * per + qh
                    if ul[i] == 0:
                        continue
                    sel = set()
                    for v, m in zip(Lg[t], masks[t]):
                        for kh in range(per):
                            if not (m >> (qh * per + kh)) & 1:
                                sel.add(int(start[int(v) * per + kh]))
                    Lb[i] = np.array(sorted(sel), dtype=np.int64)
            el, em = orc.expand_lists_masked(Lb, ul, U, T_)
            for t in range(nb):
                assert np.array_equal(el[t], Lg[t]), ("tile list", b, h, t)
                assert np.array_equal(em[t], masks[t]), ("sub-tile mask", b, h, t)
            # CSC: the transpose, each entry with the same mask
            cols = orc.csc_from_lists(Lg, nb)
            for j in range(nb):
                r = (b * w.H + h) * nb + j
                assert np.array_equal(ri[cp[r]:cp[r + 1]], cols[j]), ("csc", b, h, j)
                for e, t in zip(range(cp[r], cp[r + 1]), ri[cp[r]:cp[r + 1]]):
                    k = int(np.searchsorted(Lg[t], j))
                    assert ccm[e] == masks[t][k], ("csc mask", b, h, j, t)
            lo_, fo = Lo[(b, hi)], Fo[(b, hi)]
            for i in range(nu):
                if Lb[i] is None:
                    continue
                flagged += int(fo[i])
                if not np.array_equal(Lb[i], lo_[i]):
                    assert fo[i], f"list differs on an unflagged row (b={b}, h={h}, unit {i})"
                    diff_rows += 1
            L_use[(b, hi)] = Lb
    rep["select_rows_differing_on_near_ties"] = diff_rows
    rep["select_rows_flagged"] = flagged
    rep["masked_entries"] = int((cm > 0).sum())
    scale = 1.0 / math.sqrt(w.d)
    dOp_o = orc.permute(X["dO"][:, :, hs], perm_o)
    assert np.array_equal(f64(g["dOp"])[:, hs], dOp_o)
    Op_o, lse_o, dQ_o, dK_o, dV_o = orc.attn_blocks(Qp_o, Kp_o, Vp_o, units_o, nblk_o, L_use, U,
                                                    scale, dOp=dOp_o, o_bf16=True)
    for name, got, ref, tol in (("O", g["Op"], Op_o, O_TOL), ("dQ", g["dQp"], dQ_o, G_TOL),
                                ("dK", g["dKp"], dK_o, G_TOL), ("dV", g["dVp"], dV_o, G_TOL)):
        if name != "O" and not check_bwd:
            continue
        got = f64(got)[:, hs]
        e = max(rel_err(got[b, hi], ref[b, hi]) for b in range(w.B) for hi in range(len(hs)))
        rep[name + "_max_rel"] = e
        assert e <= tol, (name, e)
    assert np.abs(f64(g["lse"])[:, hs] - lse_o).max() <= 2e-2
    return rep


def audio_stats_slack(w, n, tau):
    """How far the audio statistics (var_n_T, var_n_H, var_n_W, nbar) of every
    (b, zone) can move when the norms n [B, N] are off by tau relative:
    [B, Z, 4] (the oracle's line-variance bound; tau nbar for the mean)."""
    out = []
    for b in range(n.shape[0]):
        gn, m = orc._grid_views(n[b][:, None], w, 1)
        dv = np.stack([orc.line_variance_bound(gn, m, a, tau) for a in range(3)], -1).reshape(-1, 3)
        mf = m.astype(np.float64)
        cnt = mf.sum(axis=(1, 3, 5))
        nbar = np.where(cnt > 0, (gn[..., 0] * mf).sum(axis=(1, 3, 5)) / np.maximum(cnt, 1), 0.0)
        out.append(np.concatenate([dv, tau * nbar.reshape(-1, 1)], -1))
    return np.stack(out)


def _compare_from_shapes(w, w_h, hs, g, X, nb, sid_use, rows, key_blocks, check_bwd, rep,
                         heads, grad_scale="result"):
    """Steps 2 (permutation, pooling) to 5b of ``compare`` for given shapes."""
    perm_o, inv_o, nval_o, tiles_o, nblk_o = orc.build_permutation(w_h, sid_use, table=True)
    assert np.array_equal(g["perm"].numpy()[:, hs], perm_o)
    assert np.array_equal(g["inv"].numpy()[:, hs], inv_o)
    assert np.array_equal(g["n_valid"].numpy()[:, hs], nval_o)
    Qp_o = orc.permute(X["Q"][:, :, hs], perm_o)
    Kp_o = orc.permute(X["K"][:, :, hs], perm_o)
    Vp_o = orc.permute(X["V"][:, :, hs], perm_o)
    assert np.array_equal(f64(g["Qp"])[:, hs], Qp_o)
    assert np.array_equal(f64(g["Kp"])[:, hs], Kp_o)
    assert np.array_equal(f64(g["Vp"])[:, hs], Vp_o)
    U = orc.slot_tokens(w)
    Qb_o = orc.pool_blocks(Qp_o, tiles_o, nblk_o, U)
    Kb_o = orc.pool_blocks(Kp_o, tiles_o, nblk_o, U)
    Qb_g = (f64(g["Qbar"]) + f64(g["Qbar_lo"]))[:, hs]
    Kb_g = (f64(g["Kbar"]) + f64(g["Kbar_lo"]))[:, hs]
    assert np.abs(Qb_g - Qb_o).max() <= 1e-11 * max(1.0, np.abs(Qb_o).max())
    assert np.abs(Kb_g - Kb_o).max() <= 1e-11 * max(1.0, np.abs(Kb_o).max())
    rep["multi_tile_blocks"] = int((tiles_o > 1).sum())
    if U < w.block:
        assert rows is None and key_blocks is None, "half-tile blocks: whole heads only"
        rep["half_tile_blocks"] = int((tiles_o == 1).sum())
        return _compare_half_tile(w, w_h, hs, g, X, nb, perm_o, inv_o, tiles_o, nblk_o, Qp_o, Kp_o,
                                  Vp_o, Qb_o, Kb_o, check_bwd, rep)

    # ---- step 3+4: selection (over blocks: their first tiles) ----
    Lg_all = gpu_lists(w, g, nb)
    Lo, Fo = orc.select_blocks(w_h, Qb_o, Kb_o, nblk_o, rows=rows)
    diff_rows = 0
    flagged = 0
    # The CUDA lists (equal to the oracle's on every unflagged row checked
    # here) are the ones the attention steps of both sides use.  With blocks
    # that span several tiles the device lists are over tiles: the block list
    # of a query block is read off its first tile (the first tiles of the
    # listed tiles) and must expand back to the device list of every one of
    # its tiles.
    L_use = {}
    for b in range(w.B):
        for hi, h in enumerate(hs):
            Lg, tl = Lg_all[(b, h)], tiles_o[b, hi]
            Lb = [None] * nb
            for i in range(nb):
                if tl[i] > 0:
                    Lb[i] = Lg[i][tl[Lg[i]] > 0]
            exp = orc.expand_lists(Lb, tl)
            for i in range(nb):
                assert np.array_equal(exp[i], Lg[i]), ("tile lists", b, h, i)
            L_use[(b, hi)] = Lg
            lo_, fo = Lo[(b, hi)], Fo[(b, hi)]
            for i in range(nb):
                if lo_[i] is None or tl[i] == 0:
                    continue
                flagged += int(fo[i])
                if not np.array_equal(Lb[i], lo_[i]):
                    assert fo[i], f"list differs on an unflagged row (b={b}, h={h}, i={i})"
                    diff_rows += 1
    L_fwd = {k: [L[i] if (rows is None or i in rows) else None for i in range(nb)]
             for k, L in L_use.items()}
    rep["select_rows_differing_on_near_ties"] = diff_rows
    rep["select_rows_flagged"] = flagged
    # CSC = transpose of CSR (exact)
    cp = g["col_ptr"].numpy()
    ri = g["row_idx"].numpy()
    for b in range(w.B):
        for h in hs:
            cols = orc.csc_from_lists(Lg_all[(b, h)], nb)
            for j in range(nb):
                r = (b * w.H + h) * nb + j
                assert np.array_equal(ri[cp[r]:cp[r + 1]], cols[j]), (b, h, j)

    # ---- step 5: attention forward ----
    scale = 1.0 / math.sqrt(w.d)
    Op_o, lse_o = orc.attn_fwd(w_h, Qp_o, Kp_o, Vp_o, nval_o, L_fwd, scale)
    Op_g = f64(g["Op"])[:, hs]
    lse_g = f64(g["lse"])[:, hs]
    row_mask = np.zeros(w.Np, bool)
    for i in (range(nb) if rows is None else rows):
        row_mask[i * w.block:(i + 1) * w.block] = True
    errs = []
    for b in range(w.B):
        for hi in range(len(hs)):
            e = rel_err(Op_g[b, hi, row_mask], Op_o[b, hi, row_mask])
            errs.append(e)
            assert e <= O_TOL, ("O", b, hs[hi], e)
            assert np.abs(lse_g[b, hi, row_mask] - lse_o[b, hi, row_mask]).max() <= 2e-2
    rep["O_max_rel"] = max(errs)
    if rows is None and heads is None:
        O_o = orc.unpermute(Op_o, inv_o)
        assert rel_err(f64(g["O"]), O_o) <= O_TOL

    if not check_bwd:
        return rep
    # ---- step 5b: backward ----
    dOp_o = orc.permute(X["dO"][:, :, hs], perm_o)
    assert np.array_equal(f64(g["dOp"])[:, hs], dOp_o)
    if key_blocks is None and rows is None:
        dQ_o, dK_o, dV_o, aQ_o, aK_o = orc.attn_bwd(w_h, Qp_o, Kp_o, Vp_o, dOp_o, nval_o, L_use,
                                                    scale, o_bf16=True, abs_terms=True)
        for name, got, ref, terms in (("dQ", g["dQp"], dQ_o, aQ_o), ("dK", g["dKp"], dK_o, aK_o),
                                      ("dV", g["dVp"], dV_o, None)):
            got = f64(got)[:, hs]
            e = max(rel_err(got[b, hi], ref[b, hi]) for b in range(w.B)
                    for hi in range(len(hs)))
            rep[name + "_max_rel"] = e
            if grad_scale == "terms" and terms is not None:
                # (1) a guard, element by element: the contract's share of the
                # head's largest value plus what the forward's bf16 roundings
                # of O can move this element by through D (TERMS_U per unit of
                # the oracle's sizes); (2) the relative error within
                # ILL_COND_TOL, the error those roundings leave once dQ and dK
                # have cancelled to their size
                use = 0.0
                for b in range(w.B):
                    for hi in range(len(hs)):
                        allow = G_TOL * np.abs(ref[b, hi]).max() + TERMS_U * terms[b, hi]
                        err = np.abs(got[b, hi] - ref[b, hi])
                        use = max(use, float((err / np.maximum(allow, 1e-300)).max()))
                rep[name + "_bound_use"] = use
                assert use <= 1.0, (name, use)
                assert e <= ILL_COND_TOL, (name, e)
            else:
                assert e <= G_TOL, (name, e)
        if heads is None:
            for name, ref in (("dQ", dQ_o), ("dK", dK_o), ("dV", dV_o)):
                assert rel_err(f64(g[name]), orc.unpermute(ref, inv_o)) <= G_TOL, name
    else:
        # dQ on the sampled rows, dK / dV on the sampled key blocks (all the
        # query blocks that selected them contribute)
        S = w.block
        if rows is not None:
            dQ_o, _, _ = orc.attn_bwd(w_h, Qp_o, Kp_o, Vp_o, dOp_o, nval_o, L_use, scale,
                                      rows_only=set(rows), o_bf16=True)
            got = f64(g["dQp"])[:, hs]
            e = 0.0
            for b in range(w.B):
                for hi in range(len(hs)):
                    e = max(e, rel_err(got[b, hi, row_mask], dQ_o[b, hi, row_mask]))
            rep["dQ_max_rel"] = e
            assert e <= G_TOL, ("dQ", e)
        if key_blocks:
            ek = 0.0
            for b in range(w.B):
                for hi in range(len(hs)):
                    cols = orc.csc_from_lists(L_use[(b, hi)], nb)
                    for j in key_blocks:
                        qs = set(int(i) for i in cols[j])
                        _, dK_o, dV_o = orc.attn_bwd(
                            w_h, Qp_o[b:b + 1, hi:hi + 1], Kp_o[b:b + 1, hi:hi + 1],
                            Vp_o[b:b + 1, hi:hi + 1], dOp_o[b:b + 1, hi:hi + 1],
                            nval_o[b:b + 1, hi:hi + 1], {(0, 0): L_use[(b, hi)]}, scale,
                            rows_only=qs, o_bf16=True)
                        sl = slice(j * S, (j + 1) * S)
                        for nm, ref in (("dKp", dK_o), ("dVp", dV_o)):
                            got = f64(g[nm])[b, hs[hi], sl]
                            ek = max(ek, rel_err(got, ref[0, 0, sl]))
            rep["dKV_sampled_max_rel"] = ek
            assert ek <= G_TOL, ("dK/dV", ek)
    return rep


def _head_slices(att, w, b, h, nb):
    """What the sampled comparison reads back of one (b, h): host copies."""
    sl = (slice(b, b + 1), slice(h, h + 1))
    o, L = att.perm_out, att.lists
    rp = L["row_ptr"].cpu().numpy().astype(np.int64)
    cp = L["col_ptr"].cpu().numpy().astype(np.int64)
    base = (b * w.H + h) * nb
    lo_, hi_ = int(rp[base]), int(rp[base + nb])
    ci = L["col_idx"][lo_:hi_].cpu().numpy().astype(np.int64)
    c_lo, c_hi = int(cp[base]), int(cp[base + nb])
    ri = L["row_idx"][c_lo:c_hi].cpu().numpy().astype(np.int64)
    g = dict(
        stats=f64(att.stats[sl]),
        shape_id=o["shape_id"][sl].cpu().numpy().astype(np.int64),
        perm=o["perm"][sl].cpu().numpy(), inv=o["inv"][sl].cpu().numpy(),
        n_valid=o["n_valid"][sl].cpu().numpy(),
        Qbar=f64(o["Qbar"][sl]) + f64(o["Qbar_lo"][sl]),
        Kbar=f64(o["Kbar"][sl]) + f64(o["Kbar_lo"][sl]),
        lists=[ci[int(rp[base + i]) - lo_:int(rp[base + i + 1]) - lo_] for i in range(nb)],
        csc=[ri[int(cp[base + j]) - c_lo:int(cp[base + j + 1]) - c_lo] for j in range(nb)],
        sel_tie=L["sel_tie"][sl].cpu().numpy())
    for nm in ("Qp", "Kp", "Vp"):
        g[nm] = f64(o[nm][sl])
    for nm in ("Op", "lse", "dQp", "dKp", "dVp", "dOp"):
        g[nm] = f64(getattr(att, nm)[sl])
    for nm in ("O", "dQ"):
        g[nm] = f64(getattr(att, nm)[b:b + 1, :, h:h + 1])
    return g


def compare_sampled(w, heads, n_rows=6, key_clusters=2, cluster_len=4, seed=0, report=None,
                    key_chunk_blocks=(0,)):
    """Full-size check on a sample, in the launch configuration bench.py
    times.  Inputs are generated on the device.  For each sampled head the
    oracle runs every step of that head (statistics, shapes, permutation,
    pooling) and the selection of EVERY query block of the head; attention
    forward and dQ run on `n_rows` sampled query blocks (always including one
    partially real block when there is one, and the block with the longest
    list), and dK / dV on `key_clusters` runs of `cluster_len` consecutive
    key blocks (every query block that selected them contributes).

    key_chunk_blocks: the attention kernels' range settings to run (0 =
    automatic, as the bench; a value >= nb = one pass over each list); each
    setting is run on the device and compared with the same oracle results,
    and its errors are reported under rep["runs"]."""
    assert w.per_head, "sampled comparison needs per-head shapes"
    rep = {} if report is None else report
    dev = torch.device("cuda")
    x = synth.generate(w, dev)
    runs = []
    for kcb in key_chunk_blocks:
        att = prism.PrismAttention(w, dev, key_chunk_blocks=kcb)
        att.forward(x["Q"], x["K"], x["V"], x["a2v"])
        att.backward(x["dO"])
        torch.cuda.synchronize()
        assert att.status() == 0, "device status word set"
        nb = att.plan.nb
        grab = {(b, h): _head_slices(att, w, b, h, nb) for b in range(w.B) for h in heads}
        rp_all = att.lists["row_ptr"].cpu().numpy()
        runs.append(dict(key_chunks=att.plan.sz.key_chunks, g=grab,
                         density=float(rp_all[-1]) / (w.B * w.H * nb * nb)))
        del att
        torch.cuda.empty_cache()
    S = w.block
    w1 = w.with_(H=1)
    scale = 1.0 / math.sqrt(w.d)
    rng = np.random.default_rng(seed)
    a2v = f64(x["a2v"])
    errs = [dict(key_chunks=r["key_chunks"], O=0.0, dQ=0.0, dKV=0.0, lse=0.0, dK_bound_use=0.0)
            for r in runs]
    rep.update(select_rows_compared=0, select_rows_flagged=0,
               select_rows_differing_on_near_ties=0, key_blocks_compared=0)
    for b in range(w.B):
        for h in heads:
            g0 = runs[0]["g"][(b, h)]
            X = {k: f64(x[k][b:b + 1, :, h:h + 1]) for k in ("Q", "K", "V", "dO")}
            # the discrete steps do not depend on the attention kernels' ranges
            for r in runs[1:]:
                gr = r["g"][(b, h)]
                for nm in ("shape_id", "perm", "n_valid"):
                    assert np.array_equal(gr[nm], g0[nm]), nm
                assert all(np.array_equal(a, c) for a, c in zip(gr["lists"], g0["lists"]))
            # ---- statistics, shapes, permutation, pooling (whole head) ----
            st_o = orc.zone_stats(w1, X["V"], a2v[b:b + 1])
            for k in range(8):
                sc = max(1e-30, np.abs(st_o[..., k]).max())
                assert np.abs(g0["stats"][..., k] - st_o[..., k]).max() / sc <= 2e-5, ("stats", k)
            sid_o, tie_o = orc.assign_shapes(w1, st_o)
            mism = g0["shape_id"] != sid_o
            assert not (mism & ~tie_o).any(), "shape id differs on a zone that is not a near tie"
            sid_use = np.where(mism, g0["shape_id"], sid_o)
            perm_o, inv_o, nval_o = orc.build_permutation(w1, sid_use)
            assert np.array_equal(g0["perm"], perm_o)
            assert np.array_equal(g0["inv"], inv_o)
            assert np.array_equal(g0["n_valid"], nval_o)
            nb = nval_o.shape[2]
            Qp_o, Kp_o = orc.permute(X["Q"], perm_o), orc.permute(X["K"], perm_o)
            Vp_o, dOp_o = orc.permute(X["V"], perm_o), orc.permute(X["dO"], perm_o)
            for nm, ref in (("Qp", Qp_o), ("Kp", Kp_o), ("Vp", Vp_o), ("dOp", dOp_o)):
                assert np.array_equal(g0[nm], ref), nm
            Qb_o, Kb_o = orc.pool(Qp_o, nval_o, S), orc.pool(Kp_o, nval_o, S)
            assert np.abs(g0["Qbar"] - Qb_o).max() <= 1e-11 * max(1.0, np.abs(Qb_o).max())
            assert np.abs(g0["Kbar"] - Kb_o).max() <= 1e-11 * max(1.0, np.abs(Kb_o).max())
            # ---- selection: every query block of the head ----
            Lg = g0["lists"]
            Lo, Fo = orc.select_blocks(w1, Qb_o, Kb_o, nval_o)
            for i in range(nb):
                rep["select_rows_compared"] += 1
                rep["select_rows_flagged"] += int(Fo[(0, 0)][i])
                if not np.array_equal(Lg[i], Lo[(0, 0)][i]):
                    assert Fo[(0, 0)][i], f"list differs on an unflagged row (b={b}, h={h}, i={i})"
                    rep["select_rows_differing_on_near_ties"] += 1
            cols = orc.csc_from_lists(Lg, nb)
            for j in range(nb):
                assert np.array_equal(g0["csc"][j], cols[j]), ("csc", j)
            # ---- sampled query blocks: O, LSE, dQ ----
            realq = np.nonzero(nval_o[0, 0] > 0)[0]
            partial = [i for i in realq if nval_o[0, 0, i] < S]
            rows = [int(i) for i in rng.choice(realq, size=min(n_rows, len(realq)), replace=False)]
            if partial and not any(i in partial for i in rows):
                rows[0] = int(rng.choice(partial))
            longest = int(max(realq, key=lambda i: len(Lg[i])))
            if longest not in rows:
                rows[-1] = longest
            rows = sorted(set(rows))
            Lfull = {(0, 0): Lg}
            Lrows = {(0, 0): [Lg[i] if i in rows else None for i in range(nb)]}
            Op_o, lse_o = orc.attn_fwd(w1, Qp_o, Kp_o, Vp_o, nval_o, Lrows, scale)
            dQ_o, _, _ = orc.attn_bwd(w1, Qp_o, Kp_o, Vp_o, dOp_o, nval_o, Lfull, scale,
                                      rows_only=set(rows), o_bf16=True)
            rr = np.concatenate([np.arange(i * S, (i + 1) * S) for i in rows])
            # ---- sampled key blocks: dK, dV over every query block that selected them ----
            realk = [j for j in range(nb) if len(cols[j]) > 0]
            kbs = []
            for _ in range(key_clusters):
                j0 = int(rng.integers(0, max(1, len(realk) - cluster_len + 1)))
                kbs += [j for j in realk[j0:j0 + cluster_len] if j not in kbs]
            kv_o = orc.attn_bwd_key_blocks(Qp_o[0, 0], Kp_o[0, 0], Vp_o[0, 0], dOp_o[0, 0],
                                           nval_o[0, 0], Lg, kbs, S, scale, o_bf16=True, abs_terms=True)
            rep["key_blocks_compared"] += len(kbs)
            for r, er in zip(runs, errs):
                gr = r["g"][(b, h)]
                # the contract is per tensor (per head): max |err| / max |ref|; on a
                # sample the maxima run over the sampled rows (a smaller, stricter
                # denominator than the whole head's)
                eo = rel_err(gr["Op"][0, 0, rr], Op_o[0, 0, rr])
                eq = rel_err(gr["dQp"][0, 0, rr], dQ_o[0, 0, rr])
                el = np.abs(gr["lse"][0, 0, rr] - lse_o[0, 0, rr]).max()
                assert eo <= O_TOL, ("O", r["key_chunks"], b, h, eo)
                assert eq <= G_TOL, ("dQ", r["key_chunks"], b, h, eq)
                assert el <= 2e-2, ("lse", r["key_chunks"], b, h, el)
                er["O"], er["dQ"], er["lse"] = max(er["O"], eo), max(er["dQ"], eq), max(er["lse"], el)
                for i in rows:  # model order: the unpermuted outputs carry the same rows
                    rs = slice(i * S, (i + 1) * S)
                    toks = perm_o[0, 0, rs]
                    real = toks >= 0
                    for nm, got in (("O", gr["Op"]), ("dQ", gr["dQp"])):
                        assert np.array_equal(gr[nm][0, toks[real], 0], got[0, 0, rs][real]), nm
                for j in kbs:
                    rs = slice(j * S, (j + 1) * S)
                    # one key block: its own maximum.  dV within G_TOL; dK also
                    # element by element within G_TOL of its maximum plus what
                    # the forward's bf16 roundings of O move it by through D
                    # (TERMS_U per unit of the oracle's sizes; a key block whose
                    # dK cancels against D is as exact as that), and within
                    # ILL_COND_TOL relative
                    ev = rel_err(gr["dVp"][0, 0, rs], kv_o[j][1])
                    assert ev <= G_TOL, ("dVp", r["key_chunks"], b, h, j, ev)
                    got, ref = np.asarray(gr["dKp"][0, 0, rs], dtype=np.float64), kv_o[j][0]
                    allow = G_TOL * np.abs(ref).max() + TERMS_U * kv_o[j][2]
                    use = float((np.abs(got - ref) / np.maximum(allow, 1e-300)).max())
                    ek = rel_err(got, ref)
                    assert use <= 1.0 and ek <= ILL_COND_TOL, ("dKp", r["key_chunks"], b, h, j, ek, use)
                    er["dKV"] = max(er["dKV"], ek, ev)
                    er["dK_bound_use"] = max(er["dK_bound_use"], use)
    rep["runs"] = errs
    rep.update({k: errs[0][k] for k in ("O", "dQ", "dKV")})
    rep["block_density"] = runs[0]["density"]
    return rep

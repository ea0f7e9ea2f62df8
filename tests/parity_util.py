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


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(w, inputs, attn_kernel=0, shape_id=None, key_chunk_blocks=0):
    dev = torch.device("cuda")
    x = {k: inputs[k].to(dev) for k in ("Q", "K", "V", "a2v", "dO")}
    att = prism.PrismAttention(w, dev, attn_kernel=attn_kernel, key_chunk_blocks=key_chunk_blocks)
    sid = None if shape_id is None else torch.as_tensor(shape_id, dtype=torch.uint8).to(dev)
    O = att.forward(x["Q"], x["K"], x["V"], x["a2v"], shape_id=sid)
    dQ, dK, dV = att.backward(x["dO"])
    torch.cuda.synchronize()
    assert att.status() == 0, "device status word set"
    g = {k: v.cpu() for k, v in att.perm_out.items()}
    g.update({k: v.cpu() for k, v in att.lists.items()})
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
            attn_kernel=0, shape_id=None, key_chunk_blocks=0, grad_scale="result"):
    """Run both sides on the seeded inputs of `w`; assert the contract.
    heads / rows / key_blocks restrict the oracle's attention work (a sample
    of the (b, h), query blocks and key blocks).  shape_id ([B, H, Z] ints):
    block shapes given to both sides instead of the statistics and Eq. 7.
    grad_scale "terms" adds to the dQ / dK tolerance the error that a 2^-7
    relative error in D = rowsum(dO * O) carries into them (two bf16
    roundings of O: the forward's and the stored value's), for inputs whose
    softmax rows are nearly one-hot, where dQ and dK cancel to that size."""
    inputs = synth.generate(w, "cpu")
    att, g = run_gpu(w, inputs, attn_kernel, shape_id, key_chunk_blocks)
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
    st_o = orc.zone_stats(w_h, Vs, X["a2v"])
    st_g = f64(g["stats"])[:, hs]
    for k in range(8):
        scale = max(1e-30, np.abs(st_o[..., k]).max())
        err = np.abs(st_g[..., k] - st_o[..., k]).max() / scale
        assert err <= 2e-5, (k, err)
    if not w.per_head:
        st_o = orc.zone_stats(w, X["V"], X["a2v"])

    # ---- step 2: shapes, permutation, pooling ----
    if w.per_head:
        sid_o, tie_o = orc.assign_shapes(w_h, st_o)
    else:
        sid_o, tie_o = orc.assign_shapes(w, st_o)
        sid_o, tie_o = sid_o[:, hs], tie_o[:, hs]
    sid_g = g["shape_id"].numpy().astype(np.int64)[:, hs]
    mism = sid_g != sid_o
    assert not (mism & ~tie_o).any(), "shape id differs on a zone that is not a near tie"
    rep["shape_ties_taken"] = int(mism.sum())
    sid_use = np.where(mism, sid_g, sid_o)
    return _compare_from_shapes(w, w_h, hs, g, X, nb, sid_use, rows, key_blocks, check_bwd, rep,
                                heads, grad_scale)


def _compare_from_shapes(w, w_h, hs, g, X, nb, sid_use, rows, key_blocks, check_bwd, rep,
                         heads, grad_scale="result"):
    """Steps 2 (permutation, pooling) to 5b of ``compare`` for given shapes."""
    perm_o, inv_o, nval_o = orc.build_permutation(w_h, sid_use)
    assert np.array_equal(g["perm"].numpy()[:, hs], perm_o)
    assert np.array_equal(g["inv"].numpy()[:, hs], inv_o)
    assert np.array_equal(g["n_valid"].numpy()[:, hs], nval_o)
    Qp_o = orc.permute(X["Q"][:, :, hs], perm_o)
    Kp_o = orc.permute(X["K"][:, :, hs], perm_o)
    Vp_o = orc.permute(X["V"][:, :, hs], perm_o)
    assert np.array_equal(f64(g["Qp"])[:, hs], Qp_o)
    assert np.array_equal(f64(g["Kp"])[:, hs], Kp_o)
    assert np.array_equal(f64(g["Vp"])[:, hs], Vp_o)
    Qb_o = orc.pool(Qp_o, nval_o, w.block)
    Kb_o = orc.pool(Kp_o, nval_o, w.block)
    Qb_g = (f64(g["Qbar"]) + f64(g["Qbar_lo"]))[:, hs]
    Kb_g = (f64(g["Kbar"]) + f64(g["Kbar_lo"]))[:, hs]
    assert np.abs(Qb_g - Qb_o).max() <= 1e-11 * max(1.0, np.abs(Qb_o).max())
    assert np.abs(Kb_g - Kb_o).max() <= 1e-11 * max(1.0, np.abs(Kb_o).max())

    # ---- step 3+4: selection ----
    Lg_all = gpu_lists(w, g, nb)
    Lo, Fo = orc.select_blocks(w_h, Qb_o, Kb_o, nval_o, rows=rows)
    diff_rows = 0
    flagged = 0
    # The CUDA lists (equal to the oracle's on every unflagged row checked
    # here) are the ones the attention steps of both sides use.
    L_use = {(b, hi): Lg_all[(b, h)] for b in range(w.B) for hi, h in enumerate(hs)}
    for b in range(w.B):
        for hi, h in enumerate(hs):
            Lg = Lg_all[(b, h)]
            lo_, fo = Lo[(b, hi)], Fo[(b, hi)]
            for i in range(nb):
                if lo_[i] is None:
                    continue
                flagged += int(fo[i])
                if not np.array_equal(Lg[i], lo_[i]):
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
            if grad_scale == "terms" and terms is not None:
                e = max(np.abs(got[b, hi] - ref[b, hi]).max() /
                        (np.abs(ref[b, hi]).max() + 2.0 ** -7 * terms[b, hi].max() / G_TOL)
                        for b in range(w.B) for hi in range(len(hs)))
            else:
                e = max(rel_err(got[b, hi], ref[b, hi]) for b in range(w.B)
                        for hi in range(len(hs)))
            rep[name + "_max_rel"] = e
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


def compare_sampled(w, heads, n_rows=6, n_key_blocks=1, seed=0, report=None):
    """Full-size check on a sample.  Inputs are generated on the device; for
    each sampled head the oracle runs every step of that head (statistics,
    shapes, permutation, pooling), the selection on `n_rows` sampled query
    blocks (always including one partially real block when there is one),
    attention forward and dQ on those rows, and dK / dV on `n_key_blocks`
    sampled key blocks (every query block that selected them contributes).
    Only the sampled slices are copied to the host."""
    assert w.per_head, "sampled comparison needs per-head shapes"
    rep = {} if report is None else report
    dev = torch.device("cuda")
    x = synth.generate(w, dev)
    att = prism.PrismAttention(w, dev)
    att.forward(x["Q"], x["K"], x["V"], x["a2v"])
    att.backward(x["dO"])
    torch.cuda.synchronize()
    assert att.status() == 0, "device status word set"
    nb, S = att.plan.nb, w.block
    w1 = w.with_(H=1)
    scale = 1.0 / math.sqrt(w.d)
    rng = np.random.default_rng(seed)
    a2v = f64(x["a2v"])
    o, L = att.perm_out, att.lists
    rp_all = L["row_ptr"].cpu().numpy()
    cp_all = L["col_ptr"].cpu().numpy()
    errs = dict(O=0.0, dQ=0.0, dKV=0.0)
    for b in range(w.B):
        for h in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            X = {k: f64(x[k][b:b + 1, :, h:h + 1]) for k in ("Q", "K", "V", "dO")}
            # ---- statistics, shapes, permutation, pooling (whole head) ----
            st_o = orc.zone_stats(w1, X["V"], a2v[b:b + 1])
            st_g = f64(att.stats[sl])
            for k in range(8):
                sc = max(1e-30, np.abs(st_o[..., k]).max())
                assert np.abs(st_g[..., k] - st_o[..., k]).max() / sc <= 2e-5, ("stats", k)
            sid_o, tie_o = orc.assign_shapes(w1, st_o)
            sid_g = o["shape_id"][sl].cpu().numpy().astype(np.int64)
            mism = sid_g != sid_o
            assert not (mism & ~tie_o).any(), "shape id differs on a zone that is not a near tie"
            sid_use = np.where(mism, sid_g, sid_o)
            perm_o, inv_o, nval_o = orc.build_permutation(w1, sid_use)
            assert np.array_equal(o["perm"][sl].cpu().numpy(), perm_o)
            assert np.array_equal(o["inv"][sl].cpu().numpy(), inv_o)
            assert np.array_equal(o["n_valid"][sl].cpu().numpy(), nval_o)
            Qp_o, Kp_o = orc.permute(X["Q"], perm_o), orc.permute(X["K"], perm_o)
            Vp_o, dOp_o = orc.permute(X["V"], perm_o), orc.permute(X["dO"], perm_o)
            for nm, ref in (("Qp", Qp_o), ("Kp", Kp_o), ("Vp", Vp_o)):
                assert np.array_equal(f64(o[nm][sl]), ref), nm
            assert np.array_equal(f64(att.dOp[sl]), dOp_o)
            Qb_o, Kb_o = orc.pool(Qp_o, nval_o, S), orc.pool(Kp_o, nval_o, S)
            Qb_g = f64(o["Qbar"][sl]) + f64(o["Qbar_lo"][sl])
            Kb_g = f64(o["Kbar"][sl]) + f64(o["Kbar_lo"][sl])
            assert np.abs(Qb_g - Qb_o).max() <= 1e-11 * max(1.0, np.abs(Qb_o).max())
            assert np.abs(Kb_g - Kb_o).max() <= 1e-11 * max(1.0, np.abs(Kb_o).max())
            # ---- the head's CSR lists from the device ----
            base = (b * w.H + h) * nb
            lo_, hi_ = int(rp_all[base]), int(rp_all[base + nb])
            ci = L["col_idx"][lo_:hi_].cpu().numpy().astype(np.int64)
            Lg = [ci[int(rp_all[base + i]) - lo_:int(rp_all[base + i + 1]) - lo_] for i in range(nb)]
            c_lo, c_hi = int(cp_all[base]), int(cp_all[base + nb])
            ri = L["row_idx"][c_lo:c_hi].cpu().numpy().astype(np.int64)
            cols = orc.csc_from_lists(Lg, nb)
            for j in range(nb):
                got = ri[int(cp_all[base + j]) - c_lo:int(cp_all[base + j + 1]) - c_lo]
                assert np.array_equal(got, cols[j]), ("csc", j)
            # ---- sampled query blocks: selection, O, LSE, dQ ----
            realq = np.nonzero(nval_o[0, 0] > 0)[0]
            partial = [i for i in realq if nval_o[0, 0, i] < S]
            rows = list(rng.choice(realq, size=min(n_rows, len(realq)), replace=False))
            if partial and not any(i in partial for i in rows):
                rows[0] = int(rng.choice(partial))
            rows = sorted(int(i) for i in rows)
            Lo, Fo = orc.select_blocks(w1, Qb_o, Kb_o, nval_o, rows=rows)
            for i in rows:
                if not np.array_equal(Lg[i], Lo[(0, 0)][i]):
                    assert Fo[(0, 0)][i], f"list differs on an unflagged row (b={b}, h={h}, i={i})"
            Lfull = {(0, 0): Lg}
            Lrows = {(0, 0): [Lg[i] if i in rows else None for i in range(nb)]}
            Op_o, lse_o = orc.attn_fwd(w1, Qp_o, Kp_o, Vp_o, nval_o, Lrows, scale)
            dQ_o, _, _ = orc.attn_bwd(w1, Qp_o, Kp_o, Vp_o, dOp_o, nval_o, Lfull, scale,
                                      rows_only=set(rows), o_bf16=True)
            Op_g, lse_g, dQp_g = f64(att.Op[sl]), f64(att.lse[sl]), f64(att.dQp[sl])
            # the contract is per tensor (per head): max |err| / max |ref|; on a
            # sample the maxima run over the sampled rows (a smaller, stricter
            # denominator than the whole head's)
            rr = np.concatenate([np.arange(i * S, (i + 1) * S) for i in rows])
            eo = rel_err(Op_g[0, 0, rr], Op_o[0, 0, rr])
            eq = rel_err(dQp_g[0, 0, rr], dQ_o[0, 0, rr])
            assert eo <= O_TOL, ("O", b, h, eo)
            assert eq <= G_TOL, ("dQ", b, h, eq)
            assert np.abs(lse_g[0, 0, rr] - lse_o[0, 0, rr]).max() <= 2e-2
            errs["O"], errs["dQ"] = max(errs["O"], eo), max(errs["dQ"], eq)
            for i in rows:  # per-block figures, reported only
                r = slice(i * S, (i + 1) * S)
                rep.setdefault("dQ_worst_block_rel", 0.0)
                rep["dQ_worst_block_rel"] = max(rep["dQ_worst_block_rel"],
                                                rel_err(dQp_g[0, 0, r], dQ_o[0, 0, r]))
                # model order: the unpermuted outputs carry the same rows
                toks = perm_o[0, 0, r]
                real = toks >= 0
                for nm, got in (("O", Op_g), ("dQ", dQp_g)):
                    mo = f64(getattr(att, nm)[b:b + 1, :, h:h + 1])
                    assert np.array_equal(mo[0, toks[real], 0], got[0, 0, r][real]), nm
            # ---- sampled key blocks: dK, dV over every query block that selected them ----
            realk = [j for j in range(nb) if len(cols[j]) > 0]
            for j in rng.choice(realk, size=min(n_key_blocks, len(realk)), replace=False):
                j = int(j)
                _, dK_o, dV_o = orc.attn_bwd(w1, Qp_o, Kp_o, Vp_o, dOp_o, nval_o, Lfull, scale,
                                             rows_only=set(int(i) for i in cols[j]),
                                             o_bf16=True)
                r = slice(j * S, (j + 1) * S)
                for nm, ref in (("dKp", dK_o), ("dVp", dV_o)):
                    got = f64(getattr(att, nm)[sl])[0, 0, r]
                    e = rel_err(got, ref[0, 0, r])  # one key block: its own maximum
                    assert e <= G_TOL, (nm, b, h, j, e)
                    errs["dKV"] = max(errs["dKV"], e)
    rep.update(errs)
    rep["block_density"] = float(rp_all[-1]) / (w.B * w.H * nb * nb)
    return rep

"""Block scores on the tensor cores (score_tc.cu): the unscaled dots
Qbar_i . Kbar_j that prism_block_select writes to the workspace, compared
with the exact dot of the same double-float block means, for every pair.

The kernel splits each row of means v (hi + lo) into seven 7-bit integer
digits after scaling by 2^-e (max|hi| < 2^e), multiplies digit slices on the
tensor cores with exact integer sums, and keeps the products of digit levels
s + t <= 6.  Its error bound is |S - S_exact| <= 2^(eq+ek) d 1.3 2^-49
(dropped levels and digit remainders).  The reference is an extended-precision
(64-bit mantissa) dot of hi + lo, whose own error is far below that bound.
The selection's lists are held to the oracle by the parity tests; this test
pins the score product itself."""
import numpy as np
import pytest
import torch

from content_adaptive_block_02_b300 import prism, synth

pytestmark = pytest.mark.gpu


def _exponent(m):
    """Smallest e with m < 2^e for m > 0 (frexp: m = f 2^e, 0.5 <= f < 1); 0 for m = 0."""
    _, e = np.frexp(m)
    return np.where(m > 0, e, 0).astype(np.int64)


def _check(w, **fw):
    dev = torch.device("cuda", 0)
    x = synth.generate(w, dev)
    att = prism.PrismAttention(w, dev)
    att.forward(x["Q"], x["K"], x["V"], x["a2v"], **fw)
    assert att.status() == prism.PRISM_OK
    sz = att.plan.sz
    nb, d = sz.nslots, w.d
    R = w.B * w.H * nb
    o = att.perm_out
    q = (o["Qbar"].double() + o["Qbar_lo"].double()).cpu().numpy().reshape(w.B * w.H, nb, d)
    k = (o["Kbar"].double() + o["Kbar_lo"].double()).cpu().numpy().reshape(w.B * w.H, nb, d)
    qh = o["Qbar"].cpu().numpy().reshape(w.B * w.H, nb, d)
    kh = o["Kbar"].cpu().numpy().reshape(w.B * w.H, nb, d)
    raw = att.ws[sz.ws_scores:sz.ws_scores + 8 * R * nb].view(torch.float32).cpu().numpy()
    S = raw[:R * nb].astype(np.float64) + raw[R * nb:].astype(np.float64)
    S = S.reshape(w.B * w.H, nb, nb)
    ref = np.einsum("hic,hjc->hij", q.astype(np.longdouble), k.astype(np.longdouble))
    eq = _exponent(np.abs(qh).max(axis=2).astype(np.float64))
    ek = _exponent(np.abs(kh).max(axis=2).astype(np.float64))
    bound = np.ldexp(np.float64(d * 1.3 * 2.0 ** -49), eq[:, :, None] + ek[:, None, :])
    err = np.abs(S - ref).astype(np.float64)
    assert np.all(err <= bound), (err / bound).max()
    # the hi part alone is the fp32 rounding of the score (normalised pair)
    hi = raw[:R * nb].reshape(w.B * w.H, nb, nb)
    assert np.all(np.abs(raw[R * nb:]).reshape(hi.shape) <= np.spacing(np.abs(hi)))
    return float((err / bound).max()), nb


def test_scores_several_tiles_ragged():
    # 8 x 48 x 48 padded grid: 144 blocks per head, two key tiles of 128 and
    # three query tiles of 64, both ragged
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=40, W=48, H=3, n_src=1, zone=(4, 16, 16),
                                      name="scores144")
    rel, nb = _check(w)
    assert nb == 144 and rel < 1.0


def test_scores_head_dim_64():
    # the tiny workload: d = 64 (one 64-channel box), 16-token blocks
    rel, nb = _check(synth.WORKLOADS["tiny"])
    assert rel < 1.0


def test_scores_half_tile_slots():
    # half-tile blocks: the selection runs over 64-token slots
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      menu=synth.MENU_64, class_tau=(), name="scores_half")
    rel, nb = _check(w)
    assert prism.Plan(w).sz.half_tile == 1 and nb == 2 * prism.Plan(w).sz.nb and rel < 1.0


def test_scores_large_magnitudes():
    # block means of order 1e3: the bound scales with 2^(eq+ek)
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      name="scores_big")
    dev = torch.device("cuda", 0)
    x = synth.generate(w, dev)
    for n in ("Q", "K"):
        x[n] = (x[n].float() * 1000.0).to(torch.bfloat16)
    att = prism.PrismAttention(w, dev)
    att.forward(x["Q"], x["K"], x["V"], x["a2v"])
    assert att.status() == prism.PRISM_OK
    sz = att.plan.sz
    nb, d, R = sz.nslots, w.d, w.B * w.H * sz.nslots
    o = att.perm_out
    q = (o["Qbar"].double() + o["Qbar_lo"].double()).cpu().numpy().reshape(-1, nb, d)
    k = (o["Kbar"].double() + o["Kbar_lo"].double()).cpu().numpy().reshape(-1, nb, d)
    raw = att.ws[sz.ws_scores:sz.ws_scores + 8 * R * nb].view(torch.float32).cpu().numpy()
    S = (raw[:R * nb].astype(np.float64) + raw[R * nb:]).reshape(-1, nb, nb)
    ref = np.einsum("hic,hjc->hij", q.astype(np.longdouble), k.astype(np.longdouble))
    mq = np.abs(q).max(axis=2)[:, :, None]
    mk = np.abs(k).max(axis=2)[:, None, :]
    assert np.all(np.abs(S - ref).astype(np.float64) <= 4 * mq * mk * d * 1.3 * 2.0 ** -49)

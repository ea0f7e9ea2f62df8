"""The workspace-free backward (prism_sparse_attn_bwd_noalloc), for callers
that cannot allocate device memory when they run the backward.  Its results
must equal those of the workspace entry point (prism_sparse_attn_bwd) within
the gradient tolerance of the parity tests, on two calls in a row (the second
call reuses the library's scratch array as the first left it).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

from content_adaptive_block_02_b300 import build, prism, synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu
P = ctypes.c_void_p


def _fn():
    build.build()
    fn = prism.lib().prism_sparse_attn_bwd_noalloc
    fn.argtypes = [P] * 12 + [ctypes.c_float] + [P] * 4
    fn.restype = ctypes.c_int
    return fn


def _small128():
    return synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2, n_src=1, name="small128")


@pytest.mark.parametrize("w,kcb", [(synth.WORKLOADS["tiny"], 0), (_small128(), 0),
                                   (_small128(), 16)],
                         ids=["tiny", "small128", "small128-key-ranges"])
def test_noalloc_backward_matches_workspace_backward(w, kcb):
    """kcb > 0: a plan whose attention kernels walk the blocks in ranges (the
    workspace backward combines per-range partials; the workspace-free one
    walks each list in one pass)."""
    fn = _fn()
    dev = torch.device("cuda")
    x = {k: v.to(dev) for k, v in synth.generate(w, "cpu").items() if torch.is_tensor(v)}
    att = prism.PrismAttention(w, dev, key_chunk_blocks=kcb)
    assert att.plan.sz.key_chunks == (7 if kcb else 1) or w.block != 128
    att.forward(x["Q"], x["K"], x["V"], x["a2v"])
    att.backward(x["dO"])
    torch.cuda.synchronize()
    assert att.status() == 0
    want = [t.clone() for t in (att.dQp, att.dKp, att.dVp)]
    o = att.perm_out
    ptr = prism._ptr
    for _ in range(2):
        got = [torch.full_like(t, float("nan")) for t in want]
        rc = fn(att.plan.h, ptr(o["Qp"]), ptr(o["Kp"]), ptr(o["Vp"]), ptr(att.Op), ptr(att.dOp),
                ptr(att.lse), ptr(o["n_valid"]), ptr(att.lists["row_ptr"]),
                ptr(att.lists["col_idx"]), ptr(att.lists["col_ptr"]),
                ptr(att.lists["row_idx"]), att.scale, ptr(got[0]), ptr(got[1]), ptr(got[2]),
                prism._stream())
        assert rc == 0, prism.ERRORS.get(rc, rc)
        torch.cuda.synchronize()
        for g, r in zip(got, want):
            assert pu.rel_err(pu.f64(g), pu.f64(r)) <= pu.G_TOL


def _status_fn():
    fn = prism.lib().prism_noalloc_device_status
    fn.argtypes = [P]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_reports_a_device_timeout_and_recovers():
    """A bounded wait that runs out inside the workspace-free backward is
    read back by prism_noalloc_device_status; the next call clears it.  The
    failure is made without a fault: a plan with PRISM_FAULT_STARVE_LOADS
    (producer warps issue no loads) and a short wait bound."""
    fn, status = _fn(), _status_fn()
    dev = torch.device("cuda")
    w = _small128()
    x = synth.generate(w, dev)
    good = prism.PrismAttention(w, dev)
    good.forward(x["Q"], x["K"], x["V"], x["a2v"])
    good.backward(x["dO"])
    torch.cuda.synchronize()
    want = [t.clone() for t in (good.dQp, good.dKp, good.dVp)]
    bad = prism.Plan(w, timeout_cycles=2_000_000, fault_inject=prism.FAULT_STARVE_LOADS)
    o, ptr = good.perm_out, prism._ptr

    def call(plan):
        got = [torch.zeros_like(t) for t in want]
        rc = fn(plan.h, ptr(o["Qp"]), ptr(o["Kp"]), ptr(o["Vp"]), ptr(good.Op), ptr(good.dOp),
                ptr(good.lse), ptr(o["n_valid"]), ptr(good.lists["row_ptr"]),
                ptr(good.lists["col_idx"]), ptr(good.lists["col_ptr"]),
                ptr(good.lists["row_idx"]), good.scale, ptr(got[0]), ptr(got[1]), ptr(got[2]),
                prism._stream())
        assert rc == 0
        return got, status(prism._stream())

    _, st = call(good.plan)
    assert st == prism.PRISM_OK
    _, st = call(bad)
    assert st == prism.PRISM_ERR_DEVICE_TIMEOUT
    got, st = call(good.plan)
    assert st == prism.PRISM_OK
    for g, r in zip(got, want):
        assert pu.rel_err(pu.f64(g), pu.f64(r)) <= pu.G_TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _fn()
    plan = prism.Plan(synth.WORKLOADS["2k"])
    fake = P(0x1000)  # aligned, never dereferenced: the size check comes first
    rc = fn(plan.h, *([fake] * 11), 0.1, fake, fake, fake, None)
    assert rc == -3  # PRISM_ERR_UNSUPPORTED

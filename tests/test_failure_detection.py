"""Failure detection without a GPU fault.

Every wait on an mbarrier inside the tensor-core attention kernels is bounded:
when it runs out, the kernel records PRISM_ERR_DEVICE_TIMEOUT (and where) in
the status word of the workspace, frees its tensor memory and returns.  The
failure is made by the test-only PRISM_FAULT_STARVE_LOADS setting, under which
the producer warps issue no loads at all, so no copy is in flight when the
consumers give up.  The test then checks that the CUDA context is still
usable: a normal plan, run again on the same inputs, reproduces its earlier
results bit for bit."""
import pytest
import torch

from content_adaptive_block_02_b300 import build, prism, synth

pytestmark = pytest.mark.gpu

SHORT_LIMIT = 2_000_000     # cycles, about 1 ms
FWD_SITES = range(1, 17)    # wait-site codes of the forward kernel
DKDV_SITES = range(21, 46)  # wait-site codes of the dK/dV kernel (the backward's first)


def _w128():
    return synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2, n_src=1, name="small128")


def _run(att, x):
    O = att.forward(x["Q"], x["K"], x["V"], x["a2v"]).clone()
    dQ, dK, dV = (t.clone() for t in att.backward(x["dO"]))
    return O, dQ, dK, dV


def test_starved_attention_times_out_and_the_context_stays_usable():
    build.build()
    dev = torch.device("cuda", 0)
    w = _w128()
    x = synth.generate(w, dev)
    good = prism.PrismAttention(w, dev)
    assert good.plan.sz.tensor_core_fwd == 1 and good.plan.sz.tensor_core_bwd == 1
    ref = _run(good, x)
    assert good.status() == 0

    bad = prism.PrismAttention(w, dev, timeout_cycles=SHORT_LIMIT,
                               fault_inject=prism.FAULT_STARVE_LOADS)
    # forward: the S / PV issuers and the softmax warps wait for tiles that never come
    bad.forward(x["Q"], x["K"], x["V"], x["a2v"])
    assert bad.status() == prism.PRISM_ERR_DEVICE_TIMEOUT
    info = bad.ws[16:32].view(torch.int32).tolist()    # where, parity, block, thread
    assert info[0] in FWD_SITES, info
    # backward on a cleared status word: the dK/dV kernel times out first
    bad.plan.ws_init(bad.ws)
    bad.backward(x["dO"])
    assert bad.status() == prism.PRISM_ERR_DEVICE_TIMEOUT
    info = bad.ws[16:32].view(torch.int32).tolist()
    assert info[0] in DKDV_SITES, info

    # the context is intact: the normal plan reproduces its results exactly
    again = _run(good, x)
    assert good.status() == 0
    for a, b in zip(ref, again):
        assert torch.equal(a, b)

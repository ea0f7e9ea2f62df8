"""Parity of the CUDA path (called through the C ABI) with the CPU oracle,
step by step, on seeded synthetic inputs.  The contract is stated in
tests/parity_util.py."""
import numpy as np
import pytest
import torch

from content_adaptive_block_02_b300 import build, prism, synth
from oracle import prism_oracle as orc
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    assert torch.cuda.is_available()


def test_tiny_full_pipeline():
    """16-token blocks, d = 64: the whole path, every step."""
    rep = pu.compare(synth.WORKLOADS["tiny"])
    assert rep["O_max_rel"] <= pu.O_TOL


def test_small_ragged_grid_with_padding():
    """5 x 7 x 9 grid: padding on every axis, partially real blocks."""
    w = synth.WORKLOADS["tiny"].with_(T=5, Hg=7, W=9, H=3, name="ragged")
    pu.compare(w)


@pytest.mark.parametrize("kw", [dict(per_head=False), dict(use_video=False),
                                dict(use_audio=False), dict(topp=0.5, topk_floor=1),
                                dict(topp=0.99), dict(topk_floor=0, topp=0.0),
                                dict(alpha=1.0 / 3.0), dict(alpha=2.0)])
def test_tiny_variants(kw):
    w = synth.WORKLOADS["tiny"].with_(**kw)
    pu.compare(w)


def test_topp_one_is_dense_attention():
    """Top-p = 1 keeps every block: the path is plain softmax attention."""
    import numpy as np
    from oracle import prism_oracle as orc
    w = synth.WORKLOADS["tiny"].with_(topp=1.0)
    pu.compare(w)
    inputs = synth.generate(w, "cpu")
    att, g = pu.run_gpu(w, inputs)
    nv = g["n_valid"].numpy()
    for (b, h), L in pu.gpu_lists(w, g, att.plan.nb).items():
        allv = np.nonzero(nv[b, h] > 0)[0]
        for i, sel in enumerate(L):
            assert np.array_equal(sel, allv if nv[b, h, i] > 0 else allv[:0])
    X = {k: pu.f64(inputs[k]) for k in ("Q", "K", "V")}
    for h in range(w.H):
        ref = orc.dense_attention(X["Q"][0, :, h], X["K"][0, :, h], X["V"][0, :, h],
                                  1 / np.sqrt(w.d))
        assert pu.rel_err(pu.f64(g["O"])[0, :, h], ref) <= pu.O_TOL


def _w128(**kw):
    """6 x 40 x 48 grid (padded to 6 x 48 x 48), 3 x 16 x 16 zones, 128-token
    blocks, d = 128: 108 blocks per head, several tiles and ragged padding."""
    base = synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2, n_src=1, name="small128")
    return base.with_(**kw)


@pytest.mark.parametrize("attn_kernel", [0, 1])
def test_128_blocks_both_kernels(attn_kernel):
    rep = pu.compare(_w128(), attn_kernel=attn_kernel)
    assert rep["O_max_rel"] <= pu.O_TOL


@pytest.mark.parametrize("kw", [dict(), dict(topp=1.0), dict(topp=0.5, topk_floor=2)])
def test_128_blocks_key_ranges(kw):
    """The tensor-core forward and dQ kernels walking the key blocks in ranges
    of 16 (7 ranges over 108 blocks, many (query block, range) items empty),
    with the per-range partial results combined afterwards."""
    rep = {}
    pu.compare(_w128(**kw), key_chunk_blocks=16, report=rep)
    assert rep["key_chunks"] == 7


def test_128_blocks_wide_zone():
    """3 x 8 x 32 zones: wider than the register-pencil statistics kernel
    handles (16 tokens per line), so the general statistics kernel runs."""
    pu.compare(_w128(zone=(3, 8, 32)))


def test_128_blocks_full_menu_zone():
    """4 x 16 x 16 zones admit every shape of the 128-token menu."""
    pu.compare(_w128(zone=(4, 16, 16), T=8))


@pytest.mark.parametrize("kw", [dict(topp=0.5), dict(topp=0.99), dict(topk_floor=40),
                                dict(topp=1.0)])
def test_128_blocks_selection_settings(kw):
    pu.compare(_w128(**kw))


# --------------------------------------------------------------------------
# full-size workloads, in the launch configuration of bench.py, on samples
# the oracle can compute one by one
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,heads,kcb", [("720p", [0, 13], (0,)), ("1080p", [5], (0,)),
                                            ("2k", [7], (0, 10 ** 6))])
def test_full_size_sampled(name, heads, kcb):
    """Every query block's list of the sampled heads, O / LSE / dQ on sampled
    query blocks, dK / dV on 8 sampled key blocks (dK held element by element
    to the contract plus its sensitivity to the forward's bf16 O, see
    parity_util.compare_sampled).  At 2K the attention kernels run twice,
    with the key ranges of the bench (bf16 partial results combined
    afterwards) and with one pass over each list, and both are held to the
    contract; the report gives the error of each."""
    rep = pu.compare_sampled(synth.WORKLOADS[name], heads, key_chunk_blocks=kcb)
    print(name, rep)
    assert rep["O"] <= pu.O_TOL and rep["dQ"] <= pu.G_TOL and rep["dKV"] <= pu.ILL_COND_TOL
    assert rep["key_blocks_compared"] >= 8 * len(heads)
    if name == "2k":
        ranges = prism.Plan(synth.WORKLOADS[name]).sz.key_chunks
        assert ranges > 1 and [r["key_chunks"] for r in rep["runs"]] == [ranges, 1]


def test_key_feature_variance_variant():
    """Table 9 caption: the variance can be taken on query / key features
    instead of value features; the statistics step takes any [B, N, H, d]
    tensor, here K, and matches the oracle's statistics of K."""
    w = synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2, n_src=1, name="small128")
    x = synth.generate(w, "cpu")
    dev = torch.device("cuda", 0)
    plan = prism.Plan(w)
    st = plan.zone_stats(x["K"].to(dev), x["a2v"].to(dev))
    torch.cuda.synchronize()
    ref = orc.zone_stats(w, pu.f64(x["K"]), pu.f64(x["a2v"]))
    got = pu.f64(st.cpu())
    for k in range(8):
        scale = max(1e-30, np.abs(ref[..., k]).max())
        assert np.abs(got[..., k] - ref[..., k]).max() / scale <= 2e-5, k


@pytest.mark.parametrize("variant,topp", [("white", 0.9), ("onesrc", 0.9), ("skew", 0.9),
                                          ("white", 0.5), ("onesrc", 0.99), ("skew", 0.99)])
def test_stress_variants(variant, topp):
    """The stress inputs on a small 128-token-block grid: (a) an isotropic
    white field with no anisotropic noise, (b) one audio source zone carrying
    90 % of the A2V norm mass, (c) per-zone noise with a 100:1:1 variance
    ratio along the axes; Top-p 0.5 / 0.9 / 0.99."""
    kw = dict(white=dict(field="white", noise="none"), onesrc=dict(n_src=1, src_mass=0.9),
              skew=dict(noise="skew"))[variant]
    # the white field's source zone gives nearly one-hot softmax rows (logits
    # up to ~110): there dQ and dK cancel to about what the forward's bf16
    # roundings of O move them by, and are checked element by element against
    # that (the oracle's bound terms)
    rep = {}
    pu.compare(_w128(topp=topp, **kw), grad_scale="terms" if variant == "white" else "result",
               report=rep)
    print(variant, topp, rep)


# --------------------------------------------------------------------------
# A2V cross-attention norms on the device (prism_a2v_norms)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,kw", [("tiny", {}), ("small128", {}),
                                     ("small128", dict(Na=37, B=2)),
                                     ("small128", dict(Na=256))])
def test_a2v_norms_match_the_oracle(name, kw):
    """Every token's ||softmax(Qa Ka^T / sqrt(Ca)) Va|| against the oracle:
    Ca = 64 with 32 audio tokens, Ca = 128 with 200, a ragged 37 over two
    batch entries, and the largest 256."""
    w = synth.WORKLOADS["tiny"] if name == "tiny" else _w128()
    w = w.with_(**kw)
    x = synth.generate(w, "cpu")
    dev = torch.device("cuda", 0)
    plan = prism.Plan(w)
    ws = plan.ws(dev)
    au = x["audio"].to(dev)
    n = plan.a2v_norms(x["qa"].to(dev), au, au, ws)
    torch.cuda.synchronize()
    assert plan.device_status(ws) == 0
    ref = orc.a2v_norms(pu.f64(x["qa"]), pu.f64(x["audio"]), pu.f64(x["audio"]))
    err = np.abs(pu.f64(n.cpu()) - ref) / ref
    print(name, kw, "max rel", err.max(), "mean", err.mean())
    assert err.max() <= pu.TAU_N


@pytest.mark.parametrize("w", [synth.WORKLOADS["tiny"], _w128(),
                               _w128(zone=(4, 16, 16), T=8)],
                         ids=["tiny", "small128", "small128-full-menu"])
def test_fused_a2v_pipeline(w):
    """The whole path with the A2V norms computed on the device: statistics
    within what the norm error can move them by, shapes equal to the
    oracle's except on zones that error can flip, every later step under
    the usual contract."""
    rep = {}
    pu.compare(w, fused_a2v=True, report=rep)
    print(w.name, rep)


# --------------------------------------------------------------------------
# block-size classes in one head (Table 11: C_128 and C_256; thresholds tau)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kw,kcb", [(dict(), 0), (dict(zone=(4, 16, 16), T=8), 0),
                                    (dict(zone=(4, 16, 16), T=8), 16),
                                    (dict(zone=(4, 16, 16), T=8, topp=0.5, topk_floor=2), 0)],
                         ids=["3x16x16", "4x16x16", "4x16x16-key-ranges", "4x16x16-p0.5"])
def test_mixed_block_classes(kw, kcb):
    """128- and 256-token blocks mixed within each head, the class of every
    zone from its complexity and the threshold, the shape from Eq. 7 in the
    class; selection over blocks, attention over their tiles."""
    # the small grid's zones sit higher (one source zone: large audio gates
    # everywhere); 1.25 puts about half of them below the threshold
    w = _w128(menu=synth.MENU_128 + synth.MENU_256, class_tau=(1.25,), **kw)
    rep = {}
    pu.compare(w, key_chunk_blocks=kcb, report=rep)
    print(kw, kcb, rep)
    assert rep["multi_tile_blocks"] > 0


def test_mixed_block_classes_cuda_cores():
    """The same on the CUDA-core kernels: 16- and 32-token blocks, d = 64."""
    w = synth.WORKLOADS["tiny"].with_(menu=synth.MENU_TINY + ((2, 4, 4),), class_tau=(1.4,))
    rep = {}
    pu.compare(w, report=rep)
    assert rep["multi_tile_blocks"] > 0


@pytest.mark.parametrize("kw,kcb", [(dict(Hg=32), 0), (dict(Hg=40), 0), (dict(Hg=32), 8),
                                    (dict(Hg=32, topp=0.5, topk_floor=2), 0)],
                         ids=["no-padding", "padding", "key-ranges", "p0.5"])
def test_half_tile_block_classes(kw, kcb):
    """All three classes of Table 11: 64-token blocks (two share a 128-row
    tensor-core tile, with a sub-tile mask per listed tile pair), 128 and 256
    on 4 x 16 x 16 zones; with padding, padded zones skip the 64-token class."""
    w = _w128(zone=(4, 16, 16), T=8, menu=synth.MENU_64 + synth.MENU_128 + synth.MENU_256,
              class_tau=(1.3, 1.15), **kw)
    plan = prism.Plan(w)
    assert plan.sz.half_tile == 1 and plan.sz.slot_tokens == 64
    rep = {}
    pu.compare(w, key_chunk_blocks=kcb, report=rep)
    print(kw, kcb, rep)
    assert rep["half_tile_blocks"] > 0 and rep["masked_entries"] > 0

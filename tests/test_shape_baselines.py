"""Block-shape baselines of the shape ablation (Prism, Table 9: "Random
Shape", "Fixed 4^3"): the zones' block shapes are given by the caller
(prism_permute_shapes) and the rest of the path -- permutation, pooling,
selection, attention forward and backward -- runs through the same kernels.
Both sides get the same shapes; the contract is that of the other parity
tests."""
import os

import numpy as np
import pytest
import torch

from content_adaptive_block_02_b300 import build, prism, synth
from oracle import prism_oracle as orc
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def _w_menu128(**kw):
    """4 x 16 x 16 zones admit every shape of the 128-token menu."""
    base = synth.WORKLOADS["720p"].with_(T=8, Hg=40, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                         name="menu128")
    return base.with_(**kw)


def _random_shapes(w, seed):
    adm = orc.admissible_shapes(w.menu, w.zone)
    rng = np.random.default_rng(seed)
    return rng.choice(adm, size=(w.B, w.H, w.n_zones)).astype(np.uint8)


def test_random_shapes_128_token_menu():
    w = _w_menu128()
    sid = _random_shapes(w, 7)
    assert len(set(sid.ravel().tolist())) >= 4
    rep = pu.compare(w, shape_id=sid)
    assert rep["O_max_rel"] <= pu.O_TOL


@pytest.mark.parametrize("k", [2, 5])  # (2, 8, 8) and (2, 4, 16) everywhere
def test_fixed_shape_128_token_menu(k):
    w = _w_menu128()
    pu.compare(w, shape_id=np.full((w.B, w.H, w.n_zones), k, np.uint8))


def test_fixed_4cubed_64_token_blocks():
    """Fixed 4^3: the single 64-token shape (4, 4, 4) on 4 x 16 x 16 zones
    (64-token blocks run on the CUDA-core attention kernels)."""
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      block=64, menu=((4, 4, 4),), name="fixed4")
    assert prism.Plan(w).sz.tensor_core_fwd == 0
    pu.compare(w, shape_id=np.zeros((w.B, w.H, w.n_zones), np.uint8))


def test_fixed_4cubed_on_tensor_cores():
    """Fixed 4^3 on the tensor cores: the single 64-token shape with a 128-row
    tile, so two blocks share every tile (sub-tile masks); shapes given by the
    caller, grid without padding."""
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      menu=((4, 4, 4),), class_tau=(), name="fixed4_tc")
    plan = prism.Plan(w)
    assert plan.sz.half_tile == 1 and plan.sz.tensor_core_fwd == 1
    rep = pu.compare(w, shape_id=np.zeros((w.B, w.H, w.n_zones), np.uint8))
    assert rep["half_tile_blocks"] > 0 and rep["O_max_rel"] <= pu.O_TOL


def test_shape_that_does_not_tile_the_zone_is_reported():
    """3 x 16 x 16 zones admit only (1, 8, 16) and (1, 16, 8); a given
    (2, 8, 8) or an index past the menu is reported in the status word and
    the zone falls back to the first admissible shape."""
    build.build()
    w = synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2, n_src=1, name="small128")
    assert orc.admissible_shapes(w.menu, w.zone) == [0, 1]
    dev = torch.device("cuda", 0)
    x = synth.generate(w, dev)
    for bad in (2, 200):
        att = prism.PrismAttention(w, dev)
        sid = torch.zeros(w.B, w.H, w.n_zones, dtype=torch.uint8, device=dev)
        sid[0, 1, 3] = bad
        att.forward(x["Q"], x["K"], x["V"], x["a2v"], shape_id=sid)
        assert att.status() == prism.PRISM_ERR_DEVICE_BOUNDS
        info = att.ws[16:32].view(torch.int32).tolist()
        assert info[0] == 0x5A1 and info[1] == bad, info
        # the fallback equals giving shape 0 there
        ref = prism.PrismAttention(w, dev)
        ref.forward(x["Q"], x["K"], x["V"], x["a2v"], shape_id=torch.zeros_like(sid))
        assert ref.status() == 0
        assert torch.equal(att.perm_out["perm"], ref.perm_out["perm"])
        assert torch.equal(att.O, ref.O)


def _table11_class(tokens):
    path = os.path.join(os.path.dirname(__file__), "golden", "table11_shape_names.txt")
    for line in open(path):
        f = line.split()
        if f and not line.startswith("#") and int(f[0]) == tokens:
            return tuple(tuple(int(c) for c in name) for name in f[1:])
    raise KeyError(tokens)


def test_only_c64_menu():
    """"Only C64" (Table 9): the 64-token class of Table 11 as the menu, with
    the zones' shapes from the statistics and Eq. 7 (4 x 16 x 16 zones admit
    five of its seven shapes); 64-token blocks run on the CUDA-core attention."""
    menu = _table11_class(64)
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      block=64, menu=menu, name="only_c64")
    assert len(orc.admissible_shapes(w.menu, w.zone)) == 5
    rep = pu.compare(w)
    assert rep["O_max_rel"] <= pu.O_TOL


def test_only_c64_on_tensor_cores():
    """"Only C64" (Table 9) on the tensor cores: the 64-token menu with a
    128-row tile, so two 64-token blocks share every tile and each listed tile
    pair carries a sub-tile mask; the grid has no padding (a padded zone would
    need a class of at least a tile)."""
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      menu=_table11_class(64), class_tau=(), name="only_c64_tc")
    plan = prism.Plan(w)
    assert plan.sz.half_tile == 1 and plan.sz.tensor_core_fwd == 1 and plan.sz.tensor_core_bwd == 1
    rep = pu.compare(w)
    assert rep["half_tile_blocks"] > 0 and rep["masked_entries"] > 0
    assert rep["O_max_rel"] <= pu.O_TOL


def test_fixed_8cubed_512_token_blocks():
    """Fixed 8^3 (Table 9): the single 512-token shape (8, 8, 8) on 8 x 16 x 16
    zones; every block spans four 128-slot tiles of the tensor-core kernels."""
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, n_src=1, zone=(8, 16, 16),
                                      menu=((8, 8, 8),), name="fixed8")
    plan = prism.Plan(w)
    assert plan.sz.tensor_core_fwd == 1 and plan.sz.multi_tile == 1
    rep = pu.compare(w, shape_id=np.zeros((w.B, w.H, w.n_zones), np.uint8))
    assert rep["multi_tile_blocks"] > 0


def test_only_c256_menu():
    """"Only C256" (Table 9): the 256-token class as the menu, shapes from the
    statistics and Eq. 7 on 4 x 16 x 16 zones (two tiles per block)."""
    w = synth.WORKLOADS["720p"].with_(T=8, Hg=40, W=48, H=2, n_src=1, zone=(4, 16, 16),
                                      menu=synth.MENU_256, name="only_c256")
    rep = pu.compare(w)
    assert rep["multi_tile_blocks"] > 0


def test_random_shapes_across_classes():
    """Random shapes drawn from both the 128- and the 256-token menus: blocks
    of one and of two tiles side by side in every head."""
    w = _w_menu128(menu=synth.MENU_128 + synth.MENU_256, class_tau=(synth.TAU_256,))
    sid = _random_shapes(w, 11)
    rep = pu.compare(w, shape_id=sid)
    assert rep["multi_tile_blocks"] > 0

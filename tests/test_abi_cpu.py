"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, and validates configurations and sizes
on the host exactly as the oracle's geometry says."""
import ctypes

import pytest

from content_adaptive_block_02_b300 import build, prism, synth
from oracle import prism_oracle as orc


@pytest.fixture(scope="module")
def L():
    build.build()
    return prism.lib()


def test_exports_every_declared_function(L):
    names = prism.declared_functions()
    assert len(names) == 19
    for n in names:
        assert hasattr(L, n), n


def test_strerror_names_every_code(L):
    for code in range(0, -8, -1):
        s = L.prism_strerror(code).decode()
        assert s and s != "unknown error"
    assert L.prism_strerror(-99).decode() == "unknown error"


@pytest.mark.parametrize("name", ["tiny", "720p", "1080p", "2k", "2k_long"])
def test_plan_sizes_match_oracle_geometry(L, name):
    w = synth.WORKLOADS[name]
    p = prism.Plan(w)
    Tp, Hp, Wp = orc.padded_grid(w.T, w.Hg, w.W, w.zone)
    assert (p.sz.Tp, p.sz.Hp, p.sz.Wp) == (Tp, Hp, Wp)
    assert p.sz.N == w.N and p.sz.Np == Tp * Hp * Wp == w.Np
    assert p.sz.Z == w.n_zones and p.sz.nb == w.n_blocks
    assert list(p.sz.admissible[: p.sz.n_admissible]) == orc.admissible_shapes(w.menu, w.zone)
    assert p.sz.max_pairs == w.B * w.H * w.n_blocks ** 2
    assert p.sz.ws_bytes > 0


def test_2k_sizes_are_the_documented_ones(L):
    p = prism.Plan(synth.WORKLOADS["2k"])
    assert (p.sz.Np, p.sz.Z, p.sz.nb) == (322_560, 420, 2520)
    assert p.sz.tensor_core_fwd == 1
    # ceil(nb / 900) equal key ranges once a head has more than 1024 key blocks
    assert (p.sz.key_chunks, p.sz.chunk_blocks) == (3, 840)
    assert prism.Plan(synth.WORKLOADS["720p"]).sz.key_chunks == 1
    assert (prism.Plan(synth.WORKLOADS["1080p"]).sz.key_chunks,
            prism.Plan(synth.WORKLOADS["1080p"]).sz.chunk_blocks) == (2, 840)
    small = synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2)
    q = prism.Plan(small, key_chunk_blocks=16)
    assert (q.sz.nb, q.sz.key_chunks, q.sz.chunk_blocks) == (108, 7, 16)
    assert prism.Plan(small, key_chunk_blocks=16, attn_kernel=1).sz.key_chunks == 1
    p1 = prism.Plan(synth.WORKLOADS["2k"], attn_kernel=1)
    assert p1.sz.tensor_core_fwd == 0 and p1.sz.tensor_core_bwd == 0
    assert prism.Plan(synth.WORKLOADS["tiny"]).sz.tensor_core_fwd == 0


def _err(w):
    with pytest.raises(prism.PrismError) as e:
        prism.Plan(w)
    return e.value.code


def test_plan_rejects_bad_configurations(L):
    base = synth.WORKLOADS["tiny"]
    assert _err(base.with_(B=0)) == -1                         # PRISM_ERR_ARG
    assert _err(base.with_(topk_floor=-1)) == -1
    assert _err(base.with_(topp=float("nan"))) == -1
    assert _err(base.with_(d=48)) == -3                        # not a multiple of 32
    assert _err(base.with_(menu=((1, 4, 4), (2, 2, 2)))) == -3  # unequal token counts
    assert _err(base.with_(zone=(3, 3, 3))) == -4              # nothing tiles the zone
    assert _err(base.with_(block=12, menu=((1, 3, 4),))) == -3  # block size not a power of 2


def test_null_pointers_are_rejected_before_any_launch(L):
    p = prism.Plan(synth.WORKLOADS["tiny"])
    assert L.prism_zone_stats(p.h, None, None, None, None) == -1
    assert L.prism_unpermute(p.h, None, None, None, None) == -1
    assert L.prism_plan_query(None, None) == -1


def test_misaligned_pointers_are_rejected_before_any_launch(L):
    p = prism.Plan(synth.WORKLOADS["tiny"])
    bad = ctypes.c_void_p(0x1008)     # never dereferenced: the host check rejects it
    good = ctypes.c_void_p(0x1000)
    assert L.prism_zone_stats(p.h, bad, good, good, None) == -2
    assert L.prism_permute(p.h, good, good, bad, None) == -2


def test_trace_events_can_be_set_and_cleared_without_a_gpu(L):
    # recording only happens when an attention entry point runs; setting and
    # clearing the handles touches no device
    p = prism.Plan(synth.WORKLOADS["tiny"])
    arr = (ctypes.c_void_p * (2 * len(prism.Plan.TRACE_SLOTS)))()
    assert L.prism_plan_set_trace_events(p.h, arr) == 0
    assert L.prism_plan_set_trace_events(p.h, None) == 0
    assert L.prism_plan_set_trace_events(None, None) == -1


def test_unknown_fault_injection_setting_is_rejected(L):
    w = synth.WORKLOADS["tiny"]
    assert prism.Plan(w, fault_inject=prism.FAULT_STARVE_LOADS).cfg.fault_inject == 1
    with pytest.raises(prism.PrismError) as e:
        prism.Plan(w, fault_inject=7)
    assert e.value.code == -1


def test_permute_shapes_rejects_null_pointers(L):
    p = prism.Plan(synth.WORKLOADS["tiny"])
    args = [p.h] + [None] * 16
    assert L.prism_permute_shapes(*args) == -1


def test_key_range_setting_is_validated_and_sized(L):
    w = synth.WORKLOADS["720p"].with_(T=6, Hg=40, W=48, H=2)
    with pytest.raises(prism.PrismError) as e:
        prism.Plan(w, key_chunk_blocks=-1)
    assert e.value.code == -1
    # at most 64 ranges; every block falls in one range
    p = prism.Plan(w, key_chunk_blocks=1)
    assert p.sz.key_chunks == 64 and p.sz.key_chunks * p.sz.chunk_blocks >= p.sz.nb
    # ranges larger than the head: one range, no partial-result workspace
    q = prism.Plan(w, key_chunk_blocks=10_000)
    assert q.sz.key_chunks == 1 and q.sz.ws_bytes < p.sz.ws_bytes


def test_half_tile_only_menu_needs_a_grid_without_padding(L):
    """Only C64 (Table 9) on the tensor cores: 64-token blocks share 128-row
    tiles, so every zone must be full; on a grid without padding the plan
    takes the tensor-core path, on the 2K grid (H = 90, T = 21: padded
    zones) it is rejected, since a padded zone needs a class of at least a
    tile."""
    small = synth.WORKLOADS["720p"].with_(T=8, Hg=32, W=48, H=2, zone=(4, 16, 16),
                                          menu=synth.MENU_64, class_tau=(), name="only_c64_tc")
    p = prism.Plan(small)
    assert (p.sz.half_tile, p.sz.n_classes, p.sz.tensor_core_fwd, p.sz.tensor_core_bwd) == (1, 1, 1, 1)
    with pytest.raises(prism.PrismError) as e:
        prism.Plan(synth.WORKLOADS["2k"].with_(menu=synth.MENU_64, zone=(4, 16, 16), class_tau=()))
    assert prism.ERRORS[e.value.code] == "PRISM_ERR_NO_ADMISSIBLE_SHAPE"


@pytest.mark.parametrize("name", ["tiny", "720p", "2k"])
def test_score_region_lies_inside_the_workspace(L, name):
    """The block scores (fp32 hi then lo, [B, H, nslots, nslots] each) sit at
    a 256-aligned offset inside ws_bytes, and the workspace also holds the
    scores' seven bf16 digit slices of the query and key block means (d
    rounded up to 64 channels) and their int32 exponents after them."""
    w = synth.WORKLOADS[name]
    p = prism.Plan(w)
    R = w.B * w.H * p.sz.nslots
    score_bytes = 2 * 4 * R * p.sz.nslots
    digit_bytes = 2 * (7 * R * ((w.d + 63) // 64 * 64) * 2 + 256) + 2 * 4 * R
    assert p.sz.ws_scores % 256 == 0 and p.sz.ws_scores >= 256
    assert p.sz.ws_scores + score_bytes <= p.sz.ws_bytes
    assert p.sz.ws_bytes >= score_bytes + digit_bytes

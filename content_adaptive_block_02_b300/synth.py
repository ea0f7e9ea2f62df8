"""Seeded synthetic workloads for the Prism block-sparse attention path.

This module is the single source of inputs for both the CUDA path and the CPU
oracle.  It holds workload *descriptions* (grid, zones, block menu, selection
parameters) and a seeded generator of Q/K/V, audio tokens, the
audio-to-video cross-attention output and the upstream gradient.  It does none
of the method's own arithmetic (no statistics, shapes, permutation, pooling,
selection or attention): it only makes data with the structure the Prism pages
describe -- smooth video latents with local, direction-dependent variation and
a few sound-producing regions (Prism, Abstract: "cross-modal interactions are
inherently concentrated around sound-producing regions").

It imports nothing from the package's CUDA binding or from the oracle.

Generator recipe (per head h, seed = seed_base * 1000 + h):
  * F: white N(0,1) field over the real (T, Hg, W) grid and the d channels,
    separably convolved along T, Hg and W with a Gaussian (sigma = 2 tokens,
    radius 6, clamp-to-edge), renormalised to unit variance and scaled by
    ``gamma``.
  * Q = F + eta_Q, K = F + eta_K, V = F + eta_V.  Each eta has variance 0.5 and
    is anisotropic per macro-zone: white along the zone's dominant axis and
    smoothed (sigma = 2) along the other two.  The dominant axis of every zone
    is one seeded uniform draw, shared by all heads.
  * Audio tokens A [Na, Ca] ~ N(0, 1).  In each of ``n_src`` seeded source
    zones, 2 * A[j_z] (a seeded audio index per zone) is added to Q, K and V of
    every token of the zone, in every head.
  * a2v_out_i = softmax(qbar_i A^T / sqrt(Ca)) A, with qbar_i the mean of Q_i
    over heads.  This stands in for the model's audio-to-video cross-attention
    output, which the path takes as an input.
  * dO ~ N(0, 1).
Stress variants: ``field="white"`` drops the smoothing and the anisotropic
noise; ``src_mass`` rescales the first source zone's a2v_out so that it carries
that fraction of the summed per-token norms; ``noise="skew"`` replaces eta by a
sum of three one-axis noises with variance ratio 100:1:1 (dominant axis first).
Every tensor is produced in fp32 and rounded to bf16; both sides of a parity
test consume the same bf16 values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field as dc_field, replace
from typing import Optional, Tuple

import torch

Shape3 = Tuple[int, int, int]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d: int
    T: int
    Hg: int
    W: int
    zone: Shape3
    block: int
    menu: Tuple[Shape3, ...]
    Na: int
    Ca: int
    topk_floor: int
    topp: float
    n_src: int
    gamma: float = 1.0
    seed_base: int = 0
    field: str = "smooth"          # "smooth" | "white"
    noise: str = "aniso"           # "aniso" | "skew" | "none"
    src_mass: Optional[float] = None
    alpha: float = 1.0
    eps: float = 1e-6
    per_head: bool = True
    use_video: bool = True
    use_audio: bool = True
    # block-size class thresholds, descending, one per boundary between the
    # menu's token-count classes (empty for a single-class menu)
    class_tau: Tuple[float, ...] = ()

    @property
    def N(self) -> int:
        return self.T * self.Hg * self.W

    def padded(self) -> Shape3:
        zT, zH, zW = self.zone
        return (-(-self.T // zT) * zT, -(-self.Hg // zH) * zH, -(-self.W // zW) * zW)

    @property
    def Np(self) -> int:
        a, b, c = self.padded()
        return a * b * c

    @property
    def n_zones(self) -> int:
        return self.Np // (self.zone[0] * self.zone[1] * self.zone[2])

    @property
    def n_blocks(self) -> int:
        return self.Np // self.block

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


MENU_TINY = ((1, 4, 4), (2, 2, 4), (2, 4, 2), (1, 2, 8), (1, 8, 2))
MENU_128 = ((1, 8, 16), (1, 16, 8), (2, 8, 8), (4, 4, 8), (4, 8, 4), (2, 4, 16), (2, 16, 4))
# 256-token class: Table 11's 488 and the other power-of-two shapes that fit a
# 16 x 16 frame patch
MENU_256 = ((4, 8, 8), (2, 8, 16), (2, 16, 8), (4, 4, 16), (4, 16, 4), (1, 16, 16))
# 64-token class: Table 11's shapes whose extents fit a 4 x 16 x 16 zone
MENU_64 = ((4, 4, 4), (2, 4, 8), (2, 8, 4), (4, 2, 8), (4, 8, 2))
# threshold between the 128- and 256-token classes (zone complexity; about
# half the zones of the smooth-field grids fall below it)
TAU_256 = 0.9
# threshold between the 64- and 128-token classes (about the top fifth of the
# smooth-field grids' zones lie above it)
TAU_128 = 1.3

# Block-mean field gain: chosen once so that the 720p-like grid at Top-p 0.9,
# Top-k floor 8 lands in the 85-90 % block-sparsity band (88.6 % measured on
# head 0 by the oracle), then frozen.
GAMMA = 1.95

WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, d=64, T=4, Hg=8, W=8, zone=(2, 4, 4), block=16,
                     menu=MENU_TINY, Na=32, Ca=64, topk_floor=2, topp=0.9, n_src=1,
                     gamma=GAMMA, seed_base=0),
    "720p": Workload("720p", B=1, H=24, d=128, T=21, Hg=45, W=80, zone=(3, 16, 16), block=128,
                     menu=MENU_128, Na=200, Ca=128, topk_floor=8, topp=0.9, n_src=2,
                     gamma=GAMMA, seed_base=1),
    "1080p": Workload("1080p", B=1, H=24, d=128, T=21, Hg=68, W=120, zone=(3, 16, 16), block=128,
                      menu=MENU_128, Na=200, Ca=128, topk_floor=8, topp=0.9, n_src=3,
                      gamma=GAMMA, seed_base=2),
    "2k": Workload("2k", B=1, H=24, d=128, T=21, Hg=90, W=160, zone=(3, 16, 16), block=128,
                   menu=MENU_128, Na=200, Ca=128, topk_floor=8, topp=0.9, n_src=3,
                   gamma=GAMMA, seed_base=3),
    "2k_long": Workload("2k_long", B=1, H=12, d=128, T=41, Hg=90, W=160, zone=(3, 16, 16),
                        block=128, menu=MENU_128, Na=200, Ca=128, topk_floor=8, topp=0.9,
                        n_src=3, gamma=GAMMA, seed_base=4),
}
# Mixed block-size classes (Table 11: C_128 and C_256 in one head, thresholds
# tau): the 2K grid with 128- and 256-token blocks; 3 x 16 x 16 zones admit
# (1,8,16), (1,16,8) and (1,16,16), 4 x 16 x 16 zones every shape of both menus.
WORKLOADS["2k_mc"] = WORKLOADS["2k"].with_(name="2k_mc", menu=MENU_128 + MENU_256,
                                           class_tau=(TAU_256,))
WORKLOADS["2k_mc4"] = WORKLOADS["2k"].with_(name="2k_mc4", zone=(4, 16, 16),
                                            menu=MENU_128 + MENU_256, class_tau=(TAU_256,))
# all three classes of Table 11 (C_64, C_128, C_256) on 4 x 16 x 16 zones; two
# 64-token blocks share one 128-row tensor-core tile
WORKLOADS["2k_mc3"] = WORKLOADS["2k"].with_(name="2k_mc3", zone=(4, 16, 16),
                                            menu=MENU_64 + MENU_128 + MENU_256,
                                            class_tau=(TAU_128, TAU_256))


def stress(base: str, variant: str, topp: float) -> Workload:
    """Stress sweep cases on the 2K-like grids: (a) isotropic white field,
    (b) one audio source zone carrying 90 % of the A2V norm mass, (c) strongly
    axis-skewed per-zone variance."""
    w = WORKLOADS[base].with_(topp=topp, name=f"{base}_{variant}_p{topp}")
    if variant == "white":
        return w.with_(field="white", noise="none")
    if variant == "onesrc":
        return w.with_(n_src=1, src_mass=0.9)
    if variant == "skew":
        return w.with_(noise="skew")
    raise ValueError(variant)


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def _gauss_kernel(sigma: float = 2.0, radius: int = 6, device="cpu") -> torch.Tensor:
    x = torch.arange(-radius, radius + 1, dtype=torch.float32, device=device)
    k = torch.exp(-0.5 * (x / sigma) ** 2)
    return k / k.sum()


def _smooth(x: torch.Tensor, axis: int, kern: torch.Tensor) -> torch.Tensor:
    """Convolve ``x`` along ``axis`` with ``kern`` (clamp-to-edge)."""
    r = (kern.numel() - 1) // 2
    xm = x.movedim(axis, -1)
    shp = xm.shape
    flat = xm.reshape(-1, 1, shp[-1])
    flat = torch.nn.functional.pad(flat, (r, r), mode="replicate")
    out = torch.nn.functional.conv1d(flat, kern.view(1, 1, -1))
    return out.reshape(shp).movedim(-1, axis)


def _zone_index(w: Workload, device) -> torch.Tensor:
    """Zone id of every real token, raster (zt, zh, zw) over the padded zone grid."""
    zT, zH, zW = w.zone
    Tp, Hp, Wp = w.padded()
    t = torch.arange(w.T, device=device) // zT
    h = torch.arange(w.Hg, device=device) // zH
    x = torch.arange(w.W, device=device) // zW
    nzh, nzw = Hp // zH, Wp // zW
    return (t.view(-1, 1, 1) * nzh + h.view(1, -1, 1)) * nzw + x.view(1, 1, -1)


def generate(w: Workload, device="cpu", want_dO: bool = True, a2v_f32: bool = False) -> dict:
    """Return a dict of bf16 tensors Q, K, V, dO [B, N, H, d], a2v [B, N, Ca],
    the A2V queries qa [B, N, Ca] (the head-mean of Q, rounded to bf16) and
    audio [B, Na, Ca], plus the source-zone ids (for reports).  a2v is
    computed from qa and audio as they are stored (bf16); with ``a2v_f32``
    its fp32 value before that rounding is returned too, as a2v_f32."""
    dev = torch.device(device)
    kern = _gauss_kernel(device=dev)
    zid = _zone_index(w, dev)                       # [T,Hg,W]
    out = {k: torch.empty(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=dev)
           for k in (["Q", "K", "V"] + (["dO"] if want_dO else []))}
    a2v = torch.empty(w.B, w.N, w.Ca, dtype=torch.bfloat16, device=dev)
    qa_all = torch.empty(w.B, w.N, w.Ca, dtype=torch.bfloat16, device=dev)
    a2v32 = torch.empty(w.B, w.N, w.Ca, dtype=torch.float32, device=dev) if a2v_f32 else None
    audio_all = torch.empty(w.B, w.Na, w.Ca, dtype=torch.bfloat16, device=dev)
    src_zones_all = []
    for b in range(w.B):
        gz = torch.Generator(device=dev).manual_seed(w.seed_base * 7919 + b)
        dom = torch.randint(0, 3, (w.n_zones,), generator=gz, device=dev)     # dominant axis per zone
        src = torch.randperm(w.n_zones, generator=gz, device=dev)[: w.n_src]
        # only zones that hold real tokens can be sources
        real = torch.unique(zid)
        if not bool(torch.isin(src, real).all()):
            src = real[torch.randperm(real.numel(), generator=gz, device=dev)[: w.n_src]]
        j_src = torch.randint(0, w.Na, (w.n_src,), generator=gz, device=dev)
        A = torch.randn(w.Na, w.Ca, generator=gz, device=dev)
        A = A.bfloat16().float()
        audio_all[b] = A.bfloat16()
        src_zones_all.append(src.tolist())
        src_add = torch.zeros(w.T, w.Hg, w.W, w.Ca, device=dev)
        for z, j in zip(src.tolist(), j_src.tolist()):
            src_add[zid == z] += 2.0 * A[j]
        dom_tok = dom[zid]                                                    # [T,Hg,W]
        qsum = torch.zeros(w.T, w.Hg, w.W, w.d, device=dev)
        for h in range(w.H):
            g = torch.Generator(device=dev).manual_seed(w.seed_base * 1000 + h + 100000 * b)
            F = torch.randn(w.T, w.Hg, w.W, w.d, generator=g, device=dev)
            if w.field == "smooth":
                for ax in range(3):
                    F = _smooth(F, ax, kern)
            F = F / F.std()
            F = F * w.gamma
            for name in ("Q", "K", "V"):
                X = F + _noise(w, g, dev, kern, dom_tok)
                if w.Ca == w.d:
                    X = X + src_add
                X = X.bfloat16()
                out[name][b, :, h, :] = X.reshape(w.N, w.d)
                if name == "Q":
                    qsum += X.float()
            if want_dO:
                out["dO"][b, :, h, :] = torch.randn(w.N, w.d, generator=g, device=dev).bfloat16()
        qbar = (qsum / w.H).reshape(w.N, w.d)
        qa = torch.zeros(w.N, w.Ca, device=dev)
        qa[:, : min(w.Ca, w.d)] = qbar[:, : w.Ca]
        qa = qa.bfloat16()
        qa_all[b] = qa
        att = torch.softmax(qa.float() @ A.t() / math.sqrt(w.Ca), dim=-1)
        a2 = att @ A                                                          # [N, Ca]
        if w.src_mass is not None:
            n = a2.norm(dim=-1)
            inz = (zid.reshape(-1) == src[0])
            m_in, m_out = n[inz].sum(), n[~inz].sum()
            f = w.src_mass / (1.0 - w.src_mass) * m_out / m_in
            a2[inz] *= f
        a2v[b] = a2.bfloat16()
        if a2v32 is not None:
            a2v32[b] = a2
    out["a2v"] = a2v
    out["qa"] = qa_all
    if a2v32 is not None:
        out["a2v_f32"] = a2v32
    out["audio"] = audio_all
    out["src_zones"] = src_zones_all
    return out


def _noise(w: Workload, g, dev, kern, dom_tok) -> torch.Tensor:
    shp = (w.T, w.Hg, w.W, w.d)
    if w.field == "white" or w.noise == "none":
        return torch.zeros(shp, device=dev)
    if w.noise == "aniso":
        eta = torch.zeros(shp, device=dev)
        for ax in range(3):
            e = torch.randn(shp, generator=g, device=dev)
            for other in range(3):
                if other != ax:
                    e = _smooth(e, other, kern)
            e = e / e.std() * math.sqrt(0.5)
            eta = torch.where((dom_tok == ax).unsqueeze(-1), e, eta)
        return eta
    if w.noise == "skew":
        # three noises, each varying along one axis only, std ratio 10:1:1
        comps = []
        for ax in range(3):
            sz = [1, 1, 1, w.d]
            sz[ax] = shp[ax]
            comps.append(torch.randn(sz, generator=g, device=dev).expand(shp))
        eta = torch.zeros(shp, device=dev)
        for ax in range(3):
            s = torch.ones(3, device=dev)
            s[ax] = 10.0
            mix = s[0] * comps[0] + s[1] * comps[1] + s[2] * comps[2]
            eta = torch.where((dom_tok == ax).unsqueeze(-1), mix, eta)
        return eta / eta.std() * math.sqrt(0.5)
    raise ValueError(w.noise)

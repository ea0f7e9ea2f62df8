"""Thin ctypes binding of the Prism C ABI (``include/prism.h``).

Argument marshalling only: every step of the path runs in the CUDA library
``libprism.so`` built from ``csrc/``.  PyTorch provides device memory and the
current stream.  There is no CPU fallback: if the library is missing, or no
CUDA device is present, the calls raise.

Names follow the C ABI: ``zone_stats``, ``assign_and_permute``,
``block_select``, ``sparse_attn_fwd``, ``permute``, ``sparse_attn_bwd``,
``unpermute``.  ``PrismAttention`` chains them into the forward and backward
of one Prism attention layer.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libprism.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "prism.h")
MAX_SHAPES = 32
MAX_CLASSES = 3

ERRORS = {
    0: "PRISM_OK", -1: "PRISM_ERR_ARG", -2: "PRISM_ERR_ALIGN", -3: "PRISM_ERR_UNSUPPORTED",
    -4: "PRISM_ERR_NO_ADMISSIBLE_SHAPE", -5: "PRISM_ERR_CUDA", -6: "PRISM_ERR_DEVICE_TIMEOUT",
    -7: "PRISM_ERR_DEVICE_BOUNDS",
}


class PrismError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({_lib_strerror(code)})")


class Config(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int),
        ("T", ctypes.c_int), ("Hg", ctypes.c_int), ("W", ctypes.c_int),
        ("zT", ctypes.c_int), ("zH", ctypes.c_int), ("zW", ctypes.c_int),
        ("block_tokens", ctypes.c_int), ("n_shapes", ctypes.c_int),
        ("shapes", (ctypes.c_int * 3) * MAX_SHAPES), ("Ca", ctypes.c_int),
        ("alpha", ctypes.c_double), ("eps", ctypes.c_double),
        ("per_head", ctypes.c_int), ("use_video", ctypes.c_int), ("use_audio", ctypes.c_int),
        ("topk_floor", ctypes.c_int), ("topp", ctypes.c_float),
        ("timeout_cycles", ctypes.c_ulonglong), ("attn_kernel", ctypes.c_int),
        ("fault_inject", ctypes.c_int), ("key_chunk_blocks", ctypes.c_int),
        ("class_tau", ctypes.c_double * (MAX_CLASSES - 1)),
    ]


FAULT_STARVE_LOADS = 1   # PRISM_FAULT_STARVE_LOADS: failure-detection tests only
PRISM_OK = 0
PRISM_ERR_DEVICE_TIMEOUT = -6
PRISM_ERR_DEVICE_BOUNDS = -7


class Sizes(ctypes.Structure):
    _fields_ = [
        ("Tp", ctypes.c_int), ("Hp", ctypes.c_int), ("Wp", ctypes.c_int),
        ("nzT", ctypes.c_int), ("nzH", ctypes.c_int), ("nzW", ctypes.c_int),
        ("Z", ctypes.c_int), ("nb", ctypes.c_int), ("blocks_per_zone", ctypes.c_int),
        ("N", ctypes.c_longlong), ("Np", ctypes.c_longlong),
        ("n_admissible", ctypes.c_int), ("admissible", ctypes.c_int * MAX_SHAPES),
        ("max_pairs", ctypes.c_longlong), ("ws_bytes", ctypes.c_size_t),
        ("tensor_core_fwd", ctypes.c_int), ("tensor_core_bwd", ctypes.c_int),
        ("key_chunks", ctypes.c_int), ("chunk_blocks", ctypes.c_int),
        ("n_classes", ctypes.c_int), ("class_tokens", ctypes.c_int * MAX_CLASSES),
        ("multi_tile", ctypes.c_int), ("slot_tokens", ctypes.c_int), ("nslots", ctypes.c_int),
        ("half_tile", ctypes.c_int), ("ws_csr_mask", ctypes.c_size_t),
        ("ws_csc_mask", ctypes.c_size_t), ("ws_scores", ctypes.c_size_t),
    ]


_LIB: Optional[ctypes.CDLL] = None
P = ctypes.c_void_p


def declared_functions():
    """Names of the functions ``include/prism.h`` declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(prism_\w+)\(", text, re.M)))


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libprism.so not built ({LIB_PATH}); run content_adaptive_block_02_b300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "prism_plan_create": [ctypes.POINTER(Config), ctypes.POINTER(P)],
        "prism_plan_destroy": [P],
        "prism_plan_query": [P, ctypes.POINTER(Sizes)],
        "prism_ws_init": [P, P, P],
        "prism_device_status": [P, P, P],
        "prism_strerror": [ctypes.c_int],
        "prism_zone_stats": [P, P, P, P, P],
        "prism_assign_and_permute": [P] + [P] * 17,
        "prism_block_select": [P] + [P] * 13,
        "prism_sparse_attn_fwd": [P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P],
        "prism_permute": [P, P, P, P, P],
        "prism_sparse_attn_bwd": [P] + [P] * 11 + [ctypes.c_float] + [P] * 5,
        "prism_unpermute": [P, P, P, P, P],
        "prism_plan_set_trace_events": [P, P],
        "prism_permute_shapes": [P] * 17,
        "prism_a2v_norms": [P, P, P, P, ctypes.c_int, P, P, P],
        "prism_zone_stats_norms": [P, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = None if name == "prism_plan_destroy" else ctypes.c_int
    L.prism_strerror.restype = ctypes.c_char_p
    _LIB = L
    return L


def _lib_strerror(code: int) -> str:
    try:
        return lib().prism_strerror(code).decode()
    except Exception:  # pragma: no cover - library missing
        return "?"


def _check(code: int, where: str):
    if code != 0:
        raise PrismError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def make_config(w, timeout_cycles: int = 0, attn_kernel: int = 0,
                fault_inject: int = 0, key_chunk_blocks: int = 0) -> Config:
    """Config from a workload description (``synth.Workload``-like object)."""
    c = Config()
    c.B, c.H, c.d = w.B, w.H, w.d
    c.T, c.Hg, c.W = w.T, w.Hg, w.W
    c.zT, c.zH, c.zW = w.zone
    c.block_tokens = w.block
    c.n_shapes = len(w.menu)
    for k, s in enumerate(w.menu):
        for a in range(3):
            c.shapes[k][a] = s[a]
    c.Ca = w.Ca
    c.alpha, c.eps = w.alpha, w.eps
    c.per_head = int(w.per_head)
    c.use_video, c.use_audio = int(w.use_video), int(w.use_audio)
    c.topk_floor = w.topk_floor
    c.topp = w.topp
    c.timeout_cycles = timeout_cycles
    c.attn_kernel = attn_kernel
    c.fault_inject = fault_inject
    c.key_chunk_blocks = key_chunk_blocks
    for q, t in enumerate(tuple(getattr(w, "class_tau", ()) or ())[:MAX_CLASSES - 1]):
        c.class_tau[q] = t
    return c


class Plan:
    """Host plan of one problem size (prism_plan_create / prism_plan_query)."""

    def __init__(self, w, timeout_cycles: int = 0, attn_kernel: int = 0, fault_inject: int = 0,
                 key_chunk_blocks: int = 0):
        self.w = w
        self.cfg = make_config(w, timeout_cycles, attn_kernel, fault_inject, key_chunk_blocks)
        h = ctypes.c_void_p()
        _check(lib().prism_plan_create(ctypes.byref(self.cfg), ctypes.byref(h)), "prism_plan_create")
        self.h = h
        s = Sizes()
        _check(lib().prism_plan_query(self.h, ctypes.byref(s)), "prism_plan_query")
        self.sz = s

    def __del__(self):
        h = getattr(self, "h", None)
        if h is not None and h.value and _LIB is not None:
            _LIB.prism_plan_destroy(h)
            self.h = None

    # sizes
    @property
    def nb(self):
        return self.sz.nb

    @property
    def Np(self):
        return self.sz.Np

    @property
    def Z(self):
        return self.sz.Z

    # ---- entry points ----
    def ws(self, device="cuda") -> torch.Tensor:
        t = torch.empty(self.sz.ws_bytes, dtype=torch.uint8, device=device)
        _check(lib().prism_ws_init(self.h, _ptr(t), _stream()), "prism_ws_init")
        return t

    def ws_init(self, ws: torch.Tensor):
        """prism_ws_init: clear the status word of an existing workspace."""
        _check(lib().prism_ws_init(self.h, _ptr(ws), _stream()), "prism_ws_init")

    def device_status(self, ws: torch.Tensor) -> int:
        return lib().prism_device_status(self.h, _ptr(ws), _stream())

    TRACE_SLOTS = ("attn_fwd", "bwd_pre", "attn_dkdv", "attn_dq", "zone_stats", "permute_pool",
                   "score", "select")

    def set_trace_events(self, events=None):
        """prism_plan_set_trace_events: `events` maps a slot name of
        TRACE_SLOTS to a (begin, end) pair of torch.cuda.Event(enable_timing=True),
        or is None to clear every slot.  Each event is recorded once here on
        the current stream so that its CUDA handle exists."""
        if events is None:
            _check(lib().prism_plan_set_trace_events(self.h, None), "prism_plan_set_trace_events")
            self._trace_keep = None
            return
        arr = (ctypes.c_void_p * (2 * len(self.TRACE_SLOTS)))()
        for i, name in enumerate(self.TRACE_SLOTS):
            pair = events.get(name)
            if pair is None:
                continue
            for j, e in enumerate(pair):
                if e.cuda_event == 0:
                    e.record(torch.cuda.current_stream())
                arr[2 * i + j] = e.cuda_event
        self._trace_keep = events
        _check(lib().prism_plan_set_trace_events(self.h, arr), "prism_plan_set_trace_events")

    def zone_stats(self, V, a2v, stats=None):
        w = self.w
        if stats is None:
            stats = torch.empty(w.B, w.H, self.Z, 8, dtype=torch.float32, device=V.device)
        _check(lib().prism_zone_stats(self.h, _ptr(V), _ptr(a2v), _ptr(stats), _stream()),
               "prism_zone_stats")
        return stats

    def a2v_norms(self, Qa, Ka, Va, ws, n=None):
        """prism_a2v_norms: per-token norms [B, N] (fp32) of the A2V
        cross-attention output, from the queries Qa [B, N, Ca] and the audio
        keys / values Ka, Va [B, Na, Ca] (bf16)."""
        w = self.w
        if n is None:
            n = torch.empty(w.B, w.N, dtype=torch.float32, device=Qa.device)
        _check(lib().prism_a2v_norms(self.h, _ptr(Qa), _ptr(Ka), _ptr(Va), int(Ka.shape[1]),
                                     _ptr(n), _ptr(ws), _stream()), "prism_a2v_norms")
        return n

    def zone_stats_norms(self, V, n, stats=None):
        """prism_zone_stats_norms: zone statistics from the A2V norms n [B, N]."""
        w = self.w
        if stats is None:
            stats = torch.empty(w.B, w.H, self.Z, 8, dtype=torch.float32, device=V.device)
        _check(lib().prism_zone_stats_norms(self.h, _ptr(V), _ptr(n), _ptr(stats), _stream()),
               "prism_zone_stats_norms")
        return stats

    def alloc_permuted(self, device):
        w = self.w
        e = dict(device=device)
        return dict(
            shape_id=torch.empty(w.B, w.H, self.Z, dtype=torch.uint8, **e),
            shape_tie=torch.empty(w.B, w.H, self.Z, dtype=torch.uint8, **e),
            perm=torch.empty(w.B, w.H, self.Np, dtype=torch.int32, **e),
            inv=torch.empty(w.B, w.H, w.N, dtype=torch.int32, **e),
            Qp=torch.empty(w.B, w.H, self.Np, w.d, dtype=torch.bfloat16, **e),
            Kp=torch.empty(w.B, w.H, self.Np, w.d, dtype=torch.bfloat16, **e),
            Vp=torch.empty(w.B, w.H, self.Np, w.d, dtype=torch.bfloat16, **e),
            Qbar=torch.empty(w.B, w.H, self.sz.nslots, w.d, dtype=torch.float32, **e),
            Qbar_lo=torch.empty(w.B, w.H, self.sz.nslots, w.d, dtype=torch.float32, **e),
            Kbar=torch.empty(w.B, w.H, self.sz.nslots, w.d, dtype=torch.float32, **e),
            Kbar_lo=torch.empty(w.B, w.H, self.sz.nslots, w.d, dtype=torch.float32, **e),
            n_valid=torch.empty(w.B, w.H, self.nb, dtype=torch.int32, **e),
        )

    def assign_and_permute(self, stats, Q, K, V, out=None):
        o = out if out is not None else self.alloc_permuted(Q.device)
        _check(lib().prism_assign_and_permute(
            self.h, _ptr(stats), _ptr(Q), _ptr(K), _ptr(V), _ptr(o["shape_id"]),
            _ptr(o["shape_tie"]), _ptr(o["perm"]), _ptr(o["inv"]), _ptr(o["Qp"]), _ptr(o["Kp"]),
            _ptr(o["Vp"]), _ptr(o["Qbar"]), _ptr(o["Qbar_lo"]), _ptr(o["Kbar"]),
            _ptr(o["Kbar_lo"]), _ptr(o["n_valid"]), _stream()), "prism_assign_and_permute")
        return o

    def permute_shapes(self, shape_id, Q, K, V, ws, out=None):
        """prism_permute_shapes: step 2 with caller-given shape ids
        ([B, H, Z] uint8 menu indices) instead of Eq. 7; the ids are copied
        into ``out["shape_id"]``."""
        o = out if out is not None else self.alloc_permuted(Q.device)
        o["shape_id"].copy_(shape_id)
        o["shape_tie"].zero_()
        _check(lib().prism_permute_shapes(
            self.h, _ptr(o["shape_id"]), _ptr(Q), _ptr(K), _ptr(V), _ptr(o["perm"]),
            _ptr(o["inv"]), _ptr(o["Qp"]), _ptr(o["Kp"]), _ptr(o["Vp"]), _ptr(o["Qbar"]),
            _ptr(o["Qbar_lo"]), _ptr(o["Kbar"]), _ptr(o["Kbar_lo"]), _ptr(o["n_valid"]),
            _ptr(ws), _stream()), "prism_permute_shapes")
        return o

    def alloc_lists(self, device):
        w = self.w
        rows = w.B * w.H * self.nb
        e = dict(device=device, dtype=torch.int32)
        return dict(
            row_ptr=torch.empty(rows + 1, **e), col_idx=torch.empty(max(self.sz.max_pairs, 4), **e),
            col_ptr=torch.empty(rows + 1, **e), row_idx=torch.empty(max(self.sz.max_pairs, 4), **e),
            sel_tie=torch.empty(w.B, w.H, self.sz.nslots, dtype=torch.uint8, device=device),
        )

    def block_select(self, shape_id, Qbar, Qbar_lo, Kbar, Kbar_lo, n_valid, ws, out=None):
        o = out if out is not None else self.alloc_lists(Qbar.device)
        _check(lib().prism_block_select(
            self.h, _ptr(shape_id), _ptr(Qbar), _ptr(Qbar_lo), _ptr(Kbar), _ptr(Kbar_lo),
            _ptr(n_valid),
            _ptr(o["row_ptr"]), _ptr(o["col_idx"]), _ptr(o["col_ptr"]), _ptr(o["row_idx"]),
            _ptr(o["sel_tie"]), _ptr(ws), _stream()), "prism_block_select")
        return o

    def sparse_attn_fwd(self, Qp, Kp, Vp, n_valid, row_ptr, col_idx, scale, ws, Op=None, lse=None):
        w = self.w
        if Op is None:
            Op = torch.empty_like(Qp)
        if lse is None:
            lse = torch.empty(w.B, w.H, self.Np, dtype=torch.float32, device=Qp.device)
        _check(lib().prism_sparse_attn_fwd(
            self.h, _ptr(Qp), _ptr(Kp), _ptr(Vp), _ptr(n_valid), _ptr(row_ptr), _ptr(col_idx),
            float(scale), _ptr(Op), _ptr(lse), _ptr(ws), _stream()), "prism_sparse_attn_fwd")
        return Op, lse

    def permute(self, perm, X, Xp=None):
        w = self.w
        if Xp is None:
            Xp = torch.empty(w.B, w.H, self.Np, w.d, dtype=X.dtype, device=X.device)
        _check(lib().prism_permute(self.h, _ptr(perm), _ptr(X), _ptr(Xp), _stream()),
               "prism_permute")
        return Xp

    def sparse_attn_bwd(self, Qp, Kp, Vp, Op, dOp, lse, n_valid, lists, scale, ws,
                        dQp=None, dKp=None, dVp=None):
        dQp = torch.empty_like(Qp) if dQp is None else dQp
        dKp = torch.empty_like(Kp) if dKp is None else dKp
        dVp = torch.empty_like(Vp) if dVp is None else dVp
        _check(lib().prism_sparse_attn_bwd(
            self.h, _ptr(Qp), _ptr(Kp), _ptr(Vp), _ptr(Op), _ptr(dOp), _ptr(lse), _ptr(n_valid),
            _ptr(lists["row_ptr"]), _ptr(lists["col_idx"]), _ptr(lists["col_ptr"]),
            _ptr(lists["row_idx"]), float(scale), _ptr(dQp), _ptr(dKp), _ptr(dVp), _ptr(ws),
            _stream()), "prism_sparse_attn_bwd")
        return dQp, dKp, dVp

    def unpermute(self, inv, Xp, X=None):
        w = self.w
        if X is None:
            X = torch.empty(w.B, w.N, w.H, w.d, dtype=Xp.dtype, device=Xp.device)
        _check(lib().prism_unpermute(self.h, _ptr(inv), _ptr(Xp), _ptr(X), _stream()),
               "prism_unpermute")
        return X


class PrismAttention:
    """Forward and backward of one Prism attention layer through the C ABI.

    ``forward(Q, K, V, a2v)`` runs zone statistics -> shapes and permutation
    (with pooling) -> block selection -> sparse attention -> inverse
    permutation and returns O [B, N, H, d]; ``backward(dO)`` returns
    (dQ, dK, dV) in the same layout.  Buffers are allocated once per plan and
    reused across calls."""

    def __init__(self, w, device="cuda", attn_kernel: int = 0, timeout_cycles: int = 0,
                 fault_inject: int = 0, key_chunk_blocks: int = 0):
        self.w = w
        self.plan = Plan(w, timeout_cycles=timeout_cycles, attn_kernel=attn_kernel,
                         fault_inject=fault_inject, key_chunk_blocks=key_chunk_blocks)
        self.device = torch.device(device)
        self.scale = 1.0 / math.sqrt(w.d)
        self.ws = self.plan.ws(self.device)
        self.stats = torch.empty(w.B, w.H, self.plan.Z, 8, dtype=torch.float32, device=self.device)
        self.perm_out = self.plan.alloc_permuted(self.device)
        self.lists = self.plan.alloc_lists(self.device)
        self.Op = torch.empty(w.B, w.H, self.plan.Np, w.d, dtype=torch.bfloat16, device=self.device)
        self.lse = torch.empty(w.B, w.H, self.plan.Np, dtype=torch.float32, device=self.device)
        self.O = torch.empty(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=self.device)
        self.dOp = torch.empty_like(self.Op)
        self.dQp, self.dKp, self.dVp = (torch.empty_like(self.Op) for _ in range(3))
        self.dQ, self.dK, self.dV = (torch.empty_like(self.O) for _ in range(3))

    def forward(self, Q, K, V, a2v=None, shape_id=None, qa=None, audio=None):
        """The A2V signal is either the cross-attention output ``a2v``
        [B, N, Ca], or its queries ``qa`` [B, N, Ca] and the audio tokens
        ``audio`` [B, Na, Ca] (keys and values), from which the norms are
        computed on the device (prism_a2v_norms).  ``shape_id`` ([B, H, Z]
        uint8, optional): block shapes given by the caller (fixed / random
        baselines) instead of the zone statistics and Eq. 7; the A2V signal is
        then unused."""
        p, o = self.plan, self.perm_out
        if shape_id is None:
            if qa is not None:
                self.nrm = p.a2v_norms(qa, audio, audio, self.ws, getattr(self, "nrm", None))
                p.zone_stats_norms(V, self.nrm, self.stats)
            else:
                p.zone_stats(V, a2v, self.stats)
            p.assign_and_permute(self.stats, Q, K, V, o)
        else:
            p.permute_shapes(shape_id, Q, K, V, self.ws, o)
        p.block_select(o["shape_id"], o["Qbar"], o["Qbar_lo"], o["Kbar"], o["Kbar_lo"],
                       o["n_valid"], self.ws, self.lists)
        p.sparse_attn_fwd(o["Qp"], o["Kp"], o["Vp"], o["n_valid"], self.lists["row_ptr"],
                          self.lists["col_idx"], self.scale, self.ws, self.Op, self.lse)
        p.unpermute(o["inv"], self.Op, self.O)
        return self.O

    def backward(self, dO):
        p, o = self.plan, self.perm_out
        p.permute(o["perm"], dO, self.dOp)
        p.sparse_attn_bwd(o["Qp"], o["Kp"], o["Vp"], self.Op, self.dOp, self.lse, o["n_valid"],
                          self.lists, self.scale, self.ws, self.dQp, self.dKp, self.dVp)
        p.unpermute(o["inv"], self.dQp, self.dQ)
        p.unpermute(o["inv"], self.dKp, self.dK)
        p.unpermute(o["inv"], self.dVp, self.dV)
        return self.dQ, self.dK, self.dV

    def status(self) -> int:
        return self.plan.device_status(self.ws)

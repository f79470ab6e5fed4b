"""ORACLE — test infrastructure only.

ctypes wrapper around ``oracle.c``, a plain CPU restatement of the MegaMoE
expert path (route -> L1 -> SwiGLU x top-k weight -> UE8M0/E4M3 requantise ->
L2 -> BF16 per slot -> FP32 combine -> BF16). Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import this package; the CUDA library
never does.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against library routines (PyTorch FP8/FP4/BF16
casts, NumPy float64 matmul, stable argsort), closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "oracle.c")


def so_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, "liborc.so" if mutant == 0 else f"liborc_m{mutant}.so")


def build(mutant: int = 0, verbose: bool = False) -> str:
    """Compile the oracle with gcc (a mutant build plants mistake #mutant)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = so_path(mutant)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
           f"-DORC_MUTANT={int(mutant)}", "-o", out, _SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=not verbose)
    return out


class _Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("S", ctypes.c_int), ("clamp", ctypes.c_float),
                ("weight_in_combine", ctypes.c_int), ("w_fmt", ctypes.c_int)]


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous numpy arrays"
    return a.ctypes.data


class Oracle:
    """One loaded build of the oracle (the real one, or a mutant)."""

    def __init__(self, mutant: int = 0):
        path = so_path(mutant)
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            build(mutant)
        lib = ctypes.CDLL(path)
        p, i32, l = ctypes.c_void_p, ctypes.c_int, ctypes.c_long
        for name in ("orc_decode_e4m3", "orc_decode_e2m1", "orc_decode_ue8m0", "orc_encode_e4m3",
                     "orc_encode_bf16", "orc_requant_codes"):
            getattr(lib, name).argtypes = [p, p, l]
            getattr(lib, name).restype = None
        lib.orc_route.argtypes = [i32, i32, i32, i32, p, p, p, p, p]
        lib.orc_route.restype = i32
        lib.orc_forward.argtypes = [ctypes.POINTER(_Dims)] + [p] * 13 + [i32]
        lib.orc_forward.restype = i32
        lib.orc_l2_rows.argtypes = [i32, i32, i32, i32, p, p, p, p, p, p]
        lib.orc_l2_rows.restype = None
        self.lib = lib
        self.mutant = mutant

    # -- formats --------------------------------------------------------------
    def _map(self, fn, a, out_dtype):
        a = np.ascontiguousarray(a)
        out = np.empty(a.shape, out_dtype)
        fn(_p(a), _p(out), a.size)
        return out

    def decode_e4m3(self, b):
        return self._map(self.lib.orc_decode_e4m3, np.asarray(b, np.uint8), np.float32)

    def decode_e2m1(self, c):
        return self._map(self.lib.orc_decode_e2m1, np.asarray(c, np.uint8), np.float32)

    def decode_ue8m0(self, b):
        return self._map(self.lib.orc_decode_ue8m0, np.asarray(b, np.uint8), np.float32)

    def encode_e4m3(self, v):
        return self._map(self.lib.orc_encode_e4m3, np.asarray(v, np.float32), np.uint8)

    def encode_bf16(self, v):
        return self._map(self.lib.orc_encode_bf16, np.asarray(v, np.float32), np.uint16)

    def requant_codes(self, amax):
        return self._map(self.lib.orc_requant_codes, np.asarray(amax, np.float32), np.uint8)

    # -- routing --------------------------------------------------------------
    def route(self, topk_idx, E: int, S: int = 0):
        topk_idx = np.ascontiguousarray(topk_idx, np.int32)
        T, k = topk_idx.shape
        Ep, R = E + S, T * (k + S)
        counts = np.zeros(Ep, np.int32)
        offsets = np.zeros(Ep + 1, np.int32)
        perm = np.full(max(R, 1), -1, np.int32)
        pos = np.full(max(R, 1), -1, np.int32)
        bad = self.lib.orc_route(T, k, S, E, _p(topk_idx), _p(counts), _p(offsets), _p(perm), _p(pos))
        return dict(counts=counts, offsets=offsets, perm=perm[:R], pos=pos[:R], bad=bad)

    # -- whole path -----------------------------------------------------------
    def forward(self, dims: dict, x, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf, intermediates=False,
                nthreads: int | None = None, weight_in_combine: bool = False):
        """Run the path. dims: T,H,I,E,k,S,clamp. Returns dict(out=uint16 [T,H], ...)."""
        T, H, I, E, k, S = (int(dims[n]) for n in ("T", "H", "I", "E", "k", "S"))
        # 0: E2M1 weights (MXFP4), 1: E4M3 weights (MXFP8), both UE8M0 per 32;
        # 2: the float-scale FP8 recipe (float32 scales per 128 x 128 weight block and per (row, 128))
        w_fmt = int(dims.get("w_fmt", 0))
        d = _Dims(T, H, I, E, k, S, float(dims.get("clamp", 0.0)), int(weight_in_combine), w_fmt)
        wb = 1 if w_fmt else 2  # weight elements per byte is 2 for E2M1
        R = T * (k + S)
        c = np.ascontiguousarray
        sfd = np.float32 if w_fmt == 2 else np.uint8
        x, x_sf = c(x, np.uint8), c(x_sf, sfd)
        topk_idx, topk_w = c(topk_idx, np.int32), c(topk_w, np.float32)
        w1, w1_sf, w2, w2_sf = c(w1, np.uint8), c(w1_sf, sfd), c(w2, np.uint8), c(w2_sf, sfd)
        assert topk_idx.shape == (T, k) and topk_w.shape == (T, k)
        assert w1.size == (E + S) * 2 * I * H // wb and w2.size == (E + S) * H * I // wb
        if w_fmt == 2:
            assert x.shape == (T, H) and x_sf.shape == (T, H // 128)
            assert w1_sf.size == (E + S) * 2 * I * H // (128 * 128) and w2_sf.size == (E + S) * H * I // (128 * 128)
        else:
            assert x.shape == (T, H) and x_sf.shape == (T, H // 32)
            assert w1_sf.size == (E + S) * 2 * I * H // 32 and w2_sf.size == (E + S) * H * I // 32
        out = np.zeros((T, H), np.uint16)
        res = dict(out=out)
        acc1 = q = qsf = None
        if intermediates:
            acc1 = np.zeros((R, 2 * I), np.float32)
            q = np.zeros((R, I), np.uint8)
            qsf = np.zeros((R, I // 128), np.float32) if w_fmt == 2 else np.zeros((R, I // 32), np.uint8)
            res.update(acc1=acc1, q=q, q_sf=qsf)
        z = np.zeros((R, H), np.uint16)
        res["z"] = z
        n = nthreads or max(1, min(64, os.cpu_count() or 1))
        bad = self.lib.orc_forward(ctypes.byref(d), _p(x), _p(x_sf), _p(topk_idx), _p(topk_w), _p(w1), _p(w1_sf),
                                   _p(w2), _p(w2_sf), _p(out), _p(acc1), _p(q), _p(qsf), _p(z), n)
        if bad < 0:
            raise ValueError("oracle rejected the dimensions")
        res["bad"] = bad
        res.update(self.route(topk_idx, E, S))
        return res

    def l2_rows(self, expert_of_row, q, q_sf, w2, w2_sf, H: int, I: int, w_fmt: int = 0):
        expert_of_row = np.ascontiguousarray(expert_of_row, np.int32)
        R = expert_of_row.size
        acc2 = np.zeros((R, H), np.float32)
        sfd = np.float32 if w_fmt == 2 else np.uint8
        self.lib.orc_l2_rows(R, H, I, int(w_fmt), _p(expert_of_row), _p(np.ascontiguousarray(q, np.uint8)),
                             _p(np.ascontiguousarray(q_sf, sfd)), _p(np.ascontiguousarray(w2, np.uint8)),
                             _p(np.ascontiguousarray(w2_sf, sfd)), _p(acc2))
        return acc2


_default = None


def get() -> Oracle:
    """The (non-mutant) oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def sampled_problem(w, tokens, topk_idx, topk_w, x_rows, x_sf_rows, gen_weights):
    """Oracle outputs for a subset of tokens of a large workload.

    Every token's output depends only on its own slot rows, so running the path
    on just these tokens, with the experts they touch renumbered compactly,
    yields exactly the full problem's outputs for them. ``gen_weights(which,
    expert_ids)`` must return (codes, scales) of those experts in order.
    """
    tokens = np.asarray(tokens)
    sub_idx = np.ascontiguousarray(topk_idx[tokens])
    routed = sorted({int(e) for e in sub_idx.ravel() if 0 <= e < w.E})
    remap = {e: i for i, e in enumerate(routed)}
    # out-of-range ids stay out of range (-2), disabled slots stay disabled (-1)
    new_idx = np.array([[remap[int(e)] if 0 <= e < w.E else (-1 if e == -1 else -2) for e in row]
                        for row in sub_idx], np.int32).reshape(sub_idx.shape)
    experts = routed + list(range(w.E, w.E + w.S))
    w1, w1sf = gen_weights(2, experts)
    w2, w2sf = gen_weights(3, experts)
    dims = dict(T=len(tokens), H=w.H, I=w.I, E=len(routed), k=w.k, S=w.S, clamp=w.clamp,
                w_fmt=getattr(w, "w_fmt", 0))
    return get().forward(dims, x_rows, x_sf_rows, new_idx, np.ascontiguousarray(topk_w[tokens]), w1, w1sf, w2, w2sf)

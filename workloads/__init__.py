"""Seeded synthetic workloads for the MoE expert path.

The five workloads mirror the model shapes the MegaMoE pages benchmark
(DeepSeek-style hidden 7168 x intermediate 2048, 256 routed experts, top-8)
plus a tiny case and a mid-size case with the SwiGLU clamp enabled:

  tiny     T=32    H=512  I=256  E=8   k=2          (seed 0)
  decode   T=8     H=7168 I=2048 E=256 k=8          (seed 1)
  mid      T=1024  H=4096 I=1536 E=128 k=8 clamp 7  (seed 2)
  skewed   T=4096  H=7168 I=2048 E=256 k=8 + 1 shared expert, Zipf(1.2) routing (seed 3)
  prefill  T=16384 H=7168 I=2048 E=256 k=8          (seed 4)

Value recipe (identical bytes from the host and the device builds):
  x   : bf16(N(0,1)) quantised to FP8 E4M3 with one UE8M0 scale per 32 along H
  W1  : [E+S, 2I, H] (gate rows [0,I), up rows [I,2I)), N(0, 1/H) -> E2M1 + UE8M0 per 32 along H
  W2  : [E+S, H, I], N(0, 1/I) -> E2M1 + UE8M0 per 32 along I
  topk: uniform without replacement (or Zipf for "skewed"), weights = softmax of N(0,1) logits

The FP8-weight variants (w_fmt = 1: decode_fp8w, prefill_fp8w) draw the same
weight values and quantise them to E4M3 + UE8M0 per 32 (MXFP8, one byte per
element) instead of E2M1.

This module holds no step of the expert computation; it only produces inputs.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth.so")
_DEV_SO = os.path.join(_HERE, "libsynth_cuda.so")

TAG_W1 = 2
TAG_W2 = 3


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    S: int = 0
    clamp: float = 0.0
    zipf: float = 0.0
    seed: int = 0
    # weights: 0 = E2M1 (MXFP4, two per byte), 1 = E4M3 (MXFP8, one per byte), both with UE8M0 per 32;
    # 2 = the float-scale FP8 recipe (E4M3 weights with a float32 scale per 128 x 128 block,
    # activations with a float32 scale per (token, 128))
    w_fmt: int = 0

    @property
    def Ep(self) -> int:
        """Experts including the shared ones (stacked after the routed experts)."""
        return self.E + self.S

    @property
    def Kp(self) -> int:
        """Slots per token: k routed + S shared."""
        return self.k + self.S

    @property
    def rows(self) -> int:
        """Routed + shared rows when every slot is valid."""
        return self.T * self.Kp

    @property
    def std1(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.H)))

    @property
    def std2(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.I)))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops(self, n_rows: int | None = None) -> float:
        """Algorithmic FLOPs: 2*H*2I (L1) + 2*I*H (L2) per routed or shared row."""
        n = self.rows if n_rows is None else n_rows
        return 6.0 * self.H * self.I * n

    @property
    def w_elem_bytes(self) -> float:
        """Bytes per weight element: 1/2 (E2M1) or 1 (E4M3)."""
        return 1.0 if self.w_fmt else 0.5

    @property
    def w_sf_bytes(self) -> float:
        """Weight scale bytes per element: one UE8M0 byte per 32, or one float32 per 128 x 128."""
        return 4.0 / (128 * 128) if self.w_fmt == 2 else 1.0 / 32.0

    @property
    def a_sf_bytes(self) -> float:
        """Activation scale bytes per element: one UE8M0 byte per 32, or one float32 per 128."""
        return 4.0 / 128 if self.w_fmt == 2 else 1.0 / 32.0

    def expert_bytes(self) -> float:
        """Weight bytes one expert streams: W1 + W2 codes and scales."""
        return 3.0 * self.H * self.I * (self.w_elem_bytes + self.w_sf_bytes)


CONFIGS = {
    "tiny": Workload("tiny", T=32, H=512, I=256, E=8, k=2, seed=0),
    "decode": Workload("decode", T=8, H=7168, I=2048, E=256, k=8, seed=1),
    "mid": Workload("mid", T=1024, H=4096, I=1536, E=128, k=8, clamp=7.0, seed=2),
    "skewed": Workload("skewed", T=4096, H=7168, I=2048, E=256, k=8, S=1, zipf=1.2, seed=3),
    "prefill": Workload("prefill", T=16384, H=7168, I=2048, E=256, k=8, seed=4),
    # FP8 (MXFP8) weight variants of the decode and prefill shapes
    "decode_fp8w": Workload("decode_fp8w", T=8, H=7168, I=2048, E=256, k=8, seed=5, w_fmt=1),
    "prefill_fp8w": Workload("prefill_fp8w", T=16384, H=7168, I=2048, E=256, k=8, seed=6, w_fmt=1),
    # the float-scale FP8 recipe (1, 128, 128) at the decode and prefill shapes
    "decode_fp8f128": Workload("decode_fp8f128", T=8, H=7168, I=2048, E=256, k=8, seed=7, w_fmt=2),
    "prefill_fp8f128": Workload("prefill_fp8f128", T=16384, H=7168, I=2048, E=256, k=8, seed=8, w_fmt=2),
}


# ----------------------------------------------------------------------------- build / load
def build(cuda: bool = True, verbose: bool = False) -> None:
    """Compile the host generator (gcc) and, if asked, the device generator (nvcc, sm_103a)."""
    src = os.path.join(_HERE, "synth.c")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", _HOST_SO, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=not verbose)
    if cuda:
        cu = os.path.join(_HERE, "synth_cuda.cu")
        nvcc = os.environ.get("NVCC", "nvcc")
        cmd = [nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-fmad=false",
               "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_SO, cu]
        subprocess.run(cmd, check=True, capture_output=not verbose)


_host = None
_dev = None


def _lib_host():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build(cuda=False)
        lib = ctypes.CDLL(_HOST_SO)
        u64, i32, f32, p = ctypes.c_uint64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.syn_gen_x.argtypes = [u64, i32, i32, i32, p, p]
        lib.syn_gen_x.restype = None
        lib.syn_gen_w.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, i32]
        lib.syn_gen_w.restype = None
        lib.syn_gen_w8.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, i32]
        lib.syn_gen_w8.restype = None
        lib.syn_gen_x128.argtypes = [u64, i32, i32, i32, p, p]
        lib.syn_gen_x128.restype = None
        lib.syn_gen_w8f.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, i32]
        lib.syn_gen_w8f.restype = None
        lib.syn_gen_routing.argtypes = [u64, i32, i32, i32, ctypes.c_double, p, p]
        lib.syn_gen_routing.restype = i32
        lib.syn_u64_at.argtypes = [u64, u64]
        lib.syn_u64_at.restype = u64
        lib.syn_key.argtypes = [u64, u64]
        lib.syn_key.restype = u64
        lib.syn_normal_at.argtypes = [u64, u64]
        lib.syn_normal_at.restype = f32
        _host = lib
    return _host


def _lib_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            build(cuda=True)
        lib = ctypes.CDLL(_DEV_SO)
        u64, i32, f32, p = ctypes.c_uint64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.syn_dev_gen_x.argtypes = [u64, i32, i32, p, p, p]
        lib.syn_dev_gen_x.restype = i32
        lib.syn_dev_gen_w.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, p]
        lib.syn_dev_gen_w.restype = i32
        lib.syn_dev_gen_w8.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, p]
        lib.syn_dev_gen_w8.restype = i32
        lib.syn_dev_gen_x128.argtypes = [u64, i32, i32, p, p, p]
        lib.syn_dev_gen_x128.restype = i32
        lib.syn_dev_gen_w8f.argtypes = [u64, i32, i32, i32, i32, i32, f32, p, p, p]
        lib.syn_dev_gen_w8f.restype = i32
        _dev = lib
    return _dev


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _nthreads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ----------------------------------------------------------------------------- host generation
def routing(w: Workload, T: int | None = None):
    """(topk_idx int32 [T,k], topk_w float32 [T,k]) for the workload's routing recipe."""
    T = w.T if T is None else T
    idx = np.zeros((T, w.k), np.int32)
    wt = np.zeros((T, w.k), np.float32)
    rc = _lib_host().syn_gen_routing(w.seed, T, w.E, w.k, float(w.zipf), _ptr(idx), _ptr(wt))
    if rc != 0:
        raise ValueError(f"routing generator failed ({rc})")
    return idx, wt


def x_sf_shape(w: Workload, n: int):
    """Shape and dtype of the activation scales of n rows."""
    return ((n, w.H // 128), np.float32) if w.w_fmt == 2 else ((n, w.H // 32), np.uint8)


def x_host(w: Workload, t0: int = 0, t1: int | None = None):
    """Activation rows [t0, t1): (x_fp8 uint8 [n,H], x_sf uint8 [n,H/32], or float32
    [n,H/128] for the float-scale recipe)."""
    t1 = w.T if t1 is None else t1
    n = max(0, t1 - t0)
    x = np.zeros((n, w.H), np.uint8)
    shape, dt = x_sf_shape(w, n)
    sf = np.zeros(shape, dt)
    if n:
        gen = _lib_host().syn_gen_x128 if w.w_fmt == 2 else _lib_host().syn_gen_x
        gen(w.seed, w.H, t0, t1, _ptr(x), _ptr(sf))
    return x, sf


def weight_shape(w: Workload, which: int):
    """(rows per expert, K) of W1 (which=TAG_W1) or W2 (which=TAG_W2)."""
    return (2 * w.I, w.H) if which == TAG_W1 else (w.H, w.I)


def code_bytes(w: Workload, K: int) -> int:
    """Bytes of one weight row of K elements."""
    return K if w.w_fmt else K // 2


def w_sf_shape(w: Workload, which: int, n: int):
    """Shape and dtype of the weight scales of n experts."""
    rows, K = weight_shape(w, which)
    if w.w_fmt == 2:
        return (n, rows // 128, K // 128), np.float32
    return (n, rows, K // 32), np.uint8


def w_host(w: Workload, which: int, e0: int = 0, e1: int | None = None, nthreads: int | None = None):
    """Weights of experts [e0, e1): (codes uint8 [n,rows,K/2] (E2M1) or [n,rows,K] (E4M3),
    scales uint8 [n,rows,K/32], or float32 [n,rows/128,K/128] for the float-scale recipe)."""
    e1 = w.Ep if e1 is None else e1
    rows, K = weight_shape(w, which)
    n = max(0, e1 - e0)
    codes = np.zeros((n, rows, code_bytes(w, K)), np.uint8)
    shape, dt = w_sf_shape(w, which, n)
    sf = np.zeros(shape, dt)
    std = w.std1 if which == TAG_W1 else w.std2
    if n:
        lib = _lib_host()
        gen = lib.syn_gen_w8f if w.w_fmt == 2 else lib.syn_gen_w8 if w.w_fmt else lib.syn_gen_w
        gen(w.seed, which, rows, K, e0, e1, std, _ptr(codes), _ptr(sf), nthreads or _nthreads())
    return codes, sf


def host_inputs(w: Workload):
    """Every input of the workload generated on the host (small workloads only)."""
    idx, wt = routing(w)
    x, xsf = x_host(w)
    w1, w1sf = w_host(w, TAG_W1)
    w2, w2sf = w_host(w, TAG_W2)
    return dict(topk_idx=idx, topk_w=wt, x=x, x_sf=xsf, w1=w1, w1_sf=w1sf, w2=w2, w2_sf=w2sf)


# ----------------------------------------------------------------------------- device generation
def x_device(w: Workload, x, x_sf, stream=None):
    """Fill torch CUDA uint8 tensors x [T,H] and x_sf [T,H/32] on the device."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    gen = _lib_dev().syn_dev_gen_x128 if w.w_fmt == 2 else _lib_dev().syn_dev_gen_x
    rc = gen(w.seed, x.shape[0], w.H, x.data_ptr(), x_sf.data_ptr(), s.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"device x generator failed ({rc})")


def w_device(w: Workload, which: int, codes, sf, e0: int = 0, e1: int | None = None, stream=None):
    """Fill torch CUDA uint8 tensors with the weights of experts [e0, e1)."""
    import torch
    e1 = w.Ep if e1 is None else e1
    rows, K = weight_shape(w, which)
    std = w.std1 if which == TAG_W1 else w.std2
    s = stream if stream is not None else torch.cuda.current_stream()
    lib = _lib_dev()
    gen = lib.syn_dev_gen_w8f if w.w_fmt == 2 else lib.syn_dev_gen_w8 if w.w_fmt else lib.syn_dev_gen_w
    rc = gen(w.seed, which, rows, K, e0, e1, std, codes.data_ptr(), sf.data_ptr(), s.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"device weight generator failed ({rc})")


def device_inputs(w: Workload, device="cuda"):
    """Every input of the workload resident in device memory (weights generated in HBM)."""
    import torch
    idx, wt = routing(w)
    out = dict(topk_idx=torch.from_numpy(idx).to(device), topk_w=torch.from_numpy(wt).to(device))
    x = torch.empty((w.T, w.H), dtype=torch.uint8, device=device)
    shape, dt = x_sf_shape(w, w.T)
    xsf = torch.empty(shape, dtype=torch.float32 if dt == np.float32 else torch.uint8, device=device)
    if w.T:
        x_device(w, x, xsf)
    out.update(x=x, x_sf=xsf)
    for which, name in ((TAG_W1, "w1"), (TAG_W2, "w2")):
        rows, K = weight_shape(w, which)
        c = torch.empty((w.Ep, rows, code_bytes(w, K)), dtype=torch.uint8, device=device)
        shape, dt = w_sf_shape(w, which, w.Ep)
        s = torch.empty(shape, dtype=torch.float32 if dt == np.float32 else torch.uint8, device=device)
        w_device(w, which, c, s)
        out[name] = c
        out[name + "_sf"] = s
    return out

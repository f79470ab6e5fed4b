"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, read back its intermediates, and compare with the oracle."""
from __future__ import annotations

import numpy as np

import workloads

# Output tolerance for the BF16 result (per element and relative Frobenius).
ATOL_REL_MAX = 2e-2
ATOL_ABS = 1e-3
FROB_REL = 5e-3


def bf16_to_f64(u16) -> np.ndarray:
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_out_close(got_u16, ref_u16, what="output"):
    g, r = bf16_to_f64(got_u16), bf16_to_f64(ref_u16)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    mx = np.abs(r).max() if r.size else 0.0
    err = np.abs(g - r)
    bound = ATOL_REL_MAX * mx + ATOL_ABS
    assert (err <= bound).all(), f"{what}: max |diff| {err.max():.4g} > {bound:.4g} (max|ref| {mx:.4g})"
    nr = np.linalg.norm(r)
    if nr > 0:
        rel = np.linalg.norm(g - r) / nr
        assert rel <= FROB_REL, f"{what}: relative Frobenius error {rel:.3g} > {FROB_REL}"


def e4m3_to_f64(b) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def assert_l2a_close(q_gpu, sf_gpu, q_ref, sf_ref, what="L2 activations"):
    """E4M3 L2 activations: equal up to one E4M3 step where FP32 rounding
    order decides, on at most a small fraction of elements."""
    vg = e4m3_to_f64(q_gpu) * np.repeat(np.ldexp(1.0, sf_gpu.astype(np.int64) - 127), 32, axis=1)
    vr = e4m3_to_f64(q_ref) * np.repeat(np.ldexp(1.0, sf_ref.astype(np.int64) - 127), 32, axis=1)
    diff = vg != vr
    frac = diff.mean() if diff.size else 0.0
    assert frac <= 2e-3, f"{what}: {frac:.3%} of elements differ"
    step = np.maximum(np.abs(vr) * 2.0 ** -3, np.repeat(np.ldexp(1.0, sf_ref.astype(np.int64) - 127), 32, axis=1) * 2.0 ** -9)
    assert (np.abs(vg - vr) <= step * 1.0001).all(), f"{what}: an element differs by more than one E4M3 step"
    sdiff = (sf_gpu != sf_ref).mean() if sf_ref.size else 0.0
    assert sdiff <= 2e-3, f"{what}: {sdiff:.3%} of UE8M0 scales differ"


def assert_l2a_close_float(q_gpu, sf_gpu, q_ref, sf_ref, what="L2 activations (float scales)"):
    """Float-scale recipe: each per-(row, 128) scale is amax / 448 of the row's
    SwiGLU outputs, so a last-bit difference in the largest of them (FP32
    rounding order, exp) moves the scale by an ulp: scales agree to 1e-6
    relative. The E4M3 codes are the same bytes up to one E4M3 step where the
    rounding order decides, on a small fraction of elements."""
    sg = np.ascontiguousarray(sf_gpu).view(np.float32).astype(np.float64)
    sr = np.asarray(sf_ref, np.float32).astype(np.float64)
    assert sg.shape == sr.shape
    assert (np.abs(sg - sr) <= 1e-6 * sr).all(), f"{what}: scales differ by more than 1e-6 relative"
    frac = (np.asarray(q_gpu) != np.asarray(q_ref)).mean() if sr.size else 0.0
    assert frac <= 2e-3, f"{what}: {frac:.3%} of E4M3 codes differ"
    vg = e4m3_to_f64(q_gpu) * np.repeat(sg, 128, axis=1)
    vr = e4m3_to_f64(q_ref) * np.repeat(sr, 128, axis=1)
    step = np.maximum(np.abs(vr) * 2.0 ** -3, np.repeat(sr, 128, axis=1) * 2.0 ** -9)
    assert (np.abs(vg - vr) <= step * (1 + 1e-5)).all(), f"{what}: an element differs by more than one E4M3 step"


class DeviceRun:
    """Owns a handle, device inputs and a workspace for one workload."""

    def __init__(self, w: workloads.Workload, inputs: dict | None = None, fast_math=False, device_weights=False,
                 clamp=None, schedule="auto", tiles=-1):
        import torch
        import moe_expert_layer_scan_gb300 as mm
        self.w = w
        self.mm = mm
        self.moe = mm.MegaMoE(w.E, w.H, w.I, w.k, w.S, swiglu_clamp=w.clamp if clamp is None else clamp,
                              fast_math=fast_math, schedule=schedule, weight_format=w.w_fmt, tiles=tiles)
        if inputs is None:
            if device_weights:
                self.d = workloads.device_inputs(w)
            else:
                h = workloads.host_inputs(w)
                self.d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in h.items()}
        else:
            self.d = {k: (v if isinstance(v, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(v))).cuda()
                      for k, v in inputs.items()}

    def run(self, **override):
        import torch
        d = dict(self.d, **override)
        out = self.moe(d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"])
        torch.cuda.synchronize()
        return out

    def status(self, stream=None) -> int:
        return self.moe.status(stream)

    def intermediates(self, T: int, pool: bool = False):
        """Host copies of the routing tables and the pool-order intermediates
        (with pool=True also the gathered token rows and scale rows)."""
        import torch
        v = self.moe.views(T)
        w = self.w
        R = T * w.Kp

        ws = self.moe.ws
        torch.cuda.synchronize()

        def grab(ptr, n, dtype):
            nbytes = n * np.dtype(dtype).itemsize
            off = ptr - ws.data_ptr()
            assert 0 <= off and off + nbytes <= ws.numel()
            return ws[off:off + nbytes].cpu().numpy().view(dtype).copy()

        Ep = w.Ep
        offsets = grab(v.offsets, Ep + 1, np.int32)
        n = int(offsets[-1]) if offsets.size else 0
        return dict(
            counts=grab(v.counts, Ep, np.int32), offsets=offsets, perm=grab(v.perm, R, np.int32)[:n],
            pos=grab(v.pos, R, np.int32), row_w=grab(v.row_w, R, np.float32)[:n],
            l2a=grab(v.l2a, n * w.I, np.uint8).reshape(n, w.I), l2a_sf=grab(v.l2a_sf, n * (w.I // 32), np.uint8).reshape(n, w.I // 32),
            z=grab(v.z, n * w.H, np.uint16).reshape(n, w.H),
            status=int(grab(v.status, 1, np.uint32)[0]),
            **(dict(pool_x=grab(v.pool_x, n * w.H, np.uint8).reshape(n, w.H),
                    pool_sf=grab(v.pool_sf, n * (w.H // 32), np.uint8).reshape(n, w.H // 32)) if pool else {}),
        )

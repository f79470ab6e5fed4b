"""Python binding of the GB300 MegaMoE expert-path library (libmegamoe.so).

The functions below carry the C ABI's names (``include/megamoe.h``) and only
marshal arguments: every step of the path runs in the library's CUDA kernels.
There is no fallback: if the library is missing, importing the binding's
functions raises.

    import moe_expert_layer_scan_gb300 as mm
    moe = mm.MegaMoE(E=256, H=7168, I=2048, topk=8, num_shared=0)
    out = moe(x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf)   # torch CUDA tensors
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB

MM_OK = 0
MM_DEV_BAD_ROUTING = 0x1
MM_DEV_TIMEOUT = 0x2
STATUS_NAMES = {0: "MM_OK", 1: "MM_ERR_INVALID_ARG", 2: "MM_ERR_UNSUPPORTED", 3: "MM_ERR_WORKSPACE_TOO_SMALL",
                4: "MM_ERR_CUDA", 5: "MM_ERR_DEVICE_TIMEOUT", 6: "MM_ERR_BAD_ROUTING", 7: "MM_ERR_ALIGNMENT"}
EXPORTS = ["mm_status_string", "mm_create", "mm_set_options", "mm_set_schedule", "mm_set_tile_policy",
           "mm_token_tile_width",
           "mm_set_weight_format",
           "mm_set_ep_ranks",
           "mm_set_expert_stats", "mm_transformed_scale_bytes", "mm_transform_weight_scales", "mm_workspace_bytes",
           "mm_run",
           "mm_get_status", "mm_launches_per_run", "mm_debug_views", "mm_debug_timeout_probe", "mm_debug_div_check",
           "mm_profile_enable",
           "mm_profile_last", "mm_profile_name", "mm_run_noalloc", "mm_destroy"]


class MMError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class DebugViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("counts", "offsets", "perm", "pos", "row_w", "pool_x", "pool_sf", "l2a",
                                                "l2a_sf", "z", "status")] + [("rows_capacity", ctypes.c_int),
                                                                             ("rank_offsets", ctypes.c_void_p)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmegamoe.so not found at {LIB_PATH}: build it with "
                               "moe_expert_layer_scan_gb300.build() (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, u32p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)
        L.mm_status_string.argtypes = [i32]
        L.mm_status_string.restype = ctypes.c_char_p
        L.mm_create.argtypes = [ctypes.POINTER(p), i32, i32, i32, i32, i32]
        L.mm_set_options.argtypes = [p, ctypes.c_float, i32]
        L.mm_set_schedule.argtypes = [p, i32]
        L.mm_set_ep_ranks.argtypes = [p, i32]
        L.mm_set_weight_format.argtypes = [p, i32]
        L.mm_set_tile_policy.argtypes = [p, i32]
        L.mm_token_tile_width.argtypes = [p, i32, ctypes.POINTER(ctypes.c_int)]
        L.mm_set_expert_stats.argtypes = [p, p]
        L.mm_workspace_bytes.argtypes = [p, i32, ctypes.POINTER(ctypes.c_size_t)]
        L.mm_run.argtypes = [p, i32] + [p] * 10 + [ctypes.c_size_t, p]
        L.mm_get_status.argtypes = [p, p, p, u32p]
        L.mm_launches_per_run.argtypes = [p, i32, ctypes.POINTER(ctypes.c_int)]
        L.mm_debug_views.argtypes = [p, p, i32, ctypes.POINTER(DebugViews)]
        L.mm_debug_timeout_probe.argtypes = [p, ctypes.c_uint64, p]
        L.mm_debug_div_check.argtypes = [ctypes.c_uint64, ctypes.c_uint64, p, p]
        L.mm_profile_enable.argtypes = [p, i32]
        L.mm_profile_last.argtypes = [p, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(ctypes.c_int)]
        L.mm_profile_name.argtypes = [p, i32]
        L.mm_profile_name.restype = ctypes.c_char_p
        L.mm_run_noalloc.argtypes = [p, i32] + [p] * 9 + [p]
        L.mm_transformed_scale_bytes.argtypes = [p, ctypes.POINTER(ctypes.c_size_t)]
        L.mm_transform_weight_scales.argtypes = [p, p, p, p, ctypes.c_size_t, p]
        L.mm_destroy.argtypes = [p]
        L.mm_destroy.restype = None
        for n in EXPORTS:
            if n not in ("mm_status_string", "mm_profile_name", "mm_destroy"):
                getattr(L, n).restype = i32
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != MM_OK:
        raise MMError(rc, what)


# ----------------------------------------------------------------------------- C-ABI mirrors
def mm_create(E: int, H: int, I: int, topk: int, num_shared: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(lib().mm_create(ctypes.byref(h), E, H, I, topk, num_shared), "mm_create")
    return h.value


def mm_set_options(h: int, swiglu_clamp: float = 0.0, fast_math: bool = False) -> None:
    _check(lib().mm_set_options(h, float(swiglu_clamp), int(bool(fast_math))), "mm_set_options")


MM_SCHEDULE_AUTO, MM_SCHEDULE_SPLIT, MM_SCHEDULE_FUSED = -1, 0, 1
SCHEDULES = {"auto": MM_SCHEDULE_AUTO, "split": MM_SCHEDULE_SPLIT, "fused": MM_SCHEDULE_FUSED}


def mm_set_schedule(h: int, schedule="auto") -> None:
    """schedule: "auto" | "split" | "fused" (or the MM_SCHEDULE_* value)."""
    v = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    _check(lib().mm_set_schedule(h, v), "mm_set_schedule")


MM_TILES_AUTO, MM_TILES_16, MM_TILES_64, MM_TILES_112, MM_TILES_224 = -1, 16, 64, 112, 224
MM_TILES_PER_EXPERT = 0
MM_TILES_224_PAIRS = -2


def mm_token_tile_width(h: int, T: int) -> int:
    """Token-tile width a call of T tokens runs with under the handle's policy."""
    v = ctypes.c_int(0)
    _check(lib().mm_token_tile_width(h, int(T), ctypes.byref(v)), "mm_token_tile_width")
    return v.value


def mm_set_tile_policy(h: int, policy: int = MM_TILES_AUTO) -> None:
    """Token-tile width: MM_TILES_AUTO, MM_TILES_16, MM_TILES_64, MM_TILES_112, MM_TILES_224,
    MM_TILES_PER_EXPERT or MM_TILES_224_PAIRS."""
    _check(lib().mm_set_tile_policy(h, int(policy)), "mm_set_tile_policy")


MM_WEIGHTS_MXFP4, MM_WEIGHTS_MXFP8, MM_WEIGHTS_FP8_F128 = 0, 1, 2


def mm_set_weight_format(h: int, fmt: int) -> None:
    """MM_WEIGHTS_MXFP4 (E2M1, two per byte), MM_WEIGHTS_MXFP8 (E4M3, one per byte), both with UE8M0 per
    32, or MM_WEIGHTS_FP8_F128 (E4M3 with float32 scales per 128 x 128 block; activations with float32
    scales per (token, 128))."""
    _check(lib().mm_set_weight_format(h, int(fmt)), "mm_set_weight_format")


def mm_set_ep_ranks(h: int, num_ranks: int) -> None:
    _check(lib().mm_set_ep_ranks(h, int(num_ranks)), "mm_set_ep_ranks")


def mm_set_expert_stats(h: int, cumulative_counts_ptr) -> None:
    """Device pointer to E + S int32 counters (or None to disable)."""
    _check(lib().mm_set_expert_stats(h, cumulative_counts_ptr or None), "mm_set_expert_stats")


def mm_transformed_scale_bytes(h: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().mm_transformed_scale_bytes(h, ctypes.byref(n)), "mm_transformed_scale_bytes")
    return n.value


def mm_transform_weight_scales(h: int, w1_sf: int, w2_sf: int, dst: int, dst_bytes: int, stream: int) -> None:
    """Writes the transformed copy of both weight scale tensors into dst and
    registers it for runs with these w1_sf / w2_sf pointers (dst = 0 unregisters)."""
    _check(lib().mm_transform_weight_scales(h, w1_sf or None, w2_sf or None, dst or None, dst_bytes, stream or None),
           "mm_transform_weight_scales")


def mm_workspace_bytes(h: int, T: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().mm_workspace_bytes(h, T, ctypes.byref(n)), "mm_workspace_bytes")
    return n.value


def mm_run(h: int, T: int, x_fp8: int, x_sf: int, topk_idx: int, topk_w: int, w1: int, w1_sf: int, w2: int,
           w2_sf: int, out_bf16: int, ws: int, ws_bytes: int, stream: int) -> int:
    """Raw call with device pointers; returns the status code (not raised)."""
    return lib().mm_run(h, T, x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf, out_bf16, ws, ws_bytes, stream)


def mm_run_noalloc(h: int, T: int, x_fp8: int, x_sf: int, topk_idx: int, topk_w: int, w1: int, w1_sf: int, w2: int,
                   w2_sf: int, out_bf16: int, stream: int) -> int:
    """Raw call of the allocation-free variant (scratch inside the library);
    returns the status code (not raised)."""
    return lib().mm_run_noalloc(h, T, x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf, out_bf16, stream)


def mm_get_status(h: int, ws: int, stream: int) -> int:
    v = ctypes.c_uint32()
    _check(lib().mm_get_status(h, ws, stream, ctypes.byref(v)), "mm_get_status")
    return v.value


def mm_launches_per_run(h: int, T: int) -> int:
    n = ctypes.c_int()
    _check(lib().mm_launches_per_run(h, T, ctypes.byref(n)), "mm_launches_per_run")
    return n.value


def mm_debug_views(h: int, ws: int, T: int) -> DebugViews:
    v = DebugViews()
    _check(lib().mm_debug_views(h, ws, T, ctypes.byref(v)), "mm_debug_views")
    return v


def mm_debug_timeout_probe(ws: int, timeout_ns: int, stream: int) -> None:
    _check(lib().mm_debug_timeout_probe(ws, int(timeout_ns), stream), "mm_debug_timeout_probe")


def mm_debug_div_check(pairs: int, seed: int, counts: int, stream: int) -> None:
    """counts: device address of 5 uint64 (see include/megamoe.h)."""
    _check(lib().mm_debug_div_check(int(pairs), int(seed), counts, stream), "mm_debug_div_check")


def mm_profile_enable(h: int, on: bool = True) -> None:
    _check(lib().mm_profile_enable(h, int(bool(on))), "mm_profile_enable")


def mm_profile_last(h: int) -> list:
    """Per-launch milliseconds of the last profiled mm_run, in launch order."""
    buf = (ctypes.c_float * 8)()
    n = ctypes.c_int()
    _check(lib().mm_profile_last(h, buf, 8, ctypes.byref(n)), "mm_profile_last")
    return [float(buf[i]) for i in range(n.value)]


def mm_profile_name(h: int, i: int):
    """Stage name of the i-th interval of the last profiled mm_run (None past the end)."""
    r = lib().mm_profile_name(h, i)
    return None if r is None else r.decode()


def mm_profile_stages(h: int) -> dict:
    """{stage name: milliseconds} of the last profiled mm_run."""
    ms = mm_profile_last(h)
    return {mm_profile_name(h, i): v for i, v in enumerate(ms)}


def mm_destroy(h: int) -> None:
    if h:
        lib().mm_destroy(h)


def mm_status_string(code: int) -> str:
    return lib().mm_status_string(code).decode()


# ----------------------------------------------------------------------------- torch convenience
class MegaMoE:
    """One layer shape bound to a handle; owns a reusable device workspace."""

    def __init__(self, E: int, H: int, I: int, topk: int, num_shared: int = 0, swiglu_clamp: float = 0.0,
                 fast_math: bool = False, schedule="auto", weight_format: int = MM_WEIGHTS_MXFP4,
                 tiles: int = MM_TILES_AUTO):
        self.E, self.H, self.I, self.topk, self.S = E, H, I, topk, num_shared
        self.h = mm_create(E, H, I, topk, num_shared)
        mm_set_options(self.h, swiglu_clamp, fast_math)
        mm_set_schedule(self.h, schedule)
        mm_set_weight_format(self.h, weight_format)
        mm_set_tile_policy(self.h, tiles)
        self.ws = None

    def workspace(self, T: int, device=None):
        import torch
        need = mm_workspace_bytes(self.h, T)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=device or "cuda")
        return self.ws

    def launches(self, T: int) -> int:
        return mm_launches_per_run(self.h, T)

    def transform_weight_scales(self, w1_sf, w2_sf, stream=None):
        """Weight preparation: the tcgen05 scale layout of both weight scale
        tensors in a device buffer this object keeps; later runs with these
        two tensors read it. Call again after the scales change."""
        import torch
        n = mm_transformed_scale_bytes(self.h)
        self.tsf = torch.empty(n, dtype=torch.uint8, device=w1_sf.device)
        s = (stream or torch.cuda.current_stream(w1_sf.device)).cuda_stream
        mm_transform_weight_scales(self.h, w1_sf.data_ptr(), w2_sf.data_ptr(), self.tsf.data_ptr(), n, s)

    def run(self, x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf, out=None, stream=None):
        """Enqueue one forward on `stream` (default: torch's current stream)."""
        import torch
        T = x_fp8.shape[0]
        dev = x_fp8.device
        for t in (x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf):
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("all inputs must be contiguous CUDA tensors")
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=dev)
        ws = self.workspace(T, dev)
        s = (stream or torch.cuda.current_stream(dev)).cuda_stream
        rc = mm_run(self.h, T, x_fp8.data_ptr(), x_sf.data_ptr(), topk_idx.data_ptr(), topk_w.data_ptr(),
                    w1.data_ptr(), w1_sf.data_ptr(), w2.data_ptr(), w2_sf.data_ptr(), out.data_ptr(), ws.data_ptr(),
                    ws.numel(), s)
        _check(rc, "mm_run")
        return out

    __call__ = run

    def status(self, stream=None) -> int:
        import torch
        s = (stream or torch.cuda.current_stream()).cuda_stream
        return mm_get_status(self.h, self.ws.data_ptr(), s)

    def views(self, T: int) -> DebugViews:
        return mm_debug_views(self.h, self.ws.data_ptr(), T)

    def __del__(self):
        try:
            mm_destroy(self.h)
        except Exception:
            pass

"""Pins for the oracle: each check compares the oracle with something other
than itself — a library routine (PyTorch FP8/BF16 casts, NumPy float64
matmul, stable argsort), a published format table, an exact rational
computation, or an invariant the mathematics fixes.

Every pin returns a list of failure strings (empty: pass). The test files
assert that the real oracle passes all of them; ``test_oracle_mutants.py``
asserts that every planted mistake fails at least one.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
U32 = 2.0 ** -24  # unit roundoff of float32


def gamma(n: int) -> float:
    """Higham's gamma_n = n u / (1 - n u): bound on recursive-summation error."""
    return n * U32 / (1 - n * U32)


# ----------------------------------------------------------------------------- independent decoders
def e2m1_table() -> np.ndarray:
    vals = {}
    with open(os.path.join(HERE, "golden", "e2m1_values.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = float(v)
    return np.array([vals[i] for i in range(16)], np.float64)


def deq_e4m3(b) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def deq_ue8m0(b) -> np.ndarray:
    b = np.asarray(b).astype(np.int64)
    return np.ldexp(1.0, b - 127)


def unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


def deq_w(codes, sf, fmt: int = 0) -> np.ndarray:
    """Weights from their codes: E2M1 packed two per byte (fmt 0, OCP MXFP4) or
    E4M3 one per byte (fmt 1, OCP MXFP8), times the UE8M0 scale of each 32; or
    (fmt 2, the float-scale recipe) E4M3 times the float32 scale of each
    128 x 128 block (sf [..., rows/128, K/128])."""
    if fmt == 2:
        return deq_e4m3(codes) * np.repeat(np.repeat(np.asarray(sf, np.float64), 128, axis=-2), 128, axis=-1)
    vals = deq_e4m3(codes) if fmt else e2m1_table()[unpack_e2m1(codes)]
    return vals * np.repeat(deq_ue8m0(sf), 32, axis=-1)


def deq_x(x, sf) -> np.ndarray:
    """Activations: E4M3 times the UE8M0 scale of each 32, or (float32 scales,
    the float-scale recipe) times the float scale of each 128."""
    sf = np.asarray(sf)
    if sf.dtype == np.float32:
        return deq_e4m3(x) * np.repeat(sf.astype(np.float64), 128, axis=-1)
    return deq_e4m3(x) * np.repeat(deq_ue8m0(sf), 32, axis=-1)


def bf16_bits_to_f64(u16) -> np.ndarray:
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def slot_experts(topk_idx, E: int, S: int) -> np.ndarray:
    """Expert of every flat slot t*(k+S)+j (-1 when disabled or out of range)."""
    T, k = topk_idx.shape
    ex = np.concatenate([topk_idx.astype(np.int64), np.tile(np.arange(E, E + S), (T, 1))], axis=1)
    ex[(ex < 0) | ((ex >= E) & (np.arange(k + S)[None, :] < k))] = -1
    return ex.reshape(-1)


def slot_weights(topk_w, S: int) -> np.ndarray:
    T, k = topk_w.shape
    return np.concatenate([topk_w.astype(np.float64), np.ones((T, S))], axis=1).reshape(-1)


# ----------------------------------------------------------------------------- format pins
def pin_e4m3_decode(o):
    b = np.arange(256, dtype=np.uint8)
    got = o.decode_e4m3(b).astype(np.float64)
    ref = deq_e4m3(b)
    return [] if np.array_equal(got, ref, equal_nan=True) else ["E4M3 decode differs from torch.float8_e4m3fn"]


def pin_e2m1_decode(o):
    got = o.decode_e2m1(np.arange(16, dtype=np.uint8)).astype(np.float64)
    return [] if np.array_equal(got, e2m1_table()) else ["E2M1 decode differs from the OCP MX table"]


def pin_ue8m0_decode(o):
    b = np.arange(255, dtype=np.uint8)
    got = o.decode_ue8m0(b).astype(np.float64)
    ref = torch.from_numpy(b.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    bad = []
    if not np.array_equal(got, ref):
        bad.append("UE8M0 decode differs from torch.float8_e8m0fnu")
    if not np.isnan(o.decode_ue8m0(np.array([255], np.uint8))[0]):
        bad.append("UE8M0 0xFF must be NaN")
    return bad


def _bf16_cases(rng):
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    # exact ties: upper 16 bits arbitrary, lower 16 bits = 0x8000
    u = (rng.integers(0x00800000, 0x7F000000, 4000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    ties = u.view(np.float32)
    return np.concatenate([v, ties, -ties])


def pin_bf16_encode(o):
    rng = np.random.default_rng(11)
    v = _bf16_cases(rng)
    got = o.encode_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    return [] if np.array_equal(got, ref) else ["BF16 encode differs from torch's round-to-nearest-even"]


def pin_e4m3_encode(o):
    rng = np.random.default_rng(12)
    codes = np.arange(127, dtype=np.uint8)
    vals = deq_e4m3(codes)  # non-negative finite values, increasing
    mids = (vals[:-1] + vals[1:]) / 2  # exact in float32 (one extra bit)
    m32 = mids.astype(np.float32)
    cases = [vals.astype(np.float32), m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9)),
             (rng.uniform(-448, 448, 20000)).astype(np.float32),
             (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 8, 20000))).astype(np.float32)]
    v = np.concatenate(cases)
    v = np.concatenate([v, -v])
    v = v[np.abs(v) <= 448]
    got = o.encode_e4m3(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # signed zero: the oracle normalises -0 to +0; compare values for zeros
    same = (got == ref) | ((deq_e4m3(got) == 0) & (deq_e4m3(ref) == 0))
    bad = [] if same.all() else [f"E4M3 encode differs from torch on {int((~same).sum())} values"]
    # saturating cast (OCP FP8 saturation mode): beyond the largest finite value -> +-448
    sat = o.encode_e4m3(np.array([448.0, 449.0, 464.0, 1e6, -500.0], np.float32))
    if list(sat) != [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]:
        bad.append("E4M3 encode must saturate to +-448")
    return bad


def _smallest_pow2_exponent(r: Fraction) -> int:
    """Smallest integer p with 2**p >= r (r > 0), by exact rational search."""
    p = 0
    while Fraction(2) ** p < r:
        p += 1
    while Fraction(2) ** (p - 1) >= r:
        p -= 1
    return p


def pin_requant_code(o):
    rng = np.random.default_rng(13)
    amax = np.concatenate([
        np.exp2(rng.uniform(-40, 20, 3000)).astype(np.float32),
        (448.0 * np.exp2(np.arange(-30, 10))).astype(np.float32),  # r exactly a power of two
        np.nextafter((448.0 * np.exp2(np.arange(-30, 10))).astype(np.float32), np.float32(1e30)),
        np.nextafter((448.0 * np.exp2(np.arange(-30, 10))).astype(np.float32), np.float32(0)),
    ]).astype(np.float32)
    got = o.requant_codes(amax)
    bad = 0
    for a, c in zip(amax, got):
        r = Fraction(float(np.float32(a) / np.float32(448.0)))  # float32 quotient, as the pages' amax/448
        want = min(max(127 + _smallest_pow2_exponent(r), 1), 254)
        bad += int(c) != want
    out = [] if bad == 0 else [f"requant scale code wrong on {bad} inputs"]
    if o.requant_codes(np.array([0.0], np.float32))[0] != 127:
        out.append("amax == 0 must give scale code 127")
    return out


# ----------------------------------------------------------------------------- routing pin
def pin_route(o):
    rng = np.random.default_rng(14)
    fails = []
    for trial in range(40):
        T = int(rng.integers(0, 40))
        E = int(rng.integers(1, 20))
        k = int(rng.integers(1, 6))
        S = int(rng.integers(0, 3))
        idx = rng.integers(-1, E, (T, k)).astype(np.int32)
        if trial % 3 == 0 and T:
            idx[rng.integers(0, T), 0] = E + 5  # out of range -> disabled + counted
        r = o.route(idx, E, S)
        ex = slot_experts(idx, E, S)
        valid = ex >= 0
        nbad = int(((idx >= E) | (idx < -1)).sum())
        counts = np.bincount(ex[valid], minlength=E + S)
        order = np.argsort(np.where(valid, ex, E + S), kind="stable")[: int(valid.sum())]
        pos = np.full(ex.size, -1, np.int64)
        pos[order] = np.arange(order.size)
        ok = (np.array_equal(r["counts"], counts) and np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(counts)]))
              and np.array_equal(r["perm"][: order.size], order) and np.array_equal(r["pos"], pos) and r["bad"] == nbad)
        if not ok:
            fails.append(f"routing mismatch vs stable argsort (T={T} E={E} k={k} S={S})")
            break
    return fails


# ----------------------------------------------------------------------------- path pins
PIN_WORKLOADS = [
    workloads.CONFIGS["tiny"],
    workloads.Workload("pin_shared", T=12, H=256, I=128, E=5, k=3, S=1, clamp=0.75, zipf=1.2, seed=21),
    # FP8 (MXFP8) weights
    workloads.Workload("pin_fp8w", T=10, H=256, I=128, E=4, k=2, S=1, seed=22, w_fmt=1),
    # the float-scale FP8 recipe (float32 scales per 128 x 128 weight block and per (row, 128))
    workloads.Workload("pin_fp8f128", T=10, H=384, I=256, E=4, k=2, S=1, clamp=2.0, seed=23, w_fmt=2),
]


def summation_terms(w, K: int) -> int:
    """Roundings on one accumulator's path: K for an ascending FP32 sum; for
    the float-scale recipe 128 per block sum, one each for the scale product,
    the scaled partial and its addition, and one per block in the outer sum."""
    return 128 + 3 + K // 128 if w.w_fmt == 2 else K


def run_case(o, w, topk_idx=None, topk_w=None):
    d = workloads.host_inputs(w)
    if topk_idx is not None:
        d["topk_idx"], d["topk_w"] = topk_idx, topk_w
    dims = dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp, w_fmt=w.w_fmt)
    res = o.forward(dims, d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"],
                    intermediates=True, nthreads=4)
    return d, res


def _rows(w, d, res):
    """Per pool row: token, expert, weight — derived from the inputs, not the oracle."""
    ex = slot_experts(d["topk_idx"], w.E, w.S)
    wt = slot_weights(d["topk_w"], w.S)
    order = np.argsort(np.where(ex >= 0, ex, w.Ep), kind="stable")[: int((ex >= 0).sum())]
    return order // w.Kp, ex[order], wt[order]


def pin_l1(o, w, d, res):
    tok, ex, _ = _rows(w, d, res)
    x = deq_x(d["x"], d["x_sf"])
    fails = []
    for r in range(len(tok)):
        W1 = deq_w(d["w1"][ex[r]], d["w1_sf"][ex[r]], w.w_fmt)  # [2I, H]
        ref = W1 @ x[tok[r]]
        bound = gamma(summation_terms(w, w.H)) * (np.abs(W1) @ np.abs(x[tok[r]])) + 1e-30
        err = np.abs(res["acc1"][r].astype(np.float64) - ref)
        if (err > bound).any():
            fails.append(f"{w.name}: L1 accumulator outside the FP32 summation bound at row {r}")
            break
    return fails


def pin_l1_dyadic(o):
    """Operands in {0, +-1/2, +-1, +-2} with unit scales: every partial sum is a
    multiple of 1/4 far below 2^24, so FP32 accumulation is exact."""
    rng = np.random.default_rng(15)
    H, I, E, T, k = 64, 32, 2, 3, 1
    lut_e4m3 = {0.0: 0x00, 0.5: 0x30, 1.0: 0x38, 2.0: 0x40, -0.5: 0xB0, -1.0: 0xB8, -2.0: 0xC0}
    lut_e2m1 = {0.0: 0, 0.5: 1, 1.0: 2, 2.0: 4, -0.5: 9, -1.0: 10, -2.0: 12}
    choices = np.array([0.0, 0.5, 1.0, 2.0, -0.5, -1.0, -2.0])
    xv = rng.choice(choices, (T, H))
    x = np.vectorize(lut_e4m3.get)(xv).astype(np.uint8)
    wv = rng.choice(choices, (E, 2 * I, H))
    codes = np.vectorize(lut_e2m1.get)(wv).astype(np.uint8)
    w1 = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    ones = lambda *s: np.full(s, 127, np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    idx = np.array([[0], [1], [1]], np.int32)
    res = o.forward(dict(T=T, H=H, I=I, E=E, k=k, S=0), x, ones(T, H // 32), idx, np.ones((T, k), np.float32),
                    w1, ones(E, 2 * I, H // 32), w2, ones(E, H, I // 32), intermediates=True, nthreads=1)
    ref = np.stack([wv[idx[t, 0]] @ xv[t] for t in range(T)])  # rows are in token order here
    return [] if np.array_equal(res["acc1"].astype(np.float64), ref) else ["L1 not exact on dyadic operands"]


def _silu64(g):
    return torch.nn.functional.silu(torch.from_numpy(g)).numpy()


def pin_swiglu_requant(o, w, d, res):
    """Recompute y in float64 from the oracle's L1 accumulators with torch's
    SiLU, then check scale codes and E4M3 codes (at most one E4M3 step off,
    only where float32 vs float64 rounding can decide) and the MX invariants."""
    _, _, wt = _rows(w, d, res)
    a1 = res["acc1"].astype(np.float64)
    I = w.I
    g, u = a1[:, :I], a1[:, I:]
    if w.clamp > 0:
        g, u = np.clip(g, -w.clamp, w.clamp), np.clip(u, -w.clamp, w.clamp)
    y = _silu64(g) * u * wt[:, None]
    q, qsf = res["q"][: len(wt)], res["q_sf"][: len(wt)]
    if w.w_fmt == 2:
        return _pin_requant_float(w, y, q, qsf)
    s = np.repeat(deq_ue8m0(qsf), 32, axis=1)
    fails = []
    amax = np.abs(y).reshape(len(wt), I // 32, 32).max(axis=2)
    r = amax / 448.0
    sg = deq_ue8m0(qsf)
    nz = amax > 0
    # the scale is the smallest power of two >= amax/448 (checked with a float32-rounding slack)
    if ((sg[nz] < r[nz] * (1 - 1e-6)) | (sg[nz] >= 2 * r[nz] * (1 + 1e-6))).any():
        fails.append(f"{w.name}: requant scale is not the smallest power of two >= amax/448")
    ref_q = torch.from_numpy(np.clip(y / s, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got_v, ref_v = deq_e4m3(q), deq_e4m3(ref_q)
    diff = got_v != ref_v
    if diff.mean() > 2e-3:
        fails.append(f"{w.name}: {diff.mean():.2%} of E4M3 L2 activations differ from torch's cast")
    step = np.abs(got_v - ref_v) * s
    ulp = np.maximum(np.abs(y) * 2.0 ** -3, s * 2.0 ** -9)
    if (step > ulp * 1.0001).any():
        fails.append(f"{w.name}: an E4M3 L2 activation is more than one step off")
    if (np.abs(y / s) > 448 * (1 + 1e-6)).any():
        fails.append(f"{w.name}: an L2 activation saturates")
    return fails


def _pin_requant_float(w, y, q, qsf):
    """Float-scale recipe: the scale of each (row, 128) is amax / 448 (within
    float32 rounding of the float64 amax), and each E4M3 code is torch's cast
    of y / scale, at most one E4M3 step off where float32 vs float64 decides."""
    n, I = y.shape
    fails = []
    amax = np.abs(y).reshape(n, I // 128, 128).max(axis=2)
    sc = qsf.astype(np.float64)
    want = np.where(amax > 0, amax / 448.0, 1.0)
    if (np.abs(sc - want) > 2.0 ** -20 * want).any():
        fails.append(f"{w.name}: float L2-activation scale is not amax/448")
    s = np.repeat(sc, 128, axis=1)
    ref_q = torch.from_numpy(np.clip(y / s, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got_v, ref_v = deq_e4m3(q), deq_e4m3(ref_q)
    diff = got_v != ref_v
    if diff.mean() > 2e-3:
        fails.append(f"{w.name}: {diff.mean():.2%} of E4M3 L2 activations differ from torch's cast")
    ulp = np.maximum(np.abs(y / s) * 2.0 ** -3, 2.0 ** -9)
    if (np.abs(got_v - ref_v) > ulp * 1.0001).any():
        fails.append(f"{w.name}: an E4M3 L2 activation is more than one step off")
    if (np.abs(y / s) > 448 * (1 + 1e-5)).any():
        fails.append(f"{w.name}: an L2 activation saturates")
    return fails


def pin_l2(o, w, d, res):
    tok, ex, _ = _rows(w, d, res)
    n = len(tok)
    qv = deq_x(res["q"][:n], res["q_sf"][:n])
    z = bf16_bits_to_f64(res["z"][:n])
    fails = []
    for r in range(n):
        W2 = deq_w(d["w2"][ex[r]], d["w2_sf"][ex[r]], w.w_fmt)  # [H, I]
        ref = W2 @ qv[r]
        tot = np.abs(W2) @ np.abs(qv[r])
        bound = gamma(summation_terms(w, w.I)) * tot * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref) + 1e-30
        if (np.abs(z[r] - ref) > bound).any():
            fails.append(f"{w.name}: L2 BF16 row {r} outside FP32-sum + BF16-rounding bound")
            break
    return fails


def pin_l2_rows(o, w, d, res):
    """The L2-only oracle call on the path's own E4M3 activations: within
    Higham's FP32 summation bound of a float64 matmul of the independently
    dequantised operands, and its BF16 equal to the path's per-slot rows."""
    tok, ex, _ = _rows(w, d, res)
    n = len(tok)
    if n == 0:
        return []
    q, qsf = np.ascontiguousarray(res["q"][:n]), np.ascontiguousarray(res["q_sf"][:n])
    acc2 = o.l2_rows(ex.astype(np.int32), q, qsf, d["w2"], d["w2_sf"], w.H, w.I, w.w_fmt).astype(np.float64)
    qv = deq_x(q, qsf)
    fails = []
    for r in range(n):
        W2 = deq_w(d["w2"][ex[r]], d["w2_sf"][ex[r]], w.w_fmt)  # [H, I]
        ref = W2 @ qv[r]
        bound = gamma(summation_terms(w, w.I)) * (np.abs(W2) @ np.abs(qv[r])) + 1e-30
        if (np.abs(acc2[r] - ref) > bound).any():
            fails.append(f"{w.name}: L2-only accumulator outside the FP32 summation bound at row {r}")
            break
    z16 = torch.from_numpy(acc2.astype(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()
    if not np.array_equal(z16, res["z"][:n]):
        fails.append(f"{w.name}: BF16 of the L2-only accumulators differs from the path's per-slot rows")
    return fails


def pin_combine(o, w, d, res):
    ex = slot_experts(d["topk_idx"], w.E, w.S).reshape(w.T, w.Kp)
    pos = res["pos"].reshape(w.T, w.Kp)
    z = bf16_bits_to_f64(res["z"])
    out = bf16_bits_to_f64(res["out"])
    fails = []
    for t in range(w.T):
        rows = [pos[t, j] for j in range(w.Kp) if ex[t, j] >= 0]
        ref = z[rows].sum(axis=0) if rows else np.zeros(w.H)
        tot = np.abs(z[rows]).sum(axis=0) if rows else np.zeros(w.H)
        bound = gamma(max(len(rows), 1)) * tot * 1.01 + 2.0 ** -8 * np.abs(ref) + 1e-30
        if (np.abs(out[t] - ref) > bound).any():
            fails.append(f"{w.name}: combine of token {t} is not the BF16 of the slot-row sum")
            break
    return fails


def pin_topk_invariance(o):
    """k equal slots on one expert with weights 1/k (k a power of two) reproduce
    the single-slot output with weight 1, bit for bit: scaling by 2^-j commutes
    with the UE8M0/E4M3 requantisation and the BF16 rounding, and the k equal
    parts add exactly."""
    base = workloads.Workload("inv", T=6, H=256, I=128, E=3, k=1, seed=31)
    d = workloads.host_inputs(base)
    fails = []
    e = np.array([[1], [0], [2], [1], [0], [2]], np.int32)
    ref = o.forward(dict(T=6, H=256, I=128, E=3, k=1, S=0), d["x"], d["x_sf"], e, np.ones((6, 1), np.float32),
                    d["w1"], d["w1_sf"], d["w2"], d["w2_sf"], nthreads=2)["out"]
    for k in (2, 4):
        idx = np.repeat(e, k, axis=1)
        wt = np.full((6, k), 1.0 / k, np.float32)
        got = o.forward(dict(T=6, H=256, I=128, E=3, k=k, S=0), d["x"], d["x_sf"], idx, wt,
                        d["w1"], d["w1_sf"], d["w2"], d["w2_sf"], nthreads=2)["out"]
        if not np.array_equal(got, ref):
            fails.append(f"top-{k} split of one expert with weights 1/{k} is not bit-identical to top-1")
    return fails


def pin_permutation(o):
    """Tokens are independent: permuting (and duplicating) tokens permutes
    (and duplicates) output rows exactly."""
    w = workloads.Workload("perm", T=10, H=256, I=128, E=6, k=2, S=1, seed=32)
    d = workloads.host_inputs(w)
    dims = dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S)
    ref = o.forward(dims, d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"],
                    nthreads=2)["out"]
    p = np.array([3, 3, 9, 0, 1, 7, 2, 2, 5, 4, 6, 8])
    dims["T"] = len(p)
    got = o.forward(dims, d["x"][p], d["x_sf"][p], d["topk_idx"][p], d["topk_w"][p], d["w1"], d["w1_sf"], d["w2"],
                    d["w2_sf"], nthreads=2)["out"]
    return [] if np.array_equal(got, ref[p]) else ["permuting/duplicating tokens does not permute outputs exactly"]


def pin_f64_model(o, w, d, res):
    """Against a float64 model that never requantises (dequantised x, W1, W2,
    exact SwiGLU, weighted sum): the whole path stays within 5e-2 relative
    Frobenius error, which bounds the quantisation error of the method."""
    x = deq_x(d["x"], d["x_sf"])
    ex = slot_experts(d["topk_idx"], w.E, w.S).reshape(w.T, w.Kp)
    wt = slot_weights(d["topk_w"], w.S).reshape(w.T, w.Kp)
    ref = np.zeros((w.T, w.H))
    W1 = {e: deq_w(d["w1"][e], d["w1_sf"][e], w.w_fmt) for e in range(w.Ep)}
    W2 = {e: deq_w(d["w2"][e], d["w2_sf"][e], w.w_fmt) for e in range(w.Ep)}
    for t in range(w.T):
        for j in range(w.Kp):
            e = ex[t, j]
            if e < 0:
                continue
            a = W1[e] @ x[t]
            g, u = a[: w.I], a[w.I:]
            if w.clamp > 0:
                g, u = np.clip(g, -w.clamp, w.clamp), np.clip(u, -w.clamp, w.clamp)
            ref[t] += W2[e] @ (_silu64(g) * u * wt[t, j])
    got = bf16_bits_to_f64(res["out"])
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    return [] if rel <= 5e-2 else [f"{w.name}: relative Frobenius error vs float64 model {rel:.3g} > 5e-2"]


def all_pins(o):
    """Every pin on one oracle build: name -> list of failures."""
    out = {
        "e4m3_decode": pin_e4m3_decode(o), "e2m1_decode": pin_e2m1_decode(o), "ue8m0_decode": pin_ue8m0_decode(o),
        "bf16_encode": pin_bf16_encode(o), "e4m3_encode": pin_e4m3_encode(o), "requant_code": pin_requant_code(o),
        "route": pin_route(o), "l1_dyadic": pin_l1_dyadic(o), "topk_invariance": pin_topk_invariance(o),
        "permutation": pin_permutation(o),
    }
    for w in PIN_WORKLOADS:
        d, res = run_case(o, w)
        out[f"l1[{w.name}]"] = pin_l1(o, w, d, res)
        out[f"swiglu_requant[{w.name}]"] = pin_swiglu_requant(o, w, d, res)
        out[f"l2[{w.name}]"] = pin_l2(o, w, d, res)
        out[f"l2_rows[{w.name}]"] = pin_l2_rows(o, w, d, res)
        out[f"combine[{w.name}]"] = pin_combine(o, w, d, res)
        out[f"f64_model[{w.name}]"] = pin_f64_model(o, w, d, res)
    return out

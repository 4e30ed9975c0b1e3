"""Pins for the CPU oracle: each check compares it with something other than itself.

* bf16 rounding     -- against torch's float32 -> bfloat16 cast (a library
                       routine), on ties, subnormals, infinities and NaN.
* dispatch          -- a worked example derived by hand from the definition
                       (stable scatter by flat slot index; TileOps PR #1738,
                       Summary "local dispatch" and Scope "tight/no-pad"),
                       plus a brute-force restatement and its invariants
                       (``expert_offsets[-1] == R``, bijection, stability).
* expert MLP        -- the one-expert, k=1, weight-1 special case is a dense
                       gated MLP, computed with torch fp64 matmuls and
                       ``torch.nn.functional.silu``.
* dispatch+combine  -- with an identity expert, dispatch then combine equals
                       ``(sum_j w[t,j]) * x[t]`` (closed form).
* whole forward     -- a naive fp64 restatement in pure Python loops on tiny
                       shapes, several experts, dropped slots included.
* MXFP8 (E4M3 codes, E8M0 scale per 32, OCP MX v1.0; FlashInfer moe_ep page
  PR #3980, MXFP8 path) --
                       the E4M3 values the OCP FP8 spec prints (largest and
                       smallest normal and subnormal, NaN, zeros) and the
                       powers of two; element rounding against a brute-force
                       nearest-code search (ties to the even mantissa,
                       saturation at 448); the scale rule as the bound
                       256 <= max|V| / X < 512; grid values round-tripping
                       exactly; a block of zeros; the block format the
                       FlashInfer page prints (32 elements, E8M0 scale), read
                       from ``tests/golden/mx_block_format.txt``.

``test_planted_mistakes`` then builds mutated copies of ``moe_oracle.c``
(a dropped term, a swapped operand, a wrong sign, a wrong index ...) and
checks that at least one pin fails for each, so that the pins are known to
bite.
"""
from __future__ import annotations

import math
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.nn.functional as F

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402
from oracle import Oracle, bf16_bits_to_f32

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_SRC = os.path.join(os.path.dirname(HERE), "oracle", "moe_oracle.c")


# ----------------------------------------------------------------------------- helpers

def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(shape, generator=g) * std).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def near_bf16_midpoint(v64: np.ndarray, rel: float = 1e-4, tol_abs=0.0) -> np.ndarray:
    """True where a float64 value lies within ``rel`` (relative) or ``tol_abs``
    (absolute) of a bf16 rounding midpoint."""
    v = np.asarray(v64, dtype=np.float64)
    lo = bf16_bits_to_f32(torch_bf16_bits(v.astype(np.float32))).astype(np.float64)
    # neighbour on the other side of v
    bits = torch_bf16_bits(v.astype(np.float32)).astype(np.int32)
    step = np.where((lo <= v) == (v >= 0), 1, -1)
    other = bf16_bits_to_f32((bits + step).astype(np.uint16)).astype(np.float64)
    mid = 0.5 * (lo + other)
    return np.abs(v - mid) <= np.maximum(rel * np.abs(v), tol_abs)


def silu64(g):
    return g / (1.0 + np.exp(-g))


# ----------------------------------------------------------------------------- pins

def pin_round_bf16(o: Oracle):
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000)]
    # exact ties: low 16 bits == 0x8000, both parities of the kept part
    base = rng.integers(0, 2 ** 31, 4000, dtype=np.int64).astype(np.uint32)
    ties = ((base & 0xFFFF0000) | 0x8000).view(np.float32)
    vals.append(ties[np.isfinite(ties)])
    vals.append(np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 1e-40, -1e-40, 3.3895e38, 65504.0,
                          np.float32(1.0) + np.float32(2 ** -8), np.float32(1.0) + np.float32(3 * 2 ** -9)],
                         dtype=np.float32))
    x = np.concatenate(vals).astype(np.float32)
    got = o.round_bf16(x)
    want = torch_bf16_bits(x)
    assert np.array_equal(got, want), f"bf16 rounding differs at {np.count_nonzero(got != want)} values"
    nan = o.round_bf16(np.array([np.nan], dtype=np.float32))
    assert np.isnan(bf16_bits_to_f32(nan))[0]


def pin_dispatch_hand(o: Oracle):
    # ids[T=3, k=2] with E=3. Slots s = t*k + j: s0:e2 s1:e0 s2:e0 s3:e1 s4:e2 s5:e1.
    # counts = [2, 2, 2] -> offsets = [0, 2, 4, 6].
    # Walking s ascending: e0 gets s1, s2 (rows 0, 1); e1 gets s3, s5 (rows 2, 3);
    # e2 gets s0, s4 (rows 4, 5). perm[row] = slot, inv[slot] = row.
    ids = np.array([[2, 0], [0, 1], [2, 1]], dtype=np.int32)
    counts, offsets, perm, inv, bad = o.dispatch(ids, 3)
    assert counts.tolist() == [2, 2, 2]
    assert offsets.tolist() == [0, 2, 4, 6]
    assert perm.tolist() == [1, 2, 3, 5, 0, 4]
    assert inv.tolist() == [4, 0, 1, 2, 5, 3]
    assert bad == 0
    # a dropped slot (-1) and an invalid id (7): neither gets a row.
    ids2 = np.array([[1, -1], [7, 1], [0, 1]], dtype=np.int32)
    counts, offsets, perm, inv, bad = o.dispatch(ids2, 3)
    # valid slots: s0:e1 s3:e1 s4:e0 s5:e1 -> e0: s4 (row 0); e1: s0, s3, s5 (rows 1..3)
    assert offsets.tolist() == [0, 1, 4, 4]
    assert perm.tolist() == [4, 0, 3, 5, -1, -1]
    assert inv.tolist() == [1, -1, -1, 2, 0, 3]
    assert bad == 1


def brute_dispatch(ids_flat: np.ndarray, E: int):
    """O(R * E) restatement: expert e's rows are its slots in ascending order."""
    ids_flat = [int(v) for v in ids_flat]
    offsets = [0]
    perm = []
    for e in range(E):
        mine = [s for s, v in enumerate(ids_flat) if v == e]
        perm.extend(mine)
        offsets.append(offsets[-1] + len(mine))
    inv = [-1] * len(ids_flat)
    for r, s in enumerate(perm):
        inv[s] = r
    return offsets, perm, inv


def pin_dispatch_brute(o: Oracle):
    rng = np.random.default_rng(1)
    for (T, k, E) in [(37, 3, 5), (1, 6, 384), (0, 2, 4), (50, 1, 1), (64, 8, 16)]:
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
        if T > 2:
            ids[1, 0] = -1
        counts, offsets, perm, inv, bad = o.dispatch(ids, E)
        b_off, b_perm, b_inv = brute_dispatch(ids.reshape(-1), E)
        assert offsets.tolist() == b_off, (T, k, E)
        R = T * k
        n_valid = b_off[-1]
        assert perm[:n_valid].tolist() == b_perm
        assert np.all(perm[n_valid:] == -1)
        assert inv.tolist() == b_inv
        # invariants
        assert offsets[-1] == int(np.count_nonzero(ids >= 0))
        assert np.all(np.diff(offsets) >= 0)
        flat = ids.reshape(-1)
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)          # stable
        assert sorted(perm[:n_valid].tolist()) == sorted(np.nonzero(flat >= 0)[0].tolist())
        for r in range(n_valid):
            assert inv[perm[r]] == r
        assert R == flat.size


def pin_dense_mlp(o: Oracle):
    """One expert, k = 1, weight 1: the oracle must be a dense gated MLP."""
    T, H, I = 16, 64, 96
    x = rand_bf16((T, H), 1.0, 2)
    W13 = rand_bf16((1, 2 * I, H), 0.1, 3)
    W2 = rand_bf16((1, H, I), 0.1, 4)
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)

    xf = torch.from_numpy(bf16_bits_to_f32(x).astype(np.float64))
    W1 = torch.from_numpy(bf16_bits_to_f32(W13[0, :I]).astype(np.float64))
    W3 = torch.from_numpy(bf16_bits_to_f32(W13[0, I:]).astype(np.float64))
    W2d = torch.from_numpy(bf16_bits_to_f32(W2[0]).astype(np.float64))
    g64, u64 = xf @ W1.T, xf @ W3.T
    act64 = (F.silu(g64) * u64).numpy()
    # forward-error bound of the fp32 sums (H terms each) propagated through SiLU(g) * u
    eps = 2.0 ** -24
    dg = H * eps * (xf.abs() @ W1.abs().T).numpy()
    du = H * eps * (xf.abs() @ W3.abs().T).numpy()
    dact = 1.1 * dg * np.abs(u64.numpy()) + np.abs(F.silu(g64).numpy()) * du + 4 * eps * np.abs(act64)

    a, y = o.expert_rows(x, W13[0], W2[0])
    a_ref = torch_bf16_bits(act64.astype(np.float32))
    diff = a != a_ref
    assert np.count_nonzero(diff) <= max(2, diff.size // 100), "activation differs from dense MLP"
    assert np.all(near_bf16_midpoint(act64[diff], tol_abs=dact[diff])), \
        "activation differs away from a rounding midpoint"
    assert np.all(np.abs(a.astype(np.int32) - a_ref.astype(np.int32))[diff] == 1), "more than one ulp apart"

    y_ref = (torch.from_numpy(bf16_bits_to_f32(a).astype(np.float64)) @ W2d.T).numpy()
    scale = np.sqrt(np.mean(y_ref ** 2))
    assert np.max(np.abs(y - y_ref)) <= 1e-5 * scale + 1e-7, "down projection differs from a @ W2^T"

    out_acc, out, bad = o.moe_tokens(x, ids, w, W13, W2)
    assert bad == 0
    assert np.max(np.abs(out_acc - y_ref)) <= 1e-5 * scale + 1e-7
    assert np.array_equal(out, torch_bf16_bits(out_acc))


def pin_identity_expert(o: Oracle):
    """dispatch -> identity expert (y_sorted = x_sorted) -> combine == (sum_j w) * x."""
    rng = np.random.default_rng(5)
    T, k, E, H = 50, 3, 7, 32
    x = rand_bf16((T, H), 1.0, 6)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[3, 1] = -1
    ids[10, 0] = -1
    w = rng.uniform(0.05, 1.5, (T, k)).astype(np.float32)
    counts, offsets, perm, inv, bad = o.dispatch(ids, E)
    n_rows = int(offsets[-1])
    x_sorted = bf16_bits_to_f32(x[perm[:n_rows] // k])    # gather: row -> token of its slot
    out_acc, out = o.combine_sorted(x_sorted, inv, w)
    wsum = np.where(ids >= 0, w.astype(np.float64), 0.0).sum(axis=1)
    ref = wsum[:, None] * bf16_bits_to_f32(x).astype(np.float64)
    assert np.max(np.abs(out_acc - ref)) <= 1e-6 * np.max(np.abs(ref))
    # softmax-normalised weights: out reproduces x to within one bf16 ulp
    wn = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    ids_full = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, perm, inv, _ = o.dispatch(ids_full, E)
    _, out = o.combine_sorted(bf16_bits_to_f32(x[perm // k]), inv, wn)
    xf = bf16_bits_to_f32(x)
    of = bf16_bits_to_f32(out)
    assert np.all(np.abs(of - xf) <= np.abs(xf) * 2.0 ** -7 + 1e-30)


def naive_forward64(x, ids, w, W13, W2, a_bits_hint=None):
    """Pure-Python fp64 restatement: loops over tokens, slots, outputs, inputs."""
    T, H = x.shape
    E, twoI, _ = W13.shape
    I = twoI // 2
    k = ids.shape[1]
    xf = bf16_bits_to_f32(x).astype(np.float64)
    W13f = bf16_bits_to_f32(W13).astype(np.float64)
    W2f = bf16_bits_to_f32(W2).astype(np.float64)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e < 0 or e >= E:
                continue
            a = [0.0] * I
            for n in range(I):
                g = 0.0
                u = 0.0
                for h in range(H):
                    g += xf[t, h] * W13f[e, n, h]
                    u += xf[t, h] * W13f[e, I + n, h]
                act = g / (1.0 + math.exp(-g)) * u
                ab = torch_bf16_bits(np.array([act], dtype=np.float32))[0]
                if a_bits_hint is not None:
                    hint = a_bits_hint.get((t, j, n))
                    if hint is not None and ab != hint and abs(int(ab) - int(hint)) == 1:
                        ab = hint
                a[n] = float(bf16_bits_to_f32(np.array([ab], dtype=np.uint16))[0])
            for m in range(H):
                y = 0.0
                for n in range(I):
                    y += a[n] * W2f[e, m, n]
                out[t, m] += float(w[t, j]) * y
    return out


def pin_naive_fp64(o: Oracle):
    T, E, k, H, I = 5, 3, 2, 8, 12
    rng = np.random.default_rng(7)
    x = rand_bf16((T, H), 1.0, 8)
    W13 = rand_bf16((E, 2 * I, H), 0.3, 9)
    W2 = rand_bf16((E, H, I), 0.3, 10)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[2, 1] = -1
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    hint = {}
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e >= 0:
                a, _ = o.expert_rows(x[t:t + 1], W13[e], W2[e])
                for n in range(I):
                    hint[(t, j, n)] = a[0, n]
    ref = naive_forward64(x, ids, w, W13, W2, hint)
    out_acc, out, bad = o.moe_tokens(x, ids, w, W13, W2)
    assert bad == 0
    assert np.max(np.abs(out_acc - ref)) <= 1e-5 * np.max(np.abs(ref)) + 1e-7


def pin_streamed_equals_tokens(o: Oracle):
    T, E, k, H, I = 9, 4, 3, 16, 24
    rng = np.random.default_rng(11)
    x = rand_bf16((T, H), 1.0, 12)
    W13 = rand_bf16((E, 2 * I, H), 0.2, 13)
    W2 = rand_bf16((E, H, I), 0.2, 14)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    acc_a, out_a, _ = o.moe_tokens(x, ids, w, W13, W2)
    acc_b, out_b = o.moe_forward_streamed(x, ids, w, lambda e: (W13[e], W2[e]), E)
    assert np.array_equal(acc_a.view(np.uint32), acc_b.view(np.uint32))
    sub = np.array([1, 4, 7], dtype=np.int32)
    acc_c, _, _ = o.moe_tokens(x, ids, w, W13, W2, tokens=sub)
    assert np.array_equal(acc_c.view(np.uint32), acc_a[sub].view(np.uint32))


def pin_e4m3_values(o: Oracle):
    """The E4M3 values the OCP 8-bit floating point spec prints for the format:
    max normal S.1111.110 = 448, min normal S.0001.000 = 2^-6, max subnormal
    S.0000.111 = 0.875 * 2^-6, min subnormal S.0000.001 = 2^-9, NaN
    S.1111.111, zeros S.0000.000; exponent bias 7, so 2^p is code (p+7) << 3."""
    v = o.e4m3_values().astype(np.float64)
    assert v[0x00] == 0.0 and not math.copysign(1.0, v[0x00]) < 0
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) < 0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x07] == 0.875 * 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert math.isnan(v[0x7F]) and math.isnan(v[0xFF])
    for p in range(-6, 9):
        assert v[(p + 7) << 3] == 2.0 ** p, p
    assert v[0x3C] == 1.5 and v[0x30] == 0.5 and v[0x44] == 3.0
    pos = v[1:0x7F]
    assert np.all(np.diff(pos) > 0)                       # codes increase with magnitude
    assert np.array_equal(v[0x81:0xFF], -pos)              # sign bit mirrors
    # within a binade the 8 codes are evenly spaced by 2^(p-3)
    for p in range(-6, 8):
        b = v[(p + 7) << 3: ((p + 8) << 3) + 1]
        assert np.allclose(np.diff(b), 2.0 ** (p - 3), rtol=0, atol=0), p


def _mx_block_with_unit_scale(vals):
    """bf16 bits of blocks of 32 whose largest magnitude is 256 (element 0), so
    the MX scale is 2^0 and each element is encoded as E4M3(value) itself."""
    vals = np.asarray(vals, dtype=np.float32).reshape(-1, 31)
    blocks = np.concatenate([np.full((vals.shape[0], 1), 256.0, np.float32), vals], axis=1)
    return torch_bf16_bits(blocks)


def pin_e4m3_rounding_brute(o: Oracle):
    """Element rounding = the nearest finite E4M3 value, found by searching all
    codes; a tie goes to the code with the even mantissa; |v| > 448 -> 448."""
    table = o.e4m3_values().astype(np.float64)
    finite = [c for c in range(256) if not math.isnan(table[c])]
    rng = np.random.default_rng(11)
    parts = [rng.uniform(-255, 255, 31 * 40), rng.uniform(-2, 2, 31 * 40),
             rng.uniform(-2 ** -5, 2 ** -5, 31 * 40),            # subnormal region
             np.sign(rng.uniform(-1, 1, 31 * 4)) * 2.0 ** rng.integers(-12, 8, 31 * 4)]
    # exact midpoints between neighbouring codes (ties), representable in bf16
    m = (table[1:0x7E] + table[2:0x7F]) / 2
    m = m[m < 255]
    m = m[bf16_bits_to_f32(torch_bf16_bits(m.astype(np.float32))).astype(np.float64) == m]
    mids = np.concatenate([m, -m])
    assert mids.size > 100
    mids = mids[: 31 * (mids.size // 31)]
    vals = np.concatenate(parts + [mids])
    vals = vals[: 31 * (vals.size // 31)]
    bits = _mx_block_with_unit_scale(vals)
    q, sc = o.mx_quantize(bits)
    assert np.all(sc == 127)
    vb = bf16_bits_to_f32(bits).astype(np.float64)
    for v, c in zip(vb.reshape(-1), q.reshape(-1)):
        d = np.array([abs(v - table[f]) for f in finite])
        best = np.flatnonzero(d == d.min())
        cand = [finite[i] for i in best]
        if v == 0.0:
            want = 0x80 if math.copysign(1.0, v) < 0 else 0x00
        elif len(cand) == 1:
            want = cand[0]
        else:
            even = [x for x in cand if (x & 1) == 0 and (x & 0x80) == (0x80 if v < 0 else 0)]
            want = even[0]
        assert c == want, (v, c, want)
    # saturation: magnitudes in (448, 512) with the block scale still 2^0
    sat = torch_bf16_bits(np.array([[500.0, -460.0, 449.0, 300.0] + [1.0] * 28], np.float32))
    q, sc = o.mx_quantize(sat)
    assert sc[0, 0] == 127 and q[0, 0] == 0x7E and q[0, 1] == 0xFE and q[0, 2] == 0x7E


def pin_mx_scale_rule(o: Oracle):
    """Per block: X = 2^(s - 127) with 256 <= max|V| / X < 512 (the scale puts
    the block maximum in E4M3's top binade); a block of zeros gets s = 0 and
    zero codes."""
    rng = np.random.default_rng(12)
    w = rng.standard_normal((64, 256)).astype(np.float32) * (2.0 ** rng.integers(-20, 20, (64, 1)))
    w[3, 32:64] = 0.0
    bits = torch_bf16_bits(w)
    q, sc = o.mx_quantize(bits)
    wb = bf16_bits_to_f32(bits).astype(np.float64).reshape(64, 8, 32)
    amax = np.abs(wb).max(axis=2)
    X = np.ldexp(1.0, sc.astype(np.int64) - 127)
    nz = amax > 0
    assert np.all(amax[nz] / X[nz] >= 256) and np.all(amax[nz] / X[nz] < 512)
    assert sc[3, 1] == 0 and np.all(q[3, 32:64] & 0x7F == 0)


def pin_mx_round_trip(o: Oracle):
    """Weights already on the MX grid (codes times a power of two, block
    maximum in the top binade) come back with the same codes and scale, and
    dequantize to exactly themselves."""
    rng = np.random.default_rng(13)
    rows, nb = 16, 4
    codes = rng.integers(0, 0x7F, (rows, nb * 32)).astype(np.uint8) | (rng.integers(0, 2, (rows, nb * 32)) << 7).astype(np.uint8)
    codes[:, ::32] = (0x78 + rng.integers(0, 7, (rows, nb))).astype(np.uint8)    # 256..448: top binade
    e = rng.integers(-30, 10, (rows, nb))
    table = o.e4m3_values().astype(np.float64)
    vals = table[codes] * np.repeat(np.ldexp(1.0, e), 32, axis=1)
    bits = torch_bf16_bits(vals.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(bits).astype(np.float64), vals)      # exact in bf16
    q, sc = o.mx_quantize(bits)
    assert np.array_equal(sc.astype(np.int64) - 127, e)
    same = (q == codes) | ((q & 0x7F) == 0) & ((codes & 0x7F) == 0)
    assert np.all(same)
    assert np.array_equal(o.mx_dequantize(q, sc), bits)


def read_golden(name: str) -> dict:
    """``key = value`` lines of a fixture under ``tests/golden/`` ('#' starts a comment)."""
    out = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, value = (part.strip() for part in line.split("=", 1))
                out[key] = value
    return out


def pin_mx_block_format(o: Oracle):
    """The block format the FlashInfer page prints for MXFP8 (32 E4M3 elements
    sharing one E8M0 scale; ``tests/golden/mx_block_format.txt``): every one
    of a block's elements, and none outside it, sets that block's scale, and
    each element decodes as E4M3 value times 2^(s - bias)."""
    fmt = read_golden("mx_block_format.txt")
    B, bias = int(fmt["block_elements"]), int(fmt["scale_bias"])
    assert (fmt["element"], fmt["scale"]) == ("e4m3", "e8m0")
    nb = 4
    base = np.full((1, nb * B), 1.0, np.float32)            # every block: max 1 -> s = bias - 8
    q0, s0 = o.mx_quantize(torch_bf16_bits(base))
    assert s0.shape == (1, nb) and np.all(s0.astype(int) == bias - 8)
    for b in range(nb):
        for i in range(B):
            w = base.copy()
            w[0, b * B + i] = 64.0                          # lifts only block b's maximum, by 2^6
            _, s = o.mx_quantize(torch_bf16_bits(w))
            want = s0.astype(int).copy()
            want[0, b] += 6
            assert np.array_equal(s.astype(int), want), (b, i)
    # decode: the E4M3 value of each code times 2^(s - bias), on random blocks
    rng = np.random.default_rng(14)
    w = rng.standard_normal((8, nb * B)).astype(np.float32) * np.ldexp(1.0, rng.integers(-12, 12, (8, 1)))
    q, s = o.mx_quantize(torch_bf16_bits(w))
    table = o.e4m3_values().astype(np.float64)
    scale = np.repeat(np.ldexp(1.0, s.astype(np.int64) - bias), B, axis=1)
    wb = bf16_bits_to_f32(torch_bf16_bits(w)).astype(np.float64)
    # E4M3 keeps 3 mantissa bits: a normal element is within 2^-4 relative,
    # one below the block's smallest normal within half a subnormal step; the
    # scale leaves the block maximum in [256, 512) X, so elements above 448 X
    # saturate to 448 X.
    kept = np.minimum(np.abs(wb), 448.0 * scale)
    err = np.abs(table[q] * scale - wb)
    assert np.all(err <= (np.abs(wb) - kept) + np.maximum(kept * 2.0 ** -4, scale * 2.0 ** -10))
    assert np.array_equal(np.sign(table[q]) * (wb != 0), np.sign(wb))


PINS = [pin_round_bf16, pin_dispatch_hand, pin_dispatch_brute, pin_dense_mlp,
        pin_identity_expert, pin_naive_fp64, pin_streamed_equals_tokens,
        pin_e4m3_values, pin_e4m3_rounding_brute, pin_mx_scale_rule, pin_mx_round_trip,
        pin_mx_block_format]


# ----------------------------------------------------------------------------- tests

@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_dispatch_matches_brute_force_on_random_routings(orc):
    """Property form of the dispatch pin: on random shapes and ids (dropped
    -1 slots and out-of-range ids included), the oracle's dispatch equals the
    O(R * E) restatement, and the bad-id flag is set exactly when an id lies
    outside [-1, E)."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=200, deadline=None, derandomize=True)
    @hyp.given(T=st.integers(0, 40), k=st.integers(1, 6), E=st.integers(1, 12), data=st.data())
    def check(T, k, E, data):
        flat = data.draw(st.lists(st.integers(-2, E + 1), min_size=T * k, max_size=T * k))
        ids = np.array(flat, dtype=np.int32).reshape(T, k)
        counts, offsets, perm, inv, bad = orc.dispatch(ids, E)
        b_off, b_perm, b_inv = brute_dispatch(ids.reshape(-1), E)
        assert offsets.tolist() == b_off
        assert perm[:b_off[-1]].tolist() == b_perm and np.all(perm[b_off[-1]:] == -1)
        assert inv.tolist() == b_inv
        assert counts.tolist() == np.diff(b_off).tolist()
        assert bool(bad) == any(v < -1 or v >= E for v in flat)

    check()


# Each entry: (name, text in moe_oracle.c, replacement). Every mutation is a
# plausible slip: a dropped term, a swapped or transposed operand, a wrong
# sign, a wrong index or stride, a missing rounding, an unstable scatter.
MUTATIONS = [
    ("gate_up_swapped",
     "const uint16_t *wg = W13e + (size_t)n * (size_t)H;\n    const uint16_t *wu = W13e + (size_t)(I + n) * (size_t)H;",
     "const uint16_t *wu = W13e + (size_t)n * (size_t)H;\n    const uint16_t *wg = W13e + (size_t)(I + n) * (size_t)H;"),
    ("silu_sign", "g / (1.0f + expf(-g))", "g / (1.0f + expf(g))"),
    ("dropped_last_h_term", "for (int32_t h = 0; h < H; ++h) {", "for (int32_t h = 0; h < H - 1; ++h) {"),
    ("activation_truncated", "return f32_to_bf16_bits_rne(silu * u);",
     "{ uint32_t tb; float tv = silu * u; memcpy(&tb, &tv, 4); return (uint16_t)(tb >> 16); }"),
    ("w2_row_stride", "const uint16_t *w2 = W2e + (size_t)m * (size_t)I;",
     "const uint16_t *w2 = W2e + (size_t)m * (size_t)(I - 1);"),
    ("expert_stride", "W13 + (size_t)e * per13", "W13 + (size_t)e * per2"),
    ("combine_weight_dropped", "acc[m] += wj * y[m];", "acc[m] += y[m];"),
    ("combine_sorted_weight_dropped", "acc += w[s] * y_sorted[(size_t)row * H + m];",
     "acc += y_sorted[(size_t)row * H + m];"),
    ("scatter_unstable", "for (int32_t s = 0; s < R; ++s) {\n        int32_t e = ids[s];\n        if (e >= 0 && e < E) {\n            int32_t row",
     "for (int32_t s = R - 1; s >= 0; --s) {\n        int32_t e = ids[s];\n        if (e >= 0 && e < E) {\n            int32_t row"),
    ("offsets_inclusive", "offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
    ("round_half_up", "u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    ("round_truncate", "u += 0x7fffu + keep_lsb;", "u += 0u * keep_lsb;"),
    ("mx_emax_7", "e = (ex2 - 1) - 8;", "e = (ex2 - 1) - 7;"),
    ("e4m3_round_half_up", "int q = (int)rintf(ldexpf(a, 3 - e));", "int q = (int)floorf(ldexpf(a, 3 - e) + 0.5f);"),
    ("e4m3_subnormal_step", "int q = (int)rintf(ldexpf(a, 9));", "int q = (int)rintf(ldexpf(a, 8));"),
    ("e4m3_saturate_to_nan", "if (a >= 448.0f)\n        return sign | 0x7E;", "if (a >= 448.0f)\n        return sign | 0x7F;"),
    ("e4m3_value_bias", "mag = ldexpf(1.0f + (float)man / 8.0f, ex - 7);", "mag = ldexpf(1.0f + (float)man / 8.0f, ex - 8);"),
    ("mx_dequant_scale_bias", "int e = (int)s[r * nb + k / 32] - 127;", "int e = (int)s[r * nb + k / 32] - 126;"),
    ("mx_amax_half_block", "for (int i = 0; i < 32; ++i) {\n                float a",
     "for (int i = 0; i < 16; ++i) {\n                float a"),
    ("mx_block_stride", "const uint16_t *v = w + r * K + (int64_t)b * 32;", "const uint16_t *v = w + r * K + (int64_t)b * 31;"),
    ("invalid_id_kept", "if (e >= 0 && e < E)\n            counts[e] += 1;", "if (e >= 0 && e < E + 1 && e != E)\n            counts[e] += 1;\n        if (e == E) counts[0] += 1;"),
]


def run_pins(path: str) -> list:
    """Run every pin against the oracle build at ``path``; return the names that failed."""
    lib = Oracle(path)
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as ex:  # a shape error or the like also counts as caught
            failed.append(f"{pin.__name__}:{type(ex).__name__}")
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes(tmp_path, name, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    c = tmp_path / "mut.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    "-o", str(so), str(c), "-lm"], check=True)
    # A mutant may write out of bounds, so it runs in a child process: a crash
    # there (non-zero exit without our marker) also counts as caught.
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--run-pins", str(so)],
                       capture_output=True, text=True, env=env, timeout=300)
    if r.returncode == 0:
        assert "CAUGHT" in r.stdout, r.stdout + r.stderr
    else:
        assert "NOT CAUGHT" not in r.stdout, f"no pin caught the planted mistake {name}"


if __name__ == "__main__":
    if len(sys.argv) == 3 and sys.argv[1] == "--run-pins":
        failed = run_pins(sys.argv[2])
        print(("CAUGHT " + ",".join(failed)) if failed else "NOT CAUGHT")
        sys.exit(0 if failed else 3)

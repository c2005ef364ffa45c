"""Pins of the oracle's FP4 format and of its FP4 pool.

FP4 here is the E2M1 element format of the OCP MX specification in NVIDIA's
NVFP4 arrangement: one E4M3 scale per 16 consecutive head_dim elements of a
token's K or V row, on top of the per-KV-head fp32 scale.  The pins:
  * the E2M1 decoder against the specification's code points (golden file);
  * the encoder against round-to-nearest-even derived independently here from
    the grid spacing (0.5 below 2, 1 up to 4, 2 up to 6) with numpy's
    half-to-even rounding, on every finite bf16 value, plus saturation, NaN,
    signed zero and ties;
  * the row quantizer against torch: torch.max for the group maximum, torch's
    own E4M3 conversion for the block scale, torch float32 arithmetic for the
    divisor and the quotient, and the grid rule above for the codes;
  * the block-scale rule (largest magnitude onto E2M1's 6) by the format
    itself: rows already on the FP4 grid come back losslessly, a group's
    maximum decodes to itself, and 6·448·G is the largest unsaturated group;
  * attention over an FP4 pool against dense fp64 attention (torch) on the
    values decoded from the stored codes and scales with the golden tables.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = 16


def _golden_e2m1():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_ocp_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, val = line.split()
                rows.append((int(code, 16), float(val)))
    return rows


E2M1 = np.array([v for _, v in sorted(_golden_e2m1())])          # value of code c


def _e4m3_values() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _grid_rne(q: np.ndarray) -> np.ndarray:
    """E2M1 codes of float values by the grid rule: the multiple of the local
    spacing nearest to |q|, ties to an even multiple, capped at 6; the sign bit
    from the sign of q; NaN -> +0."""
    q = np.asarray(q, np.float64)
    a = np.abs(q)
    spacing = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    mag = np.minimum(np.round(a / spacing) * spacing, 6.0)
    mag = np.where(np.isnan(q), 0.0, mag)
    code = np.array([int(np.nonzero(E2M1[:8] == m)[0][0]) for m in mag], np.uint8)
    sign = np.where(np.signbit(q) & ~np.isnan(q), 8, 0).astype(np.uint8)
    return code | sign


def test_e2m1_golden_table_is_complete():
    rows = _golden_e2m1()
    assert sorted(c for c, _ in rows) == list(range(16))


def test_e2m1_decode_ocp_code_points():
    for code, val in _golden_e2m1():
        got = oracle.e2m1_to_double(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e2m1_roundtrip_every_code():
    for c in range(16):
        assert oracle.e2m1_from_float(oracle.e2m1_to_double(c)) == c, hex(c)


def test_e2m1_encode_every_finite_bf16_matches_the_grid_rule():
    bits = np.arange(65536, dtype=np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    x = x[np.isfinite(x)]
    ref = _grid_rne(x)
    got = np.array([oracle.e2m1_from_float(float(v)) for v in x], np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.2500001, 0x1), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4),
    (3.5, 0x6), (5.0, 0x6), (5.0001, 0x7), (6.0, 0x7), (6.5, 0x7), (1e30, 0x7),
    (math.inf, 0x7), (-math.inf, 0xF), (-0.1, 0x8), (-0.0, 0x8), (0.0, 0x0),
    (math.nan, 0x0), (-2.9, 0xD),
])
def test_e2m1_encode_special_cases(x, code):
    # ties to even, saturation to 6, signed zero, NaN stored as +0
    assert oracle.e2m1_from_float(x) == code


def test_e2m1_encode_monotone():
    xs = np.linspace(-7, 7, 20001).astype(np.float32)
    vals = [oracle.e2m1_to_double(oracle.e2m1_from_float(float(x))) for x in xs]
    assert all(a <= b for a, b in zip(vals, vals[1:]))


def _torch_quantize_row(x_bf16: torch.Tensor, G: float):
    """The row quantizer restated with torch primitives (see the module doc)."""
    x = x_bf16.float().view(-1, 16)
    amax = torch.where(torch.isnan(x), torch.zeros_like(x), x.abs()).max(dim=1).values
    t = torch.tensor(6.0, dtype=torch.float32) * torch.tensor(G, dtype=torch.float32)
    sc = (amax / t).clamp(max=448.0).to(torch.float8_e4m3fn)
    S = sc.float() * torch.tensor(G, dtype=torch.float32)
    q = x / S[:, None]
    codes = _grid_rne(q.reshape(-1).numpy())
    codes[np.repeat((S == 0).numpy(), 16)] = 0
    return codes, sc.view(torch.uint8).numpy()


@pytest.mark.parametrize("G", [1.0, 0.01, 3.7 / (6 * 448), 1e-5, 0.5])
def test_fp4_row_quantizer_matches_torch(G):
    rng = np.random.default_rng(int(G * 1e6) % 1000 + 3)
    for trial in range(60):
        std = [1.0, 30.0, 1e-3, 0.2][trial % 4]
        x = torch.from_numpy(rng.normal(0, std, 128).astype(np.float32)).bfloat16()
        if trial % 7 == 0:
            x[5:21] = 0                                  # an all-zero group
        codes, scales = oracle.fp4_quantize_row(x, G)
        rc, rs = _torch_quantize_row(x, G)
        assert np.array_equal(scales, rs), (G, trial)
        assert np.array_equal(codes, rc), (G, trial)


def test_fp4_row_quantizer_bounds_the_error():
    # Away from saturation every element decodes to within half a grid step
    # (relative to the block's scale) of its value.
    rng = np.random.default_rng(4)
    G = 0.02
    ev = _e4m3_values()
    for _ in range(200):
        x = torch.from_numpy(rng.normal(0, 1, 128).astype(np.float32)).bfloat16()
        codes, scales = oracle.fp4_quantize_row(x, G)
        xv = x.double().numpy()
        S = np.repeat(ev[scales] * G, 16)
        dec = E2M1[codes] * S
        q = np.abs(xv) / S
        half_step = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0)) * S
        inside = q <= 6
        assert np.all(np.abs(dec - xv)[inside] <= half_step[inside] * (1 + 1e-12))
        # the group maximum lands in the top binade of the grid (4 or 6) unless
        # the scale saturated or the group is zero
        for j in range(8):
            if S[16 * j] > 0:
                assert np.abs(E2M1[codes[16 * j:16 * j + 16]]).max() >= 4.0


def test_fp4_row_quantizer_special_values():
    x = torch.zeros(32).bfloat16()
    x[0], x[1], x[2] = float("nan"), 3.0, -float("inf")
    x[17] = 1e-30                                  # group 1: scale rounds to 0
    codes, scales = oracle.fp4_quantize_row(x, 1.0)
    assert codes[0] == 0                           # NaN stores +0 and is left out of the maximum
    assert scales[0] == 0x7E                       # inf / 6 saturates the E4M3 scale at 448
    assert codes[2] == 0xF                         # -inf saturates at -6
    assert scales[1] == 0 and not codes[16:].any()


def _fill_identity(pool, k, v, lens, mbs):
    B = len(lens)
    tables = np.full((B, mbs), -1, np.int32)
    for b, c in enumerate(lens):
        nb = -(-c // BS)
        tables[b, :nb] = np.arange(b * mbs, b * mbs + nb)
        slots = tables[b, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS
        pool.write(k[b, :c], v[b, :c], slots)
    return tables


def test_fp4_identity_table_equals_dense_on_decoded_codes():
    torch.manual_seed(6)
    D, Hq, Hkv = 128, 16, 4
    lens = [1, 16, 29, 70]
    B, mbs = len(lens), -(-max(lens) // BS)
    q = torch.randn(B, Hq, D).bfloat16()
    k = (2 * torch.randn(B, max(lens), Hkv, D)).bfloat16()
    v = torch.randn(B, max(lens), Hkv, D).bfloat16()
    ks = np.array([0.011, 0.002, 0.02, 0.05], np.float32)
    vs = np.array([0.012, 0.009, 0.003, 0.004], np.float32)
    pool = oracle.Pool(B * mbs, BS, Hkv, D, dtype="fp4")
    pool.set_scales(ks, vs)
    tables = _fill_identity(pool, k, v, lens, mbs)
    arr, sc = pool.array(), pool.block_scales()
    ev = _e4m3_values()
    # every stored row is the row quantizer's output (the write scatters it)
    kd = torch.zeros(B, max(lens), Hkv, D, dtype=torch.float64)
    vd = torch.zeros_like(kd)
    for b, c in enumerate(lens):
        for t in range(c):
            blk, off = tables[b, t // BS], t % BS
            for h in range(Hkv):
                for kv, src, G, dst in ((0, k, ks[h], kd), (1, v, vs[h], vd)):
                    codes, scales = _torch_quantize_row(src[b, t, h], float(G))
                    assert np.array_equal(arr[blk, kv, off, h], codes)
                    assert np.array_equal(sc[blk, kv, off, h], scales)
                    dst[b, t, h] = torch.from_numpy(
                        E2M1[codes] * np.repeat(ev[scales], 16) * np.float64(G))
    scale = 1.0 / np.sqrt(D)
    got = pool.decode(q, tables, np.array(lens), scale)
    g = Hq // Hkv
    for b, c in enumerate(lens):
        qq = q[b].double().view(Hkv, g, D)
        kk = kd[b, :c].permute(1, 0, 2)                      # [Hkv, c, D]
        vv = vd[b, :c].permute(1, 0, 2)
        w = torch.softmax(scale * qq @ kk.transpose(1, 2), dim=-1)
        ref = (w @ vv).reshape(Hq, D).numpy()
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-6)


def test_fp4_block_copy_moves_codes_and_scales():
    pool = oracle.Pool(6, BS, 2, 64, dtype="fp4")
    pool.set_scales(np.array([0.01, 0.02], np.float32), np.array([0.03, 0.04], np.float32))
    torch.manual_seed(2)
    T = 6 * BS
    k, v = torch.randn(T, 2, 64).bfloat16(), torch.randn(T, 2, 64).bfloat16()
    pool.write(k, v, np.arange(T))
    arr, sc = pool.array().copy(), pool.block_scales().copy()
    pool.copy_blocks([[1, 4], [4, 0]])                       # in order: 1 -> 4, then 4 -> 0
    a2, s2 = pool.array(), pool.block_scales()
    for dst, src in ((4, 1), (0, 1)):
        assert np.array_equal(a2[dst], arr[src]) and np.array_equal(s2[dst], sc[src])
    assert np.array_equal(a2[[2, 3, 5]], arr[[2, 3, 5]])


# -- the block-scale rule, pinned by the format's own grid --------------------
#
# NVFP4 picks each 16-element block's scale so that the block's largest
# magnitude maps onto the largest E2M1 magnitude, 6.  Data that already lies
# on the format's grid -- 16 E2M1 values with at least one of magnitude 6,
# times a representable E4M3 scale s, times a power-of-two head scale G --
# must therefore come back with exactly those codes and that scale: every step
# (6·G, amax / (6·G), E4M3(s), s·G, x / S) is exact, and the quantiser is
# lossless on it.  A divisor of 4·G or 8·G (or a missing G) puts the largest
# element at 4 or 12 and breaks the round trip.

def _on_grid_row(rng, s_code: int, G: float):
    """A 128-element row whose every group is on the FP4 grid with scale code
    s_code; returns (bf16 row, element codes, scale code)."""
    ev = _e4m3_values()
    s = ev[s_code]
    codes = rng.integers(0, 16, 128).astype(np.uint8)
    for j in range(8):                                   # one ±6 per group
        codes[16 * j + rng.integers(0, 16)] = 0x7 | (8 * int(rng.integers(0, 2)))
    vals = E2M1[codes] * s * G
    x = torch.from_numpy(vals.astype(np.float32)).bfloat16()
    assert np.array_equal(x.double().numpy(), vals)      # exact in bf16 (<= 5 significant bits)
    return x, codes, s_code


@pytest.mark.parametrize("G", [1.0, 2.0 ** -7, 2.0 ** -11, 2.0 ** 3])
def test_fp4_on_grid_groups_round_trip_exactly(G):
    rng = np.random.default_rng(int(-math.log2(G)) + 40)
    ev = _e4m3_values()
    # normal E4M3 scales across the whole range, subnormal ones, and 448
    for s_code in [0x08, 0x11, 0x2A, 0x38, 0x3F, 0x40, 0x55, 0x6D, 0x7E, 0x01, 0x05]:
        x, codes, sc = _on_grid_row(rng, s_code, G)
        got_c, got_s = oracle.fp4_quantize_row(x, G)
        # -0 and +0 both decode to 0: compare values for zeros, codes otherwise
        assert np.array_equal(got_s, np.full(8, sc, np.uint8)), (hex(s_code), got_s)
        dec = E2M1[got_c] * np.repeat(ev[got_s], 16) * G
        assert np.array_equal(dec, x.double().numpy()), hex(s_code)
        nz = E2M1[codes] != 0
        assert np.array_equal(got_c[nz], codes[nz])


def test_fp4_group_maximum_decodes_to_itself():
    # For any group whose amax / (6 G) is an E4M3 value the largest element
    # is stored as code ±6 and decodes to exactly ±amax.
    rng = np.random.default_rng(77)
    ev = _e4m3_values()
    G = 2.0 ** -9
    for s_code in range(0x08, 0x7F, 3):                  # normal E4M3 scales up to 448
        s = ev[s_code]
        amax = 6 * s * G
        x = rng.uniform(-amax, amax, 128)
        x[rng.integers(0, 16) + 16 * np.arange(8)] = amax * rng.choice([-1, 1], 8)
        xb = torch.from_numpy(x.astype(np.float32)).bfloat16()
        xv = xb.double().numpy()
        got_c, got_s = oracle.fp4_quantize_row(xb, G)
        for j in range(8):
            grp = xv[16 * j:16 * j + 16]
            i = int(np.argmax(np.abs(grp)))
            if np.abs(grp[i]) != amax:                   # bf16 rounding moved the maximum
                continue
            assert got_s[j] == s_code, (hex(s_code), j)
            assert got_c[16 * j + i] & 0x7 == 0x7
            assert E2M1[got_c[16 * j + i]] * ev[got_s[j]] * G == grp[i]


def test_fp4_largest_scale_does_not_saturate_elements():
    # amax = 6 · 448 · G is the largest group the scale represents without
    # saturation: the scale is 448 (0x7E) and the maximum decodes exactly.
    G = 2.0 ** -4
    x = torch.zeros(16).bfloat16()
    x[3], x[9] = 6 * 448 * G, -3 * 448 * G
    codes, scales = oracle.fp4_quantize_row(x, G)
    assert scales[0] == 0x7E
    assert codes[3] == 0x7 and codes[9] == 0xD

"""The CPU oracle pinned to what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: hand-worked
values (tests/golden/), a library routine it does not use (torch's float8
conversion, numpy's matmul), exact rational arithmetic, closed forms and
invariants of the method.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# The E2M1 magnitudes by code (OCP microscaling FP4 E2M1: 1 sign, 2 exponent, 1 mantissa bit).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def unpack_codes(q):
    """Independent unpacking of the documented layout: element 2i in the low nibble."""
    N, Kh = q.shape
    c = np.empty((N, 2 * Kh), dtype=np.int64)
    c[:, 0::2] = q & 15
    c[:, 1::2] = q >> 4
    return c


def independent_dequant(q, sf, g):
    mag = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    e4 = torch_e4m3_values()
    return mag[unpack_codes(q)] * np.repeat(e4[sf], 16, axis=1) * float(g)


# ---------------------------------------------------------------- formats ----

def test_e2m1_decode_table(oracle_lib):
    for c in range(16):
        want = E2M1_TABLE[c & 7] * (-1.0 if c & 8 else 1.0)
        got = oracle_lib.e2m1_decode(c)
        assert got == want and math.copysign(1.0, got) == (-1.0 if c & 8 else 1.0)


def test_e4m3_decode_matches_torch(oracle_lib):
    ref = torch_e4m3_values()
    for b in range(256):
        got = oracle_lib.e4m3_decode(b)
        if np.isnan(ref[b]):
            assert math.isnan(got)
        else:
            assert got == ref[b], b


def test_e4m3_decode_monotone(oracle_lib):
    pos = [oracle_lib.e4m3_decode(b) for b in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9


def _e4m3_sweep():
    vals = torch_e4m3_values()
    pos = np.sort(vals[(vals >= 0) & np.isfinite(vals)])
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.Generator(np.random.PCG64(7))
    rand = rng.uniform(0, 464, 20000)
    small = rng.uniform(0, 2.0 ** -5, 5000)
    x = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), rand, small,
                        [464.0, 460.0, 2.0 ** -10, 3 * 2.0 ** -11]]).astype(np.float32)
    return np.concatenate([x, -x])


def test_e4m3_encode_matches_torch(oracle_lib):
    x = _e4m3_sweep()
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_lib.e4m3_encode(v) for v in x], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def test_e4m3_encode_saturates(oracle_lib):
    # Beyond 448 the oracle saturates (the pages clamp before the cast, so the
    # cast itself never sees these values).
    for v in (470.0, 1e6, float("inf")):
        assert oracle_lib.e4m3_encode(v) == 0x7E
        assert oracle_lib.e4m3_encode(-v) == 0xFE


def _e2m1_exact(x: float) -> int:
    """Nearest E2M1 code by exact rational distances; ties to the even code."""
    fx = Fraction(x)
    a = abs(fx)
    sign = 8 if math.copysign(1.0, x) < 0 else 0
    if a >= 6:
        return sign | 7
    dist = [(abs(a - Fraction(v)), c) for c, v in enumerate(E2M1_TABLE)]
    dmin = min(d for d, _ in dist)
    cands = [c for d, c in dist if d == dmin]
    if len(cands) == 1:
        return sign | cands[0]
    even = [c for c in cands if c % 2 == 0]
    assert len(even) == 1
    return sign | even[0]


def test_e2m1_encode_exhaustive(oracle_lib):
    grid = np.array(E2M1_TABLE)
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.Generator(np.random.PCG64(11))
    x = np.concatenate([grid, mids, np.nextafter(mids.astype(np.float32), 0),
                        np.nextafter(mids.astype(np.float32), 10),
                        rng.uniform(0, 7, 4000), [0.0, 6.5, 100.0]]).astype(np.float32)
    x = np.concatenate([x, -x])
    for v in x:
        assert oracle_lib.e2m1_encode(float(v)) == _e2m1_exact(float(v)), float(v)


def test_e2m1_ties_go_to_even(oracle_lib):
    ties = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6}
    for x, c in ties.items():
        assert oracle_lib.e2m1_encode(x) == c
        assert oracle_lib.e2m1_encode(-x) == c | 8
    assert oracle_lib.e2m1_encode(-0.0) == 0x8
    assert oracle_lib.e2m1_encode(-0.1) == 0x8


# ------------------------------------------------------------------ index ----

@pytest.mark.parametrize("V,n_kept,forced,N", [
    (248_320, 64_026, 1_024, 64_064),   # the 64k draft vocabulary of the DGX-Spark page
    (16_384, 4_000, 32, 4_032),
    (248_320, 98_304, 1_024, 98_304),   # already a multiple of 64: no padding
    (100, 1, 0, 64),
])
def test_index_padding(oracle_lib, V, n_kept, forced, N):
    keep = syn.keep_mask(5, V, n_kept, forced)
    idx, nk = oracle_lib.build_index(keep)
    assert nk == n_kept and idx.size == N and N % 64 == 0
    kept = np.nonzero(keep)[0]
    assert np.array_equal(idx[:nk], kept)          # ascending, as keep.nonzero() yields
    assert np.all(np.diff(idx[:nk]) > 0)
    assert np.all(idx[nk:] == idx[0])              # pads repeat the first kept id
    assert np.array_equal(idx[:forced], np.arange(forced))


def test_index_empty_keep_is_an_error(oracle_lib):
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.build_index(np.zeros(64, np.uint8))


def test_byte_ledger(oracle_lib):
    # q38_draft.py docstring: the BF16 248k x 2560 head alone is 1.27 GB.
    V, K, N = 248_320, 2_560, 64_064
    assert V * K * 2 == 1_271_398_400
    W = bf16(np.random.default_rng(1).normal(0, 0.02, (8, 64)))
    q, sf, _ = oracle_lib.nvfp4_quantize(W, np.arange(8, dtype=np.int32))
    per_row = q.shape[1] + sf.shape[1]             # bytes per head row at K = 64
    assert q.shape == (8, 32) and sf.shape == (8, 4)
    assert per_row * (K // 64) * N == 92_252_160   # 82,001,920 codes + 10,250,240 scales
    assert round(V * K * 2 / 92_252_160, 1) == 13.8


# ---------------------------------------------------------- quantisation ----

def _read_blocks():
    rows = []
    with open(os.path.join(GOLDEN, "nvfp4_blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, s, w, c = [t.strip() for t in line.split("|")]
            rows.append((name, int(s, 16), [float(v) for v in w.split()],
                         [int(v, 16) for v in c.split()]))
    return rows


def test_nvfp4_hand_worked_blocks(oracle_lib):
    rows = _read_blocks()
    # weights are rounded to BF16 as the fixture's derivation states
    W = np.stack([bf16(w) for _, _, w, _ in rows])
    q, sf, g = oracle_lib.nvfp4_quantize(W, np.arange(len(rows), dtype=np.int32))
    assert g == np.float32(1.0)
    codes = unpack_codes(q)
    for i, (name, s, _, c) in enumerate(rows):
        assert sf[i, 0] == s, name
        assert list(codes[i]) == c, name


def test_fp8_hand_worked_values(oracle_lib):
    vals, codes = [], []
    with open(os.path.join(GOLDEN, "fp8_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w, c = [t.strip() for t in line.split("|")]
            vals.append(float(w))
            codes.append(int(c, 16))
    row = np.zeros(16, np.float32)
    row[: len(vals)] = vals
    q, scale = oracle_lib.fp8_quantize(bf16(row)[None, :], np.zeros(1, np.int32))
    assert scale == np.float32(1.0)
    assert list(q[0, : len(vals)]) == codes


def _random_head(seed, V=96, K=64):
    return syn.head_bf16(seed, V, K)


def test_nvfp4_global_scale_closed_form(oracle_lib):
    W = _random_head(3)
    idx = np.arange(0, 96, 3, dtype=np.int32)
    _, _, g = oracle_lib.nvfp4_quantize(W, idx)
    amax = np.abs(syn.bf16_bits_to_f32(W[idx])).max()
    assert g == np.float32(amax) / np.float32(6 * 448)


def test_nvfp4_codes_are_nearest_and_block_max_hits_six(oracle_lib):
    W = _random_head(4, V=128, K=256)
    idx = np.arange(128, dtype=np.int32)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    w = syn.bf16_bits_to_f32(W).astype(np.float64).reshape(128, 16, 16)
    s = torch_e4m3_values()[sf]                          # independent scale decode
    # the block scale is the E4M3 value nearest to bamax / (6 g) (torch's cast)
    t = (np.abs(w).max(-1).astype(np.float32) / np.float32(6 * np.float32(g))).astype(np.float32)
    want_sf = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sf, want_sf)
    codes = unpack_codes(q).reshape(128, 16, 16)
    mag = np.array(E2M1_TABLE)
    d = s[..., None] * float(g)
    x = np.clip(w / d, -6, 6)
    err = np.abs(np.sign(x) * mag[codes & 7] - x)
    alt = np.abs(np.abs(x)[..., None] - mag).min(-1)
    assert np.all(err <= alt + 1e-12)                     # nearest grid point
    # the largest element of each block encodes to magnitude 6 (code 7) when s is normal
    normal = s >= 2.0 ** -6
    top = np.take_along_axis(codes & 7, np.abs(w).argmax(-1)[..., None], -1)[..., 0]
    assert normal.mean() > 0.9 and np.all(top[normal] == 7)


def test_nvfp4_dequant_error_bound(oracle_lib):
    W = _random_head(5, V=256, K=256)
    idx = np.arange(256, dtype=np.int32)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    w = syn.bf16_bits_to_f32(W).astype(np.float64)
    wq = independent_dequant(q, sf, g)
    d = np.repeat(torch_e4m3_values()[sf], 16, axis=1) * float(g)
    err = np.abs(w - wq)
    x = np.abs(w) / np.where(d > 0, d, 1)
    nz = d > 0
    # grid spacing 0.5 below 2, 1 below 4, 2 up to 6 (half of it is the rounding bound),
    # plus the clamp excess of at most 6/(1 - 2^-4) - 6 above 6
    bound = np.where(x <= 2, 0.25, np.where(x <= 4, 0.5, 1.0)) * d
    assert np.all(err[nz] <= bound[nz] * (1 + 1e-6))
    assert np.all(wq[~nz] == 0)
    assert np.all(np.abs(w[~nz]) < 2.0 ** -10 * 6 * float(g) * (1 + 1e-6))


def test_fp8_closed_form_and_error_bound(oracle_lib):
    W = _random_head(6, V=64, K=128)
    idx = np.arange(64, dtype=np.int32)
    q, scale = oracle_lib.fp8_quantize(W, idx)
    w = syn.bf16_bits_to_f32(W)
    assert scale == np.float32(np.abs(w).max()) / np.float32(448)
    wq = torch_e4m3_values()[q] * float(scale)
    err = np.abs(w.astype(np.float64) - wq)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(w), 2.0 ** -10 * float(scale)) * (1 + 1e-6))
    assert (q & 0x7F).max() == 0x7E                              # amax element -> +-448


def test_zero_head_uses_amax_floor(oracle_lib):
    W = np.zeros((4, 32), np.uint16)
    idx = np.arange(4, dtype=np.int32)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    assert g == np.float32(1e-12) / np.float32(2688) and not q.any() and not sf.any()
    q8, s8 = oracle_lib.fp8_quantize(W, idx)
    assert s8 == np.float32(1e-12) / np.float32(448) and not q8.any()


def test_gather_follows_idx(oracle_lib):
    W = _random_head(8, V=64, K=32)
    idx = np.array([5, 9, 9, 63, 0, 5] + [5] * 58, dtype=np.int32)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    q2, sf2, g2 = oracle_lib.nvfp4_quantize(W[idx], np.arange(64, dtype=np.int32))
    assert np.array_equal(q, q2) and np.array_equal(sf, sf2) and g == g2
    assert np.array_equal(q[1], q[2]) and np.array_equal(q[0], q[5])


# ------------------------------------------------------------- draft step ----

def _tiny_case(seed, V=192, K=64, n_kept=70, M=3):
    W = syn.head_bf16(seed, V, K)
    keep = syn.keep_mask(seed + 1, V, n_kept, 4)
    h = syn.hidden_bf16(seed + 2, M, K)
    return W, keep, h


def test_gemv_matches_numpy_matmul(oracle_lib):
    W, keep, h = _tiny_case(20)
    idx, nk = oracle_lib.build_index(keep)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    y, A = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, h)
    hf = syn.bf16_bits_to_f32(h).astype(np.float64)
    wq = independent_dequant(q, sf, g)
    assert np.allclose(y, hf @ wq.T, rtol=1e-12, atol=1e-14)
    assert np.allclose(A, np.abs(hf[:, None, :] * wq[None]).sum(-1), rtol=1e-12)


def test_gemv_fp8_and_bf16_match_numpy(oracle_lib):
    W, keep, h = _tiny_case(21)
    idx, _ = oracle_lib.build_index(keep)
    q, s = oracle_lib.fp8_quantize(W, idx)
    y8, _ = oracle_lib.gemv(oracle_lib.FMT_FP8, q, None, s, h)
    hf = syn.bf16_bits_to_f32(h).astype(np.float64)
    assert np.allclose(y8, hf @ (torch_e4m3_values()[q] * float(s)).T, rtol=1e-12, atol=1e-14)
    yb, _ = oracle_lib.gemv(oracle_lib.FMT_BF16, W, None, None, h)
    assert np.allclose(yb, hf @ syn.bf16_bits_to_f32(W).astype(np.float64).T, rtol=1e-12, atol=1e-14)


def test_one_hot_hidden_reads_one_column(oracle_lib):
    W, keep, _ = _tiny_case(22)
    idx, _ = oracle_lib.build_index(keep)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    K = W.shape[1]
    h = np.zeros((K, K), np.uint16)
    h[np.arange(K), np.arange(K)] = bf16(np.ones(K))
    y, _ = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, h)
    assert np.array_equal(y, independent_dequant(q, sf, g).T)   # y[k, n] = w'[n, k]


def test_restricted_argmax_equals_masked_full_argmax(oracle_lib):
    # "lossless" at head level: the argmax over the kept rows, mapped through
    # dh_idx, is the argmax over the full vocabulary with non-kept ids masked.
    rng = np.random.default_rng(23)
    for trial in range(40):
        V, K = 64, int(rng.choice([16, 32]))
        W = syn.head_bf16(100 + trial, V, K)
        keep = (rng.random(V) < rng.uniform(0.05, 0.9)).astype(np.uint8)
        if not keep.any():
            keep[rng.integers(V)] = 1
        h = syn.hidden_bf16(200 + trial, 2, K)
        idx, nk = oracle_lib.build_index(keep)
        q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
        y, _ = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, h)
        ids, _ = oracle_lib.top_tokens(y, idx)
        full = np.full((2, V), -np.inf)
        full[:, idx[:nk]] = y[:, :nk]
        assert np.array_equal(ids, np.argmax(full, axis=1))
        # and equals the brute-force best over kept ids (first max)
        for m in range(2):
            best = max(range(nk), key=lambda n: (y[m, n], -n))
            assert ids[m] == idx[best]


def test_scatter_is_minus_inf_off_the_kept_ids(oracle_lib):
    W, keep, h = _tiny_case(24)
    idx, nk = oracle_lib.build_index(keep)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    y, _ = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, h)
    out = oracle_lib.scatter_logits(y, idx, nk, W.shape[0])
    kept = keep.astype(bool)
    assert np.all(np.isneginf(out[:, ~kept]))
    assert np.all(np.isfinite(out[:, kept])) and np.isfinite(out).sum(1).tolist() == [nk] * 3
    assert np.array_equal(out[:, idx[:nk]], y[:, :nk].astype(np.float32))


def test_all_kept_reduces_to_plain_argmax(oracle_lib):
    W, _, h = _tiny_case(25, V=128)
    idx, nk = oracle_lib.build_index(np.ones(128, np.uint8))
    assert nk == 128 and np.array_equal(idx, np.arange(128))
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    y, _ = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, h)
    ids, _ = oracle_lib.top_tokens(y, idx)
    assert np.array_equal(ids, np.argmax(hf_dot(h, independent_dequant(q, sf, g)), axis=1))


def hf_dot(h, w):
    return syn.bf16_bits_to_f32(h).astype(np.float64) @ w.T


def test_argmax_first_max_and_pads(oracle_lib):
    y = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]])
    ids, rows = oracle_lib.top_tokens(y, np.array([10, 20, 30, 10], np.int32))
    assert rows.tolist() == [1, 0] and ids.tolist() == [20, 10]
    # identical drafts give identical results; pads (copies of row 0) never change the id
    W, keep, h = _tiny_case(26)
    idx, nk = oracle_lib.build_index(keep)
    q, sf, g = oracle_lib.nvfp4_quantize(W, idx)
    hh = np.stack([h[0], h[0]])
    y, _ = oracle_lib.gemv(oracle_lib.FMT_NVFP4, q, sf, g, hh)
    assert np.array_equal(y[0], y[1])
    assert np.all(y[:, nk:] == y[:, :1])


# ------------------------------------------------- W8A8 FP8 head (per-token) ----

def test_fp8_act_quantize_hand_worked_row(oracle_lib):
    # amax = 448 c, so s = c and every quotient below is exact; E4M3 bytes by
    # the format (bias 7, 3 mantissa bits): 448 = 1.75 * 2^8 -> 0x7E,
    # -224 -> 0xF6, 1 -> 0x38, 0 -> 0x00; 17 = 1.0625 * 2^4 lies halfway
    # between 16 (mantissa 000) and 18 (001) -> even -> 0x58; 19 lies halfway
    # between 18 (001) and 20 (010) -> even -> 0x5A.
    vals = np.array([448.0, -224.0, 1.0, 0.0, 17.0, 19.0], np.float32)
    for c in (1.0, 2.0 ** -3, 2.0 ** 5):
        qx, sx = oracle_lib.fp8_act_quantize(bf16(vals * np.float32(c))[None])
        assert [int(v) for v in qx[0]] == [0x7E, 0xF6, 0x38, 0x00, 0x58, 0x5A]
        assert sx[0] == np.float32(c)


def test_fp8_act_quantize_rows_are_independent_and_zero_row_floors(oracle_lib):
    h = syn.hidden_bf16(40, 3, 64)
    h[1] = 0
    qx, sx = oracle_lib.fp8_act_quantize(h)
    assert sx[1] == np.float32(1e-12) / np.float32(448) and not qx[1].any()
    for m in (0, 2):
        q1, s1 = oracle_lib.fp8_act_quantize(h[m:m + 1])
        assert np.array_equal(q1[0], qx[m]) and s1[0] == sx[m]
        x = syn.bf16_bits_to_f32(h[m])
        assert sx[m] == np.float32(np.abs(x).max()) / np.float32(448)


def test_fp8_act_quantize_error_bound_against_torch_values(oracle_lib):
    h = syn.hidden_bf16(41, 4, 256)
    qx, sx = oracle_lib.fp8_act_quantize(h)
    x = syn.bf16_bits_to_f32(h).astype(np.float64)
    xq = torch_e4m3_values()[qx] * sx[:, None].astype(np.float64)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * sx[:, None].astype(np.float64))
    assert np.all(np.abs(x - xq) <= bound * (1 + 1e-6))
    assert np.all((qx & 0x7F).max(axis=1) == 0x7E)                # each row's amax -> +-448


def test_w8a8_reduces_to_w8a16_when_h_is_on_the_e4m3_grid(oracle_lib):
    # h = 2^-3 * (E4M3 values with a 448 in every row): per-token quantisation
    # is then exact (s = 2^-3), so the W8A8 logits equal the W8A16 logits of the
    # same head, computed by the separately pinned or_gemv.
    rng = np.random.default_rng(42)
    e4 = torch_e4m3_values()
    finite = np.array([b for b in range(256) if np.isfinite(e4[b])])
    K, M = 128, 3
    codes = rng.choice(finite, size=(M, K))
    codes[:, 7] = 0x7E
    h = bf16((e4[codes] * 2.0 ** -3).astype(np.float32))
    W, keep, _ = _tiny_case(43, K=K)
    idx, _ = oracle_lib.build_index(keep)
    q, s = oracle_lib.fp8_quantize(W, idx)
    qx, sx = oracle_lib.fp8_act_quantize(h)
    assert np.array_equal(qx, codes) and np.all(sx == np.float32(2.0 ** -3))
    y8, A8 = oracle_lib.gemv_w8a8(q, s, qx, sx)
    y16, A16 = oracle_lib.gemv(oracle_lib.FMT_FP8, q, None, s, h)
    assert np.allclose(y8, y16, rtol=1e-13, atol=1e-15) and np.allclose(A8, A16, rtol=1e-13)


def test_w8a8_matches_numpy_on_decoded_codes(oracle_lib):
    W, keep, h = _tiny_case(44)
    idx, _ = oracle_lib.build_index(keep)
    q, s = oracle_lib.fp8_quantize(W, idx)
    qx, sx = oracle_lib.fp8_act_quantize(h)
    y, _ = oracle_lib.gemv_w8a8(q, s, qx, sx)
    e4 = torch_e4m3_values()
    ref = (e4[qx] @ e4[q].T) * float(s) * sx[:, None].astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)

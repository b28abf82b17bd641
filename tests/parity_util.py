"""Shared helpers of the parity tests: workloads, the oracle's expected values
and the tolerance rules (logits |dy| <= 2e-3 * sum|w' h| + 1e-5; an argmax row
is accepted when it is the oracle's or lies within the two rows' tolerances)."""
from __future__ import annotations

import numpy as np

import oracle
import synthetic as syn

REL_TOL = 2e-3
ABS_TOL = 1e-5


def tol(A):
    return REL_TOL * A + ABS_TOL


def check_logits(y_gpu, y_or, A, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_or)
    bound = tol(A)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{what}: {len(bad)} logits out of tolerance, first {bad[:3].tolist()}"
    return float((err / np.maximum(A, 1e-30)).max())


def check_argmax_rows(rows_gpu, y_or, A, n_kept, what=""):
    """Each GPU row must be the oracle's first-max row or tie with it within tolerance."""
    y = y_or[:, :n_kept]
    r_star = np.argmax(y, axis=1)
    exact = 0
    for m, j in enumerate(np.asarray(rows_gpu)):
        r = int(r_star[m])
        if j == r:
            exact += 1
            continue
        assert 0 <= j < n_kept, f"{what}: draft {m}: row {j} outside kept rows"
        gap = y[m, r] - y[m, j]
        assert gap <= tol(A[m, r]) + tol(A[m, j]), \
            f"{what}: draft {m}: row {j} vs oracle row {r}, gap {gap:.3g} beyond tolerance"
    return exact


def ids_to_rows(ids, idx, n_kept):
    """Map target ids back to head rows (ids are distinct over the kept rows)."""
    pos = {int(v): n for n, v in enumerate(np.asarray(idx)[:n_kept])}
    return np.array([pos.get(int(i), -1) for i in ids])


class Workload:
    """A seeded head + keep mask + hidden states, with the oracle's results."""

    def __init__(self, seed_head, V, K, n_kept, forced, seed_keep, W=None):
        self.V, self.K = V, K
        self.W = syn.head_bf16(seed_head, V, K) if W is None else W
        self.keep = syn.keep_mask(seed_keep, V, n_kept, forced)
        self.idx, self.n_kept = oracle.build_index(self.keep)
        self.N = self.idx.size
        self._nv = None
        self._f8 = None

    def nvfp4(self):
        if self._nv is None:
            self._nv = oracle.nvfp4_quantize(self.W, self.idx)
        return self._nv

    def fp8(self):
        if self._f8 is None:
            self._f8 = oracle.fp8_quantize(self.W, self.idx)
        return self._f8


def pack_reference(q, sf):
    """Tile-major layout of DH_FMT_NVFP4_PACKED written out with numpy: per
    (16-row tile, 128-k window), the 16 rows' 64 code bytes, then their scale
    bytes ordered [g][t][h][e] for tile row 8 h + g and window block 2 t + e
    (g < 8, t < 4, h < 2, e < 2)."""
    N, Kh = q.shape
    nwin = 2 * Kh // 128
    codes = q.reshape(N // 16, 16, nwin, 64).transpose(0, 2, 1, 3).reshape(N // 16, nwin, 1024)
    scales = sf.reshape(N // 16, 2, 8, nwin, 4, 2).transpose(0, 3, 2, 4, 1, 5).reshape(N // 16, nwin, 128)
    return np.concatenate([codes, scales], axis=2)


def plant_near_ties(q, sf, g, h_bits, n_kept, frac, seed, max_tries=8):
    """Move a fraction of hidden rows so that their top-2 oracle logits (over the
    kept rows) are within 1e-3. Each try takes the current top-2 rows a, b and
    shifts one hidden element k by (gap - target) / (w'_a[k] - w'_b[k]), with
    the target gap drawn from U(1e-4, 9e-4); k is the element with the smallest
    |w'_a[k] - w'_b[k]| that keeps the shift within 2, so that rounding the new
    value to BF16 moves the gap little. Returns (h_bits, planted rows, gaps)."""
    rng = np.random.default_rng(seed)
    h = h_bits.copy()
    M = h.shape[0]
    chosen = rng.choice(M, size=max(1, int(round(frac * M))), replace=False)
    planted, gaps = [], []
    for m in chosen:
        for _ in range(max_tries):
            y, _ = oracle.gemv(oracle.FMT_NVFP4, q, sf, g, h[m:m + 1], want_abs=False)
            order = np.argsort(-y[0, :n_kept], kind="stable")
            a, b = int(order[0]), int(order[1])
            gap = y[0, a] - y[0, b]
            if gap < 1e-3:
                planted.append(int(m))
                gaps.append(float(gap))
                break
            wab = oracle.dequant_nvfp4(q[[a, b]], sf[[a, b]], g)
            d = wab[0] - wab[1]
            move = gap - rng.uniform(1e-4, 9e-4)
            ok = np.abs(d) >= move / 2.0
            if not ok.any():
                break
            k = int(np.argmin(np.where(ok, np.abs(d), np.inf)))
            x = syn.bf16_bits_to_f32(h[m]).astype(np.float64)
            x[k] -= move / d[k]
            h[m] = syn.f32_to_bf16_bits(x.astype(np.float32))
    return h, planted, gaps

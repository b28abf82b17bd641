"""The packed NVFP4 layout that the GPU parity tests expect (parity_util.pack_reference)
against the rule include/drafthead.h states for nvfp4_pack_head, written out byte by
byte: for each 16-row tile and 128-wide k-window w, the rows' code bytes 64w..64w+63
row by row, then for lane 4 g + t (g < 8, t < 4) the scales of blocks 8w + 2t and
8w + 2t + 1 of tile row g, then of tile row g + 8."""
import numpy as np

from parity_util import pack_reference


def rule_packed(q, sf):
    N, Kh = q.shape
    K = 2 * Kh
    nwin = K // 128
    out = bytearray()
    for tile in range(N // 16):
        for w in range(nwin):
            for r in range(16):
                out += bytes(q[16 * tile + r, 64 * w:64 * w + 64])
            for g in range(8):
                for t in range(4):
                    for row in (16 * tile + g, 16 * tile + g + 8):
                        out += bytes([sf[row, 8 * w + 2 * t], sf[row, 8 * w + 2 * t + 1]])
    return np.frombuffer(bytes(out), dtype=np.uint8).reshape(N // 16, nwin, 1152)


def test_pack_reference_follows_the_documented_rule():
    rng = np.random.default_rng(11)
    for N, K in ((16, 128), (48, 512), (32, 2560)):
        q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
        sf = rng.integers(0, 256, (N, K // 16), dtype=np.uint8)
        assert np.array_equal(pack_reference(q, sf), rule_packed(q, sf)), (N, K)


def test_pack_reference_is_a_permutation():
    rng = np.random.default_rng(12)
    N, K = 32, 1024
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sf = rng.integers(0, 256, (N, K // 16), dtype=np.uint8)
    p = pack_reference(q, sf)
    assert p.size == q.size + sf.size
    assert np.array_equal(np.sort(p, axis=None), np.sort(np.concatenate([q.ravel(), sf.ravel()])))

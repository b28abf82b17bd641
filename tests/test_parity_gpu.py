"""GPU path vs the CPU oracle, element by element, through the C ABI.

Bit-exact: quantised codes, block scales, global / per-tensor scales, dh_idx,
ids (up to near-ties) and the -inf layout of compute_logits. Logits: within
2e-3 * sum|w' h| + 1e-5 of the oracle's fp64 value."""
import numpy as np
import pytest
import torch

import nvfp4_draft_head_gb300 as dh
import oracle
import synthetic as syn
from parity_util import (Workload, check_argmax_rows, check_logits, ids_to_rows, pack_reference,  # noqa: F401
                         plant_near_ties)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from nvfp4_draft_head_gb300 import build
    build.build()
    dh.lib()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return dev(bits.view(np.int16)).view(torch.bfloat16)


@pytest.fixture(scope="module")
def tiny():
    c = syn.TINY
    return Workload(syn.SEED_HEAD_TINY, c["V"], c["K"], c["n_kept"], c["forced"], syn.SEED_KEEP_TINY)


def gpu_nvfp4(wl, packed=False, ascending=None):
    """NVFP4 head on the GPU; by default the packed head declares its dh_idx
    ascending (argmax keys carry ids, dh_idx staged in shared memory) and the
    canonical one does not, so both code paths of the draft step run."""
    W = dev_bf16(wl.W)
    idx = dev(wl.idx)
    q, sf, g = dh.nvfp4_quantize_rows(W, idx)
    asc = packed if ascending is None else ascending
    if packed:
        qp = dh.nvfp4_pack_head(q, sf)
        return dh.DraftHead(dh.DH_FMT_NVFP4_PACKED, wl.V, qp, idx, wl.n_kept, scale=g, idx_ascending=asc), (q, sf, g)
    return dh.DraftHead(dh.DH_FMT_NVFP4, wl.V, q, idx, wl.n_kept, sf=sf, scale=g, idx_ascending=asc), (q, sf, g)


def gpu_fp8(wl, ascending=True):
    W = dev_bf16(wl.W)
    idx = dev(wl.idx)
    q, s = dh.fp8_quantize_rows(W, idx)
    return dh.DraftHead(dh.DH_FMT_FP8, wl.V, q, idx, wl.n_kept, scale=s, idx_ascending=ascending), (q, s)


def run_step(head, h_bits, fmt, q_or, sf_or, s_or, idx, n_kept, V, what):
    """top_tokens + compute_logits for one batch of hidden rows, both checked."""
    y, A = oracle.gemv(fmt, q_or, sf_or, s_or, h_bits)
    return check_step(head, h_bits, y, A, idx, n_kept, V, what)


def run_step_w8a8(head, h_bits, q_or, s_or, idx, n_kept, V, what):
    """The same for the W8A8 FP8 head: the oracle quantises h per token itself."""
    qx, sx = oracle.fp8_act_quantize(h_bits)
    y, A = oracle.gemv_w8a8(q_or, s_or, qx, sx)
    return check_step(head, h_bits, y, A, idx, n_kept, V, what)


def check_step(head, h_bits, y, A, idx, n_kept, V, what):
    """Run top_tokens + compute_logits on the GPU and check them against the
    oracle's logits y (and tolerance scales A) of every head row."""
    h = dev_bf16(h_bits)
    M = h_bits.shape[0]
    top = torch.empty(M, dtype=torch.float32, device="cuda")
    ids = head.top_tokens(h, top=top).cpu().numpy()
    out = head.compute_logits(h).cpu().numpy()
    assert head.device_error() == 0
    rows = ids_to_rows(ids, idx, n_kept) if idx is not None else ids
    exact = check_argmax_rows(rows, y, A, n_kept, what)
    check_logits(top.cpu().numpy()[:, None], y[np.arange(M), rows][:, None],
                 A[np.arange(M), rows][:, None], what + " top logit")
    ref = oracle.scatter_logits(y, idx if idx is not None else np.arange(y.shape[1], dtype=np.int32),
                                n_kept, V)
    assert np.array_equal(np.isneginf(out), np.isneginf(ref)), what + " -inf layout"
    fin = np.isfinite(ref)
    assert np.isfinite(out[fin]).all()
    kept_ids = (idx if idx is not None else np.arange(n_kept))[:n_kept]
    rel = check_logits(out[:, kept_ids], y[:, :n_kept], A[:, :n_kept], what + " logits")
    return exact, rel


# ------------------------------------------------------------------ tiny ----

def test_tiny_nvfp4_quantize_bit_exact(tiny):
    _, (q, sf, g) = gpu_nvfp4(tiny)
    q_o, sf_o, g_o = tiny.nvfp4()
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(sf.cpu().numpy(), sf_o)
    assert g.cpu().numpy()[0] == g_o


def crafted_encoder_head():
    """A 64 x 256 BF16 head whose NVFP4 quantisation meets every E2M1 decision.
    Row 0 starts with 2688 (global amax, so g = 1 exactly); 181 blocks hold a
    block maximum of 6 (block scale E4M3(1) = 1, so each quotient is the value
    itself) and 15 values from a sweep of every BF16 value with magnitude in
    [2^-8, 6.375] of both signs: every rounding midpoint (0.25 ... 5), the
    values next to them, saturation (6 < x <= 6.375), plus signed zeros.
    Remaining blocks are random."""
    K, N = 256, 64
    mags = []
    for e in range(-8, 3):
        for m in range(128):
            v = np.float32((1 + m / 128) * 2.0 ** e)
            if v <= 6.375:
                mags.append(v)
    mags = np.array(mags, np.float32)
    sweep = np.concatenate([mags, -mags, np.float32([0.0, -0.0, 2.0 ** -12, -(2.0 ** -12)])])
    W = syn.bf16_bits_to_f32(syn.head_bf16(31, N, K)).reshape(N, K // 16, 16)
    W[0, 0, 0] = 2688.0
    vals = iter(sweep)
    blk = 1
    done = False
    while not done:
        r, b = divmod(blk, K // 16)
        W[r, b, 0] = 6.0
        for j in range(1, 16):
            v = next(vals, None)
            if v is None:
                done = True
                W[r, b, j:] = 0.5
                break
            W[r, b, j] = v
        blk += 1
    return syn.f32_to_bf16_bits(W.reshape(N, K))


def test_nvfp4_encoder_midpoints_signs_and_saturation():
    Wb = crafted_encoder_head()
    idx = np.arange(Wb.shape[0], dtype=np.int32)
    q, sf, g = dh.nvfp4_quantize_rows(dev_bf16(Wb), dev(idx))
    q_o, sf_o, g_o = oracle.nvfp4_quantize(Wb, idx)
    assert g_o == 1.0 and g.cpu().numpy()[0] == g_o
    assert np.array_equal(sf.cpu().numpy(), sf_o)
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != q_o)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first (row, byte) {bad[:4].tolist()}"
    # the sweep's blocks really decode with scale 1 (so the quotients are the values)
    assert (sf_o.reshape(-1)[1:150] == 0x38).all()


def test_tiny_fp8_quantize_bit_exact(tiny):
    _, (q, s) = gpu_fp8(tiny)
    q_o, s_o = tiny.fp8()
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert s.cpu().numpy()[0] == s_o


def test_tiny_pack_bit_exact(tiny):
    head, (q, sf, g) = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, _ = tiny.nvfp4()
    assert np.array_equal(head.q.cpu().numpy(), pack_reference(q_o, sf_o))


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 13, 16])
def test_tiny_nvfp4_step(tiny, M, packed):
    head, _ = gpu_nvfp4(tiny, packed)
    q_o, sf_o, g_o = tiny.nvfp4()
    for step in range(3):
        h = syn.hidden_bf16(syn.hidden_seed(0, 100 * M + step), M, tiny.K)
        run_step(head, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, tiny.idx, tiny.n_kept, tiny.V,
                 f"tiny nvfp4 packed={packed} M={M} step={step}")


@pytest.mark.parametrize("ascending", [False, True])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_tiny_fp8_step(tiny, M, ascending):
    head, _ = gpu_fp8(tiny, ascending)
    q_o, s_o = tiny.fp8()
    h = syn.hidden_bf16(syn.hidden_seed(0, 500 + M), M, tiny.K)
    run_step(head, h, oracle.FMT_FP8, q_o, None, s_o, tiny.idx, tiny.n_kept, tiny.V,
             f"tiny fp8 M={M} ascending={ascending}")


def special_act_rows(K):
    """Hidden rows that exercise the per-token quantiser's edges: all zeros (the
    1e-12 clamp), one huge value among small ones (codes flushed towards zero,
    subnormal E4M3 codes), every value equal (all codes 448), values at BF16's
    range ends, alternating signs."""
    rows = np.zeros((6, K), np.uint16)
    r1 = syn.hidden_bf16(21, 1, K)[0].copy()
    r1[7] = syn.f32_to_bf16_bits(np.float32([3.0e5]))[0]
    rows[1] = r1
    rows[2] = syn.f32_to_bf16_bits(np.full(K, -0.8125, np.float32))
    big = np.where(np.arange(K) % 3 == 0, 1.0e30, -2.5e-30).astype(np.float32)
    rows[3] = syn.f32_to_bf16_bits(big)
    rows[4] = syn.f32_to_bf16_bits(np.where(np.arange(K) % 2 == 0, 1.0, -1.0).astype(np.float32))
    rows[5] = syn.hidden_bf16(22, 1, K)[0]
    return rows


def test_tiny_fp8_act_quantize_bit_exact(tiny):
    for M, seed in ((1, 31), (5, 32), (16, 33), (37, 34)):
        h = syn.hidden_bf16(seed, M, tiny.K)
        qx, sx = dh.fp8_quantize_activations(dev_bf16(h))
        qx_o, sx_o = oracle.fp8_act_quantize(h)
        assert np.array_equal(qx.cpu().numpy(), qx_o), f"codes M={M}"
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32)), f"scales M={M}"
    for K in (tiny.K, 2560, 16, 4112):
        h = special_act_rows(K)
        qx, sx = dh.fp8_quantize_activations(dev_bf16(h))
        qx_o, sx_o = oracle.fp8_act_quantize(h)
        assert np.array_equal(qx.cpu().numpy(), qx_o), f"special rows K={K}"
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))


@pytest.mark.parametrize("M", [1, 2, 4, 7, 16])
def test_tiny_w8a8_step(tiny, M):
    _, (q, s) = gpu_fp8(tiny)
    head = dh.DraftHead(dh.DH_FMT_FP8_W8A8, tiny.V, q, dev(tiny.idx), tiny.n_kept, scale=s, idx_ascending=M != 7)
    q_o, s_o = tiny.fp8()
    for step in range(2):
        h = syn.hidden_bf16(syn.hidden_seed(0, 600 + 10 * M + step), M, tiny.K)
        run_step_w8a8(head, h, q_o, s_o, tiny.idx, tiny.n_kept, tiny.V, f"tiny w8a8 M={M} step={step}")


def test_w8a8_special_rows_and_sizes(tiny):
    """Quantiser edge rows through the fused W8A8 step, and the other hidden
    sizes (K = 2560: 20 windows over 20 warps; K = 5120: two windows per warp)."""
    _, (q, s) = gpu_fp8(tiny)
    head = dh.DraftHead(dh.DH_FMT_FP8_W8A8, tiny.V, q, dev(tiny.idx), tiny.n_kept, scale=s, idx_ascending=True)
    q_o, s_o = tiny.fp8()
    run_step_w8a8(head, special_act_rows(tiny.K), q_o, s_o, tiny.idx, tiny.n_kept, tiny.V, "w8a8 special rows")
    for V, K, n_kept in ((3000, 5120, 700), (2000, 2560, 129)):
        wl = Workload(177 + K, V, K, n_kept, 5, 188 + n_kept)
        _, (q2, s2) = gpu_fp8(wl)
        q2_o, s2_o = wl.fp8()
        head2 = dh.DraftHead(dh.DH_FMT_FP8_W8A8, V, q2, dev(wl.idx), wl.n_kept, scale=s2, idx_ascending=True)
        for M in (1, 9):
            run_step_w8a8(head2, syn.hidden_bf16(990 + M + K, M, K), q2_o, s2_o, wl.idx, wl.n_kept, V,
                          f"w8a8 V={V} K={K} M={M}")
        run_step_w8a8(head2, special_act_rows(K), q2_o, s2_o, wl.idx, wl.n_kept, V, f"w8a8 special K={K}")


@pytest.mark.parametrize("M", [1, 2, 16])
def test_tiny_bf16_full_head_step(tiny, M):
    W = dev_bf16(tiny.W)
    head = dh.bf16_full_head(W)
    h = syn.hidden_bf16(syn.hidden_seed(0, 700 + M), M, tiny.K)
    run_step(head, h, oracle.FMT_BF16, tiny.W, None, None, None, tiny.V, tiny.V, f"tiny bf16 M={M}")


@pytest.mark.parametrize("N,K", [(128, 256), (192, 512), (1024, 1024), (640, 2048), (1024, 2560),
                                 (320, 4096), (2560, 5120)])
def test_nvfp4_linear(N, K):
    """An MTP-block linear y = x W'^T (NVFP4 W4A16, fp32 out) at every supported
    input width; N = 2560, K = 5120 is the fc projection of a 2560-wide block."""
    W = syn.head_bf16(4000 + K, N, K)
    lin = dh.NVFP4Linear(dev_bf16(W))
    idx = np.arange(N, dtype=np.int32)
    q_o, sf_o, g_o = oracle.nvfp4_quantize(W, idx)
    assert np.array_equal(lin.q.cpu().numpy(), q_o) and np.array_equal(lin.sf.cpu().numpy(), sf_o)
    assert np.array_equal(lin.packed.cpu().numpy(), pack_reference(q_o, sf_o))
    for M in (1, 2, 3, 16):  # 2 and 3 drafts: the ring kernels' per-window reads at K >= 4096
        x = syn.hidden_bf16(4100 + M + K, M, K)
        y = lin(dev_bf16(x)).cpu().numpy()
        assert lin.device_error() == 0
        y_o, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, x)
        check_logits(y, y_o, A, f"linear N={N} K={K} M={M}")


@pytest.mark.parametrize("K", [4096, 5120])
def test_k_split_over_cta_pairs(K):
    """5 to 16 drafts at K = 4,096 / 5,120, where each tile's K range is split
    over the two CTAs of a cluster: 388 tiles, so a pair takes more tiles than
    it has exchange slots, and the last round of tiles is ragged. At K = 5,120
    also a packed head in top-tokens mode (only the first CTA of a pair holds
    argmax keys)."""
    N = 6208
    W = syn.head_bf16(4200 + K, N, K)
    lin = dh.NVFP4Linear(dev_bf16(W))
    q_o, sf_o, g_o = oracle.nvfp4_quantize(W, np.arange(N, dtype=np.int32))
    for M in (6, 8, 16):
        x = syn.hidden_bf16(4300 + M + K, M, K)
        y = lin(dev_bf16(x)).cpu().numpy()
        assert lin.device_error() == 0
        y_o, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, x)
        check_logits(y, y_o, A, f"split linear K={K} M={M}")
    if K == 5120:
        wl = Workload(4400, 9000, K, 6100, 7, 4401)
        headp, _ = gpu_nvfp4(wl, packed=True)
        q_w, sf_w, g_w = wl.nvfp4()
        for M in (7, 16):
            run_step(headp, syn.hidden_bf16(4500 + M, M, K), oracle.FMT_NVFP4, q_w, sf_w, g_w, wl.idx, wl.n_kept,
                     wl.V, f"split head M={M}")


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "w8a8", "bf16"])
def test_k_split_formats(fmt):
    """The canonical NVFP4, FP8 (W8A16 and W8A8) and BF16 heads at K = 5,120,
    where every draft count splits K over a CTA pair (W8A8: the per-token
    activation scale is the max over both halves), plus 16 drafts at K =
    2,560 (one tile in flight; BF16 h fragments in shared memory). 376 tiles:
    a pair takes more tiles than it has exchange slots."""
    for K, Ms in ((5120, (1, 2, 4, 8, 16)), (2560, (16,))):
        wl = Workload(4600 + K, 8000, K, 6000, 9, 4601 + K)
        if fmt == "nvfp4":
            head, _ = gpu_nvfp4(wl)
            q_o, sf_o, g_o = wl.nvfp4()
            ref = lambda h: oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, h)
        elif fmt in ("fp8", "w8a8"):
            head, (q, s) = gpu_fp8(wl)
            q_o, s_o = wl.fp8()
            if fmt == "w8a8":
                head = dh.DraftHead(dh.DH_FMT_FP8_W8A8, wl.V, q, dev(wl.idx), wl.n_kept, scale=s, idx_ascending=True)

                def ref(h):
                    qx, sx = oracle.fp8_act_quantize(h)
                    return oracle.gemv_w8a8(q_o, s_o, qx, sx)
            else:
                ref = lambda h: oracle.gemv(oracle.FMT_FP8, q_o, None, s_o, h)
        else:
            head = dh.bf16_full_head(dev_bf16(wl.W))
            ref = lambda h: oracle.gemv(oracle.FMT_BF16, wl.W, None, None, h)
        idx = None if fmt == "bf16" else wl.idx
        n_kept = wl.V if fmt == "bf16" else wl.n_kept
        for M in Ms:
            h = syn.hidden_bf16(4700 + M + K, M, K)
            y, A = ref(h)
            check_step(head, h, y, A, idx, n_kept, wl.V, f"{fmt} K={K} M={M}")


@pytest.mark.parametrize("n_rows,M", [(4096, 1), (4096, 5), (64, 2), (16_384, 16)])
def test_tiny_bf16_truncated_head_step(tiny, n_rows, M):
    """The truncated BF16 draft head (the first n_rows ids of the target head):
    argmax over those rows, -inf beyond them in compute_logits."""
    head = dh.bf16_truncated_head(dev_bf16(tiny.W), n_rows)
    h = syn.hidden_bf16(syn.hidden_seed(0, 800 + n_rows + M), M, tiny.K)
    W_t = np.ascontiguousarray(tiny.W[:n_rows])
    idx = np.arange(n_rows, dtype=np.int32)
    y, A = oracle.gemv(oracle.FMT_BF16, W_t, None, None, h)
    check_step(head, h, y, A, idx, n_rows, tiny.V, f"tiny bf16 truncated N={n_rows} M={M}")


@pytest.mark.parametrize("V,K,n_kept,forced", [
    (64, 256, 1, 1),          # one kept id: N = 64, 63 padding rows
    (4096, 256, 4096, 0),     # every id kept: a plain full-vocabulary argmax
    (1000, 256, 65, 3),       # ragged: 65 kept -> 128 rows
    (3000, 5120, 700, 10),    # the larger hidden size
    (2000, 2560, 129, 1),     # pages' hidden size, small ragged head
])
def test_edge_shapes(V, K, n_kept, forced):
    wl = Workload(77 + K, V, K, n_kept, forced, 88 + n_kept)
    head, (q, sf, g) = gpu_nvfp4(wl)
    q_o, sf_o, g_o = wl.nvfp4()
    assert np.array_equal(q.cpu().numpy(), q_o) and np.array_equal(sf.cpu().numpy(), sf_o)
    assert g.cpu().numpy()[0] == g_o
    headp, _ = gpu_nvfp4(wl, packed=True)
    assert np.array_equal(headp.q.cpu().numpy(), pack_reference(q_o, sf_o))
    for M in (1, 5):
        h = syn.hidden_bf16(900 + M + K, M, K)
        run_step(head, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, wl.idx, wl.n_kept, V, f"edge V={V} K={K} M={M}")
        run_step(headp, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, wl.idx, wl.n_kept, V,
                 f"edge packed V={V} K={K} M={M}")
    head8, (q8, s8) = gpu_fp8(wl)
    q8_o, s8_o = wl.fp8()
    assert np.array_equal(q8.cpu().numpy(), q8_o) and s8.cpu().numpy()[0] == s8_o
    run_step(head8, syn.hidden_bf16(950 + K, 3, K), oracle.FMT_FP8, q8_o, None, s8_o, wl.idx,
             wl.n_kept, V, f"edge fp8 V={V} K={K}")


def test_special_hidden_states(tiny):
    head, _ = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, g_o = tiny.nvfp4()
    K = tiny.K
    h = np.zeros((4, K), np.uint16)
    h[1, 17] = syn.f32_to_bf16_bits(np.float32([1.0]))[0]          # one-hot: reads one column
    h[2] = syn.f32_to_bf16_bits(np.full(K, 3.0e4, np.float32))      # large values (f16 prescale)
    h[3] = syn.hidden_bf16(5, 1, K)[0]
    h[3, ::2] = 0
    run_step(head, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, tiny.idx, tiny.n_kept, tiny.V, "special h")
    # an all-zero hidden state: every logit is 0, the first kept row (id idx[0]) wins
    ids = head.top_tokens(dev_bf16(h[:1])).cpu().numpy()
    assert ids[0] == tiny.idx[0]


@pytest.mark.parametrize("fmt", ["nvfp4_packed", "nvfp4_canonical", "fp8", "fp8_rowkeys", "w8a8", "bf16_full"])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_exact_ties_resolve_to_the_lowest_id(tiny, fmt, M):
    """Three kept rows in different tiles (and CTAs) carry identical weights that
    dominate every draft's logits, so their quantised codes and logits are
    exactly equal: each draft must return the lowest of the three ids (the
    first maximum, as torch.argmax), whether the argmax keys carry ids or rows."""
    W = tiny.W.copy()
    kept = tiny.idx[: tiny.n_kept]
    dup = [int(kept[3]), int(kept[len(kept) // 2]), int(kept[-2])]
    h = np.repeat(syn.hidden_bf16(syn.hidden_seed(0, 7777), 1, tiny.K), M, axis=0)
    hv = syn.bf16_bits_to_f32(h[0])
    pattern = syn.f32_to_bf16_bits((0.25 * np.sign(hv)).astype(np.float32))
    for i in dup:
        W[i] = pattern
    if fmt == "bf16_full":
        head = dh.bf16_full_head(dev_bf16(W))
        ids = head.top_tokens(dev_bf16(h)).cpu().numpy()
        assert (ids == min(dup)).all(), ids
        return
    idx_d = dev(tiny.idx)
    Wd = dev_bf16(W)
    if fmt.startswith("nvfp4"):
        q, sf, g = dh.nvfp4_quantize_rows(Wd, idx_d)
        if fmt == "nvfp4_packed":
            head = dh.DraftHead(dh.DH_FMT_NVFP4_PACKED, tiny.V, dh.nvfp4_pack_head(q, sf), idx_d, tiny.n_kept,
                                scale=g, idx_ascending=True)
        else:
            head = dh.DraftHead(dh.DH_FMT_NVFP4, tiny.V, q, idx_d, tiny.n_kept, sf=sf, scale=g)
    else:
        q, s8 = dh.fp8_quantize_rows(Wd, idx_d)
        f = dh.DH_FMT_FP8_W8A8 if fmt == "w8a8" else dh.DH_FMT_FP8
        head = dh.DraftHead(f, tiny.V, q, idx_d, tiny.n_kept, scale=s8, idx_ascending=(fmt != "fp8_rowkeys"))
    top = torch.empty(M, dtype=torch.float32, device="cuda")
    ids = head.top_tokens(dev_bf16(h), top=top).cpu().numpy()
    assert head.device_error() == 0
    assert (ids == min(dup)).all(), (fmt, M, ids, dup)
    # compute_logits writes the three equal logits at their own ids
    out = head.compute_logits(dev_bf16(h)).cpu().numpy()
    assert (out[:, dup[0]] == out[:, dup[1]]).all() and (out[:, dup[1]] == out[:, dup[2]]).all()
    assert np.allclose(out[:, dup[0]], top.cpu().numpy())


def test_same_hidden_rows_agree(tiny):
    head, _ = gpu_nvfp4(tiny)
    h = np.repeat(syn.hidden_bf16(11, 1, tiny.K), 6, axis=0)
    top = torch.empty(6, device="cuda")
    ids = head.top_tokens(dev_bf16(h), top=top).cpu().numpy()
    assert len(set(ids.tolist())) == 1 and len(set(top.cpu().numpy().tolist())) == 1
    out = head.compute_logits(dev_bf16(h)).cpu().numpy()
    assert all(np.array_equal(out[0], out[i]) for i in range(6))


def test_cuda_graph_replay(tiny):
    head, _ = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, g_o = tiny.nvfp4()
    M = 2
    h_static = torch.empty((M, tiny.K), dtype=torch.bfloat16, device="cuda")
    ids_static = torch.empty(M, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        head.top_tokens(h_static.zero_(), ids=ids_static)    # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        head.top_tokens(h_static, ids=ids_static)
    for step in range(5):
        hb = syn.hidden_bf16(syn.hidden_seed(0, 9000 + step), M, tiny.K)
        h_static.copy_(dev_bf16(hb))
        graph.replay()
        ids = ids_static.cpu().numpy()
        y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
        check_argmax_rows(ids_to_rows(ids, tiny.idx, tiny.n_kept), y, A, tiny.n_kept, f"graph {step}")
        eager = head.top_tokens(dev_bf16(hb)).cpu().numpy()
        assert np.array_equal(ids, eager)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_point(tiny, pinned):
    """draft_head_top_tokens_host: hidden rows and ids in host memory, one call
    per step. Several steps are enqueued back to back (each reuses the staging
    area after the previous step's draft step, in stream order) before one
    synchronise; ids equal the device entry point's and meet the oracle."""
    head, _ = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, g_o = tiny.nvfp4()
    steps = [(M, syn.hidden_bf16(syn.hidden_seed(0, 9500 + i), M, tiny.K)) for i, M in enumerate((1, 5, 16, 2))]
    outs = []
    for M, hb in steps:
        h = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16)
        h = h.pin_memory() if pinned else h
        ids = torch.full((M,), -7, dtype=torch.int32, pin_memory=pinned)
        top = torch.full((M,), np.nan, dtype=torch.float32, pin_memory=pinned)
        outs.append((head.top_tokens_host(h, ids, top), top))
    torch.cuda.synchronize()
    assert head.device_error() == 0
    for (M, hb), (ids, top) in zip(steps, outs):
        ids = ids.numpy()
        assert np.array_equal(ids, head.top_tokens(dev_bf16(hb)).cpu().numpy())
        y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
        rows = ids_to_rows(ids, tiny.idx, tiny.n_kept)
        check_argmax_rows(rows, y, A, tiny.n_kept, f"host entry M={M}")
        check_logits(top.numpy()[:, None], y[np.arange(M), rows][:, None], A[np.arange(M), rows][:, None],
                     f"host entry M={M} top logit")
    # the W8A8 head through the same entry point
    W = dev_bf16(tiny.W)
    h8 = dh.fp8_head(W, tiny.keep, w8a8=True)
    hb = syn.hidden_bf16(syn.hidden_seed(0, 9600), 3, tiny.K)
    ids = h8.top_tokens_host(torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16))
    torch.cuda.synchronize()
    assert np.array_equal(ids.numpy(), h8.top_tokens(dev_bf16(hb)).cpu().numpy())
    with pytest.raises(ValueError):
        head.top_tokens_host(dev_bf16(hb))                 # a device tensor is refused


def test_host_buffer_entry_point_in_a_cuda_graph(tiny):
    """Under stream capture the host-buffer entry point copies h_host in stream
    order, so every replay reads the pinned buffer's current contents."""
    head, _ = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, g_o = tiny.nvfp4()
    M = 3
    h_pin = torch.zeros((M, tiny.K), dtype=torch.bfloat16).pin_memory()
    ids_pin = torch.full((M,), -7, dtype=torch.int32).pin_memory()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        head.top_tokens_host(h_pin, ids_pin)                 # warm-up outside capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        head.top_tokens_host(h_pin, ids_pin, stream=s)
    for step in range(3):
        hb = syn.hidden_bf16(syn.hidden_seed(0, 9700 + step), M, tiny.K)
        h_pin.copy_(torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        ids = ids_pin.numpy().copy()
        assert np.array_equal(ids, head.top_tokens(dev_bf16(hb)).cpu().numpy()), step
        y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
        check_argmax_rows(ids_to_rows(ids, tiny.idx, tiny.n_kept), y, A, tiny.n_kept, f"host graph {step}")


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_waits_give_up_and_report(tiny, kind):
    """A wait for an event that never happens (a workspace word nothing writes;
    an mbarrier nothing arrives on) gives up after its limit, sets the timeout
    bit in the error word and leaves the context usable: the next draft step on
    the same workspace is correct and reports no error."""
    head, _ = gpu_nvfp4(tiny, packed=True)
    dh.draft_head_wait_probe(head.ws, kind, 1 << 14 if kind == 0 else 1 << 11)
    assert head.device_error() == dh.DH_DEVERR_TIMEOUT
    assert head.device_error() == 0
    q_o, sf_o, g_o = tiny.nvfp4()
    h = syn.hidden_bf16(syn.hidden_seed(0, 4242 + kind), 2, tiny.K)
    run_step(head, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, tiny.idx, tiny.n_kept, tiny.V, f"after probe {kind}")


@pytest.mark.parametrize("M", [1, 3, 16])
def test_tiny_back_to_back_compute_logits(tiny, M):
    """Consecutive compute_logits steps into one output buffer (each step's
    -inf fill starts early and must wait for the step before it), eager and
    as one CUDA graph: the buffer ends bitwise equal to one step on the last
    hidden state, which meets the oracle's tolerance."""
    head, _ = gpu_nvfp4(tiny, packed=True)
    hb = [syn.hidden_bf16(syn.hidden_seed(0, 9200 + 10 * M + i), M, tiny.K) for i in range(6)]
    hs = [dev_bf16(x) for x in hb]
    want = head.compute_logits(hs[-1])
    y_o, A = oracle.gemv(oracle.FMT_NVFP4, *tiny.nvfp4(), hb[-1])
    kept = tiny.idx[: tiny.n_kept]
    got = want.cpu().numpy()
    check_logits(got[:, kept], y_o[:, : tiny.n_kept], A[:, : tiny.n_kept], f"back to back M={M}")
    assert np.isneginf(np.delete(got, kept, axis=1)).all()
    out = torch.empty((M, tiny.V), dtype=torch.float32, device="cuda")
    for h in hs:
        head.compute_logits(h, out=out)
    assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        head.compute_logits(hs[0], out=out)               # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for h in hs:
            head.compute_logits(h, out=out)
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    assert head.device_error() == 0


@pytest.mark.parametrize("path", ["nvfp4_logits", "w8a8_top", "w8a8_logits", "linear"])
def test_cuda_graph_replay_other_paths(tiny, path):
    """compute_logits (fill kernel + GEMV), the W8A8 step and the MTP-block linear
    are captured once and replayed with fresh inputs: each replay equals the
    eager call and stays within the oracle's tolerance."""
    M = 3
    if path == "linear":
        N, K = 256, 512
        W = syn.head_bf16(4321, N, K)
        lin = dh.NVFP4Linear(dev_bf16(W))
        q_o, sf_o, g_o = oracle.nvfp4_quantize(W, np.arange(N, dtype=np.int32))
        run = lambda x, y: lin(x, y=y)
        out_shape, kdim = (M, N), K
    else:
        if path == "nvfp4_logits":
            head, _ = gpu_nvfp4(tiny, packed=True)
        else:
            _, (q8, s8) = gpu_fp8(tiny)
            head = dh.DraftHead(dh.DH_FMT_FP8_W8A8, tiny.V, q8, dev(tiny.idx), tiny.n_kept, scale=s8,
                                idx_ascending=True)
        if path.endswith("logits"):
            run = lambda x, y: head.compute_logits(x, out=y)
            out_shape = (M, tiny.V)
        else:
            run = lambda x, y: head.top_tokens(x, ids=y)
            out_shape = (M,)
        kdim = tiny.K
    x_static = torch.zeros((M, kdim), dtype=torch.bfloat16, device="cuda")
    dtype = torch.int32 if path == "w8a8_top" else torch.float32
    y_static = torch.empty(out_shape, dtype=dtype, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(x_static, y_static)                            # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(x_static, y_static)
    for step in range(3):
        hb = syn.hidden_bf16(syn.hidden_seed(0, 9100 + 10 * step), M, kdim)
        x_static.copy_(dev_bf16(hb))
        graph.replay()
        got = y_static.cpu().numpy().copy()
        eager = run(dev_bf16(hb), torch.empty_like(y_static)).cpu().numpy()
        assert np.array_equal(got, eager), (path, step)
        if path == "linear":
            y_o, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
            check_logits(got, y_o, A, f"graph linear {step}")
        elif path == "w8a8_top":
            qx, sx = oracle.fp8_act_quantize(hb)
            y_o, A = oracle.gemv_w8a8(*tiny.fp8(), qx, sx)
            check_argmax_rows(ids_to_rows(got, tiny.idx, tiny.n_kept), y_o, A, tiny.n_kept, f"graph w8a8 {step}")
        else:
            if path == "w8a8_logits":
                qx, sx = oracle.fp8_act_quantize(hb)
                y_o, A = oracle.gemv_w8a8(*tiny.fp8(), qx, sx)
            else:
                y_o, A = oracle.gemv(oracle.FMT_NVFP4, *tiny.nvfp4(), hb)
            kept = tiny.idx[: tiny.n_kept]
            check_logits(got[:, kept], y_o[:, : tiny.n_kept], A[:, : tiny.n_kept], f"graph {path} {step}")
            assert np.isneginf(np.delete(got, kept, axis=1)).all()


def test_out_of_range_idx_sets_the_error_word(tiny):
    head, (q, sf, g) = gpu_nvfp4(tiny)
    bad = tiny.idx.copy()
    bad[5] = tiny.V            # one kept row points past the vocabulary
    idx_bad = dev(bad)
    head_bad = dh.DraftHead(dh.DH_FMT_NVFP4, tiny.V, q, idx_bad, tiny.n_kept, sf=sf, scale=g)
    head_bad_asc = dh.DraftHead(dh.DH_FMT_NVFP4, tiny.V, q, idx_bad, tiny.n_kept, sf=sf, scale=g,
                                idx_ascending=True)
    h = dev_bf16(syn.hidden_bf16(3, 1, tiny.K))
    head_bad.compute_logits(h)
    assert head_bad.device_error() == dh.DH_DEVERR_IDX
    assert head_bad.device_error() == 0                        # reading clears it
    head_bad_asc.compute_logits(h)                             # ids staged in shared memory too
    assert head_bad_asc.device_error() == dh.DH_DEVERR_IDX
    with pytest.raises(RuntimeError, match="device error"):
        dh.nvfp4_quantize_rows(dev_bf16(tiny.W), idx_bad)


def test_late_argmax_key_never_reaches_a_later_step(tiny):
    """A key stored after its step's collector gave up waiting lands in that
    step's slot bank, and the step marks the bank dirty. Simulated here by
    writing huge keys over the whole previous bank and the dirty word: the next
    steps (which alternate banks) return the oracle's ids, the next one zeroes
    the dirty bank and clears the mark, and the epoch advances once per step."""
    head, _ = gpu_nvfp4(tiny, packed=True)
    q_o, sf_o, g_o = tiny.nvfp4()
    M = 3
    h0 = syn.hidden_bf16(syn.hidden_seed(0, 8100), M, tiny.K)
    head.top_tokens(dev_bf16(h0))
    torch.cuda.synchronize()
    hdr = head.ws[:256].view(torch.int32)
    slots = head.ws[256:256 + 2 * 16 * 1024 * 8].view(torch.int64).view(2, 16, 1024)
    epoch = int(hdr[2].item())
    prev = (epoch - 1) & 1
    slots[prev].fill_(0x7FFFFFFFFFFFFFFF)
    hdr[3] = 1 | (prev << 1) | (16 << 2) | (1024 << 8)
    torch.cuda.synchronize()
    for step in range(4):
        hb = syn.hidden_bf16(syn.hidden_seed(0, 8101 + step), M, tiny.K)
        ids = head.top_tokens(dev_bf16(hb)).cpu().numpy()
        y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
        check_argmax_rows(ids_to_rows(ids, tiny.idx, tiny.n_kept), y, A, tiny.n_kept, f"late key, step {step}")
        if step == 0:
            assert int(hdr[3].item()) == 0
            assert int(slots[prev].abs().sum().item()) == 0
    assert int(hdr[2].item()) == epoch + 4
    assert head.device_error() == 0

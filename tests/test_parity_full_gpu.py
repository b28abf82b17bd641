"""Parity at the pages' full sizes (V = 248,320, K = 2560), GPU vs oracle:
  * the 64,064-row NVFP4 head: gather + quantise bit-exact, draft steps at
    M = 1 (fresh hidden states, the launch configuration the benchmark times),
    and through the host-buffer entry point;
  * the batch sweep M in {1, 2, 4, 8, 16} with planted near-ties (top-2 oracle
    gap < 1e-3 in 5 % of rows), both get_top_tokens and compute_logits;
  * the 98,304-row FP8 head: quantise bit-exact, M = 1 and 4, both paths,
    W8A16 and W8A8 (per-token FP8 hidden states);
  * the full-vocabulary BF16 head (the stock drafter read) at M = 1;
  * the truncated 40,960-row BF16 head (the FP8 page's draft_lm_head).
The oracle computes every output here (its fp64 GEMV over a whole head takes
about a second per draft row on one core)."""
import numpy as np
import pytest
import torch

import nvfp4_draft_head_gb300 as dh
import oracle
import synthetic as syn
from parity_util import Workload, check_argmax_rows, check_logits, ids_to_rows, plant_near_ties
from test_parity_gpu import check_step, dev, dev_bf16, pack_reference, run_step, run_step_w8a8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from nvfp4_draft_head_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def W_full():
    c = syn.QWEN_64K
    return syn.head_bf16(syn.SEED_HEAD_QWEN, c["V"], c["K"])


@pytest.fixture(scope="module")
def W_dev(W_full):
    return dev_bf16(W_full)


@pytest.fixture(scope="module")
def qwen64k(W_full):
    c = syn.QWEN_64K
    return Workload(syn.SEED_HEAD_QWEN, c["V"], c["K"], c["n_kept"], c["forced"], syn.SEED_KEEP_64K, W=W_full)


@pytest.fixture(scope="module")
def canon64k(qwen64k, W_dev):
    idx = dev(qwen64k.idx)
    q, sf, g = dh.nvfp4_quantize_rows(W_dev, idx)
    return dh.DraftHead(dh.DH_FMT_NVFP4, qwen64k.V, q, idx, qwen64k.n_kept, sf=sf, scale=g)


@pytest.fixture(scope="module")
def head64k(qwen64k, canon64k):
    """The packed head the benchmark times."""
    qp = dh.nvfp4_pack_head(canon64k.q, canon64k.sf)
    return dh.DraftHead(dh.DH_FMT_NVFP4_PACKED, qwen64k.V, qp, canon64k.idx, qwen64k.n_kept, scale=canon64k.scale,
                        idx_ascending=True)


def test_qwen64k_index_quantize_and_pack_bit_exact(qwen64k, canon64k, head64k):
    assert (qwen64k.n_kept, qwen64k.N) == (64_026, 64_064)
    q_o, sf_o, g_o = qwen64k.nvfp4()
    assert np.array_equal(canon64k.q.cpu().numpy(), q_o)
    assert np.array_equal(canon64k.sf.cpu().numpy(), sf_o)
    assert canon64k.scale.cpu().numpy()[0] == g_o
    assert np.array_equal(head64k.q.cpu().numpy(), pack_reference(q_o, sf_o))
    idx_abi, nk = dh.draft_head_build_index(qwen64k.keep)
    assert nk == qwen64k.n_kept and np.array_equal(idx_abi, qwen64k.idx)


def test_qwen64k_m1_steps(qwen64k, head64k, canon64k):
    q_o, sf_o, g_o = qwen64k.nvfp4()
    for step in range(6):
        h = syn.hidden_bf16(syn.hidden_seed(1, step), 1, qwen64k.K)
        run_step(head64k, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, qwen64k.idx, qwen64k.n_kept, qwen64k.V,
                 f"qwen64k M=1 step {step}")
        if step < 2:
            run_step(canon64k, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, qwen64k.idx, qwen64k.n_kept, qwen64k.V,
                     f"qwen64k canonical M=1 step {step}")


def test_qwen64k_host_buffer_entry_point(qwen64k, head64k):
    """draft_head_top_tokens_host on the benchmark's head, from one to sixteen
    drafts: ids equal the device entry point's; M = 1 and 5 are also checked
    against the oracle."""
    q_o, sf_o, g_o = qwen64k.nvfp4()
    for M in (1, 4, 5, 16):
        hb = syn.hidden_bf16(syn.hidden_seed(4, M), M, qwen64k.K)
        h_pin = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).pin_memory()
        top = torch.empty(M, dtype=torch.float32).pin_memory()
        ids = head64k.top_tokens_host(h_pin, top=top)
        torch.cuda.synchronize()
        ids = ids.numpy()
        assert np.array_equal(ids, head64k.top_tokens(dev_bf16(hb)).cpu().numpy()), M
        if M in (1, 5):
            y, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
            rows = ids_to_rows(ids, qwen64k.idx, qwen64k.n_kept)
            check_argmax_rows(rows, y, A, qwen64k.n_kept, f"host entry qwen64k M={M}")
            check_logits(top.numpy()[:, None], y[np.arange(M), rows][:, None], A[np.arange(M), rows][:, None],
                         f"host entry qwen64k M={M} top logit")
    assert head64k.device_error() == 0


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_batch_sweep_with_near_ties(qwen64k, head64k, M):
    q_o, sf_o, g_o = qwen64k.nvfp4()
    steps = 2 if M >= 8 else 4
    planted_total = 0
    for step in range(steps):
        h = syn.hidden_bf16(syn.hidden_seed(3, 1000 * M + step), M, qwen64k.K)
        if step == 0:
            h, planted, gaps = plant_near_ties(q_o, sf_o, g_o, h, qwen64k.n_kept, 0.05, seed=M)
            planted_total += len(planted)
            assert all(gp < 1e-3 for gp in gaps)
        run_step(head64k, h, oracle.FMT_NVFP4, q_o, sf_o, g_o, qwen64k.idx, qwen64k.n_kept, qwen64k.V,
                 f"sweep M={M} step {step}")
    assert planted_total >= 1


@pytest.mark.parametrize("M", [1, 4, 16])
def test_back_to_back_compute_logits_into_one_buffer(qwen64k, head64k, M):
    """Consecutive compute_logits steps write one output buffer; each step's
    -inf fill starts while the step before it finishes and must not write
    before it has completed. Six steps with different hidden states, eager
    and as one CUDA graph, end bitwise equal to a single step on the last."""
    hs = [dev_bf16(syn.hidden_bf16(syn.hidden_seed(4, 100 * M + i), M, qwen64k.K)) for i in range(6)]
    want = head64k.compute_logits(hs[-1])
    out = torch.empty((M, qwen64k.V), dtype=torch.float32, device="cuda")
    for h in hs:
        head64k.compute_logits(h, out=out)
    assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        head64k.compute_logits(hs[0], out=out)            # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for h in hs:
            head64k.compute_logits(h, out=out)
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    assert head64k.device_error() == 0


def test_fp8_98k_head(W_full, W_dev):
    c = syn.FP8_98K
    wl = Workload(syn.SEED_HEAD_QWEN, c["V"], c["K"], c["n_kept"], c["forced"], syn.SEED_KEEP_98K, W=W_full)
    assert wl.N == 98_304
    idx = dev(wl.idx)
    q, s = dh.fp8_quantize_rows(W_dev, idx)
    q_o, s_o = wl.fp8()
    assert np.array_equal(q.cpu().numpy(), q_o) and s.cpu().numpy()[0] == s_o
    head = dh.DraftHead(dh.DH_FMT_FP8, wl.V, q, idx, wl.n_kept, scale=s, idx_ascending=True)
    for M in (1, 4):
        h = syn.hidden_bf16(syn.hidden_seed(2, M), M, wl.K)
        run_step(head, h, oracle.FMT_FP8, q_o, None, s_o, wl.idx, wl.n_kept, wl.V, f"fp8 98k M={M}")
    # the same head run W8A8: hidden states quantised per token inside the step
    w8a8 = dh.DraftHead(dh.DH_FMT_FP8_W8A8, wl.V, q, idx, wl.n_kept, scale=s, idx_ascending=True)
    for M in (1, 4):
        h = syn.hidden_bf16(syn.hidden_seed(2, 10 + M), M, wl.K)
        run_step_w8a8(w8a8, h, q_o, s_o, wl.idx, wl.n_kept, wl.V, f"fp8 w8a8 98k M={M}")


def test_bf16_truncated_40960_head(W_full, W_dev):
    """The FP8 page's truncated 40,960-row BF16 draft_lm_head, read in place
    from the target head, M = 1 and 4, both paths."""
    head = dh.bf16_truncated_head(W_dev, 40_960)
    W_t = np.ascontiguousarray(W_full[:40_960])
    idx = np.arange(40_960, dtype=np.int32)
    for M in (1, 4):
        h = syn.hidden_bf16(syn.hidden_seed(5, M), M, W_full.shape[1])
        y, A = oracle.gemv(oracle.FMT_BF16, W_t, None, None, h)
        check_step(head, h, y, A, idx, 40_960, W_full.shape[0], f"bf16 truncated 40,960 M={M}")


def test_bf16_full_vocabulary_head(W_full, W_dev):
    head = dh.bf16_full_head(W_dev)
    for step in range(2):
        h = syn.hidden_bf16(syn.hidden_seed(4, step), 1, W_full.shape[1])
        ids = head.top_tokens(dev_bf16(h)).cpu().numpy()
        y, A = oracle.gemv(oracle.FMT_BF16, W_full, None, None, h)
        check_argmax_rows(ids, y, A, W_full.shape[0], f"bf16 full step {step}")

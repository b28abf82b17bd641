"""draft_head_top_tokens_static, the draft step for callers that cannot
allocate device memory (plugin hooks handed only their inputs and outputs,
serving loops that forbid cudaMalloc because it can synchronise the device).

It is called through the C ABI and compared with draft_head_top_tokens (the
entry point that takes a caller workspace) on two calls in a row: the same ids,
and top logits within the parity tolerance (2e-3 * sum|w' h| + 1e-5, with the
sum from the oracle). This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_draft_head_gb300 as dh
import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu


def test_static_scratch_entry_point_matches_workspace_entry_point():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from nvfp4_draft_head_gb300 import build
    build.build()
    L = dh.lib()
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    head = dh.nvfp4_head(Wd, keep)
    q_o, sf_o, g_o = oracle.nvfp4_quantize(W, oracle.build_index(keep)[0])
    stream = torch.cuda.current_stream().cuda_stream
    for call, M in enumerate((3, 16)):                      # two calls in a row
        hb = syn.hidden_bf16(syn.hidden_seed(0, 7000 + call), M, c["K"])
        h = torch.from_numpy(hb.view(np.int16)).cuda().view(torch.bfloat16)
        ids_ws = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        top_ws = torch.empty(M, dtype=torch.float32, device="cuda")
        st = L.draft_head_top_tokens(C.byref(head.desc), h.data_ptr(), M, ids_ws.data_ptr(),
                                     top_ws.data_ptr(), head.ws.data_ptr(), head.ws_bytes, stream)
        assert st == dh.DH_OK
        ids_st = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        top_st = torch.empty(M, dtype=torch.float32, device="cuda")
        st = L.draft_head_top_tokens_static(C.byref(head.desc), h.data_ptr(), M, ids_st.data_ptr(),
                                            top_st.data_ptr(), stream)
        assert st == dh.DH_OK
        torch.cuda.synchronize()
        a, b = ids_ws.cpu().numpy(), ids_st.cpu().numpy()
        assert np.array_equal(a, b), (call, a, b)
        _, A = oracle.gemv(oracle.FMT_NVFP4, q_o, sf_o, g_o, hb)
        rows = np.array([int(np.nonzero(head.idx.cpu().numpy()[: head.n_kept] == i)[0][0]) for i in a])
        bound = 2e-3 * A[np.arange(M), rows] + 1e-5
        assert np.all(np.abs(top_ws.cpu().numpy() - top_st.cpu().numpy()) <= bound)
    # more drafts than the fixed scratch holds is refused before any launch
    h17 = torch.zeros((17, c["K"]), dtype=torch.bfloat16, device="cuda")
    ids17 = torch.empty(17, dtype=torch.int32, device="cuda")
    assert L.draft_head_top_tokens_static(C.byref(head.desc), h17.data_ptr(), 17, ids17.data_ptr(),
                                          None, stream) == dh.DH_ERR_SHAPE


def test_static_scratch_entry_point_runs_the_w8a8_head():
    """The same comparison for the W8A8 FP8 head (hidden states quantised per
    token inside the step), which shares the draft-step kernel family."""
    from nvfp4_draft_head_gb300 import build
    build.build()
    L = dh.lib()
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    head = dh.fp8_head(Wd, keep, w8a8=True)
    stream = torch.cuda.current_stream().cuda_stream
    for call, M in enumerate((1, 7)):
        hb = syn.hidden_bf16(syn.hidden_seed(0, 7100 + call), M, c["K"])
        h = torch.from_numpy(hb.view(np.int16)).cuda().view(torch.bfloat16)
        ids_ws = head.top_tokens(h)
        ids_st = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        assert L.draft_head_top_tokens_static(C.byref(head.desc), h.data_ptr(), M, ids_st.data_ptr(),
                                              None, stream) == dh.DH_OK
        torch.cuda.synchronize()
        assert np.array_equal(ids_ws.cpu().numpy(), ids_st.cpu().numpy()), call


def test_static_scratch_reports_a_timed_out_wait_and_runs_on():
    """A bounded wait that runs out on the static scratch (the self-test probe,
    as a draft step whose wait ran out) sets its error word, which
    draft_head_static_read_device_error reads and clears; the next static
    draft step still matches the workspace entry point."""
    from nvfp4_draft_head_gb300 import build
    build.build()
    L = dh.lib()
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    head = dh.nvfp4_head(Wd, keep)
    stream = torch.cuda.current_stream().cuda_stream
    assert dh.draft_head_static_read_device_error() == 0
    for kind, rounds in ((0, 1 << 14), (1, 1 << 11)):
        dh.draft_head_wait_probe(None, kind, rounds)
        assert dh.draft_head_static_read_device_error() == dh.DH_DEVERR_TIMEOUT, kind
        assert dh.draft_head_static_read_device_error() == 0
        M = 4
        hb = syn.hidden_bf16(syn.hidden_seed(0, 7200 + kind), M, c["K"])
        h = torch.from_numpy(hb.view(np.int16)).cuda().view(torch.bfloat16)
        ids_st = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        assert L.draft_head_top_tokens_static(C.byref(head.desc), h.data_ptr(), M, ids_st.data_ptr(),
                                              None, stream) == dh.DH_OK
        assert np.array_equal(head.top_tokens(h).cpu().numpy(), ids_st.cpu().numpy()), kind
        assert dh.draft_head_static_read_device_error() == 0

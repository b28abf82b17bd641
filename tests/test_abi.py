"""The C-ABI library on the host: it builds, loads, exports every function
include/drafthead.h declares, and rejects bad arguments before any launch
(these calls return before touching CUDA, so they run without a GPU)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import nvfp4_draft_head_gb300 as dh
import oracle
import synthetic as syn

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "drafthead.h")


@pytest.fixture(scope="module")
def L():
    from nvfp4_draft_head_gb300 import build
    build.build()
    return dh.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(dh.EXPORTS)


def test_library_has_no_process_wide_unique_symbols(L):
    """Function-local statics of the launch templates (per-device caches) must
    stay private to each loaded copy of the library (built with
    -fno-gnu-unique), or a second copy would skip its own kernel set-up."""
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", dh.library_path()], capture_output=True, text=True).stdout
    unique = [ln for ln in out.splitlines() if " u " in ln]
    assert unique == [], unique[:3]


def test_last_cuda_error_starts_clear(L):
    name = C.c_char_p()
    assert L.draft_head_last_cuda_error(C.byref(name)) == 0
    assert name.value == b"cudaSuccess"
    assert L.draft_head_last_cuda_error(None) == 0


def test_status_strings_and_version(L):
    assert L.draft_head_abi_version() == 1
    for st in range(8):
        assert L.draft_head_status_string(st)
    assert L.draft_head_status_string(0) == b"ok"


def test_build_index_matches_oracle(L):
    rng = np.random.default_rng(3)
    for trial in range(30):
        V = int(rng.integers(1, 3000))
        keep = (rng.random(V) < rng.uniform(0.001, 1.0)).astype(np.uint8)
        if not keep.any():
            keep[rng.integers(V)] = 1
        idx, nk = dh.draft_head_build_index(keep)
        idx_o, nk_o = oracle.build_index(keep)
        assert nk == nk_o and np.array_equal(idx, idx_o)
    keep = syn.keep_mask(syn.SEED_KEEP_64K, **{k: syn.QWEN_64K[k] for k in ("V", "n_kept", "forced")})
    idx, nk = dh.draft_head_build_index(keep)
    assert (nk, idx.size) == (64_026, 64_064)


def test_build_index_errors(L):
    with pytest.raises(dh.DraftHeadError) as e:
        dh.draft_head_build_index(np.zeros(10, np.uint8))
    assert e.value.status == dh.DH_ERR_ARG
    keep = np.ones(100, np.uint8)
    idx = np.empty(100, np.int32)
    nk, N = C.c_int(), C.c_int()
    assert L.draft_head_build_index(keep.ctypes.data, 100, idx.ctypes.data, 100, C.byref(nk), C.byref(N)) \
        == dh.DH_ERR_SHAPE   # 100 kept -> 128 rows do not fit in cap = 100
    assert L.draft_head_build_index(None, 100, idx.ctypes.data, 100, C.byref(nk), C.byref(N)) == dh.DH_ERR_ARG


def _desc(**kw):
    d = dict(fmt=dh.DH_FMT_NVFP4, V=16384, K=256, N=4032, n_kept=4000, q=0x10000, sf=0x20000,
             scale=0x30000, idx=0x40000)
    d.update(kw)
    return dh.dh_head_t(d["fmt"], d["V"], d["K"], d["N"], d["n_kept"], d["q"], d["sf"], d["scale"], d["idx"], 0)


WS = 0x100000   # a fake, never dereferenced, 256-aligned device address
H = 0x200000


@pytest.mark.parametrize("kw,M,status", [
    (dict(fmt=9), 1, dh.DH_ERR_ARG),
    (dict(q=None), 1, dh.DH_ERR_ARG),
    (dict(sf=None), 1, dh.DH_ERR_ARG),
    (dict(scale=None), 1, dh.DH_ERR_ARG),
    (dict(K=300), 1, dh.DH_ERR_SHAPE),        # hidden size without a compiled kernel
    (dict(N=4000), 1, dh.DH_ERR_SHAPE),       # N % 64 != 0
    (dict(n_kept=0), 1, dh.DH_ERR_SHAPE),
    (dict(n_kept=5000), 1, dh.DH_ERR_SHAPE),  # n_kept > N
    (dict(), 0, dh.DH_ERR_SHAPE),             # M < 1
    (dict(), 17, dh.DH_ERR_SHAPE),            # M > 16
    (dict(q=0x10008), 1, dh.DH_ERR_ALIGN),
    (dict(sf=0x20004), 1, dh.DH_ERR_ALIGN),
    (dict(idx=None), 1, dh.DH_ERR_ARG),       # only a BF16 full head may omit dh_idx
    (dict(fmt=dh.DH_FMT_BF16, idx=None, n_kept=4032, N=4032, V=4000), 1, dh.DH_ERR_SHAPE),
])
def test_top_tokens_rejects_bad_arguments(L, kw, M, status):
    d = _desc(**kw)
    st = L.draft_head_top_tokens(C.byref(d), H, M, 0x300000, None, WS, 256, None)
    assert st == status
    # the static-scratch and host-buffer entry points apply the same checks before any CUDA call
    assert L.draft_head_top_tokens_static(C.byref(d), H, M, 0x300000, None, None) == status
    assert L.draft_head_top_tokens_host(C.byref(d), H, M, 0x300000, None, WS, 1 << 30, None) == status


def test_host_entry_point_checks(L):
    d = _desc()
    need = L.draft_head_workspace_bytes(C.byref(d), 4)
    # staging for 4 rows of K = 256 BF16 values (2 KB) and the ids / top logits
    assert need == L.draft_head_workspace_bytes(None, 16) + 2048 + 256
    assert L.draft_head_workspace_bytes(C.byref(d), 16) == L.draft_head_workspace_bytes(None, 16) + 8192 + 256
    assert L.draft_head_workspace_bytes(C.byref(d), 64) == L.draft_head_workspace_bytes(C.byref(d), 16)
    assert L.draft_head_top_tokens_host(C.byref(d), None, 4, 0x300000, None, WS, need, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens_host(C.byref(d), H, 4, None, None, WS, need, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens_host(None, H, 4, 0x300000, None, WS, need, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens_host(C.byref(d), H, 4, 0x300000, None, None, need, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens_host(C.byref(d), H, 4, 0x300000, None, WS + 16, need, None) == dh.DH_ERR_WORKSPACE
    # host buffers carry no alignment rule: a workspace one byte short is the first error
    assert L.draft_head_top_tokens_host(C.byref(d), H + 2, 4, 0x300001, 0x400003, WS, need - 1,
                                        None) == dh.DH_ERR_WORKSPACE
    # the draft-step part alone has no room for the staging area
    assert L.draft_head_top_tokens_host(C.byref(d), H, 1, 0x300000, None, WS,
                                        L.draft_head_workspace_bytes(None, 16), None) == dh.DH_ERR_WORKSPACE


def test_static_entry_point_pointer_checks(L):
    d = _desc()
    assert L.draft_head_top_tokens_static(C.byref(d), H, 1, None, None, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens_static(C.byref(d), H, 1, 0x300002, None, None) == dh.DH_ERR_ALIGN
    assert L.draft_head_top_tokens_static(C.byref(d), H, 1, 0x300000, 0x400001, None) == dh.DH_ERR_ALIGN
    assert L.draft_head_top_tokens_static(C.byref(d), H + 8, 1, 0x300000, None, None) == dh.DH_ERR_ALIGN
    assert L.draft_head_top_tokens_static(None, H, 1, 0x300000, None, None) == dh.DH_ERR_ARG


def test_workspace_and_pointer_checks(L):
    d = _desc()
    assert L.draft_head_top_tokens(C.byref(d), H, 1, 0x300000, None, WS, 128, None) == dh.DH_ERR_WORKSPACE
    assert L.draft_head_top_tokens(C.byref(d), H, 1, 0x300000, None, WS + 16, 256, None) == dh.DH_ERR_WORKSPACE
    assert L.draft_head_top_tokens(C.byref(d), H, 1, 0x300000, None, None, 256, None) == dh.DH_ERR_ARG
    assert L.draft_head_top_tokens(C.byref(d), H + 8, 1, 0x300000, None, WS, 256, None) == dh.DH_ERR_ALIGN
    assert L.draft_head_top_tokens(C.byref(d), H, 1, None, None, WS, 256, None) == dh.DH_ERR_ARG
    assert L.draft_head_compute_logits(C.byref(d), H, 1, 0x400008, WS, 256, None) == dh.DH_ERR_ALIGN
    assert L.draft_head_compute_logits(C.byref(d), None, 1, 0x400000, WS, 256, None) == dh.DH_ERR_ARG
    assert L.draft_head_workspace_bytes(C.byref(d), 16) % 256 == 0
    assert L.draft_head_quantize_workspace_bytes() % 256 == 0


@pytest.mark.parametrize("args,status", [
    (dict(K=24), dh.DH_ERR_SHAPE),     # K % 16 != 0
    (dict(N=100), dh.DH_ERR_SHAPE),    # N % 64 != 0
    (dict(V=0), dh.DH_ERR_SHAPE),
    (dict(W=0x10002), dh.DH_ERR_ALIGN),
    (dict(q=0x30004), dh.DH_ERR_ALIGN),
    (dict(W=None), dh.DH_ERR_ARG),
    (dict(ws=0x100010), dh.DH_ERR_WORKSPACE),
    (dict(ws_bytes=16), dh.DH_ERR_WORKSPACE),
])
def test_quantize_rejects_bad_arguments(L, args, status):
    a = dict(W=0x10000, V=16384, K=256, idx=0x20000, N=4032, q=0x30000, sf=0x40000, g=0x50000,
             ws=0x100000, ws_bytes=256)
    a.update(args)
    st = L.nvfp4_quantize_rows(a["W"], a["V"], a["K"], a["idx"], a["N"], a["q"], a["sf"], a["g"],
                               a["ws"], a["ws_bytes"], None)
    assert st == status
    st8 = L.fp8_quantize_rows(a["W"], a["V"], a["K"], a["idx"], a["N"], a["q"], a["g"], a["ws"],
                              a["ws_bytes"], None)
    assert st8 == status


@pytest.mark.parametrize("args,status", [
    (dict(h=None), dh.DH_ERR_ARG),
    (dict(qx=None), dh.DH_ERR_ARG),
    (dict(sx=None), dh.DH_ERR_ARG),
    (dict(M=0), dh.DH_ERR_SHAPE),
    (dict(K=24), dh.DH_ERR_SHAPE),     # K % 16 != 0
    (dict(K=0), dh.DH_ERR_SHAPE),
    (dict(h=0x10008), dh.DH_ERR_ALIGN),
    (dict(qx=0x20004), dh.DH_ERR_ALIGN),
    (dict(sx=0x30002), dh.DH_ERR_ALIGN),
])
def test_activation_quantize_rejects_bad_arguments(L, args, status):
    a = dict(h=0x10000, M=4, K=2560, qx=0x20000, sx=0x30000)
    a.update(args)
    assert L.fp8_quantize_activations(a["h"], a["M"], a["K"], a["qx"], a["sx"], None) == status


@pytest.mark.parametrize("kw,M,status", [
    (dict(), 0, dh.DH_ERR_SHAPE),
    (dict(), 17, dh.DH_ERR_SHAPE),
    (dict(fmt=dh.DH_FMT_NVFP4), 1, dh.DH_ERR_ARG),     # the packed layout only
    (dict(K=384), 1, dh.DH_ERR_SHAPE),                 # no kernel for this input width
    (dict(N=100), 1, dh.DH_ERR_SHAPE),                 # N % 64 != 0
    (dict(scale=None), 1, dh.DH_ERR_ARG),
    (dict(q=0x10008), 1, dh.DH_ERR_ALIGN),
])
def test_linear_rejects_bad_arguments(L, kw, M, status):
    d = _desc(**dict(dict(fmt=dh.DH_FMT_NVFP4_PACKED, sf=None, idx=None, K=1024, N=256), **kw))
    assert L.nvfp4_linear(C.byref(d), H, M, 0x500000, WS, 1 << 20, None) == status
    d = _desc(fmt=dh.DH_FMT_NVFP4_PACKED, sf=None, idx=None, K=1024, N=256)
    assert L.nvfp4_linear(C.byref(d), H, 1, 0x500008, WS, 1 << 20, None) == dh.DH_ERR_ALIGN
    assert L.nvfp4_linear(C.byref(d), H, 1, 0x500000, WS, 64, None) == dh.DH_ERR_WORKSPACE


def test_wait_probe_rejects_bad_arguments(L):
    # NULL selects the static scratch; kind and rounds are checked first
    assert L.draft_head_wait_probe(None, 0, 2, 16, None) == dh.DH_ERR_ARG
    assert L.draft_head_wait_probe(None, 0, 0, 0, None) == dh.DH_ERR_ARG
    assert L.draft_head_wait_probe(WS + 16, 256, 0, 16, None) == dh.DH_ERR_WORKSPACE
    assert L.draft_head_wait_probe(WS, 128, 0, 16, None) == dh.DH_ERR_WORKSPACE
    assert L.draft_head_wait_probe(WS, 256, 2, 16, None) == dh.DH_ERR_ARG
    assert L.draft_head_wait_probe(WS, 256, 0, 0, None) == dh.DH_ERR_ARG
    assert L.draft_head_wait_probe(WS, 256, 1, (1 << 22) + 1, None) == dh.DH_ERR_ARG


def test_w8a8_head_descriptor_checks(L):
    d = _desc(fmt=dh.DH_FMT_FP8_W8A8, sf=None, scale=None)
    assert L.draft_head_top_tokens(C.byref(d), H, 1, 0x300000, None, WS, 256, None) == dh.DH_ERR_ARG
    d = _desc(fmt=dh.DH_FMT_FP8_W8A8, sf=None, K=300)
    assert L.draft_head_top_tokens(C.byref(d), H, 1, 0x300000, None, WS, 256, None) == dh.DH_ERR_SHAPE
    d = _desc(fmt=dh.DH_FMT_FP8_W8A8, sf=None)
    assert L.draft_head_top_tokens(C.byref(d), H, 17, 0x300000, None, WS, 256, None) == dh.DH_ERR_SHAPE


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(dh, "_lib", None)
    monkeypatch.setattr(dh, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dh.lib()

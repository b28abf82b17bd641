"""Python binding of libdrafthead.so (the reduced-vocabulary NVFP4 draft head).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch provides device memory and the current stream. If the compiled
library is missing, every call raises; there is no fallback.

Names follow the C ABI in include/drafthead.h:
  draft_head_build_index   keep mask -> dh_idx (padded to N % 64 == 0)
  nvfp4_quantize_rows      gather + NVFP4 quantisation of W[dh_idx]
  fp8_quantize_rows        gather + per-tensor FP8 E4M3 quantisation
  fp8_quantize_activations per-token FP8 E4M3 codes of hidden states (W8A8)
  DraftHead.top_tokens     get_top_tokens: dh_idx[argmax_n (W_q h)]
  DraftHead.compute_logits compute_logits: -inf row + logits at dh_idx
  NVFP4Linear              nvfp4_linear: an MTP-block linear, y = x W'^T
  DraftHead.top_keys       draft_head_top_keys: a vocabulary shard's argmax keys
  keys_to_ids              draft_head_keys_to_ids: combined keys -> target ids
The vocabulary-sharded head (the local-argmax exchange) is in .sharded.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import build as _build

DH_OK, DH_ERR_ARG, DH_ERR_SHAPE, DH_ERR_ALIGN, DH_ERR_WORKSPACE, DH_ERR_CUDA = 0, 1, 2, 3, 4, 5
DH_FMT_NVFP4, DH_FMT_FP8, DH_FMT_BF16, DH_FMT_NVFP4_PACKED, DH_FMT_FP8_W8A8 = 1, 2, 3, 4, 5
DH_MAX_M = 16
DH_WORKSPACE_ALIGN = 256
DH_DEVERR_IDX = 1
DH_DEVERR_TIMEOUT = 2
DH_HEAD_IDX_ASCENDING = 1

EXPORTS = (
    "draft_head_build_index", "draft_head_quantize_workspace_bytes", "nvfp4_quantize_rows",
    "fp8_quantize_rows", "draft_head_workspace_bytes", "draft_head_workspace_init",
    "draft_head_top_tokens", "draft_head_compute_logits", "draft_head_read_device_error",
    "draft_head_status_string", "draft_head_abi_version", "draft_head_top_tokens_static",
    "nvfp4_pack_head", "fp8_quantize_activations", "draft_head_last_cuda_error", "nvfp4_linear",
    "draft_head_wait_probe", "draft_head_top_tokens_host", "draft_head_top_keys", "draft_head_keys_to_ids",
    "draft_head_static_read_device_error",
)

_lib = None


class DraftHeadError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib().draft_head_status_string(status).decode() if _lib is not None else str(status)
        self.cuda_error = 0
        if status == DH_ERR_CUDA and _lib is not None:
            name = C.c_char_p()
            self.cuda_error = _lib.draft_head_last_cuda_error(C.byref(name))
            msg += f": {name.value.decode() if name.value else self.cuda_error}"
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


class dh_head_t(C.Structure):
    _fields_ = [("fmt", C.c_int), ("V", C.c_int), ("K", C.c_int), ("N", C.c_int),
                ("n_kept", C.c_int), ("q", C.c_void_p), ("sf", C.c_void_p),
                ("scale", C.c_void_p), ("idx", C.c_void_p), ("flags", C.c_uint)]


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load libdrafthead.so (built by ``nvfp4_draft_head_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libdrafthead.so is not built ({path}); run "
                               "`python -m nvfp4_draft_head_gb300.build`")
        L = C.CDLL(path)
        P, I, S = C.c_void_p, C.c_int, C.c_size_t
        L.draft_head_build_index.argtypes = [P, I, P, I, P, P]
        L.draft_head_quantize_workspace_bytes.argtypes = []
        L.draft_head_quantize_workspace_bytes.restype = S
        L.nvfp4_quantize_rows.argtypes = [P, I, I, P, I, P, P, P, P, S, P]
        L.fp8_quantize_rows.argtypes = [P, I, I, P, I, P, P, P, S, P]
        L.draft_head_workspace_bytes.argtypes = [C.POINTER(dh_head_t), I]
        L.draft_head_workspace_bytes.restype = S
        L.draft_head_workspace_init.argtypes = [P, S, P]
        L.draft_head_top_tokens.argtypes = [C.POINTER(dh_head_t), P, I, P, P, P, S, P]
        L.draft_head_top_tokens_host.argtypes = [C.POINTER(dh_head_t), P, I, P, P, P, S, P]
        L.draft_head_compute_logits.argtypes = [C.POINTER(dh_head_t), P, I, P, P, S, P]
        L.draft_head_read_device_error.argtypes = [P, P, P]
        L.draft_head_status_string.argtypes = [I]
        L.draft_head_status_string.restype = C.c_char_p
        L.draft_head_abi_version.argtypes = []
        L.draft_head_top_tokens_static.argtypes = [C.POINTER(dh_head_t), P, I, P, P, P]
        L.nvfp4_pack_head.argtypes = [P, P, I, I, P, P]
        L.fp8_quantize_activations.argtypes = [P, I, I, P, P, P]
        L.draft_head_last_cuda_error.argtypes = [C.POINTER(C.c_char_p)]
        L.nvfp4_linear.argtypes = [C.POINTER(dh_head_t), P, I, P, P, S, P]
        L.draft_head_wait_probe.argtypes = [P, S, I, C.c_uint, P]
        L.draft_head_top_keys.argtypes = [C.POINTER(dh_head_t), P, I, P, P, S, P]
        L.draft_head_keys_to_ids.argtypes = [P, I, P, P, P]
        L.draft_head_static_read_device_error.argtypes = [P, P]
        _lib = L
    return _lib


def _check(fn: str, st: int):
    if st != DH_OK:
        raise DraftHeadError(fn, st)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> int:
    """cudaStream_t of `stream`, or of the current stream (without building a
    Stream object: this runs once per draft step)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _workspace(nbytes: int, device) -> torch.Tensor:
    """Zeroed device buffer whose data pointer is DH_WORKSPACE_ALIGN-aligned."""
    buf = torch.zeros(nbytes + DH_WORKSPACE_ALIGN, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % DH_WORKSPACE_ALIGN
    return buf[off: off + nbytes]


# ---------------------------------------------------------------- head build --

def draft_head_build_index(keep) -> tuple[np.ndarray, int]:
    """(dh_idx int32[N], n_kept) from a host keep mask (numpy or CPU tensor)."""
    keep = np.ascontiguousarray(np.asarray(keep).astype(np.uint8))
    V = keep.size
    idx = np.empty(V + 64, dtype=np.int32)
    nk, N = C.c_int(), C.c_int()
    _check("draft_head_build_index",
           lib().draft_head_build_index(keep.ctypes.data, V, idx.ctypes.data, idx.size,
                                        C.byref(nk), C.byref(N)))
    return idx[: N.value].copy(), nk.value


def _gather_args(W: torch.Tensor, idx: torch.Tensor):
    if W.dtype != torch.bfloat16 or W.dim() != 2 or not W.is_cuda or not W.is_contiguous():
        raise ValueError("W must be a contiguous [V, K] bfloat16 CUDA tensor")
    if idx.dtype != torch.int32 or idx.dim() != 1 or idx.device != W.device:
        raise ValueError("idx must be an int32 vector on W's device")
    return W.shape[0], W.shape[1], idx.numel()


def nvfp4_quantize_rows(W: torch.Tensor, idx: torch.Tensor, stream=None):
    """(q uint8[N, K/2], sf uint8[N, K/16], g float32[1]) of the rows W[idx]."""
    V, K, N = _gather_args(W, idx)
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    sf = torch.empty((N, K // 16), dtype=torch.uint8, device=W.device)
    g = torch.empty(1, dtype=torch.float32, device=W.device)
    nb = lib().draft_head_quantize_workspace_bytes()
    ws = _workspace(nb, W.device)
    _check("nvfp4_quantize_rows",
           lib().nvfp4_quantize_rows(W.data_ptr(), V, K, idx.data_ptr(), N, q.data_ptr(),
                                     sf.data_ptr(), g.data_ptr(), ws.data_ptr(), nb, _stream(stream)))
    _raise_device_error(ws, stream, "nvfp4_quantize_rows")
    return q, sf, g


def fp8_quantize_rows(W: torch.Tensor, idx: torch.Tensor, stream=None):
    """(q uint8[N, K] E4M3 codes, scale float32[1]) of the rows W[idx]."""
    V, K, N = _gather_args(W, idx)
    q = torch.empty((N, K), dtype=torch.uint8, device=W.device)
    s = torch.empty(1, dtype=torch.float32, device=W.device)
    nb = lib().draft_head_quantize_workspace_bytes()
    ws = _workspace(nb, W.device)
    _check("fp8_quantize_rows",
           lib().fp8_quantize_rows(W.data_ptr(), V, K, idx.data_ptr(), N, q.data_ptr(),
                                   s.data_ptr(), ws.data_ptr(), nb, _stream(stream)))
    _raise_device_error(ws, stream, "fp8_quantize_rows")
    return q, s


def nvfp4_pack_head(q: torch.Tensor, sf: torch.Tensor, stream=None) -> torch.Tensor:
    """Tile-major copy of an NVFP4 head (DH_FMT_NVFP4_PACKED): uint8 [N/16, K/128, 1152]."""
    N, Kh = q.shape
    K = 2 * Kh
    if sf.shape != (N, K // 16) or q.dtype != torch.uint8 or sf.dtype != torch.uint8:
        raise ValueError("q must be uint8 [N, K/2] and sf uint8 [N, K/16]")
    packed = torch.empty((N // 16, K // 128, 1152), dtype=torch.uint8, device=q.device)
    _check("nvfp4_pack_head",
           lib().nvfp4_pack_head(q.data_ptr(), sf.data_ptr(), N, K, packed.data_ptr(), _stream(stream)))
    return packed


def fp8_quantize_activations(h: torch.Tensor, stream=None):
    """(qx uint8[M, K] E4M3 codes, sx float32[M] scales): per-token dynamic FP8
    quantisation of BF16 hidden states, as the W8A8 head's draft step does it."""
    if h.dtype != torch.bfloat16 or h.dim() != 2 or not h.is_cuda or not h.is_contiguous():
        raise ValueError("h must be a contiguous [M, K] bfloat16 CUDA tensor")
    M, K = h.shape
    qx = torch.empty((M, K), dtype=torch.uint8, device=h.device)
    sx = torch.empty(M, dtype=torch.float32, device=h.device)
    _check("fp8_quantize_activations",
           lib().fp8_quantize_activations(h.data_ptr(), M, K, qx.data_ptr(), sx.data_ptr(), _stream(stream)))
    return qx, sx


def draft_head_read_device_error(ws: torch.Tensor, stream=None) -> int:
    err = C.c_int()
    _check("draft_head_read_device_error",
           lib().draft_head_read_device_error(ws.data_ptr(), C.byref(err), _stream(stream)))
    return err.value


def draft_head_static_read_device_error(stream=None) -> int:
    """Read and clear the static scratch's device error word (synchronises)."""
    err = C.c_int(0)
    _check("draft_head_static_read_device_error",
           lib().draft_head_static_read_device_error(C.byref(err), _stream(stream)))
    return err.value


def draft_head_wait_probe(ws: torch.Tensor | None, kind: int, rounds: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test on workspace ws, or on the static
    scratch of draft_head_top_tokens_static when ws is None (kind 0: a global
    word nothing writes, 1: an mbarrier nothing arrives on)."""
    _check("draft_head_wait_probe",
           lib().draft_head_wait_probe(_ptr(ws), 0 if ws is None else ws.numel(), kind, rounds,
                                       _stream(stream)))


def _raise_device_error(ws, stream, fn):
    err = draft_head_read_device_error(ws, stream)
    if err:
        raise RuntimeError(f"{fn}: device error word {err:#x} (a dh_idx entry outside [0, V))")


# ---------------------------------------------------------------- draft step --

class DraftHead:
    """A quantised draft head plus its workspace; tensors stay owned by torch.

    fmt: DH_FMT_NVFP4 (q, sf, scale=g), DH_FMT_NVFP4_PACKED (tile-major q, scale=g),
    DH_FMT_FP8 / DH_FMT_FP8_W8A8 (q, scale) or DH_FMT_BF16 (q = the BF16
    weights, idx may be None for a full-vocabulary head).
    """

    def __init__(self, fmt: int, V: int, q: torch.Tensor, idx: torch.Tensor | None, n_kept: int,
                 sf: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                 idx_ascending: bool = False):
        self.fmt, self.V, self.n_kept = fmt, int(V), int(n_kept)
        self.flags = DH_HEAD_IDX_ASCENDING if idx_ascending else 0
        self.q, self.sf, self.scale, self.idx = q, sf, scale, idx
        self.N = q.shape[0]
        if fmt == DH_FMT_NVFP4_PACKED:        # [N/16, K/128, 1152]
            self.N = q.shape[0] * 16
            self.K = q.shape[1] * 128
        elif fmt == DH_FMT_NVFP4:
            self.K = q.shape[1] * 2
        elif fmt in (DH_FMT_FP8, DH_FMT_FP8_W8A8):
            self.K = q.shape[1]
        else:
            self.K = q.shape[1] if q.dtype == torch.bfloat16 else q.shape[1] // 2
        self.desc = dh_head_t(fmt, self.V, self.K, self.N, self.n_kept, _ptr(q), _ptr(sf),
                              _ptr(scale), _ptr(idx), self.flags)
        self.ws_bytes = lib().draft_head_workspace_bytes(C.byref(self.desc), DH_MAX_M)
        self.ws = _workspace(self.ws_bytes, q.device)
        _check("draft_head_workspace_init",
               lib().draft_head_workspace_init(self.ws.data_ptr(), self.ws_bytes, _stream()))

    def with_storage(self, q: torch.Tensor, sf: torch.Tensor | None = None) -> "DraftHead":
        """The same head (same scale, idx, workspace) read from another copy of q / sf."""
        other = object.__new__(DraftHead)
        other.__dict__.update(self.__dict__)
        other.q, other.sf = q, (sf if sf is not None else self.sf)
        other.desc = dh_head_t(self.fmt, self.V, self.K, self.N, self.n_kept, _ptr(other.q),
                               _ptr(other.sf), _ptr(self.scale), _ptr(self.idx), self.flags)
        return other

    def top_tokens(self, h: torch.Tensor, ids: torch.Tensor | None = None,
                   top: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """get_top_tokens: int32[M] target ids of the argmax over kept rows."""
        M = self._check_h(h)
        if ids is None:
            ids = torch.empty(M, dtype=torch.int32, device=h.device)
        _check("draft_head_top_tokens",
               lib().draft_head_top_tokens(C.byref(self.desc), h.data_ptr(), M, ids.data_ptr(),
                                           _ptr(top), self.ws.data_ptr(), self.ws_bytes,
                                           _stream(stream)))
        return ids

    def top_keys(self, h: torch.Tensor, keys: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """This head as one vocabulary shard: int64[M] argmax keys (largest
        logit, then lowest target id) whose maximum over shards is the whole
        head's; needs an ascending dh_idx."""
        M = self._check_h(h)
        if keys is None:
            keys = torch.empty(M, dtype=torch.int64, device=h.device)
        _check("draft_head_top_keys",
               lib().draft_head_top_keys(C.byref(self.desc), h.data_ptr(), M, keys.data_ptr(),
                                         self.ws.data_ptr(), self.ws_bytes, _stream(stream)))
        return keys

    def top_tokens_host(self, h: torch.Tensor, ids: torch.Tensor | None = None,
                        top: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """get_top_tokens on host tensors: h a CPU bfloat16 [M, K] tensor; ids
        (returned) a CPU int32 [M] tensor; top an optional CPU float32 [M] tensor.
        One C call enqueues the copy of h to the device, the draft step and the
        copies back; the results are valid once the stream synchronises. Pinned
        tensors keep the copies asynchronous."""
        if h.device.type != "cpu":
            raise ValueError("h must be a host (CPU) tensor")
        M = self._check_h(h)
        if ids is None:
            ids = torch.empty(M, dtype=torch.int32, pin_memory=h.is_pinned())
        elif ids.device.type != "cpu" or ids.dtype != torch.int32 or ids.numel() != M or not ids.is_contiguous():
            raise ValueError(f"ids must be a contiguous CPU torch.int32 tensor of {M} elements")
        if top is not None and (top.device.type != "cpu" or top.dtype != torch.float32 or top.numel() != M
                                or not top.is_contiguous()):
            raise ValueError(f"top must be a contiguous CPU torch.float32 tensor of {M} elements")
        _check("draft_head_top_tokens_host",
               lib().draft_head_top_tokens_host(C.byref(self.desc), h.data_ptr(), M, ids.data_ptr(),
                                                _ptr(top), self.ws.data_ptr(), self.ws_bytes,
                                                _stream(stream)))
        return ids

    def compute_logits(self, h: torch.Tensor, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
        """compute_logits: float32[M, V], -inf outside the kept ids."""
        M = self._check_h(h)
        if out is None:
            out = torch.empty((M, self.V), dtype=torch.float32, device=h.device)
        _check("draft_head_compute_logits",
               lib().draft_head_compute_logits(C.byref(self.desc), h.data_ptr(), M, out.data_ptr(),
                                               self.ws.data_ptr(), self.ws_bytes, _stream(stream)))
        return out

    def device_error(self, stream=None) -> int:
        return draft_head_read_device_error(self.ws, stream)

    def _check_h(self, h: torch.Tensor) -> int:
        if h.dtype != torch.bfloat16 or h.dim() != 2 or h.shape[1] != self.K or not h.is_contiguous():
            raise ValueError(f"h must be a contiguous [M, {self.K}] bfloat16 tensor")
        return h.shape[0]


def keys_to_ids(keys: torch.Tensor, ids: torch.Tensor | None = None, top: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Target ids (and, into `top`, the winning logits) of argmax keys."""
    M = keys.numel()
    if keys.dtype != torch.int64 or not keys.is_contiguous():
        raise ValueError("keys must be a contiguous int64 tensor")
    if ids is None:
        ids = torch.empty(M, dtype=torch.int32, device=keys.device)
    _check("draft_head_keys_to_ids",
           lib().draft_head_keys_to_ids(keys.data_ptr(), M, ids.data_ptr(), _ptr(top), _stream(stream)))
    return ids


def nvfp4_head(W: torch.Tensor, keep, packed: bool = True, stream=None) -> DraftHead:
    """Build an NVFP4 draft head from a BF16 target head and a host keep mask
    (repacked tile-major unless packed=False)."""
    idx_np, nk = draft_head_build_index(keep)
    idx = torch.from_numpy(idx_np).to(W.device)
    q, sf, g = nvfp4_quantize_rows(W, idx, stream)
    if packed and (W.shape[1] % 128 == 0):
        qp = nvfp4_pack_head(q, sf, stream)
        return DraftHead(DH_FMT_NVFP4_PACKED, W.shape[0], qp, idx, nk, scale=g, idx_ascending=True)
    return DraftHead(DH_FMT_NVFP4, W.shape[0], q, idx, nk, sf=sf, scale=g, idx_ascending=True)


def fp8_head(W: torch.Tensor, keep, w8a8: bool = False, stream=None) -> DraftHead:
    """Build a per-tensor FP8 draft head from a BF16 target head and a host keep
    mask: W8A16 (BF16 hidden states), or W8A8 (per-token FP8 hidden states)."""
    idx_np, nk = draft_head_build_index(keep)
    idx = torch.from_numpy(idx_np).to(W.device)
    q, s = fp8_quantize_rows(W, idx, stream)
    return DraftHead(DH_FMT_FP8_W8A8 if w8a8 else DH_FMT_FP8, W.shape[0], q, idx, nk, scale=s,
                     idx_ascending=True)


class NVFP4Linear:
    """An NVFP4 W4A16 linear layer (an MTP-block linear): weight W [N, K] BF16
    quantised with the head's recipe and repacked tile-major; forward(x) =
    x W'^T in fp32. N % 64 == 0."""

    def __init__(self, W: torch.Tensor, stream=None):
        N, K = W.shape
        idx = torch.arange(N, dtype=torch.int32, device=W.device)
        q, sf, g = nvfp4_quantize_rows(W, idx, stream)
        self.q, self.sf, self.g = q, sf, g
        self.packed = nvfp4_pack_head(q, sf, stream)
        self.N, self.K = N, K
        self.desc = dh_head_t(DH_FMT_NVFP4_PACKED, N, K, N, N, _ptr(self.packed), None, _ptr(g), None, 0)
        self.ws_bytes = lib().draft_head_workspace_bytes(C.byref(self.desc), DH_MAX_M)
        self.ws = _workspace(self.ws_bytes, W.device)

    def with_storage(self, packed: torch.Tensor) -> "NVFP4Linear":
        """The same layer read from another copy of its packed bytes."""
        other = object.__new__(NVFP4Linear)
        other.__dict__.update(self.__dict__)
        other.packed = packed
        other.desc = dh_head_t(DH_FMT_NVFP4_PACKED, self.N, self.K, self.N, self.N, _ptr(packed), None,
                               _ptr(self.g), None, 0)
        return other

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError(f"x must be a contiguous [M, {self.K}] bfloat16 tensor")
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.N), dtype=torch.float32, device=x.device)
        _check("nvfp4_linear",
               lib().nvfp4_linear(C.byref(self.desc), x.data_ptr(), M, y.data_ptr(), self.ws.data_ptr(),
                                  self.ws_bytes, _stream(stream)))
        return y

    __call__ = forward

    def device_error(self, stream=None) -> int:
        return draft_head_read_device_error(self.ws, stream)


def bf16_full_head(W: torch.Tensor) -> DraftHead:
    """The stock full-vocabulary BF16 head (the row is the id)."""
    return DraftHead(DH_FMT_BF16, W.shape[0], W, None, W.shape[0])


def bf16_truncated_head(W: torch.Tensor, n_rows: int) -> DraftHead:
    """A truncated BF16 draft head: the first n_rows rows of the target head
    (ids 0 .. n_rows-1, n_rows % 64 == 0), read in place; compute_logits still
    writes full-vocabulary rows (-inf past n_rows)."""
    if n_rows % 64 or not 0 < n_rows <= W.shape[0]:
        raise ValueError("n_rows must be a multiple of 64 within the head")
    return DraftHead(DH_FMT_BF16, W.shape[0], W[:n_rows], None, n_rows)

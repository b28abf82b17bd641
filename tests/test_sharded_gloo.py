"""The vocabulary-sharded head's host side on CPU ranks (gloo): the row split,
the local-argmax key exchange checked against the oracle's unsharded argmax
(ties across the shard boundary included), and a rank that leaves between
steps. The shards' keys are formed here from the oracle's logits with the key
definition of draft_head_top_keys (include/drafthead.h); the GPU tests check
that the kernels produce exactly those keys."""
import os
import socket
import time
from datetime import timedelta

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import oracle
import synthetic as syn
from nvfp4_draft_head_gb300 import sharded


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def ordered32(y):
    """The header's ord(): fp32 -> uint32 preserving order (-0 as +0, NaN on top)."""
    f = np.asarray(y, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = np.where(f == 0, 0, u)
    out = np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000)
    return np.where(np.isnan(f), 0xFFFFFFFF, out).astype(np.uint64)


def shard_keys(y, ids):
    """Keys of one shard: y [M][rows] logits, ids [rows] target ids (ascending)."""
    y32 = np.asarray(y, dtype=np.float32)
    keys = (ordered32(y32) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ids.astype(np.uint64))[None, :]
    best = keys.max(axis=1)
    return (best ^ np.uint64(1 << 63)).view(np.int64)


def decode(keys):
    k = keys.view(np.uint64) ^ np.uint64(1 << 63)
    return (np.uint64(0xFFFFFFFF) - (k & np.uint64(0xFFFFFFFF))).astype(np.int64)


def expected_ids(y, ids):
    """Unsharded: the lowest id among the rows with the largest fp32 logit."""
    y32 = np.asarray(y, dtype=np.float32)
    out = []
    for row in y32:
        best = row.max()
        out.append(int(ids[np.flatnonzero(row == best)].min()))
    return np.array(out)


def tiny_with_cross_shard_ties(world):
    """The tiny workload with two pairs of identical dominating rows, each pair
    split over two shards (the lower id in the lower shard)."""
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    kept = np.flatnonzero(keep)
    lo1, _ = sharded.shard_rows(kept.size, 1, world)
    pairs = [(int(kept[lo1 - 3]), int(kept[lo1 + 2])), (int(kept[5]), int(kept[-4]))]
    h = syn.hidden_bf16(syn.hidden_seed(0, 4242), 4, c["K"])
    hv = syn.bf16_bits_to_f32(h[0])
    pat = syn.f32_to_bf16_bits((0.25 * np.sign(hv)).astype(np.float32))
    for a, b in pairs[:1]:
        W[a] = pat
        W[b] = pat
    # draft 1 is dominated by the second pair
    hv1 = syn.bf16_bits_to_f32(h[1])
    pat1 = syn.f32_to_bf16_bits((0.25 * np.sign(hv1)).astype(np.float32))
    for a, b in pairs[1:]:
        W[a] = pat1
        W[b] = pat1
    return W, keep, h, pairs


def test_shard_rows_partition_the_kept_rows():
    for n, world in ((4000, 2), (4000, 3), (64026, 8), (7, 7), (130, 4)):
        spans = [sharded.shard_rows(n, r, world) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == n
        assert all(spans[r][1] == spans[r + 1][0] for r in range(world - 1))
        sizes = [hi - lo for lo, hi in spans]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        sharded.shard_rows(3, 0, 4)
    keep = syn.keep_mask(5, 1000, 300, 10)
    masks = [sharded.shard_keep_mask(keep, r, 3) for r in range(3)]
    assert np.array_equal(sum(m.astype(int) for m in masks), keep.astype(int))


def _exchange_rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=60))
    try:
        W, keep, h, pairs = tiny_with_cross_shard_ties(world)
        idx, n_kept = oracle.build_index(keep)
        q, sf, g = oracle.nvfp4_quantize(W, idx)
        lo, hi = sharded.shard_rows(n_kept, rank, world)
        y, _ = oracle.gemv(oracle.FMT_NVFP4, q[lo:hi], sf[lo:hi], g, h, want_abs=False)
        keys = torch.from_numpy(shard_keys(y, idx[lo:hi]))
        sharded.exchange_keys(keys)
        np.save(os.path.join(out_dir, f"ids{rank}.npy"), decode(keys.numpy()))
    finally:
        tdist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.timeout(240)
def test_key_exchange_matches_the_unsharded_argmax(tmp_path, world):
    mp.start_processes(_exchange_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    W, keep, h, pairs = tiny_with_cross_shard_ties(world)
    idx, n_kept = oracle.build_index(keep)
    q, sf, g = oracle.nvfp4_quantize(W, idx)
    y, _ = oracle.gemv(oracle.FMT_NVFP4, q[:n_kept], sf[:n_kept], g, h, want_abs=False)
    want = expected_ids(y, idx[:n_kept])
    # the oracle's own first-max argmax agrees (ascending dh_idx: lowest row = lowest id)
    assert np.array_equal(want, oracle.top_tokens(y, idx[:n_kept])[0])
    assert want[0] == min(pairs[0]) and want[1] == min(pairs[1])
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"ids{r}.npy"), want)


def _leaver_rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=10))
    keys = torch.tensor([rank, -rank], dtype=torch.int64)
    sharded.exchange_keys(keys)                        # step 1: everyone takes part
    if rank == 1:
        os._exit(0)                                    # leaves between steps, no goodbye
    t0 = time.monotonic()
    try:
        sharded.exchange_keys(torch.zeros(2, dtype=torch.int64))  # step 2
        outcome = "no error"
    except sharded.ShardExchangeError as e:
        outcome = "ShardExchangeError"
    with open(os.path.join(out_dir, "rank0.txt"), "w") as f:
        f.write(f"{outcome} {time.monotonic() - t0:.2f} {keys.tolist()}")
    os._exit(0)


@pytest.mark.timeout(240)
def test_a_rank_that_leaves_between_steps_is_reported(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_leaver_rank, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode is not None
    outcome, secs, first = (tmp_path / "rank0.txt").read_text().split(" ", 2)
    assert outcome == "ShardExchangeError"
    assert float(secs) < 60.0
    assert first == "[1, 0]"                           # step 1's exchange was the max of both ranks

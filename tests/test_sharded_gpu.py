"""The vocabulary-sharded head on one GPU: shards of one quantised head (two
and three, run one after the other), their keys combined with a maximum as
the all-reduce does, decoded by the library. Checked against the header's key
definition, the oracle's unsharded argmax (ties across shard boundaries
resolve to the lowest id) and the unsharded head's own ids and logits."""
import numpy as np
import pytest
import torch

import nvfp4_draft_head_gb300 as dh
import oracle
import synthetic as syn
from nvfp4_draft_head_gb300 import sharded
from parity_util import check_argmax_rows, ids_to_rows
from test_sharded_gloo import tiny_with_cross_shard_ties

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return dev(bits.view(np.int16)).view(torch.bfloat16)


def full_head(W, keep):
    idx_np, n_kept = dh.draft_head_build_index(keep)
    idx = dev(idx_np)
    q, sf, g = dh.nvfp4_quantize_rows(dev_bf16(W), idx)
    return q, sf, g, idx, idx_np, n_kept


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("packed", [True, False])
def test_shards_match_the_oracle_and_the_unsharded_head(world, packed):
    W, keep, h_bits, pairs = tiny_with_cross_shard_ties(world)
    q, sf, g, idx, idx_np, n_kept = full_head(W, keep)
    V = W.shape[0]
    h = dev_bf16(h_bits)
    M = h_bits.shape[0]
    shards = [sharded.nvfp4_shard(q, sf, g, idx, n_kept, V, r, world, packed=packed) for r in range(world)]
    keys = [s.top_keys(h) for s in shards]
    for s in shards:
        assert s.device_error() == 0
    # each shard's key is the header's key of its oracle logits
    q_o, sf_o, g_o = oracle.nvfp4_quantize(W, idx_np)
    y_all, A_all = oracle.gemv(oracle.FMT_NVFP4, q_o[:n_kept], sf_o[:n_kept], g_o, h_bits)
    for r, k in enumerate(keys):
        lo, hi = sharded.shard_rows(n_kept, r, world)
        got = dh.keys_to_ids(k).cpu().numpy()
        check_argmax_rows(ids_to_rows(got, idx_np, n_kept) - lo, y_all[:, lo:hi], A_all[:, lo:hi], hi - lo,
                          f"shard {r} of {world}")
    combined = torch.stack(keys).max(dim=0).values
    top = torch.empty(M, dtype=torch.float32, device="cuda")
    ids = dh.keys_to_ids(combined, top=top).cpu().numpy()
    rows = ids_to_rows(ids, idx_np, n_kept)
    check_argmax_rows(rows, y_all, A_all, n_kept, f"{world} shards")
    assert ids[0] == min(pairs[0]) and ids[1] == min(pairs[1])
    # the unsharded head gives the same ids and top logits, bit for bit
    fmt = dh.DH_FMT_NVFP4_PACKED if packed else dh.DH_FMT_NVFP4
    qq = dh.nvfp4_pack_head(q, sf) if packed else q
    whole = dh.DraftHead(fmt, V, qq, idx, n_kept, sf=None if packed else sf, scale=g, idx_ascending=True)
    top_w = torch.empty(M, dtype=torch.float32, device="cuda")
    ids_w = whole.top_tokens(h, top=top_w).cpu().numpy()
    assert np.array_equal(ids, ids_w)
    assert np.array_equal(top.cpu().numpy(), top_w.cpu().numpy())
    # compute_logits: the maximum of the shards' rows is the whole head's row
    out = torch.stack([s.compute_logits(h) for s in shards]).max(dim=0).values
    assert torch.equal(out, whole.compute_logits(h))


def test_shard_keys_follow_the_header_definition():
    """Kernel keys decoded by hand: high word = ord(top logit), low word =
    0xFFFFFFFF - id, sign bit flipped; keys_to_ids inverts them."""
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    q, sf, g, idx, idx_np, n_kept = full_head(W, keep)
    s = sharded.nvfp4_shard(q, sf, g, idx, n_kept, W.shape[0], 0, 1)
    h_bits = syn.hidden_bf16(syn.hidden_seed(0, 5151), 5, c["K"])
    h = dev_bf16(h_bits)
    k = s.top_keys(h).cpu().numpy().view(np.uint64) ^ np.uint64(1 << 63)
    top = torch.empty(5, dtype=torch.float32, device="cuda")
    ids = s.top_tokens(h, top=top).cpu().numpy()
    assert np.array_equal(np.uint64(0xFFFFFFFF) - (k & np.uint64(0xFFFFFFFF)), ids.astype(np.uint64))
    t = top.cpu().numpy()
    ord_t = np.where(t >= 0, t.view(np.uint32).astype(np.uint64) | 0x80000000,
                     (~t.view(np.uint32)).astype(np.uint64) & 0xFFFFFFFF)
    assert np.array_equal(k >> np.uint64(32), ord_t)
    # a key of INT64_MIN decodes to id -1
    ids_min = dh.keys_to_ids(torch.full((3,), -(2 ** 63), dtype=torch.int64, device="cuda")).cpu().numpy()
    assert (ids_min == -1).all()


def test_shard_key_rejections():
    c = syn.TINY
    W = syn.head_bf16(syn.SEED_HEAD_TINY, c["V"], c["K"])
    keep = syn.keep_mask(syn.SEED_KEEP_TINY, c["V"], c["n_kept"], c["forced"])
    q, sf, g, idx, idx_np, n_kept = full_head(W, keep)
    unordered = dh.DraftHead(dh.DH_FMT_NVFP4, W.shape[0], q, idx, n_kept, sf=sf, scale=g, idx_ascending=False)
    h = dev_bf16(syn.hidden_bf16(1, 1, c["K"]))
    with pytest.raises(dh.DraftHeadError) as e:
        unordered.top_keys(h)
    assert e.value.status == dh.DH_ERR_ARG
    with pytest.raises(ValueError):
        sharded.ShardedDraftHead(unordered)


def test_full_size_two_shards():
    """The 64,064-row head split in two shards of 32,013 kept rows: combined
    ids and top logits equal the unsharded head's at one and four drafts."""
    c = syn.QWEN_64K
    Wd = dev_bf16(syn.head_bf16(syn.SEED_HEAD_QWEN, c["V"], c["K"]))
    keep = syn.keep_mask(syn.SEED_KEEP_64K, c["V"], c["n_kept"], c["forced"])
    idx_np, n_kept = dh.draft_head_build_index(keep)
    idx = dev(idx_np)
    q, sf, g = dh.nvfp4_quantize_rows(Wd, idx)
    del Wd
    V = c["V"]
    whole = dh.DraftHead(dh.DH_FMT_NVFP4_PACKED, V, dh.nvfp4_pack_head(q, sf), idx, n_kept, scale=g,
                         idx_ascending=True)
    shards = [sharded.nvfp4_shard(q, sf, g, idx, n_kept, V, r, 2) for r in range(2)]
    for M in (1, 4):
        for step in range(3):
            h = dev_bf16(syn.hidden_bf16(syn.hidden_seed(1, 6000 + 10 * M + step), M, c["K"]))
            keys = torch.stack([s.top_keys(h) for s in shards]).max(dim=0).values
            top = torch.empty(M, dtype=torch.float32, device="cuda")
            ids = dh.keys_to_ids(keys, top=top)
            top_w = torch.empty(M, dtype=torch.float32, device="cuda")
            ids_w = whole.top_tokens(h, top=top_w)
            assert torch.equal(ids, ids_w) and torch.equal(top, top_w), (M, step)
    assert all(s.device_error() == 0 for s in shards) and whole.device_error() == 0

"""Host-side checks of the seeded input generators (structure only, no method arithmetic)."""
import numpy as np
import torch

import workloads as W


def test_chunked_regeneration_is_consistent():
    w = W.small("t", [20000, 9000], [3, 1], seed=5, hot=4)
    full = w.ik_f32(0, 0, 0, 20000)
    part = w.ik_f32(0, 0, 8000, 8500)
    assert torch.equal(full[8000:8500], part)
    k1, v1 = w.kv_f32(0, 1, 0, 9000)
    k2, v2 = w.kv_f32(0, 1, 8190, 8200)
    assert torch.equal(k1[8190:8200], k2) and torch.equal(v1[8190:8200], v2)


def test_paging_and_shared_prefix():
    w = W.small("t", [16384 + 500, 20000, 3000], [2, 1, 4], seed=3, prefix_len=16384, prefix_seqs=2)
    nb = [w.nblocks(b) for b in range(w.B)]
    assert np.array_equal(w.block_table[0, :128], w.block_table[1, :128])
    used = np.concatenate([w.block_table[b, :nb[b]] for b in range(w.B)])
    assert len(set(used.tolist())) == w.unique_pages() == w.num_pages == sum(nb) - 128
    assert (w.block_table[2, nb[2]:] == -1).all()
    a = w.ik_f32(0, 0, 0, 16384)
    b = w.ik_f32(0, 1, 0, 16384)
    assert torch.equal(a, b)
    assert not torch.equal(w.ik_f32(0, 0, 16384, 16400), w.ik_f32(0, 1, 16384, 16400))


def test_hot_blocks_raise_index_scores():
    w = W.small("t", [8192], [2], seed=9, hot=6)
    hot = w.hot_blocks[0]
    assert len(hot) == 6 and hot.max() < (8192 - 2) // 128
    iq = w.iq_f32(0, 0)
    ik = w.ik_f32(0, 0, 0, 8192)
    s = (iq.reshape(-1, 128) @ ik.T).reshape(-1, 64, 128).amax(-1).mean(0)
    top = torch.topk(s[:63], 6).indices.sort().values.numpy()
    assert np.array_equal(top, hot)


def test_configs_shapes():
    for name in ("tiny", "decode", "spec", "long"):
        w = W.CONFIGS[name]()
        assert w.block_table.shape[0] == w.B
        assert w.T == sum(w.q_lens)
    r = W.ragged()
    assert r.B == 128 and len(r.layers) == 4
    assert [l.index_dtype for l in r.layers] == [0, 0, 1, 1]
    assert min(r.seq_lens) >= 1024 and max(r.seq_lens) <= 262144
    assert all(L > 16384 for L in r.seq_lens[:32])
    assert 1 <= min(r.q_lens) and max(r.q_lens) <= 8

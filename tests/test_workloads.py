"""The synthetic input recipe (CPU): workload shapes as documented, seeded
determinism, the page pool bookkeeping every parity test and the bench rely on,
and the planted blocks of the block-sparse workload."""
import numpy as np

from query_decode_attention_gb300 import workloads as W


def test_documented_shapes():
    s = W.serving_8b()
    assert (s.B, s.nq, s.nkv, s.hd, s.layers) == (64, 32, 8, 128, 36)
    assert s.seq_lens.min() >= 1024 and s.seq_lens.max() <= 32768
    q2 = W.qwen3vl_2b(4059)
    assert (q2.B, q2.nq, q2.nkv, q2.layers, int(q2.seq_lens[0])) == (1, 16, 8, 28, 4059)
    lc = W.long_context()
    assert (lc.B, lc.nq, lc.nkv) == (8, 16, 8) and set(lc.seq_lens.tolist()) == {131072}
    sp = W.sparse_planted(65536)
    assert (sp.B, sp.nq, sp.nkv, sp.block, sp.topk, sp.probe) == (16, 16, 8, 32, 32, 8)
    # 264 B per (token, KV head): 128 B of K codes, 128 B of V codes, two fp32 maxima
    assert s.kv_bytes_per_layer() == int(s.seq_lens.sum()) * 8 * 264


def test_seeded_determinism():
    a, b = W.serving_8b(seed=7), W.serving_8b(seed=7)
    assert np.array_equal(a.seq_lens, b.seq_lens)
    assert not np.array_equal(a.seq_lens, W.serving_8b(seed=8).seq_lens)
    wl = W.custom(2, 16, 8, [70, 33], seed=3)
    assert np.array_equal(W.host_q(wl), W.host_q(wl))
    k1, v1 = W.host_kv(wl, 1)
    k2, v2 = W.host_kv(wl, 1)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert k1.shape == (33, 8, 128) and v1.shape == (33, 8, 128)


def test_page_pool_is_a_permutation_and_slots_follow_it():
    wl = W.custom(5, 16, 8, [0, 1, 32, 33, 700], seed=11)
    pt, num_pages = W.page_table(wl, extra_pages=3)
    need = [0, 1, 1, 2, 22]
    assert num_pages == sum(need) + 3
    used = np.concatenate([pt[b, :need[b]] for b in range(wl.B)])
    assert len(set(used.tolist())) == len(used)                  # no page shared
    assert used.min() >= 0 and used.max() < num_pages
    for b in range(wl.B):
        assert (pt[b, need[b]:] == -1).all()                     # unused entries
    slots = W.all_slots(wl, pt)
    assert len(slots) == sum(int(n) for n in wl.seq_lens)
    assert len(set(slots.tolist())) == len(slots)                # every token its own row
    # token t of sequence b sits at row t mod 32 of its page
    s4 = W.slots_for(wl, pt, 4, 0, 700)
    t = np.arange(700)
    assert np.array_equal(s4 // 32, pt[4, t // 32]) and np.array_equal(s4 % 32, t % 32)


def test_planted_blocks_align_with_the_group_queries():
    # the planted workload's chosen blocks carry K rows aligned with the
    # group's queries, so their probe scores stand out from the N(0, 1) rest
    wl = W.sparse_planted(2048, B=1)
    q = W.host_q(wl)
    K, _ = W.host_kv(wl, 0, q=q)
    nblk = 2048 // wl.block
    planted = set(np.asarray(W.planted_blocks(wl, 0, 0)).tolist())
    assert len(planted) == min(32, nblk)
    qg = q[0, :wl.G].mean(axis=0)                                # KV head 0's group
    qg = qg / np.linalg.norm(qg)
    cos = []
    for j in range(nblk):
        rows = K[j * wl.block:(j + 1) * wl.block, 0]
        cos.append(float(np.mean(rows @ qg / np.linalg.norm(rows, axis=1))))
    top = set(np.argsort(cos)[-len(planted):].tolist())
    assert top == planted

"""Pins of the oracle's KV block bookkeeping.

The pages fix: logical blocks map to physical blocks through a per-sequence
block table; a block is taken only when the current one is full ("LLM
serving: speculative decoding and PagedAttention memory management",
PagedAttention section); on rejection only the rejected positions' blocks are
given back and accepted entries stay in place, O(1) per block ("Speculative
decoding principles and a vLLM production setup", sec. 3.1).

Checked here: a hand-worked example, the invariants (every physical block is
either free, held, or used by exactly one sequence below its length; the new
length is c + a + 1; accepted rows are byte-identical after rollback), and
all-or-nothing behaviour when the pool runs out.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_paged_gb300 import workloads as W


def _state(ctx, bs, num_blocks, free, bt_rows, max_blocks=8):
    B = len(ctx)
    bt = np.full((B, max_blocks), -1, np.int32)
    for b, row in enumerate(bt_rows):
        bt[b, :len(row)] = row
    fl = np.full(num_blocks, -1, np.int32)
    fl[:len(free)] = free
    pool = np.zeros((num_blocks, 1, bs, 2), np.float32)
    return W.KVState(bs, num_blocks, max_blocks, 1, 2, "f32", pool, pool.copy(), bt,
                     np.array(ctx, np.int32), fl, len(free))


def _step(n_q, start=100.0, d=2):
    n_q = np.array(n_q, np.int32)
    cu = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
    T = int(cu[-1])
    nk = (start + np.arange(T, dtype=np.float32))[:, None, None] * np.ones((1, 1, d), np.float32)
    return W.StepInputs(n_q, cu, 1, np.zeros((T, 1, d), np.float32), nk, -nk, 4, "f32",
                        np.zeros((T, 4), np.float32), np.zeros((T - len(n_q), 4), np.float32),
                        np.zeros(T - len(n_q), np.int32), np.zeros(T - len(n_q), np.float32),
                        np.zeros(len(n_q), np.float32), 1.0)


def test_hand_worked_example():
    # block size 4; seq 0 has 3 tokens in block 7, seq 1 has 4 tokens in block 2.
    # free stack (bottom..top): 5, 0, 9, 3  -> pops give 3, 9, 0, 5 in that order.
    st = _state([3, 4], 4, 10, [5, 0, 9, 3], [[7], [2]])
    kv = oracle.OracleKV(st)
    step = _step([4, 5])
    assert kv.append(step) is None
    # seq 0: 3+4 = 7 tokens -> 2 blocks, needs 1 more (pop 3)
    # seq 1: 4+5 = 9 tokens -> 3 blocks, had 1, needs 2 (pop 9 then 0)
    assert kv.bt[0][:3] == [7, 3, -1]
    assert kv.bt[1][:4] == [2, 9, 0, -1]
    assert kv.free == [5]
    # rows land at logical positions c + j
    assert kv.k_pool[7, 0, 3, 0] == 100.0  # seq 0 row 0 at position 3
    assert kv.k_pool[3, 0, 2, 0] == 103.0  # seq 0 row 3 at position 6
    assert kv.k_pool[9, 0, 0, 0] == 104.0  # seq 1 row 0 at position 4
    assert kv.k_pool[0, 0, 0, 0] == 108.0  # seq 1 row 4 at position 8
    assert kv.v_pool[0, 0, 0, 1] == -108.0
    # seq 0 accepts 0 drafts: new length 3+0+1 = 4 -> 1 block, block 3 goes back
    # seq 1 accepts 2: new length 4+2+1 = 7 -> 2 blocks, block 0 goes back
    kv.rollback(step, [0, 2])
    assert kv.seq_lens == [4, 7]
    assert kv.bt[0][:2] == [7, -1]
    assert kv.bt[1][:3] == [2, 9, -1]
    assert kv.free == [5, 3, 0]


def test_out_of_blocks_changes_nothing():
    st = _state([3, 4], 4, 10, [5, 0], [[7], [2]])
    kv = oracle.OracleKV(st)
    before = (kv.k_pool.copy(), [r[:] for r in kv.bt], kv.free[:])
    assert kv.append(_step([4, 5])) == oracle.OUT_OF_BLOCKS
    assert np.array_equal(kv.k_pool, before[0]) and kv.bt == before[1] and kv.free == before[2]


def test_block_table_room_is_checked():
    st = _state([7], 4, 10, [1, 2, 3], [[4, 5]], max_blocks=2)
    kv = oracle.OracleKV(st)
    assert kv.append(_step([3])) == oracle.NO_TABLE_ROOM


def _owned(kv):
    used = []
    for b, row in enumerate(kv.bt):
        nb = (kv.seq_lens[b] + kv.bs - 1) // kv.bs
        used += row[:nb]
        assert all(x == -1 for x in row[nb:]), "blocks past the end must be released"
    return used


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invariants_over_many_steps(seed):
    rng = np.random.default_rng(seed)
    case = W.custom(seed, batch=6, ctx_lens=rng.integers(0, 60, 6), n_q=np.full(6, 5), num_q_heads=2,
                    num_kv_heads=1, head_dim=4, block_size=8, vocab=8, dtype="f32", pool_factor=3.0,
                    growth_tokens=200, held_fraction=0.2, use_bank=False)
    st = case.state
    kv = oracle.OracleKV(st)
    universe = sorted(set(range(st.num_blocks)) - set(map(int, st.held_blocks)))
    assert sorted(_owned(kv) + kv.free) == universe
    for it in range(30):
        n_q = rng.integers(1, 9, 6)
        step = _step(n_q, start=1000.0 * (it + 1), d=4)
        c0 = kv.seq_lens[:]
        assert kv.append(step) is None
        # accepted prefix snapshot
        acc = [int(rng.integers(0, n)) for n in n_q]
        snap = {}
        for b in range(6):
            for j in range(acc[b] + 1):
                pos = c0[b] + j
                snap[(b, j)] = kv.k_pool[kv.bt[b][pos // kv.bs], 0, pos % kv.bs].copy()
        kv.rollback(step, acc)
        assert kv.seq_lens == [c0[b] + acc[b] + 1 for b in range(6)]
        for (b, j), row in snap.items():
            pos = c0[b] + j
            np.testing.assert_array_equal(kv.k_pool[kv.bt[b][pos // kv.bs], 0, pos % kv.bs], row)
            assert row[0] == 1000.0 * (it + 1) + step.cu_q[b] + j
        used = _owned(kv)
        assert len(used) == len(set(used))
        assert sorted(used + kv.free) == universe


def test_tree_rollback_compacts_the_accepted_path():
    st = _state([5], 4, 8, [1, 2, 3, 4, 5], [[6, 0]])
    kv = oracle.OracleKV(st)
    step = _step([7])  # root + 6 nodes at positions 5..11
    assert kv.append(step) is None
    # path: nodes 2 -> 4 -> 6 (rows 2, 4, 6 of the step)
    kv.rollback(step, [3], path_nodes=[[2, 4, 6, -1, -1, -1, -1]])
    assert kv.seq_lens == [5 + 3 + 1]
    vals = []
    for pos in range(5, 9):
        vals.append(kv.k_pool[kv.bt[0][pos // 4], 0, pos % 4, 0])
    assert vals == [100.0, 102.0, 104.0, 106.0]
    # 12 tokens used 3 blocks; 9 tokens keep 3 blocks: nothing freed
    assert kv.bt[0][:3] == [6, 0, 5] and kv.free == [1, 2, 3, 4]


def test_workload_pool_partition():
    """Context blocks, held blocks and the free list partition the pool."""
    case = W.contbatch(3, batch=16, vocab=64)
    st = case.state
    used = []
    for b in range(st.batch):
        nb = (int(st.seq_lens[b]) + st.block_size - 1) // st.block_size
        used += list(st.block_table[b, :nb])
    allids = used + list(st.held_blocks) + list(st.free_list[:st.free_top])
    assert sorted(allids) == list(range(st.num_blocks))
    assert abs(len(st.held_blocks) / st.num_blocks - 0.3) < 0.01

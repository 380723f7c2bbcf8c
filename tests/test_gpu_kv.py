"""GPU parity of sv_kv_append / sv_kv_rollback against the oracle's block
bookkeeping: block tables, seq_lens, free list and pool bytes bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import (appended_rows, assert_kv_equal, compare_samples, gpu_sample_result, kv_host, max_seq_len,
                      status_of, upload)

pytestmark = pytest.mark.gpu


def _accepts(rng, n_q):
    return np.array([int(rng.integers(0, n)) for n in n_q], np.int32)


@pytest.mark.parametrize("make", [
    lambda: W.tiny(),
    lambda: W.custom(7, batch=5, ctx_lens=[0, 1, 15, 16, 130], n_q=[1, 3, 2, 9, 64], num_q_heads=4,
                     num_kv_heads=2, head_dim=64, block_size=16, vocab=64, use_bank=False),
    lambda: W.custom(8, batch=3, ctx_lens=[127, 128, 129], n_q=[2, 5, 8], num_q_heads=8, num_kv_heads=8,
                     head_dim=128, block_size=128, vocab=64, held_fraction=0.3),
    lambda: W.custom(9, batch=4, ctx_lens=[3, 300, 17, 64], n_q=[6, 6, 6, 6], num_q_heads=4, num_kv_heads=1,
                     head_dim=32, block_size=1, vocab=64, dtype="f32"),
], ids=["tiny", "ragged-bs16", "bs128-fragmented", "bs1-f32"])
def test_append_rollback_small_exact(make):
    case = make()
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    S.append(kv, d, buf)
    assert okv.append(case.step) is None
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_kv_equal(kv, okv)
    acc = _accepts(np.random.default_rng(1), case.step.n_q)
    buf.accept.copy_(torch.from_numpy(acc))
    S.rollback(kv, d, buf)
    okv.rollback(case.step, acc)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_kv_equal(kv, okv)


@pytest.mark.parametrize("batch,n,heads,head_dim", [
    (1500, 2, 1, 32),   # the bookkeeping CTA's scans take two passes of 1024 threads
    (2100, 1, 1, 32),   # more sequences than the scatter stages cu_q for (it reads cu_q from global)
    (64, 64, 8, 128),   # 4096 rows of the longest chains
], ids=["1500-seqs", "2100-seqs", "4096-rows"])
def test_append_large_batches(batch, n, heads, head_dim):
    """Large batches pop the same blocks in the same order and write the same bytes as the oracle."""
    rng = np.random.default_rng(batch)
    ctx = rng.integers(0, 100, batch).astype(np.int32)
    case = W.custom(11, batch=batch, ctx_lens=ctx, n_q=[n] * batch, num_q_heads=heads, num_kv_heads=heads,
                    head_dim=head_dim, block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    S.append(kv, d, buf)
    assert okv.append(case.step) is None
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_kv_equal(kv, okv)
    acc = _accepts(rng, case.step.n_q)
    buf.accept.copy_(torch.from_numpy(acc))
    S.rollback(kv, d, buf)
    okv.rollback(case.step, acc)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_kv_equal(kv, okv, pools=False)


@pytest.mark.parametrize("batch,n", [(3, 5), (64, 64)], ids=["small", "4096-rows"])
def test_bad_popped_id_is_all_or_nothing(batch, n):
    """An id out of range among those about to be popped: SV_ERR_BAD_BLOCK_ID and nothing written."""
    case = W.custom(12, batch=batch, ctx_lens=[16] * batch, n_q=[n] * batch, num_q_heads=8, num_kv_heads=8,
                    head_dim=128, block_size=16, vocab=16, use_bank=False)
    st = case.state
    nb = st.k_pool.shape[0]
    st.free_list[st.free_top - 2] = nb + 5  # the second id to be popped
    kv, d, buf = upload(case)
    before = kv_host(kv)
    kbefore = kv.k_pool.clone()
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 6  # SV_ERR_BAD_BLOCK_ID
    after = kv_host(kv)
    for k in before:
        np.testing.assert_array_equal(np.asarray(before[k]), np.asarray(after[k]))
    assert torch.equal(kbefore, kv.k_pool)


@pytest.mark.parametrize("name", ["llama8b", "llama70b"])
def test_append_rollback_full_size(name):
    case = W.CONFIGS[name]()
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    c0 = list(okv.seq_lens)
    S.append(kv, d, buf)
    okv.append(case.step)
    acc = _accepts(np.random.default_rng(2), case.step.n_q)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    rows = appended_rows(okv, case.step, c0)
    assert_kv_equal(kv, okv, rows=rows)
    # untouched context rows keep their bytes: spot check one row per sequence
    kp = S.to_bits(kv.k_pool)
    for b in range(case.state.batch):
        if c0[b] > 0:
            pos = c0[b] - 1
            blk = okv.bt[b][pos // okv.bs]
            np.testing.assert_array_equal(kp[blk, :, pos % okv.bs], case.state.k_pool[blk, :, pos % okv.bs])
    buf.accept.copy_(torch.from_numpy(acc))
    S.rollback(kv, d, buf)
    okv.rollback(case.step, acc)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_kv_equal(kv, okv, pools=False)


def test_tree_rollback_compacts_path():
    case = W.tree(batch=4, ctx=1000, vocab=512)
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    c0 = list(okv.seq_lens)
    S.append(kv, d, buf)
    okv.append(case.step)
    # random root-to-node paths of the real trees
    rng = np.random.default_rng(3)
    B, mq = case.state.batch, case.step.max_q
    acc = np.zeros(B, np.int32)
    path = np.full((B, mq), -1, np.int32)
    for b in range(B):
        par = case.step.parent[case.step.cu_q[b]:case.step.cu_q[b + 1]]
        node = int(rng.integers(0, len(par)))
        chain = []
        while node > 0:
            chain.append(node)
            node = int(par[node])
        chain = chain[::-1]
        acc[b] = len(chain)
        path[b, :len(chain)] = chain
    buf.accept.copy_(torch.from_numpy(acc))
    buf.path.copy_(torch.from_numpy(path))
    S.rollback(kv, d, buf)
    okv.rollback(case.step, acc, path_nodes=path)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    rows = []
    for b in range(B):
        for j in range(acc[b] + 1):
            pos = c0[b] + j
            rows.append((okv.bt[b][pos // okv.bs], pos % okv.bs))
    assert_kv_equal(kv, okv, rows=rows)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_tree_step_at_temperature(kv_dtype):
    """The whole step with a stochastic tree: append, attention, tree rejection
    sample, rollback with the accepted path (the path's rows moved as bf16 rows
    or as E4M3 codes), against the oracle."""
    case = W.tree(batch=4, ctx=1000, vocab=512, temperature=1.0, kv_dtype=kv_dtype)
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    c0 = list(okv.seq_lens)
    msl = max_seq_len(case.state, case.step)
    S.append(kv, d, buf)
    S.attention(kv, d, buf, msl)
    S.sample(d, buf)
    okv.append(case.step)
    ref = oracle.tree_sample(case.step)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    got = gpu_sample_result(buf)
    compare_samples(case.step, got, ref)  # a divergence only at a flagged near-tie
    same = got[0] == ref.accept_cnt
    np.testing.assert_array_equal(buf.path.cpu().numpy()[same], ref.path_nodes[same])
    if not same.all():  # the rollback then takes the oracle's decisions, so the caches stay comparable
        buf.accept.copy_(torch.from_numpy(ref.accept_cnt))
        buf.path.copy_(torch.from_numpy(ref.path_nodes))
    S.rollback(kv, d, buf)
    okv.rollback(case.step, ref.accept_cnt, path_nodes=ref.path_nodes)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    rows = []
    for b in range(case.state.batch):
        for j in range(ref.accept_cnt[b] + 1):
            pos = c0[b] + j
            rows.append((okv.bt[b][pos // okv.bs], pos % okv.bs))
    assert_kv_equal(kv, okv, rows=rows)


def test_out_of_blocks_is_all_or_nothing():
    case = W.custom(4, batch=3, ctx_lens=[15, 31, 47], n_q=[5, 5, 5], num_q_heads=2, num_kv_heads=1,
                    head_dim=32, block_size=16, vocab=16, pool_factor=1.0, use_bank=False)
    st = case.state
    st.free_top = 1  # three sequences each need a new block
    kv, d, buf = upload(case)
    before = kv_host(kv)
    kbefore = kv.k_pool.clone()
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 4  # SV_ERR_OUT_OF_BLOCKS
    after = kv_host(kv)
    for k in before:
        np.testing.assert_array_equal(np.asarray(before[k]), np.asarray(after[k]))
    assert torch.equal(kbefore, kv.k_pool)
    # a recorded error makes the next state-changing calls no-ops
    buf.accept.zero_()
    S.rollback(kv, d, buf)
    torch.cuda.synchronize()
    after2 = kv_host(kv)
    for k in before:
        np.testing.assert_array_equal(np.asarray(before[k]), np.asarray(after2[k]))


def test_bad_accept_count_changes_nothing():
    case = W.tiny()
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    mid = kv_host(kv)
    buf.accept.copy_(torch.tensor([0, 1, 9, 2], dtype=torch.int32))  # 9 > K
    S.rollback(kv, d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 7
    after = kv_host(kv)
    for k in mid:
        np.testing.assert_array_equal(np.asarray(mid[k]), np.asarray(after[k]))


def test_block_table_room_is_checked():
    case = W.custom(5, batch=2, ctx_lens=[30, 10], n_q=[5, 2], num_q_heads=2, num_kv_heads=1, head_dim=32,
                    block_size=16, vocab=16, use_bank=False)
    st = case.state
    st.block_table = st.block_table[:, :2].copy()  # 30 + 5 tokens need 3 blocks
    st.max_blocks_per_seq = 2
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 7


def test_host_argument_errors():
    case = W.tiny()
    kv, d, buf = upload(case)
    with pytest.raises(L.SVError) as e:
        L.kv_append(kv, d.new_k, d.new_v, d.cu_q, None)  # status word is required
    assert e.value.code == 1
    with pytest.raises(TypeError):
        L.kv_append(kv, d.new_k.cpu(), d.new_v, d.cu_q, buf.status)

"""Pins of the oracle's attention against things other than itself.

* paged == dense: the oracle's block-table gather, checked against numpy fancy
  indexing of the pool (PagedAttention section of "LLM serving: speculative
  decoding and PagedAttention memory management": logical blocks map to
  physical blocks through the block table);
* dense == torch's scaled_dot_product_attention in fp64 with an explicit
  boolean mask (a library routine), for causal and tree masks and GQA;
* closed forms: uniform value rows, a single visible key, a chain-shaped tree
  mask equal to the causal mask.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import workloads as W


def _gather(state, b, L):
    """[L, Hkv, D] float64 keys/values of sequence b by numpy indexing."""
    pos = np.arange(L)
    blk = state.block_table[b, pos // state.block_size]
    assert (blk >= 0).all()
    k = state.k_pool[blk, :, pos % state.block_size, :]
    v = state.v_pool[blk, :, pos % state.block_size, :]
    if state.dtype == "bf16":
        k, v = W.bf16_bits_to_f32(k), W.bf16_bits_to_f32(v)
    return k.astype(np.float64), v.astype(np.float64)


def _qrows(step, b):
    q = step.q[step.cu_q[b]:step.cu_q[b + 1]]
    if q.dtype == np.uint16:
        q = W.bf16_bits_to_f32(q)
    return q.astype(np.float64)


def _sdpa(k, v, q, ctx, scale, mask_rows):
    """torch SDPA (fp64) with GQA by repeating each KV head Hq/Hkv times."""
    L, hkv, d = k.shape
    n, hq, _ = q.shape
    g = hq // hkv
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [hq, L, d]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, dim=0)
    qt = torch.from_numpy(q).permute(1, 0, 2)  # [hq, n, d]
    m = torch.zeros((n, L), dtype=torch.bool)
    m[:, :ctx] = True
    for i in range(n):
        for j in range(n):
            m[i, ctx + j] = bool(mask_rows(i, j))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o.permute(1, 0, 2).numpy()


def _small_case(seed=3, dtype="bf16", bs=16, hq=8, hkv=2, d=32, ctx=(5, 33, 70), nq=(3, 1, 6)):
    return W.custom(seed, batch=len(ctx), ctx_lens=ctx, n_q=nq, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=d, block_size=bs, vocab=64, dtype=dtype, use_bank=False)


@pytest.mark.parametrize("dtype,bs", [("bf16", 16), ("f32", 16), ("bf16", 4), ("f32", 64)])
def test_paged_equals_dense_exactly(dtype, bs):
    case = _small_case(dtype=dtype, bs=bs)
    kv = oracle.OracleKV(case.state)
    assert kv.append(case.step) is None
    st = kv.as_state()
    out = oracle.paged_attention(st, case.step)
    for b in range(st.batch):
        n = int(case.step.n_q[b])
        L = int(st.seq_lens[b]) + n
        k, v = _gather(st, b, L)
        dense = oracle.dense_attention(k, v, _qrows(case.step, b), int(st.seq_lens[b]), scale=case.step.scale)
        np.testing.assert_array_equal(out[case.step.cu_q[b]:case.step.cu_q[b + 1]], dense)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4), (6, 1)])
def test_dense_matches_torch_sdpa_causal(hq, hkv):
    rng = np.random.default_rng(11)
    ctx, n, d = 23, 5, 16
    k = rng.standard_normal((ctx + n, hkv, d))
    v = rng.standard_normal((ctx + n, hkv, d))
    q = rng.standard_normal((n, hq, d))
    scale = 0.37
    got = oracle.dense_attention(k, v, q, ctx, scale=scale)
    want = _sdpa(k, v, q, ctx, scale, lambda i, j: j <= i)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dense_matches_torch_sdpa_tree():
    rng = np.random.default_rng(12)
    parent = [-1, 0, 0, 1, 1, 2, 3, 5]
    n = len(parent)
    masks = np.zeros(n, np.uint64)
    for i in range(n):
        m, a = 0, i
        while a >= 0:
            m |= 1 << a
            a = parent[a]
        masks[i] = m
    ctx, hq, hkv, d = 9, 4, 2, 8
    k = rng.standard_normal((ctx + n, hkv, d))
    v = rng.standard_normal((ctx + n, hkv, d))
    q = rng.standard_normal((n, hq, d))
    got = oracle.dense_attention(k, v, q, ctx, mask_kind="tree", tree_mask=masks, scale=0.5)
    want = _sdpa(k, v, q, ctx, 0.5, lambda i, j: (int(masks[i]) >> j) & 1)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_uniform_values_give_that_row():
    rng = np.random.default_rng(13)
    ctx, n, hq, hkv, d = 40, 4, 4, 2, 8
    k = rng.standard_normal((ctx + n, hkv, d))
    row = rng.standard_normal((hkv, d))
    v = np.broadcast_to(row, (ctx + n, hkv, d)).copy()
    q = rng.standard_normal((n, hq, d)) * 3
    got = oracle.dense_attention(k, v, q, ctx, scale=0.25)
    for h in range(hq):
        np.testing.assert_allclose(got[:, h, :], np.broadcast_to(row[h // 2], (n, d)), rtol=1e-13, atol=1e-13)


def test_single_visible_key_gives_its_value():
    rng = np.random.default_rng(14)
    k = rng.standard_normal((1, 1, 8))
    v = rng.standard_normal((1, 1, 8))
    q = rng.standard_normal((1, 3, 8))
    got = oracle.dense_attention(k, v, q, 0, scale=1.0)
    for h in range(3):
        np.testing.assert_array_equal(got[0, h], v[0, 0])


def test_chain_tree_equals_causal():
    case = _small_case(seed=5, nq=(4, 6, 2))
    kv = oracle.OracleKV(case.state)
    kv.append(case.step)
    st = kv.as_state()
    causal = oracle.paged_attention(st, case.step)
    step = case.step
    masks = np.concatenate([np.array([(1 << (i + 1)) - 1 for i in range(int(n))], np.uint64) for n in step.n_q])
    step.mask_kind, step.tree_mask = "tree", masks
    tree = oracle.paged_attention(st, step)
    np.testing.assert_array_equal(causal, tree)


def test_masked_future_rows_do_not_matter():
    """Changing a key/value that row i may not see leaves row i unchanged."""
    rng = np.random.default_rng(15)
    ctx, n, hq, hkv, d = 12, 5, 2, 1, 8
    k = rng.standard_normal((ctx + n, hkv, d))
    v = rng.standard_normal((ctx + n, hkv, d))
    q = rng.standard_normal((n, hq, d))
    a = oracle.dense_attention(k, v, q, ctx, scale=0.3)
    k2, v2 = k.copy(), v.copy()
    k2[ctx + 3] += 5.0
    v2[ctx + 3] -= 7.0
    b = oracle.dense_attention(k2, v2, q, ctx, scale=0.3)
    np.testing.assert_array_equal(a[:3], b[:3])
    assert not np.allclose(a[3:], b[3:])


def test_bad_block_id_is_an_error():
    case = _small_case()
    st = case.state.copy()
    kv = oracle.OracleKV(st)
    kv.append(case.step)
    s2 = kv.as_state()
    s2.block_table = s2.block_table.copy()
    s2.block_table[1, 0] = s2.num_blocks + 3
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(s2, case.step)


def test_paged_attention_refuses_a_state_without_pools():
    import oracle as O
    from speculative_decoding_verify_paged_gb300 import workloads as W
    case = W.tiny()
    okv = O.OracleKV(case.state, with_pools=False)
    with pytest.raises(ValueError):
        O.paged_attention(okv.as_state(), case.step)


def test_threads_do_not_change_values():
    """The oracle's OpenMP tasks compute every value in the single-thread order."""
    import os
    import oracle as O
    from speculative_decoding_verify_paged_gb300 import workloads as W
    case = W.tiny()
    okv = O.OracleKV(case.state)
    okv.append(case.step)
    outs = []
    for t in (1, max(2, os.cpu_count() or 2)):
        O.set_threads(t)
        a = O.paged_attention(okv.as_state(), case.step)
        r = O.rejection_sample(case.step)
        outs.append((a, r.accept_cnt, r.out_tok, r.margin))
    O.set_threads(os.cpu_count() or 1)
    for x, y in zip(*outs):
        assert np.array_equal(x, y)

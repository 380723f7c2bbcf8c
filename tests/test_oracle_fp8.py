"""Pins of the oracle's E4M3 codec (the fp8 KV pool's element format) against
torch's float8_e4m3fn conversions (a library routine) and hand-worked values."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_decode_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode_table()
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_hand_worked_values():
    assert fp8.decode_table()[0x7E] == 448.0  # largest finite
    assert fp8.decode_table()[0x01] == 2.0 ** -9  # smallest subnormal
    assert fp8.decode_table()[0x38] == 1.0
    # ties go to the even mantissa: 1.0625 sits between 1.0 (0x38) and 1.125 (0x39)
    assert fp8.encode(np.float32([1.0625]))[0] == 0x38
    assert fp8.encode(np.float32([1.1875]))[0] == 0x3A  # between 1.125 (0x39) and 1.25 (0x3A)
    # saturation, NaN, signed zero
    assert list(fp8.encode(np.float32([1000.0, -1e9, 460.0]))) == [0x7E, 0xFE, 0x7E]
    assert fp8.encode(np.float32([np.nan]))[0] == 0x7F
    assert list(fp8.encode(np.float32([0.0, -0.0, -1e-12]))) == [0x00, 0x80, 0x80]


@pytest.mark.parametrize("scale", [1.0, 1.0 / 32, 3.7])
def test_encode_matches_torch_in_range(scale):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * 40 / scale).astype(np.float32)
    x = np.concatenate([x, fp8.decode_table()[:0x7F].astype(np.float32), np.float32([2.0 ** -10, 3 * 2.0 ** -11])])
    x = x[np.abs(x) <= 448.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.encode(x), want)
    # and the round trip of every finite code
    codes = np.arange(256, dtype=np.uint8)
    fin = ~np.isnan(fp8.decode_table())
    np.testing.assert_array_equal(fp8.encode(fp8.decode(codes[fin]).astype(np.float32)), codes[fin])


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_oracle_fp8_pool_append_and_attention():
    """The oracle's append stores torch's E4M3 code of x / scale (fp32 division)
    for each new row, and its attention over an E4M3 pool equals a brute-force
    softmax over the decoded keys and values (bf16 queries)."""
    import oracle
    from speculative_decoding_verify_paged_gb300 import workloads as W
    case = W.custom(41, batch=2, ctx_lens=[37, 5], n_q=[3, 4], num_q_heads=4, num_kv_heads=2, head_dim=32,
                    block_size=16, vocab=16, dtype="e4m3", use_bank=False)
    st, sp = case.state, case.step
    okv = oracle.OracleKV(st)
    assert okv.append(sp) is None
    s2 = okv.as_state()
    bs, D, Hq, G = st.block_size, st.head_dim, sp.num_q_heads, sp.num_q_heads // st.num_kv_heads
    cu = np.concatenate([[0], np.cumsum(sp.n_q)])
    for b in range(2):
        for i in range(int(sp.n_q[b])):
            t = int(st.seq_lens[b]) + i
            blk = s2.block_table[b, t // bs]
            for pool, new, scale in ((s2.k_pool, sp.new_k, st.k_scale), (s2.v_pool, sp.new_v, st.v_scale)):
                x = torch.from_numpy((_bf16_to_f64(new[cu[b] + i]).astype(np.float32) / np.float32(scale)))
                np.testing.assert_array_equal(pool[blk, :, t % bs], x.to(torch.float8_e4m3fn).view(torch.uint8))
    dec = lambda p, sc: torch.from_numpy(p).view(torch.float8_e4m3fn).to(torch.float64).numpy() * sc
    K, V = dec(s2.k_pool, st.k_scale), dec(s2.v_pool, st.v_scale)
    q = _bf16_to_f64(sp.q)
    ref = oracle.paged_attention(s2, sp)
    for b in range(2):
        for i in range(int(sp.n_q[b])):
            L = int(st.seq_lens[b]) + i + 1
            for h in range(Hq):
                ks = np.stack([K[s2.block_table[b, t // bs], h // G, t % bs] for t in range(L)])
                vs = np.stack([V[s2.block_table[b, t // bs], h // G, t % bs] for t in range(L)])
                s = ks @ q[cu[b] + i, h] / np.sqrt(D)
                p = np.exp(s - s.max())
                np.testing.assert_allclose(ref[cu[b] + i, h], p @ vs / p.sum(), rtol=0, atol=1e-12)

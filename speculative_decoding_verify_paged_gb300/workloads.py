"""Seeded synthetic inputs for the speculative-decoding verify step.

Both the fp64 CPU oracle and the CUDA library consume what this module makes.
It holds none of the verification arithmetic: no attention, no accept test, no
residual resampling and no block allocation. It stands in for the world around
the verifier:

* the KV cache of the committed context (a shuffled physical block pool, a
  per-sequence block table, and a free list of the unused blocks);
* the target model's query rows, new K/V rows and logits for the K+1 verified
  positions of each sequence;
* a draft model: its logits, and the draft tokens it proposes (x_i ~ q_i by
  inverse CDF in fp64 for T > 0, argmax for T = 0, top-k children for trees);
* the uniform random numbers that the accept test and the resample step use.

Every array is produced on the host from numpy's PCG64 generator, so it is the
same on every machine. bf16 tensors are stored as uint16 bit patterns (fp32
values rounded to nearest even); the same bits go to the oracle and the GPU.

Large normal arrays (KV pools, vocab-wide logits) are cut as windows, at
seeded random offsets, out of one N(0, 1) bank. Every row still holds N(0, 1)
values; two rows share values only if their windows overlap, which is rare
and harmless for the verify step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BANK_LOG2 = 25  # 32 Mi normals in the bank


# ----------------------------------------------------------------------------
# containers
# ----------------------------------------------------------------------------
@dataclass
class KVState:
    """Paged KV cache of the committed context, as host arrays."""

    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    num_kv_heads: int
    head_dim: int
    dtype: str  # "bf16" (uint16 bit patterns), "f32", or "e4m3" (uint8 codes of an fp8 pool)
    k_pool: np.ndarray  # [num_blocks, Hkv, block_size, D]
    v_pool: np.ndarray
    block_table: np.ndarray  # int32 [B, max_blocks_per_seq], -1 = no block
    seq_lens: np.ndarray  # int32 [B], committed tokens c_b
    free_list: np.ndarray  # int32 [num_blocks]; entries [0, free_top) are free ids
    free_top: int
    held_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    k_scale: float = 1.0  # e4m3 pools: a code's value times the scale
    v_scale: float = 1.0

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    def copy(self) -> "KVState":
        return KVState(
            self.block_size, self.num_blocks, self.max_blocks_per_seq,
            self.num_kv_heads, self.head_dim, self.dtype,
            self.k_pool.copy(), self.v_pool.copy(), self.block_table.copy(),
            self.seq_lens.copy(), self.free_list.copy(), self.free_top,
            self.held_blocks.copy(), self.k_scale, self.v_scale)


@dataclass
class StepInputs:
    """Inputs of one verify step for every sequence of the batch.

    Sequence b owns query rows cu_q[b] .. cu_q[b+1]-1. Row 0 of a sequence is
    the last emitted token; rows 1..K_b are the draft tokens (chain) or the
    draft-tree nodes in BFS order (tree). Draft-side arrays (draft logits,
    draft tokens, accept uniforms) have one entry per row except row 0, at
    index cu_q[b] - b + (i - 1) for row i.
    """

    n_q: np.ndarray  # int32 [B]
    cu_q: np.ndarray  # int32 [B+1]
    num_q_heads: int
    q: np.ndarray  # [T_q, Hq, D]   (uint16 bf16 bits or f32)
    new_k: np.ndarray  # [T_q, Hkv, D]
    new_v: np.ndarray
    vocab: int
    logits_dtype: str
    target_logits: np.ndarray  # [T_q, V]
    draft_logits: np.ndarray  # [T_q - B, V]
    draft_tokens: np.ndarray  # int32 [T_q - B]
    u_accept: np.ndarray  # float32 [T_q - B]
    u_resample: np.ndarray  # float32 [B]
    temperature: float
    mask_kind: str = "causal"  # "causal" | "tree"
    tree_mask: Optional[np.ndarray] = None  # uint64 [T_q]: bit j => row sees new row j
    parent: Optional[np.ndarray] = None  # int32 [T_q]: parent row within sequence, -1 root

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_q(self) -> int:
        return int(self.n_q.max()) if self.n_q.size else 1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.q.shape[-1])


@dataclass
class Case:
    name: str
    seed: int
    state: KVState
    step: StepInputs
    meta: dict = field(default_factory=dict)


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) as uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, *stream]))


class _Bank:
    """A seeded bank of N(0,1) values that windows are cut from."""

    _cache: dict = {}

    def __init__(self, seed: int, log2: int = BANK_LOG2):
        self.n = 1 << log2
        key = (seed, log2)
        if key not in _Bank._cache:
            if len(_Bank._cache) >= 2:
                _Bank._cache.pop(next(iter(_Bank._cache)))
            _Bank._cache[key] = _rng(seed, 0xBA4C).standard_normal(self.n, dtype=np.float32)
        self.vals = _Bank._cache[key]

    def windows(self, rng: np.random.Generator, count: int, width: int) -> np.ndarray:
        """[count, width] float32 rows, each a window at a random offset."""
        assert width <= self.n
        off = rng.integers(0, self.n - width + 1, size=count, dtype=np.int64)
        out = np.empty((count, width), np.float32)
        for i in range(count):  # row copies: memory bound, no per-element Python
            o = int(off[i])
            out[i] = self.vals[o:o + width]
        return out


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x) if dtype == "bf16" else x


def _draft_sample(rng: np.random.Generator, draft_f32: np.ndarray, temperature: float) -> np.ndarray:
    """The draft model's own token choice: x ~ softmax(l_d / T) (inverse CDF, fp64),
    or argmax (lowest index) when T == 0."""
    if draft_f32.shape[0] == 0:
        return np.zeros(0, np.int32)
    if temperature == 0.0:
        return np.argmax(draft_f32, axis=1).astype(np.int32)
    out = np.empty(draft_f32.shape[0], np.int32)
    u = rng.random(draft_f32.shape[0])
    for r in range(draft_f32.shape[0]):
        z = draft_f32[r].astype(np.float64) / temperature
        w = np.exp(z - z.max())
        c = np.cumsum(w)
        idx = int(np.searchsorted(c, u[r] * c[-1], side="right"))
        out[r] = min(idx, draft_f32.shape[1] - 1)
    return out


# ----------------------------------------------------------------------------
# KV state
# ----------------------------------------------------------------------------
def make_kv_state(seed: int, ctx_lens: np.ndarray, *, block_size: int, num_kv_heads: int,
                  head_dim: int, dtype: str, num_blocks: Optional[int] = None,
                  growth_tokens: int = 0, pool_factor: float = 1.25, held_fraction: float = 0.0,
                  max_blocks_per_seq: Optional[int] = None) -> KVState:
    """Context KV of every sequence in a shuffled physical pool.

    Physical ids are a seeded permutation of the pool. The context blocks of
    sequence 0, 1, ... take the first ids of the permutation in order; then a
    `held_fraction` of the whole pool is set aside as blocks held by other,
    unmodelled sequences (they never appear on the free list, which fragments
    it); the remaining ids form the free list in permutation order.
    """
    rng = _rng(seed, 1)
    ctx_lens = np.asarray(ctx_lens, np.int32)
    B = ctx_lens.shape[0]
    ctx_blocks = (ctx_lens + block_size - 1) // block_size
    reach = (ctx_lens + growth_tokens + block_size - 1) // block_size
    need = int(reach.sum())
    if num_blocks is None:
        num_blocks = max(int(math.ceil(need * pool_factor / (1.0 - held_fraction))), int(ctx_blocks.sum()) + 1)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(int(reach.max()) if B else 1, 1)
    assert int(ctx_blocks.sum()) <= num_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_blocks_per_seq), -1, np.int32)
    p = 0
    for b in range(B):
        nb = int(ctx_blocks[b])
        bt[b, :nb] = perm[p:p + nb]
        p += nb
    rest = perm[p:]
    n_held = int(round(held_fraction * num_blocks))
    n_held = min(n_held, rest.shape[0])
    held_idx = np.sort(rng.choice(rest.shape[0], size=n_held, replace=False)) if n_held else np.zeros(0, np.int64)
    keep = np.ones(rest.shape[0], bool)
    keep[held_idx] = False
    held = rest[~keep]
    free = rest[keep]
    free_list = np.full(num_blocks, -1, np.int32)
    free_list[:free.shape[0]] = free

    slab = block_size * head_dim
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    pools = []
    if dtype == "e4m3":
        # fp8 pools: random codes with exponent fields 3..9 and either sign (magnitudes
        # 1/16 .. 7.5), read with scale 1/8; no quantisation happens here
        for which in range(2):
            r = _rng(seed, 2, which)
            codes = (r.integers(0, 2, size=shape) << 7) | (r.integers(3, 10, size=shape) << 3) | \
                r.integers(0, 8, size=shape)
            pools.append(codes.astype(np.uint8))
        return KVState(block_size, num_blocks, max_blocks_per_seq, num_kv_heads, head_dim, dtype,
                       pools[0], pools[1], bt, ctx_lens.copy(), free_list, int(free.shape[0]),
                       held.astype(np.int32), 0.125, 0.125)
    bank = _Bank(seed)
    for which in range(2):
        w = bank.windows(_rng(seed, 2, which), num_blocks * num_kv_heads, slab)
        pools.append(_cast(w.reshape(shape), dtype))
    return KVState(block_size, num_blocks, max_blocks_per_seq, num_kv_heads, head_dim, dtype,
                   pools[0], pools[1], bt, ctx_lens.copy(), free_list, int(free.shape[0]),
                   held.astype(np.int32))


# ----------------------------------------------------------------------------
# one chain step
# ----------------------------------------------------------------------------
def make_chain_step(seed: int, n_q: np.ndarray, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    qkv_dtype: str, vocab: int, logits_dtype: str, target_sigma: float,
                    draft_coef: float, draft_sigma, temperature: float, stream: int = 0,
                    use_bank: bool = True) -> StepInputs:
    """Step inputs for chain drafts. draft = coef * target + N(0, sigma_b^2),
    with sigma_b a scalar or one value per sequence."""
    rng = _rng(seed, 10, stream)
    n_q = np.asarray(n_q, np.int32)
    B = n_q.shape[0]
    cu_q = np.zeros(B + 1, np.int32)
    cu_q[1:] = np.cumsum(n_q)
    Tq = int(cu_q[-1])
    Td = Tq - B
    q = _cast(rng.standard_normal((Tq, num_q_heads, head_dim), dtype=np.float32), qkv_dtype)
    new_k = _cast(rng.standard_normal((Tq, num_kv_heads, head_dim), dtype=np.float32), qkv_dtype)
    new_v = _cast(rng.standard_normal((Tq, num_kv_heads, head_dim), dtype=np.float32), qkv_dtype)

    if use_bank:
        bank = _Bank(seed)
        tgt = bank.windows(_rng(seed, 11, stream), Tq, vocab) * np.float32(target_sigma)
    else:
        tgt = rng.standard_normal((Tq, vocab), dtype=np.float32) * np.float32(target_sigma)
    tgt_c = _cast(tgt, logits_dtype)
    tgt_f = _as_f32(tgt_c, logits_dtype)

    # draft row for (b, i>=1) is the draft distribution of the token at target row i
    seq_of_row = np.repeat(np.arange(B), n_q)
    pos_of_row = np.arange(Tq) - np.repeat(cu_q[:-1], n_q)
    drow_src = np.nonzero(pos_of_row >= 1)[0]  # target rows 1..K_b of every sequence
    # q_i is the draft's distribution for x_i; p_i (target row i-1) scores the same
    # position, so the draft row for x_i is built from target row i-1.
    tgt_for_draft = tgt_f[drow_src - 1]
    sig = np.asarray(draft_sigma, np.float32)
    sig_rows = sig[seq_of_row[drow_src]] if sig.ndim == 1 else np.full(Td, sig, np.float32)
    if use_bank:
        noise = _Bank(seed).windows(_rng(seed, 12, stream), Td, vocab)
    else:
        noise = rng.standard_normal((Td, vocab), dtype=np.float32)
    drf = np.float32(draft_coef) * tgt_for_draft + sig_rows[:, None] * noise
    drf_c = _cast(drf, logits_dtype)
    drf_f = _as_f32(drf_c, logits_dtype)
    draft_tokens = _draft_sample(_rng(seed, 13, stream), drf_f, temperature)
    urng = _rng(seed, 14, stream)
    u_accept = urng.random(Td, dtype=np.float32)
    u_resample = urng.random(B, dtype=np.float32)
    return StepInputs(n_q, cu_q, num_q_heads, q, new_k, new_v, vocab, logits_dtype,
                      tgt_c, drf_c, draft_tokens, u_accept, u_resample, float(temperature))


# ----------------------------------------------------------------------------
# named workloads
# ----------------------------------------------------------------------------
def tiny(seed: int = 0, temperature: float = 1.0) -> Case:
    """4 sequences, contexts {37, 64, 101, 200}, 16-token blocks from a random
    permutation of 64 physical blocks, 4/2 heads of dim 64 in fp32, K = 4 causal,
    vocab 1000, target logits N(0, 2^2), draft = 0.8 target + N(0, 1)."""
    ctx = np.array([37, 64, 101, 200], np.int32)
    n_q = np.full(4, 5, np.int32)
    state = make_kv_state(seed, ctx, block_size=16, num_kv_heads=2, head_dim=64, dtype="f32",
                          num_blocks=64, max_blocks_per_seq=16)
    step = make_chain_step(seed, n_q, num_q_heads=4, num_kv_heads=2, head_dim=64, qkv_dtype="f32",
                           vocab=1000, logits_dtype="f32", target_sigma=2.0, draft_coef=0.8,
                           draft_sigma=1.0, temperature=temperature, use_bank=False)
    return Case("tiny", seed, state, step)


def llama8b(seed: int = 1, temperature: float = 1.0, *, batch: int = 32, ctx_range=(512, 4096),
            K: int = 5, vocab: int = 128256, block_size: int = 16, growth_tokens: int = 0,
            pool_factor: float = 1.25, kv_dtype: str = "bf16") -> Case:
    """Llama-3-8B-shaped: 32 q / 8 kv heads of dim 128, bf16 KV in 16-token blocks
    of a shuffled pool, contexts U[512, 4096], K = 5 causal, vocab 128256, bf16
    target logits N(0, 3^2), draft = 0.8 target + N(0, 1.5^2)."""
    rng = _rng(seed, 20)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=batch).astype(np.int32)
    n_q = np.full(batch, K + 1, np.int32)
    state = make_kv_state(seed, ctx, block_size=block_size, num_kv_heads=8, head_dim=128, dtype=kv_dtype,
                          growth_tokens=K + 1 + growth_tokens, pool_factor=pool_factor)
    step = llama8b_step(seed, 0, batch=batch, K=K, vocab=vocab, temperature=temperature)
    return Case("llama8b", seed, state, step, {"K": K})


def llama8b_step(seed: int, stream: int, *, batch: int = 32, K: int = 5, vocab: int = 128256,
                 temperature: float = 1.0) -> StepInputs:
    """The Llama-8B-shaped step inputs; stream 0 is the workload's own, others are
    further input sets of the same shapes and distributions."""
    return make_chain_step(seed, np.full(batch, K + 1, np.int32), num_q_heads=32, num_kv_heads=8, head_dim=128,
                           qkv_dtype="bf16", vocab=vocab, logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8,
                           draft_sigma=1.5, temperature=temperature, stream=stream)


def llama70b(seed: int = 2, temperature: float = 1.0, *, batch: int = 128, ctx_range=(512, 640),
             K: int = 4, vocab: int = 128256, growth_tokens: int = 0) -> Case:
    """Llama-3-70B-shaped, input-512/output-128: 64 q / 8 kv heads of dim 128,
    bf16 KV in 16-token blocks, 128 sequences with contexts U[512, 640], K = 4,
    vocab 128256, target N(0, 3^2), draft = 0.7 target + N(0, 2^2)."""
    rng = _rng(seed, 20)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=batch).astype(np.int32)
    n_q = np.full(batch, K + 1, np.int32)
    state = make_kv_state(seed, ctx, block_size=16, num_kv_heads=8, head_dim=128, dtype="bf16",
                          growth_tokens=K + 1 + growth_tokens)
    step = llama70b_step(seed, 0, batch=batch, K=K, vocab=vocab, temperature=temperature)
    return Case("llama70b", seed, state, step, {"K": K})


def llama70b_step(seed: int, stream: int, *, batch: int = 128, K: int = 4, vocab: int = 128256,
                  temperature: float = 1.0) -> StepInputs:
    """The Llama-70B-shaped step inputs (stream 0: the workload's own)."""
    return make_chain_step(seed, np.full(batch, K + 1, np.int32), num_q_heads=64, num_kv_heads=8, head_dim=128,
                           qkv_dtype="bf16", vocab=vocab, logits_dtype="bf16", target_sigma=3.0, draft_coef=0.7,
                           draft_sigma=2.0, temperature=temperature, stream=stream)


CONTBATCH_ITERS = 10


def contbatch(seed: int = 3, *, batch: int = 256, vocab: int = 128256, iterations: int = CONTBATCH_ITERS,
              ctx_median: float = 1024.0, ctx_sigma: float = 1.0, ctx_clip=(16, 32768)) -> Case:
    """Continuous-batching mix: 256 sequences, contexts lognormal (median 1024,
    sigma 1) clipped to [16, 32768], 128-token blocks from a fragmented free list
    (30% of the pool held by other sequences), 32/8 heads of dim 128 in bf16,
    vocab 128256, per-sequence draft noise sigma_b ~ U[0.5, 3]. The per-iteration
    inputs (K_b ~ U{2..8} redrawn each iteration) come from `contbatch_step`."""
    rng = _rng(seed, 20)
    ctx = np.exp(np.log(ctx_median) + ctx_sigma * rng.standard_normal(batch))
    ctx = np.clip(np.rint(ctx), ctx_clip[0], ctx_clip[1]).astype(np.int32)
    sigma_b = rng.uniform(0.5, 3.0, size=batch).astype(np.float32)
    state = make_kv_state(seed, ctx, block_size=128, num_kv_heads=8, head_dim=128, dtype="bf16",
                          growth_tokens=9 * iterations, held_fraction=0.3)
    step = contbatch_step(seed, 0, batch=batch, vocab=vocab, sigma_b=sigma_b)
    return Case("contbatch", seed, state, step, {"sigma_b": sigma_b, "iterations": iterations})


def contbatch_step(seed: int, iteration: int, *, batch: int, vocab: int, sigma_b: np.ndarray,
                   temperature: float = 1.0, K: np.ndarray | None = None) -> StepInputs:
    """One iteration's inputs; K_b ~ U{2..8} unless the draft lengths are given
    (e.g. by the adaptive-K controller)."""
    rng = _rng(seed, 30, iteration)
    K_drawn = rng.integers(2, 9, size=batch).astype(np.int32)
    K = K_drawn if K is None else np.asarray(K, dtype=np.int32)
    return make_chain_step(seed, K + 1, num_q_heads=32, num_kv_heads=8, head_dim=128, qkv_dtype="bf16",
                           vocab=vocab, logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8,
                           draft_sigma=sigma_b, temperature=temperature, stream=iteration + 1)


# ----------------------------------------------------------------------------
# draft trees
# ----------------------------------------------------------------------------
def full_tree(branching) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """BFS enumeration of a tree where every node at depth d has branching[d]
    children. Returns parent (node index, -1 for the root), depth and the rank of
    each node among its siblings. Node 0 is the root."""
    parent, depth, rank = [-1], [0], [0]
    frontier = [0]
    for d, k in enumerate(branching):
        nxt = []
        for p in frontier:
            for r in range(k):
                parent.append(p)
                depth.append(d + 1)
                rank.append(r)
                nxt.append(len(parent) - 1)
        frontier = nxt
    return np.array(parent, np.int32), np.array(depth, np.int32), np.array(rank, np.int32)


def tree(seed: int = 5, *, batch: int = 16, ctx: int = 8192, block_size: int = 64,
         branching=(4, 3, 2, 2, 1, 1), keep: int = 60, vocab: int = 32000,
         num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
         target_sigma: float = 3.0, draft_coef: float = 0.8, draft_sigma: float = 1.0,
         temperature: float = 0.0, kv_dtype: str = "bf16", growth_tokens: int = 0) -> Case:
    """EAGLE/Medusa-style draft trees at long context, greedy acceptance (or, at
    temperature > 0, the lossless tree rule with seeded uniforms).

    The drafter expands the full tree `branching` (184 nodes for {4,3,2,2,1,1});
    a node's children carry the top-k tokens of the draft distribution at that
    node (draft = 0.8 target + N(0, 1), softmax at T = 1). The `keep` nodes of
    highest cumulative draft probability are kept (ties to the lower BFS index),
    which keeps every kept node's parent. Query rows: the root (last emitted
    token) and the kept nodes in BFS order, so 61 rows per sequence.
    """
    parent_full, depth_full, rank_full = full_tree(branching)
    n_full = parent_full.shape[0]
    rng = _rng(seed, 40)
    ctx_lens = np.full(batch, ctx, np.int32)
    rows_per_seq = keep + 1
    state = make_kv_state(seed, ctx_lens, block_size=block_size, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, dtype=kv_dtype, growth_tokens=rows_per_seq + growth_tokens)
    bank = _Bank(seed)
    tgt_rows, drf_rows, toks, parents, masks = [], [], [], [], []
    for b in range(batch):
        tgt = bank.windows(_rng(seed, 41, b), n_full, vocab) * np.float32(target_sigma)
        tgt_c = to_bf16_bits(tgt)
        tgt_f = bf16_bits_to_f32(tgt_c)
        noise = bank.windows(_rng(seed, 42, b), n_full, vocab)
        drf_c = to_bf16_bits(np.float32(draft_coef) * tgt_f + np.float32(draft_sigma) * noise)
        drf_f = bf16_bits_to_f32(drf_c).astype(np.float64)
        logq = drf_f - drf_f.max(axis=1, keepdims=True)
        logq = logq - np.log(np.exp(logq).sum(axis=1, keepdims=True))
        token = np.full(n_full, -1, np.int64)
        cum = np.zeros(n_full)
        for v in range(1, n_full):
            p = parent_full[v]
            k = int(rank_full[v])
            order = np.argsort(-logq[p], kind="stable")
            token[v] = order[k]
            cum[v] = cum[p] + logq[p, token[v]]
        cand = np.arange(1, n_full)
        order = sorted(cand.tolist(), key=lambda v: (-cum[v], v))
        kept = sorted(order[:keep])
        kept_set = set(kept)
        assert all(parent_full[v] == 0 or parent_full[v] in kept_set for v in kept)
        full_to_row = {0: 0}
        for r, v in enumerate(kept):
            full_to_row[v] = r + 1
        nodes = [0] + kept
        par = np.array([-1] + [full_to_row[int(parent_full[v])] for v in kept], np.int32)
        mask = np.zeros(rows_per_seq, np.uint64)
        for r in range(rows_per_seq):
            m, a = 0, r
            while a >= 0:
                m |= 1 << a
                a = int(par[a])
            mask[r] = np.uint64(m)
        tgt_rows.append(tgt_c[nodes])
        # the draft row of a node is the draft distribution its token was drawn from
        drf_rows.append(drf_c[[int(parent_full[v]) for v in kept]])
        toks.append(token[kept].astype(np.int32))
        parents.append(par)
        masks.append(mask)
    n_q = np.full(batch, rows_per_seq, np.int32)
    cu_q = np.zeros(batch + 1, np.int32)
    cu_q[1:] = np.cumsum(n_q)
    Tq = int(cu_q[-1])
    q = to_bf16_bits(rng.standard_normal((Tq, num_q_heads, head_dim), dtype=np.float32))
    new_k = to_bf16_bits(rng.standard_normal((Tq, num_kv_heads, head_dim), dtype=np.float32))
    new_v = to_bf16_bits(rng.standard_normal((Tq, num_kv_heads, head_dim), dtype=np.float32))
    urng = _rng(seed, 43)
    u_acc = urng.random(Tq - batch, dtype=np.float32) if temperature > 0 else np.zeros(Tq - batch, np.float32)
    u_res = urng.random(batch, dtype=np.float32) if temperature > 0 else np.zeros(batch, np.float32)
    step = StepInputs(n_q, cu_q, num_q_heads, q, new_k, new_v, vocab, "bf16",
                      np.concatenate(tgt_rows), np.concatenate(drf_rows), np.concatenate(toks),
                      u_acc, u_res, float(temperature),
                      mask_kind="tree", tree_mask=np.concatenate(masks), parent=np.concatenate(parents))
    return Case("tree", seed, state, step, {"branching": tuple(branching), "keep": keep})


def custom(seed: int, *, batch: int, ctx_lens, n_q, num_q_heads: int, num_kv_heads: int, head_dim: int,
           block_size: int, vocab: int, dtype: str = "bf16", temperature: float = 1.0,
           target_sigma: float = 3.0, draft_coef: float = 0.8, draft_sigma=1.5,
           pool_factor: float = 1.25, held_fraction: float = 0.0, growth_tokens: int = 0,
           use_bank: bool = True) -> Case:
    """A chain case with explicit shapes (small parity cases, edge cases)."""
    ctx_lens = np.asarray(ctx_lens, np.int32)
    n_q = np.asarray(n_q, np.int32)
    assert ctx_lens.shape == (batch,) and n_q.shape == (batch,)
    state = make_kv_state(seed, ctx_lens, block_size=block_size, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, dtype=dtype, pool_factor=pool_factor,
                          held_fraction=held_fraction,
                          growth_tokens=int(n_q.max() if batch else 1) + growth_tokens)
    io = "bf16" if dtype == "e4m3" else dtype  # an fp8 pool takes bf16 rows and queries
    step = make_chain_step(seed, n_q, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                           qkv_dtype=io, vocab=vocab, logits_dtype=io, target_sigma=target_sigma,
                           draft_coef=draft_coef, draft_sigma=draft_sigma, temperature=temperature,
                           use_bank=use_bank)
    return Case("custom", seed, state, step)


CONFIGS = {
    "tiny": tiny,
    "llama8b": llama8b,
    "llama70b": llama70b,
    "contbatch": contbatch,
    "tree": tree,
}

"""fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the library never does. It shares
no code with the CUDA path. The arithmetic lives in ``spec_oracle.c`` (plain
fp64 loops, built here with gcc); this module marshals numpy arrays into it
and keeps the KV block bookkeeping as plain Python lists.

Every function is pinned by ``tests/test_oracle_*.py`` against something
other than itself (closed forms, brute force, a library routine, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspec_oracle.so")
_lib = None

_DT = {"bf16": 0, "f32": 1}


def build(force: bool = False) -> str:
    """Compile spec_oracle.c with gcc (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]
        try:  # OpenMP when the compiler has it (results do not depend on the thread count)
            subprocess.check_call(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.so_dense_attention.argtypes = [I, I, I, I, I, I, P, P, P, I, P, D, P]
        lib.so_paged_attention.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, I, P, I, I, P, D, P, I, P]
        lib.so_rejection_sample.argtypes = [I, I, P, P, P, I, P, P, P, D, I, P, P, P, P, P]
        lib.so_tree_greedy.argtypes = [I, I, P, P, I, P, P, I, P, P, P, P]
        lib.so_tree_sample.argtypes = [I, I, P, P, I, P, P, P, P, D, I, P, P, P, P, P, P]
        lib.so_set_threads.argtypes = [I]
        lib.so_set_threads.restype = I
        for f in (lib.so_dense_attention, lib.so_paged_attention, lib.so_rejection_sample, lib.so_tree_greedy,
                  lib.so_tree_sample):
            f.restype = I
        _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Threads of the oracle's parallel loops (OpenMP); returns the count in use.
    Values do not depend on it."""
    return int(_load().so_set_threads(int(n)))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype) if dtype is not None else np.ascontiguousarray(a)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what}: oracle error {rc}")


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def dense_attention(k: np.ndarray, v: np.ndarray, q: np.ndarray, ctx: int, *, mask_kind: str = "causal",
                    tree_mask: np.ndarray | None = None, scale: float) -> np.ndarray:
    """k, v [L, Hkv, D] and q [n, Hq, D] as float64; L = ctx + n."""
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    q = _c(q, np.float64)
    L, hkv, d = k.shape
    n, hq, _ = q.shape
    out = np.zeros((n, hq, d), np.float64)
    tm = _c(tree_mask, np.uint64) if tree_mask is not None else None
    rc = _load().so_dense_attention(L, ctx, n, hq, hkv, d, _p(k), _p(v), _p(q),
                                    0 if mask_kind == "causal" else 1, _p(tm), scale, _p(out))
    _check(rc, "dense_attention")
    return out


def paged_attention(state, step, *, seqs=None, out: np.ndarray | None = None) -> np.ndarray:
    """Attention of every query row over its sequence's KV, read through the
    block table. `state` must already hold the step's new rows (see
    OracleKV.append). Returns [T_q, Hq, D] float64 (rows of sequences not in
    `seqs` are zero / untouched)."""
    if state.k_pool is None or state.v_pool is None:
        raise ValueError("paged_attention needs a state with K/V pools (OracleKV(..., with_pools=True))")
    if state.dtype == "e4m3":  # fp8 pool: every code read as its E4M3 value times the pool's scale
        from copy import copy
        from . import fp8
        st = copy(state)
        st.k_pool = (fp8.decode(state.k_pool) * float(np.float32(state.k_scale))).astype(np.float32)
        st.v_pool = (fp8.decode(state.v_pool) * float(np.float32(state.v_scale))).astype(np.float32)
        st.dtype = "f32"
        state = st
    Tq = step.total_q
    hq = step.num_q_heads
    d = state.head_dim
    if out is None:
        out = np.zeros((Tq, hq, d), np.float64)
    sl = None if seqs is None else np.ascontiguousarray(seqs, np.int32)
    kp, vp = _c(state.k_pool), _c(state.v_pool)
    q = _c(step.q)
    q_dtype = "bf16" if q.dtype == np.uint16 else "f32"  # bf16 arrays hold bit patterns; an fp8 pool takes bf16 Q
    tm = _c(step.tree_mask, np.uint64) if step.tree_mask is not None else None
    rc = _load().so_paged_attention(
        state.batch, hq, state.num_kv_heads, d, state.block_size, state.max_blocks_per_seq,
        state.num_blocks, _p(_c(state.seq_lens, np.int32)), _p(_c(step.cu_q, np.int32)),
        _p(_c(state.block_table, np.int32)), _p(kp), _p(vp), _DT[state.dtype], _p(q),
        _DT[q_dtype], 0 if step.mask_kind == "causal" else 1, _p(tm), float(step.scale),
        _p(sl), 0 if sl is None else int(sl.shape[0]), _p(out))
    _check(rc, "paged_attention")
    return out


# ----------------------------------------------------------------------------
# sampler
# ----------------------------------------------------------------------------
@dataclass
class SampleResult:
    accept_cnt: np.ndarray
    out_tok: np.ndarray
    num_out: np.ndarray
    margin: np.ndarray | None = None
    fallback: np.ndarray | None = None
    path_nodes: np.ndarray | None = None


def rejection_sample(step, *, temperature: float | None = None, max_q: int | None = None) -> SampleResult:
    T = step.temperature if temperature is None else temperature
    B = step.n_q.shape[0]
    mq = step.max_q if max_q is None else max_q
    acc = np.zeros(B, np.int32)
    out_tok = np.full((B, mq), -1, np.int32)
    num = np.zeros(B, np.int32)
    marg = np.zeros(B, np.float64)
    fb = np.zeros(B, np.int32)
    tgt = _c(step.target_logits)
    drf = _c(step.draft_logits)
    rc = _load().so_rejection_sample(
        B, step.vocab, _p(_c(step.cu_q, np.int32)), _p(tgt), _p(drf), _DT[step.logits_dtype],
        _p(_c(step.draft_tokens, np.int32)), _p(_c(step.u_accept, np.float32)),
        _p(_c(step.u_resample, np.float32)), float(T), mq, _p(acc), _p(out_tok), _p(num), _p(marg), _p(fb))
    _check(rc, "rejection_sample")
    return SampleResult(acc, out_tok, num, marg, fb)


def tree_greedy(step, *, max_q: int | None = None) -> SampleResult:
    B = step.n_q.shape[0]
    mq = step.max_q if max_q is None else max_q
    acc = np.zeros(B, np.int32)
    path = np.full((B, mq), -1, np.int32)
    out_tok = np.full((B, mq), -1, np.int32)
    num = np.zeros(B, np.int32)
    rc = _load().so_tree_greedy(B, step.vocab, _p(_c(step.cu_q, np.int32)), _p(_c(step.target_logits)),
                                _DT[step.logits_dtype], _p(_c(step.draft_tokens, np.int32)),
                                _p(_c(step.parent, np.int32)), mq, _p(acc), _p(path), _p(out_tok), _p(num))
    _check(rc, "tree_greedy")
    return SampleResult(acc, out_tok, num, path_nodes=path)


def tree_sample(step, *, temperature: float | None = None, max_q: int | None = None) -> SampleResult:
    """Lossless tree verification at T > 0 (see so_tree_sample for the reading)."""
    T = step.temperature if temperature is None else temperature
    B = step.n_q.shape[0]
    mq = step.max_q if max_q is None else max_q
    acc = np.zeros(B, np.int32)
    path = np.full((B, mq), -1, np.int32)
    out_tok = np.full((B, mq), -1, np.int32)
    num = np.zeros(B, np.int32)
    marg = np.zeros(B, np.float64)
    fb = np.zeros(B, np.int32)
    rc = _load().so_tree_sample(B, step.vocab, _p(_c(step.cu_q, np.int32)), _p(_c(step.target_logits)),
                                _DT[step.logits_dtype], _p(_c(step.draft_tokens, np.int32)),
                                _p(_c(step.parent, np.int32)), _p(_c(step.u_accept, np.float32)),
                                _p(_c(step.u_resample, np.float32)), float(T), mq, _p(acc), _p(path), _p(out_tok),
                                _p(num), _p(marg), _p(fb))
    _check(rc, "tree_sample")
    return SampleResult(acc, out_tok, num, marg, fb, path_nodes=path)


# ----------------------------------------------------------------------------
# KV block bookkeeping (plain Python lists)
# ----------------------------------------------------------------------------
OUT_OF_BLOCKS = "out_of_blocks"
NO_TABLE_ROOM = "no_table_room"
BAD_LENGTH = "bad_length"


class OracleKV:
    """The paged cache as Python lists, following the pages' block manager:
    a sequence's logical blocks map to physical blocks through its block table
    ("LLM serving: speculative decoding and PagedAttention memory management",
    PagedAttention section); a new physical block is taken only when the
    current one is full (same section, on-demand allocation); rejected
    positions are given back a whole block at a time and accepted entries stay
    where they are ("Speculative decoding principles and a vLLM production
    setup", sec. 3.1).

    Free blocks form a LIFO stack (the free list's last element is its top).
    Reading taken where the pages are silent: append pops in (sequence,
    logical block) order; rollback pushes in sequence order, highest logical
    block first.
    """

    def __init__(self, state, with_pools: bool = True):
        self.bs = state.block_size
        self.num_blocks = state.num_blocks
        self.max_blocks = state.max_blocks_per_seq
        self.bt = [list(map(int, row)) for row in state.block_table]
        self.seq_lens = list(map(int, state.seq_lens))
        self.free = list(map(int, state.free_list[:state.free_top]))
        self.k_pool = state.k_pool.copy() if with_pools else None
        self.v_pool = state.v_pool.copy() if with_pools else None
        self._state = state
        self.ref = None  # per-block reference counts once sharing is on

    # ---- copy-on-write sharing ("LLM serving: speculative decoding and
    # PagedAttention memory management", PagedAttention section: parent and
    # child sequences of beam search / parallel sampling share physical blocks
    # copy-on-write). Reading taken: a block's count is the number of block-table
    # entries that hold it; a sequence about to write into a block whose count is
    # above one first takes a private copy of it (a fresh block, popped before its
    # new blocks) holding the rows written so far; a block goes back on the free
    # list when its count drops to zero.
    def enable_sharing(self, ref=None) -> None:
        if ref is None:
            ref = [0] * self.num_blocks
            for row, n in zip(self.bt, self.seq_lens):
                for lb in range(self._blocks(n, self.bs)):
                    ref[row[lb]] += 1
        self.ref = [int(x) for x in ref]

    def ref_count(self) -> np.ndarray:
        return np.array(self.ref, np.int32)

    def fork(self, parents, children):
        """Each child sequence slot (empty) takes its parent's blocks and length;
        every shared block's count goes up by one. All or nothing."""
        assert self.ref is not None
        B = len(self.seq_lens)
        ps, cs = [int(x) for x in parents], [int(x) for x in children]
        if (len(set(cs)) != len(cs) or set(cs) & set(ps)
                or any(not (0 <= x < B) for x in ps + cs)
                or any(self.seq_lens[c] != 0 or any(e != -1 for e in self.bt[c]) for c in cs)):
            return BAD_LENGTH
        for p_, c in zip(ps, cs):
            nb = self._blocks(self.seq_lens[p_], self.bs)
            for lb in range(nb):
                self.bt[c][lb] = self.bt[p_][lb]
                self.ref[self.bt[p_][lb]] += 1
            self.seq_lens[c] = self.seq_lens[p_]
        return None

    def release(self, seqs):
        """Drop finished sequences: in the order given, blocks from the highest
        logical one down lose one reference (every block, without sharing) and go
        back on the free list at zero; the slot becomes empty."""
        B = len(self.seq_lens)
        ss = [int(x) for x in seqs]
        if len(set(ss)) != len(ss) or any(not (0 <= x < B) for x in ss):
            return BAD_LENGTH
        for b in ss:
            for lb in range(self._blocks(self.seq_lens[b], self.bs) - 1, -1, -1):
                blk = self.bt[b][lb]
                if self.ref is not None:
                    self.ref[blk] -= 1
                if self.ref is None or self.ref[blk] == 0:
                    self.free.append(blk)
                self.bt[b][lb] = -1
            self.seq_lens[b] = 0
        return None

    @staticmethod
    def _blocks(tokens: int, bs: int) -> int:
        return (tokens + bs - 1) // bs

    def append(self, step):
        """Give each sequence the blocks its n_b new rows need, then write row j
        of sequence b at logical position c_b + j. All or nothing."""
        B = len(self.seq_lens)
        n = [int(step.cu_q[b + 1] - step.cu_q[b]) for b in range(B)]
        need = [self._blocks(self.seq_lens[b] + n[b], self.bs) - self._blocks(self.seq_lens[b], self.bs)
                for b in range(B)]
        # copy-on-write: the first new row lands in a partly filled block that is
        # still shared when this sequence's turn comes (sequences in order; each
        # copy drops the block's count by one, so the last writer of a block no
        # other sequence holds writes in place)
        cow = [False] * B
        if self.ref is not None:
            left = {}
            for b in range(B):
                if n[b] > 0 and self.seq_lens[b] % self.bs != 0:
                    blk = self.bt[b][self.seq_lens[b] // self.bs]
                    r = left.get(blk, self.ref[blk])
                    if r > 1:
                        cow[b] = True
                        left[blk] = r - 1
        if any(self._blocks(self.seq_lens[b] + n[b], self.bs) > self.max_blocks for b in range(B)):
            return NO_TABLE_ROOM
        if sum(need) + sum(cow) > len(self.free):
            return OUT_OF_BLOCKS
        for b in range(B):
            first = self._blocks(self.seq_lens[b], self.bs)
            if cow[b]:
                lb = self.seq_lens[b] // self.bs
                old, new = self.bt[b][lb], self.free.pop()
                if self.k_pool is not None:
                    used = self.seq_lens[b] % self.bs
                    self.k_pool[new, :, :used, :] = self.k_pool[old, :, :used, :]
                    self.v_pool[new, :, :used, :] = self.v_pool[old, :, :used, :]
                self.ref[old] -= 1
                self.ref[new] = 1
                self.bt[b][lb] = new
            for j in range(need[b]):
                self.bt[b][first + j] = self.free.pop()
                if self.ref is not None:
                    self.ref[self.bt[b][first + j]] = 1
        if self.k_pool is not None:
            new_k, new_v = step.new_k, step.new_v
            if self._state.dtype == "e4m3":
                # fp8 pool: the E4M3 code nearest to x / scale, x the bf16 input (fp32 division)
                from . import fp8
                wid = lambda a: (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)
                new_k = fp8.encode(wid(new_k) / np.float32(self._state.k_scale))
                new_v = fp8.encode(wid(new_v) / np.float32(self._state.v_scale))
            for b in range(B):
                for j in range(n[b]):
                    pos = self.seq_lens[b] + j
                    blk = self.bt[b][pos // self.bs]
                    row = int(step.cu_q[b]) + j
                    self.k_pool[blk, :, pos % self.bs, :] = new_k[row]
                    self.v_pool[blk, :, pos % self.bs, :] = new_v[row]
        return None

    def rollback(self, step, accept_cnt, path_nodes=None):
        """Keep the last emitted token and the a_b accepted rows: the new length
        is c_b + a_b + 1. Tree drafts first move the accepted path's rows to
        slots c_b+1 .. c_b+a_b, in path order. Whole blocks past the new end go
        back on the free list."""
        B = len(self.seq_lens)
        for b in range(B):
            c = self.seq_lens[b]
            n = int(step.cu_q[b + 1] - step.cu_q[b])
            a = int(accept_cnt[b])
            assert 0 <= a <= n - 1
            if path_nodes is not None and self.k_pool is not None:
                for j in range(1, a + 1):
                    src = c + int(path_nodes[b][j - 1])
                    dst = c + j
                    sb, db = self.bt[b][src // self.bs], self.bt[b][dst // self.bs]
                    self.k_pool[db, :, dst % self.bs, :] = self.k_pool[sb, :, src % self.bs, :]
                    self.v_pool[db, :, dst % self.bs, :] = self.v_pool[sb, :, src % self.bs, :]
            new_len = c + a + 1
            old_blocks = self._blocks(c + n, self.bs)
            keep = self._blocks(new_len, self.bs)
            for lb in range(old_blocks - 1, keep - 1, -1):
                blk = self.bt[b][lb]
                if self.ref is not None:
                    self.ref[blk] -= 1
                if self.ref is None or self.ref[blk] == 0:
                    self.free.append(blk)
                self.bt[b][lb] = -1
            self.seq_lens[b] = new_len

    # views in the library's array layout
    def block_table(self) -> np.ndarray:
        return np.array(self.bt, np.int32).reshape(len(self.bt), self.max_blocks)

    def free_list(self) -> np.ndarray:
        out = np.full(self.num_blocks, -1, np.int32)
        out[:len(self.free)] = self.free
        return out

    def as_state(self):
        """A KVState holding the oracle's current cache (for feeding the oracle's
        own attention)."""
        s = self._state
        from copy import copy
        st = copy(s)
        st.k_pool = self.k_pool
        st.v_pool = self.v_pool
        st.block_table = self.block_table()
        st.seq_lens = np.array(self.seq_lens, np.int32)
        st.free_list = self.free_list()
        st.free_top = len(self.free)
        return st

    def attention_state(self, step):
        """State for the step's attention: the cache after append, with the step's
        lengths c_b (the new rows are counted through cu_q)."""
        return self.as_state()

"""Pins of the oracle's copy-on-write block sharing ("LLM serving: speculative
decoding and PagedAttention memory management", PagedAttention section:
parent and child sequences of beam search or parallel sampling share
physical blocks copy-on-write).

Checked here: a hand-worked example (fork, the private copy on the first
write into a shared partial block, release), and, over random fork / append /
rollback / release sequences, a model without sharing: every sequence keeps
its own list of rows, and reading a sequence through the oracle's block table
must give exactly that list; every block's count equals the number of
block-table entries holding it, and free, held and referenced blocks
partition the pool.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_paged_gb300 import workloads as W

from test_oracle_kv import _state, _step


def test_hand_worked_fork_copy_release():
    # block size 4; seq 0 holds 6 tokens in blocks [7, 2]; seq 1 is empty.
    # free stack (bottom..top): 5, 0, 9, 3
    st = _state([6, 0], 4, 10, [5, 0, 9, 3], [[7, 2], []])
    kv = oracle.OracleKV(st)
    kv.k_pool[7, 0, :, 0] = [1, 2, 3, 4]
    kv.k_pool[2, 0, :2, 0] = [5, 6]
    kv.enable_sharing()
    assert kv.ref[7] == 1 and kv.ref[2] == 1
    assert kv.fork([0], [1]) is None
    assert kv.bt[1][:3] == [7, 2, -1] and kv.seq_lens[1] == 6
    assert kv.ref[7] == 2 and kv.ref[2] == 2
    # both write one row at position 6, inside shared block 2: seq 0 (first in
    # order) takes a private copy (pop 3) holding rows 4, 5; seq 1 then holds the
    # only reference to block 2 and writes in place
    step = _step([1, 1])
    assert kv.append(step) is None
    assert kv.bt[0][:2] == [7, 3] and kv.bt[1][:2] == [7, 2]
    assert kv.ref[2] == 1 and kv.ref[3] == 1 and kv.ref[7] == 2
    assert list(kv.k_pool[3, 0, :3, 0]) == [5, 6, 100]
    assert list(kv.k_pool[2, 0, :3, 0]) == [5, 6, 101]
    assert kv.free == [5, 0, 9]
    kv.rollback(step, [0, 0])  # keep the row each wrote: lengths 7
    assert kv.seq_lens == [7, 7] and kv.free == [5, 0, 9]
    # release seq 0: block 3 (count 1 -> 0) goes back, block 7 (2 -> 1) stays
    assert kv.release([0]) is None
    assert kv.free == [5, 0, 9, 3] and kv.ref[7] == 1 and kv.seq_lens[0] == 0
    assert kv.bt[0][:2] == [-1, -1]


def test_three_sharers_two_writers_both_copy():
    # a block held by three sequences, two of which write: both copy (pops 3, 9)
    st = _state([6, 0, 0], 4, 10, [5, 0, 9, 3], [[7, 2], [], []])
    kv = oracle.OracleKV(st)
    kv.enable_sharing()
    assert kv.fork([0, 0], [1, 2]) is None
    assert kv.ref[2] == 3
    assert kv.append(_step([1, 1, 1])) is None
    assert [kv.bt[b][1] for b in range(3)] == [3, 9, 2] and kv.ref[2] == 1


def test_fork_refusals_change_nothing():
    st = _state([6, 0, 3], 4, 12, [5, 0, 9, 3], [[7, 2], [], [4]])
    kv = oracle.OracleKV(st)
    kv.enable_sharing()
    before = ([r[:] for r in kv.bt], kv.seq_lens[:], kv.ref[:])
    assert kv.fork([0], [2]) == oracle.BAD_LENGTH  # child not empty
    assert kv.fork([0, 0], [1, 1]) == oracle.BAD_LENGTH  # the same child twice
    assert kv.fork([0, 1], [1, 2]) == oracle.BAD_LENGTH  # a child is also a parent
    assert kv.fork([1], [1]) == oracle.BAD_LENGTH
    assert kv.release([0, 0]) == oracle.BAD_LENGTH
    assert ([r[:] for r in kv.bt], kv.seq_lens[:], kv.ref[:]) == before


def test_copy_needs_a_free_block():
    # the private copy counts against the free list: all or nothing
    st = _state([6, 0], 4, 3, [], [[0, 1], []], max_blocks=4)
    kv = oracle.OracleKV(st)
    kv.enable_sharing()
    assert kv.fork([0], [1]) is None
    assert kv.append(_step([1, 1])) == oracle.OUT_OF_BLOCKS
    assert kv.bt[1][:2] == [0, 1] and kv.ref[1] == 2


def _read_rows(kv, b):
    return [kv.k_pool[kv.bt[b][pos // kv.bs], 0, pos % kv.bs, 0] for pos in range(kv.seq_lens[b])]


def _check_invariants(kv, held):
    refs = [0] * kv.num_blocks
    for b in range(len(kv.seq_lens)):
        for lb in range(kv.max_blocks):
            e = kv.bt[b][lb]
            if lb < kv._blocks(kv.seq_lens[b], kv.bs):
                refs[e] += 1
            else:
                assert e == -1
    assert refs == kv.ref
    free = set(kv.free)
    assert len(free) == len(kv.free)
    used = {i for i, r in enumerate(refs) if r > 0}
    assert not (free & used) and not (free & held) and not (used & held)
    assert free | used | held == set(range(kv.num_blocks))


@pytest.mark.parametrize("seed", range(4))
def test_sharing_matches_private_copies(seed):
    rng = np.random.default_rng(seed)
    B, bs, nblk = 8, 4, 160
    ctx = [int(x) for x in rng.integers(1, 14, size=4)] + [0] * 4
    perm = rng.permutation(nblk).astype(np.int32)
    rows, p = [], 0
    for c in ctx:
        k = (c + bs - 1) // bs
        rows.append(list(perm[p:p + k]))
        p += k
    st = _state(ctx, bs, nblk, list(perm[p:]), rows, max_blocks=16)
    kv = oracle.OracleKV(st)
    for b, c in enumerate(ctx):  # distinct values in every context row
        for pos in range(c):
            kv.k_pool[kv.bt[b][pos // bs], 0, pos % bs, 0] = 1000.0 * (b + 1) + pos
    kv.enable_sharing()
    model = [_read_rows(kv, b) for b in range(B)]
    tag = 10000.0
    forks = copies = 0
    for it in range(80):
        op = rng.integers(0, 3)
        if op == 0:  # fork a non-empty sequence into an empty slot
            empty = [b for b in range(B) if kv.seq_lens[b] == 0]
            full = [b for b in range(B) if kv.seq_lens[b] > 0]
            if not empty or not full:
                continue
            par, ch = int(rng.choice(full)), int(rng.choice(empty))
            assert kv.fork([par], [ch]) is None
            model[ch] = list(model[par])
            forks += 1
        elif op == 1:  # a verify step: every slot appends n_b rows and keeps a_b + 1 of them
            for b in range(B):  # keep within the table
                if kv.seq_lens[b] > 48:
                    assert kv.release([b]) is None
                    model[b] = []
            n = [int(rng.integers(1, 5)) for _ in range(B)]
            # every sequence writes: each shared partial block held by r sequences
            # is copied r - 1 times
            held = {}
            for b in range(B):
                if kv.seq_lens[b] % bs:
                    blk = kv.bt[b][kv.seq_lens[b] // bs]
                    held[blk] = kv.ref[blk]
            shared_partial = sum(r - 1 for r in held.values())
            step = _step(n, start=tag)
            tag += 1000.0
            free_before = len(kv.free)
            assert kv.append(step) is None
            grow = sum(kv._blocks(kv.seq_lens[b] + n[b], bs) - kv._blocks(kv.seq_lens[b], bs) for b in range(B))
            assert free_before - len(kv.free) == grow + shared_partial  # one private copy per shared partial block
            copies += shared_partial
            acc = [int(rng.integers(0, x)) for x in n]
            kv.rollback(step, acc)
            cu = step.cu_q
            for b in range(B):
                model[b] += [step.new_k[cu[b] + j, 0, 0] for j in range(acc[b] + 1)]
        else:  # release one sequence
            full = [b for b in range(B) if kv.seq_lens[b] > 0]
            if len(full) <= 1:
                continue
            b = int(rng.choice(full))
            assert kv.release([b]) is None
            model[b] = []
        _check_invariants(kv, set())
        for b in range(B):
            assert _read_rows(kv, b) == model[b]
    assert forks >= 3 and copies > 0

"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side argument checks answer without touching a GPU; the oracle
and the library share no code."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(sv_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sv_kv_append", "sv_spec_verify_attn", "sv_kv_rollback", "sv_spec_rejection_sample"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(sv_\w+)$", out, flags=re.M))
    assert exported == _declared() | set(L.EXPORTS)


def test_status_strings_and_version(lib):
    assert lib.sv_version() >= 10000
    for code, name in L.STATUS_NAMES.items():
        assert L.status_string(code).startswith(name)


def test_host_validation_without_gpu(lib):
    s = L.sv_paged_kv()
    # NULL cache, bad block size, missing status word: rejected on the host
    assert lib.sv_kv_append(None, None, None, None, 0, None, None) == 1
    s.block_size, s.head_dim, s.num_kv_heads, s.num_blocks, s.max_blocks_per_seq = 3, 128, 8, 16, 4
    assert lib.sv_kv_rollback(ctypes.byref(s), None, None, None, 6, None, None) == 1
    assert lib.sv_spec_rejection_sample(None, None, 7, 100, 1, None, 2, 2, None, None, None, 1.0,
                                        None, None, None, None, None, 0, None, None) == 1
    assert lib.sv_spec_rejection_sample(None, None, 0, 100, 1, None, 2, 2, None, None, None, float("nan"),
                                        None, None, None, None, None, 0, None, None) == 1
    # the sampler's workspace: 32 KB items x 8 warps x (max, sum); target (+ draft) rows
    assert lib.sv_spec_rejection_sample_workspace_bytes(0, 128256, 32, 256, 1.0) == (2 * 256 - 32) * 8 * 64
    assert lib.sv_spec_rejection_sample_workspace_bytes(0, 128256, 32, 256, 0.0) == 256 * 8 * 64
    assert lib.sv_spec_rejection_sample_workspace_bytes(1, 8192, 1, 1, 0.0) == 64
    assert lib.sv_spec_rejection_sample_workspace_bytes(7, 100, 1, 2, 1.0) == 0
    assert lib.sv_spec_rejection_sample_workspace_bytes(0, 100, 3, 2, 1.0) == 0
    # a workspace that is missing: refused on the host before anything is read
    fake = ctypes.c_void_p(256)
    assert lib.sv_spec_rejection_sample(fake, fake, 0, 100, 1, fake, 2, 2, fake, fake, fake, 1.0,
                                        fake, fake, fake, None, None, 0, None, None) == 10
    assert lib.sv_tree_greedy_accept(fake, 0, 100, 1, fake, 2, 2, fake, fake, fake, fake, fake, fake,
                                     ctypes.c_void_p(512), 16, None, None) == 10


def test_oracle_and_library_share_no_code():
    pkg = os.path.join(ROOT, "speculative_decoding_verify_paged_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            text = open(path).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), path
            assert "spec_oracle" not in text, path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*")):
        if path.endswith((".py", ".c", ".h")):
            text = open(path).read()
            assert "speculative_decoding_verify_paged_gb300" not in text, path
            assert "spec_verify.h" not in text, path


def test_no_alloc_scratch_size_matches_the_header():
    """The binding's copy of SV_ATTN_NO_ALLOC_SCRATCH_BYTES is the header's value."""
    text = open(os.path.join(ROOT, "include", "spec_verify.h")).read()
    m = re.search(r"#define\s+SV_ATTN_NO_ALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "SV_ATTN_NO_ALLOC_SCRATCH_BYTES not found in the header"
    assert L.ATTN_NO_ALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_no_alloc_refusals_on_the_host(lib):
    """sv_spec_verify_attn_no_alloc checks its arguments before any CUDA call:
    a NULL cache and an empty batch answer here, where there is no GPU."""
    assert lib.sv_spec_verify_attn_no_alloc(None, None, None, None, 8, 4, 4, 64, 0.1, 0, None, None, None) == 1
    s = L.sv_paged_kv()
    s.num_blocks, s.block_size, s.max_blocks_per_seq, s.num_kv_heads, s.head_dim, s.batch = 16, 16, 4, 2, 128, 0
    s.k_pool = s.v_pool = 256  # never read: nothing is launched for an empty batch
    assert lib.sv_spec_verify_attn_no_alloc(ctypes.byref(s), None, None, None, 8, 0, 4, 64, 0.1, 0, None, None,
                                            None) == 0


def test_failure_options_are_checked(lib):
    """The wait budget takes 1 ms .. 2 s (in microseconds); the stall hook three values."""
    for bad in (0, 999, 2_000_001, -5):
        assert lib.sv_set_option(L.SV_OPT_WAIT_BUDGET_US, bad) == L.SV_ERR_INVALID_ARG
    assert lib.sv_set_option(L.SV_OPT_STALL_FOR_TEST, 3) == L.SV_ERR_INVALID_ARG
    assert lib.sv_set_option(L.SV_OPT_STALL_FOR_TEST, -1) == L.SV_ERR_INVALID_ARG
    assert lib.sv_set_option(99, 0) == L.SV_ERR_INVALID_ARG
    assert lib.sv_set_option(L.SV_OPT_WAIT_BUDGET_US, 1000) == 0
    assert lib.sv_set_option(L.SV_OPT_WAIT_BUDGET_US, L.DEFAULT_WAIT_BUDGET_US) == 0
    assert lib.sv_set_option(L.SV_OPT_STALL_FOR_TEST, 0) == 0

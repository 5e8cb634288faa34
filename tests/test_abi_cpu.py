"""Host-side checks of the C ABI library: it builds, loads, exports every declared symbol, and
its pure host functions behave.  No compute call is made (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_verify_gb300 import _build, binding

HEADER = os.path.join(_build.ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("spec_verify_greedy", "spec_verify_rejection", "spec_verify_tree", "spec_verify_block",
              "spec_verify_workspace_bytes", "spec_verify_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_workspace_bytes(lib):
    ws = binding.spec_verify_workspace_bytes
    assert ws(binding.MODE_REJECTION, 64, 7, 128256) > 0
    assert ws(binding.MODE_REJECTION, 128, 7, 128256) >= ws(binding.MODE_REJECTION, 64, 7, 128256)
    assert ws(binding.MODE_GREEDY, 1, 0, 1) > 0
    assert ws(binding.MODE_TREE, 48, 8, 151936) > 0
    assert ws(binding.MODE_TREE, 48, 65, 151936) == 0  # more than 64 nodes
    assert ws(binding.MODE_REJECTION, 4, 64, 100) == 0  # k + 1 > 64
    assert ws(binding.MODE_REJECTION, 0, 3, 100) == 0
    assert ws(7, 4, 3, 100) == 0
    assert ws(binding.MODE_REJECTION, 4, 3, 100) % 256 == 0
    # Block verification adds per-row pending state and per-(row, chunk, warp) sums.
    assert ws(binding.MODE_BLOCK, 64, 7, 128256) > ws(binding.MODE_REJECTION, 64, 7, 128256)
    assert ws(binding.MODE_BLOCK, 4, 64, 100) == 0


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, 1, 2, 3, 4, 5, 6, 12345):
        s = binding.spec_verify_strerror(code)
        assert isinstance(s, str) and s


def test_invalid_arguments_are_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails its host checks first
    ws = ctypes.create_string_buffer(512)  # host memory; also never reached
    n = ctypes.c_size_t(1 << 30)
    assert lib.spec_verify_greedy(fake, 0, fake, 0, 3, 100, fake, fake, fake, n, None, None) == -1
    assert lib.spec_verify_greedy(None, 0, fake, 4, 3, 100, fake, fake, fake, n, None, None) == -1
    assert lib.spec_verify_greedy(fake, 7, fake, 4, 3, 100, fake, fake, fake, n, None, None) == -1
    assert lib.spec_verify_greedy(P(0x10001), 0, fake, 4, 3, 100, fake, fake, fake, n, None, None) == -1
    assert lib.spec_verify_rejection(fake, 0, fake, None, 4, 3, 100, 0.0, 1, 0, fake, fake, None,
                                     fake, n, None, None) == -1
    assert lib.spec_verify_rejection(fake, 0, fake, None, 4, 3, 100, float("nan"), 1, 0, fake,
                                     fake, None, fake, n, None, None) == -1
    assert lib.spec_verify_rejection(fake, 0, fake, None, 4, 64, 100, 1.0, 1, 0, fake, fake, None,
                                     fake, n, None, None) == -1
    assert lib.spec_verify_block(fake, 0, fake, None, 4, 3, 100, 0.0, 1, 0, fake, fake, fake, n,
                                 None, None) == -1
    assert lib.spec_verify_block(fake, 0, fake, None, 4, 64, 100, 1.0, 1, 0, fake, fake, fake, n,
                                 None, None) == -1
    assert lib.spec_verify_block(fake, 0, fake, P(0x10002), 4, 3, 100, 1.0, 1, 0, fake, fake, fake,
                                 n, None, None) == -1
    assert lib.spec_verify_block(fake, 0, fake, None, 4, 3, 100, 1.0, 1, 0, fake, fake, fake,
                                 ctypes.c_size_t(16), None, None) == -2
    assert lib.spec_verify_tree(fake, 0, fake, fake, 4, 8, 100, 2, 1.0, 1, 0, fake, fake, fake,
                                fake, n, None, None) == -1
    assert lib.spec_verify_tree(fake, 0, fake, fake, 4, 65, 100, 1, 1.0, 1, 0, fake, fake, fake,
                                fake, n, None, None) == -1
    # workspace too small / misaligned
    assert lib.spec_verify_greedy(fake, 0, fake, 4, 3, 100, fake, fake, fake, ctypes.c_size_t(16),
                                  None, None) == -2
    assert lib.spec_verify_greedy(fake, 0, fake, 4, 3, 100, fake, fake, P(0x10008), n, None,
                                  None) == -2
    assert lib.spec_verify_philox(1, 0, 0, 4, fake, None) == -1
    # Options: thresholds outside (0, 1], thresholds with draft probabilities, bad temperature.
    Opt = binding.Options
    for bad in (Opt(None, 1.0, 0.0, 1.0), Opt(None, 1.0, 1.0, 1.5), Opt(None, -1.0, 1.0, 1.0),
                Opt(None, float("nan"), 1.0, 1.0), Opt(0x10002, 1.0, 1.0, 1.0),
                Opt(None, 1.0, 1.0, 1.0, 0x10002, None), Opt(None, 1.0, 1.0, 1.0, None, 0x10001)):
        assert lib.spec_verify_rejection_ex(fake, 0, fake, None, 4, 3, 100, ctypes.byref(bad), 1, 0,
                                            fake, fake, None, fake, n, None, None) == -1
        assert lib.spec_verify_tree_ex(fake, 0, fake, fake, 4, 8, 100, ctypes.byref(bad), 1, 0, fake,
                                       fake, fake, fake, n, None, None) == -1
    relaxed = Opt(None, 1.0, 0.5, 1.0)
    assert lib.spec_verify_rejection_ex(fake, 0, fake, fake, 4, 3, 100, ctypes.byref(relaxed), 1, 0,
                                        fake, fake, None, fake, n, None, None) == -1
    assert lib.spec_verify_rejection_ex(fake, 0, fake, None, 4, 3, 100, None, 1, 0, fake, fake, None,
                                        fake, n, None, None) == -1
    # Budget planner: (conf, num_drafts, B, K, cost, admitted, budget, best_rate, stream)
    pb = lib.spec_verify_plan_budget
    assert pb(None, None, 4, 7, fake, fake, fake, None, fake, n, None) == -1
    assert pb(fake, None, 4, 65, fake, fake, fake, None, fake, n, None) == -1
    assert pb(fake, None, 2341, 7, fake, fake, fake, None, fake, n, None) == -1  # 16387 slots
    assert pb(fake, None, 0, 7, fake, fake, fake, None, fake, n, None) == -1
    assert pb(fake, None, 4, 7, P(0x10004), fake, fake, None, fake, n, None) == -1  # cost not 8-aligned
    assert pb(fake, None, 4, 7, fake, fake, fake, None, fake, ctypes.c_size_t(8), None) == -2
    assert lib.spec_verify_plan_budget_workspace_bytes(512, 7) == 256
    assert lib.spec_verify_plan_budget_workspace_bytes(2341, 7) == 0
    # KV compaction: (pool, num_slots, row_bytes, planes, plane_stride, slot_table, max_pos,
    # committed_in, committed_out, accept_index, accept_len, B, N, dev_status, stream)
    kv = lib.spec_verify_kv_compact
    c_out = P(0x20000)
    assert kv(fake, 100, 40, 1, 0, fake, 64, fake, c_out, fake, fake, 4, 8, None, None) == -1  # row % 16
    assert kv(P(0x10008), 100, 48, 1, 0, fake, 64, fake, c_out, fake, fake, 4, 8, None, None) == -1
    assert kv(fake, 100, 48, 1, 0, fake, 64, fake, fake, fake, fake, 4, 8, None, None) == -1  # alias
    assert kv(fake, 100, 48, 1, 0, fake, 64, fake, c_out, fake, fake, 4, 65, None, None) == -1
    assert kv(fake, 100, 48, 1, 0, fake, 6, fake, c_out, fake, fake, 4, 8, None, None) == -1  # max_pos < N
    assert kv(fake, 100, 48, 1, 0, fake, 64, fake, c_out, fake, fake, 0, 8, None, None) == -1
    assert kv(fake, 100, 48, 2, 48 * 99, fake, 64, fake, c_out, fake, fake, 4, 8, None, None) == -1
    assert kv(fake, 100, 48, 2, 48 * 100 + 8, fake, 64, fake, c_out, fake, fake, 4, 8, None,
              None) == -1
    assert kv(None, 100, 48, 1, 0, fake, 64, fake, c_out, fake, fake, 4, 8, None, None) == -1
    del ws

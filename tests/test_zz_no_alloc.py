"""The allocation-free entry point returns what the workspace entry point returns.

spec_verify_rejection_noalloc serves callers that cannot allocate device memory while they
verify (an allocator that forbids new allocations in the middle of a step, or device memory
owned by another framework), so they have no workspace to hand over; the library uses its own
built-in scratch instead.  This file is collected last so that a failure here cannot stop a
first-failure run before the other tests have run.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PROB_RTOL = 1e-5


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_verify_gb300 import _build, binding

    _build.build()
    torch.cuda.set_device(DEV)
    return binding.load_library()


def _call_noalloc(lib, inp, q, offset, out, alen, probs, status):
    B, k, V = inp.shape
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.spec_verify_rejection_noalloc(P(inp.logits), 0 if inp.logits.dtype == torch.bfloat16
                                             else 1, P(inp.drafts), P(q), B, k, V,
                                             inp.temperature, inp.seed, offset, P(out), P(alen),
                                             P(probs), P(status), stream)


def test_noalloc_matches_workspace_entry_point(lib):
    import speculative_decoding_verification_verify_gb300 as sv
    from speculative_decoding_verification_verify_gb300 import workloads as wl

    cases = [(wl.chain_b64k7(DEV, B=16, k=7, V=20001, seed=71), False),
             (wl.chain_sweep(DEV, B=8, k=3, V=9000, alpha=0.6), True)]
    for inp, use_q in cases:
        B, k, V = inp.shape
        q = inp.q if use_q else None
        out = torch.empty((B, k + 1), dtype=torch.int32, device=DEV)
        alen = torch.empty(B, dtype=torch.int32, device=DEV)
        probs = torch.empty((B, k + 1, 3), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        for offset in (0, 1):  # two calls in a row: the second sees the first one's leftovers
            ref = sv.spec_verify_rejection(inp.logits, inp.drafts, q, temperature=inp.temperature,
                                           seed=inp.seed, offset=offset, want_probs=True)
            assert _call_noalloc(lib, inp, q, offset, out, alen, probs, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0 and int(ref.dev_status.item()) == 0
            assert torch.equal(out, ref.out_tokens)
            assert torch.equal(alen, ref.accept_len)
            a, b = probs.double().cpu().numpy(), ref.out_probs.double().cpu().numpy()
            big = np.abs(b) > 1e-30
            assert np.all(np.abs(a[big] - b[big]) <= PROB_RTOL * np.abs(b[big]))


def test_noalloc_rejects_oversized_calls(lib):
    from speculative_decoding_verification_verify_gb300 import binding

    B, k, V = 60000, 7, 1000
    assert binding.spec_verify_workspace_bytes(binding.MODE_REJECTION, B, k, V) > \
        binding.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never reached: the size check comes first
    rc = lib.spec_verify_rejection_noalloc(fake, 0, fake, None, B, k, V, 1.0, 1, 0, fake, fake,
                                           None, None, None)
    assert rc == binding.ETOOBIG

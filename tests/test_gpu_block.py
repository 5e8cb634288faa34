"""Parity of the CUDA block verification (spec_verify_block, through its C ABI) with the oracle.

Token ids and accept lengths must match exactly, except for requests the oracle flags as
boundary draws, which are counted and must stay rare.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_verify_gb300 as sv
from speculative_decoding_verification_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_verify_gb300 import _build

    _build.build()
    oracle.build()
    torch.cuda.set_device(DEV)


def _np(t):
    return t.detach().cpu().numpy()


def _sample(B, n, seed=0):
    if B <= n:
        return np.arange(B, dtype=np.int32)
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(B, size=n - 2, replace=False))
    return np.unique(np.concatenate([[0, B - 1], idx])).astype(np.int32)


def run_block(inp, with_q, offset=0, ids=None):
    B, k, V = inp.shape
    ids = np.arange(B, dtype=np.int32) if ids is None else ids
    q = inp.q if with_q else None
    r = sv.spec_verify_block(inp.logits, inp.drafts, q, temperature=inp.temperature, seed=inp.seed,
                             offset=offset)
    ref = oracle.verify_block(wl.to_numpy_logits(inp.logits), _np(inp.drafts),
                              None if q is None else _np(q), inp.temperature, inp.seed, offset,
                              req_ids=ids)
    torch.cuda.synchronize()
    gt, gl = _np(r.out_tokens)[ids], _np(r.accept_len)[ids]
    ok = ~ref["boundary"].astype(bool)
    np.testing.assert_array_equal(gl[ok], ref["accept_len"][ok])
    np.testing.assert_array_equal(gt[ok], ref["out_tokens"][ok])
    assert (~ok).sum() <= max(2, len(ids) // 100), f"{(~ok).sum()} boundary draws"
    if len(ids) == B:
        assert int(_np(r.dev_status)[0]) == int(ref["status"].max())
    return r, ref


def _dominant(B, k, V, T, seed, p_hit):
    """Logits ~N(0,1) plus log(V) + 3 on one token per row (p ~ 0.9 there); each draft is its
    row's peak w.p. p_hit, so prefixes of varied length pass."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn((B, k + 1, V), generator=g, device=DEV)
    peak = torch.randint(0, V, (B, k + 1, 1), generator=g, device=DEV)
    x.scatter_add_(2, peak, torch.full((B, k + 1, 1), 3.0 + float(np.log(V)), device=DEV))
    hit = torch.rand((B, k), generator=g, device=DEV) < p_hit
    other = torch.randint(0, V, (B, k), generator=g, device=DEV)
    drafts = torch.where(hit, peak[:, :k, 0], other).to(torch.int32).contiguous()
    return wl.ChainInputs("dominant", x.to(torch.bfloat16).contiguous(), drafts, None, T, seed)


@pytest.mark.parametrize("with_q", [False, True])
def test_block_tiny(with_q):
    run_block(wl.chain_tiny(DEV), with_q)


@pytest.mark.parametrize("V", [20001, 4099, 131])
@pytest.mark.parametrize("alpha", [0.35, 0.8])
def test_block_with_q_ragged(V, alpha):
    inp = wl.chain_sweep(DEV, B=12, k=5, V=V, alpha=alpha)
    for off in (0, 3):
        run_block(inp, True, offset=off)


@pytest.mark.parametrize("V", [20001, 5003])
def test_block_one_hot_varied_lengths(V):
    inp = _dominant(16, 7, V, 1.0, 31 + V, 0.75)
    r, ref = run_block(inp, False)
    assert len(set(ref["accept_len"].tolist())) >= 3
    run_block(wl.chain_b64k7(DEV, B=16, k=7, V=V, seed=V), False)


def test_block_fp32_and_unaligned():
    inp = wl.chain_sweep(DEV, B=6, k=4, V=9001, alpha=0.7)
    lg32 = inp.logits.float().contiguous()
    run_block(wl.ChainInputs("fp32", lg32, inp.drafts, inp.q, inp.temperature, inp.seed), True)
    base = torch.empty(inp.logits.numel() + 3, dtype=torch.bfloat16, device=DEV)
    shifted = base[3:].view(inp.logits.shape)
    shifted.copy_(inp.logits)
    run_block(wl.ChainInputs("shifted", shifted, inp.drafts, inp.q, inp.temperature, inp.seed), True)


def test_block_absent_drafts_and_k0():
    inp = wl.chain_sweep(DEV, B=8, k=6, V=3001, alpha=0.8)
    d = inp.drafts.clone()
    d[1, 0] = -1
    d[2, 3:] = -1
    d[3, 5] = -1
    for with_q in (False, True):
        run_block(wl.ChainInputs("absent", inp.logits, d, inp.q, inp.temperature, inp.seed), with_q)
    k0 = wl.chain_b64k7(DEV, B=3, k=0, V=7777, seed=4)
    run_block(k0, False)


@pytest.mark.parametrize("k", [12, 40])
def test_block_long_chains(k):
    inp = wl.chain_sweep(DEV, B=5, k=k, V=3001, alpha=0.85)
    run_block(inp, True)
    run_block(_dominant(5, k, 3001, 1.0, 50 + k, 0.9), False)


def test_block_full_b1k3():
    inp = wl.chain_b1k3(DEV)
    for off in range(4):
        run_block(inp, True, offset=off)


def test_block_full_b64k7_sampled():
    inp = wl.chain_b64k7(DEV)
    run_block(inp, False, ids=_sample(64, 8, seed=2))


def test_block_sweep_cell_sampled():
    inp = wl.chain_sweep(DEV, B=64, k=7, alpha=0.7)
    run_block(inp, True, ids=_sample(64, 6, seed=4))


def test_block_status_codes():
    inp = wl.chain_sweep(DEV, B=5, k=3, V=2000, alpha=0.6)
    lg = inp.logits.clone()
    lg[1, 2, 7] = float("nan")
    d = inp.drafts.clone()
    d[3, 1] = 5000
    r, ref = run_block(wl.ChainInputs("bad", lg, d, inp.q, inp.temperature, inp.seed), True)
    assert list(_np(r.accept_len)[[1, 3]]) == [-1, -1]
    assert int(_np(r.dev_status)[0]) == 2

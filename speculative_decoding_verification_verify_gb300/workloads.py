"""Seeded synthetic inputs for the verifier, shared by the tests and the benchmark.

This module only draws inputs.  It holds none of the verification arithmetic (the GPU library
and the CPU oracle each implement that on their own).  Where a workload is defined through the
target distribution -- q built so that sum(min(p, q)) hits a target acceptance rate -- the
construction calls torch's softmax as an input-construction step; no verification decision is
taken here.

Workloads (all synthetic; sizes and value distributions follow the configurations the
verifier is specified on):
  chain_tiny    B=4, k=3, V=1024, fp32 logits ~ N(0, 2^2); draft logits = target + N(0, 0.5^2),
                q = softmax(draft / T), drafts ~ q, T = 1.
  chain_b1k3    B=1, k=3, V=128256, bf16 logits ~ N(0, 3^2), T = 0.8; q = lam * p +
                (1 - lam) * Dirichlet(0.1) with lam solved so that sum(min(p, q)) = 0.70 at
                every position; drafts ~ q.
  chain_b64k7   B=64, k=7, V=128256, bf16 logits ~ N(0, 3^2) plus +8 at one uniformly chosen
                token per row; each draft is the target argmax of its row with probability 0.7,
                else uniform over V; one-hot drafts (no q), T = 1.
  tree_b48      B=48, N=8 nodes (root + 7 drafts), V=151936, bf16 logits ~ N(0, 3^2); parent of
                node j uniform over earlier nodes, redrawn until fan-out <= 4 and depth <= 5;
                a node's token is its parent row's argmax with probability 0.7 (if no sibling
                has it), else a uniform token distinct from its siblings.
  chain_sweep   B x k grid, V=128256 bf16 ~ N(0, 3^2); draft logits = target + N(0, sigma^2)
                with sigma bisected so that the mean of sum(min(p, q)) is alpha; T = 1.
  kv_paged      the KV cache that tree verification's accepted path is compacted in: planes =
                layers x (K, V) = 64 and 2048-byte rows (8 KV heads x 128 dims, bf16) as in a
                Llama-3-8B-sized target, B=48 requests of N=8 nodes, max_pos=512 positions each,
                every position mapped to a distinct pool slot by a random permutation (a paged
                allocator with one-token pages); committed uniform in [0, max_pos - N]; the
                accepted path walks a tree_b48-shaped random tree from the root, taking a uniform
                child and stopping with probability 0.3 before each step; pool bits uniform.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass
class ChainInputs:
    name: str
    logits: torch.Tensor            # [B, k+1, V] bf16 / fp32
    drafts: torch.Tensor            # [B, k] int32
    q: Optional[torch.Tensor]       # [B, k, V] fp32 or None (one-hot drafts)
    temperature: float
    seed: int
    offset: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, k1, V = self.logits.shape
        return B, k1 - 1, V


@dataclass
class TreeInputs:
    name: str
    logits: torch.Tensor            # [B, N, V]
    node_tokens: torch.Tensor       # [B, N] int32
    parents: torch.Tensor           # [B, N] int32
    temperature: float
    seed: int
    offset: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return tuple(self.logits.shape)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _rows_argmax(logits: torch.Tensor) -> torch.Tensor:
    return torch.argmax(logits.float(), dim=-1)


def chain_tiny(device="cpu", seed=1234, B=4, k=3, V=1024, T=1.0) -> ChainInputs:
    g = _gen(device, seed)
    logits = torch.randn((B, k + 1, V), generator=g, device=device) * 2.0
    draft_logits = logits[:, :k] + torch.randn((B, k, V), generator=g, device=device) * 0.5
    q = torch.softmax(draft_logits / T, dim=-1).float().contiguous()
    drafts = torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(B, k).int()
    return ChainInputs("chain_tiny", logits.contiguous(), drafts.contiguous(), q, T, seed + 17)


def chain_b1k3(device="cpu", seed=1235, B=1, k=3, V=128256, T=0.8, alpha=0.70) -> ChainInputs:
    g = _gen(device, seed)
    logits = (torch.randn((B, k + 1, V), generator=g, device=device) * 3.0).to(torch.bfloat16)
    p = torch.softmax(logits[:, :k].double() / T, dim=-1).cpu().numpy()
    rng = np.random.default_rng(seed)
    q = np.empty((B, k, V), np.float64)
    for b in range(B):
        for i in range(k):
            while True:
                d = rng.gamma(0.1, size=V)
                d /= d.sum()
                m = np.minimum(p[b, i], d).sum()
                if m < alpha:
                    break
            lam = (alpha - m) / (1.0 - m)
            q[b, i] = lam * p[b, i] + (1.0 - lam) * d
    qt = torch.from_numpy(q.astype(np.float32)).to(device)
    drafts = torch.multinomial(qt.reshape(-1, V), 1, generator=g).reshape(B, k).int()
    return ChainInputs("chain_b1k3", logits.contiguous(), drafts.contiguous(), qt.contiguous(), T,
                       seed + 17, meta=dict(alpha=alpha))


def chain_b64k7(device="cpu", seed=1236, B=64, k=7, V=128256, T=1.0, p_hit=0.7,
                dtype=torch.bfloat16) -> ChainInputs:
    g = _gen(device, seed)
    x = torch.randn((B, k + 1, V), generator=g, device=device) * 3.0
    peak = torch.randint(0, V, (B, k + 1, 1), generator=g, device=device)
    x.scatter_add_(2, peak, torch.full((B, k + 1, 1), 8.0, device=device))
    logits = x.to(dtype).contiguous()
    del x
    am = _rows_argmax(logits[:, :k])
    rand_tok = torch.randint(0, V, (B, k), generator=g, device=device)
    hit = torch.rand((B, k), generator=g, device=device) < p_hit
    drafts = torch.where(hit, am, rand_tok).int().contiguous()
    return ChainInputs("chain_b64k7", logits, drafts, None, T, seed + 17)


def _random_tree(rng, N, topk, steps):
    while True:
        parents = np.full(N, -1, np.int64)
        depth = np.zeros(N, np.int64)
        for j in range(1, N):
            parents[j] = rng.integers(0, j)
            depth[j] = depth[parents[j]] + 1
        fan = np.bincount(parents[1:], minlength=N)
        if fan.max(initial=0) <= topk and depth.max(initial=0) <= steps:
            return parents


def tree_b48(device="cpu", seed=1237, B=48, N=8, V=151936, T=1.0, topk=4, steps=5,
             p_hit=0.7, dtype=torch.bfloat16) -> TreeInputs:
    g = _gen(device, seed)
    logits = (torch.randn((B, N, V), generator=g, device=device) * 3.0).to(dtype).contiguous()
    am = _rows_argmax(logits).cpu().numpy()
    rng = np.random.default_rng(seed)
    parents = np.zeros((B, N), np.int32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        pa = _random_tree(rng, N, topk, steps)
        parents[b] = pa
        tokens[b, 0] = rng.integers(0, V)
        for j in range(1, N):
            sib = {int(tokens[b, s]) for s in range(1, j) if pa[s] == pa[j]}
            want = int(am[b, pa[j]])
            if rng.random() < p_hit and want not in sib:
                tokens[b, j] = want
            else:
                while True:
                    t = int(rng.integers(0, V))
                    if t not in sib:
                        break
                tokens[b, j] = t
    return TreeInputs("tree_b48", logits, torch.from_numpy(tokens).to(device),
                      torch.from_numpy(parents).to(device), T, seed + 17,
                      meta=dict(topk=topk, steps=steps))


def _mean_overlap(target_logits, sigma, noise, T):
    p = torch.softmax(target_logits.float() / T, dim=-1)
    q = torch.softmax((target_logits.float() + sigma * noise) / T, dim=-1)
    return torch.minimum(p, q).sum(-1).mean().item()


def chain_sweep(device="cpu", seed=1238, B=8, k=3, V=128256, alpha=0.7, T=1.0) -> ChainInputs:
    g = _gen(device, seed + 1000 * B + 10 * k + int(alpha * 100))
    logits = (torch.randn((B, k + 1, V), generator=g, device=device) * 3.0).to(torch.bfloat16)
    # Calibrate sigma on a few rows so that the mean of sum(min(p, q)) is alpha.
    cal_rows = logits.reshape(-1, V)[: max(1, min(8, B * (k + 1)))]
    cal_noise = torch.randn(cal_rows.shape, generator=g, device=device)
    lo, hi = 0.0, 20.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if _mean_overlap(cal_rows, mid, cal_noise, T) > alpha:
            lo = mid
        else:
            hi = mid
    sigma = 0.5 * (lo + hi)
    noise = torch.randn((B, k, V), generator=g, device=device)
    q = torch.softmax((logits[:, :k].float() + sigma * noise) / T, dim=-1).contiguous()
    del noise
    drafts = (torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(B, k).int()
              if k > 0 else torch.zeros((B, 0), dtype=torch.int32, device=device))
    return ChainInputs(f"chain_sweep_B{B}_k{k}_a{alpha}", logits.contiguous(), drafts.contiguous(),
                       q, T, seed + 17, meta=dict(alpha=alpha, sigma=sigma))


@dataclass
class KVInputs:
    name: str
    pool: torch.Tensor              # [planes, num_slots, row_bytes / 2] int16 (KV bit patterns)
    slot_table: torch.Tensor        # [B, max_pos] int32
    committed: torch.Tensor         # [B] int32
    accept_index: torch.Tensor      # [B, N] int32 (root, then the path; -1 after it)
    accept_len: torch.Tensor        # [B] int32


def kv_paged(device="cpu", seed=1239, B=48, N=8, planes=64, row_bytes=2048, max_pos=512,
             topk=4, steps=5, p_stop=0.3, extra_slots=0, pool=None) -> KVInputs:
    """pool: reuse an existing [planes, num_slots, row_bytes / 2] int16 pool instead of drawing
    one (other seeds then give other positions, slots and paths over the same cache)."""
    rng = np.random.default_rng(seed)
    num_slots = B * max_pos + extra_slots
    slot_table = rng.permutation(num_slots)[: B * max_pos].astype(np.int32).reshape(B, max_pos)
    committed = rng.integers(0, max_pos - N + 1, B).astype(np.int32)
    accept_index = np.full((B, N), -1, np.int32)
    accept_len = np.zeros(B, np.int32)
    for b in range(B):
        parents = _random_tree(rng, N, topk, steps)
        path, cur = [0], 0
        while True:
            kids = np.flatnonzero(parents == cur)
            kids = kids[kids > 0]
            if kids.size == 0 or rng.random() < p_stop:
                break
            cur = int(rng.choice(kids))
            path.append(cur)
        accept_index[b, : len(path)] = path
        accept_len[b] = len(path) - 1
    if pool is None:
        g = _gen(device, seed)
        pool = torch.randint(-32768, 32768, (planes, num_slots, row_bytes // 2), generator=g,
                             device=device, dtype=torch.int16)
    elif tuple(pool.shape) != (planes, num_slots, row_bytes // 2) or pool.dtype != torch.int16:
        raise ValueError("pool does not match the requested shape")
    t = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
    return KVInputs(f"kv_paged_B{B}_N{N}_planes{planes}_row{row_bytes}", pool, t(slot_table),
                    t(committed), t(accept_index), t(accept_len))


# --------------------------------------------------------------------------------------------
# Host copies for the oracle (bf16 as uint16 bit patterns)
# --------------------------------------------------------------------------------------------
def to_numpy_logits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()

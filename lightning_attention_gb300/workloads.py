"""Seeded synthetic workloads for seg_la (segmented lightning attention).

This module only draws random inputs and describes their shapes.  It holds none of the method's
arithmetic (no slopes, no decay, no contraction): the CUDA path and the fp64 oracle each compute
those themselves from the same drawn tensors.  Both sides import it; it imports neither.

Every workload uses a CPU ``torch.Generator`` seeded with ``seed`` (0 by default) and draws, in
this fixed order: request lengths (when random), q, k, v (``randn`` fp32 rounded to bf16), prefix
states (``randn * 0.05``, fp32), the slot permutation (``randperm``), and finally decode-step
q/k/v (the tiny workload only).  The prefix-state scale of 0.05 follows the page
"SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
"独立参考实现" (prefix states injected at 0.05 so that a prefix bug cannot hide behind zeros).

Pool slots that no request names hold the sentinel 54321.0, and named slots of requests without a
prefix hold NaN, so that a read of either shows up (the page's state-tracking test uses the same
54321.0 sentinel for untouched slots).  The decode workload is the exception: its whole pool is
random, as its description asks.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
SENTINEL = 54321.0


@dataclass
class Workload:
    name: str
    kind: str                      # "extend", "decode", "verify" or "tree"
    H: int
    D: int
    layer_id: int
    L: int
    num_slots: int
    q: torch.Tensor                # bf16 [rows, H*D]
    k: torch.Tensor
    v: torch.Tensor
    state_idx: torch.Tensor        # int32 [B]
    prefix_mask: torch.Tensor      # uint8 [B]
    prefix_states: torch.Tensor    # fp32 [B, H, D, D] (rows of requests without prefix unused)
    cu_seqlens: torch.Tensor | None = None   # int32 [B+1] (extend)
    N: int = 1                     # draft tokens per request (verify)
    random_pool: bool = False      # decode workload: every slot random
    pool_fill: torch.Tensor | None = None    # fp32 [num_slots, H, D, D] when random_pool
    decode_steps: list = field(default_factory=list)  # tiny workload: [(q, k, v)] per step
    parents: torch.Tensor | None = None      # int32 [B, N] (tree verify)
    track_lens: torch.Tensor | None = None   # int32 [B] (extend with state tracking)
    track_idx: torch.Tensor | None = None    # int32 [B] (extend with state tracking)
    accept_idx: torch.Tensor | None = None   # int32 [B] (verify followed by the commit)
    Hkv: int | None = None                   # kv heads of a grouped-query workload (None: H);
                                             # k, v, slopes and the pool then have Hkv heads

    @property
    def B(self) -> int:
        return int(self.state_idx.shape[0])

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    def tokens(self) -> int:
        return self.T

    @property
    def state_heads(self) -> int:
        """Heads of k, v, the slopes and the states (the kv heads of a grouped workload)."""
        return self.H if self.Hkv is None else self.Hkv

    def materialize_pool(self, device="cpu") -> torch.Tensor:
        """Full fp32 pool [num_slots, H, D, D] on ``device``: sentinel everywhere, prefix states
        in the slots of prefix requests, NaN in the named slots of the other requests."""
        if self.random_pool:
            return self.pool_fill.to(device).clone()
        pool = torch.full((self.num_slots, self.state_heads, self.D, self.D), SENTINEL,
                          dtype=torch.float32, device=device)
        for b in range(self.B):
            s = int(self.state_idx[b])
            if int(self.prefix_mask[b]):
                pool[s].copy_(self.prefix_states[b].to(device))
            else:
                pool[s].fill_(float("nan"))
        return pool


def _qkv(g: torch.Generator, rows: int, width: int):
    out = []
    for _ in range(3):
        out.append(torch.randn(rows, width, generator=g, dtype=torch.float32).to(torch.bfloat16))
    return out


def tiny(seed: int = 0) -> Workload:
    """Tiny correctness case: H=2, head_dim 128, L=1 (layer 0); two requests of lengths 37 and 64;
    the second has a prefix state in slot 5 of an 8-slot pool, the first starts from zero in slot 2;
    one extend call, then 4 decode steps per request."""
    g = torch.Generator().manual_seed(seed)
    H, D = 2, HEAD_DIM
    lens = [37, 64]
    T = sum(lens)
    q, k, v = _qkv(g, T, H * D)
    prefix = torch.zeros(2, H, D, D)
    prefix[1] = torch.randn(H, D, D, generator=g) * 0.05
    steps = []
    for _ in range(4):
        steps.append(tuple(_qkv(g, 2, H * D)))
    return Workload(name="tiny", kind="extend", H=H, D=D, layer_id=0, L=1, num_slots=8,
                    q=q, k=k, v=v, state_idx=torch.tensor([2, 5], dtype=torch.int32),
                    prefix_mask=torch.tensor([0, 1], dtype=torch.uint8), prefix_states=prefix,
                    cu_seqlens=torch.tensor([0, 37, 101], dtype=torch.int32), decode_steps=steps)


def decode_batch(seed: int = 0, B: int = 256, num_slots: int = 1024) -> Workload:
    """Decode batch: 256 requests x 1 token, H=16, head_dim 128, layer 3 of L=8; a 1024-slot pool
    of random states (N(0,1)*0.05) with the 256 slots a random permutation subset."""
    g = torch.Generator().manual_seed(seed)
    H, D = 16, HEAD_DIM
    q, k, v = _qkv(g, B, H * D)
    pool = torch.randn(num_slots, H, D, D, generator=g) * 0.05
    idx = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    return Workload(name="decode_b256_h16", kind="decode", H=H, D=D, layer_id=3, L=8,
                    num_slots=num_slots, q=q, k=k, v=v, state_idx=idx,
                    prefix_mask=torch.ones(B, dtype=torch.uint8),
                    prefix_states=torch.empty(0), random_pool=True, pool_fill=pool)


def varlen_extend(seed: int = 0, B: int = 8, lo: int = 512, hi: int = 4096,
                  num_slots: int = 64) -> Workload:
    """Varlen extend: 8 requests with lengths uniform in [512, 4096], H=16, layer 0 of L=4; the
    even-indexed half of the requests carry prefix states; slots shuffled in a 64-slot pool."""
    g = torch.Generator().manual_seed(seed)
    H, D = 16, HEAD_DIM
    lens = torch.randint(lo, hi + 1, (B,), generator=g)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v = _qkv(g, T, H * D)
    pm = torch.tensor([1 if b % 2 == 0 else 0 for b in range(B)], dtype=torch.uint8)
    prefix = torch.zeros(B, H, D, D)
    for b in range(B):
        if pm[b]:
            prefix[b] = torch.randn(H, D, D, generator=g) * 0.05
    idx = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    return Workload(name="varlen_extend_b8_h16", kind="extend", H=H, D=D, layer_id=0, L=4,
                    num_slots=num_slots, q=q, k=k, v=v, state_idx=idx, prefix_mask=pm,
                    prefix_states=prefix, cu_seqlens=cu)


def varlen_extend_many(seed: int = 0, B: int = 1024, lo: int = 32, hi: int = 512,
                       num_slots: int = 2048) -> Workload:
    """Large varlen extend batch: 1024 requests with lengths uniform in [32, 512], H=16, layer 0
    of L=4; the even-indexed half carry prefix states; slots shuffled in a 2048-slot pool.  The
    same draw order as varlen_extend."""
    w = varlen_extend(seed, B=B, lo=lo, hi=hi, num_slots=num_slots)
    w.name = f"varlen_extend_b{B}_h16"
    return w


def varlen_extend_skewed(seed: int = 0, B: int = 8, n_long: int = 2, long_lo: int = 4096,
                         long_hi: int = 8192, lo: int = 256, hi: int = 1024,
                         num_slots: int = 64) -> Workload:
    """Skewed varlen extend: 8 requests, the first two with lengths uniform in [4096, 8192] and the
    other six in [256, 1024] (a couple of long prefills among short extends), H=16, layer 0 of
    L=4; the even-indexed half carry prefix states; slots shuffled in a 64-slot pool.  The same
    draw order as varlen_extend."""
    g = torch.Generator().manual_seed(seed)
    H, D = 16, HEAD_DIM
    lens = torch.cat([torch.randint(long_lo, long_hi + 1, (n_long,), generator=g),
                      torch.randint(lo, hi + 1, (B - n_long,), generator=g)])
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v = _qkv(g, T, H * D)
    pm = torch.tensor([1 if b % 2 == 0 else 0 for b in range(B)], dtype=torch.uint8)
    prefix = torch.zeros(B, H, D, D)
    for b in range(B):
        if pm[b]:
            prefix[b] = torch.randn(H, D, D, generator=g) * 0.05
    idx = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    return Workload(name=f"varlen_extend_skewed_b{B}_h16", kind="extend", H=H, D=D, layer_id=0,
                    L=4, num_slots=num_slots, q=q, k=k, v=v, state_idx=idx, prefix_mask=pm,
                    prefix_states=prefix, cu_seqlens=cu)


def long_prefill(seed: int = 0, T: int = 32768, H: int = 32) -> Workload:
    """Long single-sequence prefill: one request of 32768 tokens, H=32, layer 5 of L=12, zero
    initial state; pool of 4 slots, the request in slot 1."""
    g = torch.Generator().manual_seed(seed)
    D = HEAD_DIM
    q, k, v = _qkv(g, T, H * D)
    return Workload(name=f"long_prefill_t{T}_h{H}", kind="extend", H=H, D=D, layer_id=5, L=12,
                    num_slots=4, q=q, k=k, v=v, state_idx=torch.tensor([1], dtype=torch.int32),
                    prefix_mask=torch.zeros(1, dtype=torch.uint8),
                    prefix_states=torch.zeros(1, H, D, D),
                    cu_seqlens=torch.tensor([0, T], dtype=torch.int32))


def verify_chain(seed: int = 0, B: int = 128, N: int = 5, H: int = 64,
                 num_slots: int = 512) -> Workload:
    """Chain target verify (topk = 1): 128 requests x 5 draft tokens, H=64, layer 10 of L=20; every
    request has a prefix state in a random slot of a 512-slot pool."""
    g = torch.Generator().manual_seed(seed)
    D = HEAD_DIM
    q, k, v = _qkv(g, B * N, H * D)
    prefix = torch.randn(B, H, D, D, generator=g) * 0.05
    idx = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    return Workload(name=f"verify_chain_b{B}_n{N}_h{H}", kind="verify", H=H, D=D, layer_id=10,
                    L=20, num_slots=num_slots, q=q, k=k, v=v, state_idx=idx,
                    prefix_mask=torch.ones(B, dtype=torch.uint8), prefix_states=prefix, N=N)


# A binary draft tree of 8 tokens (two children per node, depth 4): token t forks from the state
# after token EAGLE_TREE8[t]; -1 is the verified prefix (the pool state).
EAGLE_TREE8 = (-1, 0, 0, 1, 1, 2, 2, 3)


def verify_tree(seed: int = 0, B: int = 128, H: int = 64, parents=EAGLE_TREE8,
                num_slots: int = 512) -> Workload:
    """Tree target verify (topk > 1): 128 requests x an 8-token draft tree, H=64, layer 10 of L=20;
    every request has a prefix state in a random slot of a 512-slot pool; all requests share one
    tree shape.  Same draw order as the chain-verify workload."""
    w = verify_chain(seed, B=B, N=len(parents), H=H, num_slots=num_slots)
    w.name = f"verify_tree_b{B}_n{len(parents)}_h{H}"
    w.kind = "tree"
    w.parents = torch.tensor([list(parents)] * B, dtype=torch.int32)
    return w


def varlen_extend_tracked(seed: int = 0) -> Workload:
    """The varlen extend workload with a state-tracking snapshot per request: track lengths
    uniform in [0, length], track slots drawn from the slots no request uses.  The extra draws
    come from a second generator (seed + 1000), so the base workload is unchanged."""
    w = varlen_extend(seed)
    g = torch.Generator().manual_seed(seed + 1000)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    w.track_lens = torch.tensor([int(torch.randint(0, n + 1, (1,), generator=g)) for n in lens],
                                dtype=torch.int32)
    used = set(w.state_idx.tolist())
    free = torch.tensor([s for s in range(w.num_slots) if s not in used], dtype=torch.int32)
    w.track_idx = free[torch.randperm(len(free), generator=g)[:w.B]]
    w.name = "varlen_extend_tracked_b8_h16"
    return w


def verify_commit(seed: int = 0) -> Workload:
    """The chain-verify workload followed by the accepted-state commit: accept indices uniform
    in [-1, N-1] (second generator, seed + 1000)."""
    w = verify_chain(seed)
    g = torch.Generator().manual_seed(seed + 1000)
    w.accept_idx = torch.randint(-1, w.N, (w.B,), generator=g, dtype=torch.int32)
    w.name = f"verify_commit_b{w.B}_n{w.N}_h{w.H}"
    return w


def custom_extend(lengths, H: int = 2, D: int = HEAD_DIM, layer_id: int = 0, L: int = 1,
                  prefix=None, num_slots: int | None = None, seed: int = 0,
                  shuffle_slots: bool = True) -> Workload:
    """Extend batch of given lengths (edge-case tests): same draw order as the fixed workloads."""
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    q, k, v = _qkv(g, T, H * D)
    if prefix is None:
        prefix = [b % 2 for b in range(B)]
    pm = torch.tensor(list(prefix), dtype=torch.uint8) if B else torch.zeros(0, dtype=torch.uint8)
    ps = torch.zeros(B, H, D, D)
    for b in range(B):
        if pm[b]:
            ps[b] = torch.randn(H, D, D, generator=g) * 0.05
    ns = num_slots if num_slots is not None else max(2 * B, 1)
    if shuffle_slots:
        idx = torch.randperm(ns, generator=g)[:B].to(torch.int32)
    else:
        idx = torch.arange(B, dtype=torch.int32)
    return Workload(name=f"custom_{B}req", kind="extend", H=H, D=D, layer_id=layer_id, L=L,
                    num_slots=ns, q=q, k=k, v=v, state_idx=idx, prefix_mask=pm,
                    prefix_states=ps, cu_seqlens=cu)


def custom_verify(B: int, N: int, H: int = 2, D: int = HEAD_DIM, layer_id: int = 0, L: int = 1,
                  num_slots: int | None = None, seed: int = 0) -> Workload:
    g = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(g, B * N, H * D)
    ps = torch.randn(B, H, D, D, generator=g) * 0.05
    ns = num_slots if num_slots is not None else max(2 * B, 1)
    idx = torch.randperm(ns, generator=g)[:B].to(torch.int32)
    return Workload(name=f"custom_verify_{B}x{N}", kind="verify", H=H, D=D, layer_id=layer_id,
                    L=L, num_slots=ns, q=q, k=k, v=v, state_idx=idx,
                    prefix_mask=torch.ones(B, dtype=torch.uint8), prefix_states=ps, N=N)


def custom_extend_gqa(lengths, H: int, Hkv: int, D: int = HEAD_DIM, layer_id: int = 0, L: int = 1,
                      prefix=None, num_slots: int | None = None, seed: int = 0) -> Workload:
    """Grouped-query extend batch: q with H heads, k and v with Hkv heads (H a multiple of Hkv),
    prefix states per kv head.  Draw order: q, k, v, prefix states, slot permutation."""
    g = torch.Generator().manual_seed(seed)
    B = len(lengths)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    q = torch.randn(T, H * D, generator=g).to(torch.bfloat16)
    k = torch.randn(T, Hkv * D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv * D, generator=g).to(torch.bfloat16)
    if prefix is None:
        prefix = [b % 2 for b in range(B)]
    pm = torch.tensor(list(prefix), dtype=torch.uint8) if B else torch.zeros(0, dtype=torch.uint8)
    ps = torch.zeros(B, Hkv, D, D)
    for b in range(B):
        if pm[b]:
            ps[b] = torch.randn(Hkv, D, D, generator=g) * 0.05
    ns = num_slots if num_slots is not None else max(2 * B, 1)
    idx = torch.randperm(ns, generator=g)[:B].to(torch.int32)
    return Workload(name=f"custom_gqa_{B}req_h{H}_kv{Hkv}", kind="extend", H=H, D=D,
                    layer_id=layer_id, L=L, num_slots=ns, q=q, k=k, v=v, state_idx=idx,
                    prefix_mask=pm, prefix_states=ps, cu_seqlens=cu, Hkv=Hkv)


def custom_decode_gqa(B: int, H: int, Hkv: int, D: int = HEAD_DIM, layer_id: int = 0, L: int = 1,
                      num_slots: int | None = None, seed: int = 0) -> Workload:
    """Grouped-query decode batch: q [B, H*D], k and v [B, Hkv*D], a random pool of Hkv-head
    states (N(0,1)*0.05) with the B slots a random permutation subset."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H * D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv * D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv * D, generator=g).to(torch.bfloat16)
    ns = num_slots if num_slots is not None else 2 * B
    pool = torch.randn(ns, Hkv, D, D, generator=g) * 0.05
    idx = torch.randperm(ns, generator=g)[:B].to(torch.int32)
    return Workload(name=f"custom_decode_gqa_b{B}_h{H}_kv{Hkv}", kind="decode", H=H, D=D,
                    layer_id=layer_id, L=L, num_slots=ns, q=q, k=k, v=v, state_idx=idx,
                    prefix_mask=torch.ones(B, dtype=torch.uint8), prefix_states=torch.empty(0),
                    random_pool=True, pool_fill=pool, Hkv=Hkv)


WORKLOADS = {
    "tiny": tiny,
    "decode": decode_batch,
    "varlen_extend": varlen_extend,
    "long_prefill": long_prefill,
    "verify": verify_chain,
    "verify_tree": verify_tree,
    "varlen_extend_tracked": varlen_extend_tracked,
    "verify_commit": verify_commit,
    "varlen_extend_b1024": varlen_extend_many,
    "varlen_extend_skewed": varlen_extend_skewed,
}

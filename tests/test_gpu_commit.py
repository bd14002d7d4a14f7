"""GPU parity of the accepted-state commit (la_commit_accepted) against the fp64 oracle.

After a verify, the target model accepts some prefix of the draft tokens (a root path in a tree)
and the request's state becomes the state after the last accepted token (page "SGLang Lightning
Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section "生产环境不支持", item 3).  Checked:
the committed slots equal the GPU intermediate states bit for bit and the oracle's
verify-then-commit within tolerance; -1 and unnamed slots keep their bytes; a decode from the
committed pool continues the sequence; out-of-range indices are reported and write nothing.
"""
import numpy as np
import pytest
import torch

import lightning_attention_gb300 as la
import oracle
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, oracle_slopes_fp32, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _bits(t):
    return t.detach().cpu().view(torch.int32)


@pytest.mark.parametrize("kind", ["chain", "tree"])
def test_commit_after_verify(kind):
    w = workloads.custom_verify(6, 5, H=3, layer_id=2, L=4, num_slots=16, seed=11)
    parents = (torch.tensor([[-1, 0, 0, 1, 2]] * w.B, dtype=torch.int32) if kind == "tree"
               else torch.tensor([list(range(-1, w.N - 1))] * w.B, dtype=torch.int32))
    accept = torch.tensor([4, -1, 0, 2, 3, 1], dtype=torch.int32)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    q, k, v, idx = w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), w.state_idx.to(DEV)
    if kind == "tree":
        _, inter = la.verify_tree(q, k, v, s, pool, idx, parents.to(DEV), w.N)
    else:
        _, inter = la.verify_chain(q, k, v, s, pool, idx, w.N)
    la.commit_accepted(inter, accept.to(DEV), pool, idx)
    la.poll_error()
    got = pool.cpu()
    inter_c = inter.cpu()
    named = set(w.state_idx.tolist())
    for slot in range(w.num_slots):
        if slot not in named:
            assert torch.equal(_bits(got[slot]), _bits(pool0[slot]))
    for b in range(w.B):
        a = int(accept[b])
        slot = int(w.state_idx[b])
        ref = pool0[slot] if a < 0 else inter_c[b, a]
        assert torch.equal(_bits(got[slot]), _bits(ref)), f"request {b}"
    # against the oracle's own verify + commit
    sl = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    args = (w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(), sl,
            pool0.double().numpy(), w.state_idx.numpy())
    if kind == "tree":
        _, i_ref = oracle.verify_tree(*args, parents.numpy(), w.N, w.H, w.D)
    else:
        _, i_ref = oracle.verify_chain(*args, w.N, w.H, w.D)
    p_ref = oracle.commit_accepted(i_ref, accept.numpy(), pool0.double().numpy(),
                                   w.state_idx.numpy())
    assert_close(to64(got), p_ref, f"{kind}: committed pool")
    # one decode step from the committed pool
    qn, kn, vn = (torch.randn(w.B, w.H * w.D, generator=torch.Generator().manual_seed(12 + j))
                  .to(torch.bfloat16) for j in range(3))
    o = la.decode(qn.to(DEV), kn.to(DEV), vn.to(DEV), s, pool, idx)
    la.poll_error()
    o_ref, d_ref = oracle.decode(qn.float().numpy(), kn.float().numpy(), vn.float().numpy(), sl,
                                 p_ref, w.state_idx.numpy(), w.H, w.D)
    assert_close(to64(o), o_ref, f"{kind}: decode after commit, out")
    assert_close(to64(pool.cpu()), d_ref, f"{kind}: decode after commit, pool")


def test_commit_full_size_verify_workload_sampled():
    w = workloads.verify_chain(0)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    _, inter = la.verify_chain(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s, pool,
                               w.state_idx.to(DEV), w.N)
    accept = torch.randint(-1, w.N, (w.B,), generator=torch.Generator().manual_seed(3),
                           dtype=torch.int32)
    la.commit_accepted(inter, accept.to(DEV), pool, w.state_idx.to(DEV))
    la.poll_error()
    for b in (0, 1, 63, 127):
        a = int(accept[b])
        slot = int(w.state_idx[b])
        ref = pool0[slot] if a < 0 else inter[b, a].cpu()
        assert torch.equal(_bits(pool[slot]), _bits(ref))
    assert int((accept < 0).sum()) > 0 and int((accept >= 0).sum()) > 0


def test_commit_bad_index_reported_nothing_written():
    w = workloads.custom_verify(3, 4, H=2, num_slots=8, seed=13)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    _, inter = la.verify_chain(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s, pool,
                               w.state_idx.to(DEV), w.N)
    la.poll_error()
    bad = torch.tensor([1, w.N, -2], dtype=torch.int32, device=DEV)  # requests 1 and 2 bad
    la.commit_accepted(inter, bad, pool, w.state_idx.to(DEV))
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    got = pool.cpu()
    for b in (1, 2):
        slot = int(w.state_idx[b])
        assert torch.equal(_bits(got[slot]), _bits(pool0[slot]))
    assert torch.equal(_bits(got[int(w.state_idx[0])]), _bits(inter[0, 1]))

"""GPU parity of tree verify (la_verify_tree) against the fp64 oracle's parent-aware recurrence.

The page's seg_la processes draft tokens only as a chain; its named fix is for each draft token
to fork from the state saved for its parent (section "Next Work", item 2, of "SGLang Lightning
Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析").  Checked here: the 128 x 8-token binary
tree workload (all outputs, sampled intermediate states), random trees, a chain-shaped tree
(bit-identical to la_verify_chain), a star (bit-identical to independent decodes), the pool left
untouched, and parents that do not point backwards (reported, nothing written).
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


def run_tree(w, parents, pool_dev):
    return la.verify_tree(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV),
                          la.slopes(w.H, w.layer_id, w.L).to(DEV), pool_dev, w.state_idx.to(DEV),
                          parents.to(DEV), w.N)


def test_tree_workload_full_outputs_sampled_states():
    w = workloads.verify_tree(0)
    pool0 = w.materialize_pool()
    pool_dev = pool0.to(DEV)
    out, inter = run_tree(w, w.parents, pool_dev)
    la.poll_error()
    assert torch.equal(pool_dev.cpu().view(torch.int32), pool0.view(torch.int32))
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    idx = w.state_idx.numpy()
    out64 = to64(out)
    group = 16
    for g0 in range(0, w.B, group):
        reqs = np.arange(g0, min(g0 + group, w.B))
        rows = np.concatenate([np.arange(b * w.N, (b + 1) * w.N) for b in reqs])
        sub_pool = pool0[torch.from_numpy(idx[reqs]).long()].double().numpy()
        o_ref, i_ref = oracle.verify_tree(w.q.float().numpy()[rows], w.k.float().numpy()[rows],
                                          w.v.float().numpy()[rows], s, sub_pool,
                                          np.arange(len(reqs), dtype=np.int32),
                                          w.parents.numpy()[reqs], w.N, w.H, w.D)
        assert_close(out64[rows], o_ref, f"tree: out (requests {reqs[0]}..{reqs[-1]})")
        for j, b in enumerate(reqs):
            if int(b) in (0, 77, w.B - 1):
                assert_close(inter[b].cpu().double().numpy(), i_ref[j],
                             f"tree: intermediate states of request {b}")


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_trees(seed):
    rng = np.random.default_rng(seed)
    B, N = 6, 9
    w = workloads.custom_verify(B, N, H=3, layer_id=1, L=3, seed=seed)
    parents = np.stack([np.array([rng.integers(-1, t) if t > 0 else -1 for t in range(N)])
                        for _ in range(B)]).astype(np.int32)
    pool0 = w.materialize_pool()
    out, inter = run_tree(w, torch.from_numpy(parents), pool0.to(DEV))
    la.poll_error()
    o_ref, i_ref = oracle.verify_tree(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                      oracle_slopes_fp32(w.H, w.layer_id, w.L),
                                      pool0.double().numpy(), w.state_idx.numpy(), parents, N, w.H,
                                      w.D)
    assert_close(to64(out), o_ref, "random tree: out")
    assert_close(inter.cpu().double().numpy(), i_ref, "random tree: states")


def test_chain_shaped_tree_equals_chain_verify_bitwise():
    w = workloads.custom_verify(4, 6, H=2, seed=5)
    chain = torch.tensor([list(range(-1, w.N - 1))] * w.B, dtype=torch.int32)
    pool = w.materialize_pool(DEV)
    out_t, inter_t = run_tree(w, chain, pool)
    out_c, inter_c = la.verify_chain(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV),
                                     la.slopes(w.H, w.layer_id, w.L).to(DEV), pool,
                                     w.state_idx.to(DEV), w.N)
    la.poll_error()
    assert torch.equal(out_t.cpu(), out_c.cpu())
    assert torch.equal(inter_t.cpu(), inter_c.cpu())


def test_star_tree_equals_independent_decodes_bitwise():
    w = workloads.custom_verify(3, 5, H=2, seed=6)
    star = torch.full((w.B, w.N), -1, dtype=torch.int32)
    pool = w.materialize_pool(DEV)
    out, inter = run_tree(w, star, pool)
    la.poll_error()
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    for t in range(w.N):
        rows = torch.arange(w.B) * w.N + t
        p2 = pool.clone()
        o = la.decode(w.q[rows].to(DEV), w.k[rows].to(DEV), w.v[rows].to(DEV), s, p2,
                      w.state_idx.to(DEV))
        la.poll_error()
        assert torch.equal(o.cpu(), out.cpu()[rows])
        assert torch.equal(p2.cpu()[w.state_idx.long()], inter.cpu()[:, t])


def test_parents_pointing_forward_are_reported_and_nothing_written():
    w = workloads.custom_verify(2, 4, H=2, seed=7)
    bad = torch.tensor([[-1, 0, 3, 1], [-1, 0, 1, 2]], dtype=torch.int32)  # request 0 is bad
    pool = w.materialize_pool(DEV)
    out = torch.full((w.B * w.N, w.H * w.D), 7.0, dtype=torch.bfloat16, device=DEV)
    la.verify_tree(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV), pool,
                   w.state_idx.to(DEV), bad.to(DEV), w.N, out=out)
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    assert (out[: w.N].float() == 7.0).all()          # bad request: untouched
    assert not (out[w.N:].float() == 7.0).all()       # good request: written

"""CUDA-graph capture and replay of the seg_la entry points.

A serving loop captures its per-step launches once and replays them.  The entry points launch
only on the caller's stream, take every size and pointer at call time and never synchronise, so
a captured call replays the same work on whatever the static buffers hold.  Checked: a decode
step, a verify + accepted-state commit step and a varlen extend (with max_seqlen and workspace
given) each replayed several times with fresh inputs copied into the static buffers, against
the same calls made eagerly (bit for bit) and against the fp64 oracle.
"""
import pytest
import torch

import lightning_attention_gb300 as la
import oracle
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, oracle_slopes_fp32, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _capture(fn):
    """Warm up on a side stream, then capture fn() into a graph; returns (graph, fn's result)."""
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res = fn()
    return g, res


def _rand_bf16(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)


def test_decode_step_graph_replay():
    B, H, D, S = 16, 4, 128, 40
    s = la.slopes(H, 1, 3).to(DEV)
    idx = torch.randperm(S, generator=torch.Generator().manual_seed(1))[:B].to(torch.int32)
    pool0 = torch.randn(S, H, D, D, generator=torch.Generator().manual_seed(2)) * 0.05
    qs, ks, vs = (torch.zeros(B, H * D, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    out = torch.empty(B, H * D, dtype=torch.bfloat16, device=DEV)
    pool_g = pool0.to(DEV)
    idx_d = idx.to(DEV)
    g, _ = _capture(lambda: la.decode(qs, ks, vs, s, pool_g, idx_d, out=out))
    pool_g.copy_(pool0.to(DEV))          # undo the warm-up and capture-time updates
    la.poll_error()
    pool_e = pool0.to(DEV)
    ref_pool = pool0.double().numpy()
    sl = oracle_slopes_fp32(H, 1, 3)
    for step in range(4):
        q, k, v = (_rand_bf16((B, H * D), 10 * step + j) for j in range(3))
        qs.copy_(q)
        ks.copy_(k)
        vs.copy_(v)
        g.replay()
        o_e = la.decode(q.to(DEV), k.to(DEV), v.to(DEV), s, pool_e, idx_d)
        la.poll_error()
        assert torch.equal(out.cpu(), o_e.cpu()), f"step {step}: replay != eager output"
        assert torch.equal(pool_g.cpu(), pool_e.cpu()), f"step {step}: replay != eager pool"
        o_ref, ref_pool = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                        sl, ref_pool, idx.numpy(), H, D)
        assert_close(to64(out), o_ref, f"graph decode step {step}")
    assert_close(to64(pool_g.cpu()), ref_pool, "graph decode: final pool")


def test_verify_commit_step_graph_replay():
    B, N, H, D, S = 8, 4, 2, 128, 24
    s = la.slopes(H, 0, 1).to(DEV)
    idx = torch.randperm(S, generator=torch.Generator().manual_seed(5))[:B].to(torch.int32)
    pool0 = torch.randn(S, H, D, D, generator=torch.Generator().manual_seed(6)) * 0.05
    qs, ks, vs = (torch.zeros(B * N, H * D, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    acc_s = torch.full((B,), -1, dtype=torch.int32, device=DEV)
    out = torch.empty(B * N, H * D, dtype=torch.bfloat16, device=DEV)
    inter = torch.empty(B, N, H, D, D, dtype=torch.float32, device=DEV)
    pool_g = pool0.to(DEV)
    idx_d = idx.to(DEV)

    def step_fn():
        la.verify_chain(qs, ks, vs, s, pool_g, idx_d, N, out=out, inter_states=inter)
        la.commit_accepted(inter, acc_s, pool_g, idx_d)

    g, _ = _capture(step_fn)
    pool_g.copy_(pool0.to(DEV))
    la.poll_error()
    pool_e = pool0.to(DEV)
    ref_pool = pool0.double().numpy()
    sl = oracle_slopes_fp32(H, 0, 1)
    gen = torch.Generator().manual_seed(7)
    for step in range(3):
        q, k, v = (_rand_bf16((B * N, H * D), 100 + 10 * step + j) for j in range(3))
        accept = torch.randint(-1, N, (B,), generator=gen, dtype=torch.int32)
        qs.copy_(q)
        ks.copy_(k)
        vs.copy_(v)
        acc_s.copy_(accept)
        g.replay()
        o_e, i_e = la.verify_chain(q.to(DEV), k.to(DEV), v.to(DEV), s, pool_e, idx_d, N)
        la.commit_accepted(i_e, accept.to(DEV), pool_e, idx_d)
        la.poll_error()
        assert torch.equal(out.cpu(), o_e.cpu()), f"step {step}: replay != eager output"
        assert torch.equal(pool_g.cpu(), pool_e.cpu()), f"step {step}: replay != eager pool"
        o_ref, i_ref = oracle.verify_chain(q.float().numpy(), k.float().numpy(),
                                           v.float().numpy(), sl, ref_pool, idx.numpy(), N, H, D)
        ref_pool = oracle.commit_accepted(i_ref, accept.numpy(), ref_pool, idx.numpy())
        assert_close(to64(out), o_ref, f"graph verify step {step}")
    assert_close(to64(pool_g.cpu()), ref_pool, "graph verify+commit: final pool")


def test_extend_graph_replay():
    lengths = [300, 1100, 77, 2049]
    w = workloads.custom_extend(lengths, H=4, layer_id=1, L=3, prefix=[1, 0, 1, 1], seed=21)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    T, max_len = w.T, max(lengths)
    pool0 = w.materialize_pool()
    nbytes = la.extend_workspace_size(w.B, T, w.H, w.D, max_len)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=DEV)
    qs, ks, vs = (torch.zeros(T, w.H * w.D, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    out = torch.empty(T, w.H * w.D, dtype=torch.bfloat16, device=DEV)
    pool_g = pool0.to(DEV)
    idx_d, cu_d, pm_d = w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV)
    g, _ = _capture(lambda: la.extend(qs, ks, vs, s, pool_g, idx_d, cu_d, pm_d, out=out,
                                      max_seqlen=max_len, workspace=ws))
    la.poll_error()
    sl = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    for step in range(2):
        q, k, v = (_rand_bf16((T, w.H * w.D), 300 + 10 * step + j) for j in range(3))
        pool_g.copy_(pool0.to(DEV))
        qs.copy_(q)
        ks.copy_(k)
        vs.copy_(v)
        g.replay()
        pool_e = pool0.to(DEV)
        o_e = la.extend(q.to(DEV), k.to(DEV), v.to(DEV), s, pool_e, idx_d, cu_d, pm_d,
                        max_seqlen=max_len, workspace=ws)
        la.poll_error()
        assert torch.equal(out.cpu(), o_e.cpu()), f"step {step}: replay != eager output"
        assert torch.equal(pool_g.cpu().view(torch.int32), pool_e.cpu().view(torch.int32))
        o_ref, p_ref = oracle.extend(q.float().numpy(), k.float().numpy(), v.float().numpy(), sl,
                                     pool0.double().numpy(), w.state_idx.numpy(),
                                     w.cu_seqlens.numpy(), w.prefix_mask.numpy(), w.H, w.D)
        assert_close(to64(out), o_ref, f"graph extend step {step}: out")
        named = w.state_idx.long()
        assert_close(to64(pool_g.cpu()[named]), p_ref[w.state_idx.numpy()],
                     f"graph extend step {step}: final states")

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Workloads are the five fixed ones (tiny, decode batch, varlen extend, long prefill, chain verify)
at their full sizes, in the same launch configuration the benchmark times, and every output and
state element is compared.  Where the host copies would be large (the long prefill's 1 GiB per
fp64 tensor, the chain verify's 2.7 GB of intermediate states), the oracle runs over groups of
heads or requests in turn, so host memory stays bounded.  Tolerance: atol = rtol = 3e-2 (see
la_testutil).  Slot routing is checked bit for bit: slots no request names keep their contents
exactly.
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


def gpu_slopes(w):
    return la.slopes(w.H, w.layer_id, w.L).to(DEV)


def named_slot_mask(num_slots, idx):
    m = np.zeros(num_slots, dtype=bool)
    m[np.asarray(idx)] = True
    return m


def run_gpu_extend(w, pool_dev):
    q, k, v = w.q.to(DEV), w.k.to(DEV), w.v.to(DEV)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1])
    out = la.extend(q, k, v, gpu_slopes(w), pool_dev, w.state_idx.to(DEV), w.cu_seqlens.to(DEV),
                    w.prefix_mask.to(DEV), max_seqlen=int(lens.max()) if w.B else 0)
    la.poll_error()
    return out


def oracle_extend_heads(w, pool_np, heads):
    """Oracle extend on a subset of heads (columns sliced out of q, k, v and the pool)."""
    D = w.D
    cols = torch.from_numpy(np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads]))
    # slice the bf16 tensors before widening them: a full long-prefill q is 1 GiB in fp64
    q = w.q[:, cols].float().numpy()
    k = w.k[:, cols].float().numpy()
    v = w.v[:, cols].float().numpy()
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)[heads]
    sub_pool = pool_np[:, heads]
    out, pool_after = oracle.extend(q, k, v, s, sub_pool, w.state_idx.numpy(), w.cu_seqlens.numpy(),
                                    w.prefix_mask.numpy(), len(heads), D)
    return out, pool_after


def check_extend(w, head_group=None):
    """Every output and final-state element against the oracle; the oracle runs over groups of
    head_group heads (all heads at once when None) to bound host memory."""
    pool0 = w.materialize_pool()
    pool_dev = pool0.to(DEV)
    out = run_gpu_extend(w, pool_dev)
    pool_after = pool_dev.cpu()
    pool_np = pool0.double().numpy()
    idx = w.state_idx.numpy()
    D = w.D
    step = w.H if head_group is None else head_group
    for h0 in range(0, w.H, step):
        heads = list(range(h0, min(w.H, h0 + step)))
        o_ref, p_ref = oracle_extend_heads(w, pool_np, heads)
        got = to64(out[:, heads[0] * D:(heads[-1] + 1) * D])
        assert_close(got, o_ref, f"{w.name}: out (heads {heads[0]}..{heads[-1]})")
        got_states = pool_after[torch.from_numpy(idx).long()][:, heads].double().numpy()
        assert_close(got_states, p_ref[idx], f"{w.name}: final states (heads {heads[0]}..{heads[-1]})")
        del o_ref, p_ref, got
    # untouched slots: bit-identical
    untouched = ~named_slot_mask(w.num_slots, idx)
    assert torch.equal(pool_after[torch.from_numpy(untouched)].view(torch.int32),
                       pool0[torch.from_numpy(untouched)].view(torch.int32)), \
        f"{w.name}: an untouched slot changed"
    return out, pool_dev


def test_tiny_extend_then_decode():
    w = workloads.tiny(0)
    out, pool_dev = check_extend(w)
    # 4 decode steps per request, each against the oracle continuing from the oracle's state
    pool_np = w.materialize_pool().double().numpy()
    _, pool_np = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                               oracle_slopes_fp32(w.H, w.layer_id, w.L), pool_np,
                               w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                               w.H, w.D)
    s_gpu = gpu_slopes(w)
    for step, (q, k, v) in enumerate(w.decode_steps):
        o = la.decode(q.to(DEV), k.to(DEV), v.to(DEV), s_gpu, pool_dev, w.state_idx.to(DEV))
        la.poll_error()
        o_ref, pool_np = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                       oracle_slopes_fp32(w.H, w.layer_id, w.L), pool_np,
                                       w.state_idx.numpy(), w.H, w.D)
        assert_close(to64(o), o_ref, f"tiny decode step {step}: out")
        idx = w.state_idx.numpy()
        assert_close(pool_dev.cpu().double().numpy()[idx], pool_np[idx],
                     f"tiny decode step {step}: states")
    # the sentinel slots are still exactly 54321.0
    untouched = ~named_slot_mask(w.num_slots, w.state_idx.numpy())
    assert (pool_dev.cpu()[torch.from_numpy(untouched)] == workloads.SENTINEL).all()


def test_decode_batch_full():
    w = workloads.decode_batch(0)
    pool0 = w.materialize_pool()
    pool_dev = pool0.to(DEV)
    out = la.decode(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), gpu_slopes(w), pool_dev,
                    w.state_idx.to(DEV))
    la.poll_error()
    idx = w.state_idx.numpy()
    # the oracle sees only the named slots, renumbered 0..B-1 (slot routing is checked separately)
    sub = pool0[torch.from_numpy(idx).long()].double().numpy()
    o_ref, p_ref = oracle.decode(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L), sub,
                                 np.arange(w.B, dtype=np.int32), w.H, w.D)
    assert_close(to64(out), o_ref, "decode: out")
    pool_after = pool_dev.cpu()
    assert_close(pool_after[torch.from_numpy(idx).long()].double().numpy(), p_ref,
                 "decode: updated states")
    untouched = torch.from_numpy(~named_slot_mask(w.num_slots, idx))
    assert torch.equal(pool_after[untouched].view(torch.int32), pool0[untouched].view(torch.int32))


def test_varlen_extend_full():
    check_extend(workloads.varlen_extend(0))


def test_long_prefill_full():
    # all 32 heads of the 32,768-token request, 8 heads per oracle pass
    check_extend(workloads.long_prefill(0), head_group=8)


def test_verify_chain_full():
    w = workloads.verify_chain(0)
    pool0 = w.materialize_pool()
    pool_dev = pool0.to(DEV)
    out, inter = la.verify_chain(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), gpu_slopes(w), pool_dev,
                                 w.state_idx.to(DEV), w.N)
    la.poll_error()
    assert torch.equal(pool_dev.cpu().view(torch.int32), pool0.view(torch.int32)), \
        "verify modified the pool"
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    idx = w.state_idx.numpy()
    out64 = to64(out)
    group = 16
    for g0 in range(0, w.B, group):
        reqs = np.arange(g0, min(g0 + group, w.B))
        rows = np.concatenate([np.arange(b * w.N, (b + 1) * w.N) for b in reqs])
        sub_pool = pool0[torch.from_numpy(idx[reqs]).long()].double().numpy()
        o_ref, i_ref = oracle.verify_chain(w.q.float().numpy()[rows], w.k.float().numpy()[rows],
                                           w.v.float().numpy()[rows], s, sub_pool,
                                           np.arange(len(reqs), dtype=np.int32), w.N, w.H, w.D)
        assert_close(out64[rows], o_ref, f"verify: out (requests {reqs[0]}..{reqs[-1]})")
        # every intermediate state of the group: [16, 5, 64, 128, 128]
        assert_close(inter[g0:g0 + len(reqs)].cpu().double().numpy(), i_ref,
                     f"verify: intermediate states (requests {reqs[0]}..{reqs[-1]})")
        del o_ref, i_ref

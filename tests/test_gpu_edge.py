"""GPU edge cases: ragged lengths around chunk boundaries, empty and zero-length requests, split
invariance, streams, and device-side input checks (which report through la_poll_error)."""
import numpy as np
import pytest
import torch

import lightning_attention_gb300 as la
import oracle
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, oracle_slopes_fp32, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def run_pair(w):
    pool0 = w.materialize_pool()
    pool_dev = pool0.to(DEV)
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV),
                    la.slopes(w.H, w.layer_id, w.L).to(DEV), pool_dev, w.state_idx.to(DEV),
                    w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    la.poll_error()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L),
                                 pool0.double().numpy(), w.state_idx.numpy(),
                                 w.cu_seqlens.numpy(), w.prefix_mask.numpy(), w.H, w.D)
    return out, pool_dev, pool0, o_ref, p_ref


def check(w):
    out, pool_dev, pool0, o_ref, p_ref = run_pair(w)
    assert_close(to64(out), o_ref, f"{w.name}: out")
    idx = w.state_idx.numpy()
    pa = pool_dev.cpu()
    assert_close(pa.double().numpy()[idx], p_ref[idx], f"{w.name}: states")
    untouched = np.ones(w.num_slots, bool)
    untouched[idx] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32))


@pytest.mark.parametrize("lengths", [
    [1], [2, 3], [127], [128], [129], [255, 256, 257], [37, 64],
    [1, 128, 0, 130, 383, 5, 64, 65],
    [0, 0, 0],
])
def test_ragged_lengths(lengths):
    check(workloads.custom_extend(lengths, H=3, layer_id=1, L=3, seed=len(lengths)))


def test_many_heads_and_requests():
    rng = np.random.default_rng(3)
    lengths = [int(x) for x in rng.integers(0, 300, size=24)]
    check(workloads.custom_extend(lengths, H=8, layer_id=2, L=4, seed=11))


def test_empty_batch_is_noop():
    w = workloads.custom_extend([], H=2)
    pool = torch.zeros(2, 2, 128, 128, device=DEV)
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV), pool,
                    w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    la.poll_error()
    assert out.shape == (0, 256)


@pytest.mark.parametrize("split", [1, 100, 127, 128, 129, 300])
def test_split_invariance_gpu(split):
    """extend(A) then extend(B) from the carried state matches one pass over A||B."""
    n = 400
    w = workloads.custom_extend([n], H=2, prefix=[1], seed=5)
    s = la.slopes(2, 0, 1).to(DEV)
    q, k, v = w.q.to(DEV), w.k.to(DEV), w.v.to(DEV)
    idx = w.state_idx.to(DEV)
    pool_a = w.materialize_pool(DEV)
    pool_b = pool_a.clone()
    ones = torch.ones(1, dtype=torch.uint8, device=DEV)
    full = la.extend(q, k, v, s, pool_a, idx, torch.tensor([0, n], dtype=torch.int32, device=DEV),
                     ones)
    o1 = la.extend(q[:split].contiguous(), k[:split].contiguous(), v[:split].contiguous(), s,
                   pool_b, idx, torch.tensor([0, split], dtype=torch.int32, device=DEV), ones)
    o2 = la.extend(q[split:].contiguous(), k[split:].contiguous(), v[split:].contiguous(), s,
                   pool_b, idx, torch.tensor([0, n - split], dtype=torch.int32, device=DEV), ones)
    la.poll_error()
    assert_close(to64(torch.cat([o1, o2])), to64(full), "split: out")
    assert_close(pool_b.cpu().double().numpy(), pool_a.cpu().double().numpy(), "split: state")


def test_runs_on_a_side_stream():
    w = workloads.custom_extend([70, 200], H=2, seed=9)
    out_ref, pool_ref_dev, *_ = run_pair(w)
    st = torch.cuda.Stream()
    pool_dev = w.materialize_pool(DEV)
    with torch.cuda.stream(st):
        out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV),
                        pool_dev, w.state_idx.to(DEV), w.cu_seqlens.to(DEV),
                        w.prefix_mask.to(DEV))
        la.poll_error()
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out_ref.cpu())
    assert torch.equal(pool_dev.cpu(), pool_ref_dev.cpu())


def test_slot_out_of_range_is_reported_not_written():
    w = workloads.custom_extend([10, 20], H=2, prefix=[0, 0], num_slots=4, seed=2,
                                shuffle_slots=False)
    pool = torch.zeros(4, 2, 128, 128, device=DEV)
    bad_idx = torch.tensor([1, 7], dtype=torch.int32, device=DEV)
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV), pool, bad_idx,
              w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    la.poll_error()  # cleared
    # decode and verify check the same way
    q = torch.zeros(2, 256, dtype=torch.bfloat16, device=DEV)
    la.decode(q, q, q, la.slopes(2, 0, 1).to(DEV), pool,
              torch.tensor([0, -1], dtype=torch.int32, device=DEV))
    with pytest.raises(la.LAError):
        la.poll_error()
    la.verify_chain(q, q, q, la.slopes(2, 0, 1).to(DEV), pool,
                    torch.tensor([4, 0], dtype=torch.int32, device=DEV), 1)
    with pytest.raises(la.LAError):
        la.poll_error()
    la.poll_error()


def test_bad_cu_seqlens_is_reported():
    w = workloads.custom_extend([10, 20], H=2, prefix=[0, 0], seed=2)
    pool = torch.zeros(w.num_slots, 2, 128, 128, device=DEV)
    cu = torch.tensor([0, 25, 20], dtype=torch.int32, device=DEV)  # decreasing
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV), pool,
              w.state_idx.to(DEV), cu, w.prefix_mask.to(DEV))
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5


@pytest.mark.parametrize("lengths,H,max_seqlen", [
    ([100, 300], 2, 200),          # one CTA per (request, head): no split
    ([8192, 2048], 16, 4096),      # the split schedule (block states in the workspace)
])
def test_request_longer_than_max_seqlen_is_reported_not_written(lengths, H, max_seqlen):
    """max_seqlen is the caller's bound on every request's length.  A longer request is skipped
    -- no output row, no state written -- and reported as LA_ERR_DEVICE_INPUT; the requests
    within the bound are computed as usual."""
    w = workloads.custom_extend(lengths, H=H, prefix=[1] * len(lengths), seed=41)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = torch.full((w.T, H * 128), 7.0, dtype=torch.bfloat16, device=DEV)
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(H, 0, 1).to(DEV), pool,
              w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), out=out,
              max_seqlen=max_seqlen)
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    la.poll_error()  # cleared
    cu = w.cu_seqlens.numpy()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(H, 0, 1), pool0.double().numpy(),
                                 w.state_idx.numpy(), cu, w.prefix_mask.numpy(), H, 128)
    out_h, pool_h = out.cpu(), pool.cpu()
    for b, n in enumerate(lengths):
        rows = slice(int(cu[b]), int(cu[b + 1]))
        slot = int(w.state_idx[b])
        if n > max_seqlen:
            assert (out_h[rows] == 7.0).all(), f"request {b} wrote output rows"
            assert torch.equal(pool_h[slot].view(torch.int32), pool0[slot].view(torch.int32)), \
                f"request {b} wrote its state"
        else:
            assert_close(to64(out_h[rows]), o_ref[rows], f"request {b}: out")
            assert_close(pool_h[slot].double().numpy(), p_ref[slot], f"request {b}: state")


def test_verify_small_and_decode_identity():
    """Verify outputs and states equal successive decodes from the same pool state."""
    w = workloads.custom_verify(3, 4, H=2, seed=4)
    s = la.slopes(2, 0, 1).to(DEV)
    pool = w.materialize_pool(DEV)
    out, inter = la.verify_chain(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s, pool,
                                 w.state_idx.to(DEV), w.N)
    la.poll_error()
    pool2 = pool.clone()
    for t in range(w.N):
        rows = torch.arange(w.B) * w.N + t
        o = la.decode(w.q[rows].to(DEV), w.k[rows].to(DEV), w.v[rows].to(DEV), s, pool2,
                      w.state_idx.to(DEV))
        la.poll_error()
        assert torch.equal(o.cpu(), out.cpu()[rows])
        idx = w.state_idx.long()
        assert torch.equal(pool2.cpu()[idx], inter.cpu()[:, t])


def test_large_batch_longest_first_changes_only_the_schedule():
    """Above 256 requests the longest-first order comes from a ranking pre-pass into the
    workspace.  Every (request, head) is computed the same way in any order, so the result equals
    the index-order run (no workspace) bit for bit, and the oracle within the tolerance.  Many
    equal lengths exercise the ties (broken by request index)."""
    rng = np.random.default_rng(17)
    lengths = [int(x) for x in rng.choice([0, 1, 37, 128, 129, 200, 300], size=600)]
    w = workloads.custom_extend(lengths, H=2, layer_id=1, L=3, seed=19)
    assert la.extend_workspace_size(w.B, w.T, w.H, 128, 300) >= 4 * w.B
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 1, 3).to(DEV))
    rest = (w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    pool_a, pool_b = w.materialize_pool(DEV), w.materialize_pool(DEV)
    out_a = la.extend(*args, pool_a, *rest, max_seqlen=300)                   # ranked
    out_b = la.extend(*args, pool_b, *rest, max_seqlen=300, workspace=False)  # index order
    la.poll_error()
    assert torch.equal(out_a.cpu(), out_b.cpu())
    assert torch.equal(pool_a.cpu().view(torch.int32), pool_b.cpu().view(torch.int32))
    pool0 = w.materialize_pool()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(2, 1, 3), pool0.double().numpy(),
                                 w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                 2, 128)
    assert_close(to64(out_a), o_ref, "large batch: out")
    idx = w.state_idx.numpy()
    assert_close(pool_a.cpu().double().numpy()[idx], p_ref[idx], "large batch: states")


def test_batch_above_the_ranking_limit_runs_in_index_order():
    """65,636 one-head requests (0-129 tokens, every other one with a prefix state) is above the
    65,536 requests the longest-first ranking and the persistent grid's records take, so the
    workspace asks for neither and one CTA per (request, head) runs in index order, about 430
    waves.  Every 61st request (and the last one) is compared with the oracle run on those
    requests alone; the slot past the batch keeps its bytes."""
    B, H, D = 65536 + 100, 1, 128
    cycle = [1, 2, 3, 0, 129, 5, 64, 7]
    lengths = [cycle[b % len(cycle)] for b in range(B)]
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    assert la.extend_workspace_size(B, T, H, D, 129) == 0, "no ranking, no records, no split"
    g = torch.Generator().manual_seed(23)
    q, k, v = (torch.randn(T, H * D, generator=g).to(torch.bfloat16) for _ in range(3))
    pm = torch.tensor([b % 2 for b in range(B)], dtype=torch.uint8)
    # the prefix states as a pattern cheap to rebuild on both sides: slot b holds 0.05 * N(0,1)
    # values drawn per slot from a small table, so that 4.3 GB never sits on the host
    table = torch.randn(16, H, D, D, generator=g) * 0.05
    pool = torch.empty(B + 1, H, D, D, device=DEV)
    tdev = table.to(DEV)
    for s0 in range(0, B + 1, 4096):
        s1 = min(B + 1, s0 + 4096)
        sl = torch.arange(s0, s1, device=DEV)
        pool[s0:s1] = tdev[sl % 16]
    sentinel = pool[B].clone()
    idx = torch.arange(B, dtype=torch.int32)
    s = la.slopes(H, 1, 3)
    out = la.extend(q.to(DEV), k.to(DEV), v.to(DEV), s.to(DEV), pool, idx.to(DEV),
                    torch.from_numpy(cu.astype(np.int32)).to(DEV), pm.to(DEV), max_seqlen=129)
    la.poll_error()
    assert torch.equal(pool[B].view(torch.int32), sentinel.view(torch.int32))
    pick = sorted(set(range(0, B, 61)) | {B - 1})
    sub_len = [lengths[b] for b in pick]
    sub_cu = np.zeros(len(pick) + 1, dtype=np.int32)
    sub_cu[1:] = np.cumsum(sub_len)
    rows = torch.from_numpy(np.concatenate([np.arange(cu[b], cu[b + 1]) for b in pick]))
    pool0 = np.stack([table[b % 16].double().numpy() for b in pick])
    o_ref, p_ref = oracle.extend(q[rows].float().numpy(), k[rows].float().numpy(),
                                 v[rows].float().numpy(), oracle_slopes_fp32(H, 1, 3), pool0,
                                 np.arange(len(pick), dtype=np.int32), sub_cu,
                                 pm.numpy()[pick], H, D)
    assert_close(to64(out[rows.to(DEV)]), o_ref, "above the ranking limit: out")
    got = pool[torch.tensor(pick, device=DEV)].cpu().double().numpy()
    assert_close(got, p_ref, "above the ranking limit: states")

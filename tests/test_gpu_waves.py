"""Extend batches with more (request, head) CTAs than SMs: the grid runs in several waves, and
the CTAs of later waves reuse the SMs (shared memory, tensor memory) that earlier ones freed.

Checked here through the C ABI: a many-wave batch (ragged lengths, empty and one-token requests,
mixed prefixes) against the fp64 oracle, with state-tracking snapshots and a head-major output;
every request's outputs and final state equal, bit for bit, the same request extended alone, since
a CTA computes its (request, head) the same way whichever wave it runs in; slots that no request
names keep their bytes.
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


def _lengths(B, seed):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(1, 700, size=B)]
    lens[3] = 0
    lens[7] = 1
    lens[11] = 128
    lens[12] = 129
    return lens


def _many_waves_batch(seed=61):
    # 48 requests x 8 heads = 384 items, about 2.5 per SM
    lens = _lengths(48, seed)
    return workloads.custom_extend(lens, H=8, prefix=[(b * 7) % 3 != 0 for b in range(48)],
                                   layer_id=1, L=3, seed=seed, num_slots=160)


def test_many_waves_against_the_oracle_with_snapshots_and_head_major_output():
    w = _many_waves_batch()
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert w.B * w.H > sms, "the batch must take more than one wave"
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    used = set(w.state_idx.tolist())
    free = [s for s in range(w.num_slots) if s not in used]
    tl = [(n // 2 if b % 4 == 0 else (-1 if b % 4 == 1 else n)) for b, n in enumerate(lens)]
    ti = [free[b] for b in range(w.B)]
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    hm = torch.full((w.H, w.T, w.D), 3.0, dtype=torch.bfloat16, device=DEV)
    la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV), pool,
              w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
              out=hm.transpose(0, 1), max_seqlen=max(lens),
              track_lens=torch.tensor(tl, dtype=torch.int32, device=DEV),
              track_state_idx=torch.tensor(ti, dtype=torch.int32, device=DEV))
    la.poll_error()
    o_ref, p_ref = oracle.extend_tracked(w.q.float().numpy(), w.k.float().numpy(),
                                         w.v.float().numpy(),
                                         oracle_slopes_fp32(w.H, w.layer_id, w.L),
                                         pool0.double().numpy(), w.state_idx.numpy(),
                                         w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                         np.asarray(tl, dtype=np.int32),
                                         np.asarray(ti, dtype=np.int32), w.H, w.D)
    got = to64(hm.transpose(0, 1).reshape(w.T, w.H * w.D))
    assert_close(got, o_ref, "many waves: out")
    pa = pool.cpu()
    named = sorted(set(w.state_idx.tolist()) | {t for t, x in zip(ti, tl) if x >= 0})
    assert_close(pa.double().numpy()[named], p_ref[named], "many waves: states and snapshots")
    untouched = np.ones(w.num_slots, bool)
    untouched[named] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32))


def test_every_item_equals_its_request_alone():
    w = _many_waves_batch(seed=62)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s, pool, w.state_idx.to(DEV),
                    w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), max_seqlen=max(lens))
    la.poll_error()
    cu = w.cu_seqlens.tolist()
    la.set_column_split(False)  # alone, a request would otherwise run as two column halves
    try:
        _compare_alone(w, lens, cu, s, pool0, out, pool)
    finally:
        la.set_column_split(True)


def _compare_alone(w, lens, cu, s, pool0, out, pool):
    for b in range(w.B):
        rows = slice(cu[b], cu[b + 1])
        pool_b = pool0.to(DEV)
        out_b = la.extend(w.q[rows].to(DEV), w.k[rows].to(DEV), w.v[rows].to(DEV), s, pool_b,
                          w.state_idx[b:b + 1].to(DEV),
                          torch.tensor([0, lens[b]], dtype=torch.int32, device=DEV),
                          w.prefix_mask[b:b + 1].to(DEV), max_seqlen=max(lens[b], 1),
                          workspace=False)
        la.poll_error()
        assert torch.equal(out_b.cpu(), out[rows].cpu()), f"request {b}: out differs"
        slot = int(w.state_idx[b])
        assert torch.equal(pool_b[slot].cpu().view(torch.int32), pool[slot].cpu().view(torch.int32)), \
            f"request {b}: final state differs"


def _persistent_batch(seed):
    # 40 requests x 8 heads = 320 items: zero-length ones with and without a prefix, one-token,
    # chunk-boundary and long requests
    lens = _lengths(40, seed)
    lens[0] = 0
    lens[1] = 0
    lens[20] = 1500
    return workloads.custom_extend(lens, H=8, prefix=[b % 3 != 1 for b in range(40)],
                                   layer_id=2, L=5, seed=seed, num_slots=128)


def _run(w, persistent, track=None, head_major=False, state_idx=None, max_seqlen=None):
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    pool = w.materialize_pool().to(DEV)
    out = torch.full((w.H, w.T, w.D) if head_major else (w.T, w.H * w.D), 5.0,
                     dtype=torch.bfloat16, device=DEV)
    kw = {}
    if track is not None:
        kw = dict(track_lens=torch.tensor(track[0], dtype=torch.int32, device=DEV),
                  track_state_idx=torch.tensor(track[1], dtype=torch.int32, device=DEV))
    idx = w.state_idx if state_idx is None else state_idx
    la.set_persistent(persistent)
    try:
        la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
                  pool, idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
                  out=out.transpose(0, 1) if head_major else out,
                  max_seqlen=max(lens) if max_seqlen is None else max_seqlen, **kw)
        torch.cuda.synchronize()
    finally:
        la.set_persistent(True)
    return out.cpu(), pool.cpu()


def test_persistent_grid_equals_one_cta_per_item():
    """The persistent grid (one CTA per SM over all (request, head) items) and one CTA per item
    give the same bits: outputs in the head-major layout, final states, tracking snapshots at
    token 0, mid-request and at the end, and every other slot."""
    w = _persistent_batch(71)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert w.B * w.H > sms
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    # the planner keeps the persistent grid's request records (32 bytes each) in the workspace
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, max(lens)) == 32 * w.B
    used = set(w.state_idx.tolist())
    free = [s for s in range(w.num_slots) if s not in used]
    tl = [(0, n // 3, n, -1)[b % 4] for b, n in enumerate(lens)]
    track = (tl, [free[b] for b in range(w.B)])
    o1, p1 = _run(w, True, track=track, head_major=True)
    la.poll_error()
    o0, p0 = _run(w, False, track=track, head_major=True)
    la.poll_error()
    assert torch.equal(o1, o0), "out differs between the grids"
    assert torch.equal(p1.view(torch.int32), p0.view(torch.int32)), "pool differs between the grids"
    # and the plain call (packed output, no tracking) the same way
    o1, p1 = _run(w, True)
    o0, p0 = _run(w, False)
    la.poll_error()
    assert torch.equal(o1, o0) and torch.equal(p1.view(torch.int32), p0.view(torch.int32))


def test_faulty_requests_in_a_persistent_batch_are_reported_and_skipped():
    """A slot out of range and a request longer than max_seqlen, inside a batch that takes the
    persistent grid: both are reported as LA_ERR_DEVICE_INPUT and write nothing; every other
    request is computed as one CTA per item computes it."""
    w = _persistent_batch(72)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    idx = w.state_idx.clone()
    idx[5] = w.num_slots + 3
    cap = sorted(lens)[-2]  # the single longest request (1500 tokens) exceeds it
    assert lens[20] > cap
    results = []
    for persistent in (True, False):
        o, pl = _run(w, persistent, state_idx=idx, max_seqlen=cap)
        with pytest.raises(la.LAError) as e:
            la.poll_error()
        assert e.value.status == 5
        la.poll_error()  # cleared
        results.append((o, pl))
    (o1, p1), (o0, p0) = results
    assert torch.equal(o1, o0) and torch.equal(p1.view(torch.int32), p0.view(torch.int32))
    cu = w.cu_seqlens.tolist()
    pool0 = w.materialize_pool()
    for b in (5, 20):
        assert (o1[cu[b]:cu[b + 1]] == 5.0).all(), f"request {b} wrote output rows"
    assert torch.equal(p1[int(w.state_idx[20])].view(torch.int32),
                       pool0[int(w.state_idx[20])].view(torch.int32))

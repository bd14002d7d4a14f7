"""la_extend_noalloc: the extend entry point for callers that cannot allocate device memory
(for example a plugin that receives only its input and output buffers from a host framework that
owns the device memory, or a latency-critical loop that must not call cudaMalloc).  Instead of a
caller-provided workspace it uses the library's fixed 16 MiB device scratch array.

Checked here through the C ABI:
  * on a batch that takes the segment-split schedule, two calls in a row each equal la_extend
    with a caller workspace bit for bit (the same plan runs the same kernels on the same inputs);
    between them, a call on another split batch of the same shape (other seed, other prefix
    pattern) leaves different block states in the shared array, so a kernel that read scratch it
    had not written would show;
  * the split schedule really runs: the result differs bitwise from the unsplit schedule
    (la_extend without workspace), and it also matches the fp64 oracle within the parity tolerance;
  * a warmed-up no-alloc call leaves the device's free memory unchanged;
  * a batch that needs no scratch gives la_extend's results as well;
  * on this device every batch shape's split plan fits the array.
This file is collected last so that a stop-at-first-failure run has already run every other test.
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
SCRATCH_BYTES = 16 << 20


def _inputs(w):
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    return dict(q=w.q.to(DEV), k=w.k.to(DEV), v=w.v.to(DEV),
                s=la.slopes(w.H, w.layer_id, w.L).to(DEV), idx=w.state_idx.to(DEV),
                cu=w.cu_seqlens.to(DEV), pm=w.prefix_mask.to(DEV), max_seqlen=int(lens.max()))


def _extend(a, pool, workspace=None):
    out = la.extend(a["q"], a["k"], a["v"], a["s"], pool, a["idx"], a["cu"], a["pm"],
                    max_seqlen=a["max_seqlen"], workspace=workspace)
    la.poll_error()
    return out


def _noalloc(a, pool):
    out = la.extend_noalloc(a["q"], a["k"], a["v"], a["s"], pool, a["idx"], a["cu"], a["pm"],
                            max_seqlen=a["max_seqlen"])
    la.poll_error()
    return out


def _split_batch(seed, prefix):
    # two 4096-token requests with 16 heads: too few (request, head) pairs to fill the GPU, so
    # the requests are cut into segments and the scratch array carries their block states
    return workloads.custom_extend([4096, 4096], H=16, prefix=prefix, layer_id=5, L=12, seed=seed)


def test_no_alloc_equals_la_extend_bitwise_on_split_batch():
    w = _split_batch(31, [1, 0])
    other = _split_batch(77, [0, 1])
    need = la.extend_workspace_size(w.B, w.T, w.H, w.D, 4096)
    assert 0 < need <= SCRATCH_BYTES
    a, a_other = _inputs(w), _inputs(other)
    pool_ref = w.materialize_pool(DEV)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out_ref = _extend(a, pool_ref, workspace=ws)
    idx = w.state_idx.long()
    for call in range(2):
        if call == 1:
            # leave the other batch's block states and initial states in the shared array
            _noalloc(a_other, other.materialize_pool(DEV))
        pool = w.materialize_pool(DEV)
        out = _noalloc(a, pool)
        assert torch.equal(out.cpu(), out_ref.cpu()), f"no-alloc call {call + 1}: out differs"
        assert torch.equal(pool.cpu().view(torch.int32), pool_ref.cpu().view(torch.int32)), \
            f"no-alloc call {call + 1}: pool differs"

    # the segment split really ran: the unsplit schedule rounds differently somewhere ...
    pool_u = w.materialize_pool(DEV)
    out_u = _extend(a, pool_u, workspace=False)
    assert not (torch.equal(out_u.cpu(), out_ref.cpu()) and
                torch.equal(pool_u.cpu()[idx], pool_ref.cpu()[idx])), \
        "the no-alloc result equals the unsplit schedule's bit for bit"
    # ... and both agree with the fp64 oracle
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L),
                                 w.materialize_pool().double().numpy(), w.state_idx.numpy(),
                                 w.cu_seqlens.numpy(), w.prefix_mask.numpy(), w.H, w.D)
    assert_close(to64(out_ref), o_ref, "no-alloc: out vs oracle")
    assert_close(pool_ref.cpu()[idx].double().numpy(), p_ref[w.state_idx.numpy()],
                 "no-alloc: final states vs oracle")


def test_no_alloc_allocates_nothing():
    w = _split_batch(5, [1, 1])
    a = _inputs(w)
    pool = w.materialize_pool(DEV)
    out = torch.empty_like(a["q"])
    # warm-up: loads the module (and its scratch array) and looks up the array's address
    la.extend_noalloc(a["q"], a["k"], a["v"], a["s"], pool, a["idx"], a["cu"], a["pm"], out=out,
                      max_seqlen=a["max_seqlen"])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        la.extend_noalloc(a["q"], a["k"], a["v"], a["s"], pool, a["idx"], a["cu"], a["pm"],
                          out=out, max_seqlen=a["max_seqlen"])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    la.poll_error()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"


def test_no_alloc_matches_la_extend_on_unsplit_batch():
    w = workloads.custom_extend([300, 1, 129, 0], H=16, prefix=[1, 0, 1, 0], seed=32)
    a = _inputs(w)
    # no sequence split: the only scratch is the balanced schedule's plan (a few KiB of records)
    assert 0 < la.extend_workspace_size(w.B, w.T, w.H, w.D, a["max_seqlen"]) < 65536
    pool_ref = w.materialize_pool(DEV)
    out_ref = _extend(a, pool_ref)
    for call in range(2):
        pool = w.materialize_pool(DEV)
        out = _noalloc(a, pool)
        assert torch.equal(out.cpu(), out_ref.cpu()), f"no-alloc call {call + 1}: out differs"
        assert torch.equal(pool.cpu().view(torch.int32), pool_ref.cpu().view(torch.int32)), \
            f"no-alloc call {call + 1}: pool differs"


def test_every_split_plan_fits_the_scratch_array():
    # the planner's largest request is 1.5 x SMs matrices of 64 KiB (one request, SMs / 2 heads);
    # sweep batch shapes on this device and check them against the array's size
    worst = 0
    for B in (1, 2, 3, 4, 8):
        for H in (1, 2, 4, 8, 16, 32, 48, 64, 76, 96, 128):
            for max_seqlen in (1024, 2048, 2176, 4096, 8192, 65536, 1 << 20):
                worst = max(worst, la.extend_workspace_size(B, B * max_seqlen, H, 128, max_seqlen))
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert worst <= 3 * sms * 65536 // 2
    assert worst <= SCRATCH_BYTES

"""la_extend_noalloc: the extend entry point for callers that cannot allocate device memory
(for example a plugin that receives only its input and output buffers from a host framework that
owns the device memory, or a latency-critical loop that must not call cudaMalloc).  Instead of a
caller-provided workspace it uses the library's fixed 16 MiB device scratch array.

Checked here through the C ABI: on a batch that takes the segment-split schedule (so the scratch
is really used) and on one that does not, two calls in a row must each match la_extend's output
and final states within the tolerance the other parity tests use.  The second call also checks
that nothing left in the shared scratch by the first call leaks into the result.  This file is
collected last so that a stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import lightning_attention_gb300 as la
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _inputs(w):
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    return dict(q=w.q.to(DEV), k=w.k.to(DEV), v=w.v.to(DEV),
                s=la.slopes(w.H, w.layer_id, w.L).to(DEV), idx=w.state_idx.to(DEV),
                cu=w.cu_seqlens.to(DEV), pm=w.prefix_mask.to(DEV), max_seqlen=int(lens.max()))


def _compare_two_calls(w):
    a = _inputs(w)
    pool_ref = w.materialize_pool(DEV)
    out_ref = la.extend(a["q"], a["k"], a["v"], a["s"], pool_ref, a["idx"], a["cu"], a["pm"],
                        max_seqlen=a["max_seqlen"])
    la.poll_error()
    idx = w.state_idx.numpy()
    for call in range(2):
        pool = w.materialize_pool(DEV)
        out = la.extend_noalloc(a["q"], a["k"], a["v"], a["s"], pool, a["idx"], a["cu"], a["pm"],
                                max_seqlen=a["max_seqlen"])
        la.poll_error()
        assert_close(to64(out), to64(out_ref), f"{w.name}: no-alloc call {call + 1}: out")
        assert_close(pool.cpu().double().numpy()[idx], pool_ref.cpu().double().numpy()[idx],
                     f"{w.name}: no-alloc call {call + 1}: final states")
        untouched = np.ones(w.num_slots, bool)
        untouched[idx] = False
        u = torch.from_numpy(untouched)
        assert torch.equal(pool.cpu()[u].view(torch.int32), pool_ref.cpu()[u].view(torch.int32))


def test_no_alloc_matches_la_extend_on_split_batch():
    # one 8192-token request with 32 heads: too few (request, head) pairs to fill the GPU, so the
    # request is split into segments and the scratch array carries the block states
    w = workloads.custom_extend([8192], H=32, prefix=[1], layer_id=5, L=12, seed=31)
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, 8192) > 0
    _compare_two_calls(w)


def test_no_alloc_matches_la_extend_on_unsplit_batch():
    w = workloads.custom_extend([300, 1, 129, 0], H=16, prefix=[1, 0, 1, 0], seed=32)
    _compare_two_calls(w)

"""Sequence split of long extend requests (batches too small to fill the GPU).

The split schedule reassociates the recurrence (segment start states from decayed block states);
results must match the fp64 oracle within the usual tolerance, the unsplit schedule of the same
call (workspace=False) within the same tolerance, and leave untouched and unread slots alone.
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


def run(w, workspace=None):
    pool = w.materialize_pool(DEV)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1])
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
                    pool, w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
                    max_seqlen=int(lens.max()), workspace=workspace)
    la.poll_error()
    return out, pool


def check_split(w):
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1])
    nbytes = la.extend_workspace_size(w.B, w.T, w.H, w.D, int(lens.max()))
    assert nbytes > 0, "this batch is expected to take the split schedule"
    out_s, pool_s = run(w)
    out_u, pool_u = run(w, workspace=False)
    pool0 = w.materialize_pool()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L), pool0.double().numpy(),
                                 w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                 w.H, w.D)
    idx = w.state_idx.numpy()
    assert_close(to64(out_s), o_ref, f"{w.name} split: out")
    assert_close(pool_s.cpu().double().numpy()[idx], p_ref[idx], f"{w.name} split: states")
    assert_close(to64(out_s), to64(out_u), f"{w.name}: split vs unsplit out")
    untouched = np.ones(w.num_slots, bool)
    untouched[idx] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pool_s.cpu()[u].view(torch.int32), pool0[u].view(torch.int32))


def test_single_long_request_with_prefix():
    check_split(workloads.custom_extend([5000], H=2, prefix=[1], layer_id=1, L=3, seed=21))


def test_single_long_request_without_prefix_nan_slot_unread():
    check_split(workloads.custom_extend([4099], H=2, prefix=[0], seed=22))


def test_mixed_long_and_short_requests():
    check_split(workloads.custom_extend([3000, 100, 2181, 0, 1], H=4, prefix=[1, 0, 1, 1, 0],
                                        layer_id=2, L=4, seed=23))


@pytest.mark.parametrize("n", [2048, 2049, 4096, 6143, 8192, 8193])
def test_lengths_around_segment_boundaries(n):
    check_split(workloads.custom_extend([n], H=1, prefix=[1], seed=n))


@pytest.mark.parametrize("lengths,H", [([40000], 1), ([20000, 3000], 2)])
def test_many_segments_few_heads(lengths, H):
    # one or two heads per request leave the SMs to the segments: dozens of them, so the state
    # scan between the two launches runs over many blocks (several rounds of its prefetch)
    check_split(workloads.custom_extend(lengths, H=H, prefix=[1] * len(lengths), layer_id=2, L=5,
                                        seed=sum(lengths) + H))

"""Column split of the extend kernel: when one CTA per (request, head) leaves SMs idle, the longest
requests run as two CTAs per head, each on one 64-column half of the values.

The halves compute S[:, cols] and out[:, cols] from V[:, cols] alone, so the split changes no
arithmetic but the products' column count.  Checked here against the fp64 oracle, with the split
on and off, for a batch that splits every request, one sized from the device's SM count so that
only the longest requests split, and a tracked batch into a head-major output; the slots no
request names stay bit-identical.
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


@pytest.fixture
def column_split():
    yield la.set_column_split
    la.set_column_split(True)


def run(w, split, track=None):
    la.set_column_split(split)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    kw = dict(max_seqlen=int(lens.max()), workspace=False)
    out = None
    if track is not None:
        tl, ti = track
        buf = torch.empty(w.H, w.T, 128, dtype=torch.bfloat16, device=DEV)
        out = buf.transpose(0, 1)
        kw.update(out=out, track_lens=torch.from_numpy(tl).to(DEV),
                  track_state_idx=torch.from_numpy(ti).to(DEV))
    res = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
                    pool, w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), **kw)
    la.poll_error()
    got = (out if out is not None else res).reshape(w.T, w.H * 128)
    return got, pool.cpu(), pool0


def check(w, track=None):
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    args = (w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(), s)
    tail = (w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy())
    results = {}
    for split in (True, False):
        got, pool, pool0 = run(w, split, track)
        if track is None:
            o_ref, p_ref = oracle.extend(*args, pool0.double().numpy(), *tail, w.H, w.D)
        else:
            o_ref, p_ref = oracle.extend_tracked(*args, pool0.double().numpy(), *tail, track[0],
                                                 track[1], w.H, w.D)
        tag = f"{w.name} split={split}"
        assert_close(to64(got), o_ref, f"{tag}: out")
        written = set(int(x) for x in w.state_idx.numpy())
        if track is not None:
            written |= set(int(x) for x in track[1] if x >= 0)
        idx = np.array(sorted(written), dtype=np.int64)
        assert_close(pool.double().numpy()[idx], p_ref[idx], f"{tag}: states")
        untouched = torch.ones(w.num_slots, dtype=torch.bool)
        untouched[torch.from_numpy(idx)] = False
        assert torch.equal(pool[untouched].view(torch.int32), pool0[untouched].view(torch.int32))
        results[split] = (to64(got), pool.double().numpy()[idx])
    # both schedules compute the same products: they agree far inside the tolerance (outputs to
    # about one bf16 rounding step)
    np.testing.assert_allclose(results[True][0], results[False][0], rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(results[True][1], results[False][1], rtol=1e-4, atol=1e-4)


def test_every_request_split(column_split):
    # B * H = 12 CTAs: every request runs as two CTAs per head
    w = workloads.custom_extend([1, 127, 129, 700, 0, 300], H=2, prefix=[1, 0, 1, 1, 0, 1],
                                num_slots=16, seed=71)
    check(w)


def test_longest_requests_split(column_split):
    # H = 8 and B chosen so that the idle SMs take exactly the two longest requests
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    H = 8
    B = sms // H - 2
    if B < 3:
        pytest.skip("device too small for a mixed schedule")
    rng = np.random.default_rng(72)
    lengths = [int(x) for x in rng.integers(1, 260, B)]
    lengths[3], lengths[B - 1] = 700, 640  # the two longest, not at the front of the batch
    w = workloads.custom_extend(lengths, H=H, num_slots=2 * B, seed=72)
    check(w)


def test_split_with_tracking_and_head_major_output(column_split):
    w = workloads.custom_extend([513, 96, 260, 0], H=3, prefix=[1, 1, 0, 0], num_slots=12, seed=73)
    used = set(int(x) for x in w.state_idx.numpy())
    free = [s for s in range(w.num_slots) if s not in used]
    tl = np.array([300, 96, -1, 0], dtype=np.int32)
    ti = np.array([free[0], free[1], -1, free[2]], dtype=np.int32)
    check(w, (tl, ti))

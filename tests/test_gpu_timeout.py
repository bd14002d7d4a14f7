"""The extend kernel's bounded waits: with the wait limit lowered to 1 us, its waits run out, the
kernel records LA_ERR_TIMEOUT and exits cleanly (draining its own copies and MMAs, freeing TMEM),
and the context stays usable for the next, normal call.  Nothing hangs, traps or faults."""
import pytest
import torch

import lightning_attention_gb300 as la
import oracle
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, oracle_slopes_fp32, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def test_wait_limit_drives_timeout_path_and_context_survives():
    w = workloads.custom_extend([1000, 300], H=2, seed=3)
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s)
    idx, cu, pm = w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV)
    la.set_wait_limit(1)
    try:
        la.extend(*args, w.materialize_pool(DEV), idx, cu, pm)
        with pytest.raises(la.LAError) as e:
            la.poll_error()
        assert e.value.status == 4  # LA_ERR_TIMEOUT
    finally:
        la.set_wait_limit(0)
    la.poll_error()  # the error word was cleared by the previous poll
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = la.extend(*args, pool, idx, cu, pm)
    la.poll_error()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L), pool0.double().numpy(),
                                 w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                 w.H, w.D)
    assert_close(to64(out), o_ref, "after timeout: out")
    i = w.state_idx.numpy()
    assert_close(pool.cpu().double().numpy()[i], p_ref[i], "after timeout: states")


def _timeout_then_normal(w, what, max_seqlen=None):
    """One call under a 1 us wait limit (reported as LA_ERR_TIMEOUT), then a normal call on the
    same context, compared with the oracle."""
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    ms = max(lens) if max_seqlen is None else max_seqlen
    s = la.slopes(w.H, w.layer_id, w.L).to(DEV)
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s)
    idx, cu, pm = w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV)
    la.set_wait_limit(1)
    try:
        la.extend(*args, w.materialize_pool(DEV), idx, cu, pm, max_seqlen=ms)
        with pytest.raises(la.LAError) as e:
            la.poll_error()
        assert e.value.status == 4, f"{what}: expected LA_ERR_TIMEOUT"
    finally:
        la.set_wait_limit(0)
    la.poll_error()
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = la.extend(*args, pool, idx, cu, pm, max_seqlen=ms)
    la.poll_error()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 oracle_slopes_fp32(w.H, w.layer_id, w.L), pool0.double().numpy(),
                                 w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                 w.H, w.D)
    assert_close(to64(out), o_ref, f"{what} after timeout: out")
    i = w.state_idx.numpy()
    assert_close(pool.cpu().double().numpy()[i], p_ref[i], f"{what} after timeout: states")


def test_timeout_on_the_persistent_grid():
    """A batch of more (request, head) pairs than SMs: the persistent grid's hand-over between
    items (staged final states, TMA stores and loads) leaves cleanly on a timeout."""
    lens = [(37 * b) % 400 + 1 for b in range(48)]
    w = workloads.custom_extend(lens, H=8, prefix=[b % 2 for b in range(48)], seed=71,
                                num_slots=100)
    assert w.B * w.H > torch.cuda.get_device_properties(DEV).multi_processor_count
    _timeout_then_normal(w, "persistent grid")


def test_timeout_on_the_balanced_grid():
    """A skewed one-wave batch: the plan, the prologues and the read counters of the balanced
    grid leave cleanly on a timeout."""
    w = workloads.custom_extend([4000, 300, 200, 500, 100, 700], H=16,
                                prefix=[1, 0, 1, 1, 0, 1], seed=73, num_slots=16)
    _timeout_then_normal(w, "balanced grid")


def test_timeout_on_the_split_schedule():
    """One long request cut into segments: the block-state pass, the state scan and the extend
    kernel's segments leave cleanly on a timeout."""
    w = workloads.custom_extend([9000, 50], H=2, prefix=[1, 0], seed=75, num_slots=8)
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, 9000) >= 65536
    _timeout_then_normal(w, "split schedule")

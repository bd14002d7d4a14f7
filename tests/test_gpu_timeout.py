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

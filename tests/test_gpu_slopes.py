"""Decay rates: caller-given ones from no decay to far steeper than the slope rule produces (up to
e^-100 per token, where every factor past the diagonal underflows), and the rule's slow late-layer
decays over long requests.

The recurrence is defined for any slope s >= 0; the kernels take two routes to the P decay
factors e^{-s (i - j)} (a running product for moderate s, per-element table reads for steep s), so
the slopes here straddle the switch between them.  Extend (whole-request and split schedules),
decode and chain verify are compared with the fp64 oracle given the same fp32 slopes.
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

SLOPES = np.array([0.0, 1e-3, 0.35, 0.92, 2.4, 2.6, 7.5, 100.0], dtype=np.float32)
H = len(SLOPES)


def extend_pair(w, workspace=None):
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), torch.from_numpy(SLOPES).to(DEV), pool,
                    w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
                    max_seqlen=int(lens.max()), workspace=workspace)
    la.poll_error()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                 SLOPES.astype(np.float64), pool0.double().numpy(),
                                 w.state_idx.numpy(), w.cu_seqlens.numpy(), w.prefix_mask.numpy(),
                                 w.H, w.D)
    idx = w.state_idx.numpy()
    assert_close(to64(out), o_ref, f"{w.name}: out")
    assert_close(pool.cpu().double().numpy()[idx], p_ref[idx], f"{w.name}: states")
    return pool, p_ref


def test_extend_ragged_steep_and_flat_decays():
    w = workloads.custom_extend([1, 31, 33, 128, 129, 300, 0, 64], H=H,
                                prefix=[1, 0, 1, 1, 0, 1, 1, 0], seed=41)
    extend_pair(w, workspace=False)


def test_extend_split_schedule_steep_and_flat_decays():
    w = workloads.custom_extend([4500, 7], H=H, prefix=[1, 1], seed=42)
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, int(lens.max())) > 0
    extend_pair(w)


def test_decode_and_chain_verify_steep_and_flat_decays():
    w = workloads.custom_extend([130, 5, 64], H=H, prefix=[1, 0, 1], seed=43)
    pool, p_ref = extend_pair(w, workspace=False)
    s64 = SLOPES.astype(np.float64)
    s_dev = torch.from_numpy(SLOPES).to(DEV)
    idx = w.state_idx.numpy()
    rng = np.random.default_rng(44)
    B, N = w.B, 4

    def rows(n):
        return [torch.from_numpy(rng.standard_normal((n, H * 128), dtype=np.float32)).bfloat16()
                for _ in range(3)]

    q, k, v = rows(B)
    dout = la.decode(q.to(DEV), k.to(DEV), v.to(DEV), s_dev, pool, w.state_idx.to(DEV))
    la.poll_error()
    d_ref, p_ref = oracle.decode(q.float().numpy(), k.float().numpy(), v.float().numpy(), s64,
                                 p_ref, idx, H, 128)
    assert_close(to64(dout), d_ref, "decode out")
    assert_close(pool.cpu().double().numpy()[idx], p_ref[idx], "decode states")

    q, k, v = rows(B * N)
    vout, inter = la.verify_chain(q.to(DEV), k.to(DEV), v.to(DEV), s_dev, pool,
                                  w.state_idx.to(DEV), N)
    la.poll_error()
    vo_ref, i_ref = oracle.verify_chain(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                        s64, p_ref, idx, N, H, 128)
    assert_close(to64(vout), vo_ref, "chain verify out")
    assert_close(to64(inter), i_ref, "chain verify states")


# Long memory: slow decays over thousands of tokens give states and outputs of magnitude 30-100, so
# that a relative error of a few 1e-4 in the state update already exceeds the absolute tolerance
# on outputs near zero.  The slopes are the slope rule's for late layers (1e-4 .. 6e-7).
@pytest.mark.parametrize("lengths,L,layer_id", [
    ([8192], 40, 38),
    ([16384], 8, 7),
    ([3000, 50], 8, 7),
])
@pytest.mark.parametrize("split", [True, False])
def test_extend_long_memory(lengths, L, layer_id, split):
    w = workloads.custom_extend(lengths, H=2, L=L, layer_id=layer_id, seed=12)
    lens = w.cu_seqlens[1:] - w.cu_seqlens[:-1]
    if split:
        assert la.extend_workspace_size(w.B, w.T, w.H, w.D, int(lens.max())) > 0
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, layer_id, L).to(DEV), pool,
                    w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
                    max_seqlen=int(lens.max()), workspace=None if split else False)
    la.poll_error()
    o_ref, p_ref = oracle.extend(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(), s,
                                 pool0.double().numpy(), w.state_idx.numpy(), w.cu_seqlens.numpy(),
                                 w.prefix_mask.numpy(), w.H, w.D)
    idx = w.state_idx.numpy()
    assert_close(to64(out), o_ref, f"{w.name} split={split}: out")
    assert_close(pool.cpu().double().numpy()[idx], p_ref[idx], f"{w.name} split={split}: states")

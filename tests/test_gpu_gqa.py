"""Grouped-query heads on the GPU (la_extend_gqa, la_decode_gqa) against the fp64 oracle.

The page's seg_la takes one head count for q, k and v (section "输入与配置覆盖" of "SGLang Lightning
Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析"); the grouped entry points let H query heads
share Hkv key/value heads, one state and one slope per kv head.  Checked here: outputs and final
states element by element at the parity tolerance on ragged, split and many-wave batches; with
Hkv = H the grouped calls equal the plain ones bit for bit; untouched slots keep their bytes; a
grouped extend without its workspace is refused.
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


def _check_extend_gqa(w, max_seqlen=None):
    Hkv = w.state_heads
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1])
    ms = int(lens.max()) if max_seqlen is None else max_seqlen
    out = la.extend_gqa(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV),
                        la.slopes(Hkv, w.layer_id, w.L).to(DEV), pool, w.state_idx.to(DEV),
                        w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV), max_seqlen=ms)
    la.poll_error()
    o_ref, p_ref = oracle.extend_gqa(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                     oracle_slopes_fp32(Hkv, w.layer_id, w.L),
                                     pool0.double().numpy(), w.state_idx.numpy(),
                                     w.cu_seqlens.numpy(), w.prefix_mask.numpy(), w.H, Hkv, w.D)
    assert_close(to64(out), o_ref, f"{w.name}: out")
    idx = w.state_idx.numpy()
    pa = pool.cpu()
    assert_close(pa.double().numpy()[idx], p_ref[idx], f"{w.name}: final states")
    untouched = np.ones(w.num_slots, bool)
    untouched[idx] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32))


@pytest.mark.parametrize("lengths,H,Hkv", [
    ([37, 64], 4, 2),
    ([1, 128, 0, 130, 383, 5], 8, 2),
    ([700, 129, 2000], 16, 4),
    ([300, 257], 8, 1),
])
def test_extend_gqa_matches_oracle(lengths, H, Hkv):
    _check_extend_gqa(workloads.custom_extend_gqa(lengths, H, Hkv, layer_id=1, L=3,
                                                  seed=len(lengths) + H))


def test_extend_gqa_split_schedule():
    # one 8192-token request with 16 query heads over 4 kv heads: the block states are computed
    # per kv head and shared by its four query heads' segments
    w = workloads.custom_extend_gqa([8192], 16, 4, prefix=[1], layer_id=5, L=12, seed=7)
    assert la.extend_gqa_workspace_size(w.B, w.T, w.H, 4, w.D, 8192) > 4 * 65536
    _check_extend_gqa(w)


def test_extend_gqa_many_waves_with_prefixes():
    # 24 requests x 32 query heads = 768 CTAs, several waves on the GPU: a sibling query head that
    # starts after its group's first head has written the final state back must still start from
    # the initial state
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(200, 700, size=24)]
    _check_extend_gqa(workloads.custom_extend_gqa(lengths, 32, 8, prefix=[1] * 24, seed=13))


def test_extend_gqa_with_equal_heads_is_la_extend():
    w = workloads.custom_extend([300, 45, 1000], H=4, layer_id=2, L=4, seed=21)
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(4, 2, 4).to(DEV))
    pool_a, pool_b = w.materialize_pool(DEV), w.materialize_pool(DEV)
    rest = (w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    out_a = la.extend(*args, pool_a, *rest, max_seqlen=1000)
    out_b = la.extend_gqa(*args, pool_b, *rest, max_seqlen=1000)
    la.poll_error()
    assert torch.equal(out_a.cpu(), out_b.cpu())
    assert torch.equal(pool_a.cpu().view(torch.int32), pool_b.cpu().view(torch.int32))


def test_extend_gqa_needs_its_workspace():
    w = workloads.custom_extend_gqa([50], 4, 2, seed=3)
    with pytest.raises(la.LAError) as e:
        la.extend_gqa(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(2, 0, 1).to(DEV),
                      w.materialize_pool(DEV), w.state_idx.to(DEV), w.cu_seqlens.to(DEV),
                      w.prefix_mask.to(DEV), workspace=torch.empty(16, dtype=torch.uint8,
                                                                   device=DEV))
    assert e.value.status == 1


@pytest.mark.parametrize("B,H,Hkv", [(64, 16, 4), (7, 8, 1), (33, 6, 3)])
def test_decode_gqa_matches_oracle(B, H, Hkv):
    w = workloads.custom_decode_gqa(B, H, Hkv, layer_id=3, L=8, seed=B)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    out = la.decode_gqa(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(Hkv, 3, 8).to(DEV), pool,
                        w.state_idx.to(DEV))
    la.poll_error()
    o_ref, p_ref = oracle.decode_gqa(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy(),
                                     oracle_slopes_fp32(Hkv, 3, 8), pool0.double().numpy(),
                                     w.state_idx.numpy(), H, Hkv, w.D)
    assert_close(to64(out), o_ref, "grouped decode: out")
    pa = pool.cpu()
    assert_close(pa.double().numpy(), p_ref, "grouped decode: states")
    untouched = np.ones(w.num_slots, bool)
    untouched[w.state_idx.numpy()] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32))


def test_decode_gqa_with_equal_heads_is_la_decode():
    w = workloads.custom_decode_gqa(40, 8, 8, seed=9)
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(8, 0, 1).to(DEV))
    pool_a, pool_b = w.materialize_pool(DEV), w.materialize_pool(DEV)
    out_a = la.decode(*args, pool_a, w.state_idx.to(DEV))
    out_b = la.decode_gqa(*args, pool_b, w.state_idx.to(DEV))
    la.poll_error()
    assert torch.equal(out_a.cpu(), out_b.cpu())
    assert torch.equal(pool_a.cpu(), pool_b.cpu())

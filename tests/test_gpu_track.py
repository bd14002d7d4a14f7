"""GPU parity of prefill state tracking (la_extend_ex) against the fp64 oracle.

The page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析" (section
"额外覆盖：mamba 状态跟踪与布局鲁棒性") describes the check: at the track_len-th token the running
state is copied into a track slot, the request's own slot still ends with the final state, and
every other slot keeps the sentinel 54321.0.  Checked here, with and without the sequence split:
snapshots at 0, inside the first chunk, inside and on chunk boundaries, on segment boundaries and
at the request's end, for prefix and zero-start requests; outputs, final states and snapshots
within tolerance of the oracle; requests whose chunking is unchanged (no snapshot, or one on the
128-token grid) bit-identical to la_extend; untouched slots bit-identical; bad entries reported
and not written.
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


def _bits(t):
    return t.detach().cpu().view(torch.int32)


def _run(w, tl, tidx, pool0, workspace, tracked=True):
    pool = pool0.to(DEV)
    kw = {}
    if tracked:
        kw = dict(track_lens=torch.tensor(tl, dtype=torch.int32, device=DEV),
                  track_state_idx=torch.tensor(tidx, dtype=torch.int32, device=DEV))
    out = la.extend(w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), la.slopes(w.H, w.layer_id, w.L).to(DEV),
                    pool, w.state_idx.to(DEV), w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV),
                    max_seqlen=max(int(x) for x in (w.cu_seqlens[1:] - w.cu_seqlens[:-1])) or 1,
                    workspace=workspace, **kw)
    return out, pool


def _free_slots(w, count, seed):
    used = set(w.state_idx.tolist())
    free = [s for s in range(w.num_slots) if s not in used]
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.choice(free, size=count, replace=False)]


def _same_grid(tl, n):
    """A snapshot on the 128-token chunk grid (or none) leaves the request's chunking, and so
    its rounding, exactly as in la_extend; any other track length restarts the grid there."""
    return tl < 0 or tl == n or tl % 128 == 0


def _check(w, tl, tidx, workspace, what):
    pool0 = w.materialize_pool()
    out, pool = _run(w, tl, tidx, pool0, workspace)
    la.poll_error()
    out_p, pool_p = _run(w, tl, tidx, pool0, workspace, tracked=False)
    la.poll_error()
    got, out_c, out_pc, pool_pc = pool.cpu(), out.cpu(), out_p.cpu(), pool_p.cpu()
    cu = w.cu_seqlens.tolist()
    for b in range(w.B):
        if _same_grid(tl[b], cu[b + 1] - cu[b]):
            rows = slice(cu[b], cu[b + 1])
            slot = int(w.state_idx[b])
            assert torch.equal(out_c[rows], out_pc[rows]), f"{what}: request {b} outputs"
            assert torch.equal(_bits(got[slot]), _bits(pool_pc[slot])), f"{what}: request {b}"
    written = {tidx[b] for b in range(w.B) if tl[b] >= 0}
    for s in range(w.num_slots):
        if s not in written and s not in set(w.state_idx.tolist()):
            assert torch.equal(_bits(got[s]), _bits(pool0[s])), f"{what}: slot {s} was written"
    o_ref, p_ref = oracle.extend_tracked(w.q.float().numpy(), w.k.float().numpy(),
                                         w.v.float().numpy(),
                                         oracle_slopes_fp32(w.H, w.layer_id, w.L),
                                         pool0.double().numpy(), w.state_idx.numpy(),
                                         w.cu_seqlens.numpy(), w.prefix_mask.numpy(), tl, tidx,
                                         w.H, w.D)
    assert_close(to64(out_c), o_ref, f"{what}: outputs")
    named = w.state_idx.numpy()
    assert_close(to64(got[w.state_idx.long()]), p_ref[named], f"{what}: final states")
    for b in range(w.B):
        if tl[b] >= 0:
            assert_close(to64(got[tidx[b]]), p_ref[tidx[b]],
                         f"{what}: snapshot of request {b} at token {tl[b]}")


@pytest.mark.parametrize("workspace", [None, False], ids=["split", "nosplit"])
def test_snapshots_across_chunk_positions(workspace):
    lengths = [300, 128, 0, 1000, 77, 257, 640, 5]
    tl = [0, 128, 0, 999, 5, 256, 200, -1]
    w = workloads.custom_extend(lengths, H=3, layer_id=1, L=4, prefix=[1, 0, 1, 0, 1, 1, 0, 1],
                                num_slots=32, seed=31)
    _check(w, tl, _free_slots(w, w.B, 1), workspace, "chunk positions")


@pytest.mark.parametrize("tl0,tl1", [(1000, 6000), (1024, 4096), (2048, 3000), (4095, 0),
                                     (8191, 5999), (8192, 1)])
def test_snapshots_with_sequence_split(tl0, tl1):
    # two long requests and few heads: the extend cuts them into segments processed in parallel
    w = workloads.custom_extend([8192, 6000], H=2, layer_id=0, L=2, prefix=[1, 1], num_slots=8,
                                seed=32)
    assert la.extend_workspace_size(w.B, w.T, w.H, w.D, 8192) > 0
    _check(w, [tl0, tl1], _free_slots(w, 2, 2), None, f"split ({tl0}, {tl1})")


def test_snapshot_at_request_end_is_the_final_state():
    w = workloads.custom_extend([384, 1001], H=2, prefix=[0, 1], num_slots=8, seed=33)
    tidx = _free_slots(w, 2, 3)
    pool0 = w.materialize_pool()
    _, pool = _run(w, [384, 1001], tidx, pool0, None)
    la.poll_error()
    got = pool.cpu()
    for b in range(2):
        # the end-of-request snapshot is the very state written to the request's slot
        assert torch.equal(_bits(got[tidx[b]]), _bits(got[int(w.state_idx[b])]))


def test_varlen_workload_tracked_sampled():
    w = workloads.varlen_extend(0)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    rng = np.random.default_rng(4)
    tl = [int(rng.integers(0, n + 1)) for n in lens]
    tl[1] = -1
    tidx = _free_slots(w, w.B, 5)
    pool0 = w.materialize_pool()
    out, pool = _run(w, tl, tidx, pool0, None)
    la.poll_error()
    out_p, _ = _run(w, tl, tidx, pool0, None, tracked=False)
    la.poll_error()
    out_c, out_pc = out.cpu(), out_p.cpu()
    r1 = slice(int(w.cu_seqlens[1]), int(w.cu_seqlens[2]))
    assert torch.equal(out_c[r1], out_pc[r1])   # no snapshot: la_extend's chunking, bit for bit
    got = pool.cpu()
    assert torch.equal(_bits(got[tidx[1]]), _bits(pool0[tidx[1]]))
    s = oracle_slopes_fp32(w.H, w.layer_id, w.L)
    for b in (0, 3, 6):
        t0, t1 = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
        slot = int(w.state_idx[b])
        o_ref, p_ref = oracle.extend_tracked(
            w.q[t0:t1].float().numpy(), w.k[t0:t1].float().numpy(), w.v[t0:t1].float().numpy(),
            s, pool0.double().numpy(), [slot], [0, t1 - t0], [int(w.prefix_mask[b])], [tl[b]],
            [tidx[b]], w.H, w.D)
        assert_close(to64(out_c[t0:t1]), o_ref, f"varlen: outputs of request {b}")
        assert_close(to64(got[slot]), p_ref[slot], f"varlen: final state of request {b}")
        assert_close(to64(got[tidx[b]]), p_ref[tidx[b]],
                     f"varlen: snapshot of request {b} at token {tl[b]}")


def test_bad_track_entries_reported_and_skipped():
    w = workloads.custom_extend([200, 300, 150], H=2, prefix=[1, 1, 1], num_slots=12, seed=34)
    free = _free_slots(w, 3, 6)
    # request 0: length past its end; request 1: its own slot; request 2: valid
    tl = [201, 100, 150]
    tidx = [free[0], int(w.state_idx[1]), free[2]]
    pool0 = w.materialize_pool()
    out, pool = _run(w, tl, tidx, pool0, None)
    with pytest.raises(la.LAError) as e:
        la.poll_error()
    assert e.value.status == 5
    got = pool.cpu()
    assert torch.equal(_bits(got[free[0]]), _bits(pool0[free[0]]))
    out_p, pool_p = _run(w, tl, tidx, pool0, None, tracked=False)
    la.poll_error()
    assert torch.equal(out.cpu(), out_p.cpu())
    named = w.state_idx.long()
    assert torch.equal(_bits(got[named]), _bits(pool_p.cpu()[named]))
    assert torch.equal(_bits(got[free[2]]), _bits(got[int(w.state_idx[2])]))

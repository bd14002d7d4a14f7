"""Seeded random extend calls that combine the options: ragged lengths (with zero-length requests and
lengths on both sides of chunk edges), 1-4 heads, caller-given slopes from 0 to 3 (log-uniform
over six decades, plus exact zeros), random prefix flags, state-tracking snapshots at random
offsets (including 0 and the full length), and the three output layouts.  Even seeds run with the
column split (two CTAs per head, one per value-column half, for the requests that idle SMs can
take), odd seeds without it.  Every case is compared with the fp64 oracle on outputs, final
states, snapshots, and on the slots no request names.
"""
import numpy as np
import pytest
import torch

import lightning_attention_gb300 as la
import oracle
from lightning_attention_gb300 import workloads
from la_testutil import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 7))
    H = int(rng.integers(1, 5))
    edges = [0, 1, 127, 128, 129, 255, 256, 300, 511, 640]
    lengths = [int(rng.choice(edges)) if rng.random() < 0.5 else int(rng.integers(0, 700))
               for _ in range(B)]
    slopes = np.where(rng.random(H) < 0.15, 0.0, 10.0 ** rng.uniform(-6, np.log10(3), H))
    prefix = [int(x) for x in rng.integers(0, 2, B)]
    track = rng.random() < 0.6
    layout = ["packed", "per_head", "head_major"][int(rng.integers(0, 3))]
    return rng, lengths, H, slopes.astype(np.float32), prefix, track, layout


@pytest.fixture
def column_split():
    yield la.set_column_split
    la.set_column_split(True)


@pytest.mark.parametrize("seed", range(24))
def test_extend_fuzz(seed, column_split):
    column_split(seed % 2 == 0)
    rng, lengths, H, slopes, prefix, track, layout = draw_case(seed)
    B = len(lengths)
    w = workloads.custom_extend(lengths, H=H, prefix=prefix, num_slots=2 * B + 2, seed=seed)
    T = w.T
    if track:
        tl = np.array([int(rng.integers(0, n + 1)) if rng.random() < 0.8 else -1 for n in lengths],
                      dtype=np.int32)
        used = set(int(x) for x in w.state_idx.numpy())
        free = [s for s in range(w.num_slots) if s not in used]
        ti = np.array([free[b] if tl[b] >= 0 else -1 for b in range(B)], dtype=np.int32)
    pool0 = w.materialize_pool()
    pool = pool0.to(DEV)
    s_dev = torch.from_numpy(slopes).to(DEV)
    args = (w.q.to(DEV), w.k.to(DEV), w.v.to(DEV), s_dev, pool, w.state_idx.to(DEV),
            w.cu_seqlens.to(DEV), w.prefix_mask.to(DEV))
    if layout == "packed":
        out = torch.empty(T, H * 128, dtype=torch.bfloat16, device=DEV)
        view = out
    elif layout == "per_head":
        out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=DEV)
        view = out
    else:
        buf = torch.empty(H, T, 128, dtype=torch.bfloat16, device=DEV)
        view = buf.transpose(0, 1)
    kw = dict(out=view, max_seqlen=max(lengths) if lengths else 0)
    if track:
        kw.update(track_lens=torch.from_numpy(tl).to(DEV), track_state_idx=torch.from_numpy(ti).to(DEV))
    la.extend(*args, **kw)
    la.poll_error()

    qn, kn, vn = w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy()
    s64 = slopes.astype(np.float64)
    if track:
        o_ref, p_ref = oracle.extend_tracked(qn, kn, vn, s64, pool0.double().numpy(),
                                             w.state_idx.numpy(), w.cu_seqlens.numpy(),
                                             w.prefix_mask.numpy(), tl, ti, H, 128)
    else:
        o_ref, p_ref = oracle.extend(qn, kn, vn, s64, pool0.double().numpy(), w.state_idx.numpy(),
                                     w.cu_seqlens.numpy(), w.prefix_mask.numpy(), H, 128)
    got = to64(view.reshape(T, H * 128))  # a copy in token-major order for the strided view
    tag = f"seed {seed} (B={B} H={H} lengths={lengths} track={track} {layout} split={seed % 2 == 0})"
    assert_close(got, o_ref, f"{tag}: out")
    written = set(int(x) for x in w.state_idx.numpy())
    if track:
        written |= set(int(x) for x in ti if x >= 0)
    idx = np.array(sorted(written), dtype=np.int64)
    pa = pool.cpu()
    assert_close(pa.double().numpy()[idx], p_ref[idx], f"{tag}: states")
    untouched = np.ones(w.num_slots, bool)
    untouched[idx] = False
    u = torch.from_numpy(untouched)
    assert torch.equal(pa[u].view(torch.int32), pool0[u].view(torch.int32)), f"{tag}: untouched slots"
